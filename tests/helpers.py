"""Shared test helpers: moving oracle outputs to the device and the linear tolerance."""
import contextlib

import numpy as np
import torch

import oracle

# |y - y_ref| <= 1e-3 * sum_k |x_k w_k| + 2^-8 |y_ref|  (x_k, w_k the dequantized operands)
TOL_ABS = 1e-3
TOL_REL = 2.0 ** -8


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def y_to_f64(y: torch.Tensor) -> np.ndarray:
    if y.dtype == torch.bfloat16:
        return y.float().cpu().numpy().astype(np.float64)
    return y.cpu().numpy().astype(np.float64)


# A tighter, empirical bound checked beside the stated one: fp32 accumulation in any of
# the kernels' orders stays far inside 2^-14 sum|x w| at these K, plus the rounding of y
# itself (2^-8 |y| for bf16 y, its unit roundoff; 2^-23 for fp32).  One 16-element block carries roughly
# 1/(4 sqrt(K/16)) of sum|x w| with random signs -- far above 2^-14 -- so a dropped or
# misscaled block fails here even where the stated tolerance would let it pass.
TIGHT_ABS = 2.0 ** -14


def _all_bf16_values(y: np.ndarray) -> bool:
    """True when every value has a bf16 representation: then the output may have been
    stored as bf16 and the bf16 rounding term applies (for an fp32 output that happens to
    hold only bf16 values this merely loosens the tight bound)."""
    y32 = y.astype(np.float32)
    return bool(np.all((y32.view(np.uint32) & 0xFFFF) == 0))


def check_tolerance(y_gpu: np.ndarray, y_ref: np.ndarray, absdot: np.ndarray, what=""):
    err = np.abs(y_gpu - y_ref)
    bound = TOL_ABS * absdot + TOL_REL * np.abs(y_ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError("%s: %d outputs out of tolerance; worst at %s: gpu %r ref %r "
                             "bound %r" % (what, int(bad.sum()), i, y_gpu[i], y_ref[i], bound[i]))
    rel_y = 2.0 ** -8 if _all_bf16_values(y_gpu) else 2.0 ** -23
    tight = TIGHT_ABS * absdot + rel_y * np.abs(y_ref)
    bad = err > tight
    if bad.any():
        i = np.unravel_index(np.argmax(err - tight), err.shape)
        raise AssertionError("%s: %d outputs outside the empirical fp32-accumulation bound; "
                             "worst at %s: gpu %r ref %r bound %r"
                             % (what, int(bad.sum()), i, y_gpu[i], y_ref[i], tight[i]))
    return float((err / np.maximum(absdot, 1e-300)).max())


def oracle_weights(w_cpu: torch.Tensor):
    """Oracle-quantized weights: (wq, ws_rowmajor, gw) as numpy."""
    return oracle.quantize(w_cpu.numpy())


def upload_weights(wq: np.ndarray, ws: np.ndarray, gw: float, K: int):
    """Device copies of oracle-quantized weights, scales swizzled by the library."""
    import nvfp4_weight_quantized_quantize_gb300 as nv
    d_wq = to_dev(wq)
    d_ws = to_dev(ws)
    d_swz = torch.empty(nv.nvfp4_repack_bytes(wq.shape[0], K), dtype=torch.uint8, device="cuda")
    nv.nvfp4_repack(d_ws, K, d_swz)
    d_g = torch.tensor([gw], dtype=torch.float32, device="cuda")
    return d_wq, d_swz, d_g


@contextlib.contextmanager
def w4a4_kernel(which: str):
    """Run the W4A4 GEMM (M > 16) on the given kernel: "auto" (the one-CTA kernel),
    "one_cta", "pair" or "prepass" (x quantized ahead of the GEMM)."""
    import nvfp4_weight_quantized_quantize_gb300 as nv
    nv.nvfp4_debug_w4a4_kernel(which)
    try:
        yield
    finally:
        nv.nvfp4_debug_w4a4_kernel("auto")
