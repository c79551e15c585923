"""GPU parity of nvfp4_linear_silu_mul_quantize: the gate/up projection with silu(gate) * up
quantized to NVFP4 in the same pass (FlashRT docs/qwen36_usage.md, env-var table:
FLASHRT_QWEN36_FUSE_MLP_GATE_UP, then FLASHRT_QWEN36_FUSE_SILU_MUL_QUANT).

The reference is the oracle's chain: gu = bf16 rounding (through fp32) of the oracle's
fp64 linear x . W^T, then the oracle's silu(gate) * up quantizer with the same static
global scale.  On structured inputs (one nonzero x per 16-block, nonzero weight codes,
scales in {0.5, 0.75, 1, 2}: see tests/test_gpu_exact.py) the projection is exact in the
kernels' fp32 accumulators, so the codes and scale bytes must match bit for bit -- on the
fused epilogue (M > 16, I % 128 == 0) and on the two-kernel path for other shapes.  On
random inputs an fp32 accumulation may round a gate or up value to the neighbouring bf16
value, so there a small fraction of codes may differ; the test bounds it.
"""
import numpy as np
import pytest
import torch

import nvfp4_weight_quantized_quantize_gb300 as nv
import oracle
from helpers import to_dev, upload_weights
from synth import make_inputs, sparse_block_x, structured_nvfp4_weights

pytestmark = pytest.mark.gpu


def gu_reference(x, wq, ws, gw):
    """The oracle's gate/up output as the GEMM stores it: fp64 -> fp32 -> bf16 (RNE)."""
    y, _ = oracle.linear_w4a16(x, wq, ws, gw)
    return torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16)


def rowmajor_scales(atoms: np.ndarray, rows, I: int) -> np.ndarray:
    """Scale bytes of the given rows, read out of an [M, I] tensor's atom layout."""
    nb = I // 16
    out = np.empty((len(rows), nb), dtype=np.uint8)
    for i, r in enumerate(rows):
        for cb in range(nb):
            out[i, cb] = atoms[oracle.swizzle_offset(int(r), cb, I)]
    return out


def run_fused(x, wq, ws, gw, gh, I, static_weights=False):
    M, K = x.shape
    d_wq, d_swz, d_g = upload_weights(wq, ws, gw, K)
    hq = torch.full((M, I // 2), 0xAB, dtype=torch.uint8, device="cuda")
    hs = torch.full((oracle.repack_atom_bytes(M, I),), 0xAB, dtype=torch.uint8, device="cuda")
    work = torch.zeros(nv.nvfp4_workspace_bytes(2, M, K, I), dtype=torch.uint8, device="cuda")
    d_gh = torch.tensor([gh], dtype=torch.float32, device="cuda")
    nv.nvfp4_linear_silu_mul_quantize(x.cuda(), d_wq, d_swz, d_g, d_gh, hq, hs, work,
                                      static_weights=static_weights)
    torch.cuda.synchronize()
    assert nv.nvfp4_workspace_error(work) == 0
    return hq.cpu().numpy(), hs.cpu().numpy()


@pytest.mark.parametrize("M,K,I,gh", [
    (40, 5120, 256, 2.0 ** -6),     # fused epilogue, one x tile
    (300, 2048, 512, 0.01),         # fused, two x tiles, ragged M
    (17, 1024, 128, 2.0 ** -7),     # fused, M just past the small-M kernels
    (5, 5120, 256, 2.0 ** -6),      # small M: GEMV into the workspace, then the quantizer
    (40, 1024, 96, 2.0 ** -6),      # I % 128 != 0: the two-kernel path on the GEMM
])
def test_structured_bit_exact(M, K, I, gh):
    x = sparse_block_x(M, K, seed=M + I)
    wq, ws, gw = structured_nvfp4_weights(2 * I, K, seed=K + I)
    hq, hs = run_fused(x, wq, ws, gw, gh, I, static_weights=(M % 2 == 1))
    gu = gu_reference(x, wq, ws, gw)
    rq, rs, rg = oracle.silu_mul_quantize(gu, gh)
    assert rg == np.float32(gh)
    np.testing.assert_array_equal(hq, rq)
    # the whole atom area, padding included (zero), against the oracle's layout
    np.testing.assert_array_equal(hs, oracle.repack(rs, I)[:oracle.repack_atom_bytes(M, I)])


def test_mlp_chunk_sampled_rows():
    # the 512-token chunk of the fused MLP (K 5120 -> 2 x 17408): 16 sampled rows of h,
    # every column, bit for bit, on structured inputs
    M, K, I, gh = 512, 5120, 17408, 2.0 ** -6
    x = sparse_block_x(M, K, seed=77)
    wq, ws, gw = structured_nvfp4_weights(2 * I, K, seed=78)
    hq, hs = run_fused(x, wq, ws, gw, gh, I, static_weights=True)
    rows = np.sort(np.random.default_rng(0).choice(M, 16, replace=False))
    rows[0], rows[-1] = 0, M - 1
    gu = gu_reference(x[rows], wq, ws, gw)
    rq, rs, _ = oracle.silu_mul_quantize(gu, gh)
    np.testing.assert_array_equal(hq[rows], rq)
    np.testing.assert_array_equal(rowmajor_scales(hs, rows, I), rs)


@pytest.mark.parametrize("M,K,I", [(64, 1024, 256), (8, 1024, 256)])
def test_random_inputs_codes_agree(M, K, I):
    x, _ = make_inputs(M, K, 1, seed=90 + M)
    _, w = make_inputs(1, K, 2 * I, seed=91)
    wq, ws, gw = oracle.quantize(w.numpy())
    gh = 0.004
    hq, hs = run_fused(x, wq, ws, gw, gh, I)
    gu = gu_reference(x, wq, ws, gw)
    rq, rs, _ = oracle.silu_mul_quantize(gu, gh)
    # an fp32 accumulation may land a gate/up value on the other side of a bf16 rounding
    # boundary; everything else is the same arithmetic
    assert np.mean(hq == rq) > 0.98
    assert np.mean(rowmajor_scales(hs, range(M), I) == rs) > 0.98
