"""Python binding of libnvfp4.so (include/nvfp4.h) -- argument marshalling only.

Every function has the name of the C entry point it calls, takes torch tensors (device
memory of the current CUDA device) and raises ``Nvfp4Error`` on a non-OK status.  All
compute runs in the library's CUDA kernels; there is no other path: if the library
is missing, importing the functions' backend raises.

  nvfp4_quantize(src, packed, scales, global_scale, workspace)      weights -> NVFP4
  nvfp4_repack(scales, cols, out)                                   scale swizzle
  nvfp4_linear(x, w_packed, w_scales_swizzled, w_global_scale, y,
               mode="w4a16"|"w4a4", x_global_scale=None, workspace=None)
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libnvfp4.so")

NVFP4_F32, NVFP4_BF16 = 0, 1
NVFP4_W4A16, NVFP4_W4A4 = 0, 1
NVFP4_STATIC_WEIGHTS = 0x10  # flag OR-ed into the mode (see nvfp4_linear)
STATUS = {0: "NVFP4_OK", 1: "NVFP4_ERR_NULL", 2: "NVFP4_ERR_SHAPE", 3: "NVFP4_ERR_ALIGN",
          4: "NVFP4_ERR_DTYPE", 5: "NVFP4_ERR_WORKSPACE", 6: "NVFP4_ERR_DEVICE",
          7: "NVFP4_ERR_CUDA", 8: "NVFP4_ERR_TIMEOUT", 9: "NVFP4_ERR_UNSUPPORTED"}
EXPORTS = ("nvfp4_quantize", "nvfp4_repack", "nvfp4_linear", "nvfp4_repack_bytes",
           "nvfp4_workspace_bytes", "nvfp4_w4a4_workspace_layout", "nvfp4_workspace_error",
           "nvfp4_status_str", "nvfp4_encode_elements", "nvfp4_quantize_noalloc",
           "nvfp4_last_cuda_error", "nvfp4_quantize_fp8_block128", "nvfp4_silu_mul_quantize",
           "nvfp4_linear_nvfp4_x", "nvfp4_linear_silu_mul_quantize",
           "nvfp4_debug_expire_waits", "nvfp4_debug_w4a4_kernel")


class Nvfp4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, STATUS.get(status, str(status))))


_lib = None


def load(path: str = LIB_PATH):
    """Load libnvfp4.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libnvfp4.so is not built (%s); run "
                           "`python -m nvfp4_weight_quantized_quantize_gb300.build_lib`" % path)
    lib = ctypes.CDLL(path)
    P, I64, SZ, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
    sig = {
        "nvfp4_quantize": (I, [P, I, I64, I64, P, P, P, P, SZ, P]),
        "nvfp4_repack": (I, [P, I64, I64, P, SZ, P]),
        "nvfp4_linear": (I, [P, I64, I64, P, P, P, I64, P, I, I, P, P, SZ, P]),
        "nvfp4_repack_bytes": (SZ, [I64, I64]),
        "nvfp4_workspace_bytes": (SZ, [I, I64, I64, I64, I]),
        "nvfp4_w4a4_workspace_layout": (I, [I64, I64, ctypes.POINTER(SZ), ctypes.POINTER(SZ),
                                            ctypes.POINTER(SZ)]),
        "nvfp4_workspace_error": (I, [P, P, ctypes.POINTER(ctypes.c_uint32)]),
        "nvfp4_status_str": (ctypes.c_char_p, [I]),
        "nvfp4_encode_elements": (I, [P, I64, P, P, P]),
        "nvfp4_quantize_noalloc": (I, [P, I, I64, I64, P, P, P, P]),
        "nvfp4_last_cuda_error": (ctypes.c_char_p, []),
        "nvfp4_debug_expire_waits": (None, [I]),
        "nvfp4_debug_w4a4_kernel": (None, [I]),
        "nvfp4_quantize_fp8_block128": (I, [P, P, I64, I64, P, P, P, P, SZ, P]),
        "nvfp4_silu_mul_quantize": (I, [P, I64, I64, P, P, SZ, P, P, P, SZ, P]),
        "nvfp4_linear_nvfp4_x": (I, [P, P, P, I64, I64, P, P, P, I64, P, I, I, P, SZ, P]),
        "nvfp4_linear_silu_mul_quantize": (I, [P, I64, I64, P, P, P, I64, P, P, P, SZ, I, P,
                                               SZ, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(st: int, where: str):
    if st != 0:
        if st == 7:
            where = "%s (%s)" % (where, load().nvfp4_last_cuda_error().decode())
        raise Nvfp4Error(st, where)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return NVFP4_F32
    if dt == torch.bfloat16:
        return NVFP4_BF16
    raise ValueError("unsupported dtype %s" % dt)


# ---- host helpers -------------------------------------------------------------------

def nvfp4_status_str(status: int) -> str:
    return load().nvfp4_status_str(status).decode()


def nvfp4_repack_bytes(rows: int, cols: int) -> int:
    return int(load().nvfp4_repack_bytes(rows, cols))


def nvfp4_workspace_bytes(op: int, M: int, K: int, N: int = 0, mode: int = NVFP4_W4A16) -> int:
    return int(load().nvfp4_workspace_bytes(op, M, K, N, mode))


def nvfp4_w4a4_workspace_layout(M: int, K: int):
    a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().nvfp4_w4a4_workspace_layout(M, K, ctypes.byref(a), ctypes.byref(b),
                                              ctypes.byref(c)), "nvfp4_w4a4_workspace_layout")
    return a.value, b.value, c.value


def nvfp4_workspace_error(workspace: torch.Tensor, stream=None) -> int:
    bits = ctypes.c_uint32(0)
    st = load().nvfp4_workspace_error(_p(workspace), _stream(stream), ctypes.byref(bits))
    if st not in (0, 8):
        _check(st, "nvfp4_workspace_error")
    return bits.value


# ---- the three calls -----------------------------------------------------------------

def nvfp4_quantize(src: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
                   global_scale: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    rows, cols = src.shape
    st = load().nvfp4_quantize(_p(src), _dtype_code(src.dtype), rows, cols, _p(packed),
                               _p(scales), _p(global_scale), _p(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "nvfp4_quantize")


def nvfp4_quantize_noalloc(src: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
                           global_scale: torch.Tensor, stream=None) -> None:
    """nvfp4_quantize without a workspace, for callers that cannot allocate: its scratch
    is a fixed array inside the library, shared by every call on the device (order
    calls that could overlap on the GPU)."""
    rows, cols = src.shape
    st = load().nvfp4_quantize_noalloc(_p(src), _dtype_code(src.dtype), rows, cols, _p(packed),
                                       _p(scales), _p(global_scale), _stream(stream))
    _check(st, "nvfp4_quantize_noalloc")


def nvfp4_quantize_fp8_block128(src: torch.Tensor, block_scales: torch.Tensor,
                                packed: torch.Tensor, scales: torch.Tensor,
                                global_scale: torch.Tensor, workspace: torch.Tensor,
                                stream=None) -> None:
    """FP8 E4M3 weights (uint8 bytes [rows, cols]) with fp32 scales per 128 x 128 tile
    ([ceil(rows/128), ceil(cols/128)]) to NVFP4 through bf16."""
    rows, cols = src.shape
    if src.dtype != torch.uint8 or block_scales.dtype != torch.float32:
        raise ValueError("src must be uint8 E4M3 bytes and block_scales float32")
    if tuple(block_scales.shape) != ((rows + 127) // 128, (cols + 127) // 128):
        raise ValueError("block_scales must be [ceil(rows/128), ceil(cols/128)]")
    st = load().nvfp4_quantize_fp8_block128(_p(src), _p(block_scales), rows, cols, _p(packed),
                                            _p(scales), _p(global_scale), _p(workspace),
                                            workspace.numel() * workspace.element_size(),
                                            _stream(stream))
    _check(st, "nvfp4_quantize_fp8_block128")


def nvfp4_repack(scales: torch.Tensor, cols: int, out: torch.Tensor, stream=None) -> None:
    rows = scales.shape[0]
    st = load().nvfp4_repack(_p(scales), rows, cols, _p(out), out.numel() * out.element_size(),
                             _stream(stream))
    _check(st, "nvfp4_repack")


def nvfp4_linear(x: torch.Tensor, w_packed: torch.Tensor, w_scales_swizzled: torch.Tensor,
                 w_global_scale: torch.Tensor, y: torch.Tensor, mode: str = "w4a16",
                 x_global_scale: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None, stream=None,
                 static_weights: bool = False) -> None:
    """static_weights: no kernel still in flight on the stream writes the weights
    (NVFP4_STATIC_WEIGHTS), so the decode kernels may stream them early."""
    M, K = x.shape
    N = w_packed.shape[0]
    m = {"w4a16": NVFP4_W4A16, "w4a4": NVFP4_W4A4}[mode]
    if static_weights:
        m |= NVFP4_STATIC_WEIGHTS
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().nvfp4_linear(_p(x), M, K, _p(w_packed), _p(w_scales_swizzled),
                             _p(w_global_scale), N, _p(y), _dtype_code(y.dtype), m,
                             _p(x_global_scale), _p(workspace), wsb, _stream(stream))
    _check(st, "nvfp4_linear")


def nvfp4_silu_mul_quantize(gate_up: torch.Tensor, packed: torch.Tensor,
                            scales_swizzled: torch.Tensor, global_scale: torch.Tensor,
                            given_global_scale: torch.Tensor | None = None,
                            workspace: torch.Tensor | None = None, stream=None) -> None:
    """bf16 gate_up [M, 2I] (gate, then up) -> NVFP4 codes of silu(gate) * up, scale atoms
    and the global scale (dynamic, or a copy of the given static one)."""
    M, I2 = gate_up.shape
    if gate_up.dtype != torch.bfloat16 or I2 % 2:
        raise ValueError("gate_up must be bf16 [M, 2I]")
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().nvfp4_silu_mul_quantize(_p(gate_up), M, I2 // 2, _p(packed), _p(scales_swizzled),
                                        scales_swizzled.numel() * scales_swizzled.element_size(),
                                        _p(global_scale), _p(given_global_scale), _p(workspace),
                                        wsb, _stream(stream))
    _check(st, "nvfp4_silu_mul_quantize")


def nvfp4_linear_nvfp4_x(x_packed: torch.Tensor, x_scales_swizzled: torch.Tensor,
                         x_global_scale: torch.Tensor, w_packed: torch.Tensor,
                         w_scales_swizzled: torch.Tensor, w_global_scale: torch.Tensor,
                         y: torch.Tensor, workspace: torch.Tensor, stream=None,
                         static_weights: bool = False) -> None:
    """y = x . W^T with NVFP4 x (codes [M, K/2], scale atoms, g_x)."""
    M, K = x_packed.shape[0], x_packed.shape[1] * 2
    N = w_packed.shape[0]
    st = load().nvfp4_linear_nvfp4_x(_p(x_packed), _p(x_scales_swizzled), _p(x_global_scale), M,
                                     K, _p(w_packed), _p(w_scales_swizzled), _p(w_global_scale),
                                     N, _p(y), _dtype_code(y.dtype),
                                     NVFP4_STATIC_WEIGHTS if static_weights else 0,
                                     _p(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream))
    _check(st, "nvfp4_linear_nvfp4_x")


def nvfp4_linear_silu_mul_quantize(x: torch.Tensor, w_packed: torch.Tensor,
                                   w_scales_swizzled: torch.Tensor, w_global_scale: torch.Tensor,
                                   h_global_scale: torch.Tensor, h_packed: torch.Tensor,
                                   h_scales_swizzled: torch.Tensor, workspace: torch.Tensor,
                                   stream=None, static_weights: bool = False) -> None:
    """The gate/up projection (W = [gate; up], 2I rows) with silu(gate) * up quantized to
    NVFP4 (static global scale) in the same pass: h codes [M, I/2] and scale atoms."""
    M, K = x.shape
    I = w_packed.shape[0] // 2
    st = load().nvfp4_linear_silu_mul_quantize(
        _p(x), M, K, _p(w_packed), _p(w_scales_swizzled), _p(w_global_scale), I,
        _p(h_global_scale), _p(h_packed), _p(h_scales_swizzled),
        h_scales_swizzled.numel() * h_scales_swizzled.element_size(),
        NVFP4_STATIC_WEIGHTS if static_weights else 0, _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "nvfp4_linear_silu_mul_quantize")


def nvfp4_debug_expire_waits(on: bool) -> None:
    """Test switch: the calling thread's next nvfp4_linear kernels make a bounded wait run
    out (see include/nvfp4.h)."""
    load().nvfp4_debug_expire_waits(1 if on else 0)


W4A4_KERNELS = {"auto": 0, "one_cta": 1, "pair": 2, "prepass": 3}


def nvfp4_debug_w4a4_kernel(which: str) -> None:
    """Test switch: the kernel of the calling thread's W4A4 GEMMs at M > 16 -- "auto" (the
    default, the one-CTA kernel), "one_cta", "pair" (CTA pairs) or "prepass" (x quantized
    by the quantizer kernels ahead of the GEMM); see include/nvfp4.h."""
    load().nvfp4_debug_w4a4_kernel(W4A4_KERNELS[which])


def nvfp4_encode_elements(inp: torch.Tensor, e2m1_out: torch.Tensor | None,
                          e4m3_out: torch.Tensor | None, stream=None) -> None:
    st = load().nvfp4_encode_elements(_p(inp), inp.numel(), _p(e2m1_out), _p(e4m3_out),
                                      _stream(stream))
    _check(st, "nvfp4_encode_elements")


# ---- convenience: allocate outputs with torch and run the calls -----------------------

def quantize_weight(w: torch.Tensor, stream=None):
    """Quantize + repack a device weight [N, K]; returns (packed, scales_rowmajor,
    scales_swizzled, global_scale)."""
    N, K = w.shape
    dev = w.device
    packed = torch.empty(N, K // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(N, K // 16, dtype=torch.uint8, device=dev)
    g = torch.empty(1, dtype=torch.float32, device=dev)
    ws = torch.empty(nvfp4_workspace_bytes(0, N, K), dtype=torch.uint8, device=dev)
    nvfp4_quantize(w, packed, scales, g, ws, stream)
    swz = torch.empty(nvfp4_repack_bytes(N, K), dtype=torch.uint8, device=dev)
    nvfp4_repack(scales, K, swz, stream)
    return packed, scales, swz, g
