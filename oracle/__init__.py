"""CPU oracle for the NVFP4 block-scaled projection -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
import this package.  The product library (``nvfp4_weight_quantized_quantize_gb300``)
never imports, links or loads it, and this package imports nothing from the product.

The arithmetic lives in ``nvfp4_oracle.c`` (plain C, strict IEEE, fp64 sums); this
module only compiles it with gcc and marshals numpy arrays through ctypes.  Every
function states the definition it follows in the C file's header.

How each function is pinned (tests/test_oracle_*):
  e2m1_encode / e4m3_encode  against an independent integer formulation over every
                             fp32 bit pattern (E2M1) / every pattern of the rounding
                             window plus a strided full sweep (E4M3); closed-form
                             grids, midpoint table, 448/464/480 and 2^-9/2^-10.
  quantize                   hand-worked blocks (tests/golden), exact round trips of
                             every code x every finite scale, zero / tiny blocks,
                             element error bounds on random data.
  dequant_fp8_block128       hand-worked bf16 ties (tests/golden), per-tile powers of
                             two that expose the tile index, every byte against the
                             E4M3 closed form, torch's float8_e4m3fn decode and bf16
                             cast on random data.
  exp_f32 / silu_mul         exp within 3 ulp of fp64 exp over a dense sweep, exact at 0
                             and the clamps; silu * up within a few ulp of the fp64
                             definition; zero, saturated and signed-zero cases.
  repack                     hand-derived byte offsets, bijection, zero padding; the
                             tensor-core W4A4 result on the GPU reads the same layout.
  linear_w4a16 / _w4a4       exact rational brute force on tiny shapes, one-hot and
                             permutation special cases, fp64 matmul of the decoded
                             operands.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

# fixed compile line: strict IEEE fp32, no contraction into fused multiply-adds
CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-fvisibility=hidden"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available) and return the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    base = ["gcc"] + CFLAGS + [_SRC, "-o", tmp]
    try:
        subprocess.run(base + ["-fopenmp", "-lm"], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        U32 = ctypes.c_uint32
        F = ctypes.c_float
        sig = {
            "orc_e2m1_value": (ctypes.c_double, [U32]),
            "orc_e4m3_value": (ctypes.c_double, [U32]),
            "orc_e2m1_encode": (U32, [F]),
            "orc_e4m3_encode": (U32, [F]),
            "orc_e2m1_encode_array": (None, [P, I64, P]),
            "orc_e4m3_encode_array": (None, [P, I64, P]),
            "orc_bf16_to_f32": (F, [ctypes.c_uint16]),
            "orc_round_bf16": (ctypes.c_uint16, [ctypes.c_double]),
            "orc_round_bf16_array": (None, [P, I64, P]),
            "orc_quantize": (ctypes.c_int, [P, ctypes.c_int, I64, I64, P, P, P, P]),
            "orc_repack_bytes": (I64, [I64, I64]),
            "orc_repack_atom_bytes": (I64, [I64, I64]),
            "orc_swizzle_offset": (I64, [I64, I64, I64]),
            "orc_repack": (ctypes.c_int, [P, I64, I64, P, I64]),
            "orc_dequantize": (None, [P, P, F, I64, I64, P]),
            "orc_linear_w4a16": (ctypes.c_int, [P, I64, I64, P, P, F, I64, P, P]),
            "orc_linear_w4a16_pairs": (ctypes.c_int, [P, I64, I64, P, P, F, I64,
                                                      P, P, I64, P, P]),
            "orc_linear_w4a4": (ctypes.c_int, [P, I64, I64, P, P, F, I64, P,
                                               P, P, P, P, P]),
            "orc_linear_w4a4_pairs": (ctypes.c_int, [P, P, F, I64, I64, P, P,
                                                     F, I64, P, P, I64, P, P]),
            "orc_num_threads": (ctypes.c_int, []),
            "orc_dequant_fp8_block128": (None, [P, P, I64, I64, P]),
            "orc_exp_f32": (F, [F]),
            "orc_silu_mul_f32": (F, [F, F]),
            "orc_silu_mul": (None, [P, I64, I64, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(x) -> np.ndarray:
    """Accept a bf16 torch tensor or a uint16 array of bf16 bit patterns."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch  # only to unpack a torch bf16 tensor's bits
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy()
                                .view(np.uint16))


def num_threads() -> int:
    return int(_load().orc_num_threads())


# --- value sets -------------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return _load().orc_e2m1_value(int(code))


def e4m3_value(byte: int) -> float:
    return _load().orc_e4m3_value(int(byte))


def e2m1_encode(v) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(v, dtype=np.float32).ravel())
    out = np.empty(a.size, dtype=np.uint8)
    _load().orc_e2m1_encode_array(_ptr(a), a.size, _ptr(out))
    return out.reshape(np.shape(v))


def e4m3_encode(v) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(v, dtype=np.float32).ravel())
    out = np.empty(a.size, dtype=np.uint8)
    _load().orc_e4m3_encode_array(_ptr(a), a.size, _ptr(out))
    return out.reshape(np.shape(v))


def round_bf16(v) -> np.ndarray:
    """fp64 -> fp32 (RN) -> bf16 (RNE), returned as uint16 bit patterns."""
    a = np.ascontiguousarray(np.asarray(v, dtype=np.float64).ravel())
    out = np.empty(a.size, dtype=np.uint16)
    _load().orc_round_bf16_array(_ptr(a), a.size, _ptr(out))
    return out.reshape(np.shape(v))


def bf16_to_f32(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --- quantizer and layout -----------------------------------------------------------

def quantize(src, global_scale: float | None = None):
    """Quantize a 2-D fp32 array (or a bf16 torch tensor / uint16 bf16 bit patterns).

    Returns (packed uint8 [R, C/2], scales uint8 [R, C/16] row-major, g float)."""
    import torch
    if isinstance(src, torch.Tensor) and src.dtype == torch.bfloat16:
        a, is_bf16 = _bf16_bits(src), 1
    elif isinstance(src, np.ndarray) and src.dtype == np.uint16:
        a, is_bf16 = np.ascontiguousarray(src), 1
    else:
        if isinstance(src, torch.Tensor):
            src = src.detach().cpu().numpy()
        a, is_bf16 = np.ascontiguousarray(src, dtype=np.float32), 0
    rows, cols = a.shape
    packed = np.empty((rows, cols // 2), dtype=np.uint8)
    scales = np.empty((rows, cols // 16), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    gin = None if global_scale is None else np.array([global_scale], dtype=np.float32)
    rc = _load().orc_quantize(_ptr(a), is_bf16, rows, cols,
                              None if gin is None else _ptr(gin),
                              _ptr(packed), _ptr(scales), _ptr(g))
    if rc != 0:
        raise ValueError("oracle quantize: non-finite input, bad global scale or cols % 16")
    return packed, scales, float(g[0])


def dequant_fp8_block128(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """R10: E4M3 bytes [R, C] and fp32 tile scales [ceil(R/128), ceil(C/128)] -> the bf16
    tensor bf16(e4m3(q) * s) as uint16 bit patterns [R, C]."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.float32)
    rows, cols = q.shape
    assert s.shape == ((rows + 127) // 128, (cols + 127) // 128)
    out = np.empty((rows, cols), dtype=np.uint16)
    _load().orc_dequant_fp8_block128(_ptr(q), _ptr(s), rows, cols, _ptr(out))
    return out


def quantize_fp8_block128(q: np.ndarray, s: np.ndarray):
    """FP8 block-128 weights -> BF16 -> NVFP4 (R10, then R1-R9): (packed, scales, g)."""
    return quantize(dequant_fp8_block128(q, s))


def exp_f32(x: float) -> float:
    """R11's fp32 exp (Cody-Waite reduction, degree-7 Taylor polynomial)."""
    return float(_load().orc_exp_f32(float(x)))


def silu_mul_f32(g: float, u: float) -> float:
    return float(_load().orc_silu_mul_f32(float(g), float(u)))


def silu_mul(gate_up) -> np.ndarray:
    """R11: bf16 gate_up [M, 2I] (torch bf16 or uint16 bits) -> fp32 h [M, I]."""
    a = _bf16_bits(gate_up)
    M, I2 = a.shape
    assert I2 % 2 == 0
    h = np.empty((M, I2 // 2), dtype=np.float32)
    _load().orc_silu_mul(_ptr(a), M, I2 // 2, _ptr(h))
    return h


def silu_mul_quantize(gate_up, global_scale: float | None = None):
    """R11 then R1-R9: (packed [M, I/2], scales [M, I/16] row-major, g)."""
    return quantize(silu_mul(gate_up), global_scale)


def repack_bytes(rows: int, cols: int) -> int:
    return int(_load().orc_repack_bytes(rows, cols))


def repack_atom_bytes(rows: int, cols: int) -> int:
    return int(_load().orc_repack_atom_bytes(rows, cols))


def swizzle_offset(r: int, cb: int, cols: int) -> int:
    return int(_load().orc_swizzle_offset(r, cb, cols))


def repack(scales: np.ndarray, cols: int) -> np.ndarray:
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    rows = s.shape[0]
    n = repack_bytes(rows, cols)
    out = np.empty(n, dtype=np.uint8)
    if _load().orc_repack(_ptr(s), rows, cols, _ptr(out), n) != 0:
        raise ValueError("oracle repack: bad shape")
    return out


def dequantize(packed: np.ndarray, scales: np.ndarray, g: float, cols: int) -> np.ndarray:
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    rows = p.shape[0]
    out = np.empty((rows, cols), dtype=np.float64)
    _load().orc_dequantize(_ptr(p), _ptr(s), g, rows, cols, _ptr(out))
    return out


# --- linear -------------------------------------------------------------------------

def linear_w4a16(x, wq: np.ndarray, ws: np.ndarray, gw: float):
    """y = x . dequant(W)^T in fp64, and the tolerance reference sum_k |x w|."""
    xb = _bf16_bits(x)
    M, K = xb.shape
    N = wq.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    ab = np.empty((M, N), dtype=np.float64)
    rc = _load().orc_linear_w4a16(_ptr(xb), M, K, _ptr(np.ascontiguousarray(wq)),
                                  _ptr(np.ascontiguousarray(ws)), gw, N, _ptr(y), _ptr(ab))
    if rc != 0:
        raise ValueError("oracle linear: K % 16 != 0")
    return y, ab


def linear_w4a16_pairs(x, wq, ws, gw, pm, pn):
    xb = _bf16_bits(x)
    M, K = xb.shape
    N = wq.shape[0]
    pm = np.ascontiguousarray(pm, dtype=np.int64)
    pn = np.ascontiguousarray(pn, dtype=np.int64)
    y = np.empty(pm.size, dtype=np.float64)
    ab = np.empty(pm.size, dtype=np.float64)
    rc = _load().orc_linear_w4a16_pairs(_ptr(xb), M, K, _ptr(np.ascontiguousarray(wq)),
                                        _ptr(np.ascontiguousarray(ws)), gw, N, _ptr(pm),
                                        _ptr(pn), pm.size, _ptr(y), _ptr(ab))
    if rc != 0:
        raise ValueError("oracle linear pairs: bad index or K")
    return y, ab


def linear_w4a4(x, wq, ws, gw, global_scale_x: float | None = None):
    """Quantize x (bf16), then y = dequant(x) . dequant(W)^T in fp64.

    Returns (y, absdot, xq, xs_rowmajor, gx)."""
    xb = _bf16_bits(x)
    M, K = xb.shape
    N = wq.shape[0]
    xq = np.empty((M, K // 2), dtype=np.uint8)
    xs = np.empty((M, K // 16), dtype=np.uint8)
    gx = np.zeros(1, dtype=np.float32)
    gin = None if global_scale_x is None else np.array([global_scale_x], dtype=np.float32)
    y = np.empty((M, N), dtype=np.float64)
    ab = np.empty((M, N), dtype=np.float64)
    rc = _load().orc_linear_w4a4(_ptr(xb), M, K, _ptr(np.ascontiguousarray(wq)),
                                 _ptr(np.ascontiguousarray(ws)), gw, N,
                                 None if gin is None else _ptr(gin), _ptr(xq), _ptr(xs),
                                 _ptr(gx), _ptr(y), _ptr(ab))
    if rc != 0:
        raise ValueError("oracle linear w4a4: bad input")
    return y, ab, xq, xs, float(gx[0])


def linear_w4a4_pairs(xq, xs, gx, wq, ws, gw, pm, pn):
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    M, K = xq.shape[0], xq.shape[1] * 2
    N = wq.shape[0]
    pm = np.ascontiguousarray(pm, dtype=np.int64)
    pn = np.ascontiguousarray(pn, dtype=np.int64)
    y = np.empty(pm.size, dtype=np.float64)
    ab = np.empty(pm.size, dtype=np.float64)
    rc = _load().orc_linear_w4a4_pairs(_ptr(xq), _ptr(np.ascontiguousarray(xs)), gx, M, K,
                                       _ptr(np.ascontiguousarray(wq)),
                                       _ptr(np.ascontiguousarray(ws)), gw, N, _ptr(pm),
                                       _ptr(pn), pm.size, _ptr(y), _ptr(ab))
    if rc != 0:
        raise ValueError("oracle w4a4 pairs: bad index or K")
    return y, ab
