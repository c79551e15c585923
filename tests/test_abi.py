"""The C-ABI library loads, exports every function include/nvfp4.h declares, and its
host-side argument checks reject bad calls before anything is enqueued.

Every call below has at least one argument that the host checks reject (the checks run
before the device is queried), so no kernel is launched even where a GPU is present.
"""
import ctypes
import os
import re
import subprocess

import pytest

import nvfp4_weight_quantized_quantize_gb300 as nv
from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "nvfp4.h")
OK, NULL, SHAPE, ALIGN, DTYPE, WORKSPACE = 0, 1, 2, 3, 4, 5


@pytest.fixture(scope="module")
def lib():
    from nvfp4_weight_quantized_quantize_gb300 import build_lib
    build_lib.build()
    return nv.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(nv.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", nv.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r"\bT (nvfp4_[a-z0-9_]+)", out))
    assert exported == set(declared_functions())


def test_header_is_plain_c():
    # the boundary is a C ABI: the header alone must compile as C99 and as C++
    for lang, std in (("c", "-std=c99"), ("c++", "-std=c++17")):
        out = subprocess.run(["gcc", std, "-Wall", "-Wextra", "-pedantic", "-Werror",
                              "-fsyntax-only", "-x", lang, HEADER], capture_output=True,
                             text=True)
        assert out.returncode == 0, out.stderr


def test_c_program_links_and_calls_host_helpers(lib, tmp_path):
    # a plain C caller links against the library and uses the host-only helpers (no
    # device work): sizes, status strings and a rejected call
    src = tmp_path / "caller.c"
    src.write_text(r"""
#include <stdio.h>
#include "nvfp4.h"
int main(void) {
    if (nvfp4_repack_bytes(17408, 5120) != (size_t)2 * 17408 * 320 + 16) return 1;
    if (nvfp4_workspace_bytes(1, 1, 48, 4, NVFP4_W4A16) != (size_t)-1) return 2;
    if (nvfp4_linear(NULL, 1, 64, NULL, NULL, NULL, 8, NULL, NVFP4_BF16, NVFP4_W4A16, NULL,
                     NULL, 0, NULL) != NVFP4_ERR_NULL) return 3;
    puts(nvfp4_status_str(NVFP4_ERR_SHAPE));
    return 0;
}
""")
    exe = tmp_path / "caller"
    libdir = os.path.dirname(nv.LIB_PATH)
    out = subprocess.run(["gcc", "-std=c99", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe),
                          "-L", libdir, "-lnvfp4", "-Wl,-rpath," + libdir],
                         capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0, (run.returncode, run.stderr)
    assert run.stdout.strip() == nv.nvfp4_status_str(2)


def test_status_strings(lib):
    for code in range(10):
        assert nv.nvfp4_status_str(code).startswith(nv.STATUS[code])


def test_size_helpers(lib):
    assert nv.nvfp4_repack_bytes(17408, 5120) == 2 * 17408 * 320 + 16
    assert nv.nvfp4_repack_bytes(1, 16) == 512 + 16 + 16
    assert nv.nvfp4_repack_bytes(129, 80) == 256 * 8 + 656 + 16
    assert nv.nvfp4_repack_bytes(0, 16) == 0 and nv.nvfp4_repack_bytes(4, 24) == 0
    assert nv.nvfp4_workspace_bytes(1, 1, 5120, 17408, nv.NVFP4_W4A16) == 256
    assert nv.nvfp4_workspace_bytes(1, 512, 5120, 34816, nv.NVFP4_W4A16) > 0
    assert nv.nvfp4_workspace_bytes(0, 10, 48) > 0
    assert nv.nvfp4_workspace_bytes(1, 1, 48, 4, nv.NVFP4_W4A16) == 2 ** 64 - 1  # K % 32
    xq, xs, gx = nv.nvfp4_w4a4_workspace_layout(2048, 5120)
    assert xq >= 4 and xs >= xq + 2048 * 2560 and gx >= xs + 2048 * 320
    assert xq % 16 == 0 and xs % 16 == 0 and gx % 4 == 0
    total = nv.nvfp4_workspace_bytes(1, 2048, 5120, 17408, nv.NVFP4_W4A4)
    assert total >= gx + 4


def _q(lib, src=16, dt=0, rows=4, cols=32, packed=32, scales=48, g=64, ws=4096,
       wsb=1 << 20):
    v = lambda a: None if a is None else ctypes.c_void_p(a)
    return lib.nvfp4_quantize(v(src), dt, rows, cols, v(packed), v(scales), v(g), v(ws), wsb,
                              None)


def test_quantize_rejects(lib):
    assert _q(lib, src=None) == NULL
    assert _q(lib, g=None) == NULL
    assert _q(lib, ws=None) == NULL
    assert _q(lib, dt=7) == DTYPE
    assert _q(lib, cols=24) == SHAPE
    assert _q(lib, rows=0) == SHAPE
    assert _q(lib, cols=8) == SHAPE
    assert _q(lib, src=17) == ALIGN
    assert _q(lib, packed=40) == ALIGN
    assert _q(lib, g=66) == ALIGN
    assert _q(lib, wsb=16) == WORKSPACE


def _qn(lib, src=16, dt=0, rows=4, cols=32, packed=32, scales=48, g=64):
    v = lambda a: None if a is None else ctypes.c_void_p(a)
    return lib.nvfp4_quantize_noalloc(v(src), dt, rows, cols, v(packed), v(scales), v(g),
                                      None)


def test_quantize_noalloc_rejects(lib):
    # the same host checks as nvfp4_quantize, less the workspace's
    assert _qn(lib, src=None) == NULL
    assert _qn(lib, packed=None) == NULL
    assert _qn(lib, scales=None) == NULL
    assert _qn(lib, g=None) == NULL
    assert _qn(lib, dt=7) == DTYPE
    assert _qn(lib, cols=24) == SHAPE
    assert _qn(lib, rows=0) == SHAPE
    assert _qn(lib, cols=8) == SHAPE
    assert _qn(lib, rows=(1 << 30) + 1) == SHAPE
    assert _qn(lib, src=17) == ALIGN
    assert _qn(lib, scales=56) == ALIGN
    assert _qn(lib, g=66) == ALIGN


def _q8(lib, src=16, bs=20, rows=4, cols=32, packed=32, scales=48, g=64, ws=4096,
        wsb=1 << 20):
    v = lambda a: None if a is None else ctypes.c_void_p(a)
    return lib.nvfp4_quantize_fp8_block128(v(src), v(bs), rows, cols, v(packed), v(scales),
                                           v(g), v(ws), wsb, None)


def test_quantize_fp8_block128_rejects(lib):
    assert _q8(lib, src=None) == NULL
    assert _q8(lib, bs=None) == NULL
    assert _q8(lib, ws=None) == NULL
    assert _q8(lib, cols=24) == SHAPE
    assert _q8(lib, rows=0) == SHAPE
    assert _q8(lib, src=17) == ALIGN
    assert _q8(lib, bs=22) == ALIGN
    assert _q8(lib, scales=40) == ALIGN
    assert _q8(lib, wsb=16) == WORKSPACE


def _sq(lib, gu=16, M=4, I=32, packed=32, sc=48, scb=512, g=64, given=None, ws=4096,
        wsb=1 << 20):
    v = lambda a: None if a is None else ctypes.c_void_p(a)
    return lib.nvfp4_silu_mul_quantize(v(gu), M, I, v(packed), v(sc), scb, v(g), v(given),
                                       v(ws), wsb, None)


def test_silu_mul_quantize_rejects(lib):
    assert _sq(lib, gu=None) == NULL
    assert _sq(lib, g=None) == NULL
    assert _sq(lib, ws=None) == NULL            # dynamic scale needs the workspace
    assert _sq(lib, I=24) == SHAPE
    assert _sq(lib, M=0) == SHAPE
    assert _sq(lib, scb=511) == SHAPE           # 128 rows x 4 blocks of atoms
    assert _sq(lib, gu=24) == ALIGN
    assert _sq(lib, given=66, ws=None) == ALIGN
    assert _sq(lib, wsb=16) == WORKSPACE


def _lx(lib, xq=16, xs=32, gx=48, M=4, K=64, wq=64, wsz=80, gw=96, N=8, y=112, ydt=1, flags=0,
        ws=4096, wsb=1 << 20):
    v = lambda a: None if a is None else ctypes.c_void_p(a)
    return lib.nvfp4_linear_nvfp4_x(v(xq), v(xs), v(gx), M, K, v(wq), v(wsz), v(gw), N, v(y),
                                    ydt, flags, v(ws), wsb, None)


def test_linear_nvfp4_x_rejects(lib):
    assert _lx(lib, xq=None) == NULL
    assert _lx(lib, gx=None) == NULL
    assert _lx(lib, ws=None) == NULL
    assert _lx(lib, ydt=3) == DTYPE
    assert _lx(lib, flags=1) == DTYPE
    assert _lx(lib, K=48) == SHAPE
    assert _lx(lib, N=0) == SHAPE
    assert _lx(lib, xs=40) == ALIGN
    assert _lx(lib, gx=50) == ALIGN
    assert _lx(lib, wsb=64) == WORKSPACE


def _ls(lib, x=16, M=4, K=64, wq=32, wsz=48, gw=64, I=32, gh=80, hq=96, hs=112, hsb=512,
        flags=0, ws=4096, wsb=1 << 20):
    v = lambda a: None if a is None else ctypes.c_void_p(a)
    return lib.nvfp4_linear_silu_mul_quantize(v(x), M, K, v(wq), v(wsz), v(gw), I, v(gh),
                                              v(hq), v(hs), hsb, flags, v(ws), wsb, None)


def test_linear_silu_mul_quantize_rejects(lib):
    assert _ls(lib, x=None) == NULL
    assert _ls(lib, gh=None) == NULL            # the activation scale is static
    assert _ls(lib, hq=None) == NULL
    assert _ls(lib, ws=None) == NULL
    assert _ls(lib, flags=1) == DTYPE
    assert _ls(lib, K=48) == SHAPE
    assert _ls(lib, I=24) == SHAPE
    assert _ls(lib, M=0) == SHAPE
    assert _ls(lib, hsb=511) == SHAPE           # 128 rows x 4 blocks of atoms
    assert _ls(lib, x=24) == ALIGN
    assert _ls(lib, hs=120) == ALIGN
    assert _ls(lib, gh=82) == ALIGN
    assert _ls(lib, wsb=16) == WORKSPACE


def test_linear_silu_mul_quantize_workspace_sizes():
    # fused (M > 16, I % 128 == 0): the error word alone; otherwise room for gu [M, 2I] bf16
    # fused path: the GEMM's stream-K state on 2I rows
    assert nv.nvfp4_workspace_bytes(2, 512, 5120, 17408) == \
        nv.nvfp4_workspace_bytes(1, 512, 5120, 2 * 17408, nv.NVFP4_W4A16)
    assert nv.nvfp4_workspace_bytes(2, 4, 5120, 17408) >= 256 + 4 * 2 * 17408 * 2
    assert nv.nvfp4_workspace_bytes(2, 40, 64, 96) >= 40 * 2 * 96 * 2
    assert nv.nvfp4_workspace_bytes(2, 40, 64, 24) == 2 ** 64 - 1


def _r(lib, src=16, rows=4, cols=32, out=32, nbytes=None):
    v = lambda a: None if a is None else ctypes.c_void_p(a)
    if nbytes is None:
        nbytes = nv.nvfp4_repack_bytes(rows, max(cols, 16)) or 512
    return lib.nvfp4_repack(v(src), rows, cols, v(out), nbytes, None)


def test_repack_rejects(lib):
    assert _r(lib, src=None) == NULL
    assert _r(lib, out=None) == NULL
    assert _r(lib, cols=20) == SHAPE
    assert _r(lib, rows=0) == SHAPE
    assert _r(lib, nbytes=511) == SHAPE
    assert _r(lib, out=8) == ALIGN


def _l(lib, x=16, M=1, K=64, wq=32, wsz=48, gw=64, N=8, y=80, ydt=1, mode=0, gx=None,
       ws=None, wsb=0):
    v = lambda a: None if a is None else ctypes.c_void_p(a)
    return lib.nvfp4_linear(v(x), M, K, v(wq), v(wsz), v(gw), N, v(y), ydt, mode, v(gx),
                            v(ws), wsb, None)


def test_linear_rejects(lib):
    assert _l(lib, x=None) == NULL
    assert _l(lib, gw=None) == NULL
    assert _l(lib, y=None) == NULL
    assert _l(lib, ydt=5) == DTYPE
    assert _l(lib, mode=3) == DTYPE
    assert _l(lib, gx=128) == DTYPE            # a static x scale needs W4A4
    assert _l(lib, K=48) == SHAPE              # K % 32
    assert _l(lib, K=0) == SHAPE
    assert _l(lib, M=0) == SHAPE
    assert _l(lib, N=0) == SHAPE
    assert _l(lib, x=24) == ALIGN
    assert _l(lib, y=88) == ALIGN
    assert _l(lib, gw=66) == ALIGN
    assert _l(lib, mode=1) == WORKSPACE        # W4A4 needs its workspace
    assert _l(lib, mode=1, ws=4096, wsb=64) == WORKSPACE
    assert _l(lib, M=512, K=64, N=8) == WORKSPACE  # every path needs the error word
    assert _l(lib, M=1, K=64, N=8) == WORKSPACE
    assert _l(lib, M=1, K=64, N=8, ws=4096, wsb=255) == WORKSPACE


def test_encode_elements_rejects(lib):
    assert lib.nvfp4_encode_elements(None, 4, None, None, None) == NULL
    assert lib.nvfp4_encode_elements(ctypes.c_void_p(16), -1, None, None, None) == SHAPE
    assert lib.nvfp4_encode_elements(ctypes.c_void_p(18), 4, None, None, None) == ALIGN


def test_workspace_error_rejects_null(lib):
    bits = ctypes.c_uint32(0)
    assert lib.nvfp4_workspace_error(None, None, ctypes.byref(bits)) == NULL


def test_binding_does_not_import_oracle():
    # the product package must not reach the test oracle
    src_dir = os.path.join(ROOT, "nvfp4_weight_quantized_quantize_gb300")
    for dirpath, _, files in os.walk(src_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f
