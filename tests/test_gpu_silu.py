"""silu on the device against the oracle over its whole input domain.

Every caller hands silu a bf16 value (the gate half of a bf16 gate_up tensor, or the
fused gate/up epilogue's bf16-rounded gate), so the 65,536 bf16 bit patterns are all
the inputs it can see.  Both device forms -- silu_f32 (the Cody-Waite exp, then CUDA's
correctly rounded division) and silu_f32_nobranch (the exp's ends selected rather than
branched to, then a branch-free division by P. Markstein's reciprocal-and-remainder
method) -- must give the oracle's orc_silu_mul_f32(g, 1) bit for bit on every one of
them, infinities and NaN included.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
from conftest import ROOT

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def silu_lib():
    src = os.path.join(ROOT, "tests", "pins", "device_silu.cu")
    out_dir = os.path.join(ROOT, "tests", "pins", "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "device_silu.so")
    tmp = so + ".tmp%d" % os.getpid()
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "nvfp4_weight_quantized_quantize_gb300", "csrc"),
                    "-Xcompiler", "-fPIC", "-shared", src, "-o", tmp], check=True)
    os.replace(tmp, so)
    lib = ctypes.CDLL(so)
    lib.device_silu.restype = ctypes.c_int
    lib.device_silu.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    return lib


def _check(out, want, gf, what):
    nan_w, nan_o = np.isnan(want), np.isnan(out)
    assert np.array_equal(nan_w, nan_o), "%s: NaN pattern differs" % what
    ok = ~nan_w
    bad = np.nonzero(out[ok].view(np.uint32) != want[ok].view(np.uint32))[0]
    assert bad.size == 0, "%s: %d inputs differ; first g = %r: device %r oracle %r" % (
        what, bad.size, float(gf[ok][bad[0]]), float(out[ok][bad[0]]), float(want[ok][bad[0]]))


def test_silu_every_bf16_input(silu_lib):
    g = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    n = g.size
    out = np.empty(n, np.float32)
    out_nb = np.empty(n, np.float32)
    rc = silu_lib.device_silu(g.ctypes.data, out.ctypes.data, out_nb.ctypes.data, n)
    assert rc == 0
    gf = (g.astype(np.uint32) << 16).view(np.float32)
    want = np.array([oracle.silu_mul_f32(float(v), 1.0) for v in gf], dtype=np.float32)
    _check(out, want, gf, "silu_f32")
    _check(out_nb, want, gf, "silu_f32_nobranch")
