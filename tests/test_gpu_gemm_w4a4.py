"""GPU parity of the block-scaled W4A4 GEMM (nvfp4_linear, mode w4a4, M > 16).

The in-call activation quantization must be bit-exact with the oracle (codes, swizzled
scale atoms, g_x); y must satisfy |y - y_ref| <= 1e-3 * sum_k |x_k w_k| + 2^-8 |y_ref|,
x_k, w_k the dequantized operands, y_ref the oracle's fp64 dot of them.  Shapes cover one
tile, ragged M / N / K (K = 32 and 64 mod 256: partial scale atoms and partial K steps),
several tiles, stream-K splits, a static g_x and the 2048-row workload (sampled).  The
GEMM runs on the one-CTA tensor-core kernel; the CTA-pair kernel (256 x 256 tiles over
two SMs) runs the same ragged shapes.
"""
import numpy as np
import pytest
import torch

import nvfp4_weight_quantized_quantize_gb300 as nv
import oracle
from helpers import check_tolerance, upload_weights, w4a4_kernel, y_to_f64
from synth import WORKLOADS, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu


def run_w4a4(x, wq, ws, gw, K, y_dtype, gx=None, work=None):
    M, N = x.shape[0], wq.shape[0]
    d_wq, d_swz, d_g = upload_weights(wq, ws, gw, K)
    y = torch.full((M, N), float("nan"), dtype=y_dtype, device="cuda")
    if work is None:
        work = torch.zeros(nv.nvfp4_workspace_bytes(1, M, K, N, nv.NVFP4_W4A4),
                           dtype=torch.uint8, device="cuda")
    d_gx = None if gx is None else torch.tensor([gx], dtype=torch.float32, device="cuda")
    nv.nvfp4_linear(x.cuda(), d_wq, d_swz, d_g, y, mode="w4a4", x_global_scale=d_gx,
                    workspace=work)
    torch.cuda.synchronize()
    assert nv.nvfp4_workspace_error(work) == 0
    return y, work


def check_x_quant(work, M, K, xq, xs, gxo):
    o_xq, o_xs, o_gx = nv.nvfp4_w4a4_workspace_layout(M, K)
    wsh = work.cpu().numpy()
    np.testing.assert_array_equal(wsh[o_xq:o_xq + M * K // 2].reshape(M, K // 2), xq)
    nb = oracle.repack_atom_bytes(M, K)
    np.testing.assert_array_equal(wsh[o_xs:o_xs + nb], oracle.repack(xs, K)[:nb])
    assert wsh[o_gx:o_gx + 4].view(np.float32)[0] == np.float32(gxo)


@pytest.mark.parametrize("M,K,N,ydt", [
    (17, 64, 1, torch.float32), (17, 32, 130, torch.bfloat16), (32, 256, 128, torch.float32),
    (100, 320, 200, torch.bfloat16), (129, 96, 130, torch.float32),
    (256, 1024, 384, torch.bfloat16), (300, 1056, 257, torch.float32),
    (512, 2048, 640, torch.bfloat16),
])
@pytest.mark.parametrize("kernel", ["auto", "pair"])
def test_w4a4_gemm_ragged(M, K, N, ydt, kernel):
    x, w = make_inputs(M, K, N, seed=300 + M + K + N, outliers=True)
    wq, ws, gw = oracle.quantize(w.numpy())
    with w4a4_kernel(kernel):
        y, work = run_w4a4(x, wq, ws, gw, K, ydt)
    y_ref, ab, xq, xs, gxo = oracle.linear_w4a4(x, wq, ws, gw)
    check_x_quant(work, M, K, xq, xs, gxo)
    check_tolerance(y_to_f64(y), y_ref, ab, "w4a4 M%d K%d N%d" % (M, K, N))


def test_w4a4_gemm_static_global_scale():
    M, K, N = 200, 512, 300
    x, w = make_inputs(M, K, N, seed=17)
    wq, ws, gw = oracle.quantize(w.numpy())
    gx = 0.0021
    y, work = run_w4a4(x, wq, ws, gw, K, torch.float32, gx=gx)
    y_ref, ab, xq, xs, gxo = oracle.linear_w4a4(x, wq, ws, gw, gx)
    check_x_quant(work, M, K, xq, xs, gxo)
    check_tolerance(y_to_f64(y), y_ref, ab, "w4a4 static gx")


@pytest.mark.parametrize("M,K,N", [(512, 1024, 640), (2048, 5120, 2304), (40, 5120, 3000)])
def test_w4a4_gemm_reuses_its_workspace(M, K, N):
    # repeated calls on one workspace (stream-K counters back at zero after each call,
    # the partial-tile sums in a fixed order) give the same bits, on either kernel, and a
    # workspace used by one kernel serves the other
    x, w = make_inputs(M, K, N, seed=19)
    wq, ws, gw = oracle.quantize(w.numpy())
    y1, work = run_w4a4(x, wq, ws, gw, K, torch.float32)
    y2, _ = run_w4a4(x, wq, ws, gw, K, torch.float32, work=work)
    with w4a4_kernel("pair"):
        v1, _ = run_w4a4(x, wq, ws, gw, K, torch.float32, work=work)
        v2, _ = run_w4a4(x, wq, ws, gw, K, torch.float32, work=work)
    y3, _ = run_w4a4(x, wq, ws, gw, K, torch.float32, work=work)
    assert torch.equal(y1, y2) and torch.equal(y2, y3) and torch.equal(v1, v2)
    xq, xs, gxo = oracle.quantize(x.float().numpy())
    rng = np.random.default_rng(M + N)
    pm = np.concatenate([rng.integers(0, M, 2048), np.full(N, M - 1)])
    pn = np.concatenate([rng.integers(0, N, 2048), np.arange(N)])
    y_ref, ab = oracle.linear_w4a4_pairs(xq, xs, gxo, wq, ws, gw, pm, pn)
    check_tolerance(y_to_f64(y1)[pm, pn], y_ref, ab, "w4a4 reuse")
    check_tolerance(y_to_f64(v1)[pm, pn], y_ref, ab, "w4a4 reuse, single-pair kernel")


def test_w4a4_workload_sampled():
    wl = WORKLOADS["w4a4"]
    x, w = workload_inputs("w4a4")
    wq, ws, gw = oracle.quantize(w.numpy())
    y, work = run_w4a4(x, wq, ws, gw, wl.K, torch.bfloat16)
    # the oracle quantizes x in full (bit-exact check), then evaluates sampled outputs
    o_xq, o_xs, o_gx = nv.nvfp4_w4a4_workspace_layout(wl.M, wl.K)
    xq, xs, gxo = oracle.quantize(x.float().numpy())
    check_x_quant(work, wl.M, wl.K, xq, xs, gxo)
    rng = np.random.default_rng(2)
    pm = rng.integers(0, wl.M, 4096)
    pn = rng.integers(0, wl.N, 4096)
    pm = np.concatenate([pm, np.zeros(wl.N, np.int64), np.full(wl.N, wl.M - 1)])
    pn = np.concatenate([pn, np.arange(wl.N), np.arange(wl.N)])
    y_ref, ab = oracle.linear_w4a4_pairs(xq, xs, gxo, wq, ws, gw, pm, pn)
    check_tolerance(y_to_f64(y)[pm, pn], y_ref, ab, "w4a4 workload")


@pytest.mark.parametrize("M,K,N,gx", [(300, 2080, 777, None), (300, 2080, 777, 0.003),
                                      (2048, 5120, 1000, None)])
def test_in_kernel_quantization_matches_prepass(M, K, N, gx):
    # x quantized inside the GEMM's grid and by the quantizer kernels ahead of it (the path
    # of a device that refuses the cooperative launch): the same codes, scales and g_x,
    # then the same GEMM, so y is the same to the bit
    x, w = make_inputs(M, K, N, seed=900 + M, outliers=True)
    wq, ws, gw = oracle.quantize(w.numpy())
    y1, work1 = run_w4a4(x, wq, ws, gw, K, torch.float32, gx=gx)
    with w4a4_kernel("prepass"):
        y2, work2 = run_w4a4(x, wq, ws, gw, K, torch.float32, gx=gx)
    assert torch.equal(y1, y2)
    o_xq, o_xs, o_gx = nv.nvfp4_w4a4_workspace_layout(M, K)
    a, b = work1.cpu().numpy(), work2.cpu().numpy()
    np.testing.assert_array_equal(a[o_xq:o_xs], b[o_xq:o_xs])
    assert a[o_gx:o_gx + 4].tobytes() == b[o_gx:o_gx + 4].tobytes()
