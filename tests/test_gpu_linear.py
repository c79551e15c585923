"""GPU parity of nvfp4_linear against the oracle (through the C ABI).

Weights are quantized by the oracle on the CPU and uploaded; the oracle computes the
reference from the same bytes in fp64.  Each output must satisfy
|y - y_ref| <= 1e-3 * sum_k |x_k w_k| + 2^-8 |y_ref|.
"""
import numpy as np
import pytest
import torch

import nvfp4_weight_quantized_quantize_gb300 as nv
import oracle
from helpers import check_tolerance, to_dev, upload_weights, y_to_f64
from synth import WORKLOADS, make_inputs, random_nvfp4_weights, random_x, workload_inputs

pytestmark = pytest.mark.gpu


def run_linear(x, wq, ws, gw, K, y_dtype, mode="w4a16", gx=None, static_weights=False):
    M = x.shape[0]
    N = wq.shape[0]
    d_wq, d_swz, d_g = upload_weights(wq, ws, gw, K)
    d_x = x.cuda()
    y = torch.empty(M, N, dtype=y_dtype, device="cuda")
    wsb = nv.nvfp4_workspace_bytes(1, M, K, N, nv.NVFP4_W4A4 if mode == "w4a4" else nv.NVFP4_W4A16)
    ws_t = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda") if wsb else None
    d_gx = None if gx is None else torch.tensor([gx], dtype=torch.float32, device="cuda")
    nv.nvfp4_linear(d_x, d_wq, d_swz, d_g, y, mode=mode, x_global_scale=d_gx, workspace=ws_t,
                    static_weights=static_weights)
    torch.cuda.synchronize()
    assert nv.nvfp4_workspace_error(ws_t) == 0
    return y, ws_t


@pytest.mark.parametrize("M,K,N,ydt", [
    (1, 32, 1, torch.float32), (1, 64, 3, torch.bfloat16), (1, 96, 257, torch.float32),
    (2, 160, 100, torch.bfloat16), (3, 512, 1000, torch.float32), (7, 1056, 333, torch.bfloat16),
    (8, 4096, 130, torch.float32), (11, 640, 77, torch.bfloat16), (16, 2048, 64, torch.float32),
    (5, 32, 9, torch.bfloat16), (13, 96, 200, torch.float32),
])
def test_ragged_w4a16(M, K, N, ydt):
    x, w = make_inputs(M, K, N, seed=100 + M + K + N, outliers=True)
    wq, ws, gw = oracle.quantize(w.numpy())
    y, _ = run_linear(x, wq, ws, gw, K, ydt)
    y_ref, ab = oracle.linear_w4a16(x, wq, ws, gw)
    check_tolerance(y_to_f64(y), y_ref, ab, "M%d K%d N%d" % (M, K, N))


@pytest.mark.parametrize("name", ["tiny", "decode_a", "decode_b"])
def test_workload_full(name):
    wl = WORKLOADS[name]
    x, w = workload_inputs(name)
    wq, ws, gw = oracle.quantize(w.numpy())
    ydt = torch.float32 if wl.y_dtype == "f32" else torch.bfloat16
    y, _ = run_linear(x, wq, ws, gw, wl.K, ydt)
    y_ref, ab = oracle.linear_w4a16(x, wq, ws, gw)
    check_tolerance(y_to_f64(y), y_ref, ab, name)


@pytest.mark.parametrize("name", ["verify_a", "verify_b"])
def test_verify_sampled(name):
    wl = WORKLOADS[name]
    x, w = workload_inputs(name)
    wq, ws, gw = oracle.quantize(w.numpy())
    y, _ = run_linear(x, wq, ws, gw, wl.K, torch.bfloat16)
    rng = np.random.default_rng(0)
    pm = rng.integers(0, wl.M, 4096)
    pn = rng.integers(0, wl.N, 4096)
    # plus two full output rows
    pm = np.concatenate([pm, np.zeros(wl.N, np.int64), np.full(wl.N, wl.M - 1)])
    pn = np.concatenate([pn, np.arange(wl.N), np.arange(wl.N)])
    y_ref, ab = oracle.linear_w4a16_pairs(x, wq, ws, gw, pm, pn)
    check_tolerance(y_to_f64(y)[pm, pn], y_ref, ab, name)


def test_zero_weights_and_zero_x():
    M, K, N = 3, 64, 40
    x, _ = make_inputs(M, K, N, 7)
    w = torch.zeros(N, K)
    wq, ws, gw = oracle.quantize(w.numpy())
    y, _ = run_linear(x, wq, ws, gw, K, torch.float32)
    assert not y.any()
    x0 = torch.zeros(M, K, dtype=torch.bfloat16)
    _, w = make_inputs(M, K, N, 8)
    wq, ws, gw = oracle.quantize(w.numpy())
    y, _ = run_linear(x0, wq, ws, gw, K, torch.float32)
    assert not y.any()


@pytest.mark.parametrize("M,K,N,gx", [(1, 512, 256, None), (7, 1024, 300, None),
                                      (4, 96, 50, 0.003), (16, 5120, 128, None),
                                      (1, 5120, 1000, None), (1, 17408, 300, None),
                                      (1, 2080, 77, None), (4, 5120, 1000, None),
                                      (8, 2080, 129, None), (2, 96, 50, None)])
def test_w4a4_small_m(M, K, N, gx):
    # M = 1 with a dynamic scale and K / 32 >= 64: the GEMV reduces x's amax itself and
    # leaves x's encoding in the workspace (checked below like the quantizer's); the
    # others quantize x ahead of the kernel
    x, w = make_inputs(M, K, N, seed=200 + M)
    wq, ws, gw = oracle.quantize(w.numpy())
    y, ws_t = run_linear(x, wq, ws, gw, K, torch.bfloat16, mode="w4a4", gx=gx)
    y_ref, ab, xq, xs, gxo = oracle.linear_w4a4(x, wq, ws, gw, gx)
    check_tolerance(y_to_f64(y), y_ref, ab, "w4a4 M%d" % M)
    if gx is not None and M <= 8:
        return  # quantized inside the small-M kernel: nothing lands in the workspace
    # the in-call activation quantization is bit-exact: codes, swizzled scales, g_x
    o_xq, o_xs, o_gx = nv.nvfp4_w4a4_workspace_layout(M, K)
    wsh = ws_t.cpu().numpy()
    np.testing.assert_array_equal(wsh[o_xq:o_xq + M * K // 2].reshape(M, K // 2), xq)
    nb = oracle.repack_atom_bytes(M, K)
    np.testing.assert_array_equal(wsh[o_xs:o_xs + nb], oracle.repack(xs, K)[:nb])
    assert wsh[o_gx:o_gx + 4].view(np.float32)[0] == np.float32(gxo)


@pytest.mark.parametrize("M,K,N", [(1, 96, 70), (1, 2080, 333), (1, 5120, 1000),
                                   (1, 17408, 300), (3, 96, 70), (3, 5120, 600), (8, 2080, 129),
                                   (8, 17408, 40)])
def test_w4a4_static_scale_fused(M, K, N):
    # W4A4 with a static activation scale at M <= 8 quantizes x inside the GEMV / skinny
    # kernel.  Its output must equal, bit for bit, the linear on the same activations
    # quantized by the oracle (the products are the same exact values), and the oracle
    # within the tolerance.
    gx = 0.004
    x, w = make_inputs(M, K, N, seed=500 + M + K)
    wq, ws, gw = oracle.quantize(w.numpy())
    y, _ = run_linear(x, wq, ws, gw, K, torch.bfloat16, mode="w4a4", gx=gx, static_weights=True)
    y_ref, ab, xq, xs, gxo = oracle.linear_w4a4(x, wq, ws, gw, gx)
    check_tolerance(y_to_f64(y), y_ref, ab, "fused w4a4 M%d K%d" % (M, K))
    d_wq, d_swz, d_g = upload_weights(wq, ws, gw, K)
    d_xs = to_dev(oracle.repack(xs, K)[:oracle.repack_atom_bytes(M, K)].copy())
    y2 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    work = torch.zeros(nv.nvfp4_workspace_bytes(1, M, K, N, nv.NVFP4_W4A4), dtype=torch.uint8,
                       device="cuda")
    nv.nvfp4_linear_nvfp4_x(to_dev(xq), d_xs, torch.tensor([gxo], device="cuda"), d_wq, d_swz,
                            d_g, y2, work)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)


def test_repeated_calls_are_deterministic():
    M, K, N = 7, 5120, 6144
    x, w = make_inputs(M, K, N, 3)
    wq, ws, gw = oracle.quantize(w.numpy())
    y1, _ = run_linear(x, wq, ws, gw, K, torch.bfloat16)
    y2, _ = run_linear(x, wq, ws, gw, K, torch.bfloat16)
    assert torch.equal(y1, y2)


def test_tiny_config_on_a_side_stream():
    x, w = workload_inputs("tiny")
    wq, ws, gw = oracle.quantize(w.numpy())
    d_wq, d_swz, d_g = upload_weights(wq, ws, gw, 512)
    s = torch.cuda.Stream()
    y = torch.empty(1, 256, dtype=torch.float32, device="cuda")
    d_x = x.cuda()
    work = torch.zeros(nv.nvfp4_workspace_bytes(1, 1, 512, 256), dtype=torch.uint8,
                       device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        nv.nvfp4_linear(d_x, d_wq, d_swz, d_g, y, workspace=work)
    s.synchronize()
    y_ref, ab = oracle.linear_w4a16(x, wq, ws, gw)
    check_tolerance(y_to_f64(y), y_ref, ab, "side stream")


@pytest.mark.parametrize("M,K", [(1, 320), (1, 4096), (3, 320), (9, 320), (16, 320),
                                 (7, 2048)])
def test_x_with_wide_dynamic_range(M, K):
    # a few elements far below their row's largest magnitude are not exact in fp16 after
    # the kernels' power-of-two rescale; the exact residual path must keep the result
    N = 70
    x, w = make_inputs(M, K, N, seed=300 + M)
    xf = x.float()
    xf[:, ::7] *= 1e-12
    xf[:, 5] = 3.0e4
    xf[0, 9] = -2.0e-30
    x = xf.to(torch.bfloat16)
    wq, ws, gw = oracle.quantize(w.numpy())
    for ydt in (torch.float32, torch.bfloat16):
        y, _ = run_linear(x, wq, ws, gw, K, ydt)
        y_ref, ab = oracle.linear_w4a16(x, wq, ws, gw)
        check_tolerance(y_to_f64(y), y_ref, ab, "wide range M%d" % M)


@pytest.mark.parametrize("M,K,N", [(1, 20480, 300), (8, 12288, 200), (16, 6144, 100),
                                   (1, 2048, 1000), (1, 65536, 40), (1, 98304, 20)])
def test_multiple_k_chunks(M, K, N):
    # K larger than one shared-memory chunk of x
    x, w = make_inputs(M, K, N, seed=400 + M)
    wq, ws, gw = oracle.quantize(w.numpy())
    y, _ = run_linear(x, wq, ws, gw, K, torch.float32)
    y_ref, ab = oracle.linear_w4a16(x, wq, ws, gw)
    check_tolerance(y_to_f64(y), y_ref, ab, "chunks M%d K%d" % (M, K))


@pytest.mark.parametrize("M,K,N,wide", [(5, 256, 39001, False), (7, 512, 31623, False),
                                        (2, 1024, 24000, False), (7, 256, 39001, True),
                                        (12, 512, 31623, False), (16, 256, 39001, True)])
def test_skinny_stages_of_several_row_groups(M, K, N, wide):
    # enough rows per CTA that a pipeline stage of the skinny kernel holds two to four 16-row
    # groups, the last one ragged (with one and with two token tiles); the wide-range case
    # takes the exact residual path
    x, w = make_inputs(M, K, N, seed=500 + M + K)
    if wide:
        xf = x.float()
        xf[:, ::5] *= 1e-12
        xf[:, 3] = 2.0e4
        x = xf.to(torch.bfloat16)
    wq, ws, gw = oracle.quantize(w.numpy())
    y, _ = run_linear(x, wq, ws, gw, K, torch.bfloat16)
    y_ref, ab = oracle.linear_w4a16(x, wq, ws, gw)
    check_tolerance(y_to_f64(y), y_ref, ab, "row groups M%d K%d N%d" % (M, K, N))


@pytest.mark.parametrize("M,K,N", [(1, 5120, 1000), (1, 1024, 77), (7, 5120, 600), (3, 2048, 130)])
def test_static_weights_flag(M, K, N):
    # NVFP4_STATIC_WEIGHTS only moves the weight stream ahead of the wait for the previous
    # kernel: the result is the same, here right after a kernel that wrote the weights'
    # neighbour buffers and a quantization on the same stream
    x, w = make_inputs(M, K, N, seed=700 + M + K)
    wq, ws, gw = oracle.quantize(w.numpy())
    d_wq, d_swz, d_g = upload_weights(wq, ws, gw, K)
    y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    wsb = nv.nvfp4_workspace_bytes(1, M, K, N)
    work = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
    d_x = x.cuda()
    for _ in range(3):
        nv.nvfp4_linear(d_x, d_wq, d_swz, d_g, y, workspace=work, static_weights=True)
    torch.cuda.synchronize()
    assert nv.nvfp4_workspace_error(work) == 0
    y_ref, ab = oracle.linear_w4a16(x, wq, ws, gw)
    check_tolerance(y_to_f64(y), y_ref, ab, "static M%d K%d N%d" % (M, K, N))


@pytest.mark.parametrize("K,N", [(5120, 700), (17408, 300)])
def test_m1_chunks_of_very_different_magnitude(K, N):
    # every 32-element chunk of x at its own scale (2^-60 .. 2^60): the M=1 kernel rescales
    # each lane's chunk by its own power of two and must still match the oracle
    x, w = make_inputs(1, K, N, seed=800 + K)
    xf = x.float()
    scales = 2.0 ** torch.arange(-60, 61, 7, dtype=torch.float64).float()
    for c in range(K // 32):
        xf[:, 32 * c:32 * c + 32] *= scales[c % len(scales)]
    x = xf.to(torch.bfloat16)
    wq, ws, gw = oracle.quantize(w.numpy())
    for ydt in (torch.float32, torch.bfloat16):
        y, _ = run_linear(x, wq, ws, gw, K, ydt)
        y_ref, ab = oracle.linear_w4a16(x, wq, ws, gw)
        check_tolerance(y_to_f64(y), y_ref, ab, "chunk scales K%d" % K)


def test_static_weights_flag_w4a4_small_m():
    # the flag passes through the W4A4 path for M <= 16 (in-call x quantization, then the
    # GEMV on the dequantized x): same result as without it
    M, K, N = 1, 2048, 300
    x, w = make_inputs(M, K, N, seed=901)
    wq, ws, gw = oracle.quantize(w.numpy())
    d_wq, d_swz, d_g = upload_weights(wq, ws, gw, K)
    outs = []
    for flag in (False, True):
        y = torch.empty(M, N, dtype=torch.float32, device="cuda")
        wsb = nv.nvfp4_workspace_bytes(1, M, K, N, nv.NVFP4_W4A4)
        work = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
        nv.nvfp4_linear(x.cuda(), d_wq, d_swz, d_g, y, mode="w4a4", workspace=work,
                        static_weights=flag)
        torch.cuda.synchronize()
        assert nv.nvfp4_workspace_error(work) == 0
        outs.append(y.cpu())
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("M", list(range(1, 17)))
def test_every_small_m(M):
    # the small-M curve: every M the GEMV / skinny / mma.sync kernels take, on a shape
    # with a ragged row count and several K chunks per warp
    x, w = make_inputs(M, 2080, 1203, seed=300 + M, outliers=True)
    wq, ws, gw = oracle.quantize(w.numpy())
    y, _ = run_linear(x, wq, ws, gw, 2080, torch.bfloat16, static_weights=(M % 2 == 0))
    y_ref, ab = oracle.linear_w4a16(x, wq, ws, gw)
    check_tolerance(y_to_f64(y), y_ref, ab, "M%d" % M)


@pytest.mark.parametrize("M,K,N", [(1, 4096, 120001), (1, 1024, 131075), (4, 1024, 131075)])
def test_wide_n(M, K, N):
    # lm-head-like outputs (ragged N): at K = 4096 each CTA of the M = 1 kernel keeps
    # partial sums for 790 rows, which leaves room for two shorter stages only; sampled
    # outputs plus the first and last 4096 of every row of y.  The weights are drawn as
    # NVFP4 bytes directly (quantizing 491 M floats on the CPU would dominate the test).
    x = random_x(M, K, seed=400 + M)
    wq, ws, gw = random_nvfp4_weights(N, K, seed=410 + M)
    y, _ = run_linear(x, wq, ws, gw, K, torch.bfloat16, static_weights=True)
    rng = np.random.default_rng(M)
    edge = np.concatenate([np.arange(4096), np.arange(N - 4096, N)])
    pm = np.concatenate([rng.integers(0, M, 8192), np.repeat(np.arange(M), edge.size)])
    pn = np.concatenate([rng.integers(0, N, 8192), np.tile(edge, M)])
    y_ref, ab = oracle.linear_w4a16_pairs(x, wq, ws, gw, pm, pn)
    check_tolerance(y_to_f64(y)[pm, pn], y_ref, ab, "wide N M%d" % M)


@pytest.mark.parametrize("M,K,N", [(1, 5120, 1000), (1, 17408, 300), (1, 2080, 129)])
def test_w4a4_dynamic_small_m_matches_prepass(M, K, N):
    # x quantized inside the M = 1 GEMV (dynamic scale) and by the quantizer kernels ahead
    # of it: the same encoding in the workspace and the same y, to the bit
    from helpers import w4a4_kernel
    x, w = make_inputs(M, K, N, seed=600 + M)
    wq, ws, gw = oracle.quantize(w.numpy())
    y1, ws1 = run_linear(x, wq, ws, gw, K, torch.float32, mode="w4a4")
    with w4a4_kernel("prepass"):
        y2, ws2 = run_linear(x, wq, ws, gw, K, torch.float32, mode="w4a4")
    assert torch.equal(y1, y2)
    o_xq, o_xs, o_gx = nv.nvfp4_w4a4_workspace_layout(M, K)
    a, b = ws1.cpu().numpy(), ws2.cpu().numpy()
    nb = oracle.repack_atom_bytes(M, K)
    np.testing.assert_array_equal(a[o_xq:o_xq + M * K // 2], b[o_xq:o_xq + M * K // 2])
    np.testing.assert_array_equal(a[o_xs:o_xs + nb], b[o_xs:o_xs + nb])
    assert a[o_gx:o_gx + 4].tobytes() == b[o_gx:o_gx + 4].tobytes()
