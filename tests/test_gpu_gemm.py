"""GPU parity of the tensor-core W4A16 GEMM (nvfp4_linear with M > 16) against the oracle.

Weights are quantized by the oracle on the CPU and uploaded; the oracle computes the
reference from the same bytes in fp64.  Each output must satisfy
|y - y_ref| <= 1e-3 * sum_k |x_k w_k| + 2^-8 |y_ref|.  Shapes cover one tile, ragged
M / N / K (K = 32 mod 64), several tiles in both directions, and the two prefill
workloads (sampled outputs plus full rows).
"""
import numpy as np
import pytest
import torch

import nvfp4_weight_quantized_quantize_gb300 as nv
import oracle
from helpers import check_tolerance, upload_weights, y_to_f64
from synth import WORKLOADS, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu


def run_gemm(x, wq, ws, gw, K, y_dtype):
    M, N = x.shape[0], wq.shape[0]
    d_wq, d_swz, d_g = upload_weights(wq, ws, gw, K)
    y = torch.full((M, N), float("nan"), dtype=y_dtype, device="cuda")
    work = torch.zeros(nv.nvfp4_workspace_bytes(1, M, K, N, nv.NVFP4_W4A16), dtype=torch.uint8,
                       device="cuda")
    nv.nvfp4_linear(x.cuda(), d_wq, d_swz, d_g, y, workspace=work)
    torch.cuda.synchronize()
    assert nv.nvfp4_workspace_error(work) == 0
    return y


@pytest.mark.parametrize("M,K,N,ydt", [
    (17, 64, 1, torch.float32), (17, 32, 130, torch.bfloat16), (32, 128, 128, torch.float32),
    (33, 96, 129, torch.bfloat16), (100, 160, 200, torch.float32),
    (256, 128, 128, torch.bfloat16), (257, 512, 300, torch.float32),
    (300, 1056, 257, torch.bfloat16), (512, 1024, 640, torch.bfloat16),
])
def test_gemm_ragged(M, K, N, ydt):
    x, w = make_inputs(M, K, N, seed=200 + M + K + N, outliers=True)
    wq, ws, gw = oracle.quantize(w.numpy())
    y = run_gemm(x, wq, ws, gw, K, ydt)
    y_ref, ab = oracle.linear_w4a16(x, wq, ws, gw)
    check_tolerance(y_to_f64(y), y_ref, ab, "M%d K%d N%d" % (M, K, N))


def test_gemm_wide_dynamic_range_rows():
    # rows of x scaled by powers of two from 2^-20 to 2^20 (bf16 products stay exact)
    M, K, N = 64, 320, 192
    x, w = make_inputs(M, K, N, seed=11)
    x = (x.float() * torch.pow(2.0, torch.arange(-20, 44, dtype=torch.float32)[:M, None])
         ).to(torch.bfloat16)
    wq, ws, gw = oracle.quantize(w.numpy())
    y = run_gemm(x, wq, ws, gw, K, torch.float32)
    y_ref, ab = oracle.linear_w4a16(x, wq, ws, gw)
    check_tolerance(y_to_f64(y), y_ref, ab, "wide rows")


@pytest.mark.parametrize("name", ["prefill_a", "prefill_b"])
def test_prefill_sampled(name):
    wl = WORKLOADS[name]
    x, w = workload_inputs(name)
    wq, ws, gw = oracle.quantize(w.numpy())
    y = run_gemm(x, wq, ws, gw, wl.K, torch.bfloat16)
    rng = np.random.default_rng(1)
    pm = rng.integers(0, wl.M, 4096)
    pn = rng.integers(0, wl.N, 4096)
    # plus the first and last output rows in full
    pm = np.concatenate([pm, np.zeros(wl.N, np.int64), np.full(wl.N, wl.M - 1)])
    pn = np.concatenate([pn, np.arange(wl.N), np.arange(wl.N)])
    y_ref, ab = oracle.linear_w4a16_pairs(x, wq, ws, gw, pm, pn)
    check_tolerance(y_to_f64(y)[pm, pn], y_ref, ab, name)


def test_gemm_repeated_calls_are_deterministic():
    M, K, N = 300, 640, 384
    x, w = make_inputs(M, K, N, seed=5)
    wq, ws, gw = oracle.quantize(w.numpy())
    y1 = run_gemm(x, wq, ws, gw, K, torch.float32)
    y2 = run_gemm(x, wq, ws, gw, K, torch.float32)
    assert torch.equal(y1, y2)


def test_stream_k_reuses_its_workspace():
    # 10 tiles on a 152-SM part: every tile is split over several CTAs (stream-K); the
    # per-quarter counters must come back to zero so the same workspace serves again
    M, K, N = 512, 1024, 640
    x, w = make_inputs(M, K, N, seed=9)
    wq, ws, gw = oracle.quantize(w.numpy())
    d_wq, d_swz, d_g = upload_weights(wq, ws, gw, K)
    xd = x.cuda()
    work = torch.zeros(nv.nvfp4_workspace_bytes(1, M, K, N, nv.NVFP4_W4A16), dtype=torch.uint8,
                       device="cuda")
    ys = []
    for _ in range(3):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        nv.nvfp4_linear(xd, d_wq, d_swz, d_g, y, workspace=work)
        torch.cuda.synchronize()
        assert nv.nvfp4_workspace_error(work) == 0
        ntiles = ((N + 127) // 128) * ((M + 255) // 256)
        assert not work[256:256 + 16 * ntiles].any()
        ys.append(y)
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[1], ys[2])
    y_ref, ab = oracle.linear_w4a16(x, wq, ws, gw)
    check_tolerance(y_to_f64(ys[0]), y_ref, ab, "stream-K reuse")
