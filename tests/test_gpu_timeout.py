"""The failure path of the bounded device waits, exercised without a GPU fault.

Every wait in which one role of a kernel (or one CTA) waits for another is bounded in
wall time; when it runs out the kernel ORs NVFP4_DEVERR_TIMEOUT into the workspace's
error word, every role stops, the copies and MMAs already issued are waited for, TMEM is
freed, and the kernel returns.  nvfp4_debug_expire_waits makes that happen on purpose:
the kernels launch with a 200 us limit and one role withholds its arrival (a flag that
nothing sets).  For each kernel with such waits the test checks that

- the call returns and the stream drains (bounded time, no hang),
- nvfp4_workspace_error reports the time-out (and clears the word),
- the CUDA context is still usable: the next call, on the zero-filled workspace, is
  correct against the oracle and reports no error.
"""
import time

import numpy as np
import pytest
import torch

import nvfp4_weight_quantized_quantize_gb300 as nv
import oracle
from helpers import check_tolerance, to_dev, upload_weights, w4a4_kernel, y_to_f64
from synth import random_nvfp4_weights, random_x

pytestmark = pytest.mark.gpu

NVFP4_DEVERR_TIMEOUT = 0x1


@pytest.mark.parametrize("M,K,N,mode,what", [
    (1, 5120, 17408, "w4a16", "pipelined GEMV: the consumers never release a stage"),
    (64, 1024, 512, "w4a16", "tcgen05 W4A16 GEMM: no stage is marked dequantized"),
    (64, 1024, 512, "w4a4", "block-scaled GEMM: one CTA never counts its share of x"),
    (64, 1024, 512, "w4a4-pair", "block-scaled CTA-pair GEMM: one CTA never counts"),
    (300, 2048, 1000, "w4a4-pair", "CTA pairs over several tiles: one CTA never counts"),
])
def test_expired_wait_reports_and_recovers(M, K, N, mode, what):
    kernel = mode.split("-")[1] if "-" in mode else "auto"
    mode = mode.split("-")[0]
    x = random_x(M, K, seed=M + K)
    wq, ws, gw = random_nvfp4_weights(N, K, seed=N)
    d_wq, d_swz, d_g = upload_weights(wq, ws, gw, K)
    d_x = x.cuda()
    y = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    m = nv.NVFP4_W4A4 if mode == "w4a4" else nv.NVFP4_W4A16
    work = torch.zeros(nv.nvfp4_workspace_bytes(1, M, K, N, m), dtype=torch.uint8,
                       device="cuda")
    torch.cuda.synchronize()

    t0 = time.perf_counter()
    nv.nvfp4_debug_expire_waits(True)
    try:
        with w4a4_kernel(kernel):
            nv.nvfp4_linear(d_x, d_wq, d_swz, d_g, y, mode=mode, workspace=work)
    finally:
        nv.nvfp4_debug_expire_waits(False)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 10.0, what
    bits = nv.nvfp4_workspace_error(work)
    assert bits & NVFP4_DEVERR_TIMEOUT, what
    assert nv.nvfp4_workspace_error(work) == 0  # read once, then cleared

    # the context is usable: a normal call on the zero-filled workspace is correct
    work.zero_()
    with w4a4_kernel(kernel):
        nv.nvfp4_linear(d_x, d_wq, d_swz, d_g, y, mode=mode, workspace=work)
    torch.cuda.synchronize()
    assert nv.nvfp4_workspace_error(work) == 0
    rng = np.random.default_rng(1)
    pm = np.concatenate([rng.integers(0, M, 2048), np.full(N, M - 1)])
    pn = np.concatenate([rng.integers(0, N, 2048), np.arange(N)])
    if mode == "w4a4":
        xq, xs, gx = oracle.quantize(x)  # x as the call quantizes it (dynamic scale)
        y_ref, ab = oracle.linear_w4a4_pairs(xq, xs, gx, wq, ws, gw, pm, pn)
    else:
        y_ref, ab = oracle.linear_w4a16_pairs(x, wq, ws, gw, pm, pn)
    check_tolerance(y_to_f64(y)[pm, pn], y_ref, ab, what)


@pytest.mark.parametrize("M,K,N,kernel", [(64, 1024, 512, "auto"), (300, 2048, 1000, "pair"),
                                          (64, 1024, 512, "pair")])
def test_expired_wait_nvfp4_x(M, K, N, kernel):
    # the GEMM on NVFP4 activations (no in-kernel quantization): the one-CTA kernel's scale
    # writers never mark a stage's scales written (the CTA-pair kernel's MMA issuer never
    # marks an accumulator full), so a wait runs out
    x = random_x(M, K, seed=M + 3)
    xq, xs, gx = oracle.quantize(x)
    wq, ws, gw = random_nvfp4_weights(N, K, seed=N + 3)
    d_wq, d_swz, d_g = upload_weights(wq, ws, gw, K)
    d_xq = to_dev(xq)
    d_xs = to_dev(oracle.repack(xs, K)[:oracle.repack_atom_bytes(M, K)].copy())
    d_gx = torch.tensor([gx], dtype=torch.float32, device="cuda")
    y = torch.zeros(M, N, dtype=torch.float32, device="cuda")
    work = torch.zeros(nv.nvfp4_workspace_bytes(1, M, K, N, nv.NVFP4_W4A4), dtype=torch.uint8,
                       device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    nv.nvfp4_debug_expire_waits(True)
    try:
        with w4a4_kernel(kernel):
            nv.nvfp4_linear_nvfp4_x(d_xq, d_xs, d_gx, d_wq, d_swz, d_g, y, work)
    finally:
        nv.nvfp4_debug_expire_waits(False)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 10.0
    assert nv.nvfp4_workspace_error(work) & NVFP4_DEVERR_TIMEOUT
    work.zero_()
    with w4a4_kernel(kernel):
        nv.nvfp4_linear_nvfp4_x(d_xq, d_xs, d_gx, d_wq, d_swz, d_g, y, work)
    torch.cuda.synchronize()
    assert nv.nvfp4_workspace_error(work) == 0
    rng = np.random.default_rng(4)
    pm = np.concatenate([rng.integers(0, M, 2048), np.full(N, M - 1)])
    pn = np.concatenate([rng.integers(0, N, 2048), np.arange(N)])
    y_ref, ab = oracle.linear_w4a4_pairs(xq, xs, gx, wq, ws, gw, pm, pn)
    check_tolerance(y_to_f64(y)[pm, pn], y_ref, ab, "nvfp4 x after a time-out")
