"""GPU parity of the fused silu(gate) * up -> NVFP4 activation quantizer (bit for bit) and
of the linear that takes NVFP4 activations (within the linear tolerance), through the C
ABI, against the oracle.  Every input is synthetic or oracle-made; none comes from the
CUDA path."""
import numpy as np
import pytest
import torch

import nvfp4_weight_quantized_quantize_gb300 as nv
import oracle
from helpers import check_tolerance, to_dev, upload_weights, y_to_f64
from synth import make_inputs, random_gate_up, random_x

pytestmark = pytest.mark.gpu


def gpu_silu_quant(gu: torch.Tensor, given_g=None):
    M, I2 = gu.shape
    I = I2 // 2
    packed = torch.empty(M, I // 2, dtype=torch.uint8, device="cuda")
    scales = torch.empty(oracle.repack_atom_bytes(M, I), dtype=torch.uint8, device="cuda")
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(nv.nvfp4_workspace_bytes(0, M, I), dtype=torch.uint8, device="cuda")
    gg = None if given_g is None else torch.tensor([given_g], dtype=torch.float32, device="cuda")
    nv.nvfp4_silu_mul_quantize(gu.cuda(), packed, scales, g, gg,
                               None if given_g is not None else ws)
    torch.cuda.synchronize()
    return packed.cpu().numpy(), scales.cpu().numpy(), float(g.item())


def assert_same(gu: torch.Tensor, given_g=None):
    M, I = gu.shape[0], gu.shape[1] // 2
    p, s, g = gpu_silu_quant(gu, given_g)
    po, so, go = oracle.silu_mul_quantize(gu, given_g)
    assert g == go
    np.testing.assert_array_equal(p, po)
    np.testing.assert_array_equal(s, oracle.repack(so, I)[:oracle.repack_atom_bytes(M, I)])


@pytest.mark.parametrize("M,I,seed", [(1, 16, 0), (3, 48, 1), (130, 272, 2), (257, 1040, 3),
                                      (64, 4096, 4)])
def test_silu_mul_quantize_dynamic(M, I, seed):
    assert_same(random_gate_up(M, I, seed))


@pytest.mark.parametrize("given", [0.002, 0.05, 1.0])
def test_silu_mul_quantize_static_scale(given):
    # a static activation scale: small ones saturate the block scales at 448
    assert_same(random_gate_up(40, 320, 5), given)


def test_silu_mul_quantize_clamps_and_signed_zeros():
    # gate values at and around exp's clamps (|g| near 87, 88), huge ones, zeros of both
    # signs, and up = 0 or -0: h takes -0, +0, g * u exactly and the exp branches
    gu = random_gate_up(8, 64, 6)
    special = [-200.0, -88.5, -88.0, -87.5, -87.0, -86.5, -30.0, -0.0, 0.0, 1e-30, 30.0, 86.5,
               87.0, 87.5, 88.0, 88.5, 200.0, 1e30, -1e30, 1e-38, -1e-38]
    for j, v in enumerate(special):
        gu[j % 8, (3 * j) % 64] = v
    gu[2, 64:80] = 0.0
    gu[3, 80:96] = -0.0
    gu[5, :64] = -100.0  # a row of -0 activations: scales 0, codes of -0
    assert_same(gu)


def test_silu_mul_quantize_mlp_shape():
    # the 512-token prefill chunk of the fused MLP: gate_up [512, 34816] -> h [512, 17408]
    assert_same(random_gate_up(512, 17408, 7))


@pytest.mark.parametrize("M,K,N", [(1, 64, 40), (5, 1056, 300), (12, 2048, 257), (16, 512, 129),
                                   (17, 1056, 200), (300, 512, 384), (512, 2048, 640)])
def test_linear_nvfp4_x(M, K, N):
    # x quantized by the oracle (from a silu * up activation), W by the oracle
    gu = random_gate_up(M, K, 20 + M)
    xq, xs, gx = oracle.silu_mul_quantize(gu)
    _, w = make_inputs(1, K, N, seed=30 + N)
    wq, ws, gw = oracle.quantize(w.numpy())
    d_wq, d_swz, d_g = upload_weights(wq, ws, gw, K)
    d_xs = to_dev(oracle.repack(xs, K)[:oracle.repack_atom_bytes(M, K)].copy())
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    work = torch.zeros(nv.nvfp4_workspace_bytes(1, M, K, N, nv.NVFP4_W4A4), dtype=torch.uint8,
                       device="cuda")
    nv.nvfp4_linear_nvfp4_x(to_dev(xq), d_xs, torch.tensor([gx], device="cuda"), d_wq, d_swz,
                            d_g, y, work, static_weights=(M % 2 == 1))
    torch.cuda.synchronize()
    assert nv.nvfp4_workspace_error(work) == 0
    pm, pn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    y_ref, ab = oracle.linear_w4a4_pairs(xq, xs, gx, wq, ws, gw, pm.ravel(), pn.ravel())
    check_tolerance(y_to_f64(y).ravel(), y_ref, ab, "M%d K%d N%d" % (M, K, N))


def test_linear_nvfp4_x_down_projection_shape():
    # the MLP's down projection on a 512-token chunk: K = 17408, N = 5120; sampled outputs
    # and two full rows
    M, K, N = 512, 17408, 5120
    xq, xs, gx = oracle.silu_mul_quantize(random_gate_up(M, K, 8))
    _, w = make_inputs(1, K, N, seed=9)
    wq, ws, gw = oracle.quantize(w.numpy())
    d_wq, d_swz, d_g = upload_weights(wq, ws, gw, K)
    d_xs = to_dev(oracle.repack(xs, K)[:oracle.repack_atom_bytes(M, K)].copy())
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    work = torch.zeros(nv.nvfp4_workspace_bytes(1, M, K, N, nv.NVFP4_W4A4), dtype=torch.uint8,
                       device="cuda")
    nv.nvfp4_linear_nvfp4_x(to_dev(xq), d_xs, torch.tensor([gx], device="cuda"), d_wq, d_swz,
                            d_g, y, work)
    torch.cuda.synchronize()
    assert nv.nvfp4_workspace_error(work) == 0
    rng = np.random.default_rng(0)
    pm = np.concatenate([rng.integers(0, M, 4096), np.zeros(N, np.int64), np.full(N, M - 1)])
    pn = np.concatenate([rng.integers(0, N, 4096), np.arange(N), np.arange(N)])
    y_ref, ab = oracle.linear_w4a4_pairs(xq, xs, gx, wq, ws, gw, pm, pn)
    check_tolerance(y_to_f64(y)[pm, pn], y_ref, ab, "down projection")
