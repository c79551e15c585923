"""The structured inputs of the exact-parity GPU tests (tests/test_gpu_exact.py), checked
on the CPU with the oracle:

- every term x_k * e2m1 * e4m3 * g_w is a multiple of u = 2^-4 g_w, and sum_k |x_k w_k|
  stays below 2^24 u, so any order of fp32 additions gives the exact sum (and y_ref is an
  fp32 value);
- the exact comparison sees a dropped block: zeroing the scale of any one block of K
  (what a kernel that skipped the block would compute) changes every output;
- it sees a neighbour's scale applied to a block: every output whose row has different
  scales in the two blocks changes;
- the same for W4A4, where x is first quantized to NVFP4 (one nonzero code per block):
  there the block-scaled sum S is exact in fp32 and y = S g_x g_w, which the kernels round
  once.
"""
import numpy as np
import pytest

import oracle
from synth import sparse_block_x, structured_nvfp4_weights


@pytest.mark.parametrize("M,K,N", [(2, 17408, 48), (3, 5120, 64)])
def test_terms_sum_exactly_in_fp32(M, K, N):
    x = sparse_block_x(M, K, seed=1)
    wq, ws, gw = structured_nvfp4_weights(N, K, seed=2)
    y, ab = oracle.linear_w4a16(x, wq, ws, gw)
    u = 2.0 ** -4 * gw
    assert ab.max() < 2.0 ** 24 * u
    assert np.array_equal(y.astype(np.float32).astype(np.float64), y)
    # every term is a multiple of u: so is the result
    assert np.array_equal(np.round(y / u), y / u)


def test_dropped_block_changes_every_output():
    M, K, N = 2, 17408, 40
    x = sparse_block_x(M, K, seed=3)
    wq, ws, gw = structured_nvfp4_weights(N, K, seed=4)
    y, _ = oracle.linear_w4a16(x, wq, ws, gw)
    rng = np.random.default_rng(0)
    for b in [0, K // 16 - 1] + list(rng.integers(1, K // 16 - 1, 6)):
        ws2 = ws.copy()
        ws2[:, b] = 0
        y2, _ = oracle.linear_w4a16(x, wq, ws2, gw)
        assert np.all(y2 != y), "block %d" % b


def test_neighbour_scale_changes_the_outputs_it_touches():
    M, K, N = 2, 5120, 64
    x = sparse_block_x(M, K, seed=5)
    wq, ws, gw = structured_nvfp4_weights(N, K, seed=6)
    y, _ = oracle.linear_w4a16(x, wq, ws, gw)
    for b in (0, 17, K // 16 - 2):
        ws2 = ws.copy()
        ws2[:, b] = ws[:, b + 1]
        y2, _ = oracle.linear_w4a16(x, wq, ws2, gw)
        differs = ws[:, b] != ws[:, b + 1]
        assert differs.any()
        assert np.all(y2[:, differs] != y[:, differs])
        assert np.array_equal(y2[:, ~differs], y[:, ~differs])


@pytest.mark.parametrize("gx", [None, 2.0 ** -5])
def test_w4a4_structured_inputs(gx):
    M, K, N = 3, 17408, 32
    x = sparse_block_x(M, K, seed=7)
    wq, ws, gw = structured_nvfp4_weights(N, K, seed=8)
    y, ab, xq, xs, gxo = oracle.linear_w4a4(x, wq, ws, gw, gx)
    # y = S g_x g_w with the block-scaled sum S exact in fp32 (the kernels apply g_x g_w
    # once, in one rounding, after the sum)
    S = y / (np.float64(gxo) * gw)
    assert np.array_equal(S.astype(np.float32).astype(np.float64), S)
    # one nonzero code per block of x
    codes = np.empty((M, K), dtype=np.uint8)
    codes[:, 0::2] = xq & 15
    codes[:, 1::2] = xq >> 4
    assert np.all(((codes & 7) != 0).reshape(M, K // 16, 16).sum(axis=2) == 1)
    xs2 = xs.copy()
    xs2[:, 5] = 0
    y2, _ = oracle.linear_w4a4_pairs(xq, xs2, gxo, wq, ws, gw,
                                     *[a.ravel() for a in np.meshgrid(np.arange(M),
                                                                      np.arange(N),
                                                                      indexing="ij")])
    assert np.all(y2.reshape(M, N) != y)
