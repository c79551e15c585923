"""Pins of the oracle's linear (W4A16 and W4A4).

- exact rational brute force on tiny shapes (Python Fractions from the decoded codes,
  which are pinned on their own), M != N != K so a transposed operand fails;
- special cases with exact answers: one-hot x (a dequantized column of W) and a
  permutation-like W (one nonzero code per row: a scaled gather of x);
- fp64 matmul of the decoded operands;
- the pair sampler equals the full linear;
- W4A4: the quantized x equals the quantizer's output and y is the product of the
  decoded operands.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from synth import make_inputs


def _codes(packed):
    c = np.empty((packed.shape[0], packed.shape[1] * 2), dtype=np.uint8)
    c[:, 0::2] = packed & 15
    c[:, 1::2] = packed >> 4
    return c


def _bits(x):
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("M,K,N,seed", [(1, 16, 3, 0), (3, 48, 5, 1), (5, 64, 2, 2)])
def test_exact_rational_brute_force(M, K, N, seed):
    x, w = make_inputs(M, K, N, seed)
    wq, ws, gw = oracle.quantize(w)
    y, ab = oracle.linear_w4a16(x, wq, ws, gw)
    xf = oracle.bf16_to_f32(_bits(x))
    codes = _codes(wq)
    for m in range(M):
        for n in range(N):
            exact = Fraction(0)
            exact_abs = Fraction(0)
            for k in range(K):
                term = (Fraction(float(xf[m, k])) * Fraction(oracle.e2m1_value(codes[n, k]))
                        * Fraction(oracle.e4m3_value(ws[n, k // 16])) * Fraction(gw))
                exact += term
                exact_abs += abs(term)
            # fp64 summation of K exact terms: |err| <= K * 2^-53 * sum|terms|
            assert abs(Fraction(y[m, n]) - exact) <= Fraction(K, 2 ** 53) * exact_abs
            assert abs(Fraction(ab[m, n]) - exact_abs) <= Fraction(K, 2 ** 53) * exact_abs


def test_one_hot_x_gives_a_dequantized_column():
    K, N = 64, 9
    _, w = make_inputs(1, K, N, 4)
    wq, ws, gw = oracle.quantize(w)
    deq = oracle.dequantize(wq, ws, gw, K)
    for j in (0, 17, 63):
        x = torch.zeros(1, K, dtype=torch.bfloat16)
        x[0, j] = 1.0
        y, _ = oracle.linear_w4a16(x, wq, ws, gw)
        assert np.array_equal(y[0], deq[:, j])


def test_permutation_like_w_gives_a_scaled_gather():
    K, N, M = 32, 6, 3
    rng = np.random.default_rng(5)
    perm = rng.permutation(K)[:N]
    w = np.zeros((N, K), dtype=np.float32)
    w[np.arange(N), perm] = [1.5, -3.0, 0.5, 6.0, -1.0, 2.0]
    wq, ws, gw = oracle.quantize(w)
    x, _ = make_inputs(M, K, N, 6)
    y, _ = oracle.linear_w4a16(x, wq, ws, gw)
    xf = oracle.bf16_to_f32(_bits(x)).astype(np.float64)
    deq = oracle.dequantize(wq, ws, gw, K)
    want = xf[:, perm] * deq[np.arange(N), perm][None, :]
    assert np.array_equal(y, want)


def test_matches_fp64_matmul_of_decoded_operands():
    M, K, N = 4, 96, 40
    x, w = make_inputs(M, K, N, 8, outliers=True)
    wq, ws, gw = oracle.quantize(w)
    y, ab = oracle.linear_w4a16(x, wq, ws, gw)
    xf = oracle.bf16_to_f32(_bits(x)).astype(np.float64)
    # decode here from the code/scale tables, independently of the oracle's linear
    e2 = np.array([oracle.e2m1_value(c) for c in range(16)])
    e4 = np.array([oracle.e4m3_value(s) for s in range(256)])
    wd = e2[_codes(wq)] * np.repeat(e4[ws], 16, axis=1) * gw
    ref = xf @ wd.T
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12 * np.abs(xf) .sum())
    np.testing.assert_allclose(ab, np.abs(xf) @ np.abs(wd).T, rtol=1e-12)


def test_pairs_equal_full():
    M, K, N = 3, 80, 21
    x, w = make_inputs(M, K, N, 9)
    wq, ws, gw = oracle.quantize(w)
    y, ab = oracle.linear_w4a16(x, wq, ws, gw)
    pm = np.array([0, 2, 1, 2, 0])
    pn = np.array([0, 20, 7, 3, 11])
    yp, abp = oracle.linear_w4a16_pairs(x, wq, ws, gw, pm, pn)
    assert np.array_equal(yp, y[pm, pn]) and np.array_equal(abp, ab[pm, pn])
    with pytest.raises(ValueError):
        oracle.linear_w4a16_pairs(x, wq, ws, gw, [3], [0])


@pytest.mark.parametrize("gx", [None, 0.01])
def test_w4a4_is_product_of_decoded_operands(gx):
    M, K, N = 5, 64, 12
    x, w = make_inputs(M, K, N, 10)
    wq, ws, gw = oracle.quantize(w)
    y, ab, xq, xs, gx_got = oracle.linear_w4a4(x, wq, ws, gw, gx)
    xq2, xs2, gx2 = oracle.quantize(x, gx)
    assert np.array_equal(xq, xq2) and np.array_equal(xs, xs2) and gx_got == gx2
    if gx is not None:
        assert gx_got == np.float32(gx)
    xd = oracle.dequantize(xq, xs, gx_got, K)
    wd = oracle.dequantize(wq, ws, gw, K)
    np.testing.assert_allclose(y, xd @ wd.T, rtol=0, atol=1e-12 * np.abs(xd).sum())
    yp, abp = oracle.linear_w4a4_pairs(xq, xs, gx_got, wq, ws, gw, [0, 4], [11, 3])
    assert np.array_equal(yp, y[[0, 4], [11, 3]])
