"""Pins of the oracle's NVFP4 quantizer.

- a hand-worked 3 x 32 tensor (tests/golden/hand_quantize.json): every E2M1 midpoint,
  a rounded E4M3 scale, a subnormal scale, an E4M3 tie, zero and tiny blocks;
- exact round trips: tensors built as code * scale * g with g a power of two
  re-quantize to the same codes and scales, for all 16 codes x all 126 nonzero
  finite scales;
- invariants on random data: the per-element error bound of round-to-nearest on
  the grid, and scale/global-scale consistency;
- the static global scale (given g) with saturation.
"""
import json
import os

import numpy as np
import pytest

import oracle
from conftest import GOLDEN

HAND = json.load(open(os.path.join(GOLDEN, "hand_quantize.json")))


def _hexes(rows):
    return np.array([[int(h, 16) for h in r] for r in rows], dtype=np.uint8)


def test_hand_worked_tensor():
    t = np.array([[float(v) for v in r] for r in HAND["input"]], dtype=np.float32)
    packed, scales, g = oracle.quantize(t)
    assert g == float(HAND["expected_global_scale"])
    np.testing.assert_array_equal(scales, _hexes(HAND["expected_scales_hex"]))
    np.testing.assert_array_equal(packed, _hexes(HAND["expected_packed_hex"]))


def test_hand_worked_tensor_as_bf16_bits():
    # every input of the fixture is exactly representable in bf16
    t = np.array([[float(v) for v in r] for r in HAND["input"]], dtype=np.float32)
    bits = (t.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(oracle.bf16_to_f32(bits), t)
    packed, scales, g = oracle.quantize(bits)
    np.testing.assert_array_equal(packed, _hexes(HAND["expected_packed_hex"]))
    np.testing.assert_array_equal(scales, _hexes(HAND["expected_scales_hex"]))


def _round_trip_tensor(g_exp):
    """Rows = scales 1..126 (row 0 uses 0x7E so that amax = 2688 g); each row holds all
    16 codes in a row-dependent order, times scale times g = 2^g_exp."""
    g = 2.0 ** g_exp
    scale_codes = [126] + list(range(1, 126))
    rng = np.random.default_rng(7)
    rows, want_codes = [], []
    for s in scale_codes:
        codes = rng.permutation(16)
        rows.append([oracle.e2m1_value(c) * oracle.e4m3_value(s) * g for c in codes])
        want_codes.append(codes)
    t = np.array(rows, dtype=np.float64)
    assert np.array_equal(t.astype(np.float32).astype(np.float64), t)  # exact in fp32
    return t.astype(np.float32), np.array(scale_codes), np.array(want_codes), g


@pytest.mark.parametrize("g_exp", [-20, -8, 0, 10])
def test_round_trip_every_code_every_scale(g_exp):
    t, scale_codes, want_codes, g = _round_trip_tensor(g_exp)
    packed, scales, g_got = oracle.quantize(t)
    assert g_got == g
    np.testing.assert_array_equal(scales[:, 0], scale_codes)
    codes = np.empty((t.shape[0], 16), dtype=np.uint8)
    codes[:, 0::2] = packed & 15
    codes[:, 1::2] = packed >> 4
    np.testing.assert_array_equal(codes, want_codes)
    # and the dequantized tensor is the input, exactly (signed zeros included)
    deq = oracle.dequantize(packed, scales, g_got, 16)
    assert np.array_equal(deq, t.astype(np.float64))
    assert np.array_equal(np.signbit(deq), np.signbit(t))


def test_all_zero_tensor():
    t = np.zeros((4, 32), dtype=np.float32)
    t[1, 3] = -0.0
    packed, scales, g = oracle.quantize(t)
    assert g == 1.0
    assert not scales.any()
    assert packed[1, 1] == 0x80 and packed.sum() == 0x80


def test_tiny_block_next_to_large_block():
    t = np.zeros((1, 32), dtype=np.float32)
    t[0, :16] = np.linspace(-5, 5, 16)
    t[0, 16:] = 1e-7 * np.array([1, -1] * 8)   # s_raw far below 2^-10
    packed, scales, g = oracle.quantize(t)
    assert scales[0, 1] == 0
    assert list(packed[0, 8:]) == [0x80] * 8   # signed zero codes


def test_non_finite_rejected():
    for bad in (np.inf, -np.inf, np.nan):
        t = np.ones((1, 16), dtype=np.float32)
        t[0, 5] = bad
        with pytest.raises(ValueError):
            oracle.quantize(t)
    with pytest.raises(ValueError):
        oracle.quantize(np.ones((1, 16), dtype=np.float32), global_scale=0.0)


def _grid_half_step(a):
    """Half the distance to the next E2M1 grid value above |v| (within [0, 6])."""
    return np.where(a < 2.0, 0.25, np.where(a < 4.0, 0.5, 1.0))


@pytest.mark.parametrize("seed,scale", [(0, 1.0), (1, 0.02), (2, 1e-3), (3, 300.0)])
def test_random_error_bounds(seed, scale):
    rng = np.random.default_rng(seed)
    t = (rng.standard_normal((64, 256)) * scale).astype(np.float32)
    t[3, 7] *= 50.0  # an outlier sets amax
    packed, scales, g = oracle.quantize(t)
    assert g == np.float32(np.abs(t).max()) / np.float32(2688.0)
    assert scales.max() <= 0x7E
    deq = oracle.dequantize(packed, scales, g, 256)
    d = np.repeat(np.array([[oracle.e4m3_value(s) for s in r] for r in scales]) * g, 16, axis=1)
    v = t.astype(np.float64) / np.where(d == 0, 1, d)
    # where the block max maps to <= 6, the error is at most half a grid step (times
    # d) plus the fp32 division's relative rounding; above 6 (scale rounded down) it
    # is the saturation error |v| - 6
    bound = np.where(np.abs(v) <= 6.0, _grid_half_step(np.abs(v)) * (1 + 1e-6),
                     np.abs(v) - 6.0 + 1e-6) * d
    err = np.abs(deq - t.astype(np.float64))
    assert np.all(err <= bound + 1e-30), float((err - bound).max())
    # the block scale is the E4M3 rounding of bmax / (6 g): within one E4M3 step
    bmax = np.abs(t.reshape(64, 16, 16)).max(axis=2)
    s_raw = bmax / (6.0 * g)
    sv = np.array([[oracle.e4m3_value(s) for s in r] for r in scales])
    assert np.all(np.abs(sv - s_raw) <= np.maximum(s_raw / 16.0, 2.0 ** -10) * 1.0001)


def test_static_global_scale_saturates():
    t = np.array([[10000.0, -3.0] + [0.0] * 14], dtype=np.float32)
    packed, scales, g = oracle.quantize(t, global_scale=1.0)
    assert g == 1.0
    assert scales[0, 0] == 0x7E            # 10000/6 saturates to 448
    assert packed[0, 0] & 15 == 7          # 10000/448 = 22.3 saturates to 6
    assert packed[0, 0] >> 4 == 8          # -3/448 rounds to -0
    deq = oracle.dequantize(packed, scales, g, 16)
    assert deq[0, 0] == 2688.0
