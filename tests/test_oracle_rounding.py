"""Pins of the oracle's E2M1 / E4M3 value sets and rounding functions.

The oracle rounds by a nearest-value search on the decoded grid; these tests hold it
against (a) the formats' closed-form facts (tests/golden/formats.json), (b) an
independent integer formulation (tests/pins/rounding_pin.c) over every fp32 bit
pattern (E2M1) or every pattern of the rounding window plus a strided sweep of the
full range (E4M3; outside [2^-12, 2^10) the answer is 0 or 448), and (c) round trips
of every finite code.
"""
import ctypes
import json
import math
import os

import numpy as np

import oracle
from conftest import GOLDEN

FMT = json.load(open(os.path.join(GOLDEN, "formats.json")))


def _fn(name):
    return ctypes.cast(getattr(oracle._load(), name), ctypes.c_void_p)


def _bits(x):
    return int(np.array([x], dtype=np.float32).view(np.uint32)[0])


def test_e2m1_value_table():
    vals = [float(v) for v in FMT["e2m1_values"]]
    for c in range(8):
        assert oracle.e2m1_value(c) == vals[c]
        assert oracle.e2m1_value(c | 8) == -vals[c]
        assert math.copysign(1.0, oracle.e2m1_value(c | 8)) == -1.0


def test_e2m1_midpoints_tie_to_even_code():
    for v, code in FMT["e2m1_midpoints_to_code"]:
        assert int(oracle.e2m1_encode([float(v)])[0]) == code
        assert int(oracle.e2m1_encode([-float(v)])[0]) == code | 8


def test_e2m1_sign_and_saturation():
    enc = oracle.e2m1_encode
    assert int(enc([-0.1])[0]) == 8  # the sign survives rounding to zero
    assert int(enc([-0.0])[0]) == 8
    assert int(enc([0.0])[0]) == 0
    assert list(enc([6.0, 6.5, 7.0, 1e30, 3.4e38])) == [7] * 5
    assert list(enc([-6.0, -1e30])) == [15, 15]
    assert int(enc([np.float32(1e-45)])[0]) == 0


def test_e4m3_known_values():
    for hx, val, _ in FMT["e4m3_known"]:
        got = oracle.e4m3_value(int(hx, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val), hx
    assert math.isnan(oracle.e4m3_value(0xFF))
    assert oracle.e4m3_value(0xFE) == -448.0


def test_e4m3_values_increase_with_code():
    prev = -1.0
    for c in range(127):
        v = oracle.e4m3_value(c)
        assert v > prev
        prev = v


def test_e4m3_rounding_boundaries():
    for v, hx in FMT["e4m3_rounding"]:
        assert int(oracle.e4m3_encode([float(v)])[0]) == int(hx, 16), v


def test_e4m3_round_trip_all_finite_codes():
    vals = np.array([oracle.e4m3_value(c) for c in range(127)], dtype=np.float32)
    assert list(oracle.e4m3_encode(vals)) == list(range(127))


def test_e2m1_round_trip_all_codes():
    vals = np.array([oracle.e2m1_value(c) for c in range(16)], dtype=np.float32)
    assert list(oracle.e2m1_encode(vals)) == list(range(16))


def test_pin_formulation_against_closed_forms(pin_lib):
    # the pin itself is checked first, so the sweeps compare two checked things
    for v, code in FMT["e2m1_midpoints_to_code"]:
        assert pin_lib.pin_e2m1_from_bits(_bits(float(v))) == code
    for v, hx in FMT["e4m3_rounding"]:
        assert pin_lib.pin_e4m3_from_bits(_bits(float(v))) == int(hx, 16)
    for hx, val, _ in FMT["e4m3_known"]:
        if val not in ("nan",):
            assert pin_lib.pin_e4m3_from_bits(_bits(float(val))) == int(hx, 16)


def test_e2m1_exhaustive_all_fp32_patterns(pin_lib):
    first = ctypes.c_uint32(0)
    bad = pin_lib.pin_sweep_e2m1(_fn("orc_e2m1_encode"), 0, 2 ** 32 - 1, 1, ctypes.byref(first))
    assert bad == 0, "first mismatching fp32 pattern 0x%08x" % first.value


def test_e4m3_exhaustive_rounding_window(pin_lib):
    first = ctypes.c_uint32(0)
    lo, hi = (127 - 12) << 23, ((127 + 10) << 23) - 1
    bad = pin_lib.pin_sweep_e4m3(_fn("orc_e4m3_encode"), lo, hi, 1, ctypes.byref(first))
    assert bad == 0, "first mismatching fp32 pattern 0x%08x" % first.value


def test_e4m3_strided_full_range(pin_lib):
    first = ctypes.c_uint32(0)
    bad = pin_lib.pin_sweep_e4m3(_fn("orc_e4m3_encode"), 0, 2 ** 32 - 1, 257,
                                 ctypes.byref(first))
    assert bad == 0, "first mismatching fp32 pattern 0x%08x" % first.value


def test_bf16_round_and_widen():
    assert int(oracle.round_bf16([1.0])[0]) == 0x3F80
    assert int(oracle.round_bf16([1.0 + 2 ** -8])[0]) == 0x3F80      # tie -> even (down)
    assert int(oracle.round_bf16([1.0 + 3 * 2 ** -8])[0]) == 0x3F82  # tie -> even (up)
    assert int(oracle.round_bf16([1.0 + 2 ** -8 + 2 ** -20])[0]) == 0x3F81
    assert int(oracle.round_bf16([-2.5])[0]) == 0xC020
    w = oracle.bf16_to_f32(np.array([0x3F80, 0xC020, 0x0001], dtype=np.uint16))
    assert w[0] == 1.0 and w[1] == -2.5 and w[2] == np.float32(2.0 ** -133)
