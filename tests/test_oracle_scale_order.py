"""Pin of the order of the two fp32 operations that form a block's raw scale.

The quantizer's block scale is read as s_raw = bmax / (6 g): the product 6 g rounded to
fp32 first, then the quotient rounded to fp32.  With g a power of two every other order
gives the same bits, so the hand-worked tensors of tests/golden/hand_quantize.json
cannot tell them apart.  tests/golden/scale_op_order.json holds three tensors whose g
(amax / 2688) is not a power of two and whose second block's exact quotient lies within
one fp32 ulp of a midpoint between two E4M3 values, so that

  (bmax / 6) / g,   bmax * RN(1 / (6 g))   and   RN(bmax * RN(2688 / amax)) / 6

each round that block's scale to the other E4M3 neighbour in at least one of the cases.
The element codes of the block then follow the scale's d = e4m3 * g, and the fixture
places them where the two candidate values of d give different codes.

Two checks:
- the fixture's arithmetic, redone here with exact rationals and an fp32 rounding
  written from its definition (nearest, ties to even): g, 6 g, each order's raw scale,
  each E4M3 byte, and that every alternative order differs from the reading's in some
  case (so the fixture really discriminates);
- the oracle's quantizer against the fixture's bytes, codes and global scale.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from conftest import GOLDEN

FIX = json.load(open(os.path.join(GOLDEN, "scale_op_order.json")))
CASES = FIX["cases"]


# ---- exact arithmetic for checking the fixture's derivation -------------------------

def rn32(q: Fraction) -> Fraction:
    """q rounded to the nearest fp32 value, ties to the even significand (normal range)."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    assert -126 <= e <= 127, "outside the fp32 normal range"
    ulp = Fraction(2) ** (e - 23)
    n = a / ulp
    fl = math.floor(n)
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * ulp


def e4m3_table():
    """Values of the finite non-negative E4M3 bytes 0x00..0x7E (bias 7, 3 mantissa bits)."""
    vals = []
    for b in range(0x7F):
        e, m = (b >> 3) & 15, b & 7
        vals.append(Fraction(m, 8) * Fraction(1, 64) if e == 0
                    else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7))
    return vals


E4M3 = e4m3_table()


def e4m3_byte(s: Fraction) -> int:
    """Nearest E4M3 byte, ties to the even byte, saturating at 448."""
    if s >= 448:
        return 0x7E
    best = min(range(0x7F), key=lambda b: (abs(E4M3[b] - s), b % 2))
    return best


def fx(h: str) -> Fraction:
    return Fraction(float.fromhex(h))


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_fixture_arithmetic(case):
    t = [Fraction(float(v)) for v in case["input"]]
    assert all(rn32(v) == v for v in t), "inputs must be fp32 values"
    amax = max(abs(v) for v in t)
    g = rn32(amax / 2688)
    assert g == fx(case["expected_global_scale"])
    assert g != 2 ** round(math.log2(g)), "g must not be a power of two"
    six_g = rn32(6 * g)
    bmax = max(abs(v) for v in t[16:])
    orders = {
        "(bmax/6)/g": rn32(rn32(bmax / 6) / g),
        "bmax*RN(1/(6g))": rn32(bmax * rn32(1 / six_g)),
        "RN(bmax*RN(2688/amax))/6": rn32(rn32(bmax * rn32(Fraction(2688) / amax)) / 6),
    }
    reading = e4m3_byte(rn32(bmax / six_g))
    assert "%02X" % reading == case["expected_scales_hex"][1]
    for name, s in orders.items():
        assert "%02X" % e4m3_byte(s) == case["other_orders_block1_scale_hex"][name]


def test_fixture_discriminates_every_alternative_order():
    for name in CASES[0]["other_orders_block1_scale_hex"]:
        assert any(c["other_orders_block1_scale_hex"][name] != c["expected_scales_hex"][1]
                   for c in CASES), name


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_oracle_scale_op_order(case):
    t = np.array([[float(v) for v in case["input"]]], dtype=np.float32)
    packed, scales, g = oracle.quantize(t)
    assert float(g).hex() == case["expected_global_scale"]
    assert ["%02X" % b for b in scales[0]] == case["expected_scales_hex"]
    assert ["%02X" % b for b in packed[0]] == case["expected_packed_hex"]
    codes = np.empty(32, dtype=np.uint8)
    codes[0::2] = packed[0] & 15
    codes[1::2] = packed[0] >> 4
    assert "".join("%X" % c for c in codes) == case["expected_codes_hex"]
