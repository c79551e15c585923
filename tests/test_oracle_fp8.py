"""Pins of the oracle's FP8 block-128 -> BF16 step (reading R10) and of the chain that
feeds it to the NVFP4 quantizer.

- hand-worked products and roundings (tests/golden/fp8_block128.json): bf16 ties both
  ways, two double-rounding cases that only the fp32-product-first reading produces,
  signed zeros, subnormals without flush to zero;
- every non-NaN E4M3 byte against the format's closed form;
- tile scales that are distinct powers of two, so a wrong tile index (rows and columns
  swapped, a tile width other than 128) changes the result;
- random bytes and scales against an independent route: torch's float8_e4m3fn decode,
  an fp32 multiply and torch's bf16 cast.
"""
import json
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from conftest import GOLDEN


def _f32(bits_hex):
    return struct.unpack(">f", bytes.fromhex(bits_hex))[0]


def _e4m3_magnitude(b):
    """OCP E4M3 (bias 7): 2^(e-7) * (1 + m/8), subnormal m * 2^-9; bit 7 is the sign."""
    e, m = (b >> 3) & 15, b & 7
    return Fraction(m, 512) if e == 0 else Fraction(8 + m, 8) * Fraction(2) ** (e - 7)


def _bf16_bits_exact(mag: Fraction, negative: bool) -> int:
    """bf16 bit pattern of +-mag, a value that bf16 holds exactly (checked); the sign bit
    is set for a negative zero too."""
    f = float(mag)
    assert Fraction(f) == mag
    u = struct.unpack(">I", struct.pack(">f", f))[0]
    assert u & 0xFFFF == 0
    return (u >> 16) | (0x8000 if negative else 0)


def _torch_route(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """bf16(e4m3(q) * s) by torch: float8_e4m3fn decode, fp32 multiply, bf16 cast."""
    rows, cols = q.shape
    v = torch.from_numpy(q.copy()).view(torch.float8_e4m3fn).to(torch.float32)
    t = torch.from_numpy(s).repeat_interleave(128, 0)[:rows].repeat_interleave(128, 1)[:, :cols]
    p = v * t
    return p.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _random_fp8(rows, cols, seed):
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 256, (rows, cols), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] ^= 0x01  # no NaN bytes
    s = np.exp2(rng.uniform(-14, -4, ((rows + 127) // 128, (cols + 127) // 128))).astype(np.float32)
    return q, s


def test_golden_cases():
    spec = json.load(open(os.path.join(GOLDEN, "fp8_block128.json")))
    for case in spec["cases"]:
        q = np.zeros((1, 16), dtype=np.uint8)
        q[0, 0] = int(case["q"], 16)
        s = np.array([[_f32(case["s_bits"])]], dtype=np.float32)
        got = int(oracle.dequant_fp8_block128(q, s)[0, 0])
        assert got == int(case["bf16"], 16), (case, hex(got))


def test_every_byte_against_closed_form():
    q = np.array([[b for b in range(256) if (b & 0x7F) != 0x7F]], dtype=np.uint8)
    q = np.pad(q, ((0, 0), (0, (-q.shape[1]) % 16)))
    s = np.ones((1, (q.shape[1] + 127) // 128), dtype=np.float32)
    got = oracle.dequant_fp8_block128(q, s)[0]
    for j, b in enumerate(q[0]):
        # 4 significant bits: every E4M3 value is exact in bf16
        assert got[j] == _bf16_bits_exact(_e4m3_magnitude(int(b)), bool(b & 0x80)), hex(b)


def test_nan_bytes_are_rejected_by_the_chain():
    q = np.zeros((2, 32), dtype=np.uint8)
    q[1, 5] = 0x7F
    s = np.ones((1, 1), dtype=np.float32)
    assert np.isnan(oracle.bf16_to_f32(oracle.dequant_fp8_block128(q, s)[1, 5]))
    with pytest.raises(ValueError):
        oracle.quantize_fp8_block128(q, s)


@pytest.mark.parametrize("rows,cols", [(300, 400), (129, 272), (128, 128), (5, 16)])
def test_tile_index(rows, cols):
    rng = np.random.default_rng(rows * 7 + cols)
    q = rng.integers(0, 256, (rows, cols), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x38
    ti, tj = (rows + 127) // 128, (cols + 127) // 128
    # distinct powers of two per tile: products stay exact, the tile shows in the result
    s = np.array([[2.0 ** (i - 3 * j) for j in range(tj)] for i in range(ti)], dtype=np.float32)
    got = oracle.dequant_fp8_block128(q, s)
    for r in range(0, rows, max(1, rows // 37)):
        for c in range(0, cols, max(1, cols // 41)):
            want = _e4m3_magnitude(int(q[r, c])) * Fraction(float(s[r // 128, c // 128]))
            assert got[r, c] == _bf16_bits_exact(want, bool(q[r, c] & 0x80)), (r, c)
    np.testing.assert_array_equal(got, _torch_route(q, s))


@pytest.mark.parametrize("rows,cols,seed", [(257, 1040, 1), (64, 4096, 2), (1, 16, 3)])
def test_random_against_torch(rows, cols, seed):
    q, s = _random_fp8(rows, cols, seed)
    np.testing.assert_array_equal(oracle.dequant_fp8_block128(q, s), _torch_route(q, s))


def test_chain_quantizes_the_bf16_tensor():
    # the conversion hands exactly the bf16 tensor to the quantizer: on a tensor whose
    # products are exact, the chain equals quantizing the bf16 values written out directly
    q, _ = _random_fp8(130, 272, 4)
    s = np.array([[0.25, 2.0, 1.0], [4.0, 0.5, 8.0]], dtype=np.float32)
    bits = np.zeros(q.shape, dtype=np.uint16)
    for r in range(q.shape[0]):
        for c in range(q.shape[1]):
            bits[r, c] = _bf16_bits_exact(_e4m3_magnitude(int(q[r, c]))
                                          * Fraction(float(s[r // 128, c // 128])),
                                          bool(q[r, c] & 0x80))
    a = oracle.quantize_fp8_block128(q, s)
    b = oracle.quantize(bits)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    assert a[2] == b[2]
