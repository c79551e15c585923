"""Pins of the oracle's fused activation step (reading R11): its fp32 exp against the
mathematical exp, silu(g) * u against its fp64 definition, the gate/up column layout,
and the hand-checkable special cases (zeros, the clamps, signed zeros).
"""
import math
import struct

import numpy as np
import pytest
import torch

import oracle


def _ulp(v: float) -> float:
    """Spacing of fp32 numbers at |v| (normal range)."""
    return 2.0 ** (math.frexp(abs(v))[1] - 24)


def _f32(v: float) -> float:
    return struct.unpack("<f", struct.pack("<f", v))[0]


def test_exp_within_two_ulp_of_exp():
    xs = np.concatenate([np.linspace(-87.0, 88.0, 150001, dtype=np.float32),
                         np.float32(np.log(2.0)) * np.arange(-125, 127, dtype=np.float32),
                         np.array([1e-8, -1e-8, 0.34657, -0.34657, 0.5, -0.5], np.float32)])
    worst = 0.0
    for x in xs:
        x = float(x)
        t = math.exp(x)
        if t < 2.0 ** -126:
            continue
        worst = max(worst, abs(oracle.exp_f32(x) - t) / _ulp(t))
    assert worst <= 2.0, worst


def test_exp_special_values():
    assert oracle.exp_f32(0.0) == 1.0
    assert oracle.exp_f32(-0.0) == 1.0
    assert oracle.exp_f32(88.5) == math.inf and oracle.exp_f32(1e30) == math.inf
    assert oracle.exp_f32(-87.5) == 0.0 and oracle.exp_f32(-1e30) == 0.0
    # at the clamps the result is still a normal float, within 2 ulp of exp
    for x in (88.0, -87.0):
        t = math.exp(x)
        assert abs(oracle.exp_f32(x) - t) <= 2 * _ulp(t)
    # monotone over a fine grid around 1
    xs = np.float32(1.0) + np.arange(-2000, 2000, dtype=np.float32) * np.float32(2.0 ** -20)
    ys = [oracle.exp_f32(float(x)) for x in xs]
    assert all(a <= b for a, b in zip(ys, ys[1:]))


def test_silu_mul_against_definition():
    rng = np.random.default_rng(0)
    g = rng.uniform(-30, 30, 20000).astype(np.float32)
    u = rng.normal(0, 2, 20000).astype(np.float32)
    for gi, ui in zip(g, u):
        gi, ui = float(gi), float(ui)
        want = gi / (1.0 + math.exp(-gi)) * ui
        got = oracle.silu_mul_f32(gi, ui)
        if abs(want) < 2.0 ** -100:
            assert abs(got - want) <= 2.0 ** -120
        else:
            assert abs(got - want) <= 4 * _ulp(want), (gi, ui, got, want)


def test_silu_mul_special_cases():
    assert oracle.silu_mul_f32(0.0, 3.0) == 0.0
    assert math.copysign(1.0, oracle.silu_mul_f32(0.0, -3.0)) == -1.0   # 0 * -3 = -0
    assert oracle.silu_mul_f32(5.0, 0.0) == 0.0
    # exp(-g) clamped to 0 for g > 87: silu(g) = g exactly, h = RN(g * u)
    assert oracle.silu_mul_f32(100.0, 1.5) == 150.0
    assert oracle.silu_mul_f32(90.0, _f32(1.1)) == _f32(90.0 * _f32(1.1))
    # exp(-g) = inf for g < -88: silu(g) = g / inf = -0, h = -0 * u
    h = oracle.silu_mul_f32(-100.0, 2.0)
    assert h == 0.0 and math.copysign(1.0, h) == -1.0
    h = oracle.silu_mul_f32(-100.0, -2.0)
    assert h == 0.0 and math.copysign(1.0, h) == 1.0
    # silu(g) for moderate g, u = 1: g * sigmoid(g) in closed form
    assert abs(oracle.silu_mul_f32(1.0, 1.0) - 1.0 / (1.0 + math.exp(-1.0))) <= 2 * _ulp(0.73)


def test_gate_up_layout():
    # gate in columns [0, I), up in [I, 2I): a swapped reading fails
    M, I = 3, 48
    rng = np.random.default_rng(1)
    gate = torch.tensor(rng.uniform(-6, 6, (M, I)), dtype=torch.bfloat16)
    up = torch.tensor(rng.uniform(-2, 2, (M, I)), dtype=torch.bfloat16)
    h = oracle.silu_mul(torch.cat([gate, up], dim=1))
    for m in range(M):
        for i in range(I):
            assert h[m, i] == np.float32(oracle.silu_mul_f32(float(gate[m, i]), float(up[m, i])))
    ones = torch.ones(M, I, dtype=torch.bfloat16)
    hs = oracle.silu_mul(torch.cat([gate, ones], dim=1))
    want = gate.double() / (1.0 + torch.exp(-gate.double()))
    assert np.allclose(hs, want.numpy(), rtol=1e-6, atol=1e-30)


def test_silu_mul_quantize_is_the_chain():
    rng = np.random.default_rng(2)
    gu = torch.tensor(rng.normal(0, 3, (5, 96)), dtype=torch.bfloat16)
    a = oracle.silu_mul_quantize(gu)
    b = oracle.quantize(oracle.silu_mul(gu))
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    assert a[2] == b[2]
    c = oracle.silu_mul_quantize(gu, global_scale=0.01)
    assert c[2] == np.float32(0.01)
    with pytest.raises(ValueError):
        oracle.silu_mul_quantize(torch.full((1, 32), float("nan"), dtype=torch.bfloat16))
