"""GPU parity of the quantizer, the repack and the element rounding, against the
oracle, bit for bit (all calls go through the C ABI)."""
import json
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import nvfp4_weight_quantized_quantize_gb300 as nv
import oracle
from conftest import GOLDEN
from helpers import to_dev
from synth import make_inputs, random_fp8_block128, random_w, workload_inputs

pytestmark = pytest.mark.gpu


def gpu_quantize(src: torch.Tensor):
    rows, cols = src.shape
    d = src.cuda()
    packed = torch.empty(rows, cols // 2, dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, cols // 16, dtype=torch.uint8, device="cuda")
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(nv.nvfp4_workspace_bytes(0, rows, cols), dtype=torch.uint8, device="cuda")
    nv.nvfp4_quantize(d, packed, scales, g, ws)
    torch.cuda.synchronize()
    return packed.cpu().numpy(), scales.cpu().numpy(), float(g.item())


def assert_same_quantization(src: torch.Tensor):
    p, s, g = gpu_quantize(src)
    src_o = src if src.dtype == torch.bfloat16 else src.numpy()
    po, so, go = oracle.quantize(src_o)
    assert g == go
    np.testing.assert_array_equal(s, so)
    np.testing.assert_array_equal(p, po)


def test_hand_worked_tensor():
    h = json.load(open(os.path.join(GOLDEN, "hand_quantize.json")))
    t = torch.tensor([[float(v) for v in r] for r in h["input"]], dtype=torch.float32)
    p, s, g = gpu_quantize(t)
    assert g == float(h["expected_global_scale"])
    np.testing.assert_array_equal(s, [[int(v, 16) for v in r] for r in h["expected_scales_hex"]])
    np.testing.assert_array_equal(p, [[int(v, 16) for v in r] for r in h["expected_packed_hex"]])


def test_scale_op_order_tensors():
    # g not a power of two, block quotients within one ulp of an E4M3 midpoint: only
    # the product-first order bmax / (6 g) gives the fixture's bytes
    fx = json.load(open(os.path.join(GOLDEN, "scale_op_order.json")))
    for case in fx["cases"]:
        t = torch.tensor([[float(v) for v in case["input"]]], dtype=torch.float32)
        p, s, g = gpu_quantize(t)
        assert float(g).hex() == case["expected_global_scale"], case["name"]
        assert ["%02X" % b for b in s[0]] == case["expected_scales_hex"], case["name"]
        assert ["%02X" % b for b in p[0]] == case["expected_packed_hex"], case["name"]


@pytest.mark.parametrize("rows,cols,seed", [(1, 16, 0), (3, 48, 1), (129, 80, 2),
                                            (256, 512, 3), (1000, 1040, 4)])
def test_ragged_shapes_fp32(rows, cols, seed):
    assert_same_quantization(random_w(rows, cols, seed, std=0.5))


@pytest.mark.parametrize("rows,cols,seed", [(1, 16, 5), (7, 5120, 6), (300, 96, 7)])
def test_bf16_input(rows, cols, seed):
    assert_same_quantization(random_w(rows, cols, seed).to(torch.bfloat16))


def test_round_trip_tensor_every_code_every_scale():
    rng = np.random.default_rng(11)
    g = 2.0 ** -8
    rows = []
    for s in [126] + list(range(1, 126)):
        codes = rng.permutation(16)
        rows.append([oracle.e2m1_value(c) * oracle.e4m3_value(s) * g for c in codes])
    assert_same_quantization(torch.tensor(np.array(rows), dtype=torch.float32))


def test_zero_and_tiny_blocks():
    t = torch.zeros(5, 64)
    t[1, 5] = -0.0
    assert_same_quantization(t)  # all-zero tensor: g = 1, signed zero codes
    t[2, :16] = torch.linspace(-3, 3, 16)
    t[3, 16:32] = 1e-8
    t[4, 48:] = -1e-30
    assert_same_quantization(t)


@pytest.mark.parametrize("amax", [1.0, 0.0123456, 3.3e-20, 7.7e25, 1e-36, 1e38])
def test_quotients_next_to_every_midpoint(amax):
    """Elements within +-3 ulps of every E2M1 decision point m * d, for every block scale:
    the element codes hang on the last bit of the fp32 quotient t / d."""
    f32 = np.float32
    amax = f32(amax)
    g = f32(amax / f32(2688.0))
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    rows = []
    for s in range(1, 127):
        sval = f32(oracle.e4m3_value(s))
        bmax = f32(sval * f32(6.0) * g)
        if not (0 < bmax < amax):
            continue
        s8 = int(oracle.e4m3_encode(np.array([bmax / (f32(6.0) * g)], dtype=np.float32))[0])
        d = f32(f32(oracle.e4m3_value(s8)) * g)
        if d == 0:
            continue
        vals = []
        for m in mids:
            c = f32(f32(m) * d)
            for k in (-3, -2, -1, 0, 1, 2, 3):
                v = c
                for _ in range(abs(k)):
                    v = np.nextafter(v, f32(np.inf) if k > 0 else f32(0))
                vals.append(v)
        vals = vals[:45]
        # 3 blocks: bmax first in each, then the 45 probe values (both signs)
        row = []
        for b in range(3):
            blk = vals[15 * b:15 * b + 15]
            blk = [(-x if (i + b) % 2 else x) for i, x in enumerate(blk)]
            row += [bmax] + blk
        rows.append(row)
    t = np.array(rows, dtype=np.float32)
    t[0, 0] = amax  # the tensor's amax
    assert_same_quantization(torch.from_numpy(t))


def test_outliers_and_extreme_ranges():
    for scale in (1e-30, 1e-3, 1.0, 1e30):
        assert_same_quantization(random_w(64, 256, 12, std=scale))


@pytest.mark.parametrize("name", ["tiny", "decode_a", "decode_b", "verify_b"])
def test_workload_weights(name):
    _, w = workload_inputs(name, M=1)
    assert_same_quantization(w)


@pytest.mark.parametrize("rows,cols,seed", [(1, 16, 0), (128, 64, 1), (130, 80, 2),
                                            (17408, 5120, 3)])
def test_repack_matches_oracle(rows, cols, seed):
    rng = np.random.default_rng(seed)
    s = rng.integers(0, 127, size=(rows, cols // 16), dtype=np.uint8)
    out = torch.full((nv.nvfp4_repack_bytes(rows, cols),), 0xAB, dtype=torch.uint8,
                     device="cuda")
    nv.nvfp4_repack(to_dev(s), cols, out)
    np.testing.assert_array_equal(out.cpu().numpy(), oracle.repack(s, cols))


def _oracle_encode_chunked(fn, x: np.ndarray, workers: int = 16) -> np.ndarray:
    parts = np.array_split(x, workers)
    with ThreadPoolExecutor(workers) as ex:
        return np.concatenate(list(ex.map(fn, parts)))


def test_e2m1_rounding_every_fp32_pattern():
    chunk = 1 << 27
    for start in range(0, 1 << 32, chunk):
        bits = torch.arange(start, start + chunk, dtype=torch.int64, device="cuda")
        f = bits.to(torch.int32).view(torch.float32)
        out = torch.empty(chunk, dtype=torch.uint8, device="cuda")
        nv.nvfp4_encode_elements(f, out, None)
        host = np.arange(start, start + chunk, dtype=np.uint64).astype(np.uint32)
        finite = ((host >> 23) & 0xFF) != 0xFF
        want = _oracle_encode_chunked(oracle.e2m1_encode, host.view(np.float32))
        got = out.cpu().numpy()
        bad = np.nonzero((got != want) & finite)[0]
        assert bad.size == 0, "pattern 0x%08x: gpu %d oracle %d" % (
            host[bad[0]], got[bad[0]], want[bad[0]])


def test_e4m3_rounding_window_and_strided():
    lo, hi = (127 - 12) << 23, (127 + 10) << 23
    for start in range(lo, hi, 1 << 26):
        n = min(1 << 26, hi - start)
        host = np.arange(start, start + n, dtype=np.uint32)
        d = torch.from_numpy(host.view(np.int32)).cuda().view(torch.float32)
        out = torch.empty(n, dtype=torch.uint8, device="cuda")
        nv.nvfp4_encode_elements(d, None, out)
        want = _oracle_encode_chunked(oracle.e4m3_encode, host.view(np.float32))
        np.testing.assert_array_equal(out.cpu().numpy(), want)
    host = (np.arange(0, 1 << 32, 251, dtype=np.uint64)).astype(np.uint32)
    host = host[((host >> 23) & 0xFF) != 0xFF]
    d = torch.from_numpy(host.view(np.int32)).cuda().view(torch.float32)
    out = torch.empty(host.size, dtype=torch.uint8, device="cuda")
    nv.nvfp4_encode_elements(d, None, out)
    want = _oracle_encode_chunked(oracle.e4m3_encode, host.view(np.float32))
    np.testing.assert_array_equal(out.cpu().numpy(), want)


# ---- FP8 (E4M3, block-128) weights -> BF16 -> NVFP4 ------------------------------------

def gpu_quantize_fp8(q: np.ndarray, s: np.ndarray):
    rows, cols = q.shape
    packed = torch.empty(rows, cols // 2, dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, cols // 16, dtype=torch.uint8, device="cuda")
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(nv.nvfp4_workspace_bytes(0, rows, cols), dtype=torch.uint8, device="cuda")
    nv.nvfp4_quantize_fp8_block128(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(),
                                   packed, scales, g, ws)
    torch.cuda.synchronize()
    return packed.cpu().numpy(), scales.cpu().numpy(), float(g.item())


def assert_same_fp8_quantization(q: np.ndarray, s: np.ndarray):
    p, sc, g = gpu_quantize_fp8(q, s)
    po, so, go = oracle.quantize_fp8_block128(q, s)
    assert g == go
    np.testing.assert_array_equal(sc, so)
    np.testing.assert_array_equal(p, po)


@pytest.mark.parametrize("rows,cols,seed,kind", [
    (1, 16, 0, "normal"), (5, 48, 1, "uniform"), (129, 272, 2, "normal"),
    (130, 400, 3, "uniform"), (257, 1040, 4, "normal"), (300, 4096, 5, "uniform"),
])
def test_fp8_block128_ragged(rows, cols, seed, kind):
    assert_same_fp8_quantization(*random_fp8_block128(rows, cols, seed, kind))


def test_fp8_block128_edge_tiles():
    # tiles with a zero scale (signed zeros), scales that make fp32 and bf16 subnormals,
    # and the bytes of the hand-worked cases (signed zero, subnormal, +-448) in one column
    q, s = random_fp8_block128(200, 272, 6, "uniform")
    s[0, 0] = 0.0
    s[0, 1] = 2.0 ** -125
    s[1, 2] = 2.0 ** -120
    h = json.load(open(os.path.join(GOLDEN, "fp8_block128.json")))
    for i, case in enumerate(h["cases"]):
        q[130 + i, 5] = int(case["q"], 16)
    assert_same_fp8_quantization(q, s)


def test_fp8_block128_all_zero_scales():
    q, s = random_fp8_block128(64, 160, 7, "uniform")
    s[:] = 0.0
    p, sc, g = gpu_quantize_fp8(q, s)
    assert g == 1.0 and not sc.any()
    po, so, go = oracle.quantize_fp8_block128(q, s)
    np.testing.assert_array_equal(p, po)  # sign bits of the negative zeros


def test_fp8_block128_full_size():
    # the decode projection's shape (17408 x 5120) as a checkpoint-like FP8 tensor
    assert_same_fp8_quantization(*random_fp8_block128(17408, 5120, 8, "normal"))


def test_fp8_block128_subnormal_tensor():
    # every product an fp32 / bf16 subnormal: the global scale, the block scales and the
    # codes all hang on the subnormal bf16 roundings
    q, s = random_fp8_block128(256, 512, 9, "uniform")
    s[:] = 2.0 ** -130
    s[1, 2] = 2.0 ** -133
    s[0, 3] = 2.0 ** -127
    assert_same_fp8_quantization(q, s)
