"""Seeded synthetic inputs for the NVFP4 projection workloads.

Shared by the tests, the smoke check and the bench: it draws random numbers and
nothing else (no quantization, rounding or layout arithmetic lives here), so both
the CUDA path and the CPU oracle can take their inputs from it.

Workloads (shapes of the decode / MTP-verify / prefill / W4A4 cases of batch-one
Qwen3.x serving; the fused gate+up projection doubles N):

  name        M     K      N      y     seed  notes
  tiny        1     512    256    f32   0
  decode_a    1     5120   17408  bf16  1     0.1% of W entries x20 (outliers)
  decode_b    1     17408  5120   bf16  2     same
  verify_a    7     5120   34816  bf16  3
  verify_b    7     5120   6144   bf16  3
  prefill_a   512   5120   34816  bf16  4     x rows scaled by U(0.5, 4)
  prefill_b   512   17408  5120   bf16  4     same
  w4a4        2048  5120   17408  bf16  5     x quantized to NVFP4 inside the call

Beyond these: FP8 block-128 checkpoints (random_fp8_block128), fused gate/up outputs
(random_gate_up) and already-encoded NVFP4 weights (random_nvfp4_weights) for the
conversion, activation and wide-N cases; x with one nonzero per 16-block
(sparse_block_x) and weights with nonzero codes and a few scale values
(structured_nvfp4_weights) for the exact-parity cases.

Draw order with ``torch.Generator(device='cpu').manual_seed(seed)``: W ~ N(0, 0.02)
fp32 first, then x ~ N(0, 1) fp32, then the outlier positions (uniform without
replacement: sequential draws with repeats discarded; the entries keep their sign
and are multiplied by 20), then the per-row x scales.  x is cast to bf16 last.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    K: int
    N: int
    y_dtype: str  # "f32" | "bf16"
    seed: int
    outliers: bool = False
    row_scale: bool = False
    w4a4: bool = False


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", 1, 512, 256, "f32", 0),
        Workload("decode_a", 1, 5120, 17408, "bf16", 1, outliers=True),
        Workload("decode_b", 1, 17408, 5120, "bf16", 2, outliers=True),
        Workload("verify_a", 7, 5120, 34816, "bf16", 3),
        Workload("verify_b", 7, 5120, 6144, "bf16", 3),
        Workload("prefill_a", 512, 5120, 34816, "bf16", 4, row_scale=True),
        Workload("prefill_b", 512, 17408, 5120, "bf16", 4, row_scale=True),
        Workload("w4a4", 2048, 5120, 17408, "bf16", 5, w4a4=True),
    ]
}


def _unique_positions(gen: torch.Generator, total: int, count: int) -> torch.Tensor:
    """`count` distinct indices in [0, total): sequential uniform draws, repeats dropped."""
    got = np.empty(0, dtype=np.int64)
    while got.size < count:
        cand = torch.randint(0, total, (2 * (count - got.size) + 16,), generator=gen,
                             dtype=torch.int64).numpy()
        allc = np.concatenate([got, cand])
        _, first = np.unique(allc, return_index=True)
        got = allc[np.sort(first)]
    return torch.from_numpy(got[:count].copy())


def make_inputs(M: int, K: int, N: int, seed: int, *, outliers: bool = False,
                row_scale: bool = False, w_std: float = 0.02):
    """Return (x bf16 [M,K], W fp32 [N,K]) on the CPU."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    w = torch.randn(N, K, generator=gen, dtype=torch.float32) * w_std
    x = torch.randn(M, K, generator=gen, dtype=torch.float32)
    if outliers:
        count = max(1, round(0.001 * N * K))
        pos = _unique_positions(gen, N * K, count)
        w.view(-1)[pos] *= 20.0
    if row_scale:
        s = torch.rand(M, 1, generator=gen, dtype=torch.float32) * 3.5 + 0.5
        x = x * s
    return x.to(torch.bfloat16), w


def workload_inputs(name: str, *, M: int | None = None):
    """Inputs of a named workload; M may be overridden (fewer rows of x)."""
    w = WORKLOADS[name]
    return make_inputs(M if M is not None else w.M, w.K, w.N, w.seed,
                       outliers=w.outliers, row_scale=w.row_scale)


def random_x(M: int, K: int, seed: int, scale: float = 1.0) -> torch.Tensor:
    gen = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(M, K, generator=gen, dtype=torch.float32) * scale).to(torch.bfloat16)


def random_fp8_block128(rows: int, cols: int, seed: int, kind: str = "normal"):
    """An FP8 "e4m3 block-128" weight: (E4M3 bytes uint8 [rows, cols], fp32 tile scales
    [ceil(rows/128), ceil(cols/128)]), on the CPU.

    kind "normal": bytes of N(0, 1) * 64 draws (clamped to +-448) as torch's
    float8_e4m3fn stores them, like a checkpoint whose tiles were scaled to use the
    format's range; tile scales 2^U(-14, -8) (weights of magnitude about 0.02).
    kind "uniform": every non-NaN byte equally likely (the widest spread of magnitudes
    inside a block), tile scales 2^U(-14, -4).
    """
    gen = torch.Generator(device="cpu").manual_seed(seed)
    nt = ((rows + 127) // 128, (cols + 127) // 128)
    if kind == "normal":
        v = (torch.randn(rows, cols, generator=gen, dtype=torch.float32) * 64.0).clamp(-448.0, 448.0)
        q = v.to(torch.float8_e4m3fn).view(torch.uint8)
        e = torch.rand(nt, generator=gen, dtype=torch.float64) * 6.0 - 14.0
    elif kind == "uniform":
        q = torch.randint(0, 254, (rows, cols), generator=gen, dtype=torch.int64)
        q = q + (q >= 0x7F).to(torch.int64)  # skip 0x7F; 254 values cover 0x00..0xFE
        q = q.to(torch.uint8)
        e = torch.rand(nt, generator=gen, dtype=torch.float64) * 10.0 - 14.0
    else:
        raise ValueError(kind)
    s = torch.exp2(e).to(torch.float32)
    return q.numpy().copy(), s.numpy().copy()


def random_gate_up(M: int, I: int, seed: int) -> torch.Tensor:
    """Output of a fused gate/up projection, bf16 [M, 2I]: gate ~ N(0, 3) in columns
    [0, I) (pre-activations reaching well into both tails of silu), up ~ N(0, 1) in
    [I, 2I)."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    gate = torch.randn(M, I, generator=gen, dtype=torch.float32) * 3.0
    up = torch.randn(M, I, generator=gen, dtype=torch.float32)
    return torch.cat([gate, up], dim=1).to(torch.bfloat16)


def random_nvfp4_weights(N: int, K: int, seed: int):
    """Already-encoded NVFP4 weights drawn directly (no quantizer involved): packed codes
    uint8 [N, K/2] with every nibble uniform over the 16 codes, E4M3 scale bytes uint8
    [N, K/16] uniform over 0x10 .. 0x5F (normal values 2^-5 .. 2^4 * 1.875), and a global
    scale 2^-8.  For linear tests at sizes where quantizing a float tensor on the CPU
    would take too long."""
    rng = np.random.default_rng(seed)
    packed = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scales = rng.integers(0x10, 0x60, (N, K // 16), dtype=np.uint8)
    return packed, scales, 2.0 ** -8


def sparse_block_x(M: int, K: int, seed: int) -> torch.Tensor:
    """bf16 x [M, K] with exactly one nonzero element in every 16-element block of every
    row, at a uniform position, with a value drawn uniformly from +-{0.5, 1, 2, 4}.  With
    such x every block of K adds a nonzero term to each output, and the exact result of
    a small sum of such terms is representable in fp32 (the exact-parity tests)."""
    rng = np.random.default_rng(seed)
    nb = K // 16
    x = np.zeros((M, nb, 16), dtype=np.float32)
    pos = rng.integers(0, 16, (M, nb))
    val = rng.choice(np.array([0.5, 1.0, 2.0, 4.0], dtype=np.float32), (M, nb))
    val *= np.where(rng.integers(0, 2, (M, nb)) == 1, -1.0, 1.0).astype(np.float32)
    np.put_along_axis(x, pos[:, :, None], val[:, :, None], axis=2)
    return torch.from_numpy(x.reshape(M, K)).to(torch.bfloat16)


def structured_nvfp4_weights(N: int, K: int, seed: int):
    """Already-encoded NVFP4 weights for the exact-parity tests: every nibble a nonzero
    code (magnitude bits 1..7, either sign), scale bytes drawn uniformly from the E4M3
    encodings of 0.5, 0.75, 1 and 2 (0x30, 0x34, 0x38, 0x40), global scale 2^-5.
    Returns (packed uint8 [N, K/2], scales uint8 [N, K/16] row-major, global scale)."""
    rng = np.random.default_rng(seed)
    mag = rng.integers(1, 8, (N, K), dtype=np.uint8)
    sign = rng.integers(0, 2, (N, K), dtype=np.uint8) << 3
    nib = mag | sign
    packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    scales = rng.choice(np.array([0x30, 0x34, 0x38, 0x40], dtype=np.uint8), (N, K // 16))
    return packed, scales, 2.0 ** -5


def random_w(N: int, K: int, seed: int, std: float = 0.02) -> torch.Tensor:
    gen = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randn(N, K, generator=gen, dtype=torch.float32) * std
