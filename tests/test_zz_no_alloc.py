"""nvfp4_quantize_noalloc: the quantizer for callers that cannot allocate device memory.

Such callers (runtimes that plan all device memory at start-up, code under a fixed
budget, latency-critical paths that must not wait on cudaMalloc/cudaFree) cannot pass a
workspace; this entry point keeps its scratch in a fixed array inside the library.  The
test calls it through the C ABI twice in a row -- a large tensor, then a smaller bf16
one whose first pass uses fewer scratch slots -- and checks each result against the
workspace-taking nvfp4_quantize, bit for bit (the tolerance of every quantizer test).
This file is collected last so that a run stopping at the first failure has already run
every other test.
"""
import pytest
import torch

import nvfp4_weight_quantized_quantize_gb300 as nv
from synth import random_w

pytestmark = pytest.mark.gpu


def _outputs(rows, cols):
    return (torch.empty(rows, cols // 2, dtype=torch.uint8, device="cuda"),
            torch.empty(rows, cols // 16, dtype=torch.uint8, device="cuda"),
            torch.empty(1, dtype=torch.float32, device="cuda"))


def test_noalloc_matches_workspace_quantizer_on_two_calls_in_a_row():
    from nvfp4_weight_quantized_quantize_gb300 import build_lib
    build_lib.build()
    nv.load()
    cases = [(4096, 5120, torch.float32, 21, 0.02), (40, 512, torch.bfloat16, 22, 3.0)]
    for rows, cols, dt, seed, std in cases:
        src = random_w(rows, cols, seed, std=std).to(dt).cuda()
        ref = _outputs(rows, cols)
        ws = torch.empty(nv.nvfp4_workspace_bytes(0, rows, cols), dtype=torch.uint8,
                         device="cuda")
        nv.nvfp4_quantize(src, *ref, ws)
        got = _outputs(rows, cols)
        nv.nvfp4_quantize_noalloc(src, *got)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
