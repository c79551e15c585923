"""Guard bytes around every output and workspace (a stand-in for a memory checker).

Each output buffer is carved out of a larger allocation with 4 KiB of a fill pattern
before and after it; the workspace gets a guard past its documented size.  After the
call every guard byte must be unchanged, and the inputs must be unchanged too.  The
shapes are ragged (M, N not multiples of the tiles; K = 32 mod 64, which leaves partial
scale atoms) and cover every dispatch path, so a store or a TMA write that strays past a
tile edge, a padded scale atom or the workspace's end shows up here.
"""
import numpy as np
import pytest
import torch

import nvfp4_weight_quantized_quantize_gb300 as nv
import oracle
from helpers import to_dev, upload_weights, w4a4_kernel
from synth import make_inputs, random_gate_up, random_nvfp4_weights, random_x

pytestmark = pytest.mark.gpu

GUARD = 4096
FILL = 0xA5


class Guarded:
    """A tensor of `nbytes` bytes with GUARD bytes of FILL on both sides."""

    def __init__(self, nbytes: int):
        self.nbytes = nbytes
        self.buf = torch.full((GUARD + nbytes + GUARD,), FILL, dtype=torch.uint8,
                              device="cuda")

    def view(self, dtype, shape):
        t = self.buf[GUARD:GUARD + self.nbytes]
        return t.view(dtype).view(*shape)

    def check(self, what: str):
        b = self.buf.cpu().numpy()
        head, tail = b[:GUARD], b[GUARD + self.nbytes:]
        bad_h = np.nonzero(head != FILL)[0]
        bad_t = np.nonzero(tail != FILL)[0]
        assert bad_h.size == 0, "%s: %d guard bytes before the buffer written" % (what, bad_h.size)
        assert bad_t.size == 0, "%s: %d guard bytes after the buffer written (first at +%d)" % (
            what, bad_t.size, int(bad_t[0]))


def guarded(shape, dtype):
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    g = Guarded(n)
    return g, g.view(dtype, shape)


@pytest.mark.parametrize("M,K,N,mode", [
    (1, 5120, 17411, "w4a16"), (1, 17408, 5121, "w4a16"), (1, 1056, 333, "w4a16"),
    (3, 5152, 1001, "w4a16"), (8, 2080, 129, "w4a16"), (5, 17440, 301, "w4a16"),
    (13, 1056, 257, "w4a16"), (16, 17408, 199, "w4a16"), (17, 1056, 300, "w4a16"),
    (300, 2080, 257, "w4a16"), (40, 1056, 129, "w4a4"), (300, 5152, 641, "w4a4"),
    (3, 1056, 77, "w4a4"), (12, 2080, 300, "w4a4"), (300, 5152, 641, "w4a4-pair"),
    (40, 1056, 129, "w4a4-pair"), (520, 2080, 1300, "w4a4"), (520, 2080, 1300, "w4a4-pair"),
    (700, 1056, 1500, "w4a4-pair"), (1, 2080, 300, "w4a4"), (1, 17408, 301, "w4a4"),
    (5, 2080, 300, "w4a4"), (8, 1056, 129, "w4a4"),
])
def test_linear_writes_only_its_outputs(M, K, N, mode):
    kernel = mode.split("-")[1] if "-" in mode else "auto"
    mode = mode.split("-")[0]
    x = random_x(M, K, seed=M * 7 + K)
    wq, ws, gw = random_nvfp4_weights(N, K, seed=N)
    d_wq, d_swz, d_g = upload_weights(wq, ws, gw, K)
    d_x = x.cuda()
    x_before = d_x.clone()
    gy, y = guarded((M, N), torch.bfloat16 if M % 2 else torch.float32)
    m = nv.NVFP4_W4A4 if mode == "w4a4" else nv.NVFP4_W4A16
    wsb = nv.nvfp4_workspace_bytes(1, M, K, N, m)
    gw_, work = guarded((wsb,), torch.uint8)
    work.zero_()
    with w4a4_kernel(kernel):
        nv.nvfp4_linear(d_x, d_wq, d_swz, d_g, y, mode=mode, workspace=work,
                        static_weights=(N % 2 == 1))
    torch.cuda.synchronize()
    assert nv.nvfp4_workspace_error(work) == 0
    gy.check("y")
    gw_.check("workspace")
    assert torch.equal(d_x, x_before), "x was written"


@pytest.mark.parametrize("rows,cols,bf16", [(129, 80, False), (1000, 1040, True),
                                            (7, 5136, False)])
def test_quantize_and_repack_write_only_their_outputs(rows, cols, bf16):
    _, w = make_inputs(1, cols, rows, seed=rows)
    src = (w.to(torch.bfloat16) if bf16 else w).cuda()
    gp, packed = guarded((rows, cols // 2), torch.uint8)
    gs, scales = guarded((rows, cols // 16), torch.uint8)
    gg, g = guarded((1,), torch.float32)
    gws, ws = guarded((nv.nvfp4_workspace_bytes(0, rows, cols),), torch.uint8)
    nv.nvfp4_quantize(src, packed, scales, g, ws)
    gz, swz = guarded((nv.nvfp4_repack_bytes(rows, cols),), torch.uint8)
    nv.nvfp4_repack(scales, cols, swz)
    torch.cuda.synchronize()
    for gd, what in ((gp, "packed"), (gs, "scales"), (gg, "global scale"), (gws, "workspace"),
                     (gz, "swizzled scales")):
        gd.check(what)
    po, so, go = oracle.quantize(src.cpu() if bf16 else src.cpu().numpy())
    assert np.array_equal(packed.cpu().numpy(), po)


@pytest.mark.parametrize("M,I,static", [(5, 1040, False), (130, 2064, True)])
def test_silu_mul_quantize_writes_only_its_outputs(M, I, static):
    gu = random_gate_up(M, I, 3).cuda()
    gq, hq = guarded((M, I // 2), torch.uint8)
    gs, hs = guarded((oracle.repack_atom_bytes(M, I),), torch.uint8)
    gg, hg = guarded((1,), torch.float32)
    given = torch.tensor([0.01], device="cuda") if static else None
    gws, ws = guarded((nv.nvfp4_workspace_bytes(0, M, I),), torch.uint8)
    nv.nvfp4_silu_mul_quantize(gu, hq, hs, hg, given, ws)
    torch.cuda.synchronize()
    for gd, what in ((gq, "codes"), (gs, "scale atoms"), (gg, "global scale"), (gws, "workspace")):
        gd.check(what)


@pytest.mark.parametrize("M,K,I", [(40, 1056, 256), (300, 2080, 384), (5, 1056, 256),
                                   (40, 1056, 96)])
def test_fused_gate_up_writes_only_its_outputs(M, K, I):
    x = random_x(M, K, seed=M + I)
    wq, ws, gw = random_nvfp4_weights(2 * I, K, seed=I)
    d_wq, d_swz, d_g = upload_weights(wq, ws, gw, K)
    gq, hq = guarded((M, I // 2), torch.uint8)
    gs, hs = guarded((oracle.repack_atom_bytes(M, I),), torch.uint8)
    gws, work = guarded((nv.nvfp4_workspace_bytes(2, M, K, I),), torch.uint8)
    work.zero_()
    gh = torch.tensor([0.002], device="cuda")
    nv.nvfp4_linear_silu_mul_quantize(x.cuda(), d_wq, d_swz, d_g, gh, hq, hs, work)
    torch.cuda.synchronize()
    assert nv.nvfp4_workspace_error(work) == 0
    for gd, what in ((gq, "codes"), (gs, "scale atoms"), (gws, "workspace")):
        gd.check(what)


@pytest.mark.parametrize("M,K,N", [(1, 1056, 300), (40, 2080, 257)])
def test_linear_nvfp4_x_writes_only_its_outputs(M, K, N):
    xq, xs, gx = oracle.silu_mul_quantize(random_gate_up(M, K, 4))
    wq, ws, gw = random_nvfp4_weights(N, K, seed=5)
    d_wq, d_swz, d_g = upload_weights(wq, ws, gw, K)
    d_xs = to_dev(oracle.repack(xs, K)[:oracle.repack_atom_bytes(M, K)].copy())
    gy, y = guarded((M, N), torch.float32)
    gws, work = guarded((nv.nvfp4_workspace_bytes(1, M, K, N, nv.NVFP4_W4A4),), torch.uint8)
    work.zero_()
    nv.nvfp4_linear_nvfp4_x(to_dev(xq), d_xs, torch.tensor([gx], device="cuda"), d_wq, d_swz,
                            d_g, y, work)
    torch.cuda.synchronize()
    assert nv.nvfp4_workspace_error(work) == 0
    gy.check("y")
    gws.check("workspace")
