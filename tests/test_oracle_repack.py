"""Pins of the oracle's swizzled scale layout.

The layout starts with the tensor-core block-scale layout for 16-element blocks: atoms of
128 rows x 4 scale columns stored as 512 contiguous bytes, 32 lines of 16 bytes, line
i holding rows i, i+32, i+64, i+96 (4 bytes each, one per scale column); atoms follow
each other along K first, then along rows; a plain row-major copy of the scales follows
(for the GEMV).  The offsets below are worked out by hand from that description.  The GPU W4A4 tensor-core result is the second pin: it reads
scales in this layout.
"""
import numpy as np

import oracle


def test_hand_derived_offsets():
    cols = 128  # 8 scale columns -> 2 atoms along K
    cases = {
        (0, 0): 0, (0, 1): 1, (0, 3): 3, (1, 0): 16, (31, 0): 496,
        (32, 0): 4, (33, 2): 22, (64, 0): 8, (96, 3): 15, (127, 3): 511,
        (0, 4): 512, (5, 6): 512 + 80 + 2, (128, 0): 1024, (160, 5): 1024 + 512 + 4 + 1,
    }
    for (r, cb), off in cases.items():
        assert oracle.swizzle_offset(r, cb, cols) == off, (r, cb)


def test_sizes_and_padding():
    # atom part: rows padded to 128, blocks to 4
    assert oracle.repack_atom_bytes(128, 64) == 512
    assert oracle.repack_atom_bytes(1, 16) == 512          # 1 row, 1 block -> one atom
    assert oracle.repack_atom_bytes(129, 80) == 256 * 8    # 5 blocks pad to 8
    assert oracle.repack_atom_bytes(17408, 5120) == 17408 * 320
    # then the row-major copy, padded to 16 bytes, plus 16 bytes
    assert oracle.repack_bytes(128, 64) == 512 + 512 + 16
    assert oracle.repack_bytes(1, 16) == 512 + 16 + 16
    assert oracle.repack_bytes(129, 80) == 2048 + 656 + 16   # 645 -> 656
    assert oracle.repack_bytes(17408, 5120) == 2 * 17408 * 320 + 16


def test_bijection_and_zero_padding():
    rng = np.random.default_rng(3)
    for rows, cols in [(1, 16), (7, 48), (130, 80), (256, 512), (300, 1040)]:
        s = rng.integers(1, 127, size=(rows, cols // 16), dtype=np.uint8)
        out = oracle.repack(s, cols)
        assert out.size == oracle.repack_bytes(rows, cols)
        offs = np.array([[oracle.swizzle_offset(r, c, cols) for c in range(cols // 16)]
                         for r in range(rows)])
        assert len(np.unique(offs)) == offs.size      # injective
        np.testing.assert_array_equal(out[offs], s)   # the inverse recovers the scales
        atom = oracle.repack_atom_bytes(rows, cols)
        assert offs.max() < atom
        # the row-major copy follows the atom part
        np.testing.assert_array_equal(out[atom:atom + s.size].reshape(s.shape), s)
        mask = np.ones(out.size, dtype=bool)
        mask[offs.ravel()] = False
        mask[atom:atom + s.size] = False
        assert not out[mask].any()                    # padding is zero


def test_row_scales_are_contiguous_by_four():
    # one row's 4 consecutive scale columns of an atom are 4 adjacent bytes
    cols = 256
    for r in (0, 37, 99, 200):
        for cb in (0, 4, 8, 12):
            base = oracle.swizzle_offset(r, cb, cols)
            assert [oracle.swizzle_offset(r, cb + j, cols) for j in range(4)] == \
                [base + j for j in range(4)]
