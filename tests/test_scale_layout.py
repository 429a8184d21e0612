"""Pins for the 128x4-swizzled scale layout used as a repack input (oracle/scale_layout):
a permutation of the expert's scale bytes, equal to an independent reshape/transpose
statement of the same tiling, local to 128x4 tiles, and inverted by unswizzle."""

import numpy as np
import pytest

from oracle import scale_layout


@pytest.mark.parametrize("N,C", [(128, 4), (256, 8), (384, 448), (7168, 128)])
def test_offsets_are_a_permutation(N, C):
    off = scale_layout.swizzled_offsets(N, C).reshape(-1)
    assert np.array_equal(np.sort(off), np.arange(N * C))


@pytest.mark.parametrize("N,C", [(128, 4), (256, 16), (640, 448)])
def test_matches_reshape_transpose_statement(N, C):
    """The same tiling written with reshapes: rows split as (tile, line group g, line i)
    with r = 128 t + 32 g + i, columns as (tile u, j) with c = 4 u + j; bytes ordered
    (t, u, i, g, j)."""
    rng = np.random.default_rng(N + C)
    plain = rng.integers(0, 256, size=(3, N, C), dtype=np.uint8)
    t = plain.reshape(3, N // 128, 4, 32, C // 4, 4)        # e, t, g, i, u, j
    want = t.transpose(0, 1, 4, 3, 2, 5).reshape(3, N * C)  # e, t, u, i, g, j
    assert np.array_equal(scale_layout.swizzle_128x4(plain), want)


def test_tiles_are_local_and_inverse_round_trips():
    rng = np.random.default_rng(5)
    N, C = 384, 24
    plain = rng.integers(0, 256, size=(2, N, C), dtype=np.uint8)
    swz = scale_layout.swizzle_128x4(plain)
    for t in range(N // 128):
        for u in range(C // 4):
            blk = swz[:, ((t * (C // 4)) + u) * 512:((t * (C // 4)) + u + 1) * 512]
            tile = plain[:, 128 * t:128 * (t + 1), 4 * u:4 * (u + 1)]
            assert np.array_equal(np.sort(blk, axis=1), np.sort(tile.reshape(2, -1), axis=1))
    assert np.array_equal(scale_layout.unswizzle_128x4(swz, N, C), plain)
    # a row's four scales of one tile are four consecutive bytes
    r, u = 77, 3
    o = scale_layout.swizzled_offsets(N, C)
    assert list(o[r, 4 * u:4 * u + 4]) == list(range(o[r, 4 * u], o[r, 4 * u] + 4))


def test_bad_shapes_rejected():
    with pytest.raises(ValueError):
        scale_layout.swizzled_offsets(100, 8)
    with pytest.raises(ValueError):
        scale_layout.swizzled_offsets(128, 6)


def test_packed_u32_word_holds_four_consecutive_blocks():
    """uint32-packed scales (tilelang_kernels.py page, grouped_gemm_fp4_packed_sf), read
    as: scale of K block 4g + j in bits 8j..8j+7 of word g."""
    plain = np.array([[[0x38, 0x40, 0x01, 0x7E, 0x00, 0x08, 0x30, 0x48]]], np.uint8)
    words = scale_layout.pack_u32(plain)
    assert words.shape == (1, 1, 2) and words.dtype == np.uint32
    assert int(words[0, 0, 0]) == 0x7E014038 and int(words[0, 0, 1]) == 0x48300800
    # the same bytes as a little-endian uint32 view of the plain scales
    assert np.array_equal(words, plain.view("<u4"))


def test_packed_u32_round_trip():
    rng = np.random.default_rng(9)
    plain = rng.integers(0, 256, size=(2, 256, 64), dtype=np.uint8)
    assert np.array_equal(scale_layout.unpack_u32(scale_layout.pack_u32(plain)), plain)
    with pytest.raises(ValueError):
        scale_layout.pack_u32(plain[:, :, :6])
