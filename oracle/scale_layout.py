"""Layouts of NVFP4 block scales accepted as repack inputs (test infrastructure).

TEST INFRASTRUCTURE ONLY: used by the tests to produce and check swizzled inputs;
the CUDA path never imports it.

Layout (megamoe_rm.cu page, scale_off: "128x4 swizzle within one expert", the order
FlashInfer's CUTLASS backend keeps NVFP4 block scales in): per expert, the [N][C]
scale matrix (N rows, C = K/16 scales per row; N % 128 == 0, C % 4 == 0) is cut into
tiles of 128 rows x 4 scales, tiles stored one after another with the 4-column index
fastest (offset of tile (r // 128, c // 4) = ((r // 128) * (C // 4) + c // 4) * 512).
Inside a 512-byte tile, the scale of row r and column c sits at
    (r % 32) * 16 + ((r // 32) % 4) * 4 + c % 4,
i.e. 32 lines of 16 bytes, line i holding rows i, i+32, i+64, i+96 (4 scales each).

uint32-packed scales (tilelang_kernels.py page, grouped_gemm_fp4_packed_sf: a
(E, N, sf_k_groups) uint32 tensor of packed UE4M3 that unpack_ue4m3_u32 turns into the
(E, N, K/16) scales): four scales per word, so sf_k_groups = K/64.  The page does not
give the byte order; the reading taken is that scale j of group g (the scale of K
block 4g + j) is bits 8j..8j+7 of word g, the order a little-endian uint32 view of the
plain scale bytes has.
"""

from __future__ import annotations

import numpy as np


def swizzled_offsets(N: int, C: int) -> np.ndarray:
    """[N][C] array: the byte offset, inside one expert's swizzled block, of the scale
    of row r and column c."""
    if N % 128 or C % 4:
        raise ValueError("the 128x4 layout needs N % 128 == 0 and C % 4 == 0")
    r = np.arange(N, dtype=np.int64)[:, None]
    c = np.arange(C, dtype=np.int64)[None, :]
    tile = (r // 128) * (C // 4) + c // 4
    return tile * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + c % 4


def swizzle_128x4(plain: np.ndarray) -> np.ndarray:
    """Plain scales [E][N][C] (uint8) -> swizzled [E][N * C]."""
    E, N, C = plain.shape
    off = swizzled_offsets(N, C)
    out = np.empty((E, N * C), dtype=plain.dtype)
    out[:, off.reshape(-1)] = plain.reshape(E, N * C)
    return out


def unswizzle_128x4(swz: np.ndarray, N: int, C: int) -> np.ndarray:
    """Swizzled scales [E][N * C] -> plain [E][N][C]."""
    E = swz.shape[0]
    off = swizzled_offsets(N, C)
    return swz.reshape(E, N * C)[:, off.reshape(-1)].reshape(E, N, C)


def pack_u32(plain: np.ndarray) -> np.ndarray:
    """Plain scales [E][N][C] (uint8, C % 4 == 0) -> packed [E][N][C/4] uint32, scale
    4g + j in bits 8j..8j+7 of word g."""
    E, N, C = plain.shape
    if C % 4:
        raise ValueError("uint32 packing needs C % 4 == 0")
    b = plain.astype(np.uint32).reshape(E, N, C // 4, 4)
    return b[..., 0] | (b[..., 1] << 8) | (b[..., 2] << 16) | (b[..., 3] << 24)


def unpack_u32(words: np.ndarray) -> np.ndarray:
    """Packed [E][N][G] uint32 -> plain scales [E][N][4G] uint8."""
    w = words.astype(np.uint32)
    parts = [(w >> (8 * j)) & 0xFF for j in range(4)]
    return np.stack(parts, axis=-1).reshape(*w.shape[:-1], 4 * w.shape[-1]).astype(np.uint8)
