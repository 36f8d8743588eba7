"""Scale-factor layouts of the boundary, restated for the oracle (TEST INFRASTRUCTURE).

Two layouts hold the 8-bit block scales of a rowwise-quantised, token-sorted
[M, K] tensor split into groups:

* COMPACT: row-major ``[M, K / block]``.
* GEMM_TILED: the layout the block-scaled tensor-core MMA reads ("swizzled
  scales", PR #2769 "GEMM + Swiglu fused Grouped MLP for MXFP8", Greptile
  summary: GroupedTensorStorage ``with_gemm_swizzled_scales`` and
  ``grouped_swizzle_for_gemm``).  Each group's rows are cut into 128-row tiles
  counted from the group's first row (the last tile padded); group g's tiles
  start at tile index ``T_g = sum_{h<g} ceil(m_h / 128)``.  The scales of one
  tile are cut into runs of 4 scale columns; each (tile, run) pair is a
  512-byte block, blocks ordered tile-major.  Inside a block, the scale of
  tile row ``rr`` and run column ``j`` sits at byte
  ``(rr % 32) * 16 + (rr // 32) * 4 + j``.

Padding rows of a tile are not part of the contract (their bytes are
unspecified), so comparisons use only the rows the groups own.
"""
from __future__ import annotations

import numpy as np


def group_offsets(splits) -> np.ndarray:
    s = np.asarray(splits, dtype=np.int64)
    return np.concatenate([[0], np.cumsum(s)]).astype(np.int64)


def tile_bases(splits) -> np.ndarray:
    s = np.asarray(splits, dtype=np.int64)
    return np.concatenate([[0], np.cumsum((s + 127) // 128)]).astype(np.int64)


def tiled_size(M: int, ks: int, G: int) -> int:
    """Bytes a GEMM_TILED buffer needs for any split of M rows into G groups."""
    tiles = (M + 127) // 128 + G
    return tiles * 128 * ks


def tiled_index(splits, ks: int) -> np.ndarray:
    """[M, ks] array of byte offsets of every owned scale in the GEMM_TILED layout."""
    assert ks % 4 == 0
    offs, tb = group_offsets(splits), tile_bases(splits)
    M = int(offs[-1])
    idx = np.empty((M, ks), dtype=np.int64)
    j = np.arange(ks, dtype=np.int64)
    for g in range(len(offs) - 1):
        lr = np.arange(offs[g + 1] - offs[g], dtype=np.int64)
        t, rr = lr // 128, lr % 128
        blk = (tb[g] + t)[:, None] * (ks // 4) + (j // 4)[None, :]
        idx[offs[g]:offs[g + 1]] = blk * 512 + ((rr % 32) * 16 + (rr // 32) * 4)[:, None] + (j % 4)[None, :]
    return idx


def tiled_to_compact(buf: np.ndarray, splits, ks: int) -> np.ndarray:
    return np.asarray(buf).reshape(-1)[tiled_index(splits, ks)]


def compact_to_tiled(scales: np.ndarray, splits, ks: int, fill: int = 0) -> np.ndarray:
    M = scales.shape[0]
    out = np.full(tiled_size(M, ks, len(splits)), fill, dtype=np.uint8)
    out[tiled_index(splits, ks)] = scales
    return out


def tiled_to_x4(buf: np.ndarray, pairs: int, runs: int) -> np.ndarray:
    """GEMM_TILED_X4 image of GEMM_TILED scales of `2 * pairs` 128-row tiles with
    `runs` runs of 4 scale columns each (runs % 4 == 0): for tile pair P, stage
    kb and run k of the stage, 4096 bytes = the block (2P, 4kb+k) four times,
    then the block (2P+1, 4kb+k) four times."""
    blocks = np.asarray(buf, np.uint8)[:2 * pairs * runs * 512].reshape(pairs, 2, runs // 4, 4, 512)
    img = np.broadcast_to(blocks.transpose(0, 2, 3, 1, 4)[:, :, :, :, None, :], (pairs, runs // 4, 4, 2, 4, 512))
    return np.ascontiguousarray(img).reshape(-1)
