"""Pins of the boundary's GEMM_TILED scale layout as the oracle states it (CPU only).

Expected offsets are worked by hand from the layout's definition (a 512-byte
block per 128-row tile and run of 4 scale columns; byte (r%32)*16 + (r/32)*4 + j
inside the block; groups start on fresh tiles)."""
import numpy as np


def test_tiled_offsets_worked_example(orc):
    splits = [130, 5]          # group 0: tiles 0, 1 ; group 1: tile 2
    ks = 8                     # two runs of 4 scale columns per row -> 2 blocks per tile
    idx = orc.tiled_index(splits, ks)
    assert idx[0, 0] == 0
    assert idx[1, 0] == 16
    assert idx[32, 0] == 4
    assert idx[33, 3] == 16 + 4 + 3
    assert idx[0, 1] == 1
    assert idx[0, 4] == 512
    assert idx[127, 7] == 512 + 31 * 16 + 3 * 4 + 3
    assert idx[128, 0] == 1024          # group 0, tile 1
    assert idx[130, 0] == 2048          # group 1 starts on tile 2
    assert idx[134, 5] == 2048 + 512 + 4 * 16 + 1


def test_tiled_is_injective_and_bounded(orc):
    rng = np.random.default_rng(0)
    for _ in range(20):
        G = int(rng.integers(1, 9))
        splits = rng.integers(0, 300, G)
        ks = 4 * int(rng.integers(1, 6))
        idx = orc.tiled_index(splits, ks)
        assert len(np.unique(idx)) == idx.size
        if idx.size:
            assert idx.max() < orc.tiled_size(int(np.sum(splits)), ks, G)
        sc = rng.integers(0, 256, (int(np.sum(splits)), ks)).astype(np.uint8)
        assert np.array_equal(orc.tiled_to_compact(orc.compact_to_tiled(sc, splits, ks), splits, ks), sc)
