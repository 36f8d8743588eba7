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


def test_x4_image_feeds_each_b_row_its_scales(orc):
    """GEMM_TILED_X4 checked through what the GEMM does with it: a 128-row x
    32-byte tensor-memory copy (lane L <- row L; row L = 16 bytes at 16 L and 16
    bytes at 2048 + 16 L) of each 4096-byte unit, then the MMA reading B row n
    (half h = n // 128, r = n % 128) at lane r % 32, column 4 h + r // 32, byte
    j.  Every B row must see its own compact scales, and the four lane quarters
    must hold the same bytes."""
    rng = np.random.default_rng(3)
    G, rows, cols = 2, 512, 512                       # NVFP4: 32 scale columns per row
    ks = cols // 16
    compact = rng.integers(0, 256, (G * rows, ks), dtype=np.uint8)
    splits = np.full(G, rows)
    tiled = orc.compact_to_tiled(compact, splits, ks)
    runs, KB = ks // 4, ks // 16
    x4 = orc.tiled_to_x4(tiled, G * rows // 256, runs)
    assert x4.size == 4 * G * rows * ks
    for P in range(G * rows // 256):
        for kb in range(KB):
            for k in range(4):
                unit = x4[((P * KB + kb) * 4 + k) * 4096:][:4096]
                lanes = np.stack([np.concatenate([unit[16 * L:16 * L + 16], unit[2048 + 16 * L:2048 + 16 * L + 16]])
                                  for L in range(128)])          # [128 lanes, 32 bytes = 8 columns]
                assert np.array_equal(lanes[:32], lanes[32:64]) and np.array_equal(lanes[:32], lanes[96:])
                for n in range(256):
                    h, r = divmod(n, 128)
                    col = 4 * h + r // 32
                    got = lanes[r % 32, 4 * col:4 * col + 4]
                    want = compact[256 * P + n, (4 * kb + k) * 4:(4 * kb + k) * 4 + 4]
                    assert np.array_equal(got, want), (P, kb, k, n)
