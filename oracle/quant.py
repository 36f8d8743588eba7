"""Group quantisers of the oracle (TEST INFRASTRUCTURE; see oracle/__init__.py).

Each function states the passage it restates.  All arithmetic is in
``formats.c``; this module only slices groups and calls it.
"""
from __future__ import annotations

import numpy as np

from ._lib import lib, ptr
from .layout import group_offsets

MXFP8, NVFP4 = 0, 1


def _u16(x) -> np.ndarray:
    a = np.ascontiguousarray(x)
    if a.dtype != np.uint16:
        a = a.view(np.uint16) if a.dtype.itemsize == 2 else a.astype(np.uint16)
    return a


def bf16_to_f64(x) -> np.ndarray:
    x = _u16(x)
    out = np.empty(x.shape, dtype=np.float64)
    lib().orc_bf16_to_double_array(ptr(x), x.size, ptr(out))
    return out


def f64_to_bf16(v) -> np.ndarray:
    """Round-to-nearest-even bf16 of float64 values (bit patterns as uint16)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().orc_bf16_from_double_array(ptr(v), v.size, ptr(out))
    return out


# ---------------------------------------------------------------- MXFP8

def mxfp8_quantize_rows(x) -> tuple[np.ndarray, np.ndarray]:
    """Rowwise MXFP8 (PR #2769, ``a_tensor`` "MXFP8"): 1x32 blocks along the
    row, E8M0 scale 2^(floor(log2 amax) - 8), E4M3 codes.
    Returns (codes [rows, K] u8, compact scales [rows, K/32] u8)."""
    x = _u16(x)
    rows, K = x.shape
    assert K % 32 == 0
    codes = np.empty((rows, K), dtype=np.uint8)
    scales = np.empty((rows, K // 32), dtype=np.uint8)
    lib().orc_mxfp8_quantize_rows(ptr(x), rows, K, ptr(codes), ptr(scales))
    return codes, scales


def mxfp8_dequant_rows(codes, scales) -> np.ndarray:
    codes, scales = np.ascontiguousarray(codes), np.ascontiguousarray(scales)
    rows, K = codes.shape
    out = np.empty((rows, K), dtype=np.float64)
    lib().orc_mxfp8_dequant_rows(ptr(codes), ptr(scales), rows, K, ptr(out))
    return out


# ---------------------------------------------------------------- NVFP4

def nvfp4_global_scale(amax) -> np.float32:
    """FP32 encode scale from amax (method statement: "FP32 global scale from amax")."""
    return np.float32(lib().orc_nvfp4_global_scale(float(np.float32(amax))))


def nvfp4_quantize_block(v, S) -> tuple[np.ndarray, int]:
    v = np.ascontiguousarray(v, dtype=np.float32)
    assert v.shape == (16,)
    codes = np.empty(8, dtype=np.uint8)
    sf = np.empty(1, dtype=np.uint8)
    lib().orc_nvfp4_quantize_block(ptr(v), float(S), ptr(codes), ptr(sf))
    return codes, int(sf[0])


def nvfp4_quantize_rows(x, S) -> tuple[np.ndarray, np.ndarray]:
    """Rowwise NVFP4 under one FP32 global scale S: 1x16 blocks, E4M3 block
    scales, E2M1 codes packed low nibble first.  Returns (codes [rows, K/2],
    compact scales [rows, K/16])."""
    x = _u16(x)
    rows, K = x.shape
    assert K % 16 == 0
    codes = np.empty((rows, K // 2), dtype=np.uint8)
    scales = np.empty((rows, K // 16), dtype=np.uint8)
    lib().orc_nvfp4_quantize_rows(ptr(x), rows, K, float(S), ptr(codes), ptr(scales))
    return codes, scales


def nvfp4_dequant_rows(codes, scales, S) -> np.ndarray:
    codes, scales = np.ascontiguousarray(codes), np.ascontiguousarray(scales)
    rows = codes.shape[0]
    K = codes.shape[1] * 2
    out = np.empty((rows, K), dtype=np.float64)
    lib().orc_nvfp4_dequant_rows(ptr(codes), ptr(scales), rows, K, float(S), ptr(out))
    return out


def rht16(v, mask: int) -> np.ndarray:
    """16-point randomized Hadamard transform (PR #3837, commit "pass the RHT
    sign mask to the Hadamard-fused kernel"): 1/4 * H16 * diag(s) * v in FP32."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    assert v.shape == (16,)
    out = np.empty(16, dtype=np.float32)
    lib().orc_rht16(ptr(v), int(mask) & 0xFFFF, ptr(out))
    return out


def amax_bf16(x) -> np.float32:
    x = _u16(x)
    return np.float32(lib().orc_amax_bf16(ptr(x), x.size))


def group_amax(x, splits) -> np.ndarray:
    """Per-group max |x| (the pre-RHT amax)."""
    x = _u16(x)
    offs = group_offsets(splits)
    return np.array([amax_bf16(x[offs[g]:offs[g + 1]]) for g in range(len(splits))], dtype=np.float32)


def group_hadamard_amax(x, splits, mask: int) -> tuple[np.ndarray, np.ndarray]:
    """``nvfp4_group_hadamard_amax`` (PR #3837, Changes: one pass returning the
    per-group pre-RHT and post-RHT amax; the sign mask enters the post-RHT
    amax).  The post-RHT amax runs over 16-row column chunks counted from each
    group's first row, zero-padded at the group's end."""
    x = _u16(x)
    M, K = x.shape
    s = np.ascontiguousarray(splits, dtype=np.int64)
    assert int(s.sum()) == M
    pre = np.empty(len(s), dtype=np.float32)
    post = np.empty(len(s), dtype=np.float32)
    lib().orc_group_hadamard_amax(ptr(x), M, K, ptr(s), len(s), int(mask) & 0xFFFF, ptr(pre), ptr(post))
    return pre, post


def group_quantize_with_amax(x, splits, fmt: int, amax_pre=None, amax_post=None, *, rowwise=True,
                             columnwise=False, use_rht=True, mask: int = 0) -> dict:
    """``nvfp4_group_quantize_with_amax`` (PR #3837: the cast alone, with the
    amaxes supplied by the caller).  Rowwise NVFP4 takes S_g from amax_pre;
    columnwise NVFP4 takes S_g from amax_post when the RHT is applied, else from
    amax_pre.  MXFP8 needs no amax (scales are block-local) and is rowwise only.

    Returns compact outputs: row_codes [M, K] (MX) / [M, K/2] (NV), row_scales
    [M, K/32 | K/16], and for columnwise NVFP4 the concatenated per-group
    col_codes [K, Mpad_g/2] and col_scales [K, Mpad_g/16]."""
    x = _u16(x)
    M, K = x.shape
    offs = group_offsets(splits)
    G = len(splits)
    out: dict = {}
    if fmt == MXFP8:
        assert not columnwise, "columnwise MXFP8 is not part of this path"
        if rowwise:
            out["row_codes"], out["row_scales"] = mxfp8_quantize_rows(x)
        return out
    amax_pre = np.asarray(amax_pre, dtype=np.float32)
    if rowwise:
        codes = np.empty((M, K // 2), dtype=np.uint8)
        scales = np.empty((M, K // 16), dtype=np.uint8)
        S = np.empty(G, dtype=np.float32)
        for g in range(G):
            S[g] = nvfp4_global_scale(amax_pre[g])
            if offs[g + 1] > offs[g]:
                codes[offs[g]:offs[g + 1]], scales[offs[g]:offs[g + 1]] = nvfp4_quantize_rows(
                    x[offs[g]:offs[g + 1]], S[g])
        out.update(row_codes=codes, row_scales=scales, row_S=S)
    if columnwise:
        amax_col = np.asarray(amax_post if use_rht else amax_pre, dtype=np.float32)
        s = np.ascontiguousarray(splits, dtype=np.int64)
        mpad = (s + 15) // 16 * 16
        col_codes = np.empty(int(K * mpad.sum() // 2), dtype=np.uint8)
        col_scales = np.empty(int(K * mpad.sum() // 16), dtype=np.uint8)
        lib().orc_group_quantize_col(ptr(x), M, K, ptr(s), G, int(bool(use_rht)), int(mask) & 0xFFFF,
                                     ptr(np.ascontiguousarray(amax_col)), ptr(col_codes), ptr(col_scales))
        out.update(col_codes=col_codes, col_scales=col_scales,
                   col_S=np.array([nvfp4_global_scale(a) for a in amax_col], dtype=np.float32))
    return out


def group_quantize(x, splits, fmt: int, *, rowwise=True, columnwise=False, use_rht=True, mask: int = 0) -> dict:
    """Generic group quantise (PR #3837, Description: the fc2-input group quantize
    with row- and/or column-wise output).  NVFP4 first takes the per-group amax
    pair, then casts with it."""
    out: dict = {}
    pre = post = None
    if fmt == NVFP4:
        if columnwise and use_rht:
            pre, post = group_hadamard_amax(x, splits, mask)
        else:
            pre = group_amax(x, splits)
        out["amax_pre"] = pre
        if post is not None:
            out["amax_post"] = post
    out.update(group_quantize_with_amax(x, splits, fmt, pre, post, rowwise=rowwise, columnwise=columnwise,
                                        use_rht=use_rht, mask=mask))
    return out
