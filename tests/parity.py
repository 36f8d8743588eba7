"""Comparison helpers of the parity tests (CUDA path vs oracle)."""
from __future__ import annotations

import numpy as np
import torch

E2M1_MAG = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)


def np_u8(t: torch.Tensor, n: int | None = None) -> np.ndarray:
    a = t.detach().cpu().numpy().view(np.uint8).reshape(-1)
    return a if n is None else a[:n]


def np_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def e4m3_value(codes: np.ndarray) -> np.ndarray:
    c = codes.astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    v = np.where(e == 0, m * 2.0 ** -9, (8 + m) * np.ldexp(1.0, e - 10))
    return s * v


def e2m1_value(nib: np.ndarray) -> np.ndarray:
    n = nib.astype(np.int64)
    return np.where(n & 8, -1.0, 1.0) * E2M1_MAG[n & 7]


def mx_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """codes [R, C], compact E8M0 scales [R, C/32]."""
    return e4m3_value(codes) * np.ldexp(1.0, scales.astype(np.int64) - 127).repeat(32, axis=1)


def nv_dequant(codes: np.ndarray, scales: np.ndarray, S) -> np.ndarray:
    """codes [R, C/2] packed, compact E4M3 scales [R, C/16], S per row [R]."""
    nib = np.stack([codes & 15, codes >> 4], axis=-1).reshape(codes.shape[0], -1)
    sf = e4m3_value(scales).repeat(16, axis=1)
    return e2m1_value(nib) * sf / np.asarray(S, np.float64).reshape(-1, 1)


def nvfp4_scale_of(amax) -> np.float32:
    """The FP32 global scale a GPU-side amax implies (448 * 6 / amax, 1 for a zero
    amax, FLT_MAX past the range), to dequantise the CUDA path's NVFP4 codes with
    its own scale; the oracle's scales come from the oracle alone."""
    a = np.float32(amax)
    if a == 0:
        return np.float32(1.0)
    with np.errstate(over="ignore", divide="ignore"):
        S = np.float32(2688.0) / a
    return np.float32(np.finfo(np.float32).max) if np.isinf(S) else np.float32(S)


def code_match_report(fmt: int, g_codes, o_codes, g_scales, o_scales, g_S=None, o_S=None, rows=None):
    """Fraction of identical codes, and the largest distance of a mismatched
    value in code steps at the coarser of the two block scales (c18 reading:
    blocks whose scale differs count as mismatched)."""
    if rows is not None:
        g_codes, o_codes, g_scales, o_scales = g_codes[rows], o_codes[rows], g_scales[rows], o_scales[rows]
        if g_S is not None:
            g_S, o_S = g_S[rows], o_S[rows]
    if fmt == 0:
        same = (g_codes == o_codes) & (g_scales.repeat(32, axis=1) == o_scales.repeat(32, axis=1))
        dg, do = mx_dequant(g_codes, g_scales), mx_dequant(o_codes, o_scales)
        emax = np.maximum(g_scales, o_scales).astype(np.int64).repeat(32, axis=1) - 127
        mag = np.maximum(np.abs(dg), np.abs(do))
        binade = np.floor(np.log2(np.maximum(mag, 1e-300) / np.ldexp(1.0, emax)))
        step = np.ldexp(1.0, emax + np.maximum(binade, -6).astype(np.int64) - 3)
    else:
        gn = np.stack([g_codes & 15, g_codes >> 4], axis=-1).reshape(g_codes.shape[0], -1)
        on = np.stack([o_codes & 15, o_codes >> 4], axis=-1).reshape(o_codes.shape[0], -1)
        same = (gn == on) & (g_scales.repeat(16, axis=1) == o_scales.repeat(16, axis=1))
        dg, do = nv_dequant(g_codes, g_scales, g_S), nv_dequant(o_codes, o_scales, o_S)
        unit = np.maximum(e4m3_value(g_scales), e4m3_value(o_scales)).repeat(16, axis=1) / \
            np.asarray(o_S, np.float64).reshape(-1, 1)
        mag = np.maximum(np.abs(dg), np.abs(do)) / np.maximum(unit, 1e-300)
        step = np.where(mag < 2, 0.5, np.where(mag < 4, 1.0, 2.0)) * unit
    frac = float(same.mean()) if same.size else 1.0
    diff = np.abs(dg - do)[~same]
    steps = float((diff / step[~same]).max()) if diff.size else 0.0
    return frac, steps


def frob(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    n = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (n if n > 0 else 1.0))
