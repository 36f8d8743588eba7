"""Fused grouped-MLP forward of the oracle (TEST INFRASTRUCTURE; see oracle/__init__.py).

Restates, step by step, the forward of the fused grouped MLP for MoE layers:
PR #2769 "GEMM + Swiglu fused Grouped MLP for MXFP8" (sequence diagram: FC1
GLU kernel on the MXFP8 ``a_tensor`` with ``b_tensor`` weights and the
``prob_tensor`` scales, writing the MXFP8 activation; then the FC2 kernel) and
PR #3837 (flowchart: FC1 and activation -> fc2 input and amax -> row-wise
NVFP4 quantization -> FC2 forward).  The GEMMs are float64 matrix products of
the dequantised operands (a library primitive); every other step is a call
into the format arithmetic of formats.c.
"""
from __future__ import annotations

import numpy as np

from .layout import group_offsets
from .quant import (MXFP8, NVFP4, amax_bf16, bf16_to_f64, f64_to_bf16, group_hadamard_amax,
                    mxfp8_dequant_rows, mxfp8_quantize_rows, nvfp4_dequant_rows, nvfp4_global_scale,
                    nvfp4_quantize_rows)

SWIGLU, SRELU, TANH_SRELU = 0, 1, 2


def quantize_weights(W, fmt: int) -> dict:
    """Per-expert rowwise quantisation of stacked weights W [G, R, C] along C
    (the contraction dimension).  NVFP4 takes one global scale per expert
    from that expert's amax."""
    W = np.ascontiguousarray(W)
    G, R, C = W.shape
    if fmt == MXFP8:
        codes, scales = mxfp8_quantize_rows(W.reshape(G * R, C))
        return dict(codes=codes.reshape(G, R, C), scales=scales.reshape(G, R, C // 32), S=None)
    codes = np.empty((G, R, C // 2), dtype=np.uint8)
    scales = np.empty((G, R, C // 16), dtype=np.uint8)
    S = np.empty(G, dtype=np.float32)
    amax = np.empty(G, dtype=np.float32)
    for g in range(G):
        amax[g] = amax_bf16(W[g])
        S[g] = nvfp4_global_scale(amax[g])
        codes[g], scales[g] = nvfp4_quantize_rows(W[g], S[g])
    return dict(codes=codes, scales=scales, S=S, amax=amax)


def dequant_weight(qw: dict, g: int, fmt: int) -> np.ndarray:
    if fmt == MXFP8:
        return mxfp8_dequant_rows(qw["codes"][g], qw["scales"][g])
    return nvfp4_dequant_rows(qw["codes"][g], qw["scales"][g], qw["S"][g])


def activation(h: np.ndarray, act: int, tanh_clamp_scale: float | None = None) -> np.ndarray:
    """SwiGLU: silu(gate) * up with gate = first half of the fc1 columns, up =
    second half, silu(u) = u / (1 + exp(-u)); SReLU: max(h, 0)^2; tanh-SReLU
    (PR #3837 Changes, "ScaledTanhSReLU", the SReLU soft clamp with
    tanh_clamp_scale c; reading: the soft clamp of the SReLU output at c):
    c * tanh(max(h, 0)^2 / c).  float64."""
    if act == SWIGLU:
        n = h.shape[1] // 2
        gate, up = h[:, :n], h[:, n:]
        return gate / (1.0 + np.exp(-gate)) * up
    t = np.square(np.maximum(h, 0.0))
    if act == TANH_SRELU:
        c = float(tanh_clamp_scale)
        return c * np.tanh(t / c)
    return t


def forward(x, splits, W1, W2, probs, act: int, fmt: int, *, rows=None, qw1=None, qw2=None,
            rht_mask: int = 0, tanh_clamp_scale: float | None = None, b1=None, b2=None) -> dict:
    """Oracle forward.

    x [M, K] bf16 bits (uint16), token-sorted; splits [G]; W1 [G, N1, K] with
    N1 = 2N (SwiGLU, gate rows then up rows) or N (SReLU, tanh-SReLU); W2 [G, K, N];
    probs [M] float32 or None (= 1).

    Steps per group g (rows off_g .. off_g + m_g):
      1. xq = rowwise quantisation of x (MXFP8 blocks are row-local; NVFP4 takes
         S_x,g from the group's amax).
      2. acc = dq(xq_g) @ dq(W1q_g)^T in float64 (NVFP4's 1/S factors are part of dq).
      3. h = bf16(acc)  ("rounds the accumulator through C dtype before the activation");
         returned as ``h`` [M, N1] in logical column order, the activation input
         the backward reads (PR #2769 sequence diagram: c_tensor, swiglu_in).
      4. a = act(h) in float64; f = bf16(a * prob)  (fc2_x).
      5. fc2_x quantisation: MXFP8 rowwise; NVFP4 rowwise with S_f,g from the
         group's amax of f; the post-RHT amax of f (16-row column chunks, sign
         mask ``rht_mask``) is reported alongside.
      6. y = bf16(dq(fc2xq_g) @ dq(W2q_g)^T) in float64.
    ``b1`` [G, N1] / ``b2`` [G, K]: optional per-expert biases (bf16 values, logical
    row order) added to the float64 accumulators of steps 2 and 6 before their
    bf16 rounding (PR #2769: the FC1 kernel takes a bias).

    ``rows``: optional sorted global row indices.  MXFP8 rows are independent, so
    only those rows are evaluated (the rest of y, fc2_x and the codes are zero).
    NVFP4 needs every row of a group for its amaxes and ignores ``rows``.
    """
    x = np.ascontiguousarray(x).view(np.uint16)
    M, K = x.shape
    splits = np.asarray(splits, dtype=np.int64)
    G = len(splits)
    offs = group_offsets(splits)
    N = W2.shape[2]
    probs = np.ones(M, dtype=np.float32) if probs is None else np.asarray(probs, dtype=np.float32)
    if qw1 is None:
        qw1 = quantize_weights(W1, fmt)
    if qw2 is None:
        qw2 = quantize_weights(W2, fmt)
    sel_all = np.arange(M, dtype=np.int64) if (rows is None or fmt == NVFP4) else np.asarray(rows, np.int64)

    blk = 32 if fmt == MXFP8 else 16
    cdiv = 1 if fmt == MXFP8 else 2
    out = dict(
        y=np.zeros((M, K), dtype=np.uint16),
        fc2x=np.zeros((M, N), dtype=np.uint16),
        h=np.zeros((M, W1.shape[1]), dtype=np.uint16),
        fc2x_codes=np.zeros((M, N // cdiv), dtype=np.uint8),
        fc2x_scales=np.zeros((M, N // blk), dtype=np.uint8),
        rows=sel_all,
    )
    if fmt == NVFP4:
        out.update(x_amax=np.zeros(G, np.float32), x_S=np.zeros(G, np.float32),
                   fc2x_amax_pre=np.zeros(G, np.float32), fc2x_amax_post=np.zeros(G, np.float32),
                   fc2x_S=np.zeros(G, np.float32))

    for g in range(G):
        r0, r1 = int(offs[g]), int(offs[g + 1])
        sel = sel_all[(sel_all >= r0) & (sel_all < r1)]
        if fmt == NVFP4:
            # step 1 (NVFP4): group amax of x, S_x,g; needs every row of the group
            xa = amax_bf16(x[r0:r1]) if r1 > r0 else np.float32(0)
            Sx = nvfp4_global_scale(xa)
            out["x_amax"][g], out["x_S"][g] = xa, Sx
        if len(sel) == 0:
            if fmt == NVFP4:
                out["fc2x_S"][g] = nvfp4_global_scale(0.0)
            continue
        xs = np.ascontiguousarray(x[sel])
        if fmt == MXFP8:
            xd = mxfp8_dequant_rows(*mxfp8_quantize_rows(xs))
        else:
            xd = nvfp4_dequant_rows(*nvfp4_quantize_rows(xs, Sx), Sx)
        # step 2-4
        acc = xd @ dequant_weight(qw1, g, fmt).T
        if b1 is not None:
            acc = acc + np.asarray(b1, np.float64)[g][None, :]
        out["h"][sel] = f64_to_bf16(acc)
        h = bf16_to_f64(out["h"][sel])
        a = activation(h, act, tanh_clamp_scale)
        f = f64_to_bf16(a * probs[sel].astype(np.float64)[:, None])
        out["fc2x"][sel] = f
        # step 5
        if fmt == MXFP8:
            fq, fs = mxfp8_quantize_rows(f)
            fd = mxfp8_dequant_rows(fq, fs)
        else:
            pre, post = group_hadamard_amax(f, [len(sel)], rht_mask)
            Sf = nvfp4_global_scale(pre[0])
            out["fc2x_amax_pre"][g], out["fc2x_amax_post"][g], out["fc2x_S"][g] = pre[0], post[0], Sf
            fq, fs = nvfp4_quantize_rows(f, Sf)
            fd = nvfp4_dequant_rows(fq, fs, Sf)
        out["fc2x_codes"][sel], out["fc2x_scales"][sel] = fq, fs
        # step 6
        acc2 = fd @ dequant_weight(qw2, g, fmt).T
        if b2 is not None:
            acc2 = acc2 + np.asarray(b2, np.float64)[g][None, :]
        out["y"][sel] = f64_to_bf16(acc2)
    return out
