"""Data-gradient half of the fused grouped-MLP backward, restated for the oracle
(TEST INFRASTRUCTURE; see oracle/__init__.py).

PR #2769 "GEMM + Swiglu fused Grouped MLP for MXFP8", sequence diagram,
backward pass: the "FC2 dGLU kernel" takes the MXFP8 output gradient dy, the
saved activation input (c_tensor, swiglu_in) and the FC2 weight quantised the
other way ("col"), and returns the fc1 output gradient (MXFP8, row scales) and
the gradient of the routing probabilities; the "FC1 dGrad kernel" returns the
input gradient.  The GEMMs are float64 products of the dequantised operands;
the accumulators are rounded through bf16 (the C dtype) as in the forward, and
fc1_dy is rounded through bf16 before its MXFP8 cast.
"""
from __future__ import annotations

import numpy as np

from .forward import SRELU, SWIGLU, activation, dequant_weight, quantize_weights
from .layout import group_offsets
from .quant import MXFP8, bf16_to_f64, f64_to_bf16, mxfp8_dequant_rows, mxfp8_quantize_rows


def dact(h: np.ndarray, act: int) -> tuple[np.ndarray, np.ndarray | None]:
    """Partial derivatives of the activation in float64.  SwiGLU (gate g =
    first half of h, up u = second half): d act / d g = u * silu'(g) with
    silu'(g) = s (1 + g (1 - s)), s = 1 / (1 + exp(-g)); d act / d u = silu(g).
    SReLU: d act / d h = 2 max(h, 0) (second result None)."""
    if act == SWIGLU:
        n = h.shape[1] // 2
        g, u = h[:, :n], h[:, n:]
        s = 1.0 / (1.0 + np.exp(-g))
        return u * s * (1.0 + g * (1.0 - s)), g * s
    return 2.0 * np.maximum(h, 0.0), None


def backward_dgrad(dy, splits, W1, W2, h, probs, act: int, *, qw1t=None, qw2t=None) -> dict:
    """Oracle of gmlp_backward_dgrad (MXFP8).

    dy [M, K] bf16 bits (gradient of y); W1 [G, N1, K] and W2 [G, K, N] bf16
    bits in logical row order (SwiGLU: gate rows then up rows); h [M, N1] bf16
    bits, the forward's activation input bf16(fc1 accumulator); probs [M] or
    None (= 1).  Per group g:
      1. dyq = rowwise MXFP8 of dy;  W2t_g = W2_g^T [N, K] quantised along K.
      2. d = bf16(dq(dyq) dq(W2t_g)^T)                              [m_g, N]
      3. fc1_dy = bf16(d p * dact(h))  (SwiGLU: [d p u silu'(g) | d p silu(g)])
         dprob = sum_n d * act(h)                                   (float64)
      4. fc1_dy -> rowwise MXFP8;  W1t_g = W1_g^T [K, N1] quantised along N1.
      5. dx = bf16(dq(fc1_dyq) dq(W1t_g)^T)                         [m_g, K]
    """
    dy = np.ascontiguousarray(dy).view(np.uint16)
    h = np.ascontiguousarray(h).view(np.uint16)
    M, K = dy.shape
    splits = np.asarray(splits, dtype=np.int64)
    G = len(splits)
    offs = group_offsets(splits)
    N1 = h.shape[1]
    N = N1 // 2 if act == SWIGLU else N1
    probs = np.ones(M, dtype=np.float64) if probs is None else np.asarray(probs, dtype=np.float64)
    if qw2t is None:
        qw2t = quantize_weights(np.ascontiguousarray(np.asarray(W2).transpose(0, 2, 1)), MXFP8)
    if qw1t is None:
        qw1t = quantize_weights(np.ascontiguousarray(np.asarray(W1).transpose(0, 2, 1)), MXFP8)
    out = dict(dfc2x=np.zeros((M, N), np.uint16), fc1_dy=np.zeros((M, N1), np.uint16),
               fc1_dy_codes=np.zeros((M, N1), np.uint8), fc1_dy_scales=np.zeros((M, N1 // 32), np.uint8),
               dprob=np.zeros(M, np.float64), dx=np.zeros((M, K), np.uint16))
    for g in range(G):
        r0, r1 = int(offs[g]), int(offs[g + 1])
        if r1 == r0:
            continue
        dq = mxfp8_dequant_rows(*mxfp8_quantize_rows(dy[r0:r1]))
        d = bf16_to_f64(f64_to_bf16(dq @ dequant_weight(qw2t, g, MXFP8).T))
        out["dfc2x"][r0:r1] = f64_to_bf16(d)
        hg = bf16_to_f64(h[r0:r1])
        p = probs[r0:r1][:, None]
        a = activation(hg, act)
        out["dprob"][r0:r1] = (d * a).sum(axis=1)
        d0, d1 = dact(hg, act)
        grad = np.concatenate([d * p * d0, d * p * d1], axis=1) if act == SWIGLU else d * p * d0
        f = f64_to_bf16(grad)
        out["fc1_dy"][r0:r1] = f
        fq, fs = mxfp8_quantize_rows(f)
        out["fc1_dy_codes"][r0:r1], out["fc1_dy_scales"][r0:r1] = fq, fs
        fd = mxfp8_dequant_rows(fq, fs)
        out["dx"][r0:r1] = f64_to_bf16(fd @ dequant_weight(qw1t, g, MXFP8).T)
    return out


def padded_offsets(splits) -> np.ndarray:
    """Token offsets of the groups in a columnwise (wgrad) operand: each group's
    token count rounded up to a multiple of 128 (zero tokens in the padding),
    groups side by side; the last entry is the total T."""
    p = (np.asarray(splits, dtype=np.int64) + 127) // 128 * 128
    return np.concatenate([[0], np.cumsum(p)]).astype(np.int64)


def mxfp8_colwise(x, splits) -> tuple[np.ndarray, np.ndarray]:
    """Columnwise MXFP8 of a token-sorted bf16 matrix x [M, C] (bits), the
    weight-gradient operand layout: per group g the transpose x_g^T [C, m_g],
    zero-padded to T_g = 128 ceil(m_g / 128) tokens, is quantised in 1x32 blocks
    along the tokens (blocks counted from the group's first token); groups sit
    side by side.  Returns codes [C, T] and E8M0 scales [C, T / 32] (compact)."""
    x = np.ascontiguousarray(x).view(np.uint16)
    C = x.shape[1]
    offs, pofs = group_offsets(splits), padded_offsets(splits)
    T = int(pofs[-1])
    codes = np.zeros((C, T), np.uint8)
    scales = np.zeros((C, T // 32), np.uint8)
    for g in range(len(offs) - 1):
        r0, r1, p0, p1 = int(offs[g]), int(offs[g + 1]), int(pofs[g]), int(pofs[g + 1])
        if p1 == p0:
            continue
        xt = np.zeros((C, p1 - p0), np.uint16)
        xt[:, :r1 - r0] = x[r0:r1].T
        codes[:, p0:p1], scales[:, p0 // 32:p1 // 32] = mxfp8_quantize_rows(xt)
    return codes, scales


def recompute_fc2x(h, probs, act: int, tanh_clamp_scale: float | None = None) -> np.ndarray:
    """fc2_x rebuilt from the saved activation input: bf16(act(h) * prob), the
    forward's own definition (h [M, N1] bf16 bits, probs [M] or None = 1;
    tanh_clamp_scale for tanh-SReLU)."""
    hb = bf16_to_f64(np.ascontiguousarray(h).view(np.uint16))
    p = np.ones(hb.shape[0]) if probs is None else np.asarray(probs, dtype=np.float64)
    return f64_to_bf16(activation(hb, act, tanh_clamp_scale) * p[:, None])


def backward_wgrad(x, dy, h, probs, fc1_dy, splits, act: int) -> dict:
    """Oracle of gmlp_backward_wgrad (MXFP8).

    PR #2769 "GEMM + Swiglu fused Grouped MLP for MXFP8", sequence diagram,
    backward pass: the weight gradients come from grouped GEMMs ("wgrad via
    general_grouped_gemm") beside the dGLU and dgrad kernels, on the columnwise
    MXFP8 operands (the forward's `d_col_tensor`, the dGLU's columnwise
    fc1_dy).  Per group g (m_g tokens; an empty group has zero gradients):
      fc2_x = bf16(act(h) * prob)                                   [M, N]
      dW2_g = dq(colq(dy_g)) @ dq(colq(fc2_x_g))^T                  [K, N]
      dW1_g = dq(colq(fc1_dy_g)) @ dq(colq(x_g))^T                  [N1, K]
      dbias1_g = sum_t fc1_dy[t, :],  dbias2_g = sum_t dy[t, :]      (bf16 values)
    colq = mxfp8_colwise (1x32 blocks along the tokens); float64 products.
    x [M, K], dy [M, K], h [M, N1], fc1_dy [M, N1] bf16 bits; dW1 rows in the
    logical order of fc1's outputs (SwiGLU: gate rows, then up rows)."""
    x, dy = np.ascontiguousarray(x).view(np.uint16), np.ascontiguousarray(dy).view(np.uint16)
    fc1_dy = np.ascontiguousarray(fc1_dy).view(np.uint16)
    K, N1 = x.shape[1], fc1_dy.shape[1]
    fc2x = recompute_fc2x(h, probs, act)
    N = fc2x.shape[1]
    G = len(splits)
    offs, pofs = group_offsets(splits), padded_offsets(splits)
    deq = {}
    for name, m in (("dy", dy), ("fc2x", fc2x), ("fc1_dy", fc1_dy), ("x", x)):
        deq[name] = mxfp8_dequant_rows(*mxfp8_colwise(m, splits))
    out = dict(dW1=np.zeros((G, N1, K)), dW2=np.zeros((G, K, N)), dbias1=np.zeros((G, N1)),
               dbias2=np.zeros((G, K)), fc2x=fc2x)
    for g in range(G):
        p0, p1 = int(pofs[g]), int(pofs[g + 1])
        r0, r1 = int(offs[g]), int(offs[g + 1])
        out["dW2"][g] = deq["dy"][:, p0:p1] @ deq["fc2x"][:, p0:p1].T
        out["dW1"][g] = deq["fc1_dy"][:, p0:p1] @ deq["x"][:, p0:p1].T
        out["dbias1"][g] = bf16_to_f64(fc1_dy[r0:r1]).sum(axis=0)
        out["dbias2"][g] = bf16_to_f64(dy[r0:r1]).sum(axis=0)
    return out
