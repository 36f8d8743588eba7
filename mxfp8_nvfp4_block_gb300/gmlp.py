"""Thin ctypes binding of libgmlp.so (include/gmlp.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  If the library is
missing or fails to load, :func:`load` raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgmlp.so")

OK, ERR_INVALID_ARG, ERR_INVALID_DIMS, ERR_UNSUPPORTED_RECIPE, ERR_UNSUPPORTED_DEVICE, ERR_WORKSPACE, \
    ERR_CUDA, ERR_DEVICE_TIMEOUT, ERR_DEVICE_BOUNDS = range(9)
MXFP8, NVFP4 = 0, 1
SWIGLU, SRELU, TANH_SRELU = 0, 1, 2
COMPACT, GEMM_TILED, GEMM_TILED_X4 = 0, 1, 2
SCALES_GEMM_TILED, SCALES_GEMM_TILED_X4 = GEMM_TILED, GEMM_TILED_X4

EXPORTS = ["gmlp_tiled_scales_bytes", "gmlp_group_hadamard_amax", "gmlp_group_quantize_with_amax",
           "gmlp_group_quantize", "gmlp_prepare_weights", "gmlp_forward_workspace_size", "gmlp_forward",
           "gmlp_check_device_status", "gmlp_last_error", "gmlp_version", "gmlp_forward_noalloc",
           "gmlp_selftest_bounded_wait", "gmlp_mma_peak", "gmlp_replicate_weight_scales",
           "gmlp_prepare_weights_discrete", "gmlp_backward_workspace_size", "gmlp_backward_dgrad",
           "gmlp_backward_wgrad_workspace_size", "gmlp_backward_wgrad", "gmlp_colwise_tokens",
           "gmlp_query_layout", "gmlp_fc2x_recompute"]


class Recipe(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int32), ("use_rht", ctypes.c_int32), ("rht_sign_mask", ctypes.c_uint32),
                ("scale_layout", ctypes.c_int32)]


class QTensor(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p)]


class QWeightC(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("global_scale", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("G", ctypes.c_int32),
                ("format", ctypes.c_int32), ("swiglu_interleaved", ctypes.c_int32), ("scale_layout", ctypes.c_int32),
                ("bias", ctypes.c_void_p)]


class FwdAux(ctypes.Structure):
    _fields_ = [("fc2x_codes", ctypes.c_void_p), ("fc2x_scales", ctypes.c_void_p), ("fc2x_bf16", ctypes.c_void_p),
                ("fc2x_amax_pre", ctypes.c_void_p), ("fc2x_amax_post", ctypes.c_void_p),
                ("stage_events", ctypes.POINTER(ctypes.c_void_p)), ("n_stage_events", ctypes.c_int32),
                ("gemm_mode", ctypes.c_int32), ("fc2x_col_codes", ctypes.c_void_p),
                ("fc2x_col_scales", ctypes.c_void_p), ("tanh_clamp_scale", ctypes.c_float),
                ("fc1_pre_act", ctypes.c_void_p)]


_lib = None
_vp, _i64, _i32, _u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libgmlp.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libgmlp.so not found at {path}: build it with __graft_entry__.build()")
    L = ctypes.CDLL(path)
    sigs = {
        "gmlp_tiled_scales_bytes": (ctypes.c_size_t, [_i64, _i32, _i64]),
        "gmlp_group_hadamard_amax": (_i32, [_vp, _i64, _i64, _vp, _i32, _u32, _vp, _vp, _vp]),
        "gmlp_group_quantize_with_amax": (_i32, [_vp, _i64, _i64, _vp, _i32, ctypes.POINTER(Recipe), _vp, _vp,
                                                 ctypes.POINTER(QTensor), ctypes.POINTER(QTensor), _vp]),
        "gmlp_group_quantize": (_i32, [_vp, _i64, _i64, _vp, _i32, ctypes.POINTER(Recipe),
                                       ctypes.POINTER(QTensor), ctypes.POINTER(QTensor), _vp, _vp, _vp]),
        "gmlp_prepare_weights": (_i32, [_vp, _i32, _i64, _i64, _i32, _i32, _vp, _vp, _vp, _vp, _vp]),
        "gmlp_prepare_weights_discrete": (_i32, [ctypes.POINTER(ctypes.c_void_p), _i32, _i64, _i64, _i32, _i32, _vp,
                                                 _vp, _vp, _vp, _vp]),
        "gmlp_forward_workspace_size": (ctypes.c_size_t, [_i64, _i64, _i64, _i32, _i32, ctypes.POINTER(Recipe)]),
        "gmlp_forward": (_i32, [_vp, _i64, _i64, _i64, _vp, _i32, ctypes.POINTER(QWeightC),
                                ctypes.POINTER(QWeightC), _vp, _i32, ctypes.POINTER(Recipe), _vp,
                                ctypes.POINTER(FwdAux), _vp, ctypes.c_size_t, _vp]),
        "gmlp_forward_noalloc": (_i32, [_vp, _i64, _i64, _i64, _vp, _i32, ctypes.POINTER(QWeightC),
                                        ctypes.POINTER(QWeightC), _vp, _i32, ctypes.POINTER(Recipe), _vp,
                                        ctypes.POINTER(FwdAux), _vp]),
        "gmlp_check_device_status": (_i32, [_vp]),
        "gmlp_selftest_bounded_wait": (_i32, [ctypes.c_uint64, _vp]),
        "gmlp_mma_peak": (_i32, [_i32, _i32, ctypes.c_int64, _i32, _vp]),
        "gmlp_replicate_weight_scales": (_i32, [_vp, _i32, _i64, _i64, _vp, _vp]),
        "gmlp_backward_workspace_size": (ctypes.c_size_t, [_i64, _i64, _i64, _i32, _i32]),
        "gmlp_backward_dgrad": (_i32, [_vp, _i64, _i64, _i64, _vp, _i32, ctypes.POINTER(QWeightC),
                                       ctypes.POINTER(QWeightC), _vp, _vp, _i32, ctypes.POINTER(Recipe), _vp, _vp,
                                       _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp, _i32, _vp]),
        "gmlp_backward_wgrad_workspace_size": (ctypes.c_size_t, [_i64, _i64, _i64, _i32, _i32]),
        "gmlp_colwise_tokens": (_i64, [_i64, _i32]),
        "gmlp_query_layout": (_i64, [_i32, ctypes.c_void_p, _i32, _i64, _i64, _i64]),
        "gmlp_backward_wgrad": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _i32, _i32, _vp, _vp, _vp,
                                       _vp, _i32, _vp, ctypes.c_size_t, _vp, _i32, _vp]),
        "gmlp_fc2x_recompute": (_i32, [_vp, _vp, _i64, _i64, _i32, ctypes.c_float, _vp, _vp]),
        "gmlp_last_error": (ctypes.c_char_p, []),
        "gmlp_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sigs.items():
        f = getattr(L, name)
        f.restype, f.argtypes = res, args
    _lib = L
    return L


class GmlpError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"gmlp status {status}: {msg}")
        self.status = status


def _check(st: int) -> None:
    if st != OK:
        raise GmlpError(st, load().gmlp_last_error().decode())


def _p(t) -> int | None:
    """Device address of a CUDA tensor (None stays NULL).  A host tensor is
    refused here: the kernels would dereference its host address."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"expected a torch.Tensor, got {type(t).__name__}")
    if not t.is_cuda:
        raise ValueError("gmlp takes device tensors: got a tensor on " + str(t.device))
    return t.data_ptr()


def _splits_p(splits: torch.Tensor) -> int:
    """split_sizes: a contiguous 1-D int64 CUDA tensor (it stays on the device)."""
    if not isinstance(splits, torch.Tensor) or splits.dtype != torch.int64 or splits.dim() != 1 \
            or not splits.is_contiguous():
        raise ValueError("split sizes must be a contiguous 1-D int64 tensor on the device")
    return _p(splits)


def _probs_p(probs, M: int) -> int | None:
    """probs: None (all ones) or a contiguous float32 CUDA tensor of at least M values."""
    if probs is None:
        return None
    if probs.dtype != torch.float32 or not probs.is_contiguous() or probs.numel() < M:
        raise ValueError(f"probs must be a contiguous float32 tensor of at least {M} values")
    return _p(probs)


def _out_p(t, name: str, dtype, min_numel: int, device, shape=None) -> int | None:
    """A caller-supplied output buffer the library writes into: None stays
    NULL; otherwise a contiguous tensor of `dtype` on `device` (the input's
    device) holding at least `min_numel` elements (exactly `shape` when given).
    Anything else is refused here, before the kernels could write past it."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, the inputs on {device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.numel() < min_numel:
        raise ValueError(f"{name} holds {t.numel()} elements, the call writes {min_numel}")
    return _p(t)


def _fwd_aux_ptrs(aux: dict, M: int, K: int, N: int, G: int, act: int, fmt: int, device) -> dict:
    """Checked device addresses of the forward's optional outputs (sizes as
    include/gmlp.h states them for gmlp_fwd_aux)."""
    blk, cdiv = (32, 1) if fmt == MXFP8 else (16, 2)
    n1 = 2 * N if act == SWIGLU else N
    ncol = N * (M + 16 * G)
    spec = {"fc2x_codes": (torch.uint8, M * N // cdiv), "fc2x_scales": (torch.uint8, tiled_scales_bytes(M, G, N // blk)),
            "fc2x_bf16": (torch.bfloat16, M * N), "fc2x_amax_pre": (torch.float32, G),
            "fc2x_amax_post": (torch.float32, G), "fc2x_col_codes": (torch.uint8, ncol // 2),
            "fc2x_col_scales": (torch.uint8, ncol // 16), "fc1_pre_act": (torch.bfloat16, M * n1)}
    unknown = set(aux) - set(spec)
    if unknown:
        raise ValueError(f"unknown forward outputs {sorted(unknown)}")
    return {k: _out_p(aux.get(k), k, dt, n, device) for k, (dt, n) in spec.items()}


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def recipe(fmt: int, use_rht: bool = False, mask: int = 0, layout: int = GEMM_TILED) -> Recipe:
    return Recipe(fmt, int(bool(use_rht)), int(mask) & 0xFFFF, layout)


def tiled_scales_bytes(M: int, G: int, nscale: int) -> int:
    return load().gmlp_tiled_scales_bytes(M, G, nscale)


def _u8(n, device):
    return torch.empty(max(int(n), 16), dtype=torch.uint8, device=device)


def _bits(x: torch.Tensor) -> torch.Tensor:
    """A bf16 operand: contiguous, on the device."""
    if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16 or not x.is_contiguous():
        raise ValueError("expected a contiguous bf16 tensor")
    _p(x)
    return x


# ------------------------------------------------------------------ quantisers

def group_hadamard_amax(x: torch.Tensor, splits: torch.Tensor, mask: int, stream=None):
    """Per-group (pre-RHT, post-RHT) amax of bf16 x [M, K]."""
    x = _bits(x)
    M, K = x.shape
    G = splits.numel()
    pre = torch.empty(G, dtype=torch.float32, device=x.device)
    post = torch.empty(G, dtype=torch.float32, device=x.device)
    _check(load().gmlp_group_hadamard_amax(_p(x), M, K, _splits_p(splits), G, mask, _p(pre), _p(post), _stream(stream)))
    return pre, post


def alloc_quant_outputs(M: int, K: int, G: int, fmt: int, layout: int, rowwise: bool, columnwise: bool,
                        splits_host=None, device="cuda"):
    """Caller-side device buffers for a group quantisation."""
    out = {}
    blk, cdiv = (32, 1) if fmt == MXFP8 else (16, 2)
    if rowwise:
        ns = K // blk
        sbytes = tiled_scales_bytes(M, G, ns) if layout == GEMM_TILED else M * ns
        out["row"] = (_u8(M * K // cdiv, device), _u8(sbytes, device))
    if columnwise and fmt == MXFP8:
        T = colwise_tokens(M, G)   # the weight-gradient operand layout: [K][T] codes
        out["col"] = (_u8(K * T, device), _u8(K * T // 32, device))
    elif columnwise:
        mp = sum((int(m) + 15) // 16 * 16 for m in splits_host)
        out["col"] = (_u8(K * mp // 2, device), _u8(K * mp // 16, device))
    return out


def colwise_tokens(M: int, G: int) -> int:
    """T of the columnwise MXFP8 layout (see gmlp_colwise_tokens)."""
    return int(load().gmlp_colwise_tokens(M, G))


LAYOUT_TILED_SCALE, LAYOUT_COLWISE_CODE, LAYOUT_COLWISE_SCALE = 0, 1, 2


def query_layout(kind: int, splits_host, ncols: int, row: int, col: int) -> int:
    """Byte offset of one scale or code in a swizzled layout (gmlp_query_layout;
    host only, -1 when out of range)."""
    sp = (ctypes.c_int64 * len(splits_host))(*[int(m) for m in splits_host])
    return int(load().gmlp_query_layout(kind, ctypes.cast(sp, ctypes.c_void_p), len(splits_host), ncols, row, col))


def group_quantize_with_amax(x, splits, rec: Recipe, amax_pre=None, amax_post=None, *, rowwise=True,
                             columnwise=False, splits_host=None, stream=None) -> dict:
    x = _bits(x)
    M, K = x.shape
    G = splits.numel()
    bufs = alloc_quant_outputs(M, K, G, rec.format, rec.scale_layout, rowwise, columnwise, splits_host, x.device)
    row = QTensor(bufs["row"][0].data_ptr(), bufs["row"][1].data_ptr()) if rowwise else None
    col = QTensor(bufs["col"][0].data_ptr(), bufs["col"][1].data_ptr()) if columnwise else None
    _check(load().gmlp_group_quantize_with_amax(
        _p(x), M, K, _splits_p(splits), G, ctypes.byref(rec), _p(amax_pre), _p(amax_post),
        ctypes.byref(row) if row else None, ctypes.byref(col) if col else None, _stream(stream)))
    return bufs


def group_quantize(x, splits, rec: Recipe, *, rowwise=True, columnwise=False, splits_host=None,
                   stream=None) -> dict:
    x = _bits(x)
    M, K = x.shape
    G = splits.numel()
    bufs = alloc_quant_outputs(M, K, G, rec.format, rec.scale_layout, rowwise, columnwise, splits_host, x.device)
    pre = post = None
    if rec.format == NVFP4:
        pre = torch.empty(G, dtype=torch.float32, device=x.device)
        post = torch.empty(G, dtype=torch.float32, device=x.device)
        bufs["amax_pre"], bufs["amax_post"] = pre, post
    row = QTensor(bufs["row"][0].data_ptr(), bufs["row"][1].data_ptr()) if rowwise else None
    col = QTensor(bufs["col"][0].data_ptr(), bufs["col"][1].data_ptr()) if columnwise else None
    _check(load().gmlp_group_quantize(
        _p(x), M, K, _splits_p(splits), G, ctypes.byref(rec), ctypes.byref(row) if row else None,
        ctypes.byref(col) if col else None, _p(pre), _p(post), _stream(stream)))
    return bufs


# ------------------------------------------------------------------ weights

@dataclass
class QWeight:
    codes: torch.Tensor
    scales: torch.Tensor                 # GEMM_TILED
    global_scale: torch.Tensor | None
    amax: torch.Tensor | None
    rows: int
    cols: int
    G: int
    format: int
    swiglu: bool
    scales_x4: torch.Tensor | None = None  # NVFP4: GEMM_TILED_X4 copy the forward reads when present
    bias: torch.Tensor | None = None       # optional bf16 [G, rows], logical row order

    def c(self) -> QWeightC:
        if self.scales_x4 is not None:
            return QWeightC(self.codes.data_ptr(), self.scales_x4.data_ptr(), _p(self.global_scale), self.rows,
                            self.cols, self.G, self.format, int(self.swiglu), SCALES_GEMM_TILED_X4, _p(self.bias))
        return QWeightC(self.codes.data_ptr(), self.scales.data_ptr(), _p(self.global_scale), self.rows,
                        self.cols, self.G, self.format, int(self.swiglu), SCALES_GEMM_TILED, _p(self.bias))


def replicate_weight_scales(q: "QWeight", stream=None) -> torch.Tensor:
    """GEMM_TILED_X4 copy of NVFP4 weight scales (see gmlp_replicate_weight_scales)."""
    out = _u8(4 * q.G * q.rows * (q.cols // 16), q.scales.device)
    _check(load().gmlp_replicate_weight_scales(_p(q.scales), q.G, q.rows, q.cols, _p(out), _stream(stream)))
    return out


def prepare_weights(W, fmt: int, swiglu_interleave: bool = False, x4: bool = False, bias=None,
                    stream=None) -> QWeight:
    """Quantise expert weights: W is a stacked bf16 [G, rows, cols] cuda tensor,
    or a list of G bf16 [rows, cols] tensors (discrete per-expert weights).
    x4=True (NVFP4, rows and cols multiples of 256) also makes the
    GEMM_TILED_X4 scale copy, which the forward then reads (the CTA-pair mode's
    faster layout; single-CTA NVFP4 GEMMs measure faster on GEMM_TILED scales,
    which their scale-writer warps place in tensor memory).  bias: optional
    bf16 [G, rows] added in fc1 / fc2."""
    discrete = isinstance(W, (list, tuple))
    if discrete:
        Ws = [_bits(w) for w in W]
        G, (rows, cols) = len(Ws), Ws[0].shape
        dev = Ws[0].device
    else:
        W = _bits(W)
        G, rows, cols = W.shape
        dev = W.device
    blk, cdiv = (32, 1) if fmt == MXFP8 else (16, 2)
    codes = _u8(G * rows * cols // cdiv, dev)
    scales = _u8(tiled_scales_bytes(G * rows, G, cols // blk), dev)
    gs = am = None
    if fmt == NVFP4:
        gs = torch.empty(G, dtype=torch.float32, device=dev)
        am = torch.empty(G, dtype=torch.float32, device=dev)
    if discrete:
        ptrs = (ctypes.c_void_p * G)(*[w.data_ptr() for w in Ws])
        _check(load().gmlp_prepare_weights_discrete(ptrs, G, rows, cols, int(bool(swiglu_interleave)), fmt,
                                                    _p(codes), _p(scales), _p(gs), _p(am), _stream(stream)))
    else:
        _check(load().gmlp_prepare_weights(_p(W), G, rows, cols, int(bool(swiglu_interleave)), fmt, _p(codes),
                                           _p(scales), _p(gs), _p(am), _stream(stream)))
    q = QWeight(codes, scales, gs, am, rows, cols, G, fmt, bool(swiglu_interleave))
    if bias is not None:
        q.bias = _bits(bias).reshape(G, rows).contiguous()
    if x4:
        if fmt != NVFP4 or rows % 256 or cols % 256:
            raise ValueError("x4 scales: NVFP4 weights with rows and cols multiples of 256")
        q.scales_x4 = replicate_weight_scales(q, stream)
    return q


# ------------------------------------------------------------------ forward

def forward_workspace_size(M: int, K: int, N: int, G: int, act: int, rec: Recipe) -> int:
    return load().gmlp_forward_workspace_size(M, K, N, G, act, ctypes.byref(rec))


def forward(x, splits, W1: QWeight, W2: QWeight, probs, act: int, rec: Recipe, *, y=None, workspace=None,
            aux: dict | None = None, events=None, gemm_mode: int = 0, tanh_clamp_scale: float = 0.0,
            stream=None) -> torch.Tensor:
    """y = fused grouped-MLP forward of bf16 x [M, K]."""
    x = _bits(x)
    M, K = x.shape
    N = W2.cols
    G = splits.numel()
    if y is None:
        y = torch.empty((M, K), dtype=torch.bfloat16, device=x.device)
    y_p = _out_p(y, "y", torch.bfloat16, M * K, x.device, shape=(M, K))
    need = forward_workspace_size(M, K, N, G, act, rec)
    if workspace is None:
        workspace = _u8(need, x.device)
    ws_p = _out_p(workspace, "workspace", torch.uint8, need, x.device)
    aux_c = None
    ev_arr = None
    if aux is not None or events is not None or gemm_mode or act == TANH_SRELU:
        a = _fwd_aux_ptrs(aux or {}, M, K, N, G, act, rec.format, x.device)
        aux_c = FwdAux(a["fc2x_codes"], a["fc2x_scales"], a["fc2x_bf16"], a["fc2x_amax_pre"], a["fc2x_amax_post"],
                       None, 0, int(gemm_mode), a["fc2x_col_codes"], a["fc2x_col_scales"], float(tanh_clamp_scale),
                       a["fc1_pre_act"])
        if events:
            ev_arr = _event_handles(events)
            aux_c.stage_events = ctypes.cast(ev_arr, ctypes.POINTER(ctypes.c_void_p))
            aux_c.n_stage_events = len(events)
    w1c, w2c = W1.c(), W2.c()
    _check(load().gmlp_forward(_p(x), M, K, N, _splits_p(splits), G, ctypes.byref(w1c), ctypes.byref(w2c), _probs_p(probs, M),
                               act, ctypes.byref(rec), y_p, ctypes.byref(aux_c) if aux_c else None,
                               ws_p, workspace.numel(), _stream(stream)))
    return y


def forward_noalloc(x, splits, W1: QWeight, W2: QWeight, probs, act: int, rec: Recipe, *, y=None,
                    tanh_clamp_scale: float = 0.0, stream=None) -> torch.Tensor:
    """Same as :func:`forward`, but the library uses its own fixed static scratch
    instead of a workspace (for callers that cannot allocate device memory)."""
    x = _bits(x)
    M, K = x.shape
    G = splits.numel()
    if y is None:
        y = torch.empty((M, K), dtype=torch.bfloat16, device=x.device)
    y_p = _out_p(y, "y", torch.bfloat16, M * K, x.device, shape=(M, K))
    w1c, w2c = W1.c(), W2.c()
    aux_c = FwdAux(tanh_clamp_scale=float(tanh_clamp_scale)) if act == TANH_SRELU else None
    _check(load().gmlp_forward_noalloc(_p(x), M, K, W2.cols, _splits_p(splits), G, ctypes.byref(w1c), ctypes.byref(w2c),
                                       _probs_p(probs, M), act, ctypes.byref(rec), y_p,
                                       ctypes.byref(aux_c) if aux_c else None, _stream(stream)))
    return y


# ------------------------------------------------------------------ backward (data gradients)

def prepare_transposed_weights(W: torch.Tensor, fmt: int = MXFP8, stream=None) -> "QWeight":
    """Quantise W [G, R, C] transposed ([G, C, R], quantised along R): the
    operand the backward dgrad GEMMs read (W2t from W2, W1t from W1 in logical
    gate/up order)."""
    return prepare_weights(_bits(W).transpose(1, 2).contiguous(), fmt, x4=False, stream=stream)


def _event_handles(events):
    """cudaEvent_t handles of torch.cuda.Events; torch creates an event's
    handle at its first record, so an event not yet recorded is recorded once
    here (the library records it again)."""
    for e in events:
        if not e.cuda_event:
            e.record()
    return (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])


def backward_dgrad(dy, splits, W2t: "QWeight", W1t: "QWeight", pre_act, probs, act: int, rec: Recipe, *,
                   dx=None, want_dprob: bool = True, fc1_dy: dict | None = None, fc1_dy_bf16=None, workspace=None,
                   events=None, stream=None):
    """dx (and dprob) of the fused grouped MLP (see gmlp_backward_dgrad).
    fc1_dy: optional {"codes", "scales"} outputs; fc1_dy_bf16: optional [M, N1]
    bf16 output (the weight gradient's operand); events: up to 3
    torch.cuda.Event recorded after each kernel."""
    dy = _bits(dy)
    M, K = dy.shape
    N = W2t.rows
    G = splits.numel()
    if dx is None:
        dx = torch.empty((M, K), dtype=torch.bfloat16, device=dy.device)
    n1 = 2 * N if act == SWIGLU else N
    dx_p = _out_p(dx, "dx", torch.bfloat16, M * K, dy.device, shape=(M, K))
    dprob = torch.empty(M, dtype=torch.float32, device=dy.device) if want_dprob else None
    need = load().gmlp_backward_workspace_size(M, K, N, G, act)
    if workspace is None:
        workspace = _u8(need, dy.device)
    ws_p = _out_p(workspace, "workspace", torch.uint8, need, dy.device)
    fc1_dy = fc1_dy or {}
    g_codes = _out_p(fc1_dy.get("codes"), "fc1_dy codes", torch.uint8, M * n1, dy.device)
    g_scales = _out_p(fc1_dy.get("scales"), "fc1_dy scales", torch.uint8, tiled_scales_bytes(M, G, n1 // 32), dy.device)
    g_bf16 = _out_p(fc1_dy_bf16, "fc1_dy_bf16", torch.bfloat16, M * n1, dy.device)
    h_p = _p(_bits(pre_act)) if pre_act is not None else None
    if pre_act is not None and pre_act.numel() < M * n1:
        raise ValueError(f"pre_act holds {pre_act.numel()} values, the call reads {M * n1}")
    ev_arr = _event_handles(events) if events else None
    _check(load().gmlp_backward_dgrad(_p(dy), M, K, N, _splits_p(splits), G, ctypes.byref(W2t.c()), ctypes.byref(W1t.c()),
                                      h_p, _probs_p(probs, M), act, ctypes.byref(rec), dx_p, _p(dprob),
                                      g_codes, g_scales, g_bf16,
                                      ws_p,
                                      workspace.numel(), ev_arr, len(events or ()), _stream(stream)))
    return dx, dprob


def backward_wgrad(x, dy, pre_act, probs, fc1_dy, splits, act: int, *, dW1=None, dW2=None, dbias1=None,
                   dbias2=None, want=("dW1", "dW2", "dbias1", "dbias2"), accumulate: bool = False, workspace=None,
                   events=None, stream=None) -> dict:
    """Weight and bias gradients of the fused grouped MLP (see
    gmlp_backward_wgrad); outputs FP32, allocated when not given for the names
    in `want`; events: up to 6 torch.cuda.Event recorded after each kernel.
    Returns {"dW1", "dW2", "dbias1", "dbias2"} (None where skipped)."""
    x, dy, fc1_dy = _bits(x), _bits(dy), _bits(fc1_dy)
    M, K = dy.shape
    N1 = fc1_dy.shape[1]
    N = N1 // 2 if act == SWIGLU else N1
    G = splits.numel()
    dev = dy.device
    shapes = {"dW1": (G, N1, K), "dW2": (G, K, N), "dbias1": (G, N1), "dbias2": (G, K)}
    out = {"dW1": dW1, "dW2": dW2, "dbias1": dbias1, "dbias2": dbias2}
    for k in shapes:
        if out[k] is None and k in want:
            out[k] = torch.empty(shapes[k], dtype=torch.float32, device=dev)
    op = {k: _out_p(out[k], k, torch.float32, int(np.prod(shapes[k])), dev) for k in shapes}
    need = load().gmlp_backward_wgrad_workspace_size(M, K, N, G, act)
    if workspace is None:
        workspace = _u8(need, dev)
    ws_p = _out_p(workspace, "workspace", torch.uint8, need, dev)
    for t, nm, n in ((x, "x", M * K), (pre_act, "pre_act", M * N1)):
        if t is not None and t.numel() < n:
            raise ValueError(f"{nm} holds {t.numel()} values, the call reads {n}")
    _check(load().gmlp_backward_wgrad(_p(x), _p(dy), _p(_bits(pre_act) if pre_act is not None else None), _probs_p(probs, M),
                                      _p(fc1_dy), M, K, N, _splits_p(splits), G, act, op["dW1"], op["dW2"],
                                      op["dbias1"], op["dbias2"], int(bool(accumulate)), ws_p,
                                      workspace.numel(), _event_handles(events) if events else None,
                                      len(events or ()), _stream(stream)))
    return out


def fc2x_recompute(pre_act, probs, act: int, *, tanh_clamp_scale: float = 0.0, out=None, stream=None):
    """fc2_x = bf16(act(h) * prob) rebuilt from the saved activation input h
    [M, N1] (see gmlp_fc2x_recompute); returns bf16 [M, N]."""
    h = _bits(pre_act)
    M, N1 = h.shape
    N = N1 // 2 if act == SWIGLU else N1
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=h.device)
    o = _out_p(out, "out", torch.bfloat16, M * N, h.device, shape=(M, N))
    _check(load().gmlp_fc2x_recompute(_p(h), _probs_p(probs, M), M, N, act, float(tanh_clamp_scale), o,
                                      _stream(stream)))
    return out


def selftest_bounded_wait(limit_ns: int, stream=None) -> None:
    """Make a bounded device wait run out (see gmlp_selftest_bounded_wait)."""
    _check(load().gmlp_selftest_bounded_wait(int(limit_ns), _stream(stream)))


def mma_peak(fmt: int, scale_copy: int, iters: int, ctas: int = 0, stream=None) -> None:
    """Launch the tensor-core ceiling loop (see gmlp_mma_peak); asynchronous.
    scale_copy: 0 none, 1 GEMM_TILED weight-scale copies, 2 GEMM_TILED_X4 ones."""
    _check(load().gmlp_mma_peak(int(fmt), int(scale_copy), int(iters), int(ctas), _stream(stream)))


def mma_peak_flops(fmt: int, iters: int, ctas: int) -> float:
    """Floating-point operations of one gmlp_mma_peak launch."""
    k = 32 if fmt == MXFP8 else 64
    return float(ctas) * iters * 4 * 2 * 128 * 256 * k


def check_device_status(stream=None) -> None:
    _check(load().gmlp_check_device_status(_stream(stream)))
