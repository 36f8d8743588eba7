"""The C ABI library loads, exports every symbol include/gmlp.h declares, and its
host-side checks return the documented statuses before any launch (CPU only:
no call here reaches the device)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mxfp8_nvfp4_block_gb300 import build, gmlp
    build.build()
    return gmlp.load(), gmlp


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "gmlp.h")).read()
    return sorted(set(re.findall(r"^GMLP_API [^;(]*?\b(gmlp_\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert len(names) >= 10
    out = subprocess.run(["nm", "-D", "--defined-only", lib[1].LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r" T (gmlp_\w+)", out))
    assert set(names) <= exported, set(names) - exported
    assert set(lib[1].EXPORTS) == set(names)
    for n in names:
        getattr(lib[0], n)


def test_version_and_sizes(lib):
    L, g = lib
    assert b"sm_103a" in L.gmlp_version()
    assert g.tiled_scales_bytes(512, 4, 8) == (4 + 4) * 128 * 8
    assert g.tiled_scales_bytes(0, 3, 4) == 3 * 128 * 4
    r = g.recipe(g.MXFP8)
    n = g.forward_workspace_size(512, 256, 256, 4, g.SWIGLU, r)
    assert n >= 512 * 256 * 2
    assert g.forward_workspace_size(512, 256, 256, 4, g.SWIGLU, g.recipe(g.NVFP4)) > 512 * 256 * 2


FAKE = 1 << 20   # an aligned non-null address; validation fails before anything dereferences it


def test_quantize_argument_checks(lib):
    L, g = lib
    r = g.recipe(g.MXFP8)
    qt = g.QTensor(FAKE, FAKE)
    # G out of range
    assert L.gmlp_group_quantize(FAKE, 64, 128, FAKE, 0, ctypes.byref(r), ctypes.byref(qt), None, None, None,
                                 None) == g.ERR_INVALID_DIMS
    assert L.gmlp_group_quantize(FAKE, 64, 128, FAKE, 513, ctypes.byref(r), ctypes.byref(qt), None, None, None,
                                 None) == g.ERR_INVALID_DIMS
    # K not a multiple of 128
    assert L.gmlp_group_quantize(FAKE, 64, 96, FAKE, 2, ctypes.byref(r), ctypes.byref(qt), None, None, None,
                                 None) == g.ERR_INVALID_DIMS
    assert b"K" in L.gmlp_last_error()
    # NULL recipe / split sizes / outputs
    assert L.gmlp_group_quantize(FAKE, 64, 128, FAKE, 2, None, ctypes.byref(qt), None, None, None,
                                 None) == g.ERR_INVALID_ARG
    assert L.gmlp_group_quantize(FAKE, 64, 128, None, 2, ctypes.byref(r), ctypes.byref(qt), None, None, None,
                                 None) == g.ERR_INVALID_ARG
    assert L.gmlp_group_quantize(FAKE, 64, 128, FAKE, 2, ctypes.byref(r), None, None, None, None,
                                 None) == g.ERR_INVALID_ARG
    # misaligned x
    assert L.gmlp_group_quantize(FAKE + 2, 64, 128, FAKE, 2, ctypes.byref(r), ctypes.byref(qt), None, None, None,
                                 None) == g.ERR_INVALID_ARG
    # MXFP8 columnwise codes / scales are written in 32-byte vectors
    q16 = g.QTensor(FAKE + 16, FAKE)
    assert L.gmlp_group_quantize(FAKE, 64, 128, FAKE, 2, ctypes.byref(r), None, ctypes.byref(q16),
                                 None, None, None) == g.ERR_INVALID_ARG
    assert L.gmlp_colwise_tokens(300, 3) == 128 * (3 + 3)
    assert L.gmlp_colwise_tokens(0, 1) == 128 and L.gmlp_colwise_tokens(-1, 1) == 0
    # unknown format
    bad = g.Recipe(7, 0, 0, 1)
    assert L.gmlp_group_quantize(FAKE, 64, 128, FAKE, 2, ctypes.byref(bad), ctypes.byref(qt), None, None, None,
                                 None) == g.ERR_UNSUPPORTED_RECIPE
    # NVFP4 needs amax buffers
    rn = g.recipe(g.NVFP4, use_rht=True)
    assert L.gmlp_group_quantize(FAKE, 64, 128, FAKE, 2, ctypes.byref(rn), ctypes.byref(qt), ctypes.byref(qt),
                                 FAKE, None, None) == g.ERR_INVALID_ARG
    assert L.gmlp_group_hadamard_amax(FAKE, 64, 100, FAKE, 2, 0, FAKE, FAKE, None) == g.ERR_INVALID_DIMS
    assert L.gmlp_group_hadamard_amax(FAKE, 64, 128, FAKE, 2, 0, None, FAKE, None) == g.ERR_INVALID_ARG


def test_forward_argument_checks(lib):
    L, g = lib
    r = g.recipe(g.MXFP8)
    w1 = g.QWeightC(FAKE, FAKE, None, 512, 256, 4, g.MXFP8, 1, 0)
    w2 = g.QWeightC(FAKE, FAKE, None, 256, 256, 4, g.MXFP8, 0, 0)
    need = g.forward_workspace_size(512, 256, 256, 4, g.SWIGLU, r)

    def call(M=512, K=256, N=256, G=4, W1=w1, W2=w2, act=g.SWIGLU, rec=r, ws=FAKE, wsb=need, y=FAKE):
        return L.gmlp_forward(FAKE, M, K, N, FAKE, G, ctypes.byref(W1), ctypes.byref(W2), None, act,
                              ctypes.byref(rec), y, None, ws, wsb, None)

    bad_aux = g.FwdAux(None, None, None, None, None, None, 0, 1)
    assert L.gmlp_forward(FAKE, 512, 256, 256, FAKE, 4, ctypes.byref(w1), ctypes.byref(w2), None, g.SWIGLU,
                          ctypes.byref(r), FAKE, ctypes.byref(bad_aux), FAKE, need, None) == g.ERR_INVALID_ARG
    assert call(y=FAKE + 16) == g.ERR_INVALID_ARG                   # y is stored in 32-byte vectors
    pre16 = g.FwdAux(None, None, None, None, None, None, 0, 0, None, None, 0.0, FAKE + 16)
    assert L.gmlp_forward(FAKE, 512, 256, 256, FAKE, 4, ctypes.byref(w1), ctypes.byref(w2), None, g.SWIGLU,
                          ctypes.byref(r), FAKE, ctypes.byref(pre16), FAKE, need, None) == g.ERR_INVALID_ARG
    assert call(K=128) == g.ERR_INVALID_DIMS                        # K % 256
    assert call(N=192) == g.ERR_INVALID_DIMS                        # N % 128
    assert call(G=3) == g.ERR_INVALID_DIMS                          # weights have 4 experts
    assert call(act=9) == g.ERR_INVALID_ARG
    assert call(wsb=need - 1) == g.ERR_WORKSPACE
    assert call(ws=None) == g.ERR_WORKSPACE
    assert call(rec=g.recipe(g.NVFP4)) == g.ERR_UNSUPPORTED_RECIPE  # weight format differs
    w1_plain = g.QWeightC(FAKE, FAKE, None, 512, 256, 4, g.MXFP8, 0, 0)
    assert call(W1=w1_plain) == g.ERR_INVALID_ARG                   # SwiGLU needs the interleave
    assert call(act=g.SRELU) == g.ERR_INVALID_DIMS                  # SReLU W1 has N rows
    w1_nv = g.QWeightC(FAKE, FAKE, None, 512, 256, 4, g.NVFP4, 1, 0)
    w2_nv = g.QWeightC(FAKE, FAKE, None, 256, 256, 4, g.NVFP4, 0, 0)
    rn = g.recipe(g.NVFP4)
    assert call(W1=w1_nv, W2=w2_nv, rec=rn, wsb=1 << 30) == g.ERR_INVALID_ARG   # no global scales
    assert L.gmlp_prepare_weights(FAKE, 4, 100, 256, 0, g.MXFP8, FAKE, FAKE, None, None, None) == g.ERR_INVALID_DIMS
    assert L.gmlp_prepare_weights(FAKE, 4, 128, 128, 0, g.NVFP4, FAKE, FAKE, FAKE, FAKE, None) == g.ERR_INVALID_DIMS
    assert L.gmlp_prepare_weights(FAKE, 4, 128, 256, 0, g.NVFP4, FAKE, FAKE, None, None, None) == g.ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(tmp_path):
    from mxfp8_nvfp4_block_gb300 import gmlp
    saved = gmlp._lib
    gmlp._lib = None
    try:
        with pytest.raises(RuntimeError, match="not found"):
            gmlp.load(str(tmp_path / "missing.so"))
    finally:
        gmlp._lib = saved


def test_mma_peak_argument_checks(lib):
    L, g = lib
    assert L.gmlp_mma_peak(7, 1, 100, 0, None) == g.ERR_INVALID_ARG          # format
    assert L.gmlp_mma_peak(g.MXFP8, 1, 0, 0, None) == g.ERR_INVALID_ARG      # iters < 1
    assert L.gmlp_mma_peak(g.NVFP4, 0, (1 << 24) + 1, 0, None) == g.ERR_INVALID_ARG
    assert b"iters" in L.gmlp_last_error()
    assert L.gmlp_mma_peak(g.MXFP8, 2, 100, 0, None) == g.ERR_INVALID_ARG       # X4 copies are NVFP4's
    assert L.gmlp_mma_peak(g.NVFP4, 4, 100, 0, None) == g.ERR_INVALID_ARG
    assert b"scale_copy" in L.gmlp_last_error()
    assert g.mma_peak_flops(g.MXFP8, 10, 2) == 2 * 10 * 4 * 2 * 128 * 256 * 32
    assert g.mma_peak_flops(g.NVFP4, 10, 2) == 2 * 10 * 4 * 2 * 128 * 256 * 64


def test_replicate_weight_scales_argument_checks(lib):
    L, g = lib
    assert L.gmlp_replicate_weight_scales(None, 2, 256, 256, FAKE, None) == g.ERR_INVALID_ARG
    assert L.gmlp_replicate_weight_scales(FAKE, 2, 128, 256, FAKE, None) == g.ERR_INVALID_DIMS   # rows % 256
    assert L.gmlp_replicate_weight_scales(FAKE, 2, 256, 384, FAKE, None) == g.ERR_INVALID_DIMS   # cols % 256
    assert L.gmlp_replicate_weight_scales(FAKE, 0, 256, 256, FAKE, None) == g.ERR_INVALID_DIMS


def test_forward_weight_scale_layout_checks(lib):
    L, g = lib
    rn = g.recipe(g.NVFP4)
    need = g.forward_workspace_size(512, 256, 256, 4, g.SRELU, rn)

    def call(l1=0, l2=0, fmt=g.NVFP4, aux=None):
        w1 = g.QWeightC(FAKE, FAKE, FAKE, 256, 256, 4, fmt, 0, l1)
        w2 = g.QWeightC(FAKE, FAKE, FAKE, 256, 256, 4, fmt, 0, l2)
        return L.gmlp_forward(FAKE, 512, 256, 256, FAKE, 4, ctypes.byref(w1), ctypes.byref(w2), None, g.SRELU,
                              ctypes.byref(g.recipe(fmt)), FAKE, aux, FAKE, need, None)

    assert call(l1=3) == g.ERR_INVALID_ARG
    assert call(l2=g.GEMM_TILED_X4, fmt=g.MXFP8) == g.ERR_INVALID_ARG    # X4 is an NVFP4 layout
    pair = g.FwdAux(None, None, None, None, None, None, 0, 2)
    # CTA pairs read GEMM_TILED_X4 too: the call passes the argument checks (then needs a device)
    assert call(l1=g.GEMM_TILED_X4, aux=ctypes.byref(pair)) in (g.ERR_CUDA, g.ERR_UNSUPPORTED_DEVICE)


def test_forward_columnwise_fc2x_checks(lib):
    L, g = lib
    r = g.recipe(g.MXFP8)
    w1 = g.QWeightC(FAKE, FAKE, None, 512, 256, 4, g.MXFP8, 1, 0)
    w2 = g.QWeightC(FAKE, FAKE, None, 256, 256, 4, g.MXFP8, 0, 0)
    need = g.forward_workspace_size(512, 256, 256, 4, g.SWIGLU, r)
    aux = g.FwdAux(None, None, None, None, None, None, 0, 0, FAKE, FAKE)
    assert L.gmlp_forward(FAKE, 512, 256, 256, FAKE, 4, ctypes.byref(w1), ctypes.byref(w2), None, g.SWIGLU,
                          ctypes.byref(r), FAKE, ctypes.byref(aux), FAKE, need, None) == g.ERR_INVALID_ARG
    assert b"NVFP4" in L.gmlp_last_error()


def test_forward_tanh_srelu_needs_a_clamp_scale(lib):
    L, g = lib
    r = g.recipe(g.NVFP4)
    w1 = g.QWeightC(FAKE, FAKE, FAKE, 256, 256, 4, g.NVFP4, 0, 0)
    w2 = g.QWeightC(FAKE, FAKE, FAKE, 256, 256, 4, g.NVFP4, 0, 0)
    need = g.forward_workspace_size(512, 256, 256, 4, g.TANH_SRELU, r)

    def call(aux):
        return L.gmlp_forward(FAKE, 512, 256, 256, FAKE, 4, ctypes.byref(w1), ctypes.byref(w2), None, g.TANH_SRELU,
                              ctypes.byref(r), FAKE, aux, FAKE, need, None)

    assert call(None) == g.ERR_INVALID_ARG
    assert call(ctypes.byref(g.FwdAux(tanh_clamp_scale=0.0))) == g.ERR_INVALID_ARG
    assert call(ctypes.byref(g.FwdAux(tanh_clamp_scale=float("inf")))) == g.ERR_INVALID_ARG
    assert b"tanh" in L.gmlp_last_error()


def test_prepare_weights_discrete_and_bias_checks(lib):
    L, g = lib
    ptrs = (ctypes.c_void_p * 2)(FAKE, None)
    assert L.gmlp_prepare_weights_discrete(None, 2, 256, 256, 0, g.MXFP8, FAKE, FAKE, None, None, None) \
        == g.ERR_INVALID_ARG
    assert L.gmlp_prepare_weights_discrete(ptrs, 2, 256, 256, 0, g.MXFP8, FAKE, FAKE, None, None, None) \
        == g.ERR_INVALID_ARG                                               # expert 1 NULL
    assert b"weight 1" in L.gmlp_last_error()
    assert L.gmlp_prepare_weights_discrete(ptrs, 2, 200, 256, 0, g.MXFP8, FAKE, FAKE, None, None, None) \
        == g.ERR_INVALID_DIMS
    r = g.recipe(g.MXFP8)
    need = g.forward_workspace_size(512, 256, 256, 4, g.SRELU, r)
    w1 = g.QWeightC(FAKE, FAKE, None, 256, 256, 4, g.MXFP8, 0, 0, FAKE + 2)   # misaligned bias
    w2 = g.QWeightC(FAKE, FAKE, None, 256, 256, 4, g.MXFP8, 0, 0)
    assert L.gmlp_forward(FAKE, 512, 256, 256, FAKE, 4, ctypes.byref(w1), ctypes.byref(w2), None, g.SRELU,
                          ctypes.byref(r), FAKE, None, FAKE, need, None) == g.ERR_INVALID_ARG
    assert b"bias" in L.gmlp_last_error()


def test_backward_dgrad_checks(lib):
    L, g = lib
    r = g.recipe(g.MXFP8)
    w2t = g.QWeightC(FAKE, FAKE, None, 256, 512, 4, g.MXFP8, 0, 0)   # [N x K]
    w1t = g.QWeightC(FAKE, FAKE, None, 512, 256, 4, g.MXFP8, 0, 0)   # [K x N1] (SReLU)
    need = L.gmlp_backward_workspace_size(512, 512, 256, 4, g.SRELU)

    def call(K=512, N=256, act=g.SRELU, rec=r, W2t=w2t, W1t=w1t, pre=FAKE, ev=None, n_ev=0, dx=FAKE, bf=None):
        return L.gmlp_backward_dgrad(FAKE, 512, K, N, FAKE, 4, ctypes.byref(W2t), ctypes.byref(W1t), pre, None, act,
                                     ctypes.byref(rec), dx, None, None, None, bf, FAKE, need, ev, n_ev, None)

    assert call(rec=g.recipe(g.NVFP4)) == g.ERR_UNSUPPORTED_RECIPE
    assert call(act=g.TANH_SRELU) == g.ERR_INVALID_ARG
    assert call(N=128) == g.ERR_INVALID_DIMS
    assert call(W2t=w1t) == g.ERR_INVALID_DIMS          # shapes swapped
    assert call(pre=None) == g.ERR_INVALID_ARG
    assert call(pre=FAKE + 16) == g.ERR_INVALID_ARG      # read in 32-byte vectors
    assert call(dx=FAKE + 16) == g.ERR_INVALID_ARG       # stored in 32-byte vectors
    assert call(bf=FAKE + 16) == g.ERR_INVALID_ARG       # bf16 fc1_dy too
    assert call(n_ev=4, ev=FAKE) == g.ERR_INVALID_ARG    # at most 3 stage events
    assert call(n_ev=1) == g.ERR_INVALID_ARG             # events NULL


def test_backward_wgrad_checks(lib):
    L, g = lib
    M, K, N, G = 512, 512, 256, 4
    need = L.gmlp_backward_wgrad_workspace_size(M, K, N, G, g.SWIGLU)
    T = L.gmlp_colwise_tokens(M, G)
    assert need >= (2 * K + N + 2 * N) * T

    def call(K=K, N=N, act=g.SWIGLU, x=FAKE, dy=FAKE, pre=FAKE, f=FAKE, dW1=FAKE, dW2=FAKE, db1=None, db2=None,
             acc=0, ws=FAKE, wsb=need, ev=None, n_ev=0):
        return L.gmlp_backward_wgrad(x, dy, pre, None, f, M, K, N, FAKE, G, act, dW1, dW2, db1, db2, acc, ws, wsb,
                                     ev, n_ev, None)

    assert call(act=g.TANH_SRELU) == g.ERR_INVALID_ARG
    assert call(K=384) == g.ERR_INVALID_DIMS
    assert call(N=128) == g.ERR_INVALID_DIMS
    assert call(acc=2) == g.ERR_INVALID_ARG
    assert call(pre=None) == g.ERR_INVALID_ARG            # dW2 rebuilds fc2_x from pre_act
    assert call(x=None) == g.ERR_INVALID_ARG              # dW1 needs x
    assert call(f=None) == g.ERR_INVALID_ARG
    assert call(dW1=FAKE + 16) == g.ERR_INVALID_ARG       # 32-byte vector stores
    assert call(pre=FAKE + 16) == g.ERR_INVALID_ARG
    assert call(db1=FAKE + 2) == g.ERR_INVALID_ARG
    assert call(wsb=need - 1) == g.ERR_WORKSPACE
    assert call(ws=None) == g.ERR_WORKSPACE
    assert call(n_ev=7, ev=FAKE) == g.ERR_INVALID_ARG      # at most 6 stage events
    assert call(n_ev=2) == g.ERR_INVALID_ARG               # events NULL


def test_query_layout_matches_the_oracles_layouts(lib, orc):
    """gmlp_query_layout against the oracle's own restatement of the layouts
    (oracle/layout.py for GEMM_TILED; the chunk-major columnwise MXFP8 layout
    as the weight-gradient parity tests de-swizzle it): every owned scale and
    code of a ragged split with empty groups, and -1 outside the tensor."""
    import numpy as np
    L, g = lib
    splits = [130, 0, 257, 5, 1, 128]
    M, G = sum(splits), len(splits)
    ks = 8
    want = orc.tiled_index(np.array(splits), ks)
    got = np.array([[g.query_layout(g.LAYOUT_TILED_SCALE, splits, ks, r, j) for j in range(ks)] for r in range(M)])
    assert np.array_equal(got, want)

    C = 256
    T = g.colwise_tokens(M, G)
    # code buffer [T/128][C][128] viewed as the logical [C][T] operand
    code_pos = np.arange(C * T).reshape(T // 128, C, 128).transpose(1, 0, 2).reshape(C, T)
    scale_pos = orc.tiled_index(np.array([C]), T // 32)           # a [C]-row operand, T/32 scales per row
    offs, pofs = orc.group_offsets(np.array(splits)), orc.padded_offsets(np.array(splits))
    rng = np.random.default_rng(3)
    for t in rng.integers(0, M, 64):
        grp = int(np.searchsorted(offs, t, side="right") - 1)
        p = int(pofs[grp] + t - offs[grp])
        for c in rng.integers(0, C, 8):
            assert g.query_layout(g.LAYOUT_COLWISE_CODE, splits, C, int(t), int(c)) == code_pos[c, p]
            assert g.query_layout(g.LAYOUT_COLWISE_SCALE, splits, C, int(t), int(c)) == scale_pos[c, p // 32]

    for kind, nc in ((g.LAYOUT_TILED_SCALE, ks), (g.LAYOUT_COLWISE_CODE, C), (g.LAYOUT_COLWISE_SCALE, C)):
        assert g.query_layout(kind, splits, nc, M, 0) == -1
        assert g.query_layout(kind, splits, nc, 0, nc) == -1
        assert g.query_layout(kind, splits, nc, -1, 0) == -1
    assert g.query_layout(g.LAYOUT_TILED_SCALE, splits, 6, 0, 0) == -1        # not a multiple of 4
    assert g.query_layout(g.LAYOUT_COLWISE_SCALE, splits, 96, 0, 0) == -1     # not a multiple of 128
    assert g.query_layout(7, splits, ks, 0, 0) == -1
    assert g.query_layout(g.LAYOUT_TILED_SCALE, [4, -1], ks, 0, 0) == -1


def test_feature_counts_above_2_to_20_are_rejected(lib):
    """K, N and weight rows / cols above 2^20 are INVALID_DIMS in every call
    that takes them; 2^20 itself passes the dimension checks (the call then
    stops at a later check, never at the size)."""
    L, g = lib
    big, top = (1 << 20) + 256, 1 << 20
    r = g.recipe(g.MXFP8)
    qt = g.QTensor(FAKE, FAKE)
    assert L.gmlp_group_quantize(FAKE, 64, big, FAKE, 2, ctypes.byref(r), ctypes.byref(qt), None, None, None,
                                 None) == g.ERR_INVALID_DIMS
    assert L.gmlp_group_quantize(FAKE, 64, top, FAKE, 2, ctypes.byref(r), ctypes.byref(qt), None, None, None,
                                 None) != g.ERR_INVALID_DIMS
    assert L.gmlp_group_quantize_with_amax(FAKE, 64, big, FAKE, 2, ctypes.byref(r), None, None, ctypes.byref(qt),
                                           None, None) == g.ERR_INVALID_DIMS
    assert L.gmlp_group_hadamard_amax(FAKE, 64, big, FAKE, 2, 0, FAKE, FAKE, None) == g.ERR_INVALID_DIMS
    assert L.gmlp_group_hadamard_amax(FAKE, 64, top, FAKE, 2, 0, FAKE, FAKE, None) != g.ERR_INVALID_DIMS
    assert L.gmlp_prepare_weights(FAKE, 1, big, 256, 0, g.MXFP8, FAKE, FAKE, None, None, None) == g.ERR_INVALID_DIMS
    assert L.gmlp_prepare_weights(FAKE, 1, 256, big, 0, g.MXFP8, FAKE, FAKE, None, None, None) == g.ERR_INVALID_DIMS
    assert L.gmlp_prepare_weights(FAKE, 1, top, top, 0, g.MXFP8, FAKE, FAKE, None, None, None) != g.ERR_INVALID_DIMS
    assert L.gmlp_replicate_weight_scales(FAKE, 1, big, 256, FAKE, None) == g.ERR_INVALID_DIMS
    assert L.gmlp_replicate_weight_scales(FAKE, 1, 256, top, FAKE, None) != g.ERR_INVALID_DIMS
    for K, N in ((big, 256), (256, big)):
        w1 = g.QWeightC(FAKE, FAKE, None, 2 * N, K, 1, g.MXFP8, 1, 0)
        w2 = g.QWeightC(FAKE, FAKE, None, K, N, 1, g.MXFP8, 0, 0)
        assert L.gmlp_forward(FAKE, 64, K, N, FAKE, 1, ctypes.byref(w1), ctypes.byref(w2), None, g.SWIGLU,
                              ctypes.byref(r), FAKE, None, FAKE, 1 << 40, None) == g.ERR_INVALID_DIMS
        assert L.gmlp_backward_dgrad(FAKE, 64, K, N, FAKE, 1, ctypes.byref(w2), ctypes.byref(w1), FAKE, None,
                                     g.SWIGLU, ctypes.byref(r), FAKE, None, None, None, None, FAKE, 1 << 40, None, 0,
                                     None) == g.ERR_INVALID_DIMS
        assert L.gmlp_backward_wgrad(FAKE, FAKE, FAKE, None, FAKE, 64, K, N, FAKE, 1, g.SWIGLU, FAKE, FAKE, None,
                                     None, 0, FAKE, 1 << 40, None, 0, None) == g.ERR_INVALID_DIMS
    w1 = g.QWeightC(FAKE, FAKE, None, 2 * top, top, 1, g.MXFP8, 1, 0)
    w2 = g.QWeightC(FAKE, FAKE, None, top, top, 1, g.MXFP8, 0, 0)
    assert L.gmlp_forward(FAKE, 64, top, top, FAKE, 1, ctypes.byref(w1), ctypes.byref(w2), None, g.SWIGLU,
                          ctypes.byref(r), FAKE, None, FAKE, 1 << 40, None) != g.ERR_INVALID_DIMS


def test_binding_refuses_host_and_mistyped_tensors(lib):
    """The binding passes device addresses only: a host tensor, split sizes
    that are not int64, or probs that are not float32 (or too short) raise
    before anything reaches the library (a kernel would otherwise dereference
    a host address or misread the buffer)."""
    import torch
    _, g = lib
    x = torch.zeros((64, 128), dtype=torch.bfloat16)          # host memory
    with pytest.raises(ValueError, match="device"):
        g.group_hadamard_amax(x, torch.tensor([64]), 0)
    with pytest.raises(ValueError):
        g.forward(x.float(), torch.tensor([64]), None, None, None, g.SWIGLU, g.recipe(g.MXFP8))
    with pytest.raises(ValueError, match="int64"):
        g._splits_p(torch.tensor([64], dtype=torch.int32))
    with pytest.raises(ValueError, match="device"):
        g._splits_p(torch.tensor([64]))
    with pytest.raises(ValueError, match="float32"):
        g._probs_p(torch.ones(64, dtype=torch.float64), 64)
    with pytest.raises(ValueError, match="at least 64"):
        g._probs_p(torch.ones(32), 64)
    with pytest.raises(TypeError):
        g._p([1, 2, 3])
    assert g._p(None) is None and g._probs_p(None, 64) is None


def test_binding_refuses_wrong_output_buffers(lib):
    """Output buffers are checked before their addresses reach the library:
    y must be a contiguous bf16 [M, K] tensor on the inputs' device, and every
    optional forward output must hold what the forward writes into it (a short
    or mistyped buffer would otherwise be written past its end)."""
    import torch
    _, g = lib
    cpu = torch.device("cpu")
    M, K, N, G = 64, 256, 256, 2
    with pytest.raises(ValueError, match="bfloat16"):
        g._out_p(torch.zeros((M, K), dtype=torch.float32), "y", torch.bfloat16, M * K, cpu, shape=(M, K))
    with pytest.raises(ValueError, match="shape"):
        g._out_p(torch.zeros((M, K // 2), dtype=torch.bfloat16), "y", torch.bfloat16, M * K, cpu, shape=(M, K))
    with pytest.raises(ValueError, match="contiguous"):
        g._out_p(torch.zeros((K, M), dtype=torch.bfloat16).t(), "y", torch.bfloat16, M * K, cpu, shape=(M, K))
    with pytest.raises(ValueError, match="is on"):
        g._out_p(torch.zeros((M, K), dtype=torch.bfloat16), "y", torch.bfloat16, M * K, torch.device("cuda", 0),
                 shape=(M, K))
    assert g._out_p(None, "y", torch.bfloat16, 1, cpu) is None
    for fmt, act in ((g.MXFP8, g.SWIGLU), (g.NVFP4, g.SRELU)):
        cdiv = 1 if fmt == g.MXFP8 else 2
        short = {"fc2x_codes": torch.zeros(M * N // cdiv - 1, dtype=torch.uint8),
                 "fc2x_scales": torch.zeros(16, dtype=torch.uint8),
                 "fc2x_amax_pre": torch.zeros(G - 1, dtype=torch.float32),
                 "fc2x_col_codes": torch.zeros(N * M // 2, dtype=torch.uint8),   # no room for group padding
                 "fc1_pre_act": torch.zeros((M, N), dtype=torch.bfloat16)}
        for k, v in short.items():
            if k == "fc1_pre_act" and act == g.SRELU:
                continue                                    # [M, N] is the SReLU size
            with pytest.raises(ValueError, match=k):
                g._fwd_aux_ptrs({k: v}, M, K, N, G, act, fmt, cpu)
        with pytest.raises(ValueError, match="float32"):
            g._fwd_aux_ptrs({"fc2x_amax_post": torch.zeros(G, dtype=torch.float64)}, M, K, N, G, act, fmt, cpu)
        with pytest.raises(ValueError, match="unknown"):
            g._fwd_aux_ptrs({"fc2x_code": torch.zeros(M * N, dtype=torch.uint8)}, M, K, N, G, act, fmt, cpu)
