"""Parity of the fused grouped-MLP forward (CUDA path, through the C ABI) with
the oracle.

* Lossless operands (one-hot fc1 weights, small powers of two): the block-
  scaled MMA, the scale layouts, the tile map over ragged groups and the fused
  epilogues must reproduce the oracle's y bit for bit.
* The workloads: >= 99.9% of fc2_x codes identical with the rest one code step
  apart, and normalised Frobenius error of y <= 1e-2.
* The NVFP4 epilogue's fused (pre, post)-RHT amax equals the standalone group
  Hadamard-amax of the bf16 fc2_x it stored, bitwise.
"""
import numpy as np
import pytest
import torch

from mxfp8_nvfp4_block_gb300.inputs import WORKLOADS, bits, make_inputs
from oracle.layout import tiled_index
from parity import code_match_report, frob, np_bits, np_u8, nvfp4_scale_of

pytestmark = pytest.mark.gpu

CODE_MATCH = 0.999   # fraction of identical fc2_x codes
Y_TOL = 1e-2         # normalised Frobenius error of y


def bf16_cpu(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)


def run_gpu(gm, d, fmt, act, mask=0, probs=True, gemm_mode=0, x4=None, tanh_c=0.0):
    w1 = gm.prepare_weights(d["W1"].cuda(), fmt, swiglu_interleave=(act == gm.SWIGLU), x4=x4)
    w2 = gm.prepare_weights(d["W2"].cuda(), fmt, x4=x4)
    M, N = d["x"].shape[0], d["W2"].shape[2]
    G = d["splits"].numel()
    cdiv = 1 if fmt == gm.MXFP8 else 2
    aux = {"fc2x_codes": torch.zeros(M * N // cdiv + 16, dtype=torch.uint8, device="cuda"),
           "fc2x_scales": torch.zeros(gm.tiled_scales_bytes(M, G, N // (32 if fmt == 0 else 16)) + 16,
                                      dtype=torch.uint8, device="cuda")}
    if fmt == gm.NVFP4:
        aux["fc2x_bf16"] = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
        aux["fc2x_amax_pre"] = torch.zeros(G, dtype=torch.float32, device="cuda")
        aux["fc2x_amax_post"] = torch.zeros(G, dtype=torch.float32, device="cuda")
    rec = gm.recipe(fmt, use_rht=True, mask=mask)
    p = d["probs"].cuda() if probs else None
    y = torch.full((M, d["x"].shape[1]), float("nan"), dtype=torch.bfloat16, device="cuda")
    gm.forward(d["x"].cuda(), d["splits"].cuda(), w1, w2, p, act, rec, y=y, aux=aux, gemm_mode=gemm_mode,
               tanh_clamp_scale=tanh_c)
    gm.check_device_status()
    torch.cuda.synchronize()
    return y, aux


def onehot_case(fmt, act, splits, K, N, seed):
    rng = np.random.default_rng(seed)
    G = len(splits)
    M = int(sum(splits))
    offs = np.concatenate([[0], np.cumsum(splits)])
    n1 = 2 * N if act == 0 else N
    if fmt == 0:
        x = rng.choice([0.0, 1, 2, 4, -1, -2, -4], size=(M, K))
        probs = rng.choice([0.5, 1.0], size=M).astype(np.float32)
    else:
        x = rng.choice([0.0, 2, 4, -2, -4], size=(M, K))
        probs = np.ones(M, np.float32)
        for g in range(G):
            if splits[g]:
                x[offs[g]] = 4.0
    W1 = np.zeros((G, n1, K))
    for g in range(G):
        W1[g, np.arange(n1), rng.integers(0, K, n1)] = 1.0
    if fmt == 0:
        W2 = rng.choice([0.0, 1, 2, -1, -2, 4, -4], size=(G, K, N))
    else:      # one-hot rows keep |y| <= 64 so the fc2 alpha product stays exact after bf16 rounding
        W2 = np.zeros((G, K, N))
        for g in range(G):
            W2[g, np.arange(K), rng.integers(0, N, K)] = rng.choice([1.0, -2, 4], K)
            W2[g, 0, :] = 0
            W2[g, 0, 0] = 4.0
    return dict(x=bf16_cpu(x), splits=torch.tensor(splits, dtype=torch.int64), W1=bf16_cpu(W1),
                W2=bf16_cpu(W2), probs=torch.from_numpy(probs))


@pytest.mark.parametrize("gemm_mode", [0, 2], ids=["cta", "cta_pair"])
@pytest.mark.parametrize("fmt,act", [(0, 1), (1, 1), (0, 0), (1, 0)],
                         ids=["mxfp8-srelu", "nvfp4-srelu", "mxfp8-swiglu", "nvfp4-swiglu"])
def test_forward_lossless_bitexact(orc, gm, fmt, act, gemm_mode):
    if act == 0:
        splits, K, N = [130, 0, 257, 5, 128], 512, 256      # SwiGLU: fc1 width 512
    else:
        splits, K, N = [130, 0, 257, 5, 128], 512, 512
    d = onehot_case(fmt, act, splits, K, N, seed=fmt * 10 + act)
    y, aux = run_gpu(gm, d, fmt, act, gemm_mode=gemm_mode)
    ref = orc.forward(bits(d["x"]), np.array(splits), bits(d["W1"]), bits(d["W2"]), d["probs"].numpy(), act, fmt)
    M = sum(splits)
    if act == 1:
        # SReLU on these operands is lossless end to end: bit-exact fc2_x codes and y
        cdiv = 1 if fmt == 0 else 2
        assert np.array_equal(np_u8(aux["fc2x_codes"], M * N // cdiv).reshape(M, -1), ref["fc2x_codes"])
        assert np.array_equal(np_bits(y), ref["y"])
    else:
        # SwiGLU: exact fc1 (one-hot), then silu in FP32 vs FP64
        frac, steps = code_match_report(fmt, np_u8(aux["fc2x_codes"], M * N // (1 if fmt == 0 else 2)).reshape(M, -1),
                                        ref["fc2x_codes"],
                                        orc.tiled_to_compact(np_u8(aux["fc2x_scales"]), splits, N // (32 if fmt == 0 else 16)),
                                        ref["fc2x_scales"],
                                        g_S=None if fmt == 0 else np.repeat(
                                            [nvfp4_scale_of(a) for a in aux["fc2x_amax_pre"].cpu().numpy()], splits),
                                        o_S=None if fmt == 0 else np.repeat(ref["fc2x_S"], splits))
        assert frac >= CODE_MATCH and steps <= 1.0 + 1e-9, (frac, steps)
        assert frob(y.float().cpu().numpy(), orc.bf16_to_f64(ref["y"])) <= Y_TOL


@pytest.mark.parametrize("act", [0, 1], ids=["swiglu", "srelu"])
def test_forward_nvfp4_x4_scales_match_tiled(gm, act):
    """The GEMM reading replicated weight scales (one 128x256b tensor-memory copy
    per MMA) gives bit-identical outputs to the one reading GEMM_TILED scales,
    in single-CTA and CTA-pair mode."""
    rng = np.random.default_rng(21 + act)
    splits, K, N = [130, 0, 257, 5, 128, 700], 512, 512
    G, M = len(splits), sum(splits)
    n1 = 2 * N if act == 0 else N
    d = dict(x=bf16_cpu(rng.standard_normal((M, K))), splits=torch.tensor(splits, dtype=torch.int64),
             W1=bf16_cpu(rng.standard_normal((G, n1, K)) / np.sqrt(K)),
             W2=bf16_cpu(rng.standard_normal((G, K, N)) / np.sqrt(N)),
             probs=torch.from_numpy(rng.uniform(0, 1, M).astype(np.float32)))
    yt, at = run_gpu(gm, d, 1, act, mask=0x3C5A, x4=False)
    own = torch.from_numpy(tiled_index(splits, N // 16).reshape(-1)).cuda()
    for mode, x4 in ((0, True), (2, True), (2, False)):
        y4, a4 = run_gpu(gm, d, 1, act, mask=0x3C5A, x4=x4, gemm_mode=mode)
        assert np.array_equal(np_bits(y4), np_bits(yt)), (mode, x4)
        for key in ("fc2x_codes", "fc2x_amax_pre", "fc2x_amax_post"):
            assert torch.equal(a4[key], at[key]), (key, mode, x4)
        assert torch.equal(a4["fc2x_scales"][own], at["fc2x_scales"][own]), (mode, x4)
        assert torch.equal(a4["fc2x_bf16"].view(torch.int16), at["fc2x_bf16"].view(torch.int16)), (mode, x4)


@pytest.mark.parametrize("use_rht", [True, False])
def test_forward_nvfp4_columnwise_fc2x(orc, gm, use_rht):
    """The forward's optional columnwise NVFP4 fc2_x (no-recompute training
    path) on lossless operands (one-hot fc1 weights, x from {0, +-2, +-4},
    prob 1: fc2_x is exact, and so are its amaxes and every RHT value):
    bit-exact against the oracle's quantize-with-amax of the oracle forward's
    own fc2_x and amaxes; fc2's rowwise operand and y are unchanged by the
    extra output."""
    splits, K, N = [130, 0, 257, 5, 1, 128, 700], 512, 512
    G, M = len(splits), sum(splits)
    d = onehot_case(1, 1, splits, K, N, seed=31)
    mask = 0x5AC3
    y0, a0 = run_gpu(gm, d, 1, 1, mask=mask)
    w1 = gm.prepare_weights(d["W1"].cuda(), gm.NVFP4)
    w2 = gm.prepare_weights(d["W2"].cuda(), gm.NVFP4)
    ncol = N * (M + 16 * G)
    aux = {k: torch.zeros_like(v) for k, v in a0.items()}
    aux["fc2x_col_codes"] = torch.zeros(ncol // 2, dtype=torch.uint8, device="cuda")
    aux["fc2x_col_scales"] = torch.zeros(ncol // 16, dtype=torch.uint8, device="cuda")
    rec = gm.recipe(gm.NVFP4, use_rht=use_rht, mask=mask)
    y = torch.empty_like(y0)
    gm.forward(d["x"].cuda(), d["splits"].cuda(), w1, w2, d["probs"].cuda(), gm.SRELU, rec, y=y, aux=aux)
    gm.check_device_status()
    assert np.array_equal(np_bits(y), np_bits(y0))
    assert torch.equal(aux["fc2x_codes"], a0["fc2x_codes"]) and torch.equal(aux["fc2x_scales"], a0["fc2x_scales"])
    fwd = orc.forward(bits(d["x"]), np.array(splits), bits(d["W1"]), bits(d["W2"]), d["probs"].numpy(), 1, 1,
                      rht_mask=mask)
    assert np.array_equal(np_bits(aux["fc2x_bf16"]), fwd["fc2x"])             # the lossless premise
    assert np.array_equal(aux["fc2x_amax_pre"].cpu().numpy(), fwd["fc2x_amax_pre"])
    assert np.array_equal(aux["fc2x_amax_post"].cpu().numpy(), fwd["fc2x_amax_post"])
    ref = orc.group_quantize_with_amax(fwd["fc2x"], np.array(splits), orc.NVFP4, fwd["fc2x_amax_pre"],
                                       fwd["fc2x_amax_post"], rowwise=False, columnwise=True, use_rht=use_rht,
                                       mask=mask)
    nb = len(ref["col_codes"])
    assert np.array_equal(np_u8(aux["fc2x_col_codes"], nb), ref["col_codes"])
    assert np.array_equal(np_u8(aux["fc2x_col_scales"], len(ref["col_scales"])), ref["col_scales"])


@pytest.mark.parametrize("fmt", [0, 1], ids=["mxfp8", "nvfp4"])
def test_forward_biases_lossless_bitexact(orc, gm, fmt):
    """Per-expert fc1 and fc2 biases on lossless operands (SReLU): fc2_x codes
    and y bit-exact against the oracle, ragged and empty groups."""
    rng = np.random.default_rng(23 + fmt)
    splits, K, N = [130, 0, 257, 5, 128], 512, 256
    G, M = len(splits), sum(splits)
    offs = np.concatenate([[0], np.cumsum(splits)])
    xs, bs = ([0.0, 1, 2, -1, -2], [0.0, 0.0, 1.0, -1.0, 2.0]) if fmt == 0 else ([0.0, 2, -2], [0.0, 2.0])
    x = rng.choice(xs, size=(M, K))
    for g in range(G):
        if splits[g]:
            x[offs[g]] = 2.0
    W1 = np.zeros((G, N, K))
    for g in range(G):
        W1[g, np.arange(N), rng.integers(0, K, N)] = 1.0
    W2 = np.zeros((G, K, N))
    for g in range(G):
        W2[g, np.arange(K), rng.integers(0, N, K)] = rng.choice([1.0, -1.0, 2.0], K)
    b1 = rng.choice(bs, size=(G, N))
    b2 = rng.choice([0.0, 1.0, -2.0, 4.0], size=(G, K))
    xt, W1t, W2t = bf16_cpu(x), bf16_cpu(W1), bf16_cpu(W2)
    b1t, b2t = bf16_cpu(b1), bf16_cpu(b2)
    w1 = gm.prepare_weights(W1t.cuda(), fmt, bias=b1t.cuda())
    w2 = gm.prepare_weights(W2t.cuda(), fmt, bias=b2t.cuda())
    cdiv = 1 if fmt == 0 else 2
    aux = {"fc2x_codes": torch.zeros(M * N // cdiv + 16, dtype=torch.uint8, device="cuda")}
    y = gm.forward(xt.cuda(), torch.tensor(splits).cuda(), w1, w2, None, gm.SRELU, gm.recipe(fmt), aux=aux)
    gm.check_device_status()
    ref = orc.forward(bits(xt), np.array(splits), bits(W1t), bits(W2t), None, 1, fmt, b1=b1, b2=b2)
    assert np.array_equal(np_u8(aux["fc2x_codes"], M * N // cdiv).reshape(M, -1), ref["fc2x_codes"])
    assert np.array_equal(np_bits(y), ref["y"])


def test_forward_swiglu_bias_follows_the_interleave(orc, gm):
    """fc1 bias given in logical gate/up order reaches the right accumulator
    columns of the interleaved W1 (MXFP8 SwiGLU, random data, tolerance)."""
    rng = np.random.default_rng(29)
    splits, K, N = [130, 0, 257, 5, 128], 512, 256
    G, M = len(splits), sum(splits)
    d = dict(x=bf16_cpu(rng.standard_normal((M, K))), splits=torch.tensor(splits, dtype=torch.int64),
             W1=bf16_cpu(rng.standard_normal((G, 2 * N, K)) / np.sqrt(K)),
             W2=bf16_cpu(rng.standard_normal((G, K, N)) / np.sqrt(N)),
             probs=torch.from_numpy(rng.uniform(0, 1, M).astype(np.float32)))
    b1 = bf16_cpu(rng.standard_normal((G, 2 * N)))
    b2 = bf16_cpu(rng.standard_normal((G, K)) * 0.1)
    w1 = gm.prepare_weights(d["W1"].cuda(), gm.MXFP8, swiglu_interleave=True, bias=b1.cuda())
    w2 = gm.prepare_weights(d["W2"].cuda(), gm.MXFP8, bias=b2.cuda())
    aux = {"fc2x_codes": torch.zeros(M * N + 16, dtype=torch.uint8, device="cuda"),
           "fc2x_scales": torch.zeros(gm.tiled_scales_bytes(M, G, N // 32) + 16, dtype=torch.uint8, device="cuda")}
    y = gm.forward(d["x"].cuda(), d["splits"].cuda(), w1, w2, d["probs"].cuda(), gm.SWIGLU, gm.recipe(gm.MXFP8),
                   aux=aux)
    gm.check_device_status()
    ref = orc.forward(bits(d["x"]), np.array(splits), bits(d["W1"]), bits(d["W2"]), d["probs"].numpy(), 0, 0,
                      b1=orc.bf16_to_f64(bits(b1)), b2=orc.bf16_to_f64(bits(b2)))
    frac, steps = code_match_report(0, np_u8(aux["fc2x_codes"], M * N).reshape(M, -1), ref["fc2x_codes"],
                                    orc.tiled_to_compact(np_u8(aux["fc2x_scales"]), splits, N // 32),
                                    ref["fc2x_scales"])
    assert frac >= CODE_MATCH and steps <= 1.0 + 1e-9, (frac, steps)
    assert frob(y.float().cpu().numpy(), orc.bf16_to_f64(ref["y"])) <= Y_TOL


@pytest.mark.parametrize("fmt,swiglu", [(0, True), (1, False)], ids=["mxfp8-swiglu", "nvfp4"])
def test_prepare_weights_discrete_matches_stacked(gm, fmt, swiglu):
    """One device pointer per expert gives the stacked preparation's bytes."""
    rng = np.random.default_rng(37)
    G, rows, cols = 3, 512, 512
    W = bf16_cpu(rng.standard_normal((G, rows, cols)) * np.array([1.0, 1e-3, 30.0])[:, None, None]).cuda()
    x4 = fmt == 1
    a = gm.prepare_weights(W, fmt, swiglu_interleave=swiglu, x4=x4)
    b = gm.prepare_weights([W[g].clone() for g in range(G)], fmt, swiglu_interleave=swiglu, x4=x4)
    gm.check_device_status()
    assert torch.equal(a.codes, b.codes)
    used = G * rows // 128 * (cols // (32 if fmt == 0 else 16) // 4) * 512
    assert torch.equal(a.scales[:used], b.scales[:used])
    if fmt == 1:
        assert torch.equal(a.global_scale, b.global_scale) and torch.equal(a.amax, b.amax)
        assert torch.equal(a.scales_x4, b.scales_x4)


def test_replicate_weight_scales_bitexact(orc, gm):
    rng = np.random.default_rng(4)
    G, rows, cols = 3, 512, 768
    W = bf16_cpu(rng.standard_normal((G, rows, cols)))
    q = gm.prepare_weights(W.cuda(), gm.NVFP4, x4=True)
    gm.check_device_status()
    tiled = np_u8(q.scales)
    want = orc.tiled_to_x4(tiled, G * rows // 256, cols // 64)
    assert np.array_equal(np_u8(q.scales_x4), want)


def forward_parity(orc, gm, name, rows=None, gemm_mode=0):
    d = make_inputs(name)
    w = d["workload"]
    splits = d["splits"].numpy()
    y, aux = run_gpu(gm, d, w.fmt, w.act, mask=d["mask"], gemm_mode=gemm_mode, tanh_c=w.tanh_clamp_scale)
    ref = orc.forward(bits(d["x"]), splits, bits(d["W1"]), bits(d["W2"]), d["probs"].numpy(), w.act, w.fmt,
                      rows=rows, rht_mask=d["mask"], tanh_clamp_scale=w.tanh_clamp_scale)
    sel = ref["rows"]
    cdiv, blk = (1, 32) if w.fmt == 0 else (2, 16)
    g_codes = np_u8(aux["fc2x_codes"], w.M * w.N // cdiv).reshape(w.M, -1)
    g_scales = orc.tiled_to_compact(np_u8(aux["fc2x_scales"]), splits, w.N // blk)
    gS = oS = None
    if w.fmt == 1:
        gpre = aux["fc2x_amax_pre"].cpu().numpy()
        gS = np.repeat([nvfp4_scale_of(a) for a in gpre], splits)
        oS = np.repeat(ref["fc2x_S"], splits)
    frac, steps = code_match_report(w.fmt, g_codes, ref["fc2x_codes"], g_scales, ref["fc2x_scales"], gS, oS, rows=sel)
    err = frob(y.float().cpu().numpy()[sel], orc.bf16_to_f64(ref["y"])[sel])
    print(f"{name}: code match {frac:.6f} (max {steps:.2f} steps), y error {err:.3e}")
    assert frac >= CODE_MATCH, frac
    assert steps <= 1.0 + 1e-9, steps
    assert err <= Y_TOL, err
    return d, y, aux, ref


def test_forward_tiny(orc, gm):
    forward_parity(orc, gm, "tiny")


def test_forward_mx_swiglu_full(orc, gm):
    forward_parity(orc, gm, "mx_swiglu")


@pytest.mark.parametrize("name", ["mx_swiglu", "nv_srelu"])
def test_forward_cta_pair_mode(orc, gm, name):
    """The CTA-pair GEMM mode (cta_group::2, 256 x 256 tiles) on full workloads."""
    forward_parity(orc, gm, name, gemm_mode=2)


def test_forward_nv_srelu_full(orc, gm):
    d, y, aux, ref = forward_parity(orc, gm, "nv_srelu")
    # amax of fc2_x: the oracle's from its own fc2_x; relative agreement
    np.testing.assert_allclose(aux["fc2x_amax_pre"].cpu().numpy(), ref["fc2x_amax_pre"], rtol=2e-2)
    np.testing.assert_allclose(aux["fc2x_amax_post"].cpu().numpy(), ref["fc2x_amax_post"], rtol=2e-2)


def test_forward_nv_tanh_srelu_full(orc, gm):
    """NVFP4 + RHT tanh-SReLU on the nv_srelu inputs (soft-clamp scale 8)."""
    d, y, aux, ref = forward_parity(orc, gm, "nv_tanh_srelu")
    np.testing.assert_allclose(aux["fc2x_amax_pre"].cpu().numpy(), ref["fc2x_amax_pre"], rtol=2e-2)
    assert aux["fc2x_amax_pre"].max().item() <= 8.0   # the clamp bounds fc2_x by c (probs <= 1)


@pytest.mark.parametrize("fmt", [0, 1], ids=["mxfp8", "nvfp4"])
def test_forward_tanh_srelu_small(orc, gm, fmt):
    """tanh-SReLU on ragged groups, clamp scale 0.5 so most outputs are clamped."""
    rng = np.random.default_rng(41 + fmt)
    splits, K, N = [130, 0, 257, 5, 1, 128], 512, 512
    G, M = len(splits), sum(splits)
    d = dict(x=bf16_cpu(rng.standard_normal((M, K))), splits=torch.tensor(splits, dtype=torch.int64),
             W1=bf16_cpu(rng.standard_normal((G, N, K)) / np.sqrt(K)),
             W2=bf16_cpu(rng.standard_normal((G, K, N)) / np.sqrt(N)),
             probs=torch.from_numpy(rng.uniform(0, 1, M).astype(np.float32)))
    y, aux = run_gpu(gm, d, fmt, 2, mask=0x1357, tanh_c=0.5)
    ref = orc.forward(bits(d["x"]), np.array(splits), bits(d["W1"]), bits(d["W2"]), d["probs"].numpy(), 2, fmt,
                      rht_mask=0x1357, tanh_clamp_scale=0.5)
    cdiv, blk = (1, 32) if fmt == 0 else (2, 16)
    gS = oS = None
    if fmt == 1:
        gS = np.repeat([nvfp4_scale_of(a) for a in aux["fc2x_amax_pre"].cpu().numpy()], splits)
        oS = np.repeat(ref["fc2x_S"], splits)
    frac, steps = code_match_report(fmt, np_u8(aux["fc2x_codes"], M * N // cdiv).reshape(M, -1), ref["fc2x_codes"],
                                    orc.tiled_to_compact(np_u8(aux["fc2x_scales"]), splits, N // blk),
                                    ref["fc2x_scales"], gS, oS)
    assert frac >= CODE_MATCH and steps <= 1.0 + 1e-9, (frac, steps)
    assert frob(y.float().cpu().numpy(), orc.bf16_to_f64(ref["y"])) <= Y_TOL


def test_forward_mx_skew_sampled(orc, gm):
    """Zipf-skewed 64 experts at full size; the oracle evaluates a row sample that
    covers every non-empty expert (MXFP8 rows are independent)."""
    w = WORKLOADS["mx_skew"]
    from mxfp8_nvfp4_block_gb300.inputs import make_splits
    s = make_splits(w)
    offs = np.concatenate([[0], np.cumsum(s)])
    rng = np.random.default_rng(0)
    rows = []
    for g in range(w.G):
        if s[g]:
            rows += [offs[g], offs[g + 1] - 1]
            rows += list(rng.integers(offs[g], offs[g + 1], min(8, s[g])))
    rows = np.unique(np.array(rows, dtype=np.int64))
    forward_parity(orc, gm, "mx_skew", rows=rows)


@pytest.mark.parametrize("act", [1, 2], ids=["srelu", "tanh_srelu"])
def test_fused_amax_equals_standalone_hadamard_amax(orc, gm, act):
    """The NVFP4 fc1 epilogue's (pre, post)-RHT amax of fc2_x is bit-identical to
    the standalone group Hadamard-amax pass over the bf16 fc2_x it stored (the
    pages check this for SReLU, tanh-SReLU and SwiGLU)."""
    d = make_inputs("tiny")
    d["W1"] = d["W1"][:, :256].contiguous()      # SReLU: W1 [G, N, K]
    _, aux = run_gpu(gm, d, 1, act, mask=0x9C31, tanh_c=0.5)
    pre, post = gm.group_hadamard_amax(aux["fc2x_bf16"], d["splits"].cuda(), 0x9C31)
    assert torch.equal(pre, aux["fc2x_amax_pre"])
    assert torch.equal(post, aux["fc2x_amax_post"])


def test_sign_mask_changes_post_rht_amax(orc, gm):
    """SReLU-shaped fc2_x (non-negative): the plain transform's amax exceeds the
    sign-masked one (the pages saw up to ~17% for SReLU activations)."""
    d = make_inputs("tiny")
    d["W1"] = d["W1"][:, :256].contiguous()
    _, aux = run_gpu(gm, d, 1, 1, mask=0x9C31)
    pre0, post0 = gm.group_hadamard_amax(aux["fc2x_bf16"], d["splits"].cuda(), 0)
    ratio = (post0 / aux["fc2x_amax_post"]).cpu().numpy()
    print("plain / masked post-RHT amax:", ratio)
    assert (ratio > 1.0).all()


def test_forward_no_probs_and_empty_groups(orc, gm):
    splits = [0, 300, 0, 0, 212]
    rng = np.random.default_rng(5)
    M, K, N, G = sum(splits), 256, 256, len(splits)
    d = dict(x=bf16_cpu(rng.standard_normal((M, K))), splits=torch.tensor(splits),
             W1=bf16_cpu(rng.standard_normal((G, 2 * N, K)) / 16), W2=bf16_cpu(rng.standard_normal((G, K, N)) / 16),
             probs=torch.ones(M))
    y, aux = run_gpu(gm, d, 0, 0, probs=False)
    ref = orc.forward(bits(d["x"]), np.array(splits), bits(d["W1"]), bits(d["W2"]), None, 0, 0)
    assert frob(y.float().cpu().numpy(), orc.bf16_to_f64(ref["y"])) <= Y_TOL


def test_forward_rows_past_splits_untouched(gm):
    """Rows past sum(split_sizes) (here M is larger) keep their contents."""
    rng = np.random.default_rng(6)
    splits = [100, 60]
    M, K, N, G = 256, 256, 256, 2
    d = dict(x=bf16_cpu(rng.standard_normal((M, K))), splits=torch.tensor(splits),
             W1=bf16_cpu(rng.standard_normal((G, 2 * N, K)) / 16), W2=bf16_cpu(rng.standard_normal((G, K, N)) / 16),
             probs=torch.rand(M))
    y, _ = run_gpu(gm, d, 0, 0)
    assert torch.isnan(y[160:].float()).all()
    assert not torch.isnan(y[:160].float()).any()
