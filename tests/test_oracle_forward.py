"""Pins of the oracle's forward (CPU only).

With operands whose quantisation is lossless, the quantised forward reduces to
a plain float64 MLP computed with numpy, exactly.  One-hot fc1 weights make
every index mistake visible: a wrong expert, a transposed weight, swapped
SwiGLU halves or a misplaced routing prob all change the result.
"""
import numpy as np
import pytest
import torch

from mxfp8_nvfp4_block_gb300.inputs import bits, make_inputs


def bf16_of(v64):
    """Reference bf16 rounding of exactly-float-representable values (torch)."""
    return torch.from_numpy(np.asarray(v64, np.float64).astype(np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def as_bits(a):
    return bf16_of(np.asarray(a, np.float64))


def onehot_w1(rng, G, n1, K):
    W = np.zeros((G, n1, K))
    perms = []
    for g in range(G):
        p = rng.integers(0, K, n1)
        W[g, np.arange(n1), p] = 1.0
        perms.append(p)
    return W, perms


@pytest.mark.parametrize("fmt_name", ["mxfp8", "nvfp4"])
def test_srelu_forward_lossless_equals_plain_mlp(orc, fmt_name):
    fmt = orc.MXFP8 if fmt_name == "mxfp8" else orc.NVFP4
    rng = np.random.default_rng(11)
    G, K, N = 4, 64, 64
    splits = np.array([9, 0, 33, 5])
    M = splits.sum()
    offs = np.concatenate([[0], np.cumsum(splits)])
    if fmt == orc.MXFP8:
        x = rng.choice([0.0, 1, 2, 4, -1, -2, -4], size=(M, K))
        probs = rng.choice([0.5, 1.0], size=M).astype(np.float32)
    else:
        x = rng.choice([0.0, 2, 4, -2, -4], size=(M, K))
        probs = np.ones(M, np.float32)
        for g in range(G):
            if splits[g]:
                x[offs[g]] = 4.0     # group amax of x = 4, and an fc1 output row of 4s
    W1, perms = onehot_w1(rng, G, N, K)
    W2 = rng.choice([0.0, 1, 2, -1, -2, 4, -4], size=(G, K, N))
    W2[:, 0, 0] = 4.0
    out = orc.forward(as_bits(x), splits, as_bits(W1), as_bits(W2), probs, orc.SRELU, fmt)
    for g in range(G):
        sl = slice(offs[g], offs[g + 1])
        h = x[sl][:, perms[g]]
        f = np.maximum(h, 0) ** 2 * probs[sl, None].astype(np.float64)
        assert np.array_equal(out["fc2x"][sl], bf16_of(f))
        y = f @ W2[g].T
        assert np.array_equal(out["y"][sl], bf16_of(y)), g


def test_swiglu_forward_gate_up_order_and_prob(orc):
    rng = np.random.default_rng(12)
    G, K, N = 3, 64, 64
    splits = np.array([20, 7, 0])
    M = splits.sum()
    offs = np.concatenate([[0], np.cumsum(splits)])
    x = rng.choice([0.0, 1, 2, 4, -1, -2, -4], size=(M, K))
    probs = rng.uniform(0, 1, M).astype(np.float32)
    W1, perms = onehot_w1(rng, G, 2 * N, K)
    W2 = rng.standard_normal((G, K, N)) / 8
    W2b = orc.bf16_to_f64(as_bits(W2))
    out = orc.forward(as_bits(x), splits, as_bits(W1), as_bits(W2), probs, orc.SWIGLU, orc.MXFP8)
    for g in range(2):
        sl = slice(offs[g], offs[g + 1])
        h = x[sl][:, perms[g]]                      # exact fc1 output
        gate, up = h[:, :N], h[:, N:]
        a = gate / (1 + np.exp(-gate)) * up * probs[sl, None].astype(np.float64)
        f = orc.bf16_to_f64(bf16_of(a))
        assert np.array_equal(out["fc2x"][sl], bf16_of(a))
        y_dense = f @ W2b[g].T                       # fc2 without the fc2_x quantisation
        y = orc.bf16_to_f64(out["y"][sl])
        rel = np.linalg.norm(y - y_dense) / np.linalg.norm(y_dense)
        assert rel < 0.05, rel
        a_sw = up / (1 + np.exp(-up)) * gate * probs[sl, None]   # halves swapped
        assert np.linalg.norm(orc.bf16_to_f64(bf16_of(a_sw)) - f) / np.linalg.norm(f) > 0.3


def test_nvfp4_forward_close_to_dense_mlp(orc):
    """Random operands: the NVFP4 forward stays within quantisation noise of the
    unquantised float64 MLP; the per-group scales (alpha) are applied."""
    rng = np.random.default_rng(13)
    G, K, N = 3, 128, 128
    splits = np.array([70, 0, 58])
    M = splits.sum()
    offs = np.concatenate([[0], np.cumsum(splits)])
    x = rng.standard_normal((M, K)) * 3
    W1 = rng.standard_normal((G, N, K)) / np.sqrt(K) * np.array([1, 10, 0.1])[:, None, None]
    W2 = rng.standard_normal((G, K, N)) / np.sqrt(K)
    probs = rng.uniform(0, 1, M).astype(np.float32)
    xb, W1b, W2b = as_bits(x), as_bits(W1), as_bits(W2)
    out = orc.forward(xb, splits, W1b, W2b, probs, orc.SRELU, orc.NVFP4)
    xf, W1f, W2f = (orc.bf16_to_f64(t) for t in (xb, W1b, W2b))
    for g in (0, 2):
        sl = slice(offs[g], offs[g + 1])
        h = xf[sl] @ W1f[g].T
        y = (np.maximum(h, 0) ** 2 * probs[sl, None]) @ W2f[g].T
        got = orc.bf16_to_f64(out["y"][sl])
        rel = np.linalg.norm(got - y) / np.linalg.norm(y)
        assert rel < 0.3, (g, rel)
    assert out["fc2x_S"][1] == 1.0 and out["x_amax"][1] == 0.0


def test_forward_row_subset_matches_full(orc):
    d = make_inputs("tiny")
    args = (bits(d["x"]), d["splits"].numpy(), bits(d["W1"]), bits(d["W2"]), d["probs"].numpy(),
            orc.SWIGLU, orc.MXFP8)
    full = orc.forward(*args)
    rows = np.array([0, 5, 199, 200, 349, 350, 511])
    part = orc.forward(*args, rows=rows)
    assert np.array_equal(part["y"][rows], full["y"][rows])
    assert np.array_equal(part["fc2x_codes"][rows], full["fc2x_codes"][rows])


def test_tanh_srelu_activation_closed_forms(orc):
    """c * tanh(max(h,0)^2 / c): zero for h <= 0; the SReLU value while h^2 << c
    (tanh z = z - z^3/3 + ...); exactly c once tanh saturates in float64; c/2 at
    h^2 = c * atanh(1/2); increasing in h and below c."""
    c = 8.0
    h = np.array([[-3.0, -0.0, 0.0, 1e-3, 100.0, np.sqrt(c * np.arctanh(0.5))]])
    y = orc.activation(h, orc.TANH_SRELU, c)[0]
    assert y[0] == 0.0 and y[1] == 0.0 and y[2] == 0.0
    assert abs(y[3] / 1e-6 - 1.0) < 1e-12
    assert y[4] == c
    assert abs(y[5] - c / 2) < 1e-12
    hs = np.linspace(0, 6, 1001)[None, :]
    ys = orc.activation(hs, orc.TANH_SRELU, c)[0]
    assert np.all(np.diff(ys) > 0) and ys.max() < c
    # the clamp only acts on large outputs: equal to SReLU within the cubic term
    sr = orc.activation(hs, orc.SRELU)[0]
    assert np.all(np.abs(ys - sr) <= sr ** 3 / (3 * c * c) + 1e-15)


def test_tanh_srelu_forward_reduces_to_srelu_for_a_huge_clamp(orc):
    """With c = 1e30 the clamp is the identity to far below bf16 resolution, so
    the whole forward (activation, x prob, bf16, fc2_x quantisation, fc2) gives
    SReLU's bytes: the tanh branch is wired in the same place."""
    d = make_inputs("tiny")
    x, W1, W2 = bits(d["x"]), bits(d["W1"]), bits(d["W2"])
    splits = d["splits"].numpy()
    G, N = len(splits), W2.shape[2]
    W1s = W1[:, :N, :]                    # SReLU / tanh-SReLU take N fc1 rows
    for fmt in (orc.MXFP8, orc.NVFP4):
        a = orc.forward(x, splits, W1s, W2, d["probs"].numpy(), orc.SRELU, fmt)
        b = orc.forward(x, splits, W1s, W2, d["probs"].numpy(), orc.TANH_SRELU, fmt, tanh_clamp_scale=1e30)
        assert np.array_equal(a["fc2x"], b["fc2x"]) and np.array_equal(a["y"], b["y"])


@pytest.mark.parametrize("fmt_name", ["mxfp8", "nvfp4"])
def test_biases_enter_before_rounding_exactly(orc, fmt_name):
    """Integer biases on lossless operands: fc2_x = bf16((h + b1)^2 * prob) and
    y = bf16(f @ W2^T + b2) exactly, for every group (fc1 bias before the
    activation, fc2 bias before the output rounding)."""
    fmt = orc.MXFP8 if fmt_name == "mxfp8" else orc.NVFP4
    rng = np.random.default_rng(17)
    G, K, N = 3, 64, 64
    splits = np.array([7, 0, 12])
    M = splits.sum()
    offs = np.concatenate([[0], np.cumsum(splits)])
    # operand sets kept exactly representable through both formats (NVFP4: h + b1
    # in {0, +-2, 4} so fc2_x in {0, 4, 16})
    xs, bs = ([0.0, 1, 2, -1, -2], [0.0, 0.0, 1.0, -1.0, 2.0]) if fmt == orc.MXFP8 else ([0.0, 2, -2], [0.0, 2.0])
    x = rng.choice(xs, size=(M, K))
    for g in range(G):
        if splits[g]:
            x[offs[g]] = 2.0
    W1, perms = onehot_w1(rng, G, N, K)
    b1 = rng.choice(bs, size=(G, N))
    W2 = np.zeros((G, K, N))
    for g in range(G):
        W2[g, np.arange(K), rng.integers(0, N, K)] = rng.choice([1.0, -1.0, 2.0], K)
    b2 = rng.choice([0.0, 1.0, -2.0, 4.0], size=(G, K))
    probs = np.ones(M, np.float32)
    out = orc.forward(as_bits(x), splits, as_bits(W1), as_bits(W2), probs, orc.SRELU, fmt, b1=b1, b2=b2)
    for g in range(G):
        sl = slice(offs[g], offs[g + 1])
        f = np.maximum(x[sl][:, perms[g]] + b1[g], 0) ** 2
        assert np.array_equal(out["fc2x"][sl], bf16_of(f)), g
        assert np.array_equal(out["y"][sl], bf16_of(f @ W2[g].T + b2[g])), g


@pytest.mark.parametrize("act", [0, 1], ids=["swiglu", "srelu"])
def test_dact_matches_finite_differences(orc, act):
    """The backward's activation derivatives against central differences of the
    forward activation (an independent evaluation of the same function)."""
    rng = np.random.default_rng(5)
    n = 64
    h = rng.standard_normal((4, 2 * n if act == 0 else n)) * 3
    if act == 1:
        h[np.abs(h) < 1e-3] = 0.5          # keep away from the kink at 0
    d0, d1 = orc.dact(h, act)
    eps = 1e-6
    if act == 0:
        for part, d in ((slice(0, n), d0), (slice(n, 2 * n), d1)):
            hp, hm = h.copy(), h.copy()
            hp[:, part] += eps
            hm[:, part] -= eps
            fd = (orc.activation(hp, act) - orc.activation(hm, act)) / (2 * eps)
            np.testing.assert_allclose(d, fd, rtol=1e-6, atol=1e-8)
    else:
        fd = (orc.activation(h + eps, act) - orc.activation(h - eps, act)) / (2 * eps)
        np.testing.assert_allclose(d0, fd, rtol=1e-6, atol=1e-8)


def test_backward_dgrad_lossless_equals_plain_backprop(orc):
    """SReLU with small-integer operands and one-hot weights: every step of the
    data-gradient backward is exact, so it equals plain float64 backprop:
    dfc2x = dy W2, dh = dfc2x * 2 relu(h), dx = dh W1, dprob = sum dfc2x relu(h)^2."""
    rng = np.random.default_rng(9)
    G, K, N = 3, 64, 64
    splits = np.array([5, 0, 9])
    M = splits.sum()
    offs = np.concatenate([[0], np.cumsum(splits)])
    dy = rng.choice([0.0, 1.0, -1.0], size=(M, K))
    W2 = np.zeros((G, K, N))
    W1 = np.zeros((G, N, K))
    for g in range(G):
        W2[g, rng.integers(0, K, N), np.arange(N)] = 1.0     # each fc2_x column reads one output row
        W1[g, np.arange(N), rng.integers(0, K, N)] = 1.0
    h = rng.choice([0.0, 1.0, -1.0, 2.0], size=(M, N))
    out = orc.backward_dgrad(as_bits(dy), splits, as_bits(W1), as_bits(W2), as_bits(h), None, orc.SRELU)
    for g in range(G):
        sl = slice(offs[g], offs[g + 1])
        d = dy[sl] @ W2[g]
        dh = d * 2 * np.maximum(h[sl], 0)
        assert np.array_equal(out["dfc2x"][sl], bf16_of(d))
        assert np.array_equal(out["fc1_dy"][sl], bf16_of(dh))
        assert np.array_equal(out["dx"][sl], bf16_of(dh @ W1[g])), g
        np.testing.assert_array_equal(out["dprob"][sl], (d * np.maximum(h[sl], 0) ** 2).sum(axis=1))


def test_backward_dgrad_row_sample_matches_full(orc):
    """Each row of dx, dprob and fc1_dy depends only on its own dy and h rows
    and its expert's weights (every MXFP8 block lies along a row), so the
    oracle's backward over a row sample, regrouped with the sample's split
    sizes, equals the full backward on those rows: the basis of the sampled
    full-size parity test."""
    d = make_inputs("tiny")
    rng = np.random.default_rng(33)
    M, K = d["x"].shape
    n1 = d["W1"].shape[1]
    dy = as_bits(rng.standard_normal((M, K)).astype(np.float32).astype(np.float64))
    h = as_bits((1.5 * rng.standard_normal((M, n1))).astype(np.float32).astype(np.float64))
    sp = d["splits"].numpy()
    probs = d["probs"].numpy()
    full = orc.backward_dgrad(dy, sp, bits(d["W1"]), bits(d["W2"]), h, probs, orc.SWIGLU)
    offs = orc.group_offsets(sp)
    rows = np.array([0, 5, 199, 200, 349, 350, 449, 450, 511])
    sub = np.array([np.count_nonzero((rows >= offs[g]) & (rows < offs[g + 1])) for g in range(len(sp))])
    part = orc.backward_dgrad(dy[rows], sub, bits(d["W1"]), bits(d["W2"]), h[rows], probs[rows], orc.SWIGLU)
    for k in ("dx", "fc1_dy", "fc1_dy_codes", "fc1_dy_scales", "dprob"):
        assert np.array_equal(part[k], full[k][rows]), k
