"""Oracle pins drawn from facts the pages state with numbers (fixtures in
tests/golden/, each naming its source) (CPU)."""
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name: str) -> dict:
    """`key value...` lines of a fixture; '#' starts a comment."""
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            tok = line.split("#", 1)[0].split()
            if tok:
                vals[tok[0]] = [float(v) if "." in v else int(v) for v in tok[1:]]
    return vals


def as_bits(a):
    return torch.from_numpy(np.asarray(a, np.float64).astype(np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def test_sign_mask_post_rht_amax_of_srelu_shaped_activations(orc):
    """For a non-negative column chunk v (an SReLU output) no signed sum exceeds
    the plain one, |sum_i H_ji s_i v_i| <= sum_i v_i = (H v)_0, so the plain
    transform's post-RHT amax is a quarter of the largest 16-row column-chunk
    sum and bounds every sign-masked amax from above.  The gap is the error
    of the global scale S = 448*6 / amax that taking the amax without the
    mask causes; the pages put it at up to roughly 17% on their activations,
    and i.i.d. relu(h)^2 data lands in the same range."""
    bound = read_golden("sign_mask_amax.txt")["max_global_scale_error"][0]
    rng = np.random.default_rng(17)
    splits = np.array([512, 0, 400, 512])
    M, K = int(splits.sum()), 512
    xb = as_bits(np.maximum(rng.standard_normal((M, K)), 0.0) ** 2)
    v = orc.bf16_to_f64(xb)
    offs = orc.group_offsets(splits)
    _, plain = orc.group_hadamard_amax(xb, splits, 0)
    for g in range(len(splits)):
        m = int(splits[g])
        if m == 0:
            assert plain[g] == 0
            continue
        blk = np.vstack([v[offs[g]:offs[g + 1]], np.zeros((-m % 16, K))])
        np.testing.assert_allclose(plain[g], 0.25 * blk.reshape(-1, 16, K).sum(axis=1).max(), rtol=1e-6)
    nz = splits > 0
    errs = []
    for _ in range(8):
        mask = int(rng.integers(1, 1 << 16))
        _, masked = orc.group_hadamard_amax(xb, splits, mask)
        assert np.all(plain[nz] >= masked[nz] * (1 - 1e-6)), mask     # FP32 sums: a rounding at most
        errs.append(plain[nz].astype(np.float64) / masked[nz] - 1.0)   # S_masked / S_plain - 1
    worst = float(np.max(errs))
    print(f"largest global-scale error of an unmasked amax: {worst:.3f} (pages: up to ~{bound})")
    assert 0.25 * bound <= worst <= 2.0 * bound


def test_ragged_split_from_the_review_is_supported(orc):
    """The review's split [64, 65] (129 tokens, not a multiple of 128): the
    second group's rows start a new 128-row scale tile at its own first row,
    and the lossless MXFP8 SReLU forward equals the plain float64 MLP."""
    splits = np.array(read_golden("ragged_split.txt")["splits"])
    assert list(splits) == [64, 65]
    idx = orc.tiled_index(splits, 4)
    assert idx[64, 0] == 512 and idx[63, 0] == (63 % 32) * 16 + (63 // 32) * 4
    rng = np.random.default_rng(5)
    G, K, N = 2, 64, 64
    M = int(splits.sum())
    offs = orc.group_offsets(splits)
    x = rng.choice([0.0, 1, 2, 4, -1, -2, -4], size=(M, K))
    probs = rng.choice([0.5, 1.0], size=M).astype(np.float32)
    W1 = np.zeros((G, N, K))
    perms = [rng.integers(0, K, N) for _ in range(G)]
    for g in range(G):
        W1[g, np.arange(N), perms[g]] = 1.0
    W2 = rng.choice([0.0, 1, 2, -1, -2, 4, -4], size=(G, K, N))
    out = orc.forward(as_bits(x), splits, as_bits(W1), as_bits(W2), probs, orc.SRELU, orc.MXFP8)
    for g in range(G):
        sl = slice(offs[g], offs[g + 1])
        f = np.maximum(x[sl][:, perms[g]], 0) ** 2 * probs[sl, None].astype(np.float64)
        assert np.array_equal(out["fc2x"][sl], as_bits(f))
        assert np.array_equal(out["y"][sl], as_bits(f @ W2[g].T)), g
