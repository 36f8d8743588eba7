"""Pins of the oracle's weight-gradient backward (columnwise MXFP8 operands and
grouped wgrad GEMMs) against closed forms and brute force (CPU)."""
import numpy as np
import torch


def as_bits(a):
    """bf16 bits of exactly representable values (torch rounding)."""
    return torch.from_numpy(np.asarray(a, np.float64).astype(np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def test_colwise_blocks_run_along_the_tokens_of_each_group(orc):
    """x[t, c] = s_c 2^(j + c mod 3), j = the 32-token block of t counted from
    its group's first token: every block along the tokens holds one magnitude,
    so its E8M0 byte is (j + c mod 3) - 8 + 127 and every code is E4M3(+-256) =
    0x78 | sign; tokens past a group's end are zero codes and a block with no
    tokens has byte 0.  Blocks taken along the columns, or counted from row 0
    of x, give other bytes."""
    splits = np.array([40, 0, 70, 128])
    C = 12
    offs = orc.group_offsets(splits)
    x = np.zeros((int(offs[-1]), C))
    sign = np.where(np.arange(C) % 2 == 0, 1.0, -1.0)
    for g in range(len(splits)):
        for t in range(offs[g], offs[g + 1]):
            j = (t - offs[g]) // 32
            x[t] = sign * 2.0 ** (j + np.arange(C) % 3)
    codes, scales = orc.mxfp8_colwise(as_bits(x), splits)
    pofs = orc.padded_offsets(splits)
    assert list(pofs) == [0, 128, 128, 256, 384]
    assert codes.shape == (C, 384) and scales.shape == (C, 12)
    for g in range(len(splits)):
        m = int(splits[g])
        for c in range(C):
            seg = codes[c, pofs[g]:pofs[g + 1]]
            want = 0x78 | (0x80 if sign[c] < 0 else 0)
            assert np.all(seg[:m] == want) and np.all(seg[m:] == 0), (g, c)
            for jb in range((pofs[g + 1] - pofs[g]) // 32):
                byte = scales[c, pofs[g] // 32 + jb]
                expect = (jb + c % 3) - 8 + 127 if 32 * jb < m else 0
                assert byte == expect, (g, c, jb)


def _loops_matmul_t(a, b):
    """sum_t a[t, i] b[t, j] by explicit loops (float64)."""
    out = np.zeros((a.shape[1], b.shape[1]))
    for t in range(a.shape[0]):
        for i in range(a.shape[1]):
            if a[t, i] != 0.0:
                for j in range(b.shape[1]):
                    out[i, j] += a[t, i] * b[t, j]
    return out


def test_wgrad_lossless_equals_brute_force():
    """SReLU, operands from {0, +-1, +-2, +-4} and probs from {1, 0.5}: every
    columnwise MXFP8 block is exact (block max 1, 2 or 4), so the weight
    gradients equal plain float64 sums over each expert's tokens, computed here
    by loops: dW2_g[k, n] = sum_t dy[t, k] relu(h)^2 p, dW1_g[j, k] = sum_t
    fc1_dy[t, j] x[t, k], and the bias gradients the token sums.  An empty
    expert gets zeros; K != N1 fixes the orientation of each gradient."""
    import oracle as orc

    rng = np.random.default_rng(21)
    splits = np.array([40, 0, 70])
    K, N = 48, 16
    offs = orc.group_offsets(splits)
    M = int(offs[-1])
    x = rng.choice([0.0, 1.0, -1.0], size=(M, K))
    dy = rng.choice([0.0, 1.0, -1.0, 2.0, -2.0], size=(M, K))
    h = rng.choice([0.0, 1.0, -1.0, 2.0], size=(M, N))
    fc1_dy = rng.choice([0.0, 1.0, -4.0, 2.0], size=(M, N))
    probs = rng.choice([1.0, 0.5], size=M).astype(np.float32)
    out = orc.backward_wgrad(as_bits(x), as_bits(dy), as_bits(h), probs, as_bits(fc1_dy), splits, orc.SRELU)
    fc2x = np.maximum(h, 0.0) ** 2 * probs[:, None]
    assert out["dW2"].shape == (3, K, N) and out["dW1"].shape == (3, N, K)
    for g in range(3):
        sl = slice(offs[g], offs[g + 1])
        np.testing.assert_array_equal(out["dW2"][g], _loops_matmul_t(dy[sl], fc2x[sl]))
        np.testing.assert_array_equal(out["dW1"][g], _loops_matmul_t(fc1_dy[sl], x[sl]))
        np.testing.assert_array_equal(out["dbias1"][g], fc1_dy[sl].sum(axis=0))
        np.testing.assert_array_equal(out["dbias2"][g], dy[sl].sum(axis=0))
    assert not out["dW2"][1].any() and not out["dW1"][1].any()


def test_recompute_fc2x_swiglu_closed_form(orc):
    """SwiGLU fc2_x from h = [gate | up]: gate 0 gives silu 0; gate 2, up 1,
    prob 1 gives bf16(2 / (1 + e^-2))."""
    h = np.array([[0.0, 2.0, 3.0, 1.0]])
    f = orc.recompute_fc2x(as_bits(h), np.array([1.0]), orc.SWIGLU)
    assert f[0, 0] == 0
    want = as_bits(np.array([2.0 / (1.0 + np.exp(-2.0))]))[0]
    assert f[0, 1] == want


def test_colwise_equals_rowwise_of_the_transposed_groups(orc):
    """Random bf16 x: the columnwise MXFP8 operand of each group is the rowwise
    MXFP8 quantiser applied to that group's transpose, zero-padded to a
    multiple of 128 tokens (blocks of 32 tokens from the group's first)."""
    rng = np.random.default_rng(27)
    splits = np.array([40, 0, 130, 128, 1])
    M, C = int(splits.sum()), 96
    xb = torch.from_numpy(rng.standard_normal((M, C)).astype(np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)
    codes, scales = orc.mxfp8_colwise(xb, splits)
    offs, pofs = orc.group_offsets(splits), orc.padded_offsets(splits)
    for g in range(len(splits)):
        m, mp = int(splits[g]), int(pofs[g + 1] - pofs[g])
        assert mp == (m + 127) // 128 * 128
        if mp == 0:
            continue
        t = np.zeros((C, mp), np.uint16)
        t[:, :m] = xb[offs[g]:offs[g + 1]].T
        rc, rs = orc.mxfp8_quantize_rows(t)
        assert np.array_equal(codes[:, pofs[g]:pofs[g + 1]], rc), g
        assert np.array_equal(scales[:, pofs[g] // 32:pofs[g + 1] // 32], rs), g


def test_recompute_fc2x_equals_the_forward_fc2x(orc):
    """fc2_x rebuilt from the forward's saved activation input h is the
    forward's own fc2_x bit for bit (SwiGLU and SReLU, MXFP8 and NVFP4, random
    operands; tanh-SReLU too): the rebuild reads h in logical column order and applies the prob
    and the bf16 rounding exactly where the forward does.  For NVFP4 this is
    the pages' recompute on / off equality (PR #3837, Description): the rebuilt
    tensor, cast column-wise with the forward's saved amaxes, gives the same
    codes and scales as the forward's own fc2_x."""
    from mxfp8_nvfp4_block_gb300.inputs import bits, make_inputs
    d = make_inputs("tiny")
    sp = d["splits"].numpy()
    for fmt in (orc.MXFP8, orc.NVFP4):
        for act in (orc.SWIGLU, orc.SRELU, orc.TANH_SRELU):
            W1 = d["W1"] if act == orc.SWIGLU else d["W1"][:, :d["W2"].shape[2]].contiguous()
            c = 8.0 if act == orc.TANH_SRELU else None
            fwd = orc.forward(bits(d["x"]), sp, bits(W1), bits(d["W2"]), d["probs"].numpy(), act, fmt,
                              rht_mask=0x2D4B, tanh_clamp_scale=c)
            again = orc.recompute_fc2x(fwd["h"], d["probs"].numpy(), act, c)
            assert np.array_equal(again, fwd["fc2x"]), (fmt, act)
            assert np.count_nonzero(fwd["fc2x"]) > fwd["fc2x"].size // 4
            if fmt == orc.NVFP4:
                on, off = (orc.group_quantize_with_amax(t, sp, orc.NVFP4, fwd["fc2x_amax_pre"],
                                                        fwd["fc2x_amax_post"], rowwise=True, columnwise=True,
                                                        use_rht=True, mask=0x2D4B) for t in (again, fwd["fc2x"]))
                for k in ("row_codes", "row_scales", "col_codes", "col_scales"):
                    assert np.array_equal(on[k], off[k]), k
