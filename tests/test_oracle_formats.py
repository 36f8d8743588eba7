"""Pins of the oracle's format arithmetic against the format definitions, library
routines, closed forms and brute force (CPU only).

The facts the method statement fixes: E2M1 values {0,0.5,1,1.5,2,3,4,6}; E4M3
max 448; MXFP8 scale 2^(floor(log2 amax) - 8); H16 H16^T = 16 I.
"""
import numpy as np
import pytest
import scipy.linalg
import torch


def all_finite_bf16():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):      # NaN patterns, dropped below
        f = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ok = np.isfinite(f)
    return b[ok], f[ok]


def e4m3_table_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


# ------------------------------------------------------------------ E4M3

def test_e4m3_decode_matches_torch_float8(orc):
    ref = e4m3_table_torch()
    mine = np.array([orc.lib().orc_e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.nanmax(mine) == 448.0 and mine[0x7E] == 448.0


def _nearest_even(values, table_vals, table_codes):
    """Brute force: nearest representable value; ties -> the code with an even mantissa LSB."""
    d = np.abs(values[:, None] - table_vals[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    even = (table_codes % 2 == 0)[None, :]
    pick_even = cand & even
    has_even = pick_even.any(axis=1)
    idx = np.where(has_even, np.argmax(pick_even, axis=1), np.argmax(cand, axis=1))
    return table_codes[idx]


@pytest.mark.parametrize("scale_exp", [-127, -9, 0, 8])
def test_e4m3_encode_bruteforce_all_bf16(orc, scale_exp):
    _, f = all_finite_bf16()
    v = np.ldexp(f, scale_exp)
    L = orc.lib()
    mine = np.array([L.orc_e4m3_encode(float(t)) for t in v], dtype=np.uint8)
    ref_vals = e4m3_table_torch()[:0x7F]   # non-negative finite codes 0x00..0x7E
    codes = np.arange(0x7F)
    a = np.abs(v)
    sat = a >= 448.0
    want = np.empty(len(v), dtype=np.uint8)
    want[sat] = 0x7E
    want[~sat] = _nearest_even(a[~sat], ref_vals, codes)
    want |= np.where(np.signbit(v), 0x80, 0).astype(np.uint8)
    assert np.array_equal(mine, want)


def test_e4m3_encode_matches_torch_rne_in_range(orc):
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(20000) * 1e-2,
                        rng.uniform(-447, 447, 20000)]).astype(np.float32).astype(np.float64)
    L = orc.lib()
    mine = np.array([L.orc_e4m3_encode(float(t)) for t in v], dtype=np.uint8)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


def test_e4m3_ties_and_saturation(orc):
    L = orc.lib()
    # midpoint of 1.0 (0x38) and 1.125 (0x39) -> even mantissa 0x38; of 1.125 and 1.25 -> 0x3A
    assert L.orc_e4m3_encode(1.0625) == 0x38
    assert L.orc_e4m3_encode(1.1875) == 0x3A
    # subnormal midpoint: 0.5 * 2^-9 -> 0 ; 1.5 * 2^-9 -> 2 * 2^-9
    assert L.orc_e4m3_encode(2.0 ** -10) == 0x00
    assert L.orc_e4m3_encode(1.5 * 2.0 ** -9) == 0x02
    assert L.orc_e4m3_encode(-0.0) == 0x80
    for v in (448.0, 463.9, 464.0, 500.0, 1e30):
        assert L.orc_e4m3_encode(v) == 0x7E and L.orc_e4m3_encode(-v) == 0xFE


# ------------------------------------------------------------------ E2M1

def test_e2m1_value_set(orc):
    L = orc.lib()
    vals = [L.orc_e2m1_decode(c) for c in range(8)]
    assert vals == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert [L.orc_e2m1_decode(c | 8) for c in range(8)] == [-v for v in vals]


def test_e2m1_ties(orc):
    L = orc.lib()
    dec = lambda c: L.orc_e2m1_decode(c)  # noqa: E731
    for v, want in [(0.25, 0), (0.75, 1), (1.25, 1), (1.75, 2), (2.5, 2), (3.5, 4), (5.0, 4),
                    (6.0, 6), (7.0, 6), (100.0, 6)]:
        assert dec(L.orc_e2m1_encode(v)) == want, v
        assert dec(L.orc_e2m1_encode(-v)) == -want, v
    assert L.orc_e2m1_encode(-0.0) == 8


def test_e2m1_encode_bruteforce(orc):
    _, f = all_finite_bf16()
    f = f[np.abs(f) < 64]
    L = orc.lib()
    mine = np.array([L.orc_e2m1_encode(float(t)) for t in f], dtype=np.uint8)
    table = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    codes = np.arange(8)
    a = np.abs(f)
    sat = a >= 6
    want = np.empty(len(f), dtype=np.uint8)
    want[sat] = 7
    want[~sat] = _nearest_even(a[~sat], table, codes)
    want |= np.where(np.signbit(f), 8, 0).astype(np.uint8)
    assert np.array_equal(mine, want)


# ------------------------------------------------------------------ bf16

def test_bf16_round_matches_torch_for_float_values(orc):
    rng = np.random.default_rng(1)
    with np.errstate(over="ignore"):         # values past FLT_MAX become inf on purpose
        v = np.concatenate([rng.standard_normal(50000), rng.standard_normal(5000) * 1e-39,
                            rng.standard_normal(5000) * 1e38]).astype(np.float32)
    mine = orc.f64_to_bf16(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


def test_bf16_round_exact_ties_and_no_double_rounding(orc):
    one_ulp = 2.0 ** -7
    assert orc.f64_to_bf16(np.array([1.0 + one_ulp / 2]))[0] == 0x3F80          # tie -> even (1.0)
    assert orc.f64_to_bf16(np.array([1.0 + 3 * one_ulp / 2]))[0] == 0x3F82      # tie -> even (1+2ulp)
    # just above the tie by far less than a float ulp: a float-first rounding would land on the tie
    assert orc.f64_to_bf16(np.array([1.0 + one_ulp / 2 + 2.0 ** -40]))[0] == 0x3F81
    assert orc.f64_to_bf16(np.array([3.5e38]))[0] == 0x7F80
    assert orc.f64_to_bf16(np.array([-0.0]))[0] == 0x8000


# ------------------------------------------------------------------ MXFP8

def test_mxfp8_scale_exponent_closed_form(orc):
    L = orc.lib()
    for k in range(-119, 128):
        assert L.orc_mxfp8_scale_exponent(2.0 ** k) == k - 8
        assert L.orc_mxfp8_scale_exponent(2.0 ** k * 1.999) == k - 8
    assert L.orc_mxfp8_scale_exponent(0.0) == -127
    assert L.orc_mxfp8_scale_exponent(2.0 ** -130) == -127
    assert L.orc_mxfp8_scale_exponent(2.0 ** -120) == -127   # clamped at the E8M0 floor


def _bf16(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_mxfp8_block_closed_forms(orc):
    # amax = 2^k -> scale byte k - 8 + 127, the max element's code is 256 = 0x78
    for k in (-20, -3, 0, 5, 30):
        row = np.full(32, 0.0)
        row[7] = -(2.0 ** k)
        row[3] = 2.0 ** (k - 1)
        codes, scales = orc.mxfp8_quantize_rows(_bf16(row).reshape(1, 32))
        assert scales[0, 0] == k - 8 + 127
        assert codes[0, 7] == 0x78 | 0x80 and codes[0, 3] == 0x70
    # a constant block gives equal codes
    codes, _ = orc.mxfp8_quantize_rows(_bf16(np.full(32, 3.3)).reshape(1, 32))
    assert len(set(codes[0].tolist())) == 1
    # all-zero block: scale byte 0, codes 0
    codes, scales = orc.mxfp8_quantize_rows(np.zeros((1, 32), np.uint16))
    assert scales[0, 0] == 0 and not codes.any()


def test_mxfp8_roundtrip_error_bound(orc):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((64, 256)) * np.exp(rng.uniform(-8, 8, (64, 1)))
    xb = _bf16(x.astype(np.float32)).reshape(64, 256)
    xf = orc.bf16_to_f64(xb)
    codes, scales = orc.mxfp8_quantize_rows(xb)
    dq = orc.mxfp8_dequant_rows(codes, scales)
    e = scales.astype(np.int64).repeat(32, axis=1) - 127
    scaled = np.ldexp(np.abs(xf), -e)            # in [0, 512)
    sat = scaled >= 448
    assert np.all(np.abs(np.ldexp(dq[sat], -e[sat])) == 448)
    ns = ~sat & (scaled >= 2.0 ** -6)
    # half an ulp of a 3-bit mantissa at the element's binade
    ulp = np.ldexp(1.0, np.floor(np.log2(scaled[ns])).astype(np.int64) - 3)
    assert np.all(np.abs(np.ldexp(np.abs(dq[ns]), -e[ns]) - scaled[ns]) <= ulp / 2)
    sub = ~sat & ~ns
    assert np.all(np.abs(np.ldexp(np.abs(dq[sub]), -e[sub]) - scaled[sub]) <= 2.0 ** -10)
    assert np.all(np.sign(dq[dq != 0]) == np.sign(xf[dq != 0]))


# ------------------------------------------------------------------ NVFP4

def test_nvfp4_global_scale(orc):
    assert orc.nvfp4_global_scale(2688.0) == 1.0
    assert orc.nvfp4_global_scale(0.0) == 1.0
    assert orc.nvfp4_global_scale(1.0) == 2688.0
    assert orc.nvfp4_global_scale(1e-40) == np.float32(np.finfo(np.float32).max)


def test_nvfp4_block_exact_values(orc):
    # b = 6 with S = 1 -> block scale 1.0 (E4M3 0x38), enc = 1, codes are the values themselves
    vals = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -1.5, -2, -3, -4, -6, 0], np.float32)
    codes, sf = orc.nvfp4_quantize_block(vals, 1.0)
    assert sf == 0x38
    nib = np.stack([codes & 15, codes >> 4], axis=1).reshape(-1)
    L = orc.lib()
    assert [L.orc_e2m1_decode(int(c)) for c in nib] == vals.tolist()
    assert nib[0] == 0 and nib[-1] == 0


def test_nvfp4_encode_factor_saturates(orc):
    """S = FLT_MAX (group amax below 2688 / FLT_MAX) and a block max b = 2^-126
    give t = fp32(b / 6) * FLT_MAX ~ 0.667 -> sf = E4M3 0.6875 (0x33), and
    S / sf overflows; the encode factor stays at FLT_MAX, so zeros encode to
    zero with their sign and the other values by their finite products
    (b -> 4.0, b / 2 -> 2.0, 2^-140 -> 2.4e-4 -> 0)."""
    fmax = np.float32(np.finfo(np.float32).max)
    b = np.float32(2.0 ** -126)
    tiny = np.float32(2.0 ** -140)
    vals = np.array([b, 0.0, -0.0, -b, tiny, -tiny, b / 2, 0.0] + [0.0] * 8, np.float32)
    codes, sf = orc.nvfp4_quantize_block(vals, fmax)
    assert sf == 0x33
    nib = (np.stack([codes & 15, codes >> 4], axis=1).reshape(-1)).tolist()
    assert nib[:8] == [6, 0, 8, 14, 0, 8, 4, 0]


@pytest.mark.parametrize("amax_level", [1.0, 2.0, 4.0])
def test_nvfp4_lossless_set(orc, amax_level):
    """Entries in {0, +-1, +-2, +-4} with group amax 4 round-trip exactly for any block maximum."""
    rng = np.random.default_rng(3)
    choices = np.array([0, 1, 2, 4, -1, -2, -4], np.float32)
    x = rng.choice(choices, size=(8, 64))
    x = np.clip(x, -amax_level, amax_level)
    x[0, 0] = 4.0
    xb = _bf16(x).reshape(8, 64)
    S = orc.nvfp4_global_scale(orc.amax_bf16(xb))
    codes, scales = orc.nvfp4_quantize_rows(xb, S)
    assert np.array_equal(orc.nvfp4_dequant_rows(codes, scales, S), x.astype(np.float64))


def test_nvfp4_roundtrip_error_bound(orc):
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((32, 128)) * np.exp(rng.uniform(-3, 3, (32, 1)))).astype(np.float32)
    xb = _bf16(x).reshape(32, 128)
    xf = orc.bf16_to_f64(xb)
    S = orc.nvfp4_global_scale(orc.amax_bf16(xb))
    codes, scales = orc.nvfp4_quantize_rows(xb, S)
    dq = orc.nvfp4_dequant_rows(codes, scales, S)
    L = orc.lib()
    sfv = np.vectorize(L.orc_e4m3_decode)(scales).repeat(16, axis=1)
    unit = sfv / float(S)                       # one E2M1 step of 1.0 in dequant units
    u = np.abs(xf) / unit                       # the element in E2M1 units
    half = np.where(u < 2, 0.25, np.where(u < 4, 0.5, 1.0))
    bound = (half + np.maximum(u - 6, 0)) * unit * (1 + 1e-6)
    assert np.all(np.abs(dq - xf) <= bound)
    # block scales: the block max maps close to 6 (E4M3 precision of the scale)
    bmax = np.abs(xf).reshape(32, 8, 16).max(axis=2)
    ratio = bmax / (sfv[:, ::16] / float(S))
    ok = bmax > 0
    assert np.all((ratio[ok] > 6 / 1.07) & (ratio[ok] < 6 * 1.07))


# ------------------------------------------------------------------ RHT

def test_rht_is_quarter_sylvester_hadamard(orc):
    H = scipy.linalg.hadamard(16).astype(np.float64)
    cols = np.stack([orc.rht16(np.eye(16, dtype=np.float32)[j], 0) for j in range(16)], axis=1)
    assert np.array_equal(4 * cols.astype(np.float64), H)
    Hm = 4 * cols.astype(np.float64)
    assert np.array_equal(Hm @ Hm.T, 16 * np.eye(16))


def test_rht_sign_mask_and_closed_forms(orc):
    H = scipy.linalg.hadamard(16).astype(np.float64)
    rng = np.random.default_rng(5)
    for _ in range(50):
        mask = int(rng.integers(0, 1 << 16))
        v = rng.integers(-100, 100, 16).astype(np.float32)     # exact in fp32 through every stage
        s = np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)])
        want = 0.25 * H @ (s * v.astype(np.float64))
        assert np.array_equal(orc.rht16(v, mask).astype(np.float64), want)
    c = np.float32(3.25)
    y = orc.rht16(np.full(16, c, np.float32), 0)
    assert y[0] == 4 * c and not y[1:].any()


def _dense_hadamard_amax(x, splits, mask):
    H = scipy.linalg.hadamard(16).astype(np.float64)
    s = np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)])
    offs = np.concatenate([[0], np.cumsum(splits)])
    pre, post = [], []
    for g in range(len(splits)):
        blk = x[offs[g]:offs[g + 1]]
        pre.append(np.abs(blk).max() if len(blk) else 0.0)
        m = len(blk)
        if m == 0:
            post.append(0.0)
            continue
        mp = (m + 15) // 16 * 16
        pad = np.zeros((mp, x.shape[1]))
        pad[:m] = blk
        ch = pad.reshape(mp // 16, 16, -1)
        y = 0.25 * np.einsum("ij,cjk->cik", H, s[None, :, None] * ch)
        post.append(np.abs(y).max())
    return np.array(pre), np.array(post)


def test_group_hadamard_amax_integer_exact(orc):
    rng = np.random.default_rng(6)
    splits = [0, 1, 15, 16, 17, 33, 50]
    M, K = sum(splits), 48
    xi = rng.integers(-60, 61, (M, K)).astype(np.float32)
    xb = _bf16(xi).reshape(M, K)
    mask = 0b1011001110001101
    pre, post = orc.group_hadamard_amax(xb, splits, mask)
    wpre, wpost = _dense_hadamard_amax(xi.astype(np.float64), splits, mask)
    assert np.array_equal(pre.astype(np.float64), wpre)
    assert np.array_equal(post.astype(np.float64), wpost)


def test_group_hadamard_amax_random_close(orc):
    rng = np.random.default_rng(7)
    splits = [40, 0, 77, 130]
    M, K = sum(splits), 64
    xb = _bf16(rng.standard_normal((M, K)).astype(np.float32)).reshape(M, K)
    mask = int(rng.integers(0, 1 << 16))
    pre, post = orc.group_hadamard_amax(xb, splits, mask)
    wpre, wpost = _dense_hadamard_amax(orc.bf16_to_f64(xb), splits, mask)
    assert np.array_equal(pre.astype(np.float64), wpre)
    np.testing.assert_allclose(post, wpost, rtol=1e-6)
    # the sign mask matters: the plain transform gives a different post-RHT amax
    _, post0 = orc.group_hadamard_amax(xb, splits, 0)
    assert not np.array_equal(post0[post0 > 0], post[post0 > 0])


def test_columnwise_rht_roundtrip_inverts(orc):
    """Dequantise the columnwise RHT output, undo the transform (v = diag(s) H y / 4), and
    recover x^T per group within NVFP4 error; a wrong layout, sign or direction does not."""
    H = scipy.linalg.hadamard(16).astype(np.float64)
    rng = np.random.default_rng(8)
    splits = [37, 16, 0, 75]
    M, K = sum(splits), 32
    xb = _bf16(rng.standard_normal((M, K)).astype(np.float32)).reshape(M, K)
    xf = orc.bf16_to_f64(xb)
    mask = 0x5A3C
    q = orc.group_quantize(xb, splits, orc.NVFP4, rowwise=False, columnwise=True, use_rht=True, mask=mask)
    s = np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)])
    L = orc.lib()
    offs = np.concatenate([[0], np.cumsum(splits)])
    cb = sb = 0
    for g, m in enumerate(splits):
        mp = (m + 15) // 16 * 16
        codes = q["col_codes"][cb:cb + K * mp // 2].reshape(K, mp // 2)
        sc = q["col_scales"][sb:sb + K * mp // 16].reshape(K, mp // 16)
        cb += K * mp // 2
        sb += K * mp // 16
        if m == 0:
            continue
        nib = np.stack([codes & 15, codes >> 4], axis=2).reshape(K, mp)
        y = np.vectorize(L.orc_e2m1_decode)(nib) * np.vectorize(L.orc_e4m3_decode)(sc).repeat(16, axis=1)
        y /= float(q["col_S"][g])
        v = np.einsum("ij,cnj->cni", H, y.reshape(K, mp // 16, 16)) * s[None, None, :] / 4.0
        rec = v.reshape(K, mp)[:, :m].T
        err = np.linalg.norm(rec - xf[offs[g]:offs[g + 1]]) / np.linalg.norm(xf[offs[g]:offs[g + 1]])
        assert err < 0.2, (g, err)


def _colwise_from_rowwise(orc, xf, splits, mask, use_rht, S):
    """Columnwise NVFP4 restated through the rowwise quantiser: per group, the
    transposed rows zero-padded to a multiple of 16 tokens, optionally taken
    through 1/4 H16 diag(s) over each 16-token chunk in float64, then rowwise
    NVFP4 under that group's S (the values here are exact in bf16)."""
    H = scipy.linalg.hadamard(16).astype(np.float64)
    s = np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)])
    offs = np.concatenate([[0], np.cumsum(splits)])
    K = xf.shape[1]
    codes, scales = [], []
    for g, m in enumerate(splits):
        mp = (m + 15) // 16 * 16
        if mp == 0:
            continue
        t = np.zeros((K, mp))
        t[:, :m] = xf[offs[g]:offs[g + 1]].T
        if use_rht:
            ch = t.reshape(K, mp // 16, 16)
            t = (0.25 * np.einsum("ij,cnj->cni", H, ch * s[None, None, :])).reshape(K, mp)
        tb = _bf16(t.astype(np.float32)).reshape(K, mp)
        assert np.array_equal(orc.bf16_to_f64(tb), t)          # exact in bf16
        c, sc = orc.nvfp4_quantize_rows(tb, S[g])
        codes.append(c.reshape(-1))
        scales.append(sc.reshape(-1))
    return np.concatenate(codes), np.concatenate(scales)


@pytest.mark.parametrize("use_rht", [False, True], ids=["plain", "rht"])
def test_columnwise_equals_rowwise_of_the_transposed_groups(orc, use_rht):
    """Small-integer x (every transform value exact): the columnwise NVFP4
    output equals the rowwise quantiser applied to each group's transpose
    (through the masked RHT when it is on), under the global scale of
    amax_post (RHT) or amax_pre (plain), both taken here from the dense
    float64 values."""
    rng = np.random.default_rng(19)
    splits = [37, 16, 0, 75, 1]
    M, K = sum(splits), 48
    xf = rng.integers(-3, 4, (M, K)).astype(np.float64)
    xb = _bf16(xf.astype(np.float32)).reshape(M, K)
    mask = 0x36C9
    q = orc.group_quantize(xb, splits, orc.NVFP4, rowwise=False, columnwise=True, use_rht=use_rht, mask=mask)
    H = scipy.linalg.hadamard(16).astype(np.float64)
    s = np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)])
    offs = np.concatenate([[0], np.cumsum(splits)])
    S = []
    for g, m in enumerate(splits):
        blk = xf[offs[g]:offs[g + 1]]
        if use_rht and m:
            mp = (m + 15) // 16 * 16
            t = np.zeros((mp, K))
            t[:m] = blk
            amax = np.abs(0.25 * np.einsum("ij,njc->nic", H, t.reshape(mp // 16, 16, K) * s[None, :, None])).max()
        else:
            amax = np.abs(blk).max() if m else 0.0
        S.append(orc.nvfp4_global_scale(amax))
    np.testing.assert_array_equal(q["col_S"], np.array(S, np.float32))
    codes, scales = _colwise_from_rowwise(orc, xf, splits, mask, use_rht, S)
    assert np.array_equal(q["col_scales"], scales)
    # a transform output of exactly zero carries the sign its butterfly gives it
    # (the fp32 stages' order, e.g. -0 from a negated zero padding row), which a
    # dense float64 product does not reproduce: compare codes with -0 folded
    # onto +0, and require every other code to match exactly
    def fold(c):
        lo, hi = c & 15, c >> 4
        return np.where(lo == 8, 0, lo) | (np.where(hi == 8, 0, hi) << 4)
    assert np.array_equal(fold(q["col_codes"]), fold(codes))
    if not use_rht:
        assert np.array_equal(q["col_codes"], codes)
