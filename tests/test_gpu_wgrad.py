"""Parity of the weight-gradient backward (CUDA path, through the C ABI) with
the oracle: columnwise MXFP8 operands (bit for bit), the grouped wgrad GEMMs
and the bias gradients, on seeded inputs shared by both sides."""
import numpy as np
import pytest
import torch

from mxfp8_nvfp4_block_gb300.inputs import bits, make_inputs
from parity import frob, np_u8

pytestmark = pytest.mark.gpu


def bf16_cpu(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)


def seeded_inputs(seed, splits_l, K, N, act, scale_rows=True):
    """x, dy, fc1_dy ~ N(0, 1) bf16 (a few rows scaled by 2^+-6 so blocks see
    different exponents), h = pre-activations N(0, 1.5), probs U(0.1, 1)."""
    rng = np.random.default_rng(seed)
    M = sum(splits_l)
    n1 = 2 * N if act == 0 else N

    def mat(c):
        a = rng.standard_normal((M, c))
        if scale_rows and M > 8:
            a[rng.integers(0, M, M // 8)] *= 64.0
            a[rng.integers(0, M, M // 8)] /= 64.0
        return bf16_cpu(a)

    return dict(x=mat(K), dy=mat(K), fc1_dy=mat(n1), h=bf16_cpu(1.5 * rng.standard_normal((M, n1))),
                probs=torch.from_numpy(rng.uniform(0.1, 1, M).astype(np.float32)))


def run_wgrad(gm, d, splits, act, **kw):
    out = gm.backward_wgrad(d["x"].cuda(), d["dy"].cuda(), d["h"].cuda(), d["probs"].cuda(), d["fc1_dy"].cuda(),
                            splits.cuda(), act, **kw)
    gm.check_device_status()
    return out


def test_colwise_mxfp8_bitexact(orc, gm):
    """gmlp_group_quantize(MXFP8, col_out): the weight-gradient operand layout,
    codes and scales equal to the oracle's columnwise MXFP8."""
    splits_l, K = [130, 0, 257, 5, 1, 128, 31], 384
    d = seeded_inputs(3, splits_l, K, 256, 1)
    splits = torch.tensor(splits_l, dtype=torch.int64)
    M, G = sum(splits_l), len(splits_l)
    out = gm.group_quantize(d["x"].cuda(), splits.cuda(), gm.recipe(gm.MXFP8), rowwise=True, columnwise=True,
                            splits_host=splits_l)
    gm.check_device_status()
    T = gm.colwise_tokens(M, G)
    codes, scales = orc.mxfp8_colwise(bits(d["x"]), np.array(splits_l))
    used = codes.shape[1]
    g_codes = np_u8(out["col"][0], K * T).reshape(T // 128, K, 128).transpose(1, 0, 2).reshape(K, T)[:, :used]
    g_scales = orc.tiled_to_compact(np_u8(out["col"][1]), np.array([K]), T // 32)[:, :used // 32]
    assert np.array_equal(g_codes, codes)
    assert np.array_equal(g_scales, scales)


@pytest.mark.parametrize("act", [0, 1], ids=["swiglu", "srelu"])
def test_wgrad_parity(orc, gm, act):
    splits_l, K, N = [130, 0, 257, 5, 1, 128], 512, 256
    d = seeded_inputs(11 + act, splits_l, K, N, act)
    splits = torch.tensor(splits_l, dtype=torch.int64)
    out = run_wgrad(gm, d, splits, act)
    ref = orc.backward_wgrad(bits(d["x"]), bits(d["dy"]), bits(d["h"]), d["probs"].numpy(), bits(d["fc1_dy"]),
                             np.array(splits_l), act)
    errs = {k: frob(out[k].cpu().numpy(), ref[k]) for k in ("dW1", "dW2", "dbias1", "dbias2")}
    print("wgrad relative errors", {k: f"{v:.2e}" for k, v in errs.items()})
    assert errs["dW1"] <= 1e-5 and errs["dbias1"] <= 1e-5 and errs["dbias2"] <= 1e-5
    # SwiGLU's fc2_x is rebuilt in FP32 (the forward epilogue's arithmetic), the
    # oracle's in float64: a bf16 rounding may differ by one step here and there
    assert errs["dW2"] <= (1e-3 if act == 0 else 1e-5)
    assert not out["dW1"][1].any() and not out["dW2"][1].any()      # the empty expert


def test_wgrad_lossless_bitexact_and_accumulate(orc, gm):
    """SReLU with operands from {0, +-1, +-2} and probs from {1, 0.5}: every
    block is exact and every sum fits FP32, so the gradients equal the oracle's
    bit for bit; accumulate = 1 then adds a second copy exactly."""
    rng = np.random.default_rng(23)
    splits_l, K, N = [130, 0, 257, 5, 128], 512, 256
    M = sum(splits_l)
    d = dict(x=bf16_cpu(rng.choice([0.0, 1.0, -1.0], size=(M, K))),
             dy=bf16_cpu(rng.choice([0.0, 1.0, -1.0, 2.0], size=(M, K))),
             fc1_dy=bf16_cpu(rng.choice([0.0, 1.0, -2.0], size=(M, N))),
             h=bf16_cpu(rng.choice([0.0, 1.0, -1.0, 2.0], size=(M, N))),
             probs=torch.from_numpy(rng.choice([1.0, 0.5], size=M).astype(np.float32)))
    splits = torch.tensor(splits_l, dtype=torch.int64)
    out = run_wgrad(gm, d, splits, 1)
    ref = orc.backward_wgrad(bits(d["x"]), bits(d["dy"]), bits(d["h"]), d["probs"].numpy(), bits(d["fc1_dy"]),
                             np.array(splits_l), 1)
    for k in ("dW1", "dW2", "dbias1", "dbias2"):
        assert np.array_equal(out[k].cpu().numpy().astype(np.float64), ref[k]), k
    again = run_wgrad(gm, d, splits, 1, accumulate=True, **{k: out[k] for k in ("dW1", "dW2", "dbias1", "dbias2")})
    for k in ("dW1", "dW2", "dbias1", "dbias2"):
        assert np.array_equal(again[k].cpu().numpy().astype(np.float64), 2 * ref[k]), k
    # only what is asked for is computed: dbias2 alone needs neither x nor h
    only = gm.backward_wgrad(d["x"].cuda(), d["dy"].cuda(), None, None, d["fc1_dy"].cuda(), splits.cuda(), 1,
                             want=("dbias2",))
    gm.check_device_status()
    assert only["dW1"] is None and np.array_equal(only["dbias2"].cpu().numpy().astype(np.float64), ref["dbias2"])


def test_wgrad_full_size_sampled(orc, gm):
    """The full headline workload (MXFP8 SwiGLU, 8 experts, K=2048, N=1024,
    16384 tokens, Dirichlet splits with an empty expert), sampled: entries of
    dW1 / dW2 / dbias computed one by one by the oracle from single columns
    (columnwise blocks never mix columns)."""
    w = make_inputs("mx_swiglu", weights=False)
    wl = w["workload"]
    splits_l = [int(v) for v in w["splits"].tolist()]
    M, K, N = wl.M, wl.K, wl.N
    gen = torch.Generator().manual_seed(97)
    d = dict(x=w["x"], probs=w["probs"],
             dy=torch.randn((M, K), generator=gen).to(torch.bfloat16),
             h=(1.5 * torch.randn((M, 2 * N), generator=gen)).to(torch.bfloat16),
             fc1_dy=torch.randn((M, 2 * N), generator=gen).to(torch.bfloat16))
    out = run_wgrad(gm, d, w["splits"], 0)
    offs = orc.group_offsets(np.array(splits_l))
    sp = np.array(splits_l)
    x, dy, h, f1 = bits(d["x"]), bits(d["dy"]), bits(d["h"]), bits(d["fc1_dy"])
    probs = d["probs"].numpy()
    rng = np.random.default_rng(5)

    def col_deq(m, c):
        return orc.mxfp8_dequant_rows(*orc.mxfp8_colwise(np.ascontiguousarray(m[:, [c]]), sp))[0]

    pofs = orc.padded_offsets(sp)
    worst = 0.0
    for _ in range(24):
        g = int(rng.choice([i for i in range(len(sp)) if sp[i] > 0]))
        i, j = int(rng.integers(0, K)), int(rng.integers(0, N))
        hj = np.ascontiguousarray(h[:, [j, N + j]])
        fj = orc.mxfp8_dequant_rows(*orc.mxfp8_colwise(orc.recompute_fc2x(hj, probs, 0), sp))[0]
        a, b = col_deq(dy, i)[pofs[g]:pofs[g + 1]], fj[pofs[g]:pofs[g + 1]]
        ref2, bound2 = float(a @ b), float(np.abs(a) @ np.abs(b))
        i1, j1 = int(rng.integers(0, 2 * N)), int(rng.integers(0, K))
        a1, b1 = col_deq(f1, i1)[pofs[g]:pofs[g + 1]], col_deq(x, j1)[pofs[g]:pofs[g + 1]]
        ref1, bound1 = float(a1 @ b1), float(np.abs(a1) @ np.abs(b1))
        got2, got1 = float(out["dW2"][g, i, j]), float(out["dW1"][g, i1, j1])
        e2, e1 = abs(got2 - ref2) / max(bound2, 1e-30), abs(got1 - ref1) / max(bound1, 1e-30)
        worst = max(worst, e2, e1)
        # FP32 accumulation over at most a few thousand tokens
        assert e2 <= 2e-4 and e1 <= 2e-4, (g, i, j, got2, ref2, got1, ref1)
        r0, r1 = offs[g], offs[g + 1]
        db2 = orc.bf16_to_f64(dy[r0:r1, i]).sum()
        db1 = orc.bf16_to_f64(f1[r0:r1, i1]).sum()
        s2, s1 = np.abs(orc.bf16_to_f64(dy[r0:r1, i])).sum(), np.abs(orc.bf16_to_f64(f1[r0:r1, i1])).sum()
        assert abs(float(out["dbias2"][g, i]) - db2) <= 1e-5 * s2 + 1e-6
        assert abs(float(out["dbias1"][g, i1]) - db1) <= 1e-5 * s1 + 1e-6
    empty = [i for i in range(len(sp)) if sp[i] == 0]
    for g in empty:
        assert not out["dW1"][g].any() and not out["dW2"][g].any()
    print(f"full-size wgrad: worst sampled error {worst:.2e} of sum |a b|")


@pytest.mark.parametrize("case", ["many_tiny", "one_group", "under_one_chunk"])
def test_wgrad_group_edge_cases(orc, gm, case):
    """Ragged extremes: 64 experts, most empty or of 1-8 tokens with a few large
    ones (the skewed workload's tail); one expert holding every token; fewer
    tokens than one 128-token chunk.  SReLU keeps the fc2_x rebuild exact, so
    only FP32 summation order separates the two sides."""
    rng = np.random.default_rng(31)
    if case == "many_tiny":
        splits_l = [int(v) for v in rng.integers(0, 9, 64)]
        splits_l[3], splits_l[40], splits_l[63] = 300, 129, 0
    elif case == "one_group":
        splits_l = [777]
    else:
        splits_l = [0, 37, 0, 60]
    K, N = 256, 256
    d = seeded_inputs(41, splits_l, K, N, 1)
    splits = torch.tensor(splits_l, dtype=torch.int64)
    out = run_wgrad(gm, d, splits, 1)
    ref = orc.backward_wgrad(bits(d["x"]), bits(d["dy"]), bits(d["h"]), d["probs"].numpy(), bits(d["fc1_dy"]),
                             np.array(splits_l), 1)
    for k in ("dW1", "dW2", "dbias1", "dbias2"):
        err = frob(out[k].cpu().numpy(), ref[k])
        assert err <= 1e-5, (k, err)
    for g, m in enumerate(splits_l):
        if m == 0:
            assert not out["dW1"][g].any() and not out["dW2"][g].any() and not out["dbias1"][g].any()
