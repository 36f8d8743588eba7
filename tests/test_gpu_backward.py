"""Parity of the data-gradient backward (CUDA path, through the C ABI) with the
oracle: fc2 dGLU (dSwiGLU / dSReLU x prob, dprob, fc1_dy in MXFP8 and bf16)
and the fc1 dgrad, on seeded inputs shared by both sides; and the forward's
saved activation input against the oracle forward's."""
import numpy as np
import pytest
import torch

from mxfp8_nvfp4_block_gb300.inputs import bits
from parity import code_match_report, frob, np_bits, np_u8

pytestmark = pytest.mark.gpu


def bf16_cpu(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)


def forward_with_h(gm, x, splits, W1, W2, probs, act):
    """Forward that also returns the saved activation input h [M, N1]."""
    M, N = x.shape[0], W2.shape[2]
    n1 = W1.shape[1]
    w1 = gm.prepare_weights(W1.cuda(), gm.MXFP8, swiglu_interleave=(act == gm.SWIGLU))
    w2 = gm.prepare_weights(W2.cuda(), gm.MXFP8)
    h = torch.full((M, n1), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = gm.forward(x.cuda(), splits.cuda(), w1, w2, probs, act, gm.recipe(gm.MXFP8), aux={"fc1_pre_act": h})
    gm.check_device_status()
    return y, h


def run_backward(gm, dy, splits, W1, W2, h, probs, act):
    M, N1 = h.shape
    G = splits.numel()
    w2t = gm.prepare_transposed_weights(W2.cuda())
    w1t = gm.prepare_transposed_weights(W1.cuda())
    fc1 = {"codes": torch.zeros(M * N1 + 16, dtype=torch.uint8, device="cuda"),
           "scales": torch.zeros(gm.tiled_scales_bytes(M, G, N1 // 32) + 16, dtype=torch.uint8, device="cuda"),
           "bf16": torch.full((M, N1), float("nan"), dtype=torch.bfloat16, device="cuda")}
    dx, dprob = gm.backward_dgrad(dy.cuda(), splits.cuda(), w2t, w1t, h, probs, act, gm.recipe(gm.MXFP8),
                                  fc1_dy={"codes": fc1["codes"], "scales": fc1["scales"]}, fc1_dy_bf16=fc1["bf16"])
    gm.check_device_status()
    return dx, dprob, fc1


@pytest.mark.parametrize("act", [0, 1], ids=["swiglu", "srelu"])
def test_forward_saves_activation_input(orc, gm, act):
    """gmlp_fwd_aux.fc1_pre_act = bf16(fc1 accumulator) in logical column order
    (SwiGLU: gate then up), against the oracle forward's h."""
    rng = np.random.default_rng(41 + act)
    splits_l, K, N = [130, 0, 257, 5, 1, 128], 512, 256
    G, M = len(splits_l), sum(splits_l)
    n1 = 2 * N if act == 0 else N
    splits = torch.tensor(splits_l, dtype=torch.int64)
    x = bf16_cpu(rng.standard_normal((M, K)))
    W1 = bf16_cpu(rng.standard_normal((G, n1, K)) / np.sqrt(K))
    W2 = bf16_cpu(rng.standard_normal((G, K, N)) / np.sqrt(N))
    probs = torch.from_numpy(rng.uniform(0.1, 1, M).astype(np.float32))
    _, h = forward_with_h(gm, x, splits, W1, W2, probs.cuda(), act)
    ref = orc.forward(bits(x), np.array(splits_l), bits(W1), bits(W2), probs.numpy(), act, orc.MXFP8)
    hb = np_bits(h)
    match = float(np.mean(hb == ref["h"]))
    err = frob(orc.bf16_to_f64(hb), orc.bf16_to_f64(ref["h"]))
    print(f"fc1_pre_act bf16 match {match:.6f}, relative error {err:.2e}")
    # FP32 tensor-core sums against float64: a bf16 rounding may flip by one step
    assert match >= 0.99 and err <= 1e-2


@pytest.mark.parametrize("act", [0, 1], ids=["swiglu", "srelu"])
def test_backward_dgrad_parity(orc, gm, act):
    rng = np.random.default_rng(61 + act)
    splits_l, K, N = [130, 0, 257, 5, 1, 128], 512, 256
    G, M = len(splits_l), sum(splits_l)
    n1 = 2 * N if act == 0 else N
    splits = torch.tensor(splits_l, dtype=torch.int64)
    W1 = bf16_cpu(rng.standard_normal((G, n1, K)) / np.sqrt(K))
    W2 = bf16_cpu(rng.standard_normal((G, K, N)) / np.sqrt(N))
    probs_h = torch.from_numpy(rng.uniform(0.1, 1, M).astype(np.float32))
    h_host = bf16_cpu(1.5 * rng.standard_normal((M, n1)))   # the saved activation input (pre-activations)
    dy = bf16_cpu(rng.standard_normal((M, K)))
    dx, dprob, fc1 = run_backward(gm, dy, splits, W1, W2, h_host.cuda(), probs_h.cuda(), act)
    ref = orc.backward_dgrad(bits(dy), np.array(splits_l), bits(W1), bits(W2), bits(h_host), probs_h.numpy(), act)
    fb = np_bits(fc1["bf16"])
    bmatch = float(np.mean(fb == ref["fc1_dy"]))
    print(f"fc1_dy bf16 match {bmatch:.6f}")
    assert bmatch >= 0.99 and frob(orc.bf16_to_f64(fb), orc.bf16_to_f64(ref["fc1_dy"])) <= 1e-2
    frac, steps = code_match_report(0, np_u8(fc1["codes"], M * n1).reshape(M, n1), ref["fc1_dy_codes"],
                                    orc.tiled_to_compact(np_u8(fc1["scales"]), np.array(splits_l), n1 // 32),
                                    ref["fc1_dy_scales"])
    print(f"fc1_dy code match {frac:.6f} (max {steps:.2f} steps)")
    assert frac >= 0.999 and steps <= 1.0 + 1e-9, (frac, steps)
    err = frob(dx.float().cpu().numpy(), orc.bf16_to_f64(ref["dx"]))
    perr = frob(dprob.cpu().numpy(), ref["dprob"])
    print(f"dx error {err:.3e}, dprob error {perr:.3e}")
    assert err <= 1e-2 and perr <= 1e-2


def test_backward_dgrad_lossless_bitexact(orc, gm):
    """SReLU, small-integer operands, one-hot weights: dx and fc1_dy exact."""
    rng = np.random.default_rng(71)
    splits_l, K, N = [130, 0, 257, 5, 128], 512, 256
    G, M = len(splits_l), sum(splits_l)
    splits = torch.tensor(splits_l, dtype=torch.int64)
    W2 = np.zeros((G, K, N))
    W1 = np.zeros((G, N, K))
    for g in range(G):
        W2[g, rng.integers(0, K, N), np.arange(N)] = 1.0
        W1[g, np.arange(N), rng.integers(0, K, N)] = 1.0
    h_host = bf16_cpu(rng.choice([0.0, 1.0, -1.0, 2.0], size=(M, N)))
    dy = bf16_cpu(rng.choice([0.0, 1.0, -1.0], size=(M, K)))
    dx, dprob, fc1 = run_backward(gm, dy, splits, bf16_cpu(W1), bf16_cpu(W2), h_host.cuda(), None, 1)
    ref = orc.backward_dgrad(bits(dy), np.array(splits_l), bits(bf16_cpu(W1)), bits(bf16_cpu(W2)), bits(h_host),
                             None, 1)
    assert np.array_equal(np_u8(fc1["codes"], M * N).reshape(M, N), ref["fc1_dy_codes"])
    assert np.array_equal(np_bits(dx), ref["dx"])
    assert np.array_equal(dprob.cpu().numpy().astype(np.float64), ref["dprob"])


def test_backward_dgrad_many_tiny_groups(orc, gm):
    """64 experts, most empty or of 1-8 tokens, a few large: every tile of the
    dGLU and dgrad GEMMs is a ragged one."""
    rng = np.random.default_rng(81)
    splits_l = [int(v) for v in rng.integers(0, 9, 64)]
    splits_l[5], splits_l[50] = 260, 131
    K, N = 256, 256
    G, M = len(splits_l), sum(splits_l)
    splits = torch.tensor(splits_l, dtype=torch.int64)
    W1 = bf16_cpu(rng.standard_normal((G, 2 * N, K)) / np.sqrt(K))
    W2 = bf16_cpu(rng.standard_normal((G, K, N)) / np.sqrt(N))
    probs_h = torch.from_numpy(rng.uniform(0.1, 1, M).astype(np.float32))
    h_host = bf16_cpu(1.5 * rng.standard_normal((M, 2 * N)))
    dy = bf16_cpu(rng.standard_normal((M, K)))
    dx, dprob, fc1 = run_backward(gm, dy, splits, W1, W2, h_host.cuda(), probs_h.cuda(), 0)
    ref = orc.backward_dgrad(bits(dy), np.array(splits_l), bits(W1), bits(W2), bits(h_host), probs_h.numpy(), 0)
    assert frob(dx.float().cpu().numpy(), orc.bf16_to_f64(ref["dx"])) <= 1e-2
    assert frob(dprob.cpu().numpy(), ref["dprob"]) <= 1e-2
    assert float(np.mean(np_bits(fc1["bf16"]) == ref["fc1_dy"])) >= 0.99


def test_backward_dgrad_full_size_sampled(orc, gm):
    """The full headline workload (MXFP8 SwiGLU, 8 experts, K=2048, N=1024,
    16384 tokens, Dirichlet splits with an empty expert) in the launch
    configuration the benchmark times.  Each row of dx, dprob and fc1_dy
    depends only on its own dy and h rows and its expert's weights, and every
    MXFP8 block lies along a row, so the oracle evaluates a row sample covering
    every non-empty expert (its first and last rows included)."""
    from mxfp8_nvfp4_block_gb300.inputs import make_inputs
    w = make_inputs("mx_swiglu")
    wl = w["workload"]
    sp = w["splits"].numpy()
    M, K, N = wl.M, wl.K, wl.N
    gen = torch.Generator().manual_seed(99)
    dy = torch.randn((M, K), generator=gen).to(torch.bfloat16)
    h = (1.5 * torch.randn((M, 2 * N), generator=gen)).to(torch.bfloat16)
    probs = w["probs"]
    dx, dprob, fc1 = run_backward(gm, dy, w["splits"], w["W1"], w["W2"], h.cuda(), probs.cuda(), 0)
    offs = orc.group_offsets(sp)
    rng = np.random.default_rng(9)
    rows = []
    for g in range(len(sp)):
        if sp[g]:
            pick = [offs[g], offs[g + 1] - 1] + list(rng.integers(offs[g], offs[g + 1], min(16, int(sp[g]))))
            rows += sorted(set(int(r) for r in pick))
    rows = np.array(rows, dtype=np.int64)
    sub = np.array([np.count_nonzero((rows >= offs[g]) & (rows < offs[g + 1])) for g in range(len(sp))])
    ref = orc.backward_dgrad(bits(dy)[rows], sub, bits(w["W1"]), bits(w["W2"]), bits(h)[rows], probs.numpy()[rows],
                             0)
    fb = np_bits(fc1["bf16"])[rows]
    bmatch = float(np.mean(fb == ref["fc1_dy"]))
    frac, steps = code_match_report(0, np_u8(fc1["codes"], M * 2 * N).reshape(M, 2 * N)[rows], ref["fc1_dy_codes"],
                                    orc.tiled_to_compact(np_u8(fc1["scales"]), sp, 2 * N // 32)[rows],
                                    ref["fc1_dy_scales"])
    err = frob(dx.float().cpu().numpy()[rows], orc.bf16_to_f64(ref["dx"]))
    perr = frob(dprob.cpu().numpy()[rows], ref["dprob"])
    print(f"full-size dgrad, {len(rows)} rows: fc1_dy bf16 match {bmatch:.6f}, code match {frac:.6f} "
          f"(max {steps:.2f} steps), dx error {err:.3e}, dprob error {perr:.3e}")
    assert bmatch >= 0.99 and frac >= 0.999 and steps <= 1.0 + 1e-9, (bmatch, frac, steps)
    assert err <= 1e-2 and perr <= 1e-2
