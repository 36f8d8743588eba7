"""The NVFP4 activation-recompute path (PR #3837, Description: with activation
recompute the backward rebuilds fc2_x instead of keeping it, and "recompute on
and off give bitwise-equal output and gradients"; Changes: the column-wise
NVFP4 cast of the rebuilt fc2_x reuses the forward's amaxes through
quantize-with-amax).

* gmlp_fc2x_recompute against the oracle on seeded activation inputs: bit for
  bit for SReLU (exact FP32 arithmetic), within one bf16 step for SwiGLU and
  tanh-SReLU (FP32 exp / tanh on the GPU against the oracle's float64).
* Recompute on / off: fc2_x rebuilt on the GPU from the forward's saved
  activation input equals the forward's own fc2_x bit for bit, and its
  quantize-with-amax cast with the forward's saved amaxes reproduces the
  forward's rowwise operand and its columnwise (RHT) output bit for bit, for
  SReLU, tanh-SReLU and SwiGLU.
"""
import numpy as np
import pytest
import torch

from mxfp8_nvfp4_block_gb300.inputs import bits
from parity import np_bits

pytestmark = pytest.mark.gpu

CLAMP = 8.0


def bf16_cpu(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)


def _sync(gm):
    gm.check_device_status()
    torch.cuda.synchronize()


@pytest.mark.parametrize("act", [0, 1, 2], ids=["swiglu", "srelu", "tanh_srelu"])
def test_fc2x_recompute_matches_oracle(orc, gm, act):
    rng = np.random.default_rng(40 + act)
    M, N = 777, 384
    n1 = 2 * N if act == gm.SWIGLU else N
    h = bf16_cpu(rng.standard_normal((M, n1)) * 2.5)
    h[5, :] = 0.0
    probs = torch.from_numpy(rng.uniform(0, 1, M).astype(np.float32))
    c = CLAMP if act == gm.TANH_SRELU else 0.0
    out = gm.fc2x_recompute(h.cuda(), probs.cuda(), act, tanh_clamp_scale=c)
    _sync(gm)
    got = np_bits(out)
    ref = orc.recompute_fc2x(bits(h), probs.numpy(), act, c or None)
    if act == gm.SRELU:
        assert np.array_equal(got, ref)
        return
    gv, rv = orc.bf16_to_f64(got), orc.bf16_to_f64(ref)
    step = np.ldexp(1.0, np.floor(np.log2(np.maximum(np.abs(rv), 1e-30))).astype(np.int64) - 7)
    assert (np.abs(gv - rv) <= step).all()              # at most one bf16 step apart
    assert (got == ref).mean() > 0.99


@pytest.mark.parametrize("act", [0, 1, 2], ids=["swiglu", "srelu", "tanh_srelu"])
def test_nvfp4_recompute_on_off_bitwise_equal(orc, gm, act):
    splits = [130, 0, 257, 5, 300, 1]
    G, M, K, N = len(splits), sum(splits), 512, 512
    n1 = 2 * N if act == gm.SWIGLU else N
    rng = np.random.default_rng(70 + act)
    x = bf16_cpu(rng.standard_normal((M, K)))
    W1 = bf16_cpu(rng.standard_normal((G, n1, K)) / np.sqrt(K))
    W2 = bf16_cpu(rng.standard_normal((G, K, N)) / np.sqrt(N))
    probs = torch.from_numpy(rng.uniform(0, 1, M).astype(np.float32)).cuda()
    sp = torch.tensor(splits, dtype=torch.int64).cuda()
    mask = 0x6B2D
    rec = gm.recipe(gm.NVFP4, use_rht=True, mask=mask)
    w1 = gm.prepare_weights(W1.cuda(), gm.NVFP4, swiglu_interleave=(act == gm.SWIGLU))
    w2 = gm.prepare_weights(W2.cuda(), gm.NVFP4)
    ncol = N * (M + 16 * G)
    aux = {"fc1_pre_act": torch.zeros((M, n1), dtype=torch.bfloat16, device="cuda"),
           "fc2x_bf16": torch.zeros((M, N), dtype=torch.bfloat16, device="cuda"),
           "fc2x_codes": torch.zeros(M * N // 2, dtype=torch.uint8, device="cuda"),
           "fc2x_scales": torch.zeros(gm.tiled_scales_bytes(M, G, N // 16), dtype=torch.uint8, device="cuda"),
           "fc2x_amax_pre": torch.zeros(G, dtype=torch.float32, device="cuda"),
           "fc2x_amax_post": torch.zeros(G, dtype=torch.float32, device="cuda"),
           "fc2x_col_codes": torch.zeros(ncol // 2, dtype=torch.uint8, device="cuda"),
           "fc2x_col_scales": torch.zeros(ncol // 16, dtype=torch.uint8, device="cuda")}
    c = CLAMP if act == gm.TANH_SRELU else 0.0
    gm.forward(x.cuda(), sp, w1, w2, probs, act, rec, aux=aux, tanh_clamp_scale=c)
    _sync(gm)
    assert torch.count_nonzero(aux["fc2x_bf16"]) > M * N // 4

    # recompute on: rebuild fc2_x from the saved activation input, then the cast
    f = gm.fc2x_recompute(aux["fc1_pre_act"], probs, act, tanh_clamp_scale=c)
    _sync(gm)
    assert torch.equal(f.view(torch.int16), aux["fc2x_bf16"].view(torch.int16))
    out = gm.group_quantize_with_amax(f, sp, rec, aux["fc2x_amax_pre"], aux["fc2x_amax_post"], rowwise=True,
                                      columnwise=True, splits_host=splits)
    _sync(gm)
    mpad = sum((m + 15) // 16 * 16 for m in splits)
    nb, ns = N * mpad // 2, N * mpad // 16
    assert torch.equal(out["col"][0][:nb], aux["fc2x_col_codes"][:nb])
    assert torch.equal(out["col"][1][:ns], aux["fc2x_col_scales"][:ns])
    assert torch.equal(out["row"][0][:M * N // 2], aux["fc2x_codes"])
    # rowwise scales: compare the bytes the groups own (padding rows unspecified)
    own = torch.from_numpy(orc.tiled_index(splits, N // 16).reshape(-1)).cuda()
    assert torch.equal(out["row"][1][own], aux["fc2x_scales"][own])
