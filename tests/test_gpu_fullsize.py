"""Full-size parity of the group quantisers (CUDA path, through the C ABI) with
the oracle, bit for bit, on the workloads' own inputs and in the launch
configuration the benchmark uses (persistent grids, many work units per CTA).

* The standalone NVFP4 quantiser on bf16 [131072, 4096] in 8 Dirichlet(0.5)
  groups with the workload's sign mask (PR #3837, Changes: the group
  Hadamard-amax pass and the quantize-with-amax cast; Description: the
  fc2-input group quantize, row + column): amax_pre / amax_post, rowwise codes
  and GEMM_TILED scales, columnwise RHT codes and scales.
* The NVFP4 forward's fc2_x amaxes on the nv_srelu workload against the
  standalone Hadamard-amax kernel and the oracle over the stored bf16 fc2_x.
* The forward's x casts on each forward workload's whole x: MXFP8 at K = 256
  (512 tokens in 4 ragged experts) and K = 2048 (16384 tokens, Dirichlet
  routing with an empty expert), NVFP4 at K = 4096 (32768 tokens with 0.1%
  outliers x50) and MXFP8 at K = 7168 (65536 tokens in 64 Zipf-routed experts,
  tail experts of 0-8 tokens).

Inputs come from the seeded generators; the oracle sees only their host
copies and its own results.
"""
import numpy as np
import pytest
import torch

from mxfp8_nvfp4_block_gb300.inputs import bits, make_inputs
from parity import np_u8

pytestmark = pytest.mark.gpu


def _check(gm, out):
    gm.check_device_status()
    torch.cuda.synchronize()
    return out


@pytest.fixture(scope="module")
def nv_quant(orc):
    d = make_inputs("nv_quant")
    xb = bits(d["x"])
    s = d["splits"].numpy()
    pre, post = orc.group_hadamard_amax(xb, s, d["mask"])
    ref = orc.group_quantize_with_amax(xb, s, orc.NVFP4, pre, post, rowwise=True, columnwise=True, use_rht=True,
                                       mask=d["mask"])
    return d, xb, s, pre, post, ref


def test_nv_quant_hadamard_amax_fullsize(gm, nv_quant):
    d, _, s, pre, post, _ = nv_quant
    assert (s > 0).all() and s.max() > 4 * s.min()          # uneven groups
    gpre, gpost = _check(gm, gm.group_hadamard_amax(d["x"].cuda(), d["splits"].cuda(), d["mask"]))
    assert np.array_equal(gpre.cpu().numpy(), pre)
    assert np.array_equal(gpost.cpu().numpy(), post)


def _compare_row_col(orc, out, ref, s, M, K):
    assert np.array_equal(np_u8(out["row"][0], M * K // 2).reshape(M, K // 2), ref["row_codes"])
    assert np.array_equal(orc.tiled_to_compact(np_u8(out["row"][1]), s, K // 16), ref["row_scales"])
    nb, ns = len(ref["col_codes"]), len(ref["col_scales"])
    assert np.array_equal(np_u8(out["col"][0], nb), ref["col_codes"])
    assert np.array_equal(np_u8(out["col"][1], ns), ref["col_scales"])


def test_nv_quant_quantize_with_amax_fullsize(orc, gm, nv_quant):
    """The cast alone with the oracle's amaxes handed to it (host copies)."""
    d, _, s, pre, post, ref = nv_quant
    M, K = d["x"].shape
    rec = gm.recipe(gm.NVFP4, use_rht=True, mask=d["mask"], layout=gm.GEMM_TILED)
    out = _check(gm, gm.group_quantize_with_amax(d["x"].cuda(), d["splits"].cuda(), rec, torch.from_numpy(pre).cuda(),
                                                 torch.from_numpy(post).cuda(), rowwise=True, columnwise=True,
                                                 splits_host=s.tolist()))
    _compare_row_col(orc, out, ref, s, M, K)


def test_nv_quant_group_quantize_fullsize(orc, gm, nv_quant):
    """The generic call: amaxes on the device, then the cast, in one call."""
    d, _, s, pre, post, ref = nv_quant
    M, K = d["x"].shape
    rec = gm.recipe(gm.NVFP4, use_rht=True, mask=d["mask"], layout=gm.GEMM_TILED)
    out = _check(gm, gm.group_quantize(d["x"].cuda(), d["splits"].cuda(), rec, rowwise=True, columnwise=True,
                                       splits_host=s.tolist()))
    assert np.array_equal(out["amax_pre"].cpu().numpy(), pre)
    assert np.array_equal(out["amax_post"].cpu().numpy(), post)
    _compare_row_col(orc, out, ref, s, M, K)


@pytest.mark.parametrize("name,fmt", [("tiny", 0), ("mx_swiglu", 0), ("nv_srelu", 1), ("mx_skew", 0)],
                         ids=["mxfp8_K256", "mxfp8_K2048", "nvfp4_K4096", "mxfp8_K7168"])
def test_forward_x_cast_fullsize(orc, gm, name, fmt):
    """The forward's x cast (rowwise, GEMM_TILED scales: fc1's A operand) on
    the workload's whole x."""
    d = make_inputs(name, weights=False)
    M, K = d["x"].shape
    s = d["splits"].numpy()
    out = _check(gm, gm.group_quantize(d["x"].cuda(), d["splits"].cuda(), gm.recipe(fmt, layout=gm.GEMM_TILED)))
    ref = orc.group_quantize(bits(d["x"]), s, fmt)
    cdiv, blk = (1, 32) if fmt == 0 else (2, 16)
    assert np.array_equal(np_u8(out["row"][0], M * K // cdiv).reshape(M, K // cdiv), ref["row_codes"])
    assert np.array_equal(orc.tiled_to_compact(np_u8(out["row"][1]), s, K // blk), ref["row_scales"])
    if fmt == 1:
        assert np.array_equal(out["amax_pre"].cpu().numpy(), ref["amax_pre"])


@pytest.mark.parametrize("colwise", [False, True], ids=["cast_pass", "epilogue"])
def test_nv_srelu_forward_amaxes_fullsize(orc, gm, colwise):
    """The NVFP4 forward's fc2_x amaxes on the nv_srelu workload (32768 tokens,
    N = 2048): pre- and post-RHT amax equal, bit for bit, both the standalone
    Hadamard-amax kernel and the oracle's group Hadamard-amax over the bf16
    fc2_x the forward stored (PR #3837, Description: the fused amax equals the
    quantizer's own).  cast_pass: the post-RHT amax comes from the rowwise
    fc2_x cast; epilogue: from the fc1 epilogue (the columnwise variant)."""
    d = make_inputs("nv_srelu")
    w = d["workload"]
    M, N, G = w.M, w.N, w.G
    w1 = gm.prepare_weights(d["W1"].cuda(), gm.NVFP4)
    w2 = gm.prepare_weights(d["W2"].cuda(), gm.NVFP4)
    aux = {"fc2x_bf16": torch.zeros((M, N), dtype=torch.bfloat16, device="cuda"),
           "fc2x_amax_pre": torch.zeros(G, dtype=torch.float32, device="cuda"),
           "fc2x_amax_post": torch.zeros(G, dtype=torch.float32, device="cuda")}
    if colwise:
        ncol = N * (M + 16 * G)
        aux["fc2x_col_codes"] = torch.zeros(ncol // 2, dtype=torch.uint8, device="cuda")
        aux["fc2x_col_scales"] = torch.zeros(ncol // 16, dtype=torch.uint8, device="cuda")
    rec = gm.recipe(gm.NVFP4, use_rht=True, mask=d["mask"])
    gm.forward(d["x"].cuda(), d["splits"].cuda(), w1, w2, d["probs"].cuda(), w.act, rec, aux=aux)
    _check(gm, None)
    pre, post = gm.group_hadamard_amax(aux["fc2x_bf16"], d["splits"].cuda(), d["mask"])
    _check(gm, None)
    assert torch.equal(pre, aux["fc2x_amax_pre"]) and torch.equal(post, aux["fc2x_amax_post"])
    opre, opost = orc.group_hadamard_amax(bits(aux["fc2x_bf16"].cpu()), d["splits"].numpy(), d["mask"])
    assert np.array_equal(aux["fc2x_amax_pre"].cpu().numpy(), opre)
    assert np.array_equal(aux["fc2x_amax_post"].cpu().numpy(), opost)
