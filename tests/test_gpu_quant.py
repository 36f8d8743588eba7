"""Parity of the group quantisers (CUDA path, through the C ABI) with the oracle:
codes, block scales and amaxes bit-exact for the same bf16 input."""
import numpy as np
import pytest
import torch

from mxfp8_nvfp4_block_gb300.inputs import bits
from parity import np_u8

pytestmark = pytest.mark.gpu

SPLITS = {
    "tiny": [200, 150, 100, 62],
    "edges": [0, 1, 15, 16, 17, 31, 33, 0, 128, 129, 255, 257],
    "empty_first": [0, 0, 300],
    "single_row": [1],
}


def bf16_cpu(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)


def rich_x(M: int, K: int, seed: int) -> torch.Tensor:
    """Rows with magnitudes over many binades, finite bf16 bit patterns (|v| < 1e30,
    so 16-term Hadamard sums stay finite) scattered in, exact E4M3 rounding
    midpoints and signed zeros."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)) * np.exp2(rng.integers(-40, 40, (M, 1)))
    t = bf16_cpu(x)
    flat = t.view(torch.int16).view(-1)
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = (pats.astype(np.uint32) << 16).view(np.float32)
    pats = pats[np.isfinite(f) & (np.abs(f) < 1e30)]
    n = min(flat.numel() // 3, len(pats))
    pos = torch.from_numpy(rng.choice(flat.numel(), n, replace=False))
    flat[pos] = torch.from_numpy(rng.choice(pats, n, replace=False).view(np.int16))
    if M >= 4 and K >= 64:
        # row 1, block 0: amax 16 (scale exponent -4) and the other 31 values on
        # E4M3 rounding midpoints of the scaled block; row 2: zeros and -0
        mids = np.array([(8 + m + 0.5) * 2.0 ** (j - 3) for j in range(4) for m in range(8)]) / 16.0
        mids[0] = 16.0
        mids[1::3] *= -1
        t[1, :32] = bf16_cpu(mids)
        t[2, :64] = 0.0
        t[2, 1:64:2] = -0.0
    return t


def gpu_call(gm, fn, *a, **k):
    out = fn(*a, **k)
    gm.check_device_status()
    return out


# K = 128, 384: rows shorter than one 128-chunk pass; 1152: one full pass and a
# ragged one; 2048: full passes only
@pytest.mark.parametrize("layout", [0, 1], ids=["compact", "tiled"])
@pytest.mark.parametrize("K", [128, 384, 1152, 2048])
@pytest.mark.parametrize("case", list(SPLITS))
def test_mxfp8_rowwise_bitexact(orc, gm, case, K, layout):
    splits = np.array(SPLITS[case], dtype=np.int64)
    M = int(splits.sum())
    x = rich_x(M, K, seed=K + len(splits))
    out = gpu_call(gm, gm.group_quantize, x.cuda(), torch.from_numpy(splits).cuda(), gm.recipe(gm.MXFP8, layout=layout))
    ref = orc.group_quantize(bits(x), splits, orc.MXFP8)
    assert np.array_equal(np_u8(out["row"][0], M * K).reshape(M, K), ref["row_codes"])
    sc = np_u8(out["row"][1])
    got = orc.tiled_to_compact(sc, splits, K // 32) if layout else sc[:M * K // 32].reshape(M, K // 32)
    assert np.array_equal(got, ref["row_scales"])


@pytest.mark.parametrize("layout", [0, 1], ids=["compact", "tiled"])
@pytest.mark.parametrize("K", [256, 1152, 2048])
@pytest.mark.parametrize("case", list(SPLITS))
def test_nvfp4_rowwise_bitexact(orc, gm, case, K, layout):
    splits = np.array(SPLITS[case], dtype=np.int64)
    M = int(splits.sum())
    x = rich_x(M, K, seed=7 + len(splits))
    out = gpu_call(gm, gm.group_quantize, x.cuda(), torch.from_numpy(splits).cuda(),
                   gm.recipe(gm.NVFP4, layout=layout))
    ref = orc.group_quantize(bits(x), splits, orc.NVFP4)
    assert np.array_equal(out["amax_pre"].cpu().numpy(), ref["amax_pre"])
    assert np.array_equal(np_u8(out["row"][0], M * K // 2).reshape(M, K // 2), ref["row_codes"])
    sc = np_u8(out["row"][1])
    got = orc.tiled_to_compact(sc, splits, K // 16) if layout else sc[:M * K // 16].reshape(M, K // 16)
    assert np.array_equal(got, ref["row_scales"])


def test_nvfp4_rowwise_every_bf16_block_max(orc, gm):
    """Every positive finite bf16 magnitude is the max of one 16-element block
    (one row of 128 consecutive magnitudes per group, so the block scales span
    the E4M3 range); codes, scales and amaxes bit-exact."""
    K = 2048
    pats = np.arange(1, 0x7F80, dtype=np.uint32)
    M = -(-len(pats) // (K // 16))
    pats = np.concatenate([pats, np.full(M * (K // 16) - len(pats), 0x3F80, np.uint32)])
    rng = np.random.default_rng(11)
    top = (pats << 16).view(np.float32).astype(np.float64)
    x = top[:, None] * rng.uniform(0.0, 1.0, (len(pats), 16))
    x[:, 0] = top
    x *= rng.choice([-1.0, 1.0], x.shape)
    xt = bf16_cpu(x.reshape(M, K))
    splits = np.ones(M, dtype=np.int64)
    for lo in range(0, M, 512):  # at most 512 groups per call
        part = xt[lo:lo + 512]
        sp = splits[lo:lo + 512]
        m = part.shape[0]
        out = gpu_call(gm, gm.group_quantize, part.cuda(), torch.from_numpy(sp).cuda(), gm.recipe(gm.NVFP4, layout=0))
        ref = orc.group_quantize(bits(part), sp, orc.NVFP4)
        assert np.array_equal(out["amax_pre"].cpu().numpy(), ref["amax_pre"])
        assert np.array_equal(np_u8(out["row"][0], m * K // 2).reshape(m, K // 2), ref["row_codes"])
        assert np.array_equal(np_u8(out["row"][1])[:m * K // 16].reshape(m, K // 16), ref["row_scales"])


@pytest.mark.parametrize("mask", [0, 0xFFFF, 0x5A3C, 0x8001])
@pytest.mark.parametrize("case", ["tiny", "edges", "empty_first"])
def test_hadamard_amax_bitexact(orc, gm, case, mask):
    splits = np.array(SPLITS[case], dtype=np.int64)
    M, K = int(splits.sum()), 384
    x = rich_x(M, K, seed=mask & 255)
    pre, post = gpu_call(gm, gm.group_hadamard_amax, x.cuda(), torch.from_numpy(splits).cuda(), mask)
    rpre, rpost = orc.group_hadamard_amax(bits(x), splits, mask)
    assert np.array_equal(pre.cpu().numpy(), rpre)
    assert np.array_equal(post.cpu().numpy(), rpost)


@pytest.mark.parametrize("use_rht", [True, False])
@pytest.mark.parametrize("rowwise", [True, False])
@pytest.mark.parametrize("case", ["tiny", "edges"])
def test_nvfp4_row_col_with_amax_bitexact(orc, gm, case, rowwise, use_rht):
    """Caller-supplied amaxes (deliberately not the tensor's own) reach both sides."""
    splits = np.array(SPLITS[case], dtype=np.int64)
    M, K = int(splits.sum()), 256
    x = rich_x(M, K, 5)
    rng = np.random.default_rng(9)
    pre, post = orc.group_hadamard_amax(bits(x), splits, 0x1234)
    pre = (pre * rng.uniform(1.0, 1.5, len(splits))).astype(np.float32)
    post = (post * rng.uniform(1.0, 1.5, len(splits))).astype(np.float32)
    rec = gm.recipe(gm.NVFP4, use_rht=use_rht, mask=0x1234, layout=1)
    out = gpu_call(gm, gm.group_quantize_with_amax, x.cuda(), torch.from_numpy(splits).cuda(), rec,
                   torch.from_numpy(pre).cuda(), torch.from_numpy(post).cuda(), rowwise=rowwise,
                   columnwise=True, splits_host=splits.tolist())
    ref = orc.group_quantize_with_amax(bits(x), splits, orc.NVFP4, pre, post, rowwise=rowwise, columnwise=True,
                                       use_rht=use_rht, mask=0x1234)
    nb = len(ref["col_codes"])
    assert np.array_equal(np_u8(out["col"][0], nb), ref["col_codes"])
    assert np.array_equal(np_u8(out["col"][1], len(ref["col_scales"])), ref["col_scales"])
    if rowwise:
        assert np.array_equal(np_u8(out["row"][0], M * K // 2).reshape(M, K // 2), ref["row_codes"])
        assert np.array_equal(orc.tiled_to_compact(np_u8(out["row"][1]), splits, K // 16), ref["row_scales"])


@pytest.mark.parametrize("scale_exp", [-110, -126, -133])
def test_nvfp4_row_col_tiny_groups_bitexact(orc, gm, scale_exp):
    """Groups whose values all lie far below 2^-100 (down to bf16 subnormals),
    beside a group of ordinary magnitude: the columnwise RHT cast's quarter
    scaling cannot fold into the encode factor there and takes the plain path;
    codes and scales bit-exact, own amaxes."""
    splits = np.array([48, 37, 16, 1], dtype=np.int64)
    M, K = int(splits.sum()), 384
    rng = np.random.default_rng(-scale_exp)
    x = rng.standard_normal((M, K))
    x[48:] *= 2.0 ** scale_exp
    x = bf16_cpu(x)
    pre, post = orc.group_hadamard_amax(bits(x), splits, 0x9E37)
    rec = gm.recipe(gm.NVFP4, use_rht=True, mask=0x9E37, layout=1)
    out = gpu_call(gm, gm.group_quantize_with_amax, x.cuda(), torch.from_numpy(splits).cuda(), rec,
                   torch.from_numpy(pre).cuda(), torch.from_numpy(post).cuda(), rowwise=True, columnwise=True,
                   splits_host=splits.tolist())
    ref = orc.group_quantize_with_amax(bits(x), splits, orc.NVFP4, pre, post, rowwise=True, columnwise=True,
                                       use_rht=True, mask=0x9E37)
    assert np.array_equal(np_u8(out["col"][0], len(ref["col_codes"])), ref["col_codes"])
    assert np.array_equal(np_u8(out["col"][1], len(ref["col_scales"])), ref["col_scales"])
    assert np.array_equal(np_u8(out["row"][0], M * K // 2).reshape(M, K // 2), ref["row_codes"])
    assert np.array_equal(orc.tiled_to_compact(np_u8(out["row"][1]), splits, K // 16), ref["row_scales"])


@pytest.mark.parametrize("fmt", [0, 1], ids=["mxfp8", "nvfp4"])
@pytest.mark.parametrize("swiglu", [False, True])
def test_prepare_weights_bitexact(orc, gm, fmt, swiglu):
    G, rows, cols = 3, 256, 512
    rng = np.random.default_rng(fmt * 2 + swiglu)
    W = bf16_cpu(rng.standard_normal((G, rows, cols)) * np.array([1.0, 1e-3, 30.0])[:, None, None])
    qw = gpu_call(gm, gm.prepare_weights, W.cuda(), fmt, swiglu_interleave=swiglu)
    ref = orc.quantize_weights(bits(W), fmt)
    blk, cdiv = (32, 1) if fmt == 0 else (16, 2)
    codes = np_u8(qw.codes, G * rows * cols // cdiv).reshape(G, rows, cols // cdiv)
    scales = orc.tiled_to_compact(np_u8(qw.scales), [rows] * G, cols // blk).reshape(G, rows, cols // blk)
    if swiglu:   # prepared row p of an expert holds logical row perm[p]
        n = rows // 2
        perm = np.array([(32 * (p // 64) + p % 64) if p % 64 < 32 else (n + 32 * (p // 64) + p % 64 - 32)
                         for p in range(rows)])
        codes, scales = codes[:, np.argsort(perm)], scales[:, np.argsort(perm)]
    assert np.array_equal(codes, ref["codes"])
    assert np.array_equal(scales, ref["scales"])
    if fmt == 1:
        assert np.array_equal(qw.global_scale.cpu().numpy(), ref["S"])
        assert np.array_equal(qw.amax.cpu().numpy(), ref["amax"])


def test_all_empty_groups(orc, gm):
    splits = torch.zeros(5, dtype=torch.int64).cuda()
    x = torch.zeros((0, 128), dtype=torch.bfloat16).cuda()
    pre, post = gpu_call(gm, gm.group_hadamard_amax, x, splits, 0xBEEF)
    assert not pre.cpu().numpy().any() and not post.cpu().numpy().any()


def test_split_sizes_past_M_reported(gm):
    """A host-made failure: split sizes summing past M are caught on the device,
    nothing is written, and the status comes back through the status word."""
    x = torch.ones((64, 128), dtype=torch.bfloat16).cuda()
    splits = torch.tensor([40, 40], dtype=torch.int64).cuda()
    out = gm.group_quantize(x, splits, gm.recipe(gm.MXFP8))
    with pytest.raises(gm.GmlpError) as e:
        gm.check_device_status()
    assert e.value.status == gm.ERR_DEVICE_BOUNDS
    gm.check_device_status()        # cleared
    neg = torch.tensor([-1, 65], dtype=torch.int64).cuda()
    gm.group_hadamard_amax(x, neg, 0)
    with pytest.raises(gm.GmlpError):
        gm.check_device_status()
    del out


def test_bounded_wait_times_out_and_reports(gm):
    """A wait that nothing completes gives up after its limit; the host reads
    GMLP_ERR_DEVICE_TIMEOUT and the context keeps working."""
    import time
    t0 = time.time()
    gm.selftest_bounded_wait(50_000_000)           # 50 ms
    with pytest.raises(gm.GmlpError) as e:
        gm.check_device_status()
    assert e.value.status == gm.ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 10
    gm.check_device_status()                        # cleared
    x = torch.ones((32, 128), dtype=torch.bfloat16).cuda()
    pre, post = gm.group_hadamard_amax(x, torch.tensor([32]).cuda(), 0)
    gm.check_device_status()
    assert pre.item() == 1.0 and post.item() == 4.0


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", [0, 1])
def test_mma_peak_loop_runs_at_a_plausible_rate(gm, fmt):
    """The tensor-core ceiling loop completes, reports no device error and runs
    at a rate between a tenth of and just above the nominal dense peak (FP8
    4.5 PFLOP/s, FP4 13.5 PFLOP/s): far above would mean it skips work.  The
    lower bound only rules out a loop that barely runs: the short loop's rate
    varies with the shared GPU's clocks (the NVFP4 12-copy mode, ~3.9 PFLOP/s
    on an idle GPU, once measured 2.1)."""
    nominal = 4500.0 if fmt == gm.MXFP8 else 13500.0
    ctas = torch.cuda.get_device_properties(0).multi_processor_count
    for copy in ((1, 2, 3, 0) if fmt == gm.NVFP4 else (1, 3, 0)):
        gm.mma_peak(fmt, copy, 256)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        gm.mma_peak(fmt, copy, 8192)
        e1.record()
        torch.cuda.synchronize()
        gm.check_device_status()
        tflops = gm.mma_peak_flops(fmt, 8192, ctas) / (e0.elapsed_time(e1) * 1e-3) / 1e12
        assert nominal / 10 < tflops < nominal * 1.1, (copy, tflops)
