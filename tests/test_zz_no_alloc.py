"""gmlp_forward_noalloc: the forward for callers that cannot allocate device
memory (a host framework that owns all device memory through its own pool, a
loop that must not pay cudaMalloc's device synchronisation, a binding without a
device allocator).  It runs gmlp_forward's kernels on a fixed static scratch
inside the library instead of a caller workspace.

Checked through the C ABI against gmlp_forward (with a caller workspace) on
two calls in a row with different formats, so the second call starts from the
scratch contents the first one left behind.  This file is collected last so
that a run stopping at its first failure has run every other test already."""
import numpy as np
import pytest
import torch

from mxfp8_nvfp4_block_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

Y_TOL = 1e-2   # normalised Frobenius error, as in the forward parity tests


def frob(a, b):
    a, b = a.double().cpu().numpy(), b.double().cpu().numpy()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def case(gm, fmt, act):
    d = make_inputs("tiny")
    if act == gm.SRELU:
        d["W1"] = d["W1"][:, :256].contiguous()
    w1 = gm.prepare_weights(d["W1"].cuda(), fmt, swiglu_interleave=(act == gm.SWIGLU))
    w2 = gm.prepare_weights(d["W2"].cuda(), fmt)
    return d, w1, w2, gm.recipe(fmt, use_rht=True, mask=0x3C5A)


def test_noalloc_matches_forward_two_calls(gm):
    for fmt, act in ((gm.MXFP8, gm.SWIGLU), (gm.NVFP4, gm.SRELU)):
        d, w1, w2, rec = case(gm, fmt, act)
        x, s, p = d["x"].cuda(), d["splits"].cuda(), d["probs"].cuda()
        y_ref = gm.forward(x, s, w1, w2, p, act, rec)
        y = torch.full_like(y_ref, float("nan"))
        gm.forward_noalloc(x, s, w1, w2, p, act, rec, y=y)
        gm.check_device_status()
        torch.cuda.synchronize()
        assert not torch.isnan(y.float()).any()
        assert frob(y, y_ref) <= Y_TOL
        assert torch.equal(y, y_ref)      # same kernels, same inputs


def test_noalloc_rejects_sizes_beyond_its_scratch(gm):
    """131072 tokens at K = N = 256 need about 66 MB of scratch, above the fixed
    64 MiB: the call is refused before any launch.  Every buffer is a real
    device tensor of the right size, so a regression in the size check would
    still only touch valid memory."""
    d, w1, w2, rec = case(gm, gm.MXFP8, gm.SWIGLU)
    M, K, N, G = 1 << 17, 256, 256, 4
    assert gm.forward_workspace_size(M, K, N, G, gm.SWIGLU, rec) > 64 << 20
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    s = torch.tensor([M // 4] * 4, dtype=torch.int64, device="cuda")
    with pytest.raises(gm.GmlpError) as e:
        gm.forward_noalloc(x, s, w1, w2, None, gm.SWIGLU, rec, y=y)
    assert e.value.status == gm.ERR_WORKSPACE
    assert "scratch" in str(e.value)
    gm.check_device_status()
