"""The forward and the backward captured in a CUDA graph and replayed: the
library allocates nothing and keeps split sizes on the device, so a captured
step replays on new inputs and new split sizes written into the captured
buffers and gives the eager call's bits (outputs reduced by atomics, dprob
and dbias, are left out: their summation order may differ)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).cuda()


def new_case(rng, splits_l, K, N, n1):
    M = sum(splits_l)
    return dict(x=bf16(rng.standard_normal((M, K))), splits=torch.tensor(splits_l, dtype=torch.int64).cuda(),
                probs=torch.from_numpy(rng.uniform(0.1, 1, M).astype(np.float32)).cuda(),
                dy=bf16(rng.standard_normal((M, K))), h=bf16(1.5 * rng.standard_normal((M, n1))))


@pytest.mark.parametrize("fmt", [0, 1], ids=["mxfp8", "nvfp4"])
def test_forward_graph_replay(gm, fmt):
    rng = np.random.default_rng(51 + fmt)
    G, K, N = 4, 512, 256
    act = gm.SWIGLU if fmt == gm.MXFP8 else gm.SRELU
    n1 = 2 * N if act == gm.SWIGLU else N
    W1 = gm.prepare_weights(bf16(rng.standard_normal((G, n1, K)) / np.sqrt(K)), fmt,
                            swiglu_interleave=(act == gm.SWIGLU))
    W2 = gm.prepare_weights(bf16(rng.standard_normal((G, K, N)) / np.sqrt(N)), fmt)
    rec = gm.recipe(fmt, use_rht=True, mask=0x5A3C)
    M = 520
    cases = [new_case(rng, s, K, N, n1) for s in ([130, 0, 257, 133], [5, 300, 0, 215], [0, 0, 520, 0])]
    buf = {k: v.clone() for k, v in cases[0].items()}
    y = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(gm.forward_workspace_size(M, K, N, G, act, rec), dtype=torch.uint8, device="cuda")
    gm.forward(buf["x"], buf["splits"], W1, W2, buf["probs"], act, rec, y=y, workspace=ws)  # warm-up
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gm.forward(buf["x"], buf["splits"], W1, W2, buf["probs"], act, rec, y=y, workspace=ws)
    for c in cases:
        for k in ("x", "splits", "probs"):
            buf[k].copy_(c[k])
        graph.replay()
        torch.cuda.synchronize()
        want = gm.forward(c["x"], c["splits"], W1, W2, c["probs"], act, rec)
        gm.check_device_status()
        assert torch.equal(y.view(torch.int16), want.view(torch.int16))


def test_backward_graph_replay(gm):
    """dgrad (dy cast, dGLU, dgrad) and wgrad (four columnwise casts, two
    grouped GEMMs) captured as one graph."""
    rng = np.random.default_rng(61)
    G, K, N = 4, 512, 256
    n1 = 2 * N
    W1b = bf16(rng.standard_normal((G, n1, K)) / np.sqrt(K))
    W2b = bf16(rng.standard_normal((G, K, N)) / np.sqrt(N))
    w2t, w1t = gm.prepare_transposed_weights(W2b), gm.prepare_transposed_weights(W1b)
    rec = gm.recipe(gm.MXFP8)
    M = 520
    cases = [new_case(rng, s, K, N, n1) for s in ([130, 0, 257, 133], [5, 300, 0, 215])]
    buf = {k: v.clone() for k, v in cases[0].items()}
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    f1 = torch.empty((M, n1), dtype=torch.bfloat16, device="cuda")
    wsd = torch.empty(gm.load().gmlp_backward_workspace_size(M, K, N, G, gm.SWIGLU), dtype=torch.uint8,
                      device="cuda")
    wsw = torch.empty(gm.load().gmlp_backward_wgrad_workspace_size(M, K, N, G, gm.SWIGLU), dtype=torch.uint8,
                      device="cuda")
    grads = {"dW1": torch.empty((G, n1, K), device="cuda"), "dW2": torch.empty((G, K, N), device="cuda")}

    def step(b):
        gm.backward_dgrad(b["dy"], b["splits"], w2t, w1t, b["h"], b["probs"], gm.SWIGLU, rec, dx=dx,
                          fc1_dy_bf16=f1, workspace=wsd, want_dprob=False)
        gm.backward_wgrad(b["x"], b["dy"], b["h"], b["probs"], f1, b["splits"], gm.SWIGLU, want=("dW1", "dW2"),
                          workspace=wsw, **grads)

    step(buf)  # warm-up
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(buf)
    for c in cases:
        for k in buf:
            buf[k].copy_(c[k])
        graph.replay()
        torch.cuda.synchronize()
        got = {"dx": dx.clone(), "f1": f1.clone(), "dW1": grads["dW1"].clone(), "dW2": grads["dW2"].clone()}
        wdx, _ = gm.backward_dgrad(c["dy"], c["splits"], w2t, w1t, c["h"], c["probs"], gm.SWIGLU, rec,
                                   fc1_dy_bf16=f1, want_dprob=False)
        wg = gm.backward_wgrad(c["x"], c["dy"], c["h"], c["probs"], f1, c["splits"], gm.SWIGLU, want=("dW1", "dW2"))
        gm.check_device_status()
        assert torch.equal(got["dx"].view(torch.int16), wdx.view(torch.int16))
        assert torch.equal(got["f1"].view(torch.int16), f1.view(torch.int16))
        assert torch.equal(got["dW1"], wg["dW1"]) and torch.equal(got["dW2"], wg["dW2"])
