"""The oracle's backward pinned to an independent derivative: torch's float64
autograd of the plain (unquantised) MLP.  SReLU, one-hot +-1 weights and
small-integer operands keep every quantised step of the forward and of both
backward halves exact (every fc1_dy value has at most four significant bits),
so the oracle's data, probability and weight gradients must equal autograd's
bit for bit (CPU)."""
import numpy as np
import torch


def as_bits(a):
    return torch.from_numpy(np.asarray(a, np.float64).astype(np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def test_backward_equals_autograd_of_the_plain_mlp(orc):
    rng = np.random.default_rng(13)
    splits = np.array([40, 0, 70, 33])
    G, K, N = len(splits), 64, 32
    offs = orc.group_offsets(splits)
    M = int(offs[-1])
    x = rng.choice([0.0, 1.0, -1.0, 2.0], size=(M, K))
    dy = rng.choice([0.0, 1.0, -1.0, 2.0, -2.0], size=(M, K))
    probs = rng.choice([1.0, 0.5], size=M).astype(np.float32)
    W1 = np.zeros((G, N, K))
    W2 = np.zeros((G, K, N))
    for g in range(G):
        W1[g, np.arange(N), rng.integers(0, K, N)] = rng.choice([1.0, -1.0], size=N)   # h = +-x[:, j]
        W2[g, np.arange(K), rng.integers(0, N, K)] = rng.choice([1.0, -1.0], size=K)   # y reads one fc2_x column

    # autograd of y_g = (relu(x_g W1_g^T)^2 * p) W2_g^T, L = sum(y * dy)
    xt = torch.tensor(x, requires_grad=True)
    pt = torch.tensor(probs.astype(np.float64), requires_grad=True)
    W1t = torch.tensor(W1, requires_grad=True)
    W2t = torch.tensor(W2, requires_grad=True)
    loss = 0.0
    for g in range(G):
        r0, r1 = int(offs[g]), int(offs[g + 1])
        if r1 == r0:
            continue
        h = xt[r0:r1] @ W1t[g].T
        f = torch.relu(h) ** 2 * pt[r0:r1, None]
        loss = loss + ((f @ W2t[g].T) * torch.tensor(dy[r0:r1])).sum()
    loss.backward()

    fwd = orc.forward(as_bits(x), splits, as_bits(W1), as_bits(W2), probs, orc.SRELU, orc.MXFP8)
    bd = orc.backward_dgrad(as_bits(dy), splits, as_bits(W1), as_bits(W2), fwd["h"], probs, orc.SRELU)
    bw = orc.backward_wgrad(as_bits(x), as_bits(dy), fwd["h"], probs, bd["fc1_dy"], splits, orc.SRELU)
    np.testing.assert_array_equal(orc.bf16_to_f64(bd["dx"]), xt.grad.numpy())
    np.testing.assert_array_equal(bd["dprob"], pt.grad.numpy())
    np.testing.assert_array_equal(bw["dW1"], W1t.grad.numpy())
    np.testing.assert_array_equal(bw["dW2"], W2t.grad.numpy())
    assert np.abs(xt.grad.numpy()).max() > 0 and np.abs(W2t.grad.numpy()).max() > 0


def test_swiglu_backward_close_to_autograd_of_the_plain_mlp(orc):
    """SwiGLU with random operands: the oracle's quantised backward against
    torch's float64 autograd of the unquantised MLP y_g = (silu(x W1g_gate^T) *
    (x W1g_up^T) * p) W2_g^T.  Each MXFP8 cast (3 mantissa bits) adds about
    2.5% RMS relative error and every gradient passes through five or six of
    them, so 6-8% is expected and 12% is the bound; a wrong wiring (gate and
    up swapped, the prob misplaced, a missing term of the SwiGLU derivative, a
    transposed weight) gives errors of order one."""
    rng = np.random.default_rng(29)
    splits = np.array([70, 0, 130, 33])
    G, K, N = len(splits), 128, 64
    offs = orc.group_offsets(splits)
    M = int(offs[-1])
    bfr = lambda a: orc.bf16_to_f64(as_bits(np.asarray(a, np.float32)))   # values as the bf16 inputs hold them
    x, dy = bfr(rng.standard_normal((M, K))), bfr(rng.standard_normal((M, K)))
    W1, W2 = bfr(rng.standard_normal((G, 2 * N, K)) / np.sqrt(K)), bfr(rng.standard_normal((G, K, N)) / np.sqrt(N))
    probs = rng.uniform(0.1, 1.0, M).astype(np.float32)

    xt = torch.tensor(x, requires_grad=True)
    pt = torch.tensor(probs.astype(np.float64), requires_grad=True)
    W1t, W2t = torch.tensor(W1, requires_grad=True), torch.tensor(W2, requires_grad=True)
    loss = 0.0
    for g in range(G):
        r0, r1 = int(offs[g]), int(offs[g + 1])
        if r1 == r0:
            continue
        h = xt[r0:r1] @ W1t[g].T
        f = torch.nn.functional.silu(h[:, :N]) * h[:, N:] * pt[r0:r1, None]
        loss = loss + ((f @ W2t[g].T) * torch.tensor(dy[r0:r1])).sum()
    loss.backward()

    def rel(a, b):
        return float(np.linalg.norm(a - b) / np.linalg.norm(b))

    fwd = orc.forward(as_bits(x), splits, as_bits(W1), as_bits(W2), probs, orc.SWIGLU, orc.MXFP8)
    bd = orc.backward_dgrad(as_bits(dy), splits, as_bits(W1), as_bits(W2), fwd["h"], probs, orc.SWIGLU)
    bw = orc.backward_wgrad(as_bits(x), as_bits(dy), fwd["h"], probs, bd["fc1_dy"], splits, orc.SWIGLU)
    errs = dict(dx=rel(orc.bf16_to_f64(bd["dx"]), xt.grad.numpy()), dprob=rel(bd["dprob"], pt.grad.numpy()),
                dW1=rel(bw["dW1"], W1t.grad.numpy()), dW2=rel(bw["dW2"], W2t.grad.numpy()))
    print("SwiGLU backward vs float64 autograd:", {k: f"{v:.3e}" for k, v in errs.items()})
    for k, v in errs.items():
        assert v <= 0.12, (k, v)
    # the same comparison with gate and up swapped in the oracle's inputs fails
    W1s = np.concatenate([W1[:, N:], W1[:, :N]], axis=1)
    fwd_s = orc.forward(as_bits(x), splits, as_bits(W1s), as_bits(W2), probs, orc.SWIGLU, orc.MXFP8)
    bd_s = orc.backward_dgrad(as_bits(dy), splits, as_bits(W1s), as_bits(W2), fwd_s["h"], probs, orc.SWIGLU)
    swapped = rel(orc.bf16_to_f64(bd_s["dx"]), xt.grad.numpy())
    print(f"gate and up swapped: dx error {swapped:.3f}")
    assert swapped > 0.5
