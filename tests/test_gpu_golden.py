"""The review's ragged split (tests/golden/ragged_split.txt: [64, 65], a token
count that is not a multiple of 128) through the CUDA path, bit for bit against
the oracle on lossless operands: the forward in both formats and the weight
gradients."""
import numpy as np
import pytest
import torch

from mxfp8_nvfp4_block_gb300.inputs import bits
from parity import np_bits, np_u8
from test_gpu_forward import onehot_case, run_gpu
from test_gpu_wgrad import bf16_cpu, run_wgrad
from test_oracle_golden import read_golden

pytestmark = pytest.mark.gpu

SPLITS = read_golden("ragged_split.txt")["splits"]


@pytest.mark.parametrize("fmt", [0, 1], ids=["mxfp8", "nvfp4"])
def test_forward_review_split_bitexact(orc, gm, fmt):
    K, N = 256, 256
    d = onehot_case(fmt, 1, SPLITS, K, N, seed=70 + fmt)
    y, aux = run_gpu(gm, d, fmt, 1)
    ref = orc.forward(bits(d["x"]), np.array(SPLITS), bits(d["W1"]), bits(d["W2"]), d["probs"].numpy(), 1, fmt)
    M = sum(SPLITS)
    cdiv = 1 if fmt == 0 else 2
    assert np.array_equal(np_u8(aux["fc2x_codes"], M * N // cdiv).reshape(M, -1), ref["fc2x_codes"])
    assert np.array_equal(np_bits(y), ref["y"])


def test_wgrad_review_split_bitexact(orc, gm):
    rng = np.random.default_rng(71)
    K, N = 256, 256
    M = sum(SPLITS)
    d = dict(x=bf16_cpu(rng.choice([0.0, 1.0, -1.0], size=(M, K))),
             dy=bf16_cpu(rng.choice([0.0, 1.0, -1.0, 2.0], size=(M, K))),
             fc1_dy=bf16_cpu(rng.choice([0.0, 1.0, -2.0], size=(M, N))),
             h=bf16_cpu(rng.choice([0.0, 1.0, -1.0, 2.0], size=(M, N))),
             probs=torch.from_numpy(rng.choice([1.0, 0.5], size=M).astype(np.float32)))
    splits = torch.tensor(SPLITS, dtype=torch.int64)
    out = run_wgrad(gm, d, splits, 1)
    ref = orc.backward_wgrad(bits(d["x"]), bits(d["dy"]), bits(d["h"]), d["probs"].numpy(), bits(d["fc1_dy"]),
                             np.array(SPLITS), 1)
    for k in ("dW1", "dW2", "dbias1", "dbias2"):
        assert np.array_equal(out[k].cpu().numpy().astype(np.float64), ref[k]), k
