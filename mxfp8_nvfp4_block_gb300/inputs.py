"""Seeded synthetic inputs for the five workloads of the fused grouped-MLP forward.

This module holds no arithmetic of the method: it only draws random tensors.
It is the one module that both the CUDA path's tests/bench and the oracle's
tests use, so both sides see the same bytes.

Workloads (x ~ N(0,1) bf16 token-sorted [M, K]; W ~ N(0, 1/K) bf16; probs ~
U(0,1) fp32):

* ``tiny``      MXFP8 SwiGLU, G=4, K=256, N=256, splits [200,150,100,62], seed 0.
* ``mx_swiglu`` MXFP8 SwiGLU, G=8, K=2048, N=1024, M=16384; splits multinomial
  over Dirichlet(alpha=1) expert weights with expert 7's weight set to zero
  (so it gets no tokens), seed 1.
* ``nv_srelu``  NVFP4 + RHT squared-ReLU, G=8, K=4096, N=2048, M=32768 split
  uniformly; exactly round(0.001*M*K) entries of x (a random permutation's
  prefix) multiplied by 50; a random 16-bit RHT sign mask; seed 2.
* ``nv_tanh_srelu`` the ``nv_srelu`` inputs (same seed, same bytes) with the
  tanh-SReLU activation, soft-clamp scale 8.
* ``mx_skew``   MXFP8 SwiGLU, G=64, K=7168, N=2048, M=65536; counts multinomial
  over p_k ~ k^-1.1, then experts 56..63 overwritten with uniform integers in
  [0, 8] (expert 63 forced to 0) and expert 0 absorbing the difference; seed 3.
* ``nv_quant``  standalone NVFP4 group quantiser, G=8, x [131072, 4096],
  Dirichlet(alpha=0.5) splits, row + column outputs, random sign mask; seed 4.

Splits and masks come from ``numpy.random.default_rng(seed)``; tensors from a
``torch.Generator`` seeded with ``seed`` (x, then W1 expert by expert, then W2,
then probs).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

MXFP8, NVFP4 = 0, 1
SWIGLU, SRELU, TANH_SRELU = 0, 1, 2


@dataclass(frozen=True)
class Workload:
    name: str
    fmt: int
    act: int
    G: int
    K: int
    N: int
    M: int
    seed: int
    quant_only: bool = False
    tanh_clamp_scale: float = 0.0   # tanh-SReLU soft-clamp scale

    @property
    def n1(self) -> int:
        return 2 * self.N if self.act == SWIGLU else self.N

    @property
    def flops(self) -> float:
        """Dense GEMM flops of one forward: 2*M*K*N1 + 2*M*N*K."""
        return 2.0 * self.M * self.K * self.n1 + 2.0 * self.M * self.N * self.K


WORKLOADS = {
    "tiny": Workload("tiny", MXFP8, SWIGLU, 4, 256, 256, 512, 0),
    "mx_swiglu": Workload("mx_swiglu", MXFP8, SWIGLU, 8, 2048, 1024, 16384, 1),
    "nv_srelu": Workload("nv_srelu", NVFP4, SRELU, 8, 4096, 2048, 32768, 2),
    "mx_skew": Workload("mx_skew", MXFP8, SWIGLU, 64, 7168, 2048, 65536, 3),
    "nv_tanh_srelu": Workload("nv_tanh_srelu", NVFP4, TANH_SRELU, 8, 4096, 2048, 32768, 2, tanh_clamp_scale=8.0),
    "nv_quant": Workload("nv_quant", NVFP4, SRELU, 8, 4096, 0, 131072, 4, quant_only=True),
}


def make_splits(w: Workload) -> np.ndarray:
    rng = np.random.default_rng(w.seed)
    if w.name == "tiny":
        s = np.array([200, 150, 100, 62])
    elif w.name == "mx_swiglu":
        p = rng.dirichlet(np.ones(w.G))
        p[w.G - 1] = 0.0
        s = rng.multinomial(w.M, p / p.sum())
    elif w.name in ("nv_srelu", "nv_tanh_srelu"):
        s = np.full(w.G, w.M // w.G)
    elif w.name == "mx_skew":
        p = np.arange(1, w.G + 1, dtype=np.float64) ** -1.1
        s = rng.multinomial(w.M, p / p.sum())
        s[56:] = rng.integers(0, 9, 8)
        s[63] = 0
        s[0] += w.M - s.sum()
    elif w.name == "nv_quant":
        s = rng.multinomial(w.M, rng.dirichlet(np.full(w.G, 0.5)))
    else:
        raise KeyError(w.name)
    s = np.asarray(s, dtype=np.int64)
    assert s.sum() == w.M and (s >= 0).all()
    return s


def make_mask(w: Workload) -> int:
    rng = np.random.default_rng(w.seed + 1000)
    return int(rng.integers(0, 1 << 16))


def _normal(gen, shape, std=1.0):
    return torch.randn(shape, generator=gen, dtype=torch.float32).mul_(std).to(torch.bfloat16)


def make_x(w: Workload, gen: torch.Generator) -> torch.Tensor:
    x = torch.randn((w.M, w.K), generator=gen, dtype=torch.float32)
    if w.name in ("nv_srelu", "nv_tanh_srelu"):
        n_out = int(round(0.001 * w.M * w.K))
        idx = torch.randperm(w.M * w.K, generator=gen)[:n_out]
        x.view(-1)[idx] *= 50.0
    return x.to(torch.bfloat16)


def make_inputs(name: str, *, weights: bool = True) -> dict:
    """CPU tensors of one workload (bf16 / fp32 / int64)."""
    w = WORKLOADS[name]
    gen = torch.Generator().manual_seed(w.seed)
    out = dict(workload=w, splits=torch.from_numpy(make_splits(w)), mask=make_mask(w))
    out["x"] = make_x(w, gen)
    if w.quant_only:
        return out
    std = 1.0 / np.sqrt(w.K)
    if weights:
        W1 = torch.empty((w.G, w.n1, w.K), dtype=torch.bfloat16)
        for g in range(w.G):
            W1[g] = _normal(gen, (w.n1, w.K), std)
        W2 = torch.empty((w.G, w.K, w.N), dtype=torch.bfloat16)
        for g in range(w.G):
            W2[g] = _normal(gen, (w.K, w.N), std)
        out["W1"], out["W2"] = W1, W2
    out["probs"] = torch.rand((w.M,), generator=gen, dtype=torch.float32)
    return out


def random_splits(M: int, G: int, seed: int, zero_groups: int = 0) -> np.ndarray:
    """Ragged splits for edge-case tests: Dirichlet(1) multinomial with some groups emptied."""
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.ones(G))
    if zero_groups:
        p[rng.choice(G, zero_groups, replace=False)] = 0.0
    return rng.multinomial(M, p / p.sum()).astype(np.int64)


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a CPU bf16 tensor (for the oracle)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
