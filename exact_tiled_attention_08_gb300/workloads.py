"""Seeded synthetic inputs for exact attention.

This module only draws random numbers and casts them: it holds none of the
attention arithmetic, and is the one module that the CUDA-path tests and the
CPU oracle tests share.  It imports torch (for the seeded CPU generator and
bf16) and nothing from the product's CUDA binding.

Every tensor is drawn as fp32 ``randn`` from ``torch.Generator('cpu')`` in the
order Q, K, V, dO, then cast to bf16 (round to nearest even), laid out
``[B, H, N, d]`` contiguous.  The rescale-stress workload multiplies
ceil(1% of N) key rows, drawn from the last quarter of the sequence, by 8
(exact in bf16), the same rows for every (batch, head): the scores those keys
produce are about 8x larger and arrive late in every row, so the running
maximum jumps after several blocks have already been accumulated.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    key_outliers: bool
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def fwd_flops(self) -> float:
        """4 N^2 d per (batch, head), halved when causal."""
        f = 4.0 * self.N * self.N * self.d * self.B * self.H
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        """Five N x N x d matmuls: 2.5x the forward count."""
        return 2.5 * self.fwd_flops()


# The five workloads the pages' method is measured on.  Head dim 128 (and 64
# for the rescale stress), 128 to 32k tokens, bf16.
WORKLOADS = {
    "tiny_b1_h1_n128_d128": Workload("tiny_b1_h1_n128_d128", 1, 1, 128, 128, False, False, 1001),
    "b4_h16_n2048_d128": Workload("b4_h16_n2048_d128", 4, 16, 2048, 128, False, False, 1002),
    "causal_b2_h32_n8192_d128": Workload("causal_b2_h32_n8192_d128", 2, 32, 8192, 128, True, False, 1003),
    "causal_long_b1_h8_n32768_d128": Workload("causal_long_b1_h8_n32768_d128", 1, 8, 32768, 128, True, False, 1004),
    "rescale_stress_b16_h16_n1024_d64": Workload("rescale_stress_b16_h16_n1024_d64", 16, 16, 1024, 64, False, True, 1005),
}


def outlier_key_rows(n: int, gen: torch.Generator) -> torch.Tensor:
    """ceil(1% of n) distinct key indices drawn from [3n/4, n)."""
    count = max(1, math.ceil(0.01 * n))
    lo = (3 * n) // 4
    count = min(count, n - lo)
    return torch.randperm(n - lo, generator=gen)[:count] + lo


def make_inputs(B: int, H: int, N: int, d: int, seed: int, key_outliers: bool = False,
                with_dout: bool = True) -> dict:
    """bf16 CPU tensors ``q, k, v`` (and ``do``) of shape [B, H, N, d]."""
    gen = torch.Generator("cpu").manual_seed(seed)
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=gen, dtype=torch.float32)
    k = torch.randn(shape, generator=gen, dtype=torch.float32)
    v = torch.randn(shape, generator=gen, dtype=torch.float32)
    do = torch.randn(shape, generator=gen, dtype=torch.float32) if with_dout else None
    if key_outliers:
        rows = outlier_key_rows(N, gen)
        k[:, :, rows, :] *= 8.0
    out = {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16)}
    if with_dout:
        out["do"] = do.to(torch.bfloat16)
    return out


def workload_inputs(w: Workload, with_dout: bool = True) -> dict:
    return make_inputs(w.B, w.H, w.N, w.d, w.seed, w.key_outliers, with_dout)


def to_f32_numpy(t: torch.Tensor):
    """Exact widening of a (bf16) tensor to a float32 numpy array on the host."""
    return t.detach().to("cpu", torch.float32).numpy()


def rotation_signs(d: int, seed: int) -> torch.Tensor:
    """d random signs (+1 / -1, int8) for the FP8 forward's Hadamard rotation."""
    gen = torch.Generator("cpu").manual_seed(seed)
    return (torch.randint(0, 2, (d,), generator=gen, dtype=torch.int8) * 2 - 1).to(torch.int8)


def make_outlier_inputs(B: int, H: int, N: int, d: int, seed: int, frac: float = 1e-3,
                        outlier_std: float = 10.0) -> dict:
    """bf16 ``q, k, v`` whose entries are N(0, 1) plus, with probability
    ``frac``, an extra N(0, outlier_std^2): a few large entries scattered over
    the tensors, the case per-tensor FP8 scaling handles badly."""
    gen = torch.Generator("cpu").manual_seed(seed)
    shape = (B, H, N, d)
    out = {}
    for name in ("q", "k", "v"):
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
        hit = torch.rand(shape, generator=gen) < frac
        x = x + hit * outlier_std * torch.randn(shape, generator=gen, dtype=torch.float32)
        out[name] = x.to(torch.bfloat16)
    return out
