"""Seeded synthetic inputs for the virtual-rank collectives.

This module only draws random numbers; it holds none of the collectives'
arithmetic.  The tests, the smoke check and the benchmark all take their
inputs from here, so the CUDA library and the CPU oracle always see the same
bytes.

Recipes (one per workload; every rank u of workload c is seeded with
``SEED + 1000 * c + u``):

* ``uniform``    -- fp32 uniform on [-1, 1] (reduce-scatter / message sweeps);
* ``gradient``   -- fp32 normal(0, 1e-3), gradient-like;
* ``outliers``   -- bf16 from fp32 normal(0, 1e-2), with a Bernoulli(0.01) mask
                    of elements multiplied by 100;
* ``fusion_counts`` -- element counts round(exp(U[ln 1024, ln 4194304])) for the
                    tensor-fusion workload, from a seeded host generator (the
                    same list on every rank).

Generation runs on whatever device is given: on the GPU for full-size
workloads (then copied to the host for the oracle), on the CPU for small
oracle-only cases.  Parity depends only on the bytes, never on where they were
drawn.
"""
from __future__ import annotations

import math

import numpy as np
import torch

SEED = 20261202

# workload ids used in the seed formula
RS_W4 = 1          # reduce-scatter / allreduce sum, W=4, fp32, n=2^20, uniform
AR_W8_F32 = 2      # allreduce sum, W=8, fp32, n=2^26, gradient-like
AR_W8_BF16 = 3     # allreduce avg, W=8, bf16, n=2^28, normal + outliers
FUSION_W8 = 4      # tensor fusion, W=8, 200 fp32 tensors per rank
SWEEP = 5          # message-size sweep, fp32 uniform


def rank_seed(workload: int, rank: int) -> int:
    return SEED + 1000 * workload + rank


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def uniform(n: int, seed: int, device="cpu") -> torch.Tensor:
    """fp32 uniform on [-1, 1]."""
    g = _gen(seed, device)
    return torch.rand(n, generator=g, device=device, dtype=torch.float32).mul_(2.0).sub_(1.0)


def gradient(n: int, seed: int, device="cpu", std: float = 1e-3) -> torch.Tensor:
    """fp32 normal(0, std)."""
    g = _gen(seed, device)
    return torch.randn(n, generator=g, device=device, dtype=torch.float32).mul_(std)


def outliers(n: int, seed: int, device="cpu", std: float = 1e-2, p: float = 0.01,
             factor: float = 100.0) -> torch.Tensor:
    """bf16 normal(0, std) with a Bernoulli(p) mask of elements times ``factor``."""
    g = _gen(seed, device)
    x = torch.randn(n, generator=g, device=device, dtype=torch.float32).mul_(std)
    mask = torch.rand(n, generator=g, device=device, dtype=torch.float32) < p
    x[mask] *= factor
    return x.to(torch.bfloat16)


def fusion_counts(T: int = 200, seed: int = SEED + 1000 * FUSION_W8,
                  lo: int = 1024, hi: int = 4194304) -> np.ndarray:
    """Log-uniform element counts in [lo, hi] (int64)."""
    rng = np.random.default_rng(seed)
    return np.round(np.exp(rng.uniform(math.log(lo), math.log(hi), T))).astype(np.int64)


def rank_buffers(kind: str, W: int, n: int, workload: int, device="cpu") -> list[torch.Tensor]:
    """W rank buffers of n elements drawn with the named recipe."""
    make = {"uniform": uniform, "gradient": gradient, "outliers": outliers}[kind]
    return [make(n, rank_seed(workload, u), device) for u in range(W)]


def fusion_tensors(counts, W: int, device="cpu", workload: int = FUSION_W8):
    """tensors[u][t]: fp32 normal(0, 1e-3) tensor t of rank u."""
    out = []
    for u in range(W):
        g = _gen(rank_seed(workload, u), device)
        out.append([torch.randn(int(c), generator=g, device=device, dtype=torch.float32).mul_(1e-3)
                    for c in counts])
    return out
