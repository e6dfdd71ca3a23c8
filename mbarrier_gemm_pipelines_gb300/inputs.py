"""Seeded synthetic inputs for the five workloads (random draws only).

This module holds no arithmetic of the operators: it only draws the inputs.
The tests, the smoke check and the benchmark pass the same host tensors to the
CUDA path and to the CPU oracle, so the choice of generator never affects a
parity result.  Generator: ``torch.Generator('cpu').manual_seed(seed)``; draw
order A, B, bias (grouped: counts, X, W, b); "N(0, s)" means standard
deviation s; bf16 tensors are the fp32 draw rounded to nearest even.

Workloads
  gemm_small      fp32 M=N=K=256, U[-1, 1] (seed 0)
  copy            fp32 [16384, 4096] = 256 MiB, U[-1e3, 1e3] (seed 1)
  gemm_fp32       fp32 M=N=K=4096, A, B ~ N(0, 1)/sqrt(K), bias ~ N(0, 0.1) (seed 2)
  gemm_bf16       bf16 M=N=K=8192, A, B ~ N(0, 1)/sqrt(K), bias fp32 ~ N(0, 0.1) (seed 3)
  grouped_bf16    4096 tokens over 8 experts, counts ~ Multinomial(4096, uniform),
                  X[4096, 4096], W[8, 4096, 14336] ~ N(0, 1)/sqrt(4096),
                  b[8, 14336] ~ N(0, 0.1) (seed 4)
"""
from __future__ import annotations

import math

import torch


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def uniform(shape, lo, hi, g):
    return torch.rand(shape, generator=g, dtype=torch.float32) * (hi - lo) + lo


def normal(shape, std, g):
    return torch.randn(shape, generator=g, dtype=torch.float32) * std


def gemm_uniform(M, N, K, seed=0, lo=-1.0, hi=1.0):
    g = _gen(seed)
    return uniform((M, K), lo, hi, g), uniform((K, N), lo, hi, g), uniform((N,), lo, hi, g)


def gemm_normal(M, N, K, seed, bias_std=0.1, dtype=torch.float32):
    """A, B ~ N(0, 1)/sqrt(K) (as `dtype`), bias fp32 ~ N(0, bias_std)."""
    g = _gen(seed)
    s = 1.0 / math.sqrt(K) if K > 0 else 1.0
    A = normal((M, K), s, g)
    B = normal((K, N), s, g)
    bias = normal((N,), bias_std, g)
    return A.to(dtype), B.to(dtype), bias


def copy_tensor(rows=16384, cols=4096, seed=1, lo=-1e3, hi=1e3):
    return uniform((rows, cols), lo, hi, _gen(seed))


def grouped(tokens=4096, experts=8, K=4096, N=14336, seed=4, bias_std=0.1,
            dtype=torch.bfloat16):
    """Counts ~ Multinomial(tokens, uniform over experts); X, W ~ N(0,1)/sqrt(K)."""
    g = _gen(seed)
    pick = torch.multinomial(torch.ones(experts), tokens, replacement=True, generator=g)
    counts = torch.bincount(pick, minlength=experts).tolist()
    s = 1.0 / math.sqrt(K)
    X = normal((tokens, K), s, g).to(dtype)
    W = normal((experts, K, N), s, g).to(dtype)
    b = normal((experts, N), bias_std, g)
    return counts, X, W, b


# The workloads by name (sizes as listed in the module docstring).
def workload(name: str):
    if name == "gemm_small":
        return gemm_uniform(256, 256, 256, seed=0)
    if name == "copy":
        return copy_tensor()
    if name == "gemm_fp32":
        return gemm_normal(4096, 4096, 4096, seed=2)
    if name == "gemm_bf16":
        return gemm_normal(8192, 8192, 8192, seed=3, dtype=torch.bfloat16)
    if name == "grouped_bf16":
        return grouped()
    raise KeyError(name)
