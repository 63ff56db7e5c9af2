"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no arithmetic of the GEMM/GEMV themselves: it only draws
numbers.  Everything is drawn on the CPU with a ``torch.Generator`` seeded by
the caller, so the GPU path and the oracle see the same fp16 bytes.

Recipes (the pages give shapes and distributions, not generators):
  * GEMM operands: i.i.d. uniform[-1, 1) in fp32, rounded to fp16 (RNE);
    A (M x K) is drawn first, then B (N x K).
  * GEMV operands: i.i.d. normal(0, 0.02) in fp32, rounded to fp16; x (K) first,
    then W (N x K) — the nn.Linear weight layout of "Learning TileLang with
    GEMV", §01 GEMV (N = 4096, K = 14336: a Llama-3-8B MLP down projection).
  * Integer-valued operands: i.i.d. uniform on {lo..hi}, exactly representable.
"""
from __future__ import annotations

import torch

# The five workloads, named by what they are.
WORKLOADS = {
    "gemm_256": dict(kind="gemm", M=256, N=256, K=256),
    "gemm_4096": dict(kind="gemm", M=4096, N=4096, K=4096),
    "gemv_4096x14336": dict(kind="gemv", N=4096, K=14336),
    "gemm_ragged_4000x3000x4160": dict(kind="gemm", M=4000, N=3000, K=4160),
    "gemm_8192": dict(kind="gemm", M=8192, N=8192, K=8192),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def uniform_f16(shape, g: torch.Generator) -> torch.Tensor:
    return (torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0).half()


def normal_f16(shape, g: torch.Generator, std: float = 0.02) -> torch.Tensor:
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std).half()


def gemm_inputs(M: int, N: int, K: int, seed: int = 0):
    """(A, B): CPU fp16 tensors, A (M, K) then B (N, K), uniform[-1, 1)."""
    g = _gen(seed)
    A = uniform_f16((M, K), g)
    B = uniform_f16((N, K), g)
    return A, B


def gemv_inputs(N: int, K: int, seed: int = 0):
    """(x, W): CPU fp16 tensors, x (K,) then W (N, K), normal(0, 0.02)."""
    g = _gen(seed)
    x = normal_f16((K,), g)
    W = normal_f16((N, K), g)
    return x, W


def integer_f16(shape, seed: int, lo: int = -2, hi: int = 2) -> torch.Tensor:
    """Integer-valued fp16 tensor with entries in {lo..hi}."""
    g = _gen(seed)
    return torch.randint(lo, hi + 1, shape, generator=g, dtype=torch.int32).to(torch.float16)


def l2_rotation_count(bytes_per_set: int, l2_bytes: int, factor: float = 4.0) -> int:
    """How many distinct input sets to rotate so that each launch misses L2:
    enough that a set is read again only after `factor` x L2 bytes of other
    sets (at 2 x L2, ncu still counted 10-30 % of a 117 MB weight set as L2
    hits on the next pass)."""
    if bytes_per_set <= 0:
        return 1
    n = 1
    while n * bytes_per_set < factor * l2_bytes:
        n += 1
    return max(n, 2)
