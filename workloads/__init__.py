"""Seeded synthetic inputs shaped like the pages' workloads.

Used by both the GPU path's tests/benchmark and the oracle's tests; it holds
none of the method's arithmetic (no reduction, no codec), only random draws
and dtype casts.  Every generator draws rank by rank from one
``torch.Generator`` seeded once, so the values depend only on the seed, the
shape and the device the generator runs on.

Workloads (sizes as the configurations name them):
  lossless_n4   N=4, T=4096 fp32, N(0,1), seed 0
  bfp8_bucket   N=8, T=13,107,200 (25 MiB of fp16), N(0, 1e-3^2) -> fp16, seed 1
  sparse_n16    N=16, T=64 Mi bf16; zero with probability 0.6 (Bernoulli mask
                per rank), else N(0, 0.02^2) -> bf16; zeros are +0.0; seed 2
  diloco_n8     N=8, T=10^9 fp32: prev = N(0, 1e-4^2), then a fresh
                perturbation N(0, 1e-5^2) from the same generator,
                cur = prev + perturbation (fp32); seed 3
  sweep         T fp32 elements in {256 * 4^k}, U(-1, 1), seed 4 + case index
"""
from __future__ import annotations

import torch

CONFIGS = {
    "lossless_n4": dict(N=4, T=4096, dtype="f32", seed=0),
    "bfp8_bucket": dict(N=8, T=13_107_200, dtype="f16", seed=1),
    "sparse_n16": dict(N=16, T=64 * 2 ** 20, dtype="bf16", seed=2),
    "diloco_n8": dict(N=8, T=10 ** 9, dtype="f32", seed=3),
    # the bucket's tensors as parameters gathered compressed (allgather alone)
    "bfp8_allgather": dict(N=8, T=13_107_200, dtype="f16", seed=1),
    # the same tensors broadcast compressed from rank 0 (binomial tree)
    "bfp8_broadcast": dict(N=8, T=13_107_200, dtype="f16", seed=1),
}
SWEEP_N = (2, 4, 8, 16, 64)
SWEEP_T = tuple(256 * 4 ** k for k in range(11))  # 1 KiB .. 1 GiB of fp32


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def lossless(N: int, T: int, seed: int = 0, device="cuda"):
    g = _gen(seed, device)
    return [torch.randn(T, generator=g, device=device, dtype=torch.float32) for _ in range(N)]


def bfp_bucket(N: int, T: int, seed: int = 1, device="cuda", std: float = 1e-3):
    g = _gen(seed, device)
    out = []
    for _ in range(N):
        x = torch.randn(T, generator=g, device=device, dtype=torch.float32)
        out.append((x * std).to(torch.float16))
    return out


def sparse(N: int, T: int, seed: int = 2, device="cuda", p_zero: float = 0.6, std: float = 0.02,
           dtype=torch.bfloat16):
    g = _gen(seed, device)
    out = []
    for _ in range(N):
        keep = torch.rand(T, generator=g, device=device) >= p_zero
        v = torch.randn(T, generator=g, device=device, dtype=torch.float32) * std
        v = v.to(dtype)
        out.append(torch.where(keep, v, torch.zeros((), dtype=dtype, device=device)))
    return out


def diloco(N: int, T: int, seed: int = 3, device="cuda", std_prev: float = 1e-4,
           std_pert: float = 1e-5):
    """Returns (cur, prev): lists of N fp32 tensors."""
    g = _gen(seed, device)
    prev, cur = [], []
    for _ in range(N):
        p = torch.randn(T, generator=g, device=device, dtype=torch.float32) * std_prev
        prev.append(p)
    for r in range(N):
        pert = torch.randn(T, generator=g, device=device, dtype=torch.float32) * std_pert
        cur.append(prev[r] + pert)
    return cur, prev


def uniform(N: int, T: int, seed: int = 4, device="cuda"):
    g = _gen(seed, device)
    return [torch.rand(T, generator=g, device=device, dtype=torch.float32) * 2 - 1
            for _ in range(N)]
