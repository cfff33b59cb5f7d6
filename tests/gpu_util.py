"""Helpers shared by the GPU parity tests: host copies of device tensors for
the oracle, bitwise comparison, and oracle runs on sampled sub-problems."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O

TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
DT_NAME = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}


def host(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> numpy array in the oracle's representation."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def bitsof(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    return a.view({4: np.uint32, 2: np.uint16, 1: np.uint8}[a.dtype.itemsize])


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str = ""):
    g, w = bitsof(got), bitsof(want)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    bad = np.nonzero(g != w)[0]
    if bad.size:
        i = bad[0]
        raise AssertionError(f"{what}: {bad.size} of {g.size} elements differ; first at {i}: "
                             f"got {got[i]!r} (0x{int(g[i]):x}) want {want[i]!r} (0x{int(w[i]):x})")


def rand_f32(N, T, seed, scale=1.0, device="cuda"):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return [torch.randn(T, generator=g, device=device) * scale for _ in range(N)]


def cast(ts, name):
    return [t.to(TORCH_DT[name]) for t in ts]


def sample_offsets(n: int, count: int, seed: int, align: int = 256):
    """Sorted, distinct slice-aligned offsets inside a chunk of length n; the
    last (possibly partial) slice is always included."""
    nsl = -(-n // align)
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(nsl, size=min(count, nsl), replace=False).tolist())
    pick.add(nsl - 1)
    pick.add(0)
    return sorted(pick)


def gather_subproblem(ts, N, T, slices, align=256):
    """Host arrays of a mini ring problem made of the chosen slice positions
    of every chunk.  Slices are independent in the ring (the BFP blocks and
    sparse messages never cross a slice), so the mini problem's chunk c holds
    exactly the values the full problem has at those positions of chunk c.
    Requires every chunk to have the same length n (N divides T) and the
    ragged slice, if any, to be the last one picked."""
    n = T // N
    assert n * N == T
    idx = []
    for c in range(N):
        for s in slices:
            lo = c * n + s * align
            hi = min(c * n + (s + 1) * align, (c + 1) * n)
            idx.append(np.arange(lo, hi))
    idx = np.concatenate(idx)
    it = torch.from_numpy(idx).to(ts[0].device)
    return [host(t.index_select(0, it)) for t in ts], idx
