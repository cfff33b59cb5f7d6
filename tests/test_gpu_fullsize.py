"""GPU parity at the configurations' full sizes, in the launch configuration
bench.py times (the library chooses it from N, T and the dtypes alone).

The oracle cannot redo 10^9-element rings in a test, so it computes sampled
positions: slices of 256 elements are independent in the BFP and lossless
rings (BFP blocks never cross a slice boundary, and every element's chain
depends only on its chunk index), so the ring over the chosen slices of every
chunk is an exact sub-problem.  The per-chunk sparse ring is not sliceable
(each chunk's format depends on all of it): it runs the whole oracle.  Properties that hold at any size are checked
on the whole output: every rank bit-identical, the sparse ring equal to the
lossless ring, closed-form byte counters."""
import numpy as np
import pytest
import torch

import oracle as O
import ring_allreduce_compressed_gb300 as rra
import workloads as W
from gpu_util import assert_bits_equal, gather_subproblem, host, sample_offsets

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rra.build()
    rra.lib()


def check_sampled(xs, outs, N, T, seed, in_dt, out_dt, count=24, **kw):
    n = T // N
    slices = sample_offsets(n, count, seed)
    sub_in, idx = gather_subproblem(xs, N, T, slices)
    extra = {}
    if "diff_prev" in kw:
        extra["diff_prev"] = gather_subproblem(kw.pop("diff_prev"), N, T, slices)[0]
        base_sub = gather_subproblem([kw.pop("diff_base")], N, T, slices)[0][0]
        extra["diff_base"] = base_sub
    ref, _, _ = O.ring(sub_in, in_dt, out_dt, **kw, **extra)
    it = torch.from_numpy(idx).cuda()
    for r in range(N):
        got = host(outs[r].index_select(0, it))
        assert_bits_equal(got, ref[r], f"rank {r}")


def all_ranks_identical(outs):
    for r in range(1, len(outs)):
        assert torch.equal(outs[r].view(torch.uint8), outs[0].view(torch.uint8)), r


def test_bfp8_bucket_full_size():
    """N=8, 25 MiB fp16 bucket, block-FP8, fp16 out."""
    c = W.CONFIGS["bfp8_bucket"]
    N, T = c["N"], c["T"]
    xs = W.bfp_bucket(N, T, seed=c["seed"])
    outs = [torch.empty(T, dtype=torch.float16, device="cuda") for _ in range(N)]
    comm = rra.Comm(N, T, torch.float16)
    comm.ring_allreduce(xs, outs, rra.Codec("bfp", bits=8))
    sent, recv = comm.get_bytes()
    assert comm.status() == rra.RRA_OK
    n = T // N
    per_msg = n // 128 + n
    assert sent == [2 * (N - 1) * per_msg] * N == recv  # 23,116,800 B per rank
    assert sent[0] == 23_116_800
    all_ranks_identical(outs)
    check_sampled(xs, outs, N, T, 1, "f16", "f16", codec="bfp", bits=8)
    comm.close()


def test_sparse_n16_full_size():
    """N=16, 64 Mi bf16 with 60% zeros, threshold 0.5, fp32 out, one sparse
    message per chunk and hop: the whole output and the byte counters
    against the whole oracle (a per-chunk format depends on every slice of
    the chunk, so no slice sample is an exact sub-problem), and equal to the
    lossless ring."""
    c = W.CONFIGS["sparse_n16"]
    N, T = c["N"], c["T"]
    xs = W.sparse(N, T, seed=c["seed"])
    comm = rra.Comm(N, T, torch.bfloat16)
    outs = [torch.empty(T, dtype=torch.float32, device="cuda") for _ in range(N)]
    comm.ring_allreduce(xs, outs, rra.Codec("sparse", sparsity_threshold=0.5))
    sparse_sent, sparse_recv = comm.get_bytes()
    assert comm.status() == rra.RRA_OK
    ref, rsent, rrecv = O.ring([host(x) for x in xs], "bf16", "f32", codec="sparse", threshold=0.5)
    assert sparse_sent == [int(v) for v in rsent] and sparse_recv == [int(v) for v in rrecv]
    for r in range(N):
        assert_bits_equal(host(outs[r]), ref[r], f"rank {r}")
    del ref
    lossless = [torch.empty(T, dtype=torch.float32, device="cuda") for _ in range(N)]
    comm.ring_allreduce(xs, lossless)
    lossless_sent, _ = comm.get_bytes()
    for r in range(N):
        assert torch.equal(outs[r].view(torch.int32), lossless[r].view(torch.int32)), r
    # hop 1 (density 0.4) goes sparse, every later hop dense: 8 + 8 nnz bytes
    # once, 8 + 4 n bytes for the other 29 messages a rank sends
    n = T // N
    assert 29 * (8 + 4 * n) < sparse_sent[0] < 30 * (8 + 4 * n)
    assert lossless_sent[0] == 30 * n * 4
    comm.close()


def test_sparse_n16_full_size_per_slice():
    """The per-slice option at full size: sampled slices are exact
    sub-problems there (every slice decides on its own)."""
    c = W.CONFIGS["sparse_n16"]
    N, T = c["N"], c["T"]
    xs = W.sparse(N, T, seed=c["seed"])
    comm = rra.Comm(N, T, torch.bfloat16)
    outs = [torch.empty(T, dtype=torch.float32, device="cuda") for _ in range(N)]
    comm.ring_allreduce(xs, outs, rra.Codec("sparse", sparsity_threshold=0.5, granularity="slice"))
    assert comm.status() == rra.RRA_OK
    check_sampled(xs, outs, N, T, 2, "bf16", "f32", codec="sparse", threshold=0.5,
                  slice=rra.RING_SLICE)
    all_ranks_identical(outs)
    comm.close()


def test_diloco_n8_full_size():
    """N=8, 10^9 fp32 per rank: diff against prev, block-FP4, average 1/N,
    previous result added back (the 64-element tail block of every chunk is
    always among the sampled slices)."""
    c = W.CONFIGS["diloco_n8"]
    N, T = c["N"], c["T"]
    torch.cuda.empty_cache()  # blocks cached by earlier tests count as free
    free, _ = torch.cuda.mem_get_info()
    if free < 110 * 2 ** 30:
        pytest.skip("needs ~110 GB of device memory")
    cur, prev = W.diloco(N, T, seed=c["seed"])
    base = torch.empty(T, device="cuda")
    comm = rra.Comm(N, T)
    # previous round's result: lossless mean of prev; reduce-scatter writes
    # chunk r of every output, so one shared output buffer collects the mean
    comm.reduce_scatter(prev, [base] * N, rra.Codec("none", average=True))
    assert comm.status() == rra.RRA_OK
    outs = [torch.empty(T, device="cuda") for _ in range(N)]
    codec = rra.Codec("bfp", bits=4, diff_prev=prev, diff_base=base, average=True)
    comm.ring_allreduce(cur, outs, codec)
    sent, _ = comm.get_bytes()
    assert comm.status() == rra.RRA_OK
    n = T // N
    assert sent[0] == 2 * (N - 1) * (-(-n // 128) + -(-n // 2))
    check_sampled(cur, outs, N, T, 3, "f32", "f32", count=12, codec="bfp", bits=4,
                  diff_prev=prev, diff_base=base, average=True)
    # the base itself: sampled against the oracle's lossless mean
    n_sl = sample_offsets(n, 8, 5)
    sub_prev, idx = gather_subproblem(prev, N, T, n_sl)
    ref = O.ring(sub_prev, average=True)[0][0]
    assert_bits_equal(host(base.index_select(0, torch.from_numpy(idx).cuda())), ref, "base")
    comm.close()


@pytest.mark.parametrize("N,T", [(2, 256 * 4 ** 10), (64, 256 * 4 ** 10), (64, 256), (16, 256 * 4 ** 7)])
def test_sweep_extremes_ring_and_tree(N, T):
    """Message-size sweep corners: 1 KiB and 1 GiB per rank, N up to 64,
    lossless fp32, ring and tree, in place."""
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    if free < N * T * 4 * 1.3 + 2 ** 30:
        pytest.skip("not enough device memory")
    bufs = W.uniform(N, T, seed=4)
    if T * N <= 2 ** 22:
        ref = O.ring([host(b) for b in bufs])[0]
        tref = O.tree_allreduce([host(b) for b in bufs])[0]
    comm = rra.Comm(N, T)
    snapshot = None
    if T * N <= 2 ** 22:
        snapshot = [b.clone() for b in bufs]
    n = -(-T // N)
    slices = sample_offsets(n, 6, 6)
    sub = gather_subproblem(bufs, N, T, slices)[0] if T % N == 0 else None
    sub_ref = O.ring(sub)[0] if sub is not None else None
    idx = gather_subproblem(bufs, N, T, slices)[1] if T % N == 0 else None
    comm.ring_allreduce(bufs, bufs)
    assert comm.status() == rra.RRA_OK
    sent, _ = comm.get_bytes()
    assert sent[0] == 2 * (N - 1) * n * 4
    if snapshot is not None:
        for r in range(N):
            assert_bits_equal(host(bufs[r]), ref[r], f"ring rank {r}")
    elif sub_ref is not None:
        it = torch.from_numpy(idx).cuda()
        for r in (0, N // 2, N - 1):
            assert_bits_equal(host(bufs[r].index_select(0, it)), sub_ref[r], f"ring rank {r}")
    all_ranks_identical(bufs)
    if snapshot is not None:
        comm.tree_allreduce(snapshot)
        assert comm.status() == rra.RRA_OK
        for r in range(N):
            assert_bits_equal(host(snapshot[r]), tref[r], f"tree rank {r}")
    comm.close()
