"""GPU parity: every op and codec of the CUDA path, called through the C ABI
(Python binding), against the CPU oracle on the same seeded inputs.

The bar is bit-exactness everywhere: lossless sums follow the ring's fixed
order, the codecs round to nearest even exactly as the oracle does, byte
counters are exact.  Sizes span several 256-element slices, ragged tails,
chunk counts that do not divide T, the N=1 and N=2 special cases, both the
bulk-copy fast path (16-byte aligned buffers and chunk sizes) and the generic
path, and N up to the 64-rank maximum."""
import numpy as np
import pytest
import torch

import oracle as O
import ring_allreduce_compressed_gb300 as rra
import workloads as W
from gpu_util import (TORCH_DT, assert_bits_equal, cast, host, rand_f32)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rra.build()
    rra.lib()
    torch.cuda.init()


def run_ring(xs, out_dt, codec=None, mode="allreduce", outs=None):
    N = len(xs)
    comm = rra.Comm(N, xs[0].numel(), xs[0].dtype)
    if outs is None:
        outs = [torch.zeros(xs[0].numel(), dtype=TORCH_DT[out_dt], device="cuda") for _ in range(N)]
    if mode == "allreduce":
        comm.ring_allreduce(xs, outs, codec)
    else:
        comm.reduce_scatter(xs, outs, codec)
    sent, recv = comm.get_bytes()
    assert comm.status() == rra.RRA_OK
    comm.close()
    return outs, np.array(sent, np.uint64), np.array(recv, np.uint64)


def oracle_ring(xs, in_dt, out_dt, mode="allreduce", **kw):
    outs = None
    if mode == "reduce_scatter":
        outs = [np.zeros(xs[0].numel(), O.NP_DTYPES[out_dt]) for _ in xs]
    return O.ring([host(x) for x in xs], in_dt, out_dt, mode=mode, outputs=outs, **kw)


def compare(gpu, ref, what):
    g_outs, g_sent, g_recv = gpu
    r_outs, r_sent, r_recv = ref
    for r, (g, w) in enumerate(zip(g_outs, r_outs)):
        assert_bits_equal(host(g), w, f"{what} rank {r}")
    assert list(g_sent) == list(r_sent), (what, g_sent, r_sent)
    assert list(g_recv) == list(r_recv), (what, g_recv, r_recv)


# ------------------------------------------------------------------ lossless

def test_config1_lossless_all_ops():
    """N=4, T=4096 fp32, N(0,1) seed 0: ring allreduce, reduce-scatter,
    allgather, broadcast from rank 0 and the tree, bit-exact, with the
    closed-form byte counter 2T(N-1)/N * 4 = 24,576 B per rank."""
    xs = W.lossless(4, 4096, seed=0)
    gpu = run_ring(xs, "f32")
    ref = oracle_ring(xs, "f32", "f32")
    compare(gpu, ref, "ring")
    assert list(gpu[1]) == [24576] * 4
    for r in range(1, 4):
        assert torch.equal(gpu[0][r], gpu[0][0])

    rs_out = [torch.full((4096,), 7.0, device="cuda") for _ in range(4)]
    gpu = run_ring(xs, "f32", mode="reduce_scatter", outs=rs_out)
    rs_ref_out = [np.full(4096, 7.0, np.float32) for _ in range(4)]
    ref = O.ring([host(x) for x in xs], mode="reduce_scatter", outputs=rs_ref_out)
    compare(gpu, ref, "reduce_scatter")

    comm = rra.Comm(4, 4096)
    bufs = [x.clone() for x in xs]
    comm.allgather(bufs)
    ref_bufs, s, r = O.allgather([host(x) for x in xs])
    for q in range(4):
        assert_bits_equal(host(bufs[q]), ref_bufs[q], f"allgather {q}")
    assert comm.get_bytes() == (list(s), list(r))

    bufs = [x.clone() for x in xs]
    comm.broadcast(bufs, root=0)
    ref_bufs, s, r = O.broadcast([host(x) for x in xs], "f32", 0)
    for q in range(4):
        assert_bits_equal(host(bufs[q]), ref_bufs[q], f"broadcast {q}")
    assert comm.get_bytes() == (list(s), list(r))

    bufs = [x.clone() for x in xs]
    comm.tree_allreduce(bufs)
    ref_bufs, s, r = O.tree_allreduce([host(x) for x in xs])
    for q in range(4):
        assert_bits_equal(host(bufs[q]), ref_bufs[q], f"tree {q}")
    assert comm.get_bytes() == (list(s), list(r))
    assert comm.status() == rra.RRA_OK
    comm.close()


@pytest.mark.parametrize("N", [1, 2, 3, 5, 8, 16, 17, 33, 64])
@pytest.mark.parametrize("T", [1, 100, 256, 1000, 4096, 70001])
def test_lossless_ring_shapes(N, T):
    xs = rand_f32(N, T, seed=N * 7919 + T)
    compare(run_ring(xs, "f32"), oracle_ring(xs, "f32", "f32"), f"N={N} T={T}")


@pytest.mark.parametrize("N,n,G", [(12, 152 * 512, 2), (16, 152 * 1024, 4), (32, 152 * 512, 2)])
def test_lossless_wide_default_shape(N, n, G):
    """Lossless rings of 12 or more ranks on the staged path take two slots
    per edge, one stage and the widest slice that leaves every SM a slice
    position and fits 16 resident warps per SM (one block of 16 warps, two
    of 12); bit-exact in ring order."""
    T = N * n
    xs = rand_f32(N, T, seed=N + G)
    comm = rra.Comm(N, T)
    outs = [torch.empty_like(x) for x in xs]
    comm.ring_allreduce(xs, outs)
    assert comm.status() == rra.RRA_OK
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert comm.last_shape()[1:] == (2, 1, G)
    sent, recv = comm.get_bytes()
    comm.close()
    compare((outs, np.array(sent, np.uint64), np.array(recv, np.uint64)),
            oracle_ring(xs, "f32", "f32"), f"N={N} wide default")


@pytest.mark.parametrize("in_dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("out_dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("T", [4096 * 3, 5003])
def test_lossless_dtypes(in_dt, out_dt, T):
    xs = cast(rand_f32(4, T, seed=11), in_dt)
    compare(run_ring(xs, out_dt), oracle_ring(xs, in_dt, out_dt), f"{in_dt}->{out_dt}")


def test_lossless_misaligned_buffers_take_generic_path():
    """Views starting 4 bytes into their storage are not 16-byte aligned: the
    generic (element-wise) path must give the same bits."""
    N, T = 4, 8192
    base = rand_f32(N, T + 1, seed=12)
    xs = [b[1:] for b in base]
    outs_store = [torch.zeros(T + 1, device="cuda") for _ in range(N)]
    outs = [o[1:] for o in outs_store]
    comm = rra.Comm(N, T)
    comm.ring_allreduce(xs, outs)
    ref = O.ring([host(x) for x in xs])
    for r in range(N):
        assert_bits_equal(host(outs[r]), ref[0][r], f"rank {r}")
    comm.close()


def test_in_place_allreduce():
    N, T = 8, 65536
    xs = rand_f32(N, T, seed=13)
    ref = O.ring([host(x) for x in xs])
    comm = rra.Comm(N, T)
    comm.ring_allreduce(xs, xs)
    for r in range(N):
        assert_bits_equal(host(xs[r]), ref[0][r], f"rank {r}")
    comm.close()


# ------------------------------------------------------------------ block floating point

@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("in_dt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("N,T", [(2, 512), (3, 1000), (8, 8 * 4096), (8, 40017), (5, 256 * 5 * 3 + 70)])
def test_bfp_ring(bits, in_dt, N, T):
    xs = cast(rand_f32(N, T, seed=bits * 100 + N + T, scale=1e-3), in_dt)
    out_dt = "f16" if in_dt == "f16" else "f32"
    codec = rra.Codec("bfp", bits=bits)
    gpu = run_ring(xs, out_dt, codec)
    ref = oracle_ring(xs, in_dt, out_dt, codec="bfp", bits=bits)
    compare(gpu, ref, f"bfp{bits} {in_dt}")


@pytest.mark.parametrize("bits", [8, 4])
def test_bfp_ring_degenerate_blocks(bits):
    """All-zero blocks, subnormal maxima, huge and tiny magnitudes in the same
    slice, values that round to the clamp: exponents from the bits, clamp at
    -126, codes clamped to +-(2^(bits-1)-1)."""
    N, T = 4, 4 * 1024
    g = torch.Generator(device="cuda")
    g.manual_seed(99)
    xs = []
    for r in range(N):
        x = torch.randn(T, generator=g, device="cuda")
        x[:128] = 0.0
        x[128:256] = torch.randn(128, generator=g, device="cuda") * 1e-39  # subnormal
        x[256:384] *= 1e30
        x[384:512] = 1.9921875 * (1 if r % 2 else -1)
        x[512:640] *= 1e-30
        xs.append(x)
    codec = rra.Codec("bfp", bits=bits)
    compare(run_ring(xs, "f32", codec), oracle_ring(xs, "f32", "f32", codec="bfp", bits=bits),
            "degenerate")


def test_bfp8_config2_shape_small():
    """The headline codec on a shrunken bucket: N=8, fp16 N(0,1e-3^2), fp16 out."""
    xs = W.bfp_bucket(8, 8 * 2048 * 8, seed=1)
    codec = rra.Codec("bfp", bits=8)
    gpu = run_ring(xs, "f16", codec)
    compare(gpu, oracle_ring(xs, "f16", "f16", codec="bfp", bits=8), "cfg2 small")
    n = xs[0].numel() // 8
    assert all(int(s) == 14 * (n // 128 + n) for s in gpu[1])


@pytest.mark.parametrize("in_dt", ["f32", "f16"])
@pytest.mark.parametrize("G", [0, 1, 2, 8])
def test_bfp8_f16_outputs_across_exponents(in_dt, G):
    """fp16 outputs of BFP8 codes for block exponents from far below the fp16
    subnormals to past the fp16 maximum.  Where 2^(e-q) and the offset term
    are fp16 numbers the allgather writes fp16 straight from the codes, else
    it rounds the fp32 decode; both must give the oracle's bits (the exact
    decoded value rounded once to fp16), on full slices and the ragged tail,
    for every slice width."""
    N, T = 8, 8 * 2048 * 6 + 8 * 40
    g = torch.Generator(device="cuda")
    g.manual_seed(70 + G)
    lo, hi = (-48, 21) if in_dt == "f32" else (-30, 13)
    nb = -(-T // 128)
    j = (torch.arange(nb, device="cuda") * 7) % (hi - lo + 1) + lo
    scale = torch.pow(2.0, j.float()).repeat_interleave(128)[:T]
    xs = cast([torch.randn(T, generator=g, device="cuda") * scale for _ in range(N)], in_dt)
    comm = rra.Comm(N, T, xs[0].dtype)
    if G:
        comm.set_tuning(0, 0, 0, G)
    outs = [torch.zeros(T, dtype=torch.float16, device="cuda") for _ in range(N)]
    codec = rra.Codec("bfp", bits=8)
    comm.ring_allreduce(xs, outs, codec)
    assert comm.status() == rra.RRA_OK
    if G:
        assert comm.last_shape()[3] == G
    sent, recv = comm.get_bytes()
    comm.close()
    ref = oracle_ring(xs, in_dt, "f16", codec="bfp", bits=8)
    compare((outs, np.array(sent, np.uint64), np.array(recv, np.uint64)), ref,
            f"bfp8 {in_dt}->f16 G={G}")


# ------------------------------------------------------------------ sparse

SLICE_OF = {"chunk": None, "slice": rra.RING_SLICE}


@pytest.mark.parametrize("gran", ["chunk", "slice"])
@pytest.mark.parametrize("thr", [0.5, 0.2, 0.9])
@pytest.mark.parametrize("in_dt", ["bf16", "f32", "f16"])
@pytest.mark.parametrize("N,T", [(2, 1000), (5, 256 * 5 * 4), (16, 16 * 3000 + 5)])
def test_sparse_ring(gran, thr, in_dt, N, T):
    xs = W.sparse(N, T, seed=N + T, dtype=TORCH_DT[in_dt])
    thr32 = float(np.float32(thr))
    out_dt = "f32"
    codec = rra.Codec("sparse", sparsity_threshold=thr, granularity=gran)
    gpu = run_ring(xs, out_dt, codec)
    ref = oracle_ring(xs, in_dt, out_dt, codec="sparse", threshold=thr32, slice=SLICE_OF[gran])
    compare(gpu, ref, f"sparse {gran} thr={thr}")
    # lossless: equals the lossless ring bit for bit
    compare(run_ring(xs, out_dt), (ref[0], *oracle_ring(xs, in_dt, out_dt)[1:]), "vs lossless")


@pytest.mark.parametrize("gran", ["chunk", "slice"])
def test_sparse_ring_all_zero_and_dense(gran):
    N, T = 4, 4096
    zeros = [torch.zeros(T, device="cuda") for _ in range(N)]
    codec = rra.Codec("sparse", granularity=gran)
    gpu = run_ring(zeros, "f32", codec)
    compare(gpu, oracle_ring(zeros, "f32", "f32", codec="sparse", slice=SLICE_OF[gran]), "zeros")
    msgs = 1 if gran == "chunk" else T // N // 256
    assert all(int(s) == 2 * (N - 1) * msgs * 8 for s in gpu[1])  # headers only
    dense = rand_f32(N, T, seed=5)
    compare(run_ring(dense, "f32", codec),
            oracle_ring(dense, "f32", "f32", codec="sparse", slice=SLICE_OF[gran]), "dense")


def _sparse_with_minus_zero(N, T, seed, dt, p_zero=0.6):
    xs = W.sparse(N, T, seed=seed, p_zero=p_zero, dtype=TORCH_DT[dt])
    for r, x in enumerate(xs):
        x[(r * 7) % 13::29] = -0.0
    return xs


@pytest.mark.parametrize("gran", ["chunk", "slice"])
@pytest.mark.parametrize("in_dt", ["bf16", "f32"])
def test_sparse_ring_minus_zero_is_lossless(gran, in_dt):
    """The receiver adds the whole restored message, so -0.0 inputs give the
    lossless ring's bits (a -0.0 meeting an omitted +0.0 becomes +0.0)."""
    N, T = 6, 6 * 2048 + 30
    xs = _sparse_with_minus_zero(N, T, 41, in_dt)
    codec = rra.Codec("sparse", granularity=gran)
    gpu = run_ring(xs, "f32", codec)
    compare(gpu, oracle_ring(xs, in_dt, "f32", codec="sparse", slice=SLICE_OF[gran]), "-0.0")
    lossless = run_ring(xs, "f32")
    for r in range(N):
        assert torch.equal(gpu[0][r].view(torch.int32), lossless[0][r].view(torch.int32))


def _tie_inputs(N, T, dt, thr=0.5):
    """Inputs whose hop-1 messages sit at the per-chunk decision's edge:
    chunk c of rank c+1 has exactly ceil((1 - thr) n) nonzeros for even c
    (dense, since sparse needs nnz < (1 - thr) n) and one fewer for odd c."""
    n = -(-T // N)
    g = torch.Generator(device="cuda")
    g.manual_seed(1234 + N)
    xs = []
    for r in range(N):
        x = torch.zeros(T, device="cuda")
        for c in range(N):
            lo, hi = min(c * n, T), min((c + 1) * n, T)
            if hi == lo:
                continue
            want = int(np.ceil((1 - thr) * (hi - lo)))
            k = want - (c % 2) if (c + 1) % N == r else (hi - lo) // 3
            k = max(0, min(k, hi - lo))
            pos = torch.randperm(hi - lo, generator=g, device="cuda")[:k] + lo
            x[pos] = torch.randn(k, generator=g, device="cuda") * 0.02 + 0.5
        xs.append(x.to(TORCH_DT[dt]))
    return xs


@pytest.mark.parametrize("in_dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N,T", [(2, 2 * 4096), (5, 5 * 1000 + 3), (16, 16 * 2048 + 17)])
def test_sparse_ring_per_chunk_decision_at_the_tie(in_dt, N, T):
    """Per-chunk decisions on both sides of nnz = (1 - threshold) * n: values
    and byte counters bit-exact against the oracle, allreduce and
    reduce-scatter."""
    xs = _tie_inputs(N, T, in_dt)
    codec = rra.Codec("sparse", sparsity_threshold=0.5)
    compare(run_ring(xs, "f32", codec), oracle_ring(xs, in_dt, "f32", codec="sparse"), "tie")
    outs = [torch.full((T,), 7.0, device="cuda") for _ in range(N)]
    ref_outs = [np.full(T, 7.0, np.float32) for _ in range(N)]
    gpu = run_ring(xs, "f32", codec, mode="reduce_scatter", outs=outs)
    ref = O.ring([host(x) for x in xs], in_dt, "f32", codec="sparse", mode="reduce_scatter",
                 outputs=ref_outs)
    compare(gpu, ref, "tie rs")


@pytest.mark.parametrize("G", [1, 2, 4])
def test_sparse_ring_per_chunk_clustered_nonzeros(G):
    """A chunk can be sparse overall while some of its 256-element groups are
    dense: their pairs beyond the 128 a slot holds take the spill path.  Every
    chunk here has its nonzeros packed at its start (a fifth of it), so whole
    groups are fully nonzero in sparse messages."""
    N, T = 8, 8 * 4096 * 2
    n = T // N
    g = torch.Generator(device="cuda")
    g.manual_seed(99)
    xs = []
    for r in range(N):
        x = torch.zeros(T, device="cuda")
        for c in range(N):
            k = n // 5 + 37 * r
            x[c * n: c * n + k] = torch.randn(k, generator=g, device="cuda") + 3.0
        xs.append(x)
    comm = rra.Comm(N, T)
    comm.set_tuning(0, 0, 0, G)
    outs = [torch.empty(T, device="cuda") for _ in range(N)]
    comm.ring_allreduce(xs, outs, rra.Codec("sparse"))
    sent, recv = comm.get_bytes()
    assert comm.status() == rra.RRA_OK
    comm.close()
    ref = oracle_ring(xs, "f32", "f32", codec="sparse")
    compare((outs, sent, recv), ref, f"clustered G={G}")
    # every hop's partial keeps the packed prefix: all messages sparse
    assert all(int(v) < 2 * (N - 1) * (8 + 4 * n) * 0.5 for v in sent)


@pytest.mark.parametrize("G,K", [(1, 1), (1, 2), (2, 2), (4, 2)])
@pytest.mark.parametrize("N", [3, 8, 16])
def test_sparse_ring_per_chunk_launch_shapes(G, K, N):
    """Every slice width and mailbox depth moves the same per-chunk messages."""
    T = N * 4096 * 3 + 8 * N
    xs = _sparse_with_minus_zero(N, T, 50 + N, "bf16", p_zero=0.7)
    comm = rra.Comm(N, T, torch.bfloat16)
    comm.set_tuning(0, K, 0, G)
    outs = [torch.empty(T, device="cuda") for _ in range(N)]
    comm.ring_allreduce(xs, outs, rra.Codec("sparse"))
    sent, recv = comm.get_bytes()
    assert comm.status() == rra.RRA_OK
    shape = comm.last_shape()
    assert shape[3] == G, shape
    comm.close()
    compare((outs, sent, recv), oracle_ring(xs, "bf16", "f32", codec="sparse"), f"G={G} K={K}")


@pytest.mark.parametrize("N", [17, 20, 33])
@pytest.mark.parametrize("kind", ["bf16", "diff"])
def test_sparse_ring_per_chunk_many_ranks(N, kind):
    """More than 16 ranks: warps play several ranks each, and the count pass
    takes its path for more than 16 hops (per-position warp sums); with a
    diff stream the counts are of the fp32 differences."""
    T = N * 2048 + 3 * N + 1
    if kind == "bf16":
        xs = _sparse_with_minus_zero(N, T, 80 + N, "bf16", p_zero=0.7)
        compare(run_ring(xs, "f32", rra.Codec("sparse")),
                oracle_ring(xs, "bf16", "f32", codec="sparse"), f"N={N}")
    else:
        cur, prev = W.diloco(N, T, seed=N)
        for q in range(N):  # unchanged positions: zero differences
            cur[q][: T // 2] = prev[q][: T // 2]
        codec = rra.Codec("sparse", diff_prev=prev, average=True)
        ref = O.ring([host(c) for c in cur], codec="sparse", diff_prev=[host(p) for p in prev],
                     average=True)
        compare(run_ring(cur, "f32", codec), ref, f"diff N={N}")


def test_sparse_ring_per_chunk_generic_path_and_in_place():
    """Buffers off the 16-byte grid take the generic path (bounds-checked
    loads, the count pass's scalar loads); in place, out = in."""
    N, T = 5, 5 * 3001
    base = _sparse_with_minus_zero(N, T + 1, 61, "f32")
    xs = [b[1:] for b in base]  # 4-byte offset: no bulk copies
    ref = oracle_ring(xs, "f32", "f32", codec="sparse")
    compare(run_ring(xs, "f32", rra.Codec("sparse")), ref, "generic")
    bufs = [x.clone() for x in _sparse_with_minus_zero(N, T, 62, "f32")]
    ref = oracle_ring(bufs, "f32", "f32", codec="sparse")
    comm = rra.Comm(N, T)
    comm.ring_allreduce(bufs, bufs, rra.Codec("sparse"))
    sent, recv = comm.get_bytes()
    assert comm.status() == rra.RRA_OK
    comm.close()
    compare((bufs, sent, recv), ref, "in place")


def test_sparse_ring_per_chunk_repeated_calls_and_other_ops():
    """The count tables are reset by every call: a per-chunk sparse call
    after other calls, and twice in a row on other data, on one comm."""
    N, T = 8, 8 * 2048
    comm = rra.Comm(N, T)
    for seed in (1, 2):
        xs = _sparse_with_minus_zero(N, T, 70 + seed, "f32", p_zero=0.3 + 0.4 * seed)
        outs = [torch.empty(T, device="cuda") for _ in range(N)]
        comm.ring_allreduce(xs, outs, rra.Codec("sparse"))
        sent, recv = comm.get_bytes()
        assert comm.status() == rra.RRA_OK
        compare((outs, sent, recv), oracle_ring(xs, "f32", "f32", codec="sparse"), f"call {seed}")
        comm.allgather([o.clone() for o in outs])
        assert comm.status() == rra.RRA_OK
    comm.close()


# ------------------------------------------------------------------ diff / average / base

@pytest.mark.parametrize("codec_kind,bits", [("bfp", 4), ("bfp", 8), ("none", 8), ("sparse", 8)])
@pytest.mark.parametrize("N,T", [(8, 8 * 1000 + 8 * 64), (3, 3000)])
def test_diff_average_base(codec_kind, bits, N, T):
    cur, prev = W.diloco(N, T, seed=3)
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    base = torch.randn(T, generator=g, device="cuda") * 1e-4
    codec = rra.Codec(codec_kind, bits=bits, diff_prev=prev, diff_base=base, average=True)
    gpu = run_ring(cur, "f32", codec)
    ref = O.ring([host(c) for c in cur], codec=codec_kind, bits=bits,
                 diff_prev=[host(p) for p in prev], diff_base=host(base), average=True)
    compare(gpu, ref, f"diff {codec_kind}{bits}")


def test_average_without_base():
    xs = rand_f32(5, 5000, seed=21)
    codec = rra.Codec("none", average=True)
    compare(run_ring(xs, "f32", codec), O.ring([host(x) for x in xs], average=True), "avg")


# ------------------------------------------------------------------ reduce-scatter

@pytest.mark.parametrize("codec_kind,bits,in_dt", [("none", 8, "f32"), ("bfp", 8, "f16"),
                                                   ("bfp", 4, "f32"), ("sparse", 8, "bf16")])
@pytest.mark.parametrize("N,T", [(4, 4096), (7, 10007), (16, 16 * 512)])
def test_reduce_scatter(codec_kind, bits, in_dt, N, T):
    if codec_kind == "sparse":
        xs = W.sparse(N, T, seed=N, dtype=TORCH_DT[in_dt])
    else:
        xs = cast(rand_f32(N, T, seed=N + T, scale=1e-3), in_dt)
    outs = [torch.full((T,), 3.0, device="cuda") for _ in range(N)]
    codec = rra.Codec(codec_kind, bits=bits)
    gpu = run_ring(xs, "f32", codec, mode="reduce_scatter", outs=outs)
    ref_outs = [np.full(T, 3.0, np.float32) for _ in range(N)]
    ref = O.ring([host(x) for x in xs], in_dt, "f32", codec=codec_kind, bits=bits,
                 mode="reduce_scatter", outputs=ref_outs)
    compare(gpu, ref, f"rs {codec_kind}")


def test_reduce_scatter_into_one_shared_buffer():
    """Reduce-scatter writes chunk r of out[r] only, so all ranks may point at
    one buffer; it then holds the whole reduced vector (here the mean)."""
    N, T = 8, 8 * 3000 + 5
    xs = rand_f32(N, T, seed=77)
    shared = torch.zeros(T, device="cuda")
    comm = rra.Comm(N, T)
    comm.reduce_scatter(xs, [shared] * N, rra.Codec("none", average=True))
    assert comm.status() == rra.RRA_OK
    ref = O.ring([host(x) for x in xs], average=True)[0][0]
    assert_bits_equal(host(shared), ref, "shared")
    comm.close()


# ------------------------------------------------------------------ allgather / broadcast / tree

@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N,T", [(1, 10), (2, 1000), (4, 4096), (7, 7 * 300 + 3), (64, 64 * 256)])
def test_allgather(dt, N, T):
    bufs = cast(rand_f32(N, T, seed=N + T), dt)
    ref, s, r = O.allgather([host(b) for b in bufs], dt)
    comm = rra.Comm(N, T, bufs[0].dtype)
    comm.allgather(bufs)
    for q in range(N):
        assert_bits_equal(host(bufs[q]), ref[q], f"allgather {q}")
    assert comm.get_bytes() == (list(s), list(r))
    comm.close()


def _allgather_inputs(N, T, dt, codec, seed):
    xs = rand_f32(N, T, seed=seed, scale=1e-2)
    if codec == "sparse":  # mostly +0.0, with some -0.0 kept as values
        g = torch.Generator(device="cuda")
        g.manual_seed(seed + 1)
        keep = torch.rand(N, T, generator=g, device="cuda") < 0.3
        xs = [torch.where(keep[r], x, torch.zeros_like(x)) for r, x in enumerate(xs)]
        for x in xs:
            x[5::211] = -0.0
    return cast(xs, dt)


@pytest.mark.parametrize("codec,bits", [("bfp", 8), ("bfp", 4), ("sparse", 8)])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N,T", [(1, 300), (2, 512), (3, 1000), (8, 8 * 2048 * 5 + 8 * 24),
                                 (5, 256 * 5 * 3 + 70), (16, 16 * 1024 * 3), (33, 33 * 512 + 7),
                                 (64, 64 * 256 * 2)])
def test_allgather_codec(codec, bits, dt, N, T):
    """Compressed allgather: every buffer holds every owner's decoded chunk,
    bit for bit as the oracle; byte counters exact (full slices, a ragged
    tail, chunk sizes that are and are not 16-byte multiples)."""
    bufs = _allgather_inputs(N, T, dt, codec, seed=N * 101 + T + bits)
    ref, s, r = O.allgather_codec([host(b) for b in bufs], dt, codec, bits)
    comm = rra.Comm(N, T, bufs[0].dtype)
    c = rra.Codec("bfp", bits=bits) if codec == "bfp" else rra.Codec("sparse", sparsity_threshold=0.5)
    comm.allgather(bufs, codec=c)
    assert comm.status() == rra.RRA_OK
    for q in range(N):
        assert_bits_equal(host(bufs[q]), ref[q], f"allgather {codec}{bits} {dt} rank {q}")
    assert comm.get_bytes() == (list(s), list(r))
    comm.close()


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_allgather_codec_launch_shapes(G):
    """Every slice width gives the same bits (fp16 BFP8: the direct fp16 path
    on full slices, the fp32 decode on the ragged tail)."""
    N, T = 8, 8 * 2048 * 7 + 8 * 56
    bufs = _allgather_inputs(N, T, "f16", "bfp", seed=G)
    ref, s, r = O.allgather_codec([host(b) for b in bufs], "f16", "bfp", 8)
    comm = rra.Comm(N, T, torch.float16)
    comm.set_tuning(0, 0, 0, G)
    comm.allgather(bufs, codec=rra.Codec("bfp", bits=8))
    assert comm.status() == rra.RRA_OK and comm.last_shape()[3] == G
    for q in range(N):
        assert_bits_equal(host(bufs[q]), ref[q], f"G={G} rank {q}")
    assert comm.get_bytes() == (list(s), list(r))
    comm.close()


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("N,T", [(3, 1000), (8, 8 * 2048 * 2 + 8 * 24), (16, 16 * 1024 * 3)])
def test_allgather_codec_sparse_per_slice(dt, N, T):
    """The per-slice option of the compressed allgather: one message per 256
    elements of every owner's chunk."""
    bufs = _allgather_inputs(N, T, dt, "sparse", seed=N * 7 + T)
    ref, s, r = O.allgather_codec([host(b) for b in bufs], dt, "sparse", 8, slice=rra.RING_SLICE)
    comm = rra.Comm(N, T, bufs[0].dtype)
    comm.allgather(bufs, codec=rra.Codec("sparse", granularity="slice"))
    assert comm.status() == rra.RRA_OK
    for q in range(N):
        assert_bits_equal(host(bufs[q]), ref[q], f"rank {q}")
    assert comm.get_bytes() == (list(s), list(r))
    comm.close()


def test_sparse_allgather_equals_the_plain_allgather():
    """Sparse codes restore every element: the same bits as the uncompressed
    allgather, including -0.0, with fewer bytes on the wire for fp32."""
    N, T = 8, 8 * 4096
    bufs = _allgather_inputs(N, T, "f32", "sparse", seed=3)
    plain = [b.clone() for b in bufs]
    comm = rra.Comm(N, T)
    comm.allgather(plain)
    _, plain_bytes = comm.get_bytes()
    comm.allgather(bufs, codec=rra.Codec("sparse", sparsity_threshold=0.5))
    _, sparse_bytes = comm.get_bytes()
    for q in range(N):
        assert_bits_equal(host(bufs[q]), host(plain[q]), f"rank {q}")
    assert all(a < b for a, b in zip(sparse_bytes, plain_bytes))
    comm.close()


def test_allgather_codec_after_allreduce_on_one_comm():
    """The allreduce, the compressed allgather and the allreduce again on one
    communicator: each keeps its own launch-shape key and result."""
    N, T = 4, 4 * 2048 * 3
    xs = rand_f32(N, T, seed=8)
    codec = rra.Codec("bfp", bits=8)
    comm = rra.Comm(N, T)
    outs = [torch.zeros(T, device="cuda") for _ in range(N)]
    ref_ar = oracle_ring(xs, "f32", "f32", codec="bfp", bits=8)[0]
    comm.ring_allreduce(xs, outs, codec)
    bufs = [x.clone() for x in xs]
    ref_ag = O.allgather_codec([host(b) for b in bufs], "f32", "bfp", 8)[0]
    comm.allgather(bufs, codec=codec)
    comm.ring_allreduce(xs, outs, codec)
    assert comm.status() == rra.RRA_OK
    for q in range(N):
        assert_bits_equal(host(outs[q]), ref_ar[q], f"allreduce {q}")
        assert_bits_equal(host(bufs[q]), ref_ag[q], f"allgather {q}")
    comm.close()


def test_allgather_codec_argument_errors():
    N, T = 4, 1024
    comm = rra.Comm(N, T)
    bufs = rand_f32(N, T, seed=1)
    for bad in (rra.Codec("bfp", bits=8, average=True), rra.Codec("bfp", bits=5)):
        with pytest.raises(RuntimeError):
            comm.allgather(bufs, codec=bad)
    comm.close()


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("N,root", [(N, root) for N in (1, 2, 3, 5, 8, 13, 64) for root in (0, 2)
                                    if root < N])
@pytest.mark.parametrize("T", [777, 8192])
def test_broadcast(dt, N, root, T):
    bufs = cast(rand_f32(N, T, seed=N * 3 + root), dt)
    ref, s, r = O.broadcast([host(b) for b in bufs], dt, root)
    comm = rra.Comm(N, T, bufs[0].dtype)
    comm.broadcast(bufs, root=root)
    for q in range(N):
        assert_bits_equal(host(bufs[q]), ref[q], f"broadcast {q}")
    assert comm.get_bytes() == (list(s), list(r))
    comm.close()


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N,root", [(1, 0), (2, 1), (5, 2), (8, 3), (16, 0), (33, 7)])
@pytest.mark.parametrize("T", [777, 8192, 3 * 4096 + 128 * 5 + 3])
def test_broadcast_codec(bits, dt, N, root, T):
    """BFP-compressed broadcast: every buffer, the root's included, holds the
    decoded codes of the root's buffer, bit for bit as the oracle; byte
    counters exact (fast and generic paths, one rank per warp and several)."""
    bufs = cast(rand_f32(N, T, seed=N * 13 + root + T + bits, scale=1e-2), dt)
    ref, s, r = O.broadcast_codec([host(b) for b in bufs], dt, root, bits)
    comm = rra.Comm(N, T, bufs[0].dtype)
    comm.broadcast(bufs, root=root, codec=rra.Codec("bfp", bits=bits))
    assert comm.status() == rra.RRA_OK
    for q in range(N):
        assert_bits_equal(host(bufs[q]), ref[q], f"bfp{bits} {dt} broadcast rank {q}")
    assert comm.get_bytes() == (list(s), list(r))
    comm.close()


@pytest.mark.parametrize("G", [1, 2, 4])
def test_broadcast_codec_slice_widths_and_blocks(G):
    """Every slice width, and blocks that are all zero, subnormal, huge or
    round to the clamp, give the oracle's bits."""
    N, T, root = 8, 4096 * 6 + 256 + 40, 5
    g = torch.Generator(device="cuda")
    g.manual_seed(G)
    bufs = [torch.randn(T, generator=g, device="cuda") for _ in range(N)]
    x = bufs[root]
    x[:128] = 0.0
    x[128:256] = torch.randn(128, generator=g, device="cuda") * 1e-39
    x[256:384] *= 1e30
    x[384:512] = 1.9921875
    ref, s, r = O.broadcast_codec([host(b) for b in bufs], "f32", root, 8)
    comm = rra.Comm(N, T)
    comm.set_tuning(0, 0, 0, G)
    comm.broadcast(bufs, root=root, codec=rra.Codec("bfp", bits=8))
    assert comm.status() == rra.RRA_OK
    for q in range(N):
        assert_bits_equal(host(bufs[q]), ref[q], f"G={G} rank {q}")
    assert comm.get_bytes() == (list(s), list(r))
    comm.close()


@pytest.mark.parametrize("G", [0, 1, 2, 4])
def test_broadcast_codec_f16_outputs_across_exponents(G):
    """fp16 buffers of a BFP8 broadcast for block exponents from below the
    fp16 subnormals to near the fp16 maximum, full slices and a ragged tail:
    every rank (the root included) holds the decoded value rounded once to
    fp16, the oracle's bits."""
    N, T, root = 8, 4096 * 5 + 8 * 40 + 3, 2
    g = torch.Generator(device="cuda")
    g.manual_seed(90 + G)
    lo, hi = -30, 13
    nb = -(-T // 128)
    j = (torch.arange(nb, device="cuda") * 5) % (hi - lo + 1) + lo
    scale = torch.pow(2.0, j.float()).repeat_interleave(128)[:T]
    bufs = [(torch.randn(T, generator=g, device="cuda") * scale).half() for _ in range(N)]
    ref, s, r = O.broadcast_codec([host(b) for b in bufs], "f16", root, 8)
    comm = rra.Comm(N, T, torch.float16)
    if G:
        comm.set_tuning(0, 0, 0, G)
    comm.broadcast(bufs, root=root, codec=rra.Codec("bfp", bits=8))
    assert comm.status() == rra.RRA_OK
    for q in range(N):
        assert_bits_equal(host(bufs[q]), ref[q], f"G={G} rank {q}")
    assert comm.get_bytes() == (list(s), list(r))
    comm.close()


def test_broadcast_codec_misaligned_takes_generic_path():
    N, T, root = 4, 5000, 1
    store = cast(rand_f32(N, T + 1, seed=4, scale=1e-2), "f16")
    bufs = [b[1:] for b in store]
    ref, s, r = O.broadcast_codec([host(b) for b in bufs], "f16", root, 8)
    comm = rra.Comm(N, T, torch.float16)
    comm.broadcast(bufs, root=root, codec=rra.Codec("bfp", bits=8))
    assert comm.status() == rra.RRA_OK
    for q in range(N):
        assert_bits_equal(host(bufs[q]), ref[q], f"rank {q}")
    comm.close()


def test_broadcast_codec_argument_errors():
    N, T = 4, 1024
    comm = rra.Comm(N, T)
    bufs = rand_f32(N, T, seed=1)
    for bad, code in ((rra.Codec("sparse", sparsity_threshold=0.5), rra.RRA_ERR_UNSUPPORTED),
                      (rra.Codec("bfp", bits=6), rra.RRA_ERR_INVALID)):
        with pytest.raises(rra.RRAError) as ei:
            comm.broadcast(bufs, root=0, codec=bad)
        assert ei.value.code == code
    with pytest.raises(rra.RRAError):
        comm.broadcast(bufs, root=N, codec=rra.Codec("bfp", bits=8))
    comm.close()


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8, 16, 33, 64])
@pytest.mark.parametrize("T", [300, 8192])
def test_tree_allreduce(N, T):
    bufs = rand_f32(N, T, seed=N * 5 + T)
    ref, s, r = O.tree_allreduce([host(b) for b in bufs])
    comm = rra.Comm(N, T)
    comm.tree_allreduce(bufs)
    for q in range(N):
        assert_bits_equal(host(bufs[q]), ref[q], f"tree {q}")
    assert comm.get_bytes() == (list(s), list(r))
    comm.close()


# ------------------------------------------------------------------ standalone codecs

@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("n", [1, 127, 128, 1000, 65536 + 77])
def test_bfp_codec(bits, dt, n):
    x = cast(rand_f32(1, n, seed=n + bits, scale=3e-2), dt)[0]
    nb = -(-n // 128)
    mb = n if bits == 8 else -(-n // 2)
    exps = torch.zeros(nb, dtype=torch.int8, device="cuda")
    mants = torch.zeros(mb, dtype=torch.uint8, device="cuda")
    rra.bfp_encode(x, bits, exps, mants)
    rx = O.to_f32(host(x), dt)
    re, rm = O.bfp_encode(rx, bits)
    assert np.array_equal(host(exps), re) and np.array_equal(host(mants), rm)
    out = torch.full((n,), 0.5, device="cuda")
    rra.bfp_decode(exps, mants, n, bits, out)
    assert_bits_equal(host(out), O.bfp_decode(re, rm, n, bits), "decode")
    rra.bfp_decode(exps, mants, n, bits, out, accumulate=True)
    acc = O.bfp_decode(re, rm, n, bits)
    O.bfp_decode(re, rm, n, bits, out=acc, accumulate=True)
    assert_bits_equal(host(out), acc, "decode accumulate")


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("p_zero,thr", [(0.6, 0.5), (0.3, 0.5), (0.5, 0.5), (0.95, 0.9)])
@pytest.mark.parametrize("n", [1, 1000, 4096 * 3 + 11, 300000])
def test_sparse_codec(dt, p_zero, thr, n):
    x = W.sparse(1, n, seed=n, p_zero=p_zero, dtype=TORCH_DT[dt])[0]
    hdr = torch.zeros(2, dtype=torch.int32, device="cuda")
    vals = torch.zeros(n, dtype=TORCH_DT[dt], device="cuda")
    idx = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    rra.sparse_encode(x, thr, hdr, vals, idx)
    rh, rv, ri = O.sparse_encode(host(x), dt, float(np.float32(thr)))
    h = host(hdr).view(np.uint32)
    assert list(h) == list(rh)
    k = int(rh[1]) if rh[0] else n
    assert np.array_equal(bitsof_any(host(vals)[:k]), bitsof_any(rv))
    if rh[0]:
        assert np.array_equal(host(idx)[:k], ri)
    acc = torch.full((n,), 2.0, device="cuda")
    rra.sparse_decode(hdr, vals, idx, n, acc)
    assert_bits_equal(host(acc), O.sparse_decode(rh, rv, ri, n, dt), "decode")
    rra.sparse_decode(hdr, vals, idx, n, acc, accumulate=True)
    ra = O.sparse_decode(rh, rv, ri, n, dt)
    O.sparse_decode(rh, rv, ri, n, dt, acc=ra, accumulate=True)
    assert_bits_equal(host(acc), ra, "decode accumulate")


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("offset", [0, 1])
def test_sparse_codec_many_tiles(dt, offset):
    """Long inputs: every block of the encoder and the one-pass decoder walks
    several 4096-element tiles; the decoded view may start off 16-byte
    alignment (element-wise stores)."""
    n = (1 << 24) + 333
    x = W.sparse(1, n, seed=77, p_zero=0.6, dtype=TORCH_DT[dt])[0]
    hdr = torch.zeros(2, dtype=torch.int32, device="cuda")
    vals = torch.zeros(n, dtype=TORCH_DT[dt], device="cuda")
    idx = torch.zeros(n, dtype=torch.int32, device="cuda")
    rra.sparse_encode(x, 0.5, hdr, vals, idx)
    rh, rv, ri = O.sparse_encode(host(x), dt, 0.5)
    assert list(host(hdr).view(np.uint32)) == list(rh) and rh[0] == 1
    k = int(rh[1])
    assert np.array_equal(bitsof_any(host(vals)[:k]), bitsof_any(rv))
    assert np.array_equal(host(idx)[:k], ri)
    store = torch.full((n + offset,), 3.0, device="cuda")
    acc = store[offset:]
    rra.sparse_decode(hdr, vals, idx, n, acc)
    assert_bits_equal(host(acc), O.sparse_decode(rh, rv, ri, n, dt), "decode")
    assert float(store[0]) == 3.0 or offset == 0
    # accumulating, tile by tile, onto a base with no zeros (the last tile is
    # ragged, so the whole-tile and element paths both run)
    base = torch.randn(n, generator=torch.Generator(device="cuda").manual_seed(5), device="cuda")
    acc.copy_(base)
    rra.sparse_decode(hdr, vals, idx, n, acc, accumulate=True)
    ra = host(base).copy()
    O.sparse_decode(rh, rv, ri, n, dt, acc=ra, accumulate=True)
    assert_bits_equal(host(acc), ra, "decode accumulate")
    assert float(store[0]) == 3.0 or offset == 0


def _encode_and_check(x, dt, thr, stream=None):
    n = x.numel()
    hdr = torch.zeros(2, dtype=torch.int32, device="cuda")
    vals = torch.zeros(n, dtype=x.dtype, device="cuda")
    idx = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    rra.sparse_encode(x, thr, hdr, vals, idx, stream=stream)
    torch.cuda.synchronize()
    rh, rv, ri = O.sparse_encode(host(x), dt, float(np.float32(thr)))
    assert list(host(hdr).view(np.uint32)) == list(rh)
    k = int(rh[1]) if rh[0] else n
    assert np.array_equal(bitsof_any(host(vals)[:k]), bitsof_any(rv))
    if rh[0]:
        assert np.array_equal(host(idx)[:k], ri)
    return int(rh[0])


@pytest.mark.parametrize("dt", ["bf16", "f32", "f16"])
@pytest.mark.parametrize("dense_frac,thr", [(0.6, 0.5), (0.97, 0.5), (0.2, 0.9), (0.45, 0.5)])
def test_sparse_encode_dense_prefix_inputs(dt, dense_frac, thr):
    """Nonzeros only in a leading part of x, zeros after it: the format
    follows the total count alone, and a dense message copies the zeros
    too.  (0.45, 0.5) stays sparse."""
    n = 40 * 4096 + 1234
    x = W.sparse(1, n, seed=int(dense_frac * 100), p_zero=0.0, dtype=TORCH_DT[dt])[0]
    x[int(dense_frac * n):] = 0
    fmt = _encode_and_check(x, dt, thr)
    assert fmt == (1 if dense_frac < 1 - thr else 0)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("off", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (0, 2, 2), (3, 3, 3)])
def test_sparse_encode_misaligned_buffers(dt, off):
    """x, vals and idx starting off their 16-byte alignment (element offsets
    1..3): the encoder falls back to element loads and to single-element
    stores of the run; the result is the same bits."""
    n = 5 * 1024 + 77
    ox, ov, oi = off
    big = W.sparse(1, n + ox, seed=ox + 10 * ov + 100 * oi, p_zero=0.6, dtype=TORCH_DT[dt])[0]
    x = big[ox:]
    hdr = torch.zeros(2, dtype=torch.int32, device="cuda")
    vstore = torch.zeros(n + ov, dtype=TORCH_DT[dt], device="cuda")
    istore = torch.full((n + oi,), -1, dtype=torch.int32, device="cuda")
    vals, idx = vstore[ov:], istore[oi:]
    rra.sparse_encode(x, 0.5, hdr, vals, idx)
    rh, rv, ri = O.sparse_encode(host(x), dt, 0.5)
    assert list(host(hdr).view(np.uint32)) == list(rh) and rh[0] == 1
    k = int(rh[1])
    assert np.array_equal(bitsof_any(host(vals)[:k]), bitsof_any(rv))
    assert np.array_equal(host(idx)[:k], ri)
    # nothing written before the views
    assert all(int(v) == 0 for v in host(vstore[:ov]).view(np.uint16 if dt == "bf16" else np.uint32))
    assert all(int(v) == -1 for v in host(istore[:oi]))


@pytest.mark.parametrize("n", [1023, 1024, 1025, 4096 * 1024, 4096 * 1024 + 1])
def test_sparse_encode_chunk_and_segment_edges(n):
    """Sizes at the encoder's 1024-element chunk and 4096-chunk segment
    boundaries, sparse and dense."""
    for pz, fmt in ((0.7, 1), (0.2, 0)):
        x = W.sparse(1, n, seed=n % 97 + int(10 * pz), p_zero=pz, dtype=torch.bfloat16)[0]
        assert _encode_and_check(x, "bf16", 0.5) == fmt


def test_sparse_encode_calls_in_a_row():
    """Encodes of different sizes and dtypes on one stream, sharing the
    stream's scratch: larger and smaller chunk counts in turn, so that a
    count or offset left by an earlier call would show."""
    cases = [((1 << 22) + 17, 0.6, "bf16"), (70_001, 0.7, "f32"), ((1 << 22) + 17, 0.3, "bf16"),
             (5_000_000, 0.8, "f16"), (4096, 0.5, "f32"), ((1 << 22) + 17, 0.6, "bf16")]
    fmts = set()
    for i, (n, pz, dt) in enumerate(cases):
        x = W.sparse(1, n, seed=200 + i, p_zero=pz, dtype=TORCH_DT[dt])[0]
        fmts.add(_encode_and_check(x, dt, 0.5))
    assert fmts == {0, 1}


def test_sparse_codec_concurrent_streams():
    """Encodes and decodes queued on two streams without ordering between
    them: each stream has its own scratch, so both results match the oracle."""
    sizes = [(1 << 22) + 5, (1 << 21) + 4099]
    xs = [W.sparse(1, n, seed=90 + i, p_zero=0.7, dtype=torch.float32)[0]
          for i, n in enumerate(sizes)]
    streams = [torch.cuda.Stream() for _ in sizes]
    outs = []
    for x, n in zip(xs, sizes):
        outs.append((torch.zeros(2, dtype=torch.int32, device="cuda"),
                     torch.zeros(n, device="cuda"),
                     torch.zeros(n, dtype=torch.int32, device="cuda"),
                     torch.full((n,), 5.0, device="cuda")))
    torch.cuda.synchronize()
    for _ in range(3):
        for x, st, (hdr, vals, idx, _) in zip(xs, streams, outs):
            rra.sparse_encode(x, 0.5, hdr, vals, idx, stream=st)
        for n, st, (hdr, vals, idx, acc) in zip(sizes, streams, outs):
            rra.sparse_decode(hdr, vals, idx, n, acc, stream=st)
    torch.cuda.synchronize()
    for x, n, (hdr, vals, idx, acc) in zip(xs, sizes, outs):
        rh, rv, ri = O.sparse_encode(host(x), "f32", 0.5)
        assert list(host(hdr).view(np.uint32)) == list(rh) and rh[0] == 1
        k = int(rh[1])
        assert np.array_equal(host(vals)[:k].view(np.uint32), rv.view(np.uint32))
        assert np.array_equal(host(idx)[:k], ri)
        assert_bits_equal(host(acc), O.sparse_decode(rh, rv, ri, n, "f32"), "decode")


def bitsof_any(a):
    return a.view({4: np.uint32, 2: np.uint16}[a.dtype.itemsize])


@pytest.mark.parametrize("n", [1, 7, 4096, 100003])
def test_diff_codec(n):
    cur, prev = W.diloco(1, n, seed=n)
    d = torch.empty(n, device="cuda")
    rra.diff_encode(cur[0], prev[0], d)
    assert_bits_equal(host(d), O.diff_encode(host(cur[0]), host(prev[0])), "diff")


# ------------------------------------------------------------------ failure detection, determinism

@pytest.mark.parametrize("op", ["ring", "allgather", "broadcast", "tree", "allgather_codec",
                                "broadcast_codec"])
def test_withheld_message_times_out(op):
    """A simulated rank that never publishes one message: its receiver's
    bounded wait runs out, the launch returns, the communicator reports
    RRA_ERR_TIMEOUT, and the next call works again."""
    N, T = 4, 4096
    xs = rand_f32(N, T, seed=31)
    comm = rra.Comm(N, T)
    comm.set_timeout(20_000_000)  # 20 ms
    # rank 1 sends at the first step of the ring, the allgather and the tree's
    # first reduce level; in the broadcasts only the root sends at level 0;
    # the compressed allgather's first send is the owner's, at ring step N
    comm.debug_withhold(0 if op.startswith("broadcast") else 1, N if op == "allgather_codec" else 1)
    outs = [torch.zeros(T, device="cuda") for _ in range(N)]
    bufs = [x.clone() for x in xs]
    bfp8 = rra.Codec("bfp", bits=8)
    if op == "ring":
        comm.ring_allreduce(xs, outs)
    elif op == "allgather":
        comm.allgather(bufs)
    elif op == "broadcast":
        comm.broadcast(bufs, root=0)
    elif op == "allgather_codec":
        comm.allgather(bufs, codec=bfp8)
    elif op == "broadcast_codec":
        comm.broadcast(bufs, root=0, codec=bfp8)
    else:
        comm.tree_allreduce(bufs)
    assert comm.status() == rra.RRA_ERR_TIMEOUT
    assert comm.status() == rra.RRA_OK  # reading clears it
    comm.set_timeout(0)
    comm.ring_allreduce(xs, outs)
    assert comm.status() == rra.RRA_OK
    ref = O.ring([host(x) for x in xs])
    assert_bits_equal(host(outs[2]), ref[0][2], "after recovery")
    comm.close()


def test_repeat_runs_bit_identical():
    N, T = 8, 8 * 4096 + 100
    xs = cast(rand_f32(N, T, seed=41, scale=1e-3), "f16")
    comm = rra.Comm(N, T, torch.float16)
    codec = rra.Codec("bfp", bits=8)
    first = None
    for _ in range(10):
        outs = [torch.empty(T, dtype=torch.float16, device="cuda") for _ in range(N)]
        comm.ring_allreduce(xs, outs, codec)
        cur = torch.stack(outs).cpu()
        if first is None:
            first = cur
        assert torch.equal(cur.view(torch.int16), first.view(torch.int16))
    comm.close()


def test_argument_errors_are_reported_on_the_host():
    comm = rra.Comm(4, 1000)
    xs = rand_f32(4, 1000, seed=1)
    with pytest.raises(rra.RRAError):
        comm.ring_allreduce(xs, xs, rra.Codec("bfp", bits=5))
    with pytest.raises(rra.RRAError):
        comm.ring_allreduce(xs, [xs[0]] * 4)  # outputs overlap
    big = rand_f32(4, 2000, seed=1)
    with pytest.raises(rra.RRAError):
        comm.ring_allreduce(big, big)  # count > max_count
    with pytest.raises(rra.RRAError):
        comm.broadcast(xs, root=4)
    with pytest.raises(rra.RRAError):
        comm.tree_allreduce(cast(xs, "f16"))
    comm.close()


# ------------------------------------------------------------------ forced launch shapes

@pytest.mark.parametrize("codec_kind,bits,in_dt", [("none", 8, "f32"), ("bfp", 8, "f16"),
                                                   ("bfp", 4, "bf16"), ("sparse", 8, "bf16")])
@pytest.mark.parametrize("N,T", [(8, 8 * 2048 * 3 + 8 * 700 + 3), (5, 5 * 1300 + 2),
                                 (20, 20 * 1024 + 7)])
def test_forced_launch_shapes(codec_kind, bits, in_dt, N, T):
    """Every slice width (1, 2, 4, 8 groups of 256), staging depth and block
    count gives the oracle's bits and byte counts: the shape changes only how
    the work is cut, never what is computed.  Covers multi-group sparse
    slices (one sub-message per group) and ranks shared by a warp (N=20)."""
    if codec_kind == "sparse":
        xs = W.sparse(N, T, seed=N + T, dtype=TORCH_DT[in_dt])
    else:
        xs = cast(rand_f32(N, T, seed=N + T, scale=1e-3), in_dt)
    codec = rra.Codec(codec_kind, bits=bits)
    ref = oracle_ring(xs, in_dt, "f32", codec=codec_kind, bits=bits)
    comm = rra.Comm(N, T, xs[0].dtype)
    for G in (1, 2, 4, 8):
        for D, blocks in ((1, 0), (3, 1)):
            comm.set_tuning(blocks, 0, D, G)
            outs = [torch.zeros(T, device="cuda") for _ in range(N)]
            comm.ring_allreduce(xs, outs, codec)
            sent, recv = comm.get_bytes()
            assert comm.status() == rra.RRA_OK
            got_G = comm.last_shape()[3]
            # a width that does not fit the shared memory falls back to a narrower one;
            # with one stage and at most 8 ranks every instantiated width fits
            if N <= 8 and D == 1 and not (codec_kind == "sparse" and G == 8):
                assert got_G == G, (G, got_G)
            compare((outs, np.array(sent, np.uint64), np.array(recv, np.uint64)), ref,
                    f"{codec_kind}{bits} G={G} D={D} blocks={blocks}")
    comm.close()
