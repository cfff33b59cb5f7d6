"""Property-based pins for the CPU oracle: random shapes, magnitudes and zero
patterns drawn by hypothesis, each case checked against the pure-Python brute
force or a closed form -- never against the oracle itself.  No GPU is needed.

Sources: "从零实现集合通信", "两趟实现 ring allreduce" (the two-pass schedule and
its 2T(N-1)/N bytes per rank); "CCCL通信压缩库" §2.1 (block floating point with
a shared exponent per block, sparse values + indices above a threshold) and
its operator-aware layer (compressed allgather and broadcast) and its
error feedback (§5: carry what one round's compression lost into the next)."""
import math

import numpy as np
import pytest

import brute
import oracle as O

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import HealthCheck, given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

SETTINGS = settings(max_examples=40, deadline=None,
                    suppress_health_check=[HealthCheck.too_slow])


@st.composite
def vectors(draw, max_len=300):
    """float32 vectors mixing magnitudes, exact zeros and -0.0."""
    n = draw(st.integers(1, max_len))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(n) * 10.0 ** rng.integers(-30, 30, n).astype(np.float64)
    x[rng.random(n) < draw(st.floats(0.0, 0.95))] = 0.0
    x[rng.random(n) < 0.05] = -0.0
    return x.astype(np.float32)


@SETTINGS
@given(x=vectors(), bits=st.sampled_from([8, 4]))
def test_bfp_round_trip_equals_brute_force(x, bits):
    """Encode then decode block by block: the oracle's values equal the
    brute force's (frexp/ldexp/round-half-even restatement), bit for bit."""
    exps, mants = O.bfp_encode(x, bits)
    got = O.bfp_decode(exps, mants, x.size, bits)
    want, nbytes = brute.bfp_roundtrip([np.float32(v) for v in x], bits)
    assert np.array_equal(got.view(np.uint32), np.array(want, np.float32).view(np.uint32))
    assert O.bfp_bytes(x.size, bits) == nbytes


@SETTINGS
@given(x=vectors(), bits=st.sampled_from([8, 4]))
def test_bfp_error_bound(x, bits):
    """Every element is within half a code step 2^(e-q-1) of its input, or
    within one step when its code was clamped (e: the block exponent)."""
    q, M = bits - 2, 2 ** (bits - 1) - 1
    exps, mants = O.bfp_encode(x, bits)
    y = O.bfp_decode(exps, mants, x.size, bits)
    for b in range(0, x.size, 128):
        blk = x[b:b + 128]
        e = O.bfp_block_exponent(blk)
        step = math.ldexp(1.0, e - q)
        for v, w in zip(blk, y[b:b + 128]):
            clamped = abs(float(v)) / step > M + 0.5
            assert abs(float(v) - float(w)) <= (step if clamped else step / 2)


@SETTINGS
@given(x=vectors(), thr=st.sampled_from([0.2, 0.5, 0.9]))
def test_sparse_round_trip_is_exact(x, thr):
    """The sparse codec restores every element bit for bit (-0.0 included),
    and chooses the sparse form exactly when nnz < (1 - threshold) * n."""
    hdr, vals, idx = O.sparse_encode(x, "f32", thr)
    nnz = sum(1 for v in x if brute.nonzero(v))
    assert int(hdr[1]) == nnz
    assert bool(hdr[0]) == (nnz < (1.0 - thr) * x.size)
    if hdr[0]:
        assert list(idx) == sorted(set(int(i) for i in idx))
    y = O.sparse_decode(hdr, vals, idx, x.size, "f32")
    assert np.array_equal(y.view(np.uint32), x.view(np.uint32))


@SETTINGS
@given(N=st.integers(1, 4), T=st.integers(1, 64), seed=st.integers(0, 2 ** 31 - 1),
       codec=st.sampled_from(["none", "bfp8", "bfp4", "sparse"]))
def test_ring_allreduce_equals_brute_force(N, T, seed, codec):
    """The two-pass ring (every codec) against the brute force's literal
    restatement: outputs bit for bit and per-rank byte counts."""
    xs = [x for x in O_rand(N, T, seed)]
    kind, bits = ("bfp", int(codec[3])) if codec.startswith("bfp") else (codec, 8)
    outs, sent, recv = O.ring([x.copy() for x in xs], codec=kind, bits=bits)
    ref, bs, br = brute.ring([list(x) for x in xs], codec=kind, bits=bits)
    for r in range(N):
        assert np.array_equal(outs[r].view(np.uint32), np.array(ref[r], np.float32).view(np.uint32))
    assert list(sent) == bs and list(recv) == br
    if codec == "none" and T % N == 0:
        assert all(int(s) == 2 * (N - 1) * (T // N) * 4 for s in sent)


@SETTINGS
@given(N=st.integers(1, 5), T=st.integers(1, 80), seed=st.integers(0, 2 ** 31 - 1),
       sl=st.sampled_from([None, 1, 3, 8, 16]), zero_p=st.sampled_from([0.3, 0.6, 0.9]),
       thr=st.sampled_from([0.0, 0.25, 0.5, 0.75]))
def test_sparse_ring_is_the_lossless_ring_with_message_bytes(N, T, seed, sl, zero_p, thr):
    """Sparse codes (one message per chunk, or per slice) restore every value
    and the receiver adds the restored message, so the outputs are the
    lossless ring's bit for bit (-0.0 included); the byte counts are the
    brute force's."""
    rng = np.random.default_rng(seed)
    xs = []
    for _ in range(N):
        x = rng.standard_normal(T).astype(np.float32)
        x[rng.random(T) < zero_p] = 0.0
        x[rng.random(T) < 0.05] = -0.0
        xs.append(x)
    outs, sent, recv = O.ring([x.copy() for x in xs], codec="sparse", threshold=thr, slice=sl)
    ls, _, _ = O.ring([x.copy() for x in xs])
    _, bs, br = brute.ring([list(x) for x in xs], codec="sparse", threshold=thr, slice_len=sl)
    for r in range(N):
        assert np.array_equal(outs[r].view(np.uint32), ls[r].view(np.uint32))
    assert list(sent) == bs and list(recv) == br


@SETTINGS
@given(N=st.integers(1, 5), T=st.integers(1, 700), seed=st.integers(0, 2 ** 31 - 1),
       bits=st.sampled_from([8, 4]))
def test_compressed_allgather_is_each_chunks_round_trip(N, T, seed, bits):
    """Every buffer ends with the BFP round trip of each owner's chunk, and
    every rank forwards all chunks but its successor's."""
    xs = O_rand(N, T, seed)
    out, sent, _ = O.allgather_codec([x.copy() for x in xs], "f32", "bfp", bits)
    n = -(-T // N)
    msg = []
    for c in range(N):
        lo, hi = min(c * n, T), min((c + 1) * n, T)
        want, nb = brute.bfp_roundtrip([np.float32(v) for v in xs[c][lo:hi]], bits)
        msg.append(nb if hi > lo else 0)
        for r in range(N):
            assert np.array_equal(out[r][lo:hi].view(np.uint32),
                                  np.array(want, np.float32).view(np.uint32))
    assert [int(s) for s in sent] == [sum(msg) - msg[(r + 1) % N] for r in range(N)]


@SETTINGS
@given(N=st.integers(1, 9), T=st.integers(1, 600), pick=st.integers(0, 2 ** 20),
       seed=st.integers(0, 2 ** 31 - 1), bits=st.sampled_from([8, 4]))
def test_compressed_broadcast_is_the_roots_round_trip(N, T, pick, seed, bits):
    """Every buffer, the root's included, ends with the BFP round trip of the
    root's buffer; each non-root rank receives one message, and the root
    sends one to each of its ceil(log2 N) children in the binomial tree."""
    root = pick % N
    xs = O_rand(N, T, seed)
    out, sent, recv = O.broadcast_codec([x.copy() for x in xs], "f32", root, bits)
    want, nb = brute.bfp_roundtrip([np.float32(v) for v in xs[root]], bits)
    for r in range(N):
        assert np.array_equal(out[r].view(np.uint32), np.array(want, np.float32).view(np.uint32))
    assert [int(v) for v in recv] == [0 if r == root else nb for r in range(N)]
    assert int(sum(sent)) == (N - 1) * nb
    assert int(sent[root]) == brute.ceil_log2(N) * nb


@SETTINGS
@given(N=st.integers(1, 4), T=st.integers(1, 300), seed=st.integers(0, 2 ** 31 - 1),
       bits=st.sampled_from([8, 4]))
def test_error_feedback_from_zero_residual_is_the_plain_ring(N, T, seed, bits):
    """With every residual zero, adding it changes no code (v + 0 only turns
    -0.0 into +0.0, which encodes the same), so the first round of error
    feedback delivers exactly the plain compressed ring's result."""
    xs = O_rand(N, T, seed)
    res = [np.zeros(T, np.float32) for _ in range(N)]
    ef, s_ef, _ = O.ring([x.copy() for x in xs], codec="bfp", bits=bits, residual=res)
    plain, s_plain, _ = O.ring([x.copy() for x in xs], codec="bfp", bits=bits)
    for r in range(N):
        assert np.array_equal(ef[r].view(np.uint32), plain[r].view(np.uint32))
    assert list(s_ef) == list(s_plain)


@SETTINGS
@given(N=st.integers(1, 9), T=st.integers(1, 80), seed=st.integers(0, 2 ** 31 - 1))
def test_tree_allreduce_equals_brute_force(N, T, seed):
    """The binomial-tree allreduce (reduce to rank 0, then broadcast) against
    the brute force: every buffer bit for bit, and the per-rank byte counts."""
    xs = O_rand(N, T, seed)
    out, sent, recv = O.tree_allreduce([x.copy() for x in xs])
    ref, bs, br = brute.tree_allreduce([list(x) for x in xs])
    for r in range(N):
        assert np.array_equal(out[r].view(np.uint32), np.array(ref[r], np.float32).view(np.uint32))
    assert [int(v) for v in sent] == bs and [int(v) for v in recv] == br


@SETTINGS
@given(N=st.integers(1, 5), T=st.integers(1, 64), seed=st.integers(0, 2 ** 31 - 1),
       codec=st.sampled_from(["none", "bfp8", "sparse"]))
def test_reduce_scatter_equals_brute_force(N, T, seed, codec):
    """The first pass alone: chunk r of rank r's output against the brute
    force, and the byte counts of N-1 steps."""
    xs = O_rand(N, T, seed)
    kind, bits = ("bfp", 8) if codec == "bfp8" else (codec, 8)
    outs, sent, recv = O.ring([x.copy() for x in xs], codec=kind, bits=bits,
                              mode="reduce_scatter")
    ref, bs, br = brute.ring([list(x) for x in xs], codec=kind, bits=bits,
                             mode="reduce_scatter")
    for r, (lo, hi) in enumerate(brute.chunks(T, N)):
        want = np.array(ref[r][lo:hi], np.float32)
        assert np.array_equal(outs[r][lo:hi].view(np.uint32), want.view(np.uint32))
    assert list(sent) == bs and list(recv) == br


@SETTINGS
@given(N=st.integers(1, 5), T=st.integers(1, 300), seed=st.integers(0, 2 ** 31 - 1),
       bits=st.sampled_from([8, 4]), average=st.booleans())
def test_difference_ring_equals_brute_force(N, T, seed, bits, average):
    """The ring on cur - prev with the base added back (and the average
    taken) against the brute force, on every rank."""
    rng = np.random.default_rng(seed)
    prev = [(rng.standard_normal(T) * 1e-4).astype(np.float32) for _ in range(N)]
    cur = [(p + (rng.standard_normal(T) * 1e-5).astype(np.float32)).astype(np.float32)
           for p in prev]
    base = (rng.standard_normal(T) * 1e-4).astype(np.float32)
    outs, sent, _ = O.ring([c.copy() for c in cur], codec="bfp", bits=bits, diff_prev=prev,
                           diff_base=base, average=average)
    ref, bs, _ = brute.ring([list(c) for c in cur], codec="bfp", bits=bits,
                            diff_prev=[list(p) for p in prev], diff_base=list(base),
                            average=average)
    for r in range(N):
        assert np.array_equal(outs[r].view(np.uint32), np.array(ref[r], np.float32).view(np.uint32))
    assert list(sent) == bs


@SETTINGS
@given(N=st.integers(1, 5), T=st.integers(1, 700), seed=st.integers(0, 2 ** 31 - 1),
       op=st.sampled_from(["allreduce", "allgather", "broadcast"]), pick=st.integers(0, 99))
def test_codec_statistics_equal_brute_force(N, T, seed, op, pick):
    """The statistics behind the adaptive codec choice, per operation,
    against the brute force over exactly the elements that operation
    encodes (all chunks of all buffers; chunk r of buffer r; the root's
    buffer as one message)."""
    xs = O_rand(N, T, seed, tiny=True)
    root = pick % N
    got = [int(v) for v in O.codec_stats_op([x.copy() for x in xs], "f32", op, root)]
    if op == "allreduce":
        want = brute.codec_stats([list(x) for x in xs])
    elif op == "broadcast":
        want = brute.codec_stats([list(xs[root])])
    else:
        want = [0, 0, 0, 0]
        for r, (lo, hi) in enumerate(brute.chunks(T, N)):
            part = brute.codec_stats([list(xs[r][lo:hi])]) if hi > lo else [0, 0, 0, 0]
            want = [a + b for a, b in zip(want, part)]
    assert got == want


def O_rand(N, T, seed, tiny=False):
    rng = np.random.default_rng(seed)
    xs = []
    for _ in range(N):
        # tiny: magnitudes over 12 decades, so that blocks flush small elements
        span = 6 if tiny else 3
        x = rng.standard_normal(T) * 10.0 ** rng.integers(-span, span, T).astype(np.float64)
        x[rng.random(T) < 0.3] = 0.0
        xs.append(x.astype(np.float32))
    return xs
