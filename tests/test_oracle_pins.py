"""Pins for the CPU oracle: each test ties the oracle to something other than
itself -- values derived by hand from the pages' definitions (tests/golden),
closed forms, invariants, textbook special cases, library routines (numpy /
torch conversions and float32 arithmetic, math.fsum, frexp), error bounds and
an independent brute force on tiny inputs.  No GPU is needed.

Sources: "从零实现集合通信" (collective ops from scratch), section "两趟实现
ring allreduce" (schedule, 2T(N-1)/N bytes per rank, byte/step table) and
"用 gloo 来验证" (check against a reference within float32 epsilon);
"CCCL通信压缩库" §2.1 / §3.3 (block floating point, sparse values+indices,
difference encoding, threshold 0.5).
"""
import math
import os
import struct

import numpy as np
import pytest
import torch

import brute
import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U = 2.0 ** -24  # unit roundoff of binary32


def rand_ranks(N, T, seed, dtype=np.float32, scale=1.0):
    rng = np.random.default_rng(seed)
    return [(rng.standard_normal(T) * scale).astype(dtype) for _ in range(N)]


def bits32(a):
    return np.asarray(a, np.float32).view(np.uint32)


# --------------------------------------------------------------- conversions

def test_f16_conversion_matches_numpy():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 20000),
        np.array([0.0, -0.0, 65504, 65519.99, 65520, 65536, 1e9, -1e9, 2 ** -14, 2 ** -24, 2 ** -25,
                  3 * 2 ** -26, 2 ** -25 * 1.0000001, 5.960464477539063e-08, np.inf, -np.inf],
                 np.float32)]).astype(np.float32)
    ours = O.from_f32(vals, "f16")
    with np.errstate(over="ignore"):  # overflow to infinity is one of the cases
        ref = vals.astype(np.float16)
    assert np.array_equal(ours.view(np.uint16), ref.view(np.uint16))
    back = O.to_f32(ours, "f16")
    assert np.array_equal(bits32(back), bits32(ref.astype(np.float32)))


def test_bf16_conversion_matches_torch():
    rng = np.random.default_rng(2)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 20000),
        np.array([0.0, -0.0, 3.3895314e38, 3.4e38, 1e-39, 1e-45, -1e-40, np.inf, -np.inf,
                  1.00390625, 1.01171875, 1.0078125 + 2 ** -20], np.float32)]).astype(np.float32)
    ours = O.from_f32(vals, "bf16")
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = O.to_f32(ours, "bf16")
    assert np.array_equal(bits32(back), bits32((ours.astype(np.uint32) << 16).view(np.float32)))


def test_scalar_casts_match_library_routines():
    """The scalar fp32 -> fp16 / bf16 helpers agree with numpy's and torch's
    round-to-nearest-even conversions, ties and overflow included."""
    vals = [0.0, -0.0, 1.0, 65504.0, 65520.0, 2.0 ** -25, 3 * 2.0 ** -26, 1.00390625,
            1.01171875, -3.3895314e38, 1e-40, 0.1, -7.3e-5]
    for v in vals:
        f = np.float32(v)
        with np.errstate(over="ignore"):  # 65520 rounds to infinity
            half = np.array(f).astype(np.float16)
        assert O.f32_to_f16_bits(float(f)) == int(half.view(np.uint16))
        want = torch.tensor([f]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)[0]
        assert O.f32_to_bf16_bits(float(f)) == int(want)


# --------------------------------------------------------------- lossless ring

@pytest.mark.parametrize("N", [1, 2, 3, 4])
@pytest.mark.parametrize("T", [1, 3, 7, 16, 33, 64])
def test_ring_lossless_brute_force(N, T):
    xs = rand_ranks(N, T, seed=N * 100 + T)
    outs, sent, recv = O.ring(xs)
    ref, bs, br = brute.ring([list(x) for x in xs])
    for r in range(N):
        assert np.array_equal(bits32(outs[r]), bits32(np.array(ref[r], np.float32)))
    assert list(sent) == bs and list(recv) == br


@pytest.mark.parametrize("N,T", [(2, 4096), (4, 4096), (5, 1000), (8, 12345), (16, 4096)])
def test_ring_lossless_invariants(N, T):
    """All ranks end bit-identical; each element is within the classical
    recursive-summation bound (N-1) u sum|x| of the exact sum (math.fsum)."""
    xs = rand_ranks(N, T, seed=N + T)
    outs, sent, recv = O.ring(xs)
    for r in range(1, N):
        assert np.array_equal(bits32(outs[r]), bits32(outs[0]))
    X = np.stack(xs).astype(np.float64)
    for i in range(0, T, max(1, T // 97)):
        exact = math.fsum(X[:, i])
        bound = (N - 1) * U * math.fsum(np.abs(X[:, i])) * (1 + 1e-6)
        assert abs(float(outs[0][i]) - exact) <= bound


def test_ring_lossless_order_is_the_ring_order():
    """The oracle's sum for chunk c is ((x_{c+1}+x_{c+2})+...)+x_c in float32:
    checked against numpy float32 adds in that order, for a case where a
    different association gives a different answer."""
    N, T = 4, 4
    big, tiny = np.float32(2.0 ** 24), np.float32(1.0)
    xs = [np.full(T, v, np.float32) for v in (big, tiny, tiny, -big)]
    outs, _, _ = O.ring(xs)
    n = 1
    for c in range(N):
        acc = xs[(c + 1) % N][c * n]
        for k in range(2, N + 1):
            acc = np.float32(acc + xs[(c + k) % N][c * n])
        assert outs[0][c] == acc
    assert len(set(float(v) for v in outs[0])) > 1  # association visibly matters


def test_ring_N1_identity_zero_bytes():
    x = rand_ranks(1, 100, 3)
    outs, sent, recv = O.ring(x)
    assert np.array_equal(bits32(outs[0]), bits32(x[0])) and sent[0] == 0 and recv[0] == 0


def test_ring_N2_is_one_float32_add():
    a, b = rand_ranks(2, 1000, 4)
    outs, _, _ = O.ring([a, b])
    ref = (a + b).astype(np.float32)  # numpy float32 add, RNE
    assert np.array_equal(bits32(outs[0]), bits32(ref)) and np.array_equal(bits32(outs[1]), bits32(ref))


@pytest.mark.parametrize("N,T", [(4, 4096), (8, 8192), (3, 10), (7, 100), (5, 3)])
def test_ring_byte_counter_closed_form(N, T):
    """Lossless: every rank sends and receives 2(N-1) chunk messages of 4 B
    per element: 2T(N-1)/N * 4 bytes when N divides T ("two-pass ring")."""
    xs = rand_ranks(N, T, 5)
    _, sent, recv = O.ring(xs)
    n = -(-T // N)
    lens = [max(0, min(T, (c + 1) * n) - c * n) for c in range(N)]
    for r in range(N):
        rs = sum(lens[(r - s) % N] for s in range(1, N))
        ag = sum(lens[(r - s + 1) % N] for s in range(1, N))
        assert sent[r] == 4 * (rs + ag)
        assert recv[(r + 1) % N] == sent[r]
    if T % N == 0:
        assert all(int(s) == 2 * T * (N - 1) // N * 4 for s in sent)


def test_ring_config1_byte_counter():
    xs = rand_ranks(4, 4096, 0)
    _, sent, recv = O.ring(xs)
    assert list(sent) == [24576] * 4 and list(recv) == [24576] * 4


@pytest.mark.parametrize("in_t,out_t", [("f16", "f32"), ("bf16", "bf16"), ("f32", "f16")])
def test_ring_dtypes_widen_then_cast(in_t, out_t):
    N, T = 3, 50
    rng = np.random.default_rng(7)
    xs32 = [rng.standard_normal(T).astype(np.float32) for _ in range(N)]
    xs = [O.from_f32(x, in_t) for x in xs32]
    outs, sent, _ = O.ring(xs, in_t, out_t)
    wide = [O.to_f32(x, in_t) for x in xs]
    ref, _, _ = O.ring(wide)
    assert np.array_equal(outs[1], O.from_f32(ref[1], out_t))
    assert sent[0] == 4 * 2 * (T - -(-T // N))  # fp32 on the wire


# --------------------------------------------------------------- reduce-scatter / allgather

@pytest.mark.parametrize("N,T", [(2, 10), (3, 64), (4, 64), (4, 4096)])
def test_reduce_scatter(N, T):
    xs = rand_ranks(N, T, 11)
    fill = [np.full(T, 7.0, np.float32) for _ in range(N)]
    outs, sent, recv = O.ring(xs, mode="reduce_scatter", outputs=fill)
    full, _, _ = O.ring(xs)
    n = -(-T // N)
    for r in range(N):
        lo, hi = min(r * n, T), min((r + 1) * n, T)
        assert np.array_equal(bits32(outs[r][lo:hi]), bits32(full[0][lo:hi]))
        rest = np.concatenate([outs[r][:lo], outs[r][hi:]])
        assert (rest == 7.0).all()
    if T % N == 0:
        assert all(int(s) == 4 * T * (N - 1) // N for s in sent)
    if N <= 4 and T <= 64:
        ref, bs, _ = brute.ring([list(x) for x in xs], mode="reduce_scatter")
        for r in range(N):
            lo, hi = min(r * n, T), min((r + 1) * n, T)
            assert np.array_equal(bits32(outs[r][lo:hi]), bits32(np.array(ref[r][lo:hi], np.float32)))
        assert list(sent) == bs


@pytest.mark.parametrize("N,T,dt", [(2, 10, "f32"), (4, 4096, "f32"), (3, 11, "f16"), (4, 64, "bf16")])
def test_allgather(N, T, dt):
    rng = np.random.default_rng(12)
    bufs = [O.from_f32(rng.standard_normal(T).astype(np.float32), dt) for _ in range(N)]
    n = -(-T // N)
    expect = np.concatenate([bufs[c][min(c * n, T):min((c + 1) * n, T)] for c in range(N)])
    orig = [b.copy() for b in bufs]
    out, sent, recv = O.allgather(bufs, dt)
    for r in range(N):
        assert np.array_equal(out[r].view(np.uint8), expect.view(np.uint8))
    es = 4 if dt == "f32" else 2
    if T % N == 0:
        assert all(int(s) == es * T * (N - 1) // N for s in sent)
    ref, bs, _ = brute.allgather([list(b.view(np.uint32 if es == 4 else np.uint16)) for b in orig], es)
    assert list(sent) == bs
    for r in range(N):
        assert np.array_equal(np.array(ref[r]), out[r].view(np.uint32 if es == 4 else np.uint16))


# --------------------------------------------------------------- compressed allgather
# Reading AG: the owner encodes its chunk once, the codes travel the ring
# unchanged, every rank (owner included) stores the decoded chunk.

@pytest.mark.parametrize("codec,bits", [("bfp", 8), ("bfp", 4), ("sparse", 8)])
@pytest.mark.parametrize("N,T", [(1, 10), (2, 64), (3, 50), (4, 64), (4, 17)])
def test_allgather_codec_brute_force(codec, bits, N, T):
    rng = np.random.default_rng(N * 31 + T)
    xs = [(rng.standard_normal(T) * (rng.random(T) < 0.3)).astype(np.float32) for _ in range(N)]
    out, sent, recv = O.allgather_codec([x.copy() for x in xs], "f32", codec, bits)
    ref, bs, br = brute.allgather_codec([list(x) for x in xs], codec, bits)
    for r in range(N):
        assert np.array_equal(out[r].view(np.uint32), np.array(ref[r], np.float32).view(np.uint32))
    assert list(sent) == bs and list(recv) == br


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_allgather_codec_is_the_chunk_codec_everywhere(bits, dt):
    """Every buffer ends with, for each chunk c, the standalone codec's round
    trip of the owner's chunk c, cast to the buffer's dtype; the byte counts
    are the message sizes of the N - 1 chunks each rank forwards (all but
    chunk r + 1)."""
    N, T = 5, 5 * 300 + 7
    rng = np.random.default_rng(bits + len(dt))
    bufs = [O.from_f32((rng.standard_normal(T) * 1e-2).astype(np.float32), dt) for _ in range(N)]
    n = -(-T // N)
    lims = [(min(c * n, T), min((c + 1) * n, T)) for c in range(N)]
    want, msg = [], []
    for c, (lo, hi) in enumerate(lims):
        x = O.to_f32(bufs[c][lo:hi], dt)
        exps, mants = O.bfp_encode(x, bits)
        want.append(O.from_f32(O.bfp_decode(exps, mants, hi - lo, bits), dt))
        msg.append(O.bfp_bytes(hi - lo, bits))
    out, sent, recv = O.allgather_codec([b.copy() for b in bufs], dt, "bfp", bits)
    for r in range(N):
        for c, (lo, hi) in enumerate(lims):
            assert np.array_equal(out[r][lo:hi], want[c]), (r, c)
        assert int(sent[r]) == sum(msg) - msg[(r + 1) % N]
        assert int(recv[r]) == sum(msg) - msg[r]


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("N,T", [(2, 512), (4, 4096), (5, 1001)])
def test_allgather_codec_is_the_allreduce_second_pass(bits, N, T):
    """The compressed allreduce is its reduce-scatter followed by this
    allgather of the owners' fp32 sums: outputs and byte counts add up."""
    rng = np.random.default_rng(N + T + bits)
    xs = [rng.standard_normal(T).astype(np.float32) for _ in range(N)]
    ar, s_ar, r_ar = O.ring([x.copy() for x in xs], codec="bfp", bits=bits)
    rs_out = [np.zeros(T, np.float32) for _ in range(N)]
    rs, s_rs, r_rs = O.ring([x.copy() for x in xs], codec="bfp", bits=bits,
                            mode="reduce_scatter", outputs=rs_out)
    out, s_ag, r_ag = O.allgather_codec(rs, "f32", "bfp", bits)
    for r in range(N):
        assert np.array_equal(out[r].view(np.uint32), ar[r].view(np.uint32))
    assert list(s_ar) == [a + b for a, b in zip(s_rs, s_ag)]
    assert list(r_ar) == [a + b for a, b in zip(r_rs, r_ag)]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_sparse_allgather_is_an_exact_copy(dt):
    """Sparse codes restore every element, -0.0 included: the buffers equal the
    lossless allgather's, while the bytes are the sparse messages' (fp32
    values and int32 indices, so fewer than fp32 elements would take)."""
    N, T = 4, 4 * 700
    rng = np.random.default_rng(5)
    vals = rng.standard_normal(T).astype(np.float32)
    vals[rng.random(T) < 0.7] = 0.0
    vals[::97] = -0.0
    bufs = [O.from_f32(np.roll(vals, 13 * r), dt) for r in range(N)]
    out, sent, _ = O.allgather_codec([b.copy() for b in bufs], dt, "sparse")
    ref, _, _ = O.allgather([b.copy() for b in bufs], dt)
    for r in range(N):
        assert np.array_equal(out[r].view(np.uint8), ref[r].view(np.uint8))
    n = T // N
    msg = [brute.sparse_roundtrip(list(O.to_f32(bufs[c][c * n:(c + 1) * n], dt)), 0.5)[1]
           for c in range(N)]
    # one message per chunk: 70 % zeros, so each is sparse (8 + 8 nnz bytes)
    assert all(m == 8 + 8 * int(np.count_nonzero(O.to_f32(bufs[c][c * n:(c + 1) * n], dt).view(np.uint32)))
               for c, m in enumerate(msg))
    assert [int(x) for x in sent] == [sum(msg) - msg[(r + 1) % N] for r in range(N)]
    assert all(int(x) < 4 * n * (N - 1) for x in sent)


# Reading AB: the root's BFP codes travel the binomial tree unchanged.

@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("N,root", [(1, 0), (2, 1), (3, 0), (5, 2), (4, 3)])
@pytest.mark.parametrize("T", [1, 37, 64, 130])
def test_broadcast_codec_brute_force(bits, N, root, T):
    rng = np.random.default_rng(N * 7 + root + T)
    xs = [rng.standard_normal(T).astype(np.float32) for _ in range(N)]
    out, sent, recv = O.broadcast_codec([x.copy() for x in xs], "f32", root, bits)
    ref, bs, br = brute.broadcast_codec([list(x) for x in xs], root, bits)
    for r in range(N):
        assert np.array_equal(out[r].view(np.uint32), np.array(ref[r], np.float32).view(np.uint32))
    assert list(sent) == bs and list(recv) == br


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_broadcast_codec_is_the_codec_round_trip_everywhere(bits, dt):
    """Every buffer, the root's included, holds the standalone codec's round
    trip of the root's buffer in its dtype; the root sends ceil(log2 N)
    messages of the codec's size, every other rank receives one."""
    N, T, root = 8, 1000, 3
    rng = np.random.default_rng(bits)
    bufs = [O.from_f32((rng.standard_normal(T) * 1e-3).astype(np.float32), dt) for _ in range(N)]
    exps, mants = O.bfp_encode(O.to_f32(bufs[root], dt), bits)
    want = O.from_f32(O.bfp_decode(exps, mants, T, bits), dt)
    out, sent, recv = O.broadcast_codec([b.copy() for b in bufs], dt, root, bits)
    msg = O.bfp_bytes(T, bits)
    for r in range(N):
        assert np.array_equal(out[r], want)
    assert int(sent[root]) == 3 * msg and int(sum(sent)) == (N - 1) * msg
    assert [int(x) for x in recv] == [0 if r == root else msg for r in range(N)]


# Reading F4op: the statistics of what each operation encodes.

@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_codec_stats_per_operation(dt):
    """The allgather counts chunk r of buffer r alone, the broadcast the
    root's buffer with blocks from its start: each equals the statistics of
    those elements as a one-rank problem; the allreduce's are the sum over
    every (buffer, chunk)."""
    N, T, root = 5, 5 * 300 + 77, 2
    rng = np.random.default_rng(len(dt))
    bufs = []
    for r in range(N):
        x = (rng.standard_normal(T) * 10.0 ** rng.integers(-4, 2, T)).astype(np.float32)
        x[rng.random(T) < 0.3] = 0.0
        bufs.append(O.from_f32(x, dt))
    n = -(-T // N)
    own = [bufs[r][min(r * n, T):min((r + 1) * n, T)] for r in range(N)]
    want_ag = sum(O.codec_stats([np.ascontiguousarray(o)], dt) for o in own)
    assert list(O.codec_stats_op(bufs, dt, "allgather")) == list(want_ag)
    assert list(O.codec_stats_op(bufs, dt, "broadcast", root)) == list(O.codec_stats([bufs[root]], dt))
    assert list(O.codec_stats_op(bufs, dt, "allreduce")) == list(O.codec_stats(bufs, dt))
    # the allreduce counts every buffer over every chunk: N times T elements
    assert int(O.codec_stats_op(bufs, dt, "allreduce")[0]) == N * T


def test_codec_stats_per_operation_brute_force():
    N, T, root = 3, 40, 1
    rng = np.random.default_rng(2)
    xs = [(rng.standard_normal(T) * (rng.random(T) < 0.6)).astype(np.float32) for _ in range(N)]
    n = -(-T // N)
    ag = [0, 0, 0, 0]
    for r in range(N):
        piece = list(xs[r][min(r * n, T):min((r + 1) * n, T)])
        ag = [a + b for a, b in zip(ag, brute.codec_stats([piece]))]
    assert list(O.codec_stats_op([x.copy() for x in xs], "f32", "allgather")) == ag
    assert list(O.codec_stats_op([x.copy() for x in xs], "f32", "broadcast", root)) == \
        brute.codec_stats([list(xs[root])])


# --------------------------------------------------------------- broadcast / tree

@pytest.mark.parametrize("N,root", [(N, root) for N in (1, 2, 3, 4, 5, 8, 13)
                                     for root in (0, 1, 4) if root < N])
def test_broadcast(N, root):
    T = 37
    bufs = rand_ranks(N, T, 20 + N)
    src = bufs[root].copy()
    out, sent, recv = O.broadcast(bufs, "f32", root)
    for r in range(N):
        assert np.array_equal(bits32(out[r]), bits32(src))
    # every non-root rank receives the buffer exactly once (T bytes per rank)
    for r in range(N):
        assert recv[r] == (0 if r == root else 4 * T)
    L = brute.ceil_log2(N)
    if N == 1 << L:
        assert sent[root] == 4 * T * L
    assert sum(sent) == 4 * T * (N - 1)


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8, 16])
def test_tree_allreduce(N):
    T = 64
    bufs = rand_ranks(N, T, 40 + N)
    ref_in = [list(b) for b in bufs]
    X = np.stack(bufs).astype(np.float64)
    out, sent, recv = O.tree_allreduce([b.copy() for b in bufs])
    for r in range(1, N):
        assert np.array_equal(bits32(out[r]), bits32(out[0]))
    for i in range(T):
        exact = math.fsum(X[:, i])
        assert abs(float(out[0][i]) - exact) <= (N - 1) * U * math.fsum(np.abs(X[:, i])) * (1 + 1e-6)
    ref, bs, br = brute.tree_allreduce(ref_in)
    assert np.array_equal(bits32(out[0]), bits32(np.array(ref[0], np.float32)))
    assert list(sent) == bs and list(recv) == br
    L = brute.ceil_log2(N)
    assert recv[0] == 4 * T * L  # the root receives once per level


def test_tree_N4_binomial_order():
    """N = 4: (x0 + x1) + (x2 + x3), float32 adds in that order."""
    xs = rand_ranks(4, 256, 50)
    out, _, _ = O.tree_allreduce([x.copy() for x in xs])
    ref = ((xs[0] + xs[1]).astype(np.float32) + (xs[2] + xs[3]).astype(np.float32)).astype(np.float32)
    assert np.array_equal(bits32(out[3]), bits32(ref))


# --------------------------------------------------------------- BFP codec

def load_bfp_golden():
    cases = []
    with open(os.path.join(GOLDEN, "bfp_closed_form.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            bits, e, xs, codes = [p.strip() for p in line.split("|")]
            cases.append((int(bits), int(e), [float.fromhex(v) for v in xs.split(",")],
                          [int(c) for c in codes.split(",")]))
    return cases


@pytest.mark.parametrize("case", load_bfp_golden())
def test_bfp_golden_codes(case):
    bits, e, xs, codes = case
    x = np.array(xs, np.float32)
    assert O.bfp_block_exponent(x) == e
    exps, mants = O.bfp_encode(x, bits)
    assert int(exps[0]) == e
    if bits == 8:
        got = list(mants.view(np.int8))
    else:
        got = [int((mants[i // 2] >> (4 * (i % 2))) & 0xF) for i in range(len(xs))]
        got = [g - 16 if g >= 8 else g for g in got]
    assert got == codes
    dec = O.bfp_decode(exps, mants, len(xs), bits)
    for m, d in zip(codes, dec):
        assert d == np.float32(math.ldexp(m, e - (bits - 2)))
    # the per-element helpers give the same codes and values one at a time
    for v, m in zip(xs, codes):
        assert O.bfp_code(np.float32(v), e, bits) == m
        assert O.bfp_value(m, e, bits) == math.ldexp(m, e - (bits - 2))


def test_bfp4_nibble_packing_by_hand():
    # codes 4,2 | 0,2 | -4,7 | 1 -> bytes 0x24, 0x20, 0x7C, 0x01 (element 2j low nibble)
    x = np.array([1.0, 0.5, 0.0, 0.5, -1.0, 1.75, 0.25], np.float32)  # max 1.75 -> e=0, step 1/4
    exps, mants = O.bfp_encode(x, 4)
    assert int(exps[0]) == 0 and list(mants) == [0x24, 0x20, 0x7C, 0x01]


@pytest.mark.parametrize("bits", [8, 4])
def test_bfp_exponent_is_floor_log2(bits):
    rng = np.random.default_rng(60 + bits)
    for _ in range(500):
        blk = (rng.standard_normal(128) * 10.0 ** rng.uniform(-30, 30)).astype(np.float32)
        e = O.bfp_block_exponent(blk)
        amax = float(np.abs(blk).max())
        assert 2.0 ** e <= amax < 2.0 ** (e + 1)


@pytest.mark.parametrize("bits", [8, 4])
def test_bfp_error_bound(bits):
    """Unclamped elements: |x - dec| <= 2^(e-q-1) (for 8 bits: 2^(e-7), the
    bound the spec states); clamped ones: |x - dec| < 2^(e-q)."""
    rng = np.random.default_rng(70 + bits)
    q, M = bits - 2, 2 ** (bits - 1) - 1
    x = (rng.standard_normal(128 * 400) * 10.0 ** rng.uniform(-20, 20, 128 * 400)).astype(np.float32)
    exps, mants = O.bfp_encode(x, bits)
    dec = O.bfp_decode(exps, mants, x.size, bits).astype(np.float64)
    e = np.repeat(exps.astype(np.int64), 128)[: x.size]
    err = np.abs(x.astype(np.float64) - dec)
    scaled = np.abs(x.astype(np.float64)) * np.exp2((q - e).astype(np.float64))
    clamped = scaled > M + 0.5
    assert (err[~clamped] <= np.exp2(e[~clamped] - q - 1.0)).all()
    assert (err[clamped] < np.exp2(e[clamped] - q * 1.0)).all()
    assert clamped.any() or bits == 8


@pytest.mark.parametrize("bits", [8, 4])
def test_bfp_brute_force_and_idempotent(bits):
    rng = np.random.default_rng(80 + bits)
    x = (rng.standard_normal(300) * 1e-3).astype(np.float32)
    exps, mants = O.bfp_encode(x, bits)
    dec = O.bfp_decode(exps, mants, x.size, bits)
    ref, nbytes = brute.bfp_roundtrip(list(x), bits)
    assert np.array_equal(bits32(dec), bits32(np.array(ref, np.float32)))
    assert nbytes == exps.size + mants.size == O.bfp_bytes(x.size, bits)
    e2, m2 = O.bfp_encode(dec, bits)  # decode(encode) is a fixed point
    assert np.array_equal(e2, exps) and np.array_equal(m2, mants)


def test_bfp_decode_accumulate():
    x = np.array([1.0, -0.5, 0.25], np.float32)
    exps, mants = O.bfp_encode(x, 8)
    acc = np.array([1.0, 1.0, 1.0], np.float32)
    O.bfp_decode(exps, mants, 3, 8, out=acc, accumulate=True)
    assert list(acc) == [2.0, 0.5, 1.25]


# --------------------------------------------------------------- sparse codec

def test_sparse_roundtrip_exact_and_indices():
    rng = np.random.default_rng(90)
    x = rng.standard_normal(1000).astype(np.float32)
    x[rng.random(1000) < 0.7] = 0.0
    x[5] = -0.0  # kept: only +0.0 counts as zero
    hdr, vals, idx = O.sparse_encode(x)
    nz = bits32(x) != 0
    assert hdr[0] == 1 and hdr[1] == nz.sum()
    assert np.array_equal(idx, np.nonzero(nz)[0]) and 5 in idx
    assert (np.diff(idx) > 0).all()
    back = O.sparse_decode(hdr, vals, idx, x.size)
    assert np.array_equal(bits32(back), bits32(x))


@pytest.mark.parametrize("nnz,expect_sparse", [(49, True), (50, False), (51, False), (0, True)])
def test_sparse_threshold_boundary(nnz, expect_sparse):
    """threshold 0.5, n = 100: sparse iff sparsity (n-nnz)/n > 0.5 strictly;
    the tie (density exactly 0.5) stays dense."""
    x = np.zeros(100, np.float32)
    x[:nnz] = 1.5
    hdr, vals, idx = O.sparse_encode(x, threshold=0.5)
    assert bool(hdr[0]) == expect_sparse and hdr[1] == nnz
    assert O.sparse_is_sparse(nnz, 100, 0.5) == expect_sparse
    back = O.sparse_decode(hdr, vals, idx, 100)
    assert np.array_equal(bits32(back), bits32(x))


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_sparse_keeps_input_dtype(dt):
    x32 = np.array([0, 0, 1.5, 0, -2.25, 0, 0, 0, 0, 3.0], np.float32)
    x = O.from_f32(x32, dt)
    hdr, vals, idx = O.sparse_encode(x, dt)
    assert hdr[0] == 1 and list(idx) == [2, 4, 9] and vals.dtype == O.NP_DTYPES[dt]
    acc = np.ones(10, np.float32)
    O.sparse_decode(hdr, vals, idx, 10, dt, acc=acc, accumulate=True)
    assert list(acc) == [1, 1, 2.5, 1, -1.25, 1, 1, 1, 1, 4.0]


def test_sparse_decode_overwrites_or_adds_by_hand():
    """Without accumulation the restored message replaces acc (+0.0 where a
    sparse message lists nothing); with it every carried value is added: a
    sparse message adds at its listed positions only, a dense one everywhere
    (the values below are exact in fp32, so the sums are by hand)."""
    garbage = np.full(6, 7.0, np.float32)
    # sparse: two values listed at 1 and 4
    hdr = np.array([1, 2], np.uint32)
    vals = np.array([0.5, -3.0], np.float32)
    idx = np.array([1, 4], np.int32)
    got = O.sparse_decode(hdr, vals, idx, 6, acc=garbage.copy())
    assert list(got) == [0.0, 0.5, 0.0, 0.0, -3.0, 0.0]
    got = O.sparse_decode(hdr, vals, idx, 6, acc=garbage.copy(), accumulate=True)
    assert list(got) == [7.0, 7.5, 7.0, 7.0, 4.0, 7.0]
    # dense: all six values
    hdr = np.array([0, 6], np.uint32)
    vals = np.array([1.0, 0.0, -2.0, 0.25, 0.0, 3.0], np.float32)
    got = O.sparse_decode(hdr, vals, np.zeros(0, np.int32), 6, acc=garbage.copy())
    assert list(got) == [1.0, 0.0, -2.0, 0.25, 0.0, 3.0]
    got = O.sparse_decode(hdr, vals, np.zeros(0, np.int32), 6, acc=garbage.copy(), accumulate=True)
    assert list(got) == [8.0, 7.0, 5.0, 7.25, 7.0, 10.0]


# --------------------------------------------------------------- diff

def test_diff_encode():
    rng = np.random.default_rng(95)
    prev = rng.standard_normal(5000).astype(np.float32)
    cur = (prev * rng.uniform(0.6, 1.9, 5000)).astype(np.float32)  # within 2x: Sterbenz
    d = O.diff_encode(cur, prev)
    assert np.array_equal(bits32(d), bits32((cur - prev).astype(np.float32)))
    exact = cur.astype(np.float64) - prev.astype(np.float64)
    same_sign = np.sign(cur) == np.sign(prev)
    assert (d[same_sign].astype(np.float64) == exact[same_sign]).all()


# --------------------------------------------------------------- compressed ring

@pytest.mark.parametrize("codec,bits,sl", [("bfp", 8, None), ("bfp", 4, None), ("sparse", 8, None),
                                           ("sparse", 8, 8)])
@pytest.mark.parametrize("N,T", [(1, 10), (2, 64), (3, 50), (4, 64), (4, 17)])
def test_compressed_ring_brute_force(codec, bits, sl, N, T):
    rng = np.random.default_rng(N * 1000 + T + bits)
    xs = [(rng.standard_normal(T) * 1e-3).astype(np.float32) for _ in range(N)]
    if codec == "sparse":
        for x in xs:
            x[rng.random(T) < 0.6] = 0.0
    outs, sent, recv = O.ring(xs, codec=codec, bits=bits, slice=sl)
    ref, bs, br = brute.ring([list(x) for x in xs], codec=codec, bits=bits, slice_len=sl)
    for r in range(N):
        assert np.array_equal(bits32(outs[r]), bits32(np.array(ref[r], np.float32)))
    assert list(sent) == bs and list(recv) == br
    for r in range(1, N):
        assert np.array_equal(bits32(outs[r]), bits32(outs[0]))


@pytest.mark.parametrize("N", [3, 4])
def test_diff_average_base_brute_force(N):
    T = 40
    rng = np.random.default_rng(123)
    prev = [(rng.standard_normal(T) * 1e-4).astype(np.float32) for _ in range(N)]
    cur = [(p + (rng.standard_normal(T) * 1e-5).astype(np.float32)).astype(np.float32) for p in prev]
    base = (rng.standard_normal(T) * 1e-4).astype(np.float32)
    outs, sent, _ = O.ring(cur, codec="bfp", bits=4, diff_prev=prev, diff_base=base, average=True)
    ref, bs, _ = brute.ring([list(c) for c in cur], codec="bfp", bits=4,
                            diff_prev=[list(p) for p in prev], diff_base=list(base), average=True)
    assert np.array_equal(bits32(outs[2]), bits32(np.array(ref[2], np.float32)))
    assert list(sent) == bs


def test_bfp_ring_byte_counter_closed_form():
    """Every message of a BFP ring is ceil(len/128) exponent bytes plus the
    mantissas (len bytes at 8 bits, ceil(len/2) at 4 bits)."""
    N, T = 8, 8 * 1000
    xs = rand_ranks(N, T, 130, scale=1e-3)
    for bits, per in ((8, 8 + 1000), (4, 8 + 500)):
        _, sent, recv = O.ring(xs, codec="bfp", bits=bits)
        assert all(int(s) == 2 * (N - 1) * per for s in sent)


def test_bfp_ring_error_within_per_hop_bounds():
    """|out - exact sum| <= sum over the N hops that quantise (N-1 partial
    sums and the final sum) of the half-step 2^(e-7) at that hop's block
    exponent, plus the float32 add roundings; exponents are bounded by the
    largest partial-sum magnitude."""
    N, T = 8, 128 * 6
    xs = rand_ranks(N, T, 140, scale=1e-3)
    outs, _, _ = O.ring(xs, codec="bfp", bits=8)
    X = np.stack(xs).astype(np.float64)
    n = T // N
    for c in range(N):
        for b in range(0, n, 128):
            sl = slice(c * n + b, c * n + min(b + 128, n))
            partial_max = 0.0
            acc = np.zeros(sl.stop - sl.start)
            for k in range(1, N + 1):
                acc = acc + X[(c + k) % N, sl]
                partial_max = max(partial_max, float(np.abs(acc).max()))
            e_max = math.floor(math.log2(partial_max * 1.01))
            bound = N * 2.0 ** (e_max - 7) + N * U * float(np.abs(X[:, sl]).sum(0).max()) * 2
            err = np.abs(outs[0][sl].astype(np.float64) - X[:, sl].sum(0))
            assert err.max() <= bound


def _sparse_inputs(N, T, seed, zero_p=0.6, minus_zero_every=0):
    rng = np.random.default_rng(seed)
    xs = []
    for _ in range(N):
        x = (rng.standard_normal(T) * 0.02).astype(np.float32)
        x[rng.random(T) < zero_p] = 0.0
        if minus_zero_every:
            x[rng.integers(0, minus_zero_every):: minus_zero_every] = -0.0
        xs.append(x)
    return xs


@pytest.mark.parametrize("sl", [None, 256, 7])
def test_sparse_ring_equals_lossless_ring(sl):
    """The sparse codec is lossless and the receiver adds the whole restored
    message (S4), so the sparse ring's result is the lossless ring's bit for
    bit, -0.0 inputs included, in either message granularity."""
    N, T = 5, 3000
    xs = _sparse_inputs(N, T, 150, minus_zero_every=37)
    sp, ssent, _ = O.ring(xs, codec="sparse", slice=sl)
    ls, lsent, _ = O.ring(xs)
    for r in range(N):
        assert np.array_equal(bits32(sp[r]), bits32(ls[r]))
    _, bs, _ = brute.ring([list(x) for x in xs], codec="sparse", slice_len=sl)
    assert list(ssent) == bs


def test_sparse_ring_adds_the_restored_message():
    """S4: an omitted position is restored as +0.0 and added, so a -0.0 own
    input meets +0.0 and gives +0.0, as in the lossless ring."""
    # N = 2, T = 4: rank 1 owns chunk 1 = [2, 4) and receives it from rank 0,
    # whose values there are +0.0, so the sparse message lists nothing
    xs = [np.zeros(4, np.float32), np.array([0, 0, -0.0, 0], np.float32)]
    for sl in (None, 4):
        sp, sent, _ = O.ring(xs, codec="sparse", slice=sl, mode="reduce_scatter")
        assert struct.pack("<f", float(sp[1][2])) == struct.pack("<f", 0.0)
        # each rank sends one all-zero chunk of 2: a sparse header, no pairs
        assert list(sent) == [8, 8]
        ref, _, _ = brute.ring([list(x) for x in xs], codec="sparse", slice_len=sl,
                               mode="reduce_scatter")
        assert struct.pack("<f", float(ref[1][2])) == struct.pack("<f", 0.0)


def _per_chunk_message_bytes(xs, thr=0.5):
    """bytes[h][c] of the message of chunk c at hop h (h = 1..N-1 the
    reduce-scatter partials, h = N the owner's full sum), with numpy: the
    partial of hop h is x_{c+1} + ... + x_{c+h}, added one float32 add at a
    time in ring order; a message is 8 + 8 nnz bytes when nnz < (1 - thr)
    len, else 8 + 4 len; an empty chunk sends nothing."""
    N, T = len(xs), xs[0].size
    n = -(-T // N)
    out = np.zeros((N + 1, N), np.int64)
    for c in range(N):
        lo, hi = min(c * n, T), min((c + 1) * n, T)
        if hi == lo:
            continue
        p = None
        for h in range(1, N + 1):
            x = xs[(c + h) % N][lo:hi]
            p = x.copy() if p is None else (p + x).astype(np.float32)
            nnz = int(np.count_nonzero(p.view(np.uint32)))
            out[h][c] = 8 + 8 * nnz if nnz < (1.0 - thr) * (hi - lo) else 8 + 4 * (hi - lo)
    return out


@pytest.mark.parametrize("N,T,zero_p", [(4, 4 * 500, 0.6), (5, 3001, 0.75), (6, 6 * 90, 0.9),
                                        (3, 2, 0.5), (8, 13, 0.3)])
def test_sparse_ring_per_chunk_bytes_closed_form(N, T, zero_p):
    """One message per chunk and hop (reading S3): reduce-scatter step s,
    rank r sends chunk (r - s) mod N's hop-s partial; allgather step s, rank r
    forwards the owner's message of chunk (r - s + 1) mod N."""
    xs = _sparse_inputs(N, T, 160 + N, zero_p=zero_p)
    _, sent, recv = O.ring(xs, codec="sparse")
    B = _per_chunk_message_bytes(xs)
    want = [sum(B[s][(r - s) % N] for s in range(1, N)) +
            sum(B[N][(r - s + 1) % N] for s in range(1, N)) for r in range(N)]
    assert [int(v) for v in sent] == want
    assert [int(v) for v in recv] == [want[(r - 1) % N] for r in range(N)]
    _, rs_sent, _ = O.ring(xs, codec="sparse", mode="reduce_scatter")
    assert [int(v) for v in rs_sent] == [sum(B[s][(r - s) % N] for s in range(1, N))
                                         for r in range(N)]


def test_sparse_ring_per_chunk_decision_at_the_tie():
    """Chunk length 8, threshold 0.5: a hop whose partial has 4 nonzeros is
    dense (8 + 32 bytes), 3 nonzeros sparse (8 + 24); per-slice messages of 4
    elements decide each half on its own."""
    N, T = 2, 16
    a = np.zeros(T, np.float32)
    b = np.zeros(T, np.float32)
    a[8:12] = [1, 2, 3, 4]      # chunk 1 of rank 0, sent at step 1: 4 of 8 nonzero
    b[0:3] = [5, 6, 7]          # chunk 0 of rank 1, sent at step 1: 3 of 8 nonzero
    _, sent, _ = O.ring([a, b], codec="sparse", mode="reduce_scatter")
    assert [int(v) for v in sent] == [8 + 4 * 8, 8 + 8 * 3]
    _, sent4, _ = O.ring([a, b], codec="sparse", slice=4, mode="reduce_scatter")
    # rank 0: [1 2 3 4] dense (8 + 16) and [0 0 0 0] sparse (8); rank 1:
    # [5 6 7 0] dense (8 + 16) and [0 0 0 0] sparse (8)
    assert [int(v) for v in sent4] == [8 + 16 + 8, 8 + 16 + 8]
# --------------------------------------------------------------- error feedback

@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("mode", ["allreduce", "reduce_scatter"])
@pytest.mark.parametrize("N,T", [(1, 10), (2, 64), (3, 50), (4, 17)])
def test_error_feedback_brute_force(bits, mode, N, T):
    """Two rounds with carried residuals against the independent brute force:
    outputs, byte counts and every residual bit for bit."""
    rng = np.random.default_rng(N * 100 + T + bits)
    res_o = [(rng.standard_normal(T) * 1e-5).astype(np.float32) for _ in range(N)]
    res_b = [list(r.copy()) for r in res_o]
    for rnd in range(2):
        xs = [(rng.standard_normal(T) * 1e-3).astype(np.float32) for _ in range(N)]
        outs = [np.zeros(T, np.float32) for _ in range(N)]
        outs, sent, recv = O.ring(xs, codec="bfp", bits=bits, mode=mode, outputs=outs,
                                  residual=res_o)
        ref, bs, br = brute.ring([list(x) for x in xs], codec="bfp", bits=bits, mode=mode,
                                 residual=res_b)
        for r in range(N):
            want = np.array([0.0 if v is None else v for v in ref[r]], np.float32)
            assert np.array_equal(bits32(outs[r]), bits32(want)), (rnd, r)
            assert np.array_equal(bits32(res_o[r]), bits32(np.array(res_b[r], np.float32))), (rnd, r)
        assert list(sent) == bs and list(recv) == br


def test_error_feedback_zero_residual_first_round_is_the_plain_ring():
    rng = np.random.default_rng(4)
    N, T = 4, 700
    xs = [(rng.standard_normal(T) * 1e-3).astype(np.float32) for _ in range(N)]
    res = [np.zeros(T, np.float32) for _ in range(N)]
    with_ef = O.ring(xs, codec="bfp", bits=4, residual=res)
    plain = O.ring(xs, codec="bfp", bits=4)
    for r in range(N):
        assert np.array_equal(bits32(with_ef[0][r]), bits32(plain[0][r]))
    assert any(np.any(e != 0) for e in res)  # BFP4 loses something, so residuals are set


@pytest.mark.parametrize("bits", [4, 8])
def test_error_feedback_conserves_the_total(bits):
    """Over K rounds, everything sent and not yet delivered sits in the
    residuals.  Each chunk's result D = sum_r x_r + sum_r (e_old - e_new), up
    to fp32 rounding of the sums.  So sum_k D_k + sum_r e_r(K) equals
    sum_k sum_r x_{r,k}, and the error of sum_k D_k stays bounded instead of
    growing with K as it does without feedback."""
    rng = np.random.default_rng(11 + bits)
    N, T, K = 4, 1024, 24
    res = [np.zeros(T, np.float32) for _ in range(N)]
    tot_in = np.zeros(T)
    tot_ef = np.zeros(T)
    tot_plain = np.zeros(T)
    mag = 0.0
    for _ in range(K):
        xs = [(rng.standard_normal(T) * 1e-3).astype(np.float32) for _ in range(N)]
        tot_in += np.sum([x.astype(np.float64) for x in xs], axis=0)
        mag += np.sum([np.abs(x.astype(np.float64)) for x in xs], axis=0)
        tot_ef += O.ring(xs, codec="bfp", bits=bits, residual=res)[0][0]
        tot_plain += O.ring(xs, codec="bfp", bits=bits)[0][0]
    left = np.sum([e.astype(np.float64) for e in res], axis=0)
    # fp32 rounding of the adds along the chain: a few ulps of the magnitudes involved
    bound = 4 * N * 2.0 ** -24 * (mag + K * np.max([np.abs(e) for e in res]))
    assert np.all(np.abs(tot_ef + left - tot_in) <= bound + 1e-12)
    drift_ef = np.abs(tot_ef - tot_in).mean()
    drift_plain = np.abs(tot_plain - tot_in).mean()
    assert drift_ef < drift_plain / 2, (drift_ef, drift_plain)


def test_error_feedback_needs_a_lossy_codec():
    xs = [np.ones(16, np.float32)] * 2
    res = [np.zeros(16, np.float32)] * 2
    for codec in ("none", "sparse"):
        with pytest.raises(ValueError):
            O.ring(xs, codec=codec, residual=res)


# --------------------------------------------------------------- codec statistics

def test_codec_stats_closed_form():
    """One block with maximum 1.0 (e = 0): BFP8 rounds |x| <= 2^-7 to code 0
    (1/128 is the tie and goes to even 0; 1/127 does not), BFP4 rounds
    |x| <= 2^-3 to 0.  +0.0 is not counted as nonzero; -0.0 is, and flushes."""
    x = np.array([1.0, 1 / 128, 1 / 127, 0.125, 0.13, 0.0, -0.0], np.float32)
    st = O.codec_stats([x])
    assert list(st) == [7, 6, 4, 2]


def test_codec_stats_blocks_start_at_chunk_starts():
    """Blocks are cut from each ring chunk's start, so the same values give
    different counts for different N when a block straddles a chunk edge."""
    T = 256
    x = np.full(T, 1e-3, np.float32)
    x[0] = 1.0  # a large value only in the first 128 elements of the buffer
    st1 = O.codec_stats([x])  # one chunk: the block of x[0] holds 127 small values
    assert list(st1) == [T, T, 127, 127]
    xs = [x.copy(), x.copy(), x.copy()]
    st3 = O.codec_stats(xs)  # chunks of 86: only x[0]'s block (86 values) sees 1.0
    assert list(st3) == [3 * T, 3 * T, 3 * 85, 3 * 85]


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N,T", [(1, 300), (2, 257), (3, 1000), (5, 64)])
def test_codec_stats_brute_force(dt, N, T):
    rng = np.random.default_rng(N * 31 + T)
    xs = []
    for _ in range(N):
        x = (rng.standard_normal(T) * 10.0 ** rng.integers(-6, 2, T)).astype(np.float32)
        x[rng.random(T) < 0.3] = 0.0
        x[rng.random(T) < 0.02] = -0.0
        xs.append(x)
    if dt != "f32":
        hs = [O.from_f32(x, dt) for x in xs]
        vals = [O.to_f32(h, dt) for h in hs]
    else:
        hs, vals = xs, xs
    st = O.codec_stats(hs, dt)
    assert list(st) == brute.codec_stats([list(v) for v in vals])
