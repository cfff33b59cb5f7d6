"""Pure-Python brute force of the ring collectives and codecs, for tiny inputs.

An independent second implementation used only to pin the C oracle (N <= 4,
T <= 64): plain Python loops, one numpy float32 scalar operation per IEEE
binary32 add, ``math.frexp``/``math.ldexp`` for exponents and exact
power-of-two scaling (in double, where every scaled value here is exact) and
Python's ``round`` (round half to even) for the integer codes.  It shares no
code with the C oracle or with the GPU library.

Schedules (collective ops from scratch lesson, "two-pass ring allreduce"):
reduce-scatter step s = 1..N-1, rank r sends chunk (r-s) mod N to r+1;
allgather step s = 1..N-1, rank r sends chunk (r-s+1) mod N.
"""
from __future__ import annotations

import math
import struct

import numpy as np

F = np.float32


def chunks(T, N):
    n = -(-T // N)
    return [(min(c * n, T), min((c + 1) * n, T)) for c in range(N)]


def nonzero(v) -> bool:
    return struct.pack("<f", float(v)) != b"\x00\x00\x00\x00"


# ---------------------------------------------------------------- codecs

def bfp_exponent(vals) -> int:
    amax = max((abs(float(v)) for v in vals), default=0.0)
    if amax < 2.0 ** -126:
        return -126
    _, E = math.frexp(amax)  # amax = f * 2^E, 0.5 <= f < 1
    return E - 1


def bfp_code(v, e, bits) -> int:
    q, M = bits - 2, 2 ** (bits - 1) - 1
    r = round(math.ldexp(float(v), q - e))  # half to even
    return max(-M, min(M, r))


def bfp_value(m, e, bits):
    return F(math.ldexp(m, e - (bits - 2)))


def bfp_roundtrip(vals, bits):
    """Encode and decode a list of float32 values block by block."""
    out, nbytes = [], 0
    for lo in range(0, len(vals), 128):
        blk = vals[lo:lo + 128]
        e = bfp_exponent(blk)
        out += [bfp_value(bfp_code(v, e, bits), e, bits) for v in blk]
        nbytes += 1
    nbytes += len(vals) if bits == 8 else (len(vals) + 1) // 2
    return out, nbytes


def sparse_roundtrip(vals, threshold, slice_len=None):
    """Returns (restored values, wire bytes) of one chunk's message: one
    message for the whole list (slice_len None) or one per slice_len
    elements.  A sparse message lists (value, index) pairs; the receiver
    puts the values back by index into zeros."""
    out, nbytes = [], 0
    step = slice_len or max(len(vals), 1)
    for lo in range(0, len(vals), step):
        sl = vals[lo:lo + step]
        pairs = [(v, i) for i, v in enumerate(sl) if nonzero(v)]
        if len(pairs) < (1.0 - threshold) * len(sl):
            piece = [F(0.0)] * len(sl)
            for v, i in pairs:
                piece[i] = v
            out += piece
            nbytes += 8 + 8 * len(pairs)
        else:
            out += list(sl)
            nbytes += 8 + 4 * len(sl)
    return out, nbytes


# ---------------------------------------------------------------- ring

def ring(xs, codec="none", bits=8, threshold=0.5, slice_len=None, mode="allreduce",
         diff_prev=None, diff_base=None, average=False, residual=None):
    """xs: list of N lists of float32 scalars.  Returns (results, sent, recv)
    where results[r] is a list with None at chunks rank r does not produce.
    residual: N lists of float32 error-feedback residuals, updated in place
    (a rank encodes u = v + e and keeps e = u - decoded)."""
    N, T = len(xs), len(xs[0])
    ch = chunks(T, N)
    if diff_prev is not None:
        local = [[F(xs[r][i] - diff_prev[r][i]) for i in range(T)] for r in range(N)]
    else:
        local = [[F(v) for v in x] for x in xs]
    sent, recv = [0] * N, [0] * N

    def encode(vals):
        """(decoded values, wire bytes) of one message"""
        if codec == "none":
            return list(vals), 4 * len(vals)
        if codec == "bfp":
            return bfp_roundtrip(vals, bits)
        return sparse_roundtrip(vals, threshold, slice_len)

    def encode_at(r, lo, hi, vals):
        if residual is None:
            return encode(vals)
        u = [F(v + residual[r][lo + k]) for k, v in enumerate(vals)]
        msg = encode(u)
        for k in range(hi - lo):
            residual[r][lo + k] = F(u[k] - msg[0][k])
        return msg

    for s in range(1, N):
        inbox = [None] * N
        for r in range(N):
            lo, hi = ch[(r - s) % N]
            inbox[(r + 1) % N] = encode_at(r, lo, hi, local[r][lo:hi])
            sent[r] += inbox[(r + 1) % N][1]
            recv[(r + 1) % N] += inbox[(r + 1) % N][1]
        for r in range(N):
            lo, hi = ch[(r - s - 1) % N]
            vals, _ = inbox[r]
            for i in range(lo, hi):  # decompressed message added element by element
                local[r][i] = F(local[r][i] + vals[i - lo])

    res = [[None] * T for _ in range(N)]
    held = [None] * N
    for r in range(N):
        lo, hi = ch[r]
        if mode == "reduce_scatter" or codec == "none":
            for i in range(lo, hi):
                res[r][i] = local[r][i]
        if mode == "allreduce":
            held[r] = encode_at(r, lo, hi, local[r][lo:hi])
            if codec != "none":
                for i in range(lo, hi):
                    res[r][i] = held[r][0][i - lo]
    if mode == "allreduce":
        for s in range(1, N):
            inbox = [None] * N
            for r in range(N):
                inbox[(r + 1) % N] = held[r]
                sent[r] += held[r][1]
                recv[(r + 1) % N] += held[r][1]
            for r in range(N):
                lo, hi = ch[(r - s) % N]
                vals, _ = inbox[r]
                for i in range(lo, hi):
                    res[r][i] = vals[i - lo]
                held[r] = inbox[r]
    for r in range(N):
        for i in range(T):
            if res[r][i] is None:
                continue
            w = res[r][i]
            if average:
                w = F(w / F(N))
            if diff_base is not None:
                w = F(diff_base[i] + w)
            res[r][i] = w
    return res, sent, recv


# ---------------------------------------------------------------- tree / bcast / allgather

def ceil_log2(N):
    L = 0
    while (1 << L) < N:
        L += 1
    return L


def broadcast(bufs, root, elem_bytes):
    N, T = len(bufs), len(bufs[0])
    bufs = [list(b) for b in bufs]
    sent, recv = [0] * N, [0] * N
    for k in range(ceil_log2(N)):
        for q in range(1 << k):
            if q + (1 << k) < N:
                src, dst = (q + root) % N, (q + (1 << k) + root) % N
                bufs[dst] = list(bufs[src])
                sent[src] += T * elem_bytes
                recv[dst] += T * elem_bytes
    return bufs, sent, recv


def broadcast_codec(bufs, root, bits):
    """BFP-compressed broadcast of N lists of float32 scalars: the root's
    buffer is encoded once (blocks from its start), every tree edge carries
    the codes, every rank holds the decoded buffer."""
    N, T = len(bufs), len(bufs[0])
    out, nb = bfp_roundtrip([F(v) for v in bufs[root]], bits)
    sent, recv = [0] * N, [0] * N
    for k in range(ceil_log2(N)):
        for q in range(1 << k):
            if q + (1 << k) < N:
                sent[(q + root) % N] += nb
                recv[(q + (1 << k) + root) % N] += nb
    return [list(out) for _ in range(N)], sent, recv


def tree_allreduce(bufs):
    N, T = len(bufs), len(bufs[0])
    acc = [[F(v) for v in b] for b in bufs]
    sent, recv = [0] * N, [0] * N
    for k in range(ceil_log2(N)):
        st = 1 << k
        for r in range(0, N, 2 * st):
            if r + st < N:
                acc[r] = [F(a + b) for a, b in zip(acc[r], acc[r + st])]
                sent[r + st] += 4 * T
                recv[r] += 4 * T
    out, s2, r2 = broadcast(acc, 0, 4)
    return out, [a + b for a, b in zip(sent, s2)], [a + b for a, b in zip(recv, r2)]


def allgather(bufs, elem_bytes):
    N, T = len(bufs), len(bufs[0])
    ch = chunks(T, N)
    bufs = [list(b) for b in bufs]
    sent, recv = [0] * N, [0] * N
    for s in range(1, N):
        msgs = [None] * N
        for r in range(N):
            lo, hi = ch[(r - s + 1) % N]
            msgs[(r + 1) % N] = bufs[r][lo:hi]
            sent[r] += (hi - lo) * elem_bytes
            recv[(r + 1) % N] += (hi - lo) * elem_bytes
        for r in range(N):
            lo, hi = ch[(r - s) % N]
            bufs[r][lo:hi] = msgs[r]
    return bufs, sent, recv


def allgather_codec(xs, codec="bfp", bits=8, threshold=0.5, slice_len=None):
    """Compressed allgather of N lists of float32 scalars: the owner of chunk
    c encodes its own elements once, the codes travel the ring unchanged, and
    every rank (owner included) holds the decoded chunk.  Returns (results,
    sent, recv)."""
    N, T = len(xs), len(xs[0])
    ch = chunks(T, N)
    held = []
    for r in range(N):
        lo, hi = ch[r]
        vals = [F(v) for v in xs[r][lo:hi]]
        if codec == "bfp":
            out, nb = bfp_roundtrip(vals, bits)
        else:
            out, nb = sparse_roundtrip(vals, threshold, slice_len)
        held.append((out, nb))
    res = [[F(v) for v in x] for x in xs]
    for r in range(N):
        lo, hi = ch[r]
        res[r][lo:hi] = held[r][0]
    sent, recv = [0] * N, [0] * N
    cur = held
    for s in range(1, N):
        nxt = [None] * N
        for r in range(N):
            nxt[(r + 1) % N] = cur[r]
            sent[r] += cur[r][1]
            recv[(r + 1) % N] += cur[r][1]
        for r in range(N):
            lo, hi = ch[(r - s) % N]
            res[r][lo:hi] = nxt[r][0]
        cur = nxt
    return res, sent, recv


# ---------------------------------------------------------------- codec statistics

def codec_stats(xs):
    """[elements, nonzero, flushed by BFP4, flushed by BFP8] over N lists of
    float32 scalars: 128-element blocks from each ring chunk's start; a
    nonzero element (bits not +0.0) is flushed when its code rounds to 0,
    i.e. when |x| * 2^(q - e) <= 1/2."""
    N, T = len(xs), len(xs[0])
    st = [0, 0, 0, 0]
    for x in xs:
        for lo, hi in chunks(T, N):
            for b in range(lo, hi, 128):
                blk = [F(v) for v in x[b:min(b + 128, hi)]]
                e = bfp_exponent(blk)
                for v in blk:
                    st[0] += 1
                    if not nonzero(v):
                        continue
                    st[1] += 1
                    for k, bits in ((2, 4), (3, 8)):
                        if bfp_code(v, e, bits) == 0:
                            st[k] += 1
    return st
