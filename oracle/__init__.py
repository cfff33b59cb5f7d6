"""CPU oracle for the chunked ring allreduce with compression codecs.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg (``bench.py --impl reference`` and its
``cpu_baseline`` field) are the only code that may import this package.  The
GPU library (``ring_allreduce_compressed_gb300``) never imports it and it never
imports the GPU library: the two share no code, headers, tables or constants.

The arithmetic lives in ``oracle.c`` (plain C, single-threaded, IEEE binary32
without FMA contraction); this module only compiles it with gcc, loads it with
ctypes and marshals numpy arrays.  Every function cites the page and section it
follows in ``oracle.c``.

Dtype tags: ``"f32"`` (numpy float32), ``"f16"`` (numpy float16) and ``"bf16"``
(numpy uint16 holding bfloat16 bit patterns; numpy has no bfloat16).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
# A test that plants a mistake in the oracle compiles a mutated copy of
# oracle.c elsewhere and points this variable at it.
_LIB_OVERRIDE = os.environ.get("RRA_ORACLE_LIB")
_lock = threading.Lock()
_lib = None

DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
NP_DTYPES = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}
CODECS = {"none": 0, "bfp": 1, "sparse": 2}
BFP_BLOCK = 128
# Sparse codec message granularity (reading S3).  slice=None (the default):
# one message per ring chunk and hop, its format chosen from the nonzero count
# of the whole chunk.  slice=RING_SLICE: the per-slice option, one message per
# 256 elements, each with its own header and its own sparse/dense decision.
RING_SLICE = 256


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, no fast-math)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            if _LIB_OVERRIDE:
                L = C.CDLL(_LIB_OVERRIDE)
            else:
                build()
                L = C.CDLL(_LIB)
            vp, sz, i32, u64p = C.c_void_p, C.c_size_t, C.c_int, C.POINTER(C.c_uint64)
            L.oracle_ring.argtypes = [i32, i32, sz, vp, i32, vp, i32, i32, i32, C.c_double, sz,
                                      vp, vp, i32, u64p, u64p]
            L.oracle_ring.restype = i32
            L.oracle_ring_ef.argtypes = [i32, i32, sz, vp, i32, vp, i32, i32, i32, C.c_double,
                                         sz, vp, vp, i32, vp, u64p, u64p]
            L.oracle_ring_ef.restype = i32
            L.oracle_allgather.argtypes = [i32, sz, vp, i32, u64p, u64p]
            L.oracle_allgather_codec.argtypes = [i32, sz, vp, i32, i32, i32, C.c_double, sz,
                                                 u64p, u64p]
            L.oracle_allgather_codec.restype = i32
            L.oracle_codec_stats.argtypes = [i32, sz, vp, i32, u64p]
            L.oracle_codec_stats.restype = i32
            L.oracle_codec_stats_op.argtypes = [i32, i32, i32, sz, vp, i32, u64p]
            L.oracle_codec_stats_op.restype = i32
            L.oracle_broadcast.argtypes = [i32, sz, vp, i32, i32, u64p, u64p]
            L.oracle_broadcast_codec.argtypes = [i32, sz, vp, i32, i32, i32, u64p, u64p]
            L.oracle_broadcast_codec.restype = i32
            L.oracle_tree_allreduce.argtypes = [i32, sz, vp, u64p, u64p]
            for f in (L.oracle_allgather, L.oracle_broadcast, L.oracle_tree_allreduce):
                f.restype = i32
            L.oracle_bfp_encode.argtypes = [vp, sz, i32, vp, vp]
            L.oracle_bfp_decode.argtypes = [vp, vp, sz, i32, vp, i32]
            L.oracle_bfp_block_exponent.argtypes = [vp, sz]
            L.oracle_bfp_block_exponent.restype = i32
            L.oracle_bfp_code.argtypes = [C.c_float, i32, i32]
            L.oracle_bfp_code.restype = i32
            L.oracle_bfp_value.argtypes = [i32, i32, i32]
            L.oracle_bfp_value.restype = C.c_float
            L.oracle_bfp_bytes.argtypes = [sz, i32]
            L.oracle_bfp_bytes.restype = sz
            L.oracle_sparse_encode.argtypes = [vp, sz, i32, C.c_double, vp, vp, vp]
            L.oracle_sparse_decode.argtypes = [vp, vp, vp, sz, i32, vp, i32]
            L.oracle_sparse_is_sparse.argtypes = [sz, sz, C.c_double]
            L.oracle_sparse_is_sparse.restype = i32
            L.oracle_diff_encode.argtypes = [vp, vp, vp, sz]
            L.oracle_cast_to_f32.argtypes = [vp, sz, i32, vp]
            L.oracle_cast_from_f32.argtypes = [vp, sz, i32, vp]
            L.oracle_f32_to_f16.argtypes = [C.c_float]
            L.oracle_f32_to_f16.restype = C.c_uint16
            L.oracle_f16_to_f32.argtypes = [C.c_uint16]
            L.oracle_f16_to_f32.restype = C.c_float
            L.oracle_f32_to_bf16.argtypes = [C.c_float]
            L.oracle_f32_to_bf16.restype = C.c_uint16
            L.oracle_bf16_to_f32.argtypes = [C.c_uint16]
            L.oracle_bf16_to_f32.restype = C.c_float
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _ptrs(arrs) -> C.Array:
    return (C.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])


def _check(arrs, T, dtype):
    for a in arrs:
        assert a.dtype == NP_DTYPES[dtype] and a.size == T and a.flags["C_CONTIGUOUS"], \
            (a.dtype, a.size, dtype, T)


def _counters(N):
    return (C.c_uint64 * N)(), (C.c_uint64 * N)()


# ---------------------------------------------------------------------------
# collectives
# ---------------------------------------------------------------------------

def ring(inputs, in_dtype="f32", out_dtype="f32", codec="none", bits=8, threshold=0.5,
         slice=None, diff_prev=None, diff_base=None, average=False,
         mode="allreduce", outputs=None, residual=None):
    """Two-pass ring allreduce (mode="allreduce") or its first pass alone
    (mode="reduce_scatter") over N host arrays.  Returns (outputs, sent, recv).
    ``slice``: sparse codec only -- None for one message per chunk and hop,
    else the elements of each per-slice message.

    For reduce_scatter only chunk r of outputs[r] is written; pass ``outputs``
    to control what the other chunks hold (default: zeros).  ``residual``:
    N float32 arrays of T error-feedback residuals (BFP only), updated in
    place."""
    N = len(inputs)
    T = inputs[0].size
    _check(inputs, T, in_dtype)
    if outputs is None:
        outputs = [np.zeros(T, NP_DTYPES[out_dtype]) for _ in range(N)]
    _check(outputs, T, out_dtype)
    dp = None
    if diff_prev is not None:
        _check(diff_prev, T, "f32")
        dp = _ptrs(diff_prev)
    db = None
    if diff_base is not None:
        _check([diff_base], T, "f32")
        db = _ptr(diff_base)
    rp = None
    if residual is not None:
        _check(residual, T, "f32")
        rp = _ptrs(residual)
    sent, recv = _counters(N)
    rc = lib().oracle_ring_ef({"allreduce": 0, "reduce_scatter": 1}[mode], N, T, _ptrs(inputs),
                              DTYPES[in_dtype], _ptrs(outputs), DTYPES[out_dtype], CODECS[codec],
                              bits, float(threshold), int(slice or 0),
                              C.cast(dp, C.c_void_p) if dp is not None else None, db,
                              int(bool(average)), C.cast(rp, C.c_void_p) if rp is not None else None,
                              sent, recv)
    if rc != 0:
        raise ValueError("oracle_ring: bad arguments")
    return outputs, np.array(sent[:], np.uint64), np.array(recv[:], np.uint64)


def codec_stats(bufs, dtype="f32"):
    """Statistics of N input buffers for the adaptive codec choice:
    [elements, nonzero (fp32 bits not +0.0), nonzero flushed to code 0 by
    BFP4, nonzero flushed to code 0 by BFP8], with 128-element blocks cut
    from each ring chunk's start."""
    N, T = len(bufs), bufs[0].size
    _check(bufs, T, dtype)
    st = (C.c_uint64 * 4)()
    if lib().oracle_codec_stats(N, T, _ptrs(bufs), DTYPES[dtype], st) != 0:
        raise ValueError("oracle_codec_stats: bad arguments")
    return np.array(st[:], np.uint64)


OPS = {"allreduce": 0, "allgather": 1, "broadcast": 2}


def codec_stats_op(bufs, dtype="f32", op="allreduce", root=0):
    """Statistics of what an operation encodes (reading F4op): the allreduce
    every chunk of every buffer, the compressed allgather chunk r of buffer
    r, the compressed broadcast the root's buffer (blocks from its start)."""
    N, T = len(bufs), bufs[0].size
    _check(bufs, T, dtype)
    st = (C.c_uint64 * 4)()
    if lib().oracle_codec_stats_op(OPS[op], root, N, T, _ptrs(bufs), DTYPES[dtype], st) != 0:
        raise ValueError("oracle_codec_stats_op: bad arguments")
    return np.array(st[:], np.uint64)


def allgather(bufs, dtype="f32"):
    """In-place allgather: chunk r of bufs[r] is rank r's contribution."""
    N, T = len(bufs), bufs[0].size
    _check(bufs, T, dtype)
    sent, recv = _counters(N)
    assert lib().oracle_allgather(N, T, _ptrs(bufs), DTYPES[dtype], sent, recv) == 0
    return bufs, np.array(sent[:], np.uint64), np.array(recv[:], np.uint64)


def allgather_codec(bufs, dtype="f32", codec="bfp", bits=8, threshold=0.5, slice=None):
    """In-place compressed allgather (reading AG): chunk r of bufs[r] is rank
    r's contribution; every buffer ends with decode(codes) of every chunk.
    ``slice`` as for ``ring``."""
    N, T = len(bufs), bufs[0].size
    _check(bufs, T, dtype)
    sent, recv = _counters(N)
    if lib().oracle_allgather_codec(N, T, _ptrs(bufs), DTYPES[dtype], CODECS[codec], bits,
                                    float(threshold), int(slice or 0), sent, recv) != 0:
        raise ValueError("oracle_allgather_codec: bad arguments")
    return bufs, np.array(sent[:], np.uint64), np.array(recv[:], np.uint64)


def broadcast(bufs, dtype="f32", root=0):
    N, T = len(bufs), bufs[0].size
    _check(bufs, T, dtype)
    sent, recv = _counters(N)
    if lib().oracle_broadcast(N, T, _ptrs(bufs), DTYPES[dtype], root, sent, recv) != 0:
        raise ValueError("oracle_broadcast: bad arguments")
    return bufs, np.array(sent[:], np.uint64), np.array(recv[:], np.uint64)


def broadcast_codec(bufs, dtype="f32", root=0, bits=8):
    """In-place BFP-compressed broadcast (reading AB): every buffer ends with
    the decoded codes of the root's buffer."""
    N, T = len(bufs), bufs[0].size
    _check(bufs, T, dtype)
    sent, recv = _counters(N)
    if lib().oracle_broadcast_codec(N, T, _ptrs(bufs), DTYPES[dtype], root, bits, sent,
                                    recv) != 0:
        raise ValueError("oracle_broadcast_codec: bad arguments")
    return bufs, np.array(sent[:], np.uint64), np.array(recv[:], np.uint64)


def tree_allreduce(bufs):
    N, T = len(bufs), bufs[0].size
    _check(bufs, T, "f32")
    sent, recv = _counters(N)
    assert lib().oracle_tree_allreduce(N, T, _ptrs(bufs), sent, recv) == 0
    return bufs, np.array(sent[:], np.uint64), np.array(recv[:], np.uint64)


# ---------------------------------------------------------------------------
# codecs
# ---------------------------------------------------------------------------

def bfp_encode(x: np.ndarray, bits: int):
    """x: float32 array.  Returns (exps int8[ceil(n/128)], mants uint8)."""
    x = np.ascontiguousarray(x, np.float32)
    n = x.size
    exps = np.zeros((n + BFP_BLOCK - 1) // BFP_BLOCK, np.int8)
    mants = np.zeros(n if bits == 8 else (n + 1) // 2, np.uint8)
    lib().oracle_bfp_encode(_ptr(x), n, bits, _ptr(exps), _ptr(mants))
    return exps, mants


def bfp_decode(exps, mants, n, bits, out=None, accumulate=False):
    if out is None:
        out = np.zeros(n, np.float32)
    lib().oracle_bfp_decode(_ptr(exps), _ptr(mants), n, bits, _ptr(out), int(bool(accumulate)))
    return out


def bfp_block_exponent(x) -> int:
    x = np.ascontiguousarray(x, np.float32)
    return lib().oracle_bfp_block_exponent(_ptr(x), x.size)


def bfp_code(x: float, e: int, bits: int) -> int:
    return lib().oracle_bfp_code(float(x), e, bits)


def bfp_value(m: int, e: int, bits: int) -> float:
    return lib().oracle_bfp_value(m, e, bits)


def bfp_bytes(n: int, bits: int) -> int:
    return lib().oracle_bfp_bytes(n, bits)


def sparse_encode(x: np.ndarray, dtype="f32", threshold=0.5):
    """Returns (hdr uint32[2] = {fmt, nnz}, vals (input dtype), idx int32).
    vals/idx are trimmed to the payload the header describes."""
    n = x.size
    _check([x], n, dtype)
    hdr = np.zeros(2, np.uint32)
    vals = np.zeros(max(n, 1), NP_DTYPES[dtype])
    idx = np.zeros(max(n, 1), np.int32)
    lib().oracle_sparse_encode(_ptr(x), n, DTYPES[dtype], float(threshold), _ptr(hdr), _ptr(vals),
                               _ptr(idx))
    if hdr[0] == 1:
        return hdr, vals[: hdr[1]].copy(), idx[: hdr[1]].copy()
    return hdr, vals[:n].copy(), idx[:0].copy()


def sparse_decode(hdr, vals, idx, n, dtype="f32", acc=None, accumulate=False):
    if acc is None:
        acc = np.zeros(n, np.float32)
    vals = np.ascontiguousarray(vals) if vals.size else np.zeros(1, NP_DTYPES[dtype])
    idx = np.ascontiguousarray(idx, np.int32) if idx.size else np.zeros(1, np.int32)
    lib().oracle_sparse_decode(_ptr(np.ascontiguousarray(hdr, np.uint32)), _ptr(vals), _ptr(idx),
                               n, DTYPES[dtype], _ptr(acc), int(bool(accumulate)))
    return acc


def sparse_is_sparse(nnz: int, n: int, threshold: float) -> bool:
    return bool(lib().oracle_sparse_is_sparse(nnz, n, float(threshold)))


def diff_encode(cur, prev):
    cur = np.ascontiguousarray(cur, np.float32)
    prev = np.ascontiguousarray(prev, np.float32)
    out = np.empty_like(cur)
    lib().oracle_diff_encode(_ptr(cur), _ptr(prev), _ptr(out), cur.size)
    return out


def to_f32(x, dtype):
    x = np.ascontiguousarray(x)
    out = np.empty(x.size, np.float32)
    lib().oracle_cast_to_f32(_ptr(x), x.size, DTYPES[dtype], _ptr(out))
    return out


def from_f32(x, dtype):
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(x.size, NP_DTYPES[dtype])
    lib().oracle_cast_from_f32(_ptr(x), x.size, DTYPES[dtype], _ptr(out))
    return out


def f32_to_f16_bits(v: float) -> int:
    return lib().oracle_f32_to_f16(v)


def f32_to_bf16_bits(v: float) -> int:
    return lib().oracle_f32_to_bf16(v)
