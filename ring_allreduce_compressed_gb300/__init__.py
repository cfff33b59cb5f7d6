"""Python binding of librra (include/rra.h): the chunked ring allreduce with
gradient-compression codecs for N ranks simulated on one GB300 (sm_103a).

This module only marshals arguments (tensor pointers, dtype codes, the
current CUDA stream) into the C ABI; every step of every collective and codec
runs in the library's CUDA kernels.  PyTorch supplies device memory and
streams.  There is no CPU fallback: importing works without a GPU, but every
call needs the built library and a CUDA device, and raises otherwise.

Names follow the C ABI: ``Comm.ring_allreduce``, ``Comm.reduce_scatter``,
``Comm.allgather``, ``Comm.broadcast``, ``Comm.tree_allreduce``,
``bfp_encode``/``bfp_decode``, ``sparse_encode``/``sparse_decode``,
``diff_encode``.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass
from typing import Optional, Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "librra.so")

RRA_OK, RRA_ERR_INVALID, RRA_ERR_UNSUPPORTED, RRA_ERR_CUDA, RRA_ERR_TIMEOUT, RRA_ERR_NOMEM = range(6)
RRA_ALGO_RING, RRA_ALGO_TREE = 0, 1
# operations for the operator-aware codec choice (rra_codec_*_op)
RRA_OP_ALLREDUCE, RRA_OP_ALLGATHER, RRA_OP_BROADCAST = 0, 1, 2
RRA_DEFAULT_CROSSOVER = 256 << 20          # N <= 4
RRA_DEFAULT_CROSSOVER_WIDE = (1 << 30) + 1  # N >= 5


def default_crossover(N: int) -> int:
    """rra_allreduce_auto's crossover for N ranks until one is set or measured."""
    return RRA_DEFAULT_CROSSOVER if N <= 4 else RRA_DEFAULT_CROSSOVER_WIDE
RRA_F32, RRA_F16, RRA_BF16 = 0, 1, 2
CODEC_NONE, CODEC_BFP, CODEC_SPARSE = 0, 1, 2
MAX_RANKS = 64
BFP_BLOCK = 128
RING_SLICE = 256
SPARSE_PER_CHUNK, SPARSE_PER_SLICE = 0, 1

_lib = None


class RRAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)}")


class _Codec(C.Structure):
    _fields_ = [("kind", C.c_int), ("bits", C.c_int), ("sparsity_threshold", C.c_float),
                ("diff_prev", C.c_void_p), ("diff_base", C.c_void_p), ("average", C.c_int),
                ("residual", C.c_void_p), ("sparse_granularity", C.c_int)]


class _Stats(C.Structure):
    _fields_ = [("elements", C.c_uint64), ("nonzero", C.c_uint64),
                ("bfp4_flushed", C.c_uint64), ("bfp8_flushed", C.c_uint64)]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile librra.so in-tree (see _compile.py)."""
    from . import _compile
    return _compile.build(force=force, verbose=verbose)


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"librra.so is not built ({LIB_PATH}); run "
                               "ring_allreduce_compressed_gb300.build() first")
        L = C.CDLL(LIB_PATH)
        vp, sz, i32, st = C.c_void_p, C.c_size_t, C.c_int, C.c_int
        L.rra_comm_create.argtypes = [i32, sz, i32, C.POINTER(C.c_void_p)]
        L.rra_comm_destroy.argtypes = [vp]
        L.rra_ring_allreduce.argtypes = [vp, vp, vp, sz, i32, i32, vp, vp]
        L.rra_reduce_scatter.argtypes = [vp, vp, vp, sz, i32, i32, vp, vp]
        L.rra_allgather.argtypes = [vp, vp, sz, i32, vp]
        L.rra_allgather_codec.argtypes = [vp, vp, sz, i32, vp, vp]
        L.rra_broadcast.argtypes = [vp, vp, sz, i32, i32, vp]
        L.rra_broadcast_codec.argtypes = [vp, vp, sz, i32, i32, vp, vp]
        L.rra_tree_allreduce.argtypes = [vp, vp, sz, i32, vp]
        L.rra_bfp_encode.argtypes = [vp, sz, i32, i32, vp, vp, vp]
        L.rra_bfp_decode.argtypes = [vp, vp, sz, i32, vp, i32, vp]
        L.rra_sparse_encode.argtypes = [vp, sz, i32, C.c_float, vp, vp, vp, vp]
        L.rra_sparse_encode_noalloc.argtypes = [vp, sz, i32, C.c_float, vp, vp, vp, vp]
        L.rra_sparse_decode.argtypes = [vp, vp, vp, sz, i32, vp, i32, vp]
        L.rra_diff_encode.argtypes = [vp, vp, vp, sz, vp]
        L.rra_get_bytes.argtypes = [vp, C.POINTER(C.c_uint64), C.POINTER(C.c_uint64)]
        L.rra_comm_status.argtypes = [vp]
        L.rra_set_timeout.argtypes = [vp, C.c_uint64]
        L.rra_debug_withhold.argtypes = [vp, i32, i32]
        L.rra_comm_set_tuning.argtypes = [vp, i32, i32, i32, i32]
        L.rra_comm_last_shape.argtypes = [vp] + [C.POINTER(C.c_int)] * 4
        L.rra_autotune.argtypes = [vp, vp, vp, sz, i32, i32, vp, vp]
        L.rra_allreduce_auto.argtypes = [vp, vp, sz, i32, vp, C.POINTER(C.c_int)]
        L.rra_set_crossover.argtypes = [vp, sz]
        L.rra_get_crossover.argtypes = [vp, C.POINTER(C.c_size_t)]
        L.rra_autotune_crossover.argtypes = [vp, vp, sz, i32, vp, C.POINTER(C.c_size_t)]
        L.rra_codec_measure.argtypes = [vp, vp, sz, i32, C.POINTER(_Stats), vp]
        L.rra_codec_measure_op.argtypes = [vp, i32, i32, vp, sz, i32, C.POINTER(_Stats), vp]
        L.rra_codec_advise_op.argtypes = [vp, i32, i32, vp, sz, i32, C.c_float, C.c_float, i32,
                                          C.POINTER(_Codec), C.POINTER(_Stats), vp]
        L.rra_codec_advise.argtypes = [vp, vp, sz, i32, C.c_float, C.c_float,
                                       C.POINTER(_Codec), C.POINTER(_Stats), vp]
        L.rra_status_string.argtypes = [i32]
        L.rra_status_string.restype = C.c_char_p
        for name in ("rra_comm_create", "rra_comm_destroy", "rra_ring_allreduce",
                     "rra_reduce_scatter", "rra_allgather", "rra_allgather_codec", "rra_broadcast",
                     "rra_broadcast_codec",
                     "rra_tree_allreduce",
                     "rra_bfp_encode", "rra_bfp_decode", "rra_sparse_encode",
                     "rra_sparse_encode_noalloc", "rra_sparse_decode",
                     "rra_diff_encode", "rra_get_bytes", "rra_comm_status", "rra_set_timeout",
                     "rra_debug_withhold", "rra_comm_set_tuning", "rra_comm_last_shape",
                     "rra_autotune", "rra_allreduce_auto", "rra_set_crossover",
                     "rra_get_crossover", "rra_autotune_crossover", "rra_codec_measure",
                     "rra_codec_advise", "rra_codec_measure_op", "rra_codec_advise_op"):
            getattr(L, name).restype = st
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().rra_status_string(code).decode()


def _check(code: int, where: str):
    if code != RRA_OK:
        raise RRAError(code, where)


def _dtype_code(t) -> int:
    import torch
    m = {torch.float32: RRA_F32, torch.float16: RRA_F16, torch.bfloat16: RRA_BF16}
    if t not in m:
        raise TypeError(f"unsupported dtype {t}")
    return m[t]


def _stream(stream) -> C.c_void_p:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _dev(t, name):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA tensor")
    return t.data_ptr()


def _ptrs(ts: Sequence, name: str):
    return (C.c_void_p * len(ts))(*[_dev(t, name) for t in ts])


@dataclass
class Codec:
    """Codec of a reducing call (rra_codec).  kind: "none" | "bfp" | "sparse"."""
    kind: str = "none"
    bits: int = 8
    sparsity_threshold: float = 0.5
    diff_prev: Optional[Sequence] = None  # N fp32 tensors (previous round)
    diff_base: Optional[object] = None    # fp32 tensor (previous result)
    average: bool = False
    residual: Optional[Sequence] = None   # N fp32 tensors: error-feedback residuals (BFP)
    granularity: str = "chunk"            # sparse: one message per "chunk" and hop, or per "slice"

    def _marshal(self):
        kinds = {"none": CODEC_NONE, "bfp": CODEC_BFP, "sparse": CODEC_SPARSE}
        keep = []
        c = _Codec()
        c.kind = kinds[self.kind]
        c.bits = int(self.bits)
        c.sparsity_threshold = float(self.sparsity_threshold)
        if self.diff_prev is not None:
            arr = _ptrs(self.diff_prev, "diff_prev")
            keep.append(arr)
            c.diff_prev = C.cast(arr, C.c_void_p)
        if self.diff_base is not None:
            c.diff_base = _dev(self.diff_base, "diff_base")
        c.average = 1 if self.average else 0
        c.sparse_granularity = {"chunk": SPARSE_PER_CHUNK, "slice": SPARSE_PER_SLICE}[self.granularity]
        if self.residual is not None:
            arr = _ptrs(self.residual, "residual")
            keep.append(arr)
            c.residual = C.cast(arr, C.c_void_p)
        return c, keep


class Comm:
    """A communicator of ``nranks`` simulated ranks on the current device."""

    def __init__(self, nranks: int, max_count: int, max_dtype=None):
        import torch
        code = _dtype_code(max_dtype if max_dtype is not None else torch.float32)
        h = C.c_void_p()
        _check(lib().rra_comm_create(nranks, max_count, code, C.byref(h)), "rra_comm_create")
        self._h = h
        self.nranks = nranks

    def close(self):
        if getattr(self, "_h", None):
            lib().rra_comm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _reduce(self, fn, name, inputs, outputs, codec, stream):
        if len(inputs) != self.nranks or len(outputs) != self.nranks:
            raise ValueError(f"{name}: need {self.nranks} inputs and outputs")
        c, keep = (codec or Codec())._marshal()
        _check(fn(self._h, _ptrs(inputs, "inputs"), _ptrs(outputs, "outputs"), inputs[0].numel(),
                  _dtype_code(inputs[0].dtype), _dtype_code(outputs[0].dtype), C.byref(c),
                  _stream(stream)), name)
        del keep

    def ring_allreduce(self, inputs, outputs, codec: Optional[Codec] = None, stream=None):
        self._reduce(lib().rra_ring_allreduce, "rra_ring_allreduce", inputs, outputs, codec, stream)

    def reduce_scatter(self, inputs, outputs, codec: Optional[Codec] = None, stream=None):
        self._reduce(lib().rra_reduce_scatter, "rra_reduce_scatter", inputs, outputs, codec, stream)

    def allgather(self, bufs, codec: Optional[Codec] = None, stream=None):
        """In-place allgather; with a BFP or sparse codec every chunk travels
        as its owner's codes and every rank stores the decoded chunk."""
        if codec is None:
            _check(lib().rra_allgather(self._h, _ptrs(bufs, "bufs"), bufs[0].numel(),
                                       _dtype_code(bufs[0].dtype), _stream(stream)),
                   "rra_allgather")
            return
        c, keep = codec._marshal()
        _check(lib().rra_allgather_codec(self._h, _ptrs(bufs, "bufs"), bufs[0].numel(),
                                         _dtype_code(bufs[0].dtype), C.byref(c),
                                         _stream(stream)), "rra_allgather_codec")
        del keep

    def broadcast(self, bufs, root: int = 0, codec: Optional[Codec] = None, stream=None):
        """In-place broadcast from root; with a BFP codec the root's codes
        travel the tree and every rank (root included) stores the decoded
        buffer."""
        if codec is None:
            _check(lib().rra_broadcast(self._h, _ptrs(bufs, "bufs"), bufs[0].numel(),
                                       _dtype_code(bufs[0].dtype), root, _stream(stream)),
                   "rra_broadcast")
            return
        c, keep = codec._marshal()
        _check(lib().rra_broadcast_codec(self._h, _ptrs(bufs, "bufs"), bufs[0].numel(),
                                         _dtype_code(bufs[0].dtype), root, C.byref(c),
                                         _stream(stream)), "rra_broadcast_codec")
        del keep

    def tree_allreduce(self, bufs, stream=None):
        _check(lib().rra_tree_allreduce(self._h, _ptrs(bufs, "bufs"), bufs[0].numel(),
                                        _dtype_code(bufs[0].dtype), _stream(stream)),
               "rra_tree_allreduce")

    def get_bytes(self):
        sent = (C.c_uint64 * self.nranks)()
        recv = (C.c_uint64 * self.nranks)()
        _check(lib().rra_get_bytes(self._h, sent, recv), "rra_get_bytes")
        return list(sent), list(recv)

    def status(self) -> int:
        """Latched device-side status of the last call (cleared by reading)."""
        return lib().rra_comm_status(self._h)

    def set_timeout(self, ns: int):
        _check(lib().rra_set_timeout(self._h, int(ns)), "rra_set_timeout")

    def set_tuning(self, blocks_per_sm: int = 0, mailbox_depth: int = 0, stage_depth: int = 0,
                   slice_groups: int = 0):
        """Launch tuning of the fused kernels (0 = automatic)."""
        _check(lib().rra_comm_set_tuning(self._h, blocks_per_sm, mailbox_depth, stage_depth,
                                         slice_groups), "rra_comm_set_tuning")

    def last_shape(self):
        """(blocks per SM, mailbox depth, staging depth, slice groups) of the
        last ring launch."""
        v = [C.c_int() for _ in range(4)]
        _check(lib().rra_comm_last_shape(self._h, *[C.byref(x) for x in v]),
               "rra_comm_last_shape")
        return tuple(x.value for x in v)

    def autotune(self, inputs, outputs, codec: Optional[Codec] = None, stream=None):
        """Time the ring allreduce of these arguments in every candidate
        launch shape and keep the fastest for later calls with the same
        codec, dtypes and count (rra_autotune); returns that shape."""
        self._reduce(lib().rra_autotune, "rra_autotune", inputs, outputs, codec, stream)
        return self.last_shape()

    def allreduce_auto(self, bufs, stream=None) -> int:
        """In-place allreduce, tree below the crossover (fp32), ring above;
        returns RRA_ALGO_RING or RRA_ALGO_TREE."""
        algo = C.c_int(-1)
        _check(lib().rra_allreduce_auto(self._h, _ptrs(bufs, "bufs"), bufs[0].numel(),
                                        _dtype_code(bufs[0].dtype), _stream(stream),
                                        C.byref(algo)), "rra_allreduce_auto")
        return algo.value

    def set_crossover(self, bytes_per_rank: int = 0):
        _check(lib().rra_set_crossover(self._h, int(bytes_per_rank)), "rra_set_crossover")

    def crossover(self) -> int:
        v = C.c_size_t()
        _check(lib().rra_get_crossover(self._h, C.byref(v)), "rra_get_crossover")
        return v.value

    def autotune_crossover(self, bufs, stream=None) -> int:
        """Measure the ring/tree crossover on bufs (overwritten); returns it."""
        v = C.c_size_t()
        _check(lib().rra_autotune_crossover(self._h, _ptrs(bufs, "bufs"), bufs[0].numel(),
                                            _dtype_code(bufs[0].dtype), _stream(stream),
                                            C.byref(v)), "rra_autotune_crossover")
        return v.value

    def codec_stats(self, inputs, op: int = None, root: int = 0, stream=None) -> dict:
        """rra_codec_measure: elements, nonzero, and the nonzero elements BFP4
        and BFP8 would round to code 0, over the N inputs; with an op
        (RRA_OP_*), rra_codec_measure_op: over what that operation encodes."""
        st = _Stats()
        if op is None:
            _check(lib().rra_codec_measure(self._h, _ptrs(inputs, "inputs"), inputs[0].numel(),
                                           _dtype_code(inputs[0].dtype), C.byref(st),
                                           _stream(stream)), "rra_codec_measure")
        else:
            _check(lib().rra_codec_measure_op(self._h, op, root, _ptrs(inputs, "inputs"),
                                              inputs[0].numel(), _dtype_code(inputs[0].dtype),
                                              C.byref(st), _stream(stream)),
                   "rra_codec_measure_op")
        return {k: int(getattr(st, k)) for k, _ in _Stats._fields_}

    def advise_codec(self, inputs, sparsity_threshold: float = 0.5,
                     max_flushed_fraction: float = 0.01, stream=None):
        """rra_codec_advise: (Codec, stats) -- sparse above the sparsity
        threshold, else BFP4 if it flushes at most the given share of the
        nonzero values to code 0, else BFP8."""
        st, c = _Stats(), _Codec()
        _check(lib().rra_codec_advise(self._h, _ptrs(inputs, "inputs"), inputs[0].numel(),
                                      _dtype_code(inputs[0].dtype), float(sparsity_threshold),
                                      float(max_flushed_fraction), C.byref(c), C.byref(st),
                                      _stream(stream)), "rra_codec_advise")
        kind = {CODEC_NONE: "none", CODEC_BFP: "bfp", CODEC_SPARSE: "sparse"}[c.kind]
        return (Codec(kind, bits=c.bits, sparsity_threshold=c.sparsity_threshold),
                {k: int(getattr(st, k)) for k, _ in _Stats._fields_})

    def advise_codec_op(self, op: int, inputs, root: int = 0, sparsity_threshold: float = 0.5,
                        max_flushed_fraction: float = 0.01, allow_lossy: bool = True,
                        stream=None):
        """rra_codec_advise_op: (Codec, stats) for the allreduce (as
        advise_codec), the compressed allgather (sparse if sparse enough,
        else BFP8 when allowed and harmless enough, else none) or the
        compressed broadcast (BFP8 when allowed and harmless enough, else
        none)."""
        st, c = _Stats(), _Codec()
        _check(lib().rra_codec_advise_op(self._h, op, root, _ptrs(inputs, "inputs"),
                                         inputs[0].numel(), _dtype_code(inputs[0].dtype),
                                         float(sparsity_threshold), float(max_flushed_fraction),
                                         1 if allow_lossy else 0, C.byref(c), C.byref(st),
                                         _stream(stream)), "rra_codec_advise_op")
        kind = {CODEC_NONE: "none", CODEC_BFP: "bfp", CODEC_SPARSE: "sparse"}[c.kind]
        return (Codec(kind, bits=c.bits, sparsity_threshold=c.sparsity_threshold),
                {k: int(getattr(st, k)) for k, _ in _Stats._fields_})

    def debug_withhold(self, rank: int, step: int):
        _check(lib().rra_debug_withhold(self._h, rank, step), "rra_debug_withhold")


# ---------------------------------------------------------------- codecs

def bfp_encode(x, bits: int, exps, mants, stream=None):
    _check(lib().rra_bfp_encode(_dev(x, "x"), x.numel(), _dtype_code(x.dtype), bits,
                                _dev(exps, "exps"), _dev(mants, "mants"), _stream(stream)),
           "rra_bfp_encode")


def bfp_decode(exps, mants, n: int, bits: int, out, accumulate: bool = False, stream=None):
    _check(lib().rra_bfp_decode(_dev(exps, "exps"), _dev(mants, "mants"), n, bits,
                                _dev(out, "out"), int(accumulate), _stream(stream)),
           "rra_bfp_decode")


def sparse_encode(x, threshold: float, hdr, vals, idx, stream=None):
    _check(lib().rra_sparse_encode(_dev(x, "x"), x.numel(), _dtype_code(x.dtype), threshold,
                                   _dev(hdr, "hdr"), _dev(vals, "vals"), _dev(idx, "idx"),
                                   _stream(stream)), "rra_sparse_encode")


def sparse_encode_noalloc(x, threshold: float, hdr, vals, idx, stream=None):
    """rra_sparse_encode_noalloc: the sparse encoder without any device
    allocation (fixed in-library scratch; n <= RRA_NOALLOC_MAX_COUNT), for
    callers that cannot allocate: processes whose device memory belongs to
    their own allocator or a fixed budget, latency-critical loops, libraries
    that must not call the CUDA allocator behind their framework's back."""
    _check(lib().rra_sparse_encode_noalloc(_dev(x, "x"), x.numel(), _dtype_code(x.dtype),
                                           threshold, _dev(hdr, "hdr"), _dev(vals, "vals"),
                                           _dev(idx, "idx"), _stream(stream)),
           "rra_sparse_encode_noalloc")


def sparse_decode(hdr, vals, idx, n: int, acc, accumulate: bool = False, stream=None):
    _check(lib().rra_sparse_decode(_dev(hdr, "hdr"), _dev(vals, "vals"), _dev(idx, "idx"), n,
                                   _dtype_code(vals.dtype), _dev(acc, "acc"), int(accumulate),
                                   _stream(stream)), "rra_sparse_decode")


def diff_encode(cur, prev, diff, stream=None):
    _check(lib().rra_diff_encode(_dev(cur, "cur"), _dev(prev, "prev"), _dev(diff, "diff"),
                                 cur.numel(), _stream(stream)), "rra_diff_encode")
