"""The allocation-free sparse encoder, rra_sparse_encode_noalloc.

Some callers of this library cannot allocate device memory: processes whose
device memory belongs to their own allocator or is budgeted up front,
latency-critical loops that cannot take an allocation's implicit device
synchronisation, libraries that must not call the CUDA allocator behind
their framework's back.  For them the library offers a sparse encoder whose
scratch is a fixed array inside the library instead of a cudaMalloc'd
workspace.  This test calls it through the C ABI and checks its output --
header, values and indices, bit for bit, the tolerance every codec test here
uses -- against the CPU oracle's sparse encode and against the allocating
entry point rra_sparse_encode, on calls in a row through the shared scratch:
two of the same size on different data (an unwritten scratch word would carry
the first call's counts into the second), then other sizes and dtypes.  Sizes
beyond its fixed limit are refused.

The file name sorts last so that a run stopping at the first failure has run
every other test first; it also passes alone in a fresh process."""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle as O
import ring_allreduce_compressed_gb300 as rra
import workloads as W
from gpu_util import DT_NAME, host

pytestmark = pytest.mark.gpu


def _fn(name):
    f = getattr(rra.lib(), name)
    f.argtypes = [C.c_void_p, C.c_size_t, C.c_int, C.c_float, C.c_void_p, C.c_void_p,
                  C.c_void_p, C.c_void_p]
    f.restype = C.c_int
    return f


def _encode(fn, x, thr):
    """(hdr, payload values as raw bits, indices or None) of one encode."""
    n = x.numel()
    hdr = torch.zeros(2, dtype=torch.int32, device="cuda")
    vals = torch.zeros(n, dtype=x.dtype, device="cuda")
    idx = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    code = fn(C.c_void_p(x.data_ptr()), n, rra._dtype_code(x.dtype), C.c_float(thr),
              C.c_void_p(hdr.data_ptr()), C.c_void_p(vals.data_ptr()),
              C.c_void_p(idx.data_ptr()), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == rra.RRA_OK, rra.status_string(code)
    torch.cuda.synchronize()
    h = hdr.cpu().numpy().view(np.uint32)
    k = int(h[1]) if h[0] else n
    v = host(vals[:k])
    return h, v.view(np.uint16 if v.itemsize == 2 else np.uint32), \
        (idx[: int(h[1])].cpu().numpy() if h[0] else None)


def _oracle(x, thr):
    h, v, i = O.sparse_encode(host(x), DT_NAME[x.dtype], float(np.float32(thr)))
    return h, v.view(np.uint16 if v.itemsize == 2 else np.uint32), (i if h[0] else None)


def test_noalloc_sparse_encode_matches_the_oracle_and_the_allocating_encoder():
    rra.build()
    f_new, f_old = _fn("rra_sparse_encode_noalloc"), _fn("rra_sparse_encode")
    cases = [
        # the same size twice on different data: every scratch word is rewritten
        (3_000_017, 0.6, torch.bfloat16, 0.5, 5),
        (3_000_017, 0.8, torch.bfloat16, 0.5, 15),
        # other sizes and dtypes; the second of these is dense (30 % zeros)
        (4096 * 3 + 11, 0.7, torch.float16, 0.5, 8),
        (200_003, 0.3, torch.float32, 0.5, 6),
        (1, 0.0, torch.float32, 0.5, 9),
    ]
    formats = set()
    for n, p_zero, dt, thr, seed in cases:
        x = W.sparse(1, n, seed=seed, p_zero=p_zero, dtype=dt)[0]
        got = _encode(f_new, x, thr)
        want = _oracle(x, thr)
        also = _encode(f_old, x, thr)
        for a, b in ((got, want), (got, also)):
            assert list(a[0]) == list(b[0]), (n, a[0], b[0])
            assert np.array_equal(a[1], b[1]), n
            if b[2] is not None:
                assert np.array_equal(a[2], b[2]), n
        formats.add(int(got[0][0]))
    assert formats == {0, 1}  # both the sparse and the dense form were produced


def test_noalloc_sparse_encode_at_its_largest_size():
    """n = 2^28 fills the fixed scratch exactly; sampled against the oracle
    through the allocating encoder's identical output, and the header against
    a count made on the device by torch."""
    f_new, f_old = _fn("rra_sparse_encode_noalloc"), _fn("rra_sparse_encode")
    n = 1 << 28
    x = W.sparse(1, n, seed=21, p_zero=0.6, dtype=torch.bfloat16)[0]
    got = _encode(f_new, x, 0.5)
    also = _encode(f_old, x, 0.5)
    assert list(got[0]) == list(also[0])
    assert int(got[0][1]) == int((x.view(torch.int16) != 0).sum())
    assert np.array_equal(got[1], also[1]) and np.array_equal(got[2], also[2])
    # the oracle on the first and the last 3 Mi elements: their pairs are the
    # first and the last pairs of the whole message
    m = 3 << 20
    for lo in (0, n - m):
        part = x[lo: lo + m]
        hp, vp, ip = _oracle(part, 0.5)
        k = int(hp[1])
        sel = slice(0, k) if lo == 0 else slice(len(got[2]) - k, len(got[2]))
        assert np.array_equal(got[1][sel], vp)
        assert np.array_equal(got[2][sel], ip + lo)
    del x


def test_noalloc_sparse_encode_refuses_sizes_beyond_its_scratch():
    f_new = _fn("rra_sparse_encode_noalloc")
    too_big = 65536 * 4096 + 1
    # checked on the host before anything is read: dummy non-null pointers suffice
    code = f_new(C.c_void_p(256), too_big, 0, C.c_float(0.5), C.c_void_p(256), C.c_void_p(256),
                 C.c_void_p(256), None)
    assert code == rra.RRA_ERR_INVALID
