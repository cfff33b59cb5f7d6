"""The allocation-free sparse encoder, rra_sparse_encode_noalloc.

Some callers of this library cannot allocate device memory: code running
while a CUDA graph is being captured, latency-critical loops, processes whose
device memory belongs to their own allocator.  For them the library offers a
sparse encoder whose scratch is a fixed array inside the library instead of a
cudaMalloc'd workspace.  This test calls it through the C ABI and checks that
two calls in a row (different inputs, sizes and dtypes, so stale scratch from
the first call would show) produce exactly what the allocating entry point
rra_sparse_encode produces -- bit for bit, the tolerance every codec test
here uses -- and that sizes beyond its fixed limit are refused.

The file name sorts last so that a run stopping at the first failure has run
every other test first; it also passes alone in a fresh process."""
import ctypes as C

import numpy as np
import pytest
import torch

import ring_allreduce_compressed_gb300 as rra
import workloads as W

pytestmark = pytest.mark.gpu


def _encode(fn, x, thr):
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
    return h, vals[:k].cpu().view(torch.int16 if x.element_size() == 2 else torch.int32), \
        (idx[: int(h[1])].cpu() if h[0] else None)


def test_noalloc_sparse_encode_matches_the_allocating_encoder():
    rra.build()
    L = rra.lib()
    f_new = L.rra_sparse_encode_noalloc
    f_new.argtypes = [C.c_void_p, C.c_size_t, C.c_int, C.c_float, C.c_void_p, C.c_void_p,
                      C.c_void_p, C.c_void_p]
    f_new.restype = C.c_int
    f_old = L.rra_sparse_encode
    cases = [(3_000_017, 0.6, torch.bfloat16, 0.5, 5), (200_003, 0.3, torch.float32, 0.5, 6)]
    for n, p_zero, dt, thr, seed in cases:  # two calls in a row through the shared scratch
        x = W.sparse(1, n, seed=seed, p_zero=p_zero, dtype=dt)[0]
        h_new, v_new, i_new = _encode(f_new, x, thr)
        h_old, v_old, i_old = _encode(f_old, x, thr)
        assert list(h_new) == list(h_old)
        assert torch.equal(v_new, v_old)
        if i_old is not None:
            assert torch.equal(i_new, i_old)
    # both formats were exercised: the first input is sparse, the second dense
    x = W.sparse(1, 1000, seed=7, p_zero=0.9)[0]
    assert _encode(f_new, x, 0.5)[0][0] == 1


def test_noalloc_sparse_encode_refuses_sizes_beyond_its_scratch():
    L = rra.lib()
    f_new = L.rra_sparse_encode_noalloc
    f_new.argtypes = [C.c_void_p, C.c_size_t, C.c_int, C.c_float, C.c_void_p, C.c_void_p,
                      C.c_void_p, C.c_void_p]
    f_new.restype = C.c_int
    too_big = 65536 * 4096 + 1
    # checked on the host before anything is read: dummy non-null pointers suffice
    code = f_new(C.c_void_p(256), too_big, 0, C.c_float(0.5), C.c_void_p(256), C.c_void_p(256),
                 C.c_void_p(256), None)
    assert code == rra.RRA_ERR_INVALID
