"""GPU parity of error feedback ("CCCL通信压缩库" §5, future directions: the
precision a compression loses is carried into the next round): each rank's
fp32 residual is added to every value it encodes and keeps what the encoding
lost.  Outputs, byte counts and residuals are compared with the oracle bit
for bit over several rounds, so the carried state itself is checked."""
import numpy as np
import pytest
import torch

import oracle as O
import ring_allreduce_compressed_gb300 as rra
import workloads as W
from gpu_util import assert_bits_equal, cast, host, rand_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rra.build()
    rra.lib()
    torch.cuda.init()


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("in_dt", ["f16", "f32"])
@pytest.mark.parametrize("N,T", [(8, 8 * 2048 * 5 + 8 * 300), (3, 3 * 1000 + 1), (20, 20 * 512 + 9)])
@pytest.mark.parametrize("mode", ["allreduce", "reduce_scatter"])
def test_error_feedback_rounds(bits, in_dt, N, T, mode):
    comm = rra.Comm(N, T, torch.float32)
    res = [torch.zeros(T, device="cuda") for _ in range(N)]
    res_o = [np.zeros(T, np.float32) for _ in range(N)]
    for rnd in range(3):
        xs = cast(rand_f32(N, T, seed=100 * rnd + N + T, scale=1e-3), in_dt)
        outs = [torch.zeros(T, device="cuda") for _ in range(N)]
        codec = rra.Codec("bfp", bits=bits, residual=res)
        if mode == "allreduce":
            comm.ring_allreduce(xs, outs, codec)
        else:
            comm.reduce_scatter(xs, outs, codec)
        sent, recv = comm.get_bytes()
        assert comm.status() == rra.RRA_OK
        ref_outs = [np.zeros(T, np.float32) for _ in range(N)]
        ref, rs, rr = O.ring([host(x) for x in xs], in_dt, "f32", codec="bfp", bits=bits,
                             mode=mode, outputs=ref_outs, residual=res_o)
        for r in range(N):
            assert_bits_equal(host(outs[r]), ref[r], f"round {rnd} out {r}")
            assert_bits_equal(host(res[r]), res_o[r], f"round {rnd} residual {r}")
        assert list(sent) == list(rs) and list(recv) == list(rr)
    comm.close()


def test_error_feedback_with_diff_and_forced_shapes():
    """The DiLoCo composition (difference, BFP4, average, base) with feedback,
    in every slice width: the residual follows the encoded difference."""
    N, T = 8, 8 * 1024 * 3 + 8 * 200
    cur, prev = W.diloco(N, T, seed=5)
    base = torch.randn(T, device="cuda") * 1e-4
    comm = rra.Comm(N, T)
    for G in (8, 4, 2, 1):
        comm.set_tuning(0, 0, 0, G)
        res = [torch.full((T,), 1e-6, device="cuda") for _ in range(N)]
        res_o = [host(r) for r in res]
        outs = [torch.zeros(T, device="cuda") for _ in range(N)]
        codec = rra.Codec("bfp", bits=4, diff_prev=prev, diff_base=base, average=True,
                          residual=res)
        comm.ring_allreduce(cur, outs, codec)
        assert comm.status() == rra.RRA_OK
        ref = O.ring([host(c) for c in cur], codec="bfp", bits=4,
                     diff_prev=[host(p) for p in prev], diff_base=host(base), average=True,
                     residual=res_o)[0]
        for r in (0, N - 1):
            assert_bits_equal(host(outs[r]), ref[r], f"G={G} out {r}")
        for r in range(N):
            assert_bits_equal(host(res[r]), res_o[r], f"G={G} residual {r}")
    comm.close()


def test_error_feedback_argument_checks():
    N, T = 4, 4096
    xs = rand_f32(N, T, seed=1)
    outs = [torch.zeros(T, device="cuda") for _ in range(N)]
    res = [torch.zeros(T, device="cuda") for _ in range(N)]
    comm = rra.Comm(N, T)
    with pytest.raises(rra.RRAError) as e:  # lossless and sparse lose nothing
        comm.ring_allreduce(xs, outs, rra.Codec("none", residual=res))
    assert e.value.code == rra.RRA_ERR_UNSUPPORTED
    with pytest.raises(rra.RRAError) as e:
        comm.ring_allreduce(xs, outs, rra.Codec("sparse", residual=res))
    assert e.value.code == rra.RRA_ERR_UNSUPPORTED
    with pytest.raises(rra.RRAError) as e:  # a residual that is also an output
        comm.ring_allreduce(xs, outs, rra.Codec("bfp", bits=8, residual=[outs[0]] + res[1:]))
    assert e.value.code == rra.RRA_ERR_INVALID
    with pytest.raises(rra.RRAError) as e:  # two ranks sharing a residual
        comm.ring_allreduce(xs, outs, rra.Codec("bfp", bits=8, residual=[res[0]] * N))
    assert e.value.code == rra.RRA_ERR_INVALID
    comm.close()
