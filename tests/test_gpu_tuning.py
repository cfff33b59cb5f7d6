"""GPU tests of the measured tuning layer: the launch-shape autotuner of the
ring allreduce and the size-based ring/tree choice ("从零实现集合通信",
sections "真实世界中的生产模式" and "练习": choose ring or tree by message
size and measure the crossover; CCCL §2.2/§3.3: the pipeline chunk size).

Tuning may change only the time a call takes: every result is compared with
the oracle bit for bit, whichever shape or algorithm ran."""
import numpy as np
import pytest
import torch

import oracle as O
import ring_allreduce_compressed_gb300 as rra
from gpu_util import assert_bits_equal, cast, host, rand_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rra.build()
    rra.lib()
    torch.cuda.init()


def test_autotune_keeps_results_and_remembers_the_shape():
    N, T = 8, 8 * 2048 * 40 + 8 * 96  # several slice positions and a short last slice
    xs = cast(rand_f32(N, T, seed=123, scale=1e-3), "f16")
    codec = rra.Codec("bfp", bits=8)
    ref, s_ref, r_ref = O.ring([host(x) for x in xs], "f16", "f16", codec="bfp", bits=8)
    comm = rra.Comm(N, T, torch.float16)
    outs = [torch.zeros(T, dtype=torch.float16, device="cuda") for _ in range(N)]
    shape = comm.autotune(xs, outs, codec)
    assert comm.status() == rra.RRA_OK
    blocks, K, D, G = shape
    assert G in (1, 2, 4, 8) and 1 <= K <= 8 and 1 <= D <= 16 and blocks >= 1
    for q in range(N):  # the autotuner leaves the result of a call in outs
        assert_bits_equal(host(outs[q]), ref[q], f"autotune out {q}")
    assert comm.get_bytes() == (list(s_ref), list(r_ref))
    # a later call with the same key takes the measured shape
    outs2 = [torch.zeros(T, dtype=torch.float16, device="cuda") for _ in range(N)]
    comm.ring_allreduce(xs, outs2, codec)
    assert comm.status() == rra.RRA_OK
    assert comm.last_shape() == shape
    for q in range(N):
        assert_bits_equal(host(outs2[q]), ref[q], f"tuned call {q}")
    # a manual shape overrides the measured one
    comm.set_tuning(2, 2, 1, 1)
    comm.ring_allreduce(xs, outs2, codec)
    assert comm.status() == rra.RRA_OK
    assert comm.last_shape()[3] == 1
    for q in range(N):
        assert_bits_equal(host(outs2[q]), ref[q], f"manual call {q}")
    comm.close()


def test_autotune_other_key_is_untouched():
    """The measured shape belongs to its (codec, dtypes, count) key only."""
    N, T = 4, 4 * 4096
    xs = rand_f32(N, T, seed=5)
    comm = rra.Comm(N, T)
    outs = [torch.zeros(T, device="cuda") for _ in range(N)]
    comm.ring_allreduce(xs, outs)
    auto_shape = comm.last_shape()
    comm.autotune(xs, outs, rra.Codec("bfp", bits=4))
    comm.ring_allreduce(xs, outs)  # lossless: a different key
    assert comm.last_shape() == auto_shape
    ref = O.ring([host(x) for x in xs])[0]
    for q in range(N):
        assert_bits_equal(host(outs[q]), ref[q], f"lossless {q}")
    comm.close()


@pytest.mark.parametrize("N", [2, 5, 8])
def test_allreduce_auto_follows_the_crossover(N):
    # the default for N (256 MiB per rank up to N = 4, above 1 GiB from
    # N = 5), then a 4 MiB crossover set by the caller
    T_small, T_large = 1000, (4 << 20) // 4 + 24
    comm = rra.Comm(N, T_large)
    assert comm.crossover() == rra.default_crossover(N)
    comm.set_crossover(4 << 20)
    assert comm.crossover() == 4 << 20
    for T, algo in [(T_small, rra.RRA_ALGO_TREE), (T_large, rra.RRA_ALGO_RING)]:
        xs = rand_f32(N, T, seed=N + T)
        bufs = [x.clone() for x in xs]
        assert comm.allreduce_auto(bufs) == algo
        assert comm.status() == rra.RRA_OK
        hx = [host(x) for x in xs]
        ref = (O.tree_allreduce(hx)[0] if algo == rra.RRA_ALGO_TREE else O.ring(hx)[0])
        for q in range(N):
            assert_bits_equal(host(bufs[q]), ref[q], f"auto T={T} {q}")
    # a crossover of one byte sends everything to the ring; a huge one to the tree
    xs = rand_f32(N, T_small, seed=9)
    comm.set_crossover(1)
    assert comm.allreduce_auto([x.clone() for x in xs]) == rra.RRA_ALGO_RING
    comm.set_crossover(1 << 40)
    assert comm.allreduce_auto([x.clone() for x in xs]) == rra.RRA_ALGO_TREE
    # the tree sums fp32 only: half precision always takes the ring
    h = cast(xs, "f16")
    assert comm.allreduce_auto(h) == rra.RRA_ALGO_RING
    assert comm.status() == rra.RRA_OK
    comm.set_crossover(0)
    assert comm.crossover() == rra.default_crossover(N)
    comm.close()


def test_autotune_crossover_is_consistent():
    N, T = 4, 256 * 4 ** 5  # 1 Ki .. 1 Mi bytes per rank
    comm = rra.Comm(N, T)
    bufs = rand_f32(N, T, seed=77)
    c = comm.autotune_crossover(bufs)
    assert comm.status() == rra.RRA_OK
    assert c == comm.crossover()
    # a measured size (1 KiB * 4^k), or one byte above the largest when the tree always won
    assert c in [1024 * 4 ** k for k in range(6)] + [4 * T + 1]
    xs = rand_f32(N, 300, seed=1)
    algo = comm.allreduce_auto([x.clone() for x in xs])
    assert algo == (rra.RRA_ALGO_TREE if 300 * 4 < c else rra.RRA_ALGO_RING)
    comm.close()


def test_alternating_launch_shapes():
    """Calls that alternate between launch shapes with different shared-memory
    sizes all launch: the library only ever raises a kernel's shared-memory
    limit, so a smaller shape in between cannot break a larger one."""
    N, T = 8, 8 * 2048 * 12
    xs = cast(rand_f32(N, T, seed=3, scale=1e-3), "f16")
    codec = rra.Codec("bfp", bits=8)
    ref = O.ring([host(x) for x in xs], "f16", "f16", codec="bfp", bits=8)[0]
    comm = rra.Comm(N, T, torch.float16)
    outs = [torch.zeros(T, dtype=torch.float16, device="cuda") for _ in range(N)]
    for D in (4, 1, 2, 4, 1, 4):
        comm.set_tuning(1, 2, D, 8)
        comm.ring_allreduce(xs, outs, codec)
        assert comm.status() == rra.RRA_OK
        assert comm.last_shape()[2] == D
        for q in (0, N - 1):
            assert_bits_equal(host(outs[q]), ref[q], f"D={D} {q}")
    comm.close()
