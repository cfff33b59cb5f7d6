"""GPU tests of the adaptive codec choice ("CCCL通信压缩库" §5, future
directions: watch sparsity and value distribution and switch the
compression).  The statistics are integer counts, compared with the oracle
exactly; the advice follows the documented rule from those counts."""
import numpy as np
import pytest
import torch

import oracle as O
import ring_allreduce_compressed_gb300 as rra
import workloads as W
from gpu_util import TORCH_DT, cast, host, rand_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rra.build()
    rra.lib()
    torch.cuda.init()


def _mixed(N, T, seed, dt):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    xs = []
    for _ in range(N):
        mag = 10.0 ** torch.randint(-6, 2, (T,), generator=g, device="cuda").float()
        x = torch.randn(T, generator=g, device="cuda") * mag
        x[torch.rand(T, generator=g, device="cuda") < 0.3] = 0.0
        x[torch.rand(T, generator=g, device="cuda") < 0.02] = -0.0
        xs.append(x.to(TORCH_DT[dt]))
    return xs


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N,T", [(1, 300), (2, 257), (4, 4096 * 3 + 17), (8, 8 * 1000 + 3),
                                 (20, 20 * 130 + 11)])
def test_codec_stats_match_the_oracle(dt, N, T):
    xs = _mixed(N, T, N * 7 + T, dt)
    comm = rra.Comm(N, T, xs[0].dtype)
    st = comm.codec_stats(xs)
    ref = O.codec_stats([host(x) for x in xs], dt)
    assert [st["elements"], st["nonzero"], st["bfp4_flushed"], st["bfp8_flushed"]] == list(ref)
    comm.close()


def test_advice_follows_the_rule():
    N, T = 8, 8 * 4096
    comm = rra.Comm(N, T, torch.bfloat16)
    sparse = W.sparse(N, T, seed=1)  # 60 % zeros
    codec, st = comm.advise_codec(sparse, sparsity_threshold=0.5)
    assert codec.kind == "sparse" and 1 - st["nonzero"] / st["elements"] > 0.5
    gauss = cast(rand_f32(N, T, seed=2), "bf16")  # BFP4 flushes a good share of N(0,1)
    codec, st = comm.advise_codec(gauss, max_flushed_fraction=0.01)
    assert st["bfp4_flushed"] > 0.01 * st["nonzero"]
    assert (codec.kind, codec.bits) == ("bfp", 8)
    codec, st = comm.advise_codec(gauss, max_flushed_fraction=1.0)
    assert (codec.kind, codec.bits) == ("bfp", 4)
    # a constant-magnitude signal loses nothing to the 4-bit code
    flat = [torch.full((T,), 0.5, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    codec, st = comm.advise_codec(flat)
    assert st["bfp4_flushed"] == 0 and (codec.kind, codec.bits) == ("bfp", 4)
    comm.close()


def test_advised_codec_runs_the_ring():
    """The advice is a plain codec: the ring runs with it, bit-exact."""
    N, T = 4, 4 * 2048
    xs = cast(rand_f32(N, T, seed=9, scale=1e-3), "f16")
    comm = rra.Comm(N, T, torch.float16)
    codec, _ = comm.advise_codec(xs)
    outs = [torch.zeros(T, device="cuda") for _ in range(N)]
    comm.ring_allreduce(xs, outs, codec)
    assert comm.status() == rra.RRA_OK
    ref = O.ring([host(x) for x in xs], "f16", "f32", codec=codec.kind, bits=codec.bits,
                 threshold=float(np.float32(codec.sparsity_threshold)))[0]
    for r in range(N):
        assert np.array_equal(host(outs[r]).view(np.uint32), ref[r].view(np.uint32))
    comm.close()


# ---------------------------------------------------------------- operator-aware choice

@pytest.mark.parametrize("op", ["allgather", "broadcast"])
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N,T", [(1, 300), (3, 1000), (8, 8 * 1000 + 3), (20, 20 * 130 + 11)])
def test_codec_stats_per_operation_match_the_oracle(op, dt, N, T):
    """What the compressed allgather (each owner's chunk) and broadcast (the
    root's buffer) encode, counted exactly as the oracle counts it."""
    xs = _mixed(N, T, seed=N + T + len(op), dt=dt)
    root = (N - 1) // 2
    comm = rra.Comm(N, T, xs[0].dtype)
    code = {"allgather": rra.RRA_OP_ALLGATHER, "broadcast": rra.RRA_OP_BROADCAST}[op]
    got = comm.codec_stats(xs, op=code, root=root)
    want = O.codec_stats_op([host(x) for x in xs], dt, op, root)
    assert [got[k] for k in ("elements", "nonzero", "bfp4_flushed", "bfp8_flushed")] == \
        [int(v) for v in want]
    comm.close()


def test_operator_aware_advice():
    """Allgather and broadcast take lossless sparse codes (allgather only),
    else BFP8 when lossy codes are allowed and flush little, else nothing;
    BFP4 is never advised for them.  The allreduce keeps its own rule."""
    N, T = 8, 8 * 4096
    comm = rra.Comm(N, T)
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    sparse = [torch.where(torch.rand(T, generator=g, device="cuda") < 0.2,
                          torch.randn(T, generator=g, device="cuda"), torch.zeros(T, device="cuda"))
              for _ in range(N)]
    smooth = [torch.randn(T, generator=g, device="cuda") for _ in range(N)]
    c, st = comm.advise_codec_op(rra.RRA_OP_ALLGATHER, sparse)
    assert c.kind == "sparse" and st["elements"] == T  # N owner chunks of T / N
    c, _ = comm.advise_codec_op(rra.RRA_OP_BROADCAST, sparse, root=3)
    assert c.kind in ("bfp", "none") and (c.kind == "none" or c.bits == 8)
    c, st = comm.advise_codec_op(rra.RRA_OP_ALLGATHER, smooth)
    flushed8 = st["bfp8_flushed"] <= 0.01 * st["nonzero"]
    assert (c.kind, c.bits) == (("bfp", 8) if flushed8 else ("none", 0))
    c, _ = comm.advise_codec_op(rra.RRA_OP_ALLGATHER, smooth, allow_lossy=False)
    assert c.kind == "none"
    c, st = comm.advise_codec_op(rra.RRA_OP_BROADCAST, smooth, root=0, max_flushed_fraction=1.0)
    assert (c.kind, c.bits) == ("bfp", 8) and st["elements"] == T
    c, _ = comm.advise_codec_op(rra.RRA_OP_BROADCAST, smooth, root=0, max_flushed_fraction=0.0)
    assert c.kind == ("bfp" if st["bfp8_flushed"] == 0 else "none")
    c_ar, _ = comm.advise_codec_op(rra.RRA_OP_ALLREDUCE, smooth)
    c_ref, _ = comm.advise_codec(smooth)
    assert (c_ar.kind, c_ar.bits) == (c_ref.kind, c_ref.bits)
    # the advised codec runs the compressed allgather unchanged
    bufs = [x.clone() for x in sparse]
    c, _ = comm.advise_codec_op(rra.RRA_OP_ALLGATHER, bufs)
    ref = O.allgather_codec([host(b) for b in bufs], "f32", c.kind, c.bits)[0]
    comm.allgather(bufs, codec=c)
    for q in range(N):
        assert np.array_equal(host(bufs[q]).view(np.uint32), ref[q].view(np.uint32))
    with pytest.raises(rra.RRAError):
        comm.advise_codec_op(rra.RRA_OP_BROADCAST, smooth, root=N)
    with pytest.raises(rra.RRAError):
        comm.advise_codec_op(7, smooth)
    comm.close()
