"""Pin the lossless oracle against torch.distributed's gloo collectives, the
check the collective-ops lesson ("从零实现集合通信") itself suggests: run each
primitive through gloo at the same world size on the same tensor and fail
above float32 epsilon.  gloo sums in its own order, so the comparison allows
the recursive-summation bound (N-1) u sum|x| on each element.  gloo's
broadcast and allgather are exact and are compared bit for bit, and so is the
compressed allgather against gloo gathering each chunk's BFP8 round trip.
World sizes 2 and 4, CPU processes, 127.0.0.1 rendezvous."""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import brute
import oracle as O

U = 2.0 ** -24


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, xs, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = torch.from_numpy(xs[rank].copy())
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    b = torch.from_numpy(xs[rank].copy())
    dist.broadcast(b, src=world - 1)
    parts = [torch.empty(xs[0].size // world, dtype=torch.float32) for _ in range(world)]
    n = xs[0].size // world
    dist.all_gather(parts, torch.from_numpy(xs[rank][rank * n:(rank + 1) * n].copy()))
    # compressed allgather: each rank's chunk goes through the BFP8 round trip
    # (the brute force's restatement of the codec) before gloo gathers it
    rt, _ = brute.bfp_roundtrip([np.float32(v) for v in xs[rank][rank * n:(rank + 1) * n]], 8)
    cparts = [torch.empty(n, dtype=torch.float32) for _ in range(world)]
    dist.all_gather(cparts, torch.tensor(rt, dtype=torch.float32))
    q.put((rank, t.numpy(), b.numpy(), torch.cat(parts).numpy(), torch.cat(cparts).numpy()))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_lossless_ops_agree_with_gloo(world):
    T = 4096
    rng = np.random.default_rng(world)
    xs = [rng.standard_normal(T).astype(np.float32) for _ in range(world)]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, xs, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    ours, _, _ = O.ring([x.copy() for x in xs])
    X = np.stack(xs).astype(np.float64)
    bound = (world - 1) * U * np.abs(X).sum(0) * (1 + 1e-6)
    exact = np.array([math.fsum(X[:, i]) for i in range(T)])
    for rank, red, bc, ag, cag in got:
        assert (np.abs(red.astype(np.float64) - ours[rank].astype(np.float64)) <= 2 * bound).all()
        assert (np.abs(ours[rank].astype(np.float64) - exact) <= bound).all()
        bufs, _, _ = O.broadcast([x.copy() for x in xs], "f32", root=world - 1)
        assert np.array_equal(bufs[rank].view(np.uint32), bc.view(np.uint32))
        gbufs, _, _ = O.allgather([x.copy() for x in xs], "f32")
        assert np.array_equal(gbufs[rank].view(np.uint32), ag.view(np.uint32))
        cbufs, _, _ = O.allgather_codec([x.copy() for x in xs], "f32", "bfp", 8)
        assert np.array_equal(cbufs[rank].view(np.uint32), cag.view(np.uint32))
