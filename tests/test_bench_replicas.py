"""The multi-GPU form of the benchmark is "replicas only": every rank runs the
whole simulated ring on its own GPU, nothing is sharded and there is no
data-path collective.  What bench.py does across ranks is host logic -- a
barrier, the maximum of the per-rank step times, the whole-job value -- and
that is checked here with world size 2 on the gloo backend (CPU)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    ms = [0.25, 0.30][rank]  # rank 1 is the slow replica
    m = bench.max_over_ranks(world, ms)
    q.put((rank, m, bench.whole_job_gbs(world, 26_214_400, m)))
    dist.destroy_process_group()


def test_replica_aggregation_world_size_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v in got:
        assert m == pytest.approx(0.30)  # the max over ranks, seen by every rank
        assert v == pytest.approx(2 * 26_214_400 / 0.30e-3 / 1e9)


def test_single_replica_value():
    assert bench.whole_job_gbs(1, 26_214_400, 0.25) == pytest.approx(104.8576)
