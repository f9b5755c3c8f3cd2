"""bench.py's multi-process (replica) aggregation on the CPU: two gloo ranks,
max time over ranks, units summed over ranks (no GPU)."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        assert (r, w, lr) == (rank, world, rank)
        t_local = 1.0 + rank                       # rank 1 is the slow one
        t = bench.dist_max(t_local, world)
        value, tmax = bench.aggregate([t], 100.0, world)
        bench.barrier(world)
        out[rank] = (t, value, tmax)
    finally:
        dist.destroy_process_group()


def test_replica_aggregation_two_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        t, value, tmax = out[r]
        assert t == 2.0 and tmax == 2.0
        assert value == pytest.approx(world * 100.0 / 2.0)


def test_aggregate_single():
    import bench
    v, t = bench.aggregate([0.5], 10.0, 1)
    assert v == 20.0 and t == 0.5
