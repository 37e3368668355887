"""Host logic of the multi-rank benchmark mode on CPU (gloo, world size 2):
the barrier, the max-over-ranks time and the weak-scaling aggregate."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        bench.barrier(world)
        # rank r "measured" (r + 1) * 10 ms for its steps
        t = bench.max_over_ranks((rank + 1) * 10.0, world)
        out[rank] = t
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 20.0, 1: 20.0}


def test_weak_scaling_aggregate():
    import bench
    # two ranks, each 1e12 FLOP per step, 10 steps in 5 ms (slowest rank)
    v = bench.aggregate_tflops(1e12, 10, 5.0, 2)
    assert v == pytest.approx(2 * 1e12 * 10 / 5e-3 / 1e12)
    assert bench.aggregate_tflops(1e12, 10, 5.0, 1) == pytest.approx(v / 2)
    assert bench.max_over_ranks(3.5, 1) == 3.5
