"""The benchmark's multi-GPU path is replicas: every rank runs the whole layer
on its own GPU, ranks meet at a barrier, and the job's time is the slowest
rank's.  These host-side pieces run here as two gloo processes on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        my_ms = 100.0 + 10.0 * rank               # rank 1 is the slow one
        t = bench.reduce_max(my_ms, world)
        v = bench.aggregate_tops(4.0e12, 10, t, world)
        out.put((rank, t, v))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_time_and_aggregate_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in res:
        assert t == 110.0                          # max over ranks
        assert v == pytest.approx(2 * 4.0e12 * 10 / 0.110 / 1e12)


def test_single_rank_helpers_need_no_process_group():
    assert bench.reduce_max(3.5, 1) == 3.5
    bench.barrier(1)
    assert bench.aggregate_tops(1e12, 1, 1000.0, 1) == pytest.approx(1.0)
