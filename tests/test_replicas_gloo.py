"""The multi-GPU path is replicas only (no data-path collective): each rank
runs its own copy of the workload and the job's time is the slowest rank's.
This checks that host logic with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow replica
        m = bench.max_over_ranks(local_ms)
        rate = bench.job_throughput(world, 2.0e9, 100, m)
        q.put((rank, m, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, m, rate in got:
        assert m == 15.0
        assert rate == pytest.approx(2 * 2.0e9 * 100 / 15e-3)


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(1, 10.0, 4, 2.0) == pytest.approx(10.0 * 4 / 2e-3)
