"""The N-GPU bench runs N independent replicas: timing is the maximum over
ranks and throughput counts every rank's units.  Checked with two gloo ranks
on the CPU (no GPU, no data-path collective)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(times[rank], dist, "cpu")
        q.put((rank, slowest, bench.replica_throughput(16 * 100, world, slowest)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_throughput():
    world, port = 2, _free_port()
    times = [0.50, 0.75]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, slowest, value in got:
        assert slowest == pytest.approx(0.75)
        assert value == pytest.approx(2 * 1600 / 0.75)


def test_single_process_needs_no_collective():
    assert bench.max_over_ranks(0.3) == 0.3
    assert bench.replica_throughput(10, 1, 2.0) == 5.0
