"""The replica path of bench.py on CPU: two gloo ranks report different times; the job's time
is the slowest rank's, and the job throughput counts every rank's rows."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        slowest = bench.max_over_ranks(1.0 + rank)  # rank 1 is the slower replica
        q.put((r, ws, local, slowest, bench.job_rows_per_s(ws, 32, 10, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, (r, ws, local, slowest, value) in enumerate(res):
        assert (r, ws, local) == (rank, 2, rank)
        assert slowest == 2.0
        assert value == pytest.approx(2 * 32 * 10 / 2.0)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_rows_per_s(1, 32, 100, 0.5) == pytest.approx(6400.0)
