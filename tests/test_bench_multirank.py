"""bench.py's multi-rank host logic on CPU with gloo, world size 2: the job
time is the slowest rank's, and the value counts every rank's tokens."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 100.0 * (rank + 1)  # rank 1 is the slow one
        value, ms_per_step = bench.aggregate_throughput(64, 10, mine, world)
        q.put((rank, bench.max_over_ranks(mine), value, ms_per_step))
    finally:
        dist.destroy_process_group()


def test_gloo_two_ranks_max_time_and_aggregate_value():
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
    for rank, mx, value, ms in res:
        assert mx == 200.0
        assert ms == pytest.approx(20.0)
        # 2 ranks x 64 tokens x 10 steps in 0.2 s
        assert value == pytest.approx(2 * 64 * 10 / 0.2)


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    v, ms = bench.aggregate_throughput(64, 4, 8.0, 1)
    assert ms == 2.0 and v == pytest.approx(64 * 4 / 0.008)
