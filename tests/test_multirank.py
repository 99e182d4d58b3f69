"""Multi-rank host logic of bench.py on CPU (gloo, world_size 2).

Rows are independent, so N GPUs run N copies of the workload with no
collective on the data path; the only cross-rank steps are the barrier around
the timed region and the max-over-ranks of the elapsed time. This checks those
steps and the whole-job aggregation with two CPU ranks.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench._barrier(world)
        mine = 1.0 + rank  # rank 1 is the slower rank
        slowest = bench._max_over_ranks(mine, world)
        value = bench.aggregate_value(bytes_per_step=1_000_000_000, steps=10, world=world,
                                      max_seconds=slowest)
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, slowest, value in res:
        assert slowest == 2.0                     # max over ranks, seen by every rank
        assert value == pytest.approx(10.0)       # 2 ranks x 10 steps x 1 GB / 2 s = 10 GB/s


def test_single_rank_defaults():
    import bench
    assert bench._max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate_value(2_000_000_000, 5, 1, 2.0) == pytest.approx(5.0)
