"""The N-rank path of bench.py on CPU: two gloo ranks, each timing its own replica
(requests are sharded across ranks; the step has no collective). The job's time is
the slowest rank's and its throughput counts every rank's drafted tokens."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = [3.0, 5.0][rank]  # rank 1 is the slow one
    worst = bench.world_max(ms, world, "cpu")
    value = bench.job_throughput(16 * 4, world, worst)
    dist.barrier()
    q.put((rank, worst, value))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_tokens():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(world))
    for _, worst, value in out:
        assert worst == 5.0
        assert value == pytest.approx(2 * 64 / 5e-3)


def test_single_rank_is_identity():
    import bench

    assert bench.world_max(2.5, 1, "cpu") == 2.5
    assert bench.job_throughput(32, 1, 2.0) == pytest.approx(16000.0)
