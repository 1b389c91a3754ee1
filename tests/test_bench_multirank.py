"""The benchmark's multi-GPU path is N independent replicas timed between
barriers, reported as the slowest rank.  Its aggregation runs here on CPU
with two gloo ranks (no GPU)."""
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
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local_ms = 2.0 if rank == 0 else 3.5          # rank 1 is the slow replica
        bench.barrier(world)
        step_ms, us_per_call = bench.whole_job_us_per_call(local_ms, world, torch.device("cpu"))
        q.put((rank, step_ms, us_per_call))
    finally:
        dist.destroy_process_group()


def test_replicas_report_the_slowest_rank_and_whole_job_throughput():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, step_ms, us in res:
        assert step_ms == pytest.approx(3.5)          # max over ranks
        assert us == pytest.approx(3.5e3 / 2)         # two calls per job step


def test_single_rank_is_plain_time_per_call():
    import bench
    step_ms, us = bench.whole_job_us_per_call(1.25, 1, torch.device("cpu"))
    assert step_ms == 1.25 and us == pytest.approx(1250.0)
