"""The N>1 host path of bench.py on CPU: world_size-2 gloo ranks (no GPU).
Each rank is an independent replica; the job time is the slowest rank's and
the job throughput counts both ranks' work.  The reference arm runs on rank 0
only; other ranks exit at once."""
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


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sec_local = 0.010 * (rank + 1)  # rank 1 is the slow one
        sec, value = bench.aggregate_over_ranks(sec_local, 1e12, world)
        q.put((rank, sec, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time_and_sum_work():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, sec, value in out:
        assert sec == pytest.approx(0.020)
        assert value == pytest.approx(2 * 1e12 / 0.020 / 1e12)


def test_single_rank_needs_no_process_group():
    import bench
    sec, value = bench.aggregate_over_ranks(0.5, 2e12, 1)
    assert sec == 0.5 and value == pytest.approx(4.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    import argparse

    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(workload=bench.MAIN, steps=1, warmup=3)
    assert bench.run_reference(args) == 0
