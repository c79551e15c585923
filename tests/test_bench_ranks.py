"""The multi-rank host logic of bench.py on CPU (gloo, world size 2): the job's time is
the slowest rank's, the throughput counts every replica's bytes, and the reference arm
runs on rank 0 alone.  The GPU path itself is replicas only (no collective on the data
path); these are the pieces that differ from a single process."""
import multiprocessing as mp
import os
import socket

import pytest

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.5 + rank, dist, "cpu")  # rank 1 is the slower one
        dist.barrier()
        q.put((rank, ms, bench.job_gbps(1000, 10, world, ms)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2.5 for g in got)  # max of 1.5 and 2.5 ms on both ranks
    # 2 replicas x 10 steps x 1000 bytes in 2.5 ms
    assert all(g[2] == pytest.approx(2 * 10 * 1000 / 2.5e-3 / 1e9) for g in got)


def test_single_process_keeps_its_time():
    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25
    assert bench.job_gbps(100, 4, 1, 2.0) == pytest.approx(100 * 4 / 2e-3 / 1e9)


def test_reference_arm_runs_on_rank_zero_only():
    class A:
        steps, warmup = 1, 0
    assert bench.run_reference(A(), 1, 2) is None
