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


def test_reference_arm_line_keeps_the_contract():
    # `bench.py --impl reference` on the host cores: one JSON line with the arm's metric,
    # unit and direction, its cpu_baseline and an e2e with no host<->device bytes
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.abspath(bench.__file__))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "3"], capture_output=True, text=True,
                         timeout=600, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["steps"] == 2 and line["warmup"] >= 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_algorithmic_bytes_of_the_workloads():
    # packed nibbles + E4M3 scales + x (bf16) + y (bf16) + the global scale, per call
    assert bench.algo_bytes(1, 5120, 17408) == 50_180_100     # decode, either shape
    assert bench.algo_bytes(1, 17408, 5120) == 50_180_100
    assert bench.algo_bytes(7, 5120, 34816) == 100_829_188    # MTP verify
    assert bench.algo_bytes(7, 5120, 6144) == 17_852_420
