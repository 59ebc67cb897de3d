"""The bench's multi-rank logic on the host: two gloo ranks on the CPU.

One process per GPU runs an independent replica; the step time is the
maximum over ranks, the throughput counts every rank's work, and the
reference arm runs on rank 0 alone.  No GPU is used.
"""
import os
import socket
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        seconds = bench.max_over_ranks(0.5 + rank, torch.device("cpu"))  # rank 1 is the slower one
        out.put((rank, seconds, bench.job_tflops(2e12, seconds, world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    ctx = torch.multiprocessing.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest rank's time; the job did 2 x 2e12 FLOP in 1.5 s
    assert [r[1] for r in res] == [1.5, 1.5]
    for r in res:
        assert r[2] == pytest.approx(2 * 2e12 / 1.5 / 1e12)


def test_single_process_is_its_own_maximum():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_tflops(1e12, 0.5, 1) == pytest.approx(2.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import argparse

    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = argparse.Namespace(workload=bench.DEFAULT_WORKLOAD, steps=1, warmup=0)
    assert bench.run_reference(args) is None  # returns at once, no oracle work
