"""The multi-rank bookkeeping of bench.py on CPU (gloo, two ranks).

With N processes each rank times its own replica of the step; the job's
step time is the slowest rank's and the job's throughput is N times one
rank's bytes over that time.  The path itself never exchanges data
between ranks, so the only collectives are this max and the barriers.
"""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        q.put((rank, bench.max_over_ranks(local_ms[rank], world)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    world, local_ms = 2, [3.25, 7.5]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, local_ms, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(world))
    assert got == {0: 7.5, 1: 7.5}


def test_max_over_ranks_single_process():
    assert bench.max_over_ranks(2.5, 1) == 2.5


def test_job_throughput_is_weak_scaling_sum():
    # 1 GB per rank per step, 2 ms per step on the slowest of 4 ranks
    assert bench.job_gbs(1e9, 4, 2.0) == pytest.approx(2000.0)
    assert bench.job_gbs(1e9, 1, 2.0) == pytest.approx(500.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert bench.run_reference(args) is None
