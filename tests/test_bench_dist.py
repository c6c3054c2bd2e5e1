"""The multi-rank arithmetic of bench.py (max over ranks, whole-job rate, rank-0-only
reference arm) on two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        # each rank times something different; every rank must see the slowest
        got = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        rate = bench.whole_job_rate(8 * 100, world, got / 1e3)
        ref = bench.run_reference(type("A", (), {"rows": 8, "steps": 1, "warmup": 1})()) if rank else None
        out.put((rank, got, rate, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
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
    for rank, got, rate, ref in res:
        assert got == 15.0  # max of 10 and 15 on both ranks
        assert rate == pytest.approx(2 * 800 / 0.015)  # all ranks' rows / slowest rank's time
        assert ref is None  # the reference arm runs on rank 0 only


def test_single_rank_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(80, 1, 2.0) == 40.0
