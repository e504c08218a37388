"""The bench's multi-rank aggregation (max time over ranks, whole-job rate) on
two gloo ranks over 127.0.0.1, CPU only."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 + 3.0 * rank)      # rank 1 is the slow one
        results[rank] = (ms, bench.whole_job_rate(world, 8, 20, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_on_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        ms, rate = results[r]
        assert ms == pytest.approx(13.0)
        assert rate == pytest.approx(2 * 8 * 20 / 13.0e-3)


def test_single_process_aggregation_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5) == 7.5
    assert bench.whole_job_rate(1, 8, 20, 10.0) == pytest.approx(16000.0)
