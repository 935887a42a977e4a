"""The multi-replica timing of bench.py on CPU: two gloo ranks (the GEMV has
no exchange step, so N GPUs run N independent replicas; the bench reports the
slowest rank's time and the whole-job throughput)."""
from __future__ import annotations

import multiprocessing as mp
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(torch, dist, local_ms[rank], "cpu")
        dist.barrier()
        out.put((rank, ms, bench.whole_job_gbs(world, 41_297_920, ms)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    local_ms = [0.0150, 0.0175]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, local_ms, out)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in results] == [0, 1]
    for _, ms, gbs in results:
        assert ms == pytest.approx(0.0175)                    # max over ranks, on every rank
        assert gbs == pytest.approx(2 * 41_297_920 / 0.0175e-3 / 1e9)


def test_one_process_keeps_its_own_time():
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch
    import bench
    assert bench.max_over_ranks(torch, None, 0.0123, "cpu") == 0.0123
    assert bench.whole_job_gbs(1, 1e9, 1.0) == pytest.approx(1000.0)
