"""The multi-GPU path's host logic on two CPU ranks (gloo, world size 2).

The indexer shards by request with no exchange step: each rank runs its own
replica and only the timing is reduced (max over ranks).  This checks that
reduction and the whole-job us/call it feeds, with real torch.distributed
ranks on the gloo backend.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        mine = [3.0, 7.5][rank]           # per-rank device time (ms) of 10 calls
        mx = bench.reduce_max(mine, world, "cpu")
        us = bench.whole_job_us_per_call(mx, 10, world)
        q.put((rank, mx, us))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, mx, us in got:
        assert mx == 7.5                    # the slowest rank's time
        assert us == pytest.approx(7.5e3 / 20)  # 20 calls over both ranks


def test_single_rank_identity():
    import bench
    assert bench.reduce_max(4.25, 1, "cpu") == 4.25
    assert bench.whole_job_us_per_call(4.25, 17, 1) == pytest.approx(4250 / 17)
