"""The replica path's host logic on two CPU ranks (gloo, 127.0.0.1): the time
bench.py reports is the slowest rank's, and the whole-job rate counts every
rank's units.  No GPU and no collective on the data path: the ranks only
reduce their timings."""
import os
import socket

import pytest

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = 1.0 + 0.5 * rank          # rank 1 is the slow replica
        t = bench.max_over_ranks(elapsed, world, torch.device("cpu"))
        q.put((rank, t, bench.job_rate(300.0, world, t)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.25, 1, None) == 3.25
    assert bench.job_rate(300.0, 1, 2.0) == 150.0


def test_two_ranks_take_the_slowest_time_and_count_all_units():
    torch_mp = pytest.importorskip("torch.multiprocessing")
    ctx = torch_mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=120)
    assert [p.exitcode for p in procs] == [0, 0]
    # both ranks report the slowest rank's 1.5 s and 2 x 300 units over it
    assert res == [(0, 1.5, 400.0), (1, 1.5, 400.0)]
