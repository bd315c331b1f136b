"""The multi-GPU bench path on CPU: two gloo ranks, no GPU.

Every rank runs an independent request (weak scaling); the job's time is the
slowest rank's and the value counts every rank's decode steps.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, totals, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import sys
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        total, value = bench.whole_job_value(totals[rank], 128, 10, world, torch.device("cpu"))
        out[rank] = (total, value, bench.rank_seed(0x5EED, rank))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_every_rank():
    world, port = 2, _free_port()
    totals = [50.0, 80.0]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, totals, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        total, value, _ = res[r]
        assert total == 80.0
        assert value == pytest.approx(world * 128 * 10 / 0.080)
    assert res[0][2] != res[1][2]          # independent shards


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    total, value = bench.whole_job_value(40.0, 128, 5, 1, torch.device("cpu"))
    assert total == 40.0 and value == pytest.approx(128 * 5 / 0.040)
