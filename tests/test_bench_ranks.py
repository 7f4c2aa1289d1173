"""The multi-rank path of bench.py on CPU: two gloo ranks, replicas only (no data
exchange), the job time is the slowest rank's and the value sums the ranks' tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = bench.job_ms(10.0 + 5.0 * rank, world, torch.device("cpu"))
        out[rank] = (ms, bench.job_value(world, 128, ms))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_step():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == (15.0, pytest.approx(2 * 128 / 0.015))


def test_one_rank_needs_no_process_group():
    import bench
    assert bench.job_ms(3.0, 1, torch.device("cpu")) == 3.0
    assert bench.job_value(1, 128, 2.0) == pytest.approx(64000.0)
