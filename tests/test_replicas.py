"""The multi-GPU path is replicas only: each rank runs the whole stack on its own
token, the step time is the max over ranks and the job's time per token is that
over the rank count.  Checked with two gloo ranks on the CPU."""
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


def _rank(rank, world, port, times, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        us_step, value = bench.aggregate_ranks(torch, dist, times[rank], world, "cpu")
        out[rank] = (us_step, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_divide_by_world():
    times = [5000.0, 5400.0]
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(2, _free_port(), times, out), nprocs=2, join=True)
    for r in range(2):
        assert out[r] == (pytest.approx(5400.0), pytest.approx(2700.0))


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_ranks(torch, None, 5062.5, 1, "cpu") == (5062.5, 5062.5)
