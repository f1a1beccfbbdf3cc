"""The multi-GPU path is replicas only (one process per GPU, no exchange on
the data path): the job takes as long as its slowest rank, and its value is
every rank's work over that time.  Checked with two gloo ranks on CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        total_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        m = bench.max_over_ranks(total_ms, torch.device("cpu"))
        rate = bench.job_rate(2048, world, 20, m)
        out[rank] = (m, rate)
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_count_every_rank():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as man:  # no fork of this threaded process
        out = man.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] == res[1][1] == pytest.approx(2048 * 2 * 20 / 15.0e-3)


def test_single_process_is_its_own_max():
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
    assert bench.job_rate(10, 1, 4, 2.0) == pytest.approx(10 * 4 / 2.0e-3)
