"""bench.py's multi-rank bookkeeping on CPU with the gloo backend
(world_size 2): timings are reduced with max over ranks and the whole-job
value counts every rank's bytes.  The attention path has no collective."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [10.0 + rank, 2.0 * (world - rank), 0.5]
        got = bench.max_over_ranks(mine, dist)
        out[rank] = torch.tensor(got)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    world = 2
    port = _free_port()
    out = torch.zeros(world, 3).share_memory_()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        assert out[r].tolist() == [11.0, 4.0, 0.5]


def test_whole_job_value_is_weak_scaling():
    one = bench.whole_job_value(1, 10**9, 1.0)
    assert one == pytest.approx(1000.0)
    assert bench.whole_job_value(4, 10**9, 1.0) == pytest.approx(4 * one)


def test_single_process_max_is_identity():
    assert bench.max_over_ranks([1.5, 2.5], None) == [1.5, 2.5]
