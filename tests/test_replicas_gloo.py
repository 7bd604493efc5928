"""Host logic of the replica benchmark (one process per GPU, no collective on
the data path): the slowest rank's time is the job's time and the throughput
counts the units of every rank. Two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [12.5, 20.0][rank]  # rank 1 is the slow one
        out[rank] = bench.max_over_ranks(ms, torch.device("cpu"))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert out[0] == pytest.approx(20.0) and out[1] == pytest.approx(20.0)


def test_job_throughput_counts_every_rank():
    # 2 replicas, each 100 tokens, slowest 50 ms -> 4000 tokens/s for the job
    assert bench.job_throughput(100, 2, 50.0) == pytest.approx(4000.0)
    assert bench.job_throughput(100, 1, 50.0) == pytest.approx(2000.0)
