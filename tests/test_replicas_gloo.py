"""The multi-GPU path is replicas only (tokens are independent, no exchange
inside the layer): N ranks each run the whole workload and the benchmark
reports the slowest rank's time.  This runs that aggregation with two gloo
ranks on the CPU."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = 0.5 + rank            # rank 1 is the slow one
        job_s, value = bench.aggregate_replicas(local, steps=32, tokens_per_step=1, world=world)
        out[rank] = (job_s, value)
        # the reference arm runs on rank 0 only; other ranks return without work
        args = type("A", (), {"workload": "tiny", "steps": 1, "warmup": 1, "reference_budget_s": 0.0})()
        if rank != 0:
            assert bench.run_reference(args, rank, world) is None
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        job_s, value = res[rank]
        assert job_s == pytest.approx(1.5)                 # max over ranks
        assert value == pytest.approx(2 * 32 * 1 / 1.5)    # whole-job tokens over job time


def test_single_replica_is_local_time():
    job_s, value = bench.aggregate_replicas(0.25, steps=10, tokens_per_step=8, world=1)
    assert job_s == 0.25 and value == pytest.approx(320.0)
