"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

bench.py under torch.distributed.run gives every rank its own copy of the
workload (the (sequence, head) units are independent, so no data-path
collective exists) and only reduces the step time: the job's time is the
slowest rank's, and the job's throughput counts every rank's tokens.  These
tests run that logic as two gloo processes on the host."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from gated_deltanet_chunked_device_gb300 import workloads as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        ms = 1.0 + rank * 0.5                       # rank 1 is the slow one
        dist.barrier()
        job_ms = bench.max_over_ranks(ms, dist)
        w = wl.custom(seq_lens=[130, 0, 20], hq=2, hk=2, hv=4)
        inp = wl.generate(w, seed=3)                # every rank draws the same replica
        digest = float(inp["q"].float().sum() + inp["g"].sum() + inp["beta"].sum())
        digests = [None] * world
        dist.all_gather_object(digests, digest)
        results[rank] = (job_ms, bench.job_tokens_per_s(world, inp["T"], job_ms), digests)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_time_and_count_all_tokens():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        mp.start_processes(_worker, args=(world, _free_port(), results), nprocs=world, start_method="spawn")
        res = dict(results)
    assert sorted(res) == [0, 1]
    for rank in range(world):
        job_ms, tps, digests = res[rank]
        assert job_ms == pytest.approx(1.5)        # max over ranks
        assert tps == pytest.approx(2 * 150 / 1.5e-3)
        assert digests[0] == digests[1]            # identical replicas


def test_single_process_passes_values_through():
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.job_tokens_per_s(1, 1000, 2.0) == pytest.approx(5e5)
