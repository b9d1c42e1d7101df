"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

bench.py under torch.distributed.run either gives every rank its own copy of
the workload (--shard replica) or splits one batch's state heads over the
ranks (--shard heads); the (sequence, head) units are independent, so no
data-path collective exists either way, and only the step time is reduced:
the job's time is the slowest rank's.  These tests run that logic as two gloo
processes on the host."""
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
        assert tps == pytest.approx(2 * 150 / 1.5e-3)      # two copies of the batch
        assert digests[0] == digests[1]            # identical replicas


def test_single_process_passes_values_through():
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.job_tokens_per_s(1, 1000, 2.0) == pytest.approx(5e5)


def _shard_worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = wl.WORKLOADS["gva_8seq_ckpt512_bf16"]              # 16 q/k heads, 32 v (= state) heads
        full = wl.generate(wl.custom(seq_lens=[70, 5], hq=w.hq, hk=w.hk, hv=w.hv), seed=4)
        ws, part = bench.shard_heads(w, full, rank, world)
        ranges = bench.head_shard(full["H"], w.hq, w.hk, w.hv, rank, world)
        # the shard is the same problem shape with every head count halved, holding this rank's heads
        assert (ws.hq, ws.hk, ws.hv, part["H"]) == (w.hq // world, w.hk // world, w.hv // world, full["H"] // world)
        a, b = ranges["h"]
        assert torch.equal(part["g"], full["g"][:, a:b]) and torch.equal(part["beta"], full["beta"][:, a:b])
        for key in ("q", "k", "v"):
            qa, qb = ranges[key]
            assert torch.equal(part[key], full[key][:, qa:qb]) and part[key].is_contiguous()
        # state head h of the shard reads the same q / k / v heads as state head a + h of the whole batch
        H, Hs = full["H"], part["H"]
        for h in range(Hs):
            for key, n, ns in (("q", w.hq, ws.hq), ("k", w.hk, ws.hk), ("v", w.hv, ws.hv)):
                assert ranges[key][0] + h // (Hs // ns) == (a + h) // (H // n)
        gathered = [None] * world
        dist.all_gather_object(gathered, ranges)
        results[rank] = gathered
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_split_the_state_heads_exactly():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        mp.start_processes(_shard_worker, args=(world, _free_port(), results), nprocs=world, start_method="spawn")
        res = dict(results)
    assert sorted(res) == [0, 1]
    gathered = res[0]
    assert gathered == res[1]
    w = wl.WORKLOADS["gva_8seq_ckpt512_bf16"]
    for key, n in (("h", max(w.hq, w.hv)), ("q", w.hq), ("k", w.hk), ("v", w.hv)):
        covered = sorted(r[key] for r in gathered)
        assert covered[0][0] == 0 and covered[-1][1] == n      # the ranges tile [0, n) ...
        for (a0, b0), (a1, b1) in zip(covered, covered[1:]):
            assert b0 == a1                                    # ... without gap or overlap


def test_head_shard_refuses_heads_that_do_not_divide():
    with pytest.raises(ValueError):
        bench.head_shard(32, 16, 16, 32, 0, 3)
    assert bench.head_shard(32, 32, 16, 16, 3, 4) == {"h": (24, 32), "q": (24, 32), "k": (12, 16), "v": (12, 16)}
