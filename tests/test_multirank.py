"""The multi-process host logic of bench.py on CPU: two `gloo` ranks.

The path shards into replicas (one process per GPU, each on its own seeded copy
of the workload; no data-path collective).  What the ranks share is host
logic: the torchrun environment, a per-rank seed, the max over ranks of the
timed figures (the job takes as long as its slowest rank) and the whole-job
throughput.  These tests run that logic in two real processes."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.rank_env()
        # each rank times a different step; the job's figures are the maxima
        ms, idx_ms = bench.max_over_ranks([2.0 + rank, 1.5 - 0.5 * rank], w, "cpu")
        value = bench.job_value(1376, w, ms)
        out.put((r, w, local, bench.rank_seed(7, r), ms, idx_ms, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_every_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert [r[:3] for r in res] == [(0, 2, 0), (1, 2, 1)]
    assert res[0][3] != res[1][3]                              # each replica draws its own inputs
    for r in res:
        assert r[4] == 3.0 and r[5] == 1.5                     # max over ranks, element by element
        assert r[6] == pytest.approx(2 * 1376 / 3e-3)          # both ranks' units over the slowest time


def test_single_process_defaults():
    assert bench.rank_env({}) == (0, 1, 0)
    assert bench.max_over_ranks([1.25, 2], 1, "cpu") == [1.25, 2.0]
    assert bench.job_value(10, 1, 2.0) == pytest.approx(5000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(None, None) == 0                # other ranks exit without work

