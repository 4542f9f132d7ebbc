"""The multi-GPU path is replicas only: every rank runs the whole decode step on
its own sequences, with no collective on the data path. What crosses ranks is
the bench's timing (the slowest replica's time, max over ranks) and the rule
that only rank 0 reports. Checked here with two gloo ranks on the CPU."""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", init_method="env://")
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        elapsed = [120.0, 150.0][rank]           # rank 1 is the slow replica
        job = bench.max_over_ranks(elapsed, "cpu")
        out[rank] = (job, bench.whole_job_rate(w, 36, 10, job))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time_and_add_their_work():
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
        assert all(p.exitcode == 0 for p in procs)
        res = dict(out)
    for r in range(world):
        job, rate = res[r]
        assert job == 150.0
        assert rate == pytest.approx(2 * 36 * 10 / 0.150)


def test_reference_arm_runs_on_rank_0_only(monkeypatch, capsys):
    import argparse

    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(argparse.Namespace(ref_seqs=1, steps=1, warmup=0))
    assert capsys.readouterr().out == ""
