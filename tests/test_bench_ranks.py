"""The benchmark's multi-rank logic on CPU, with two gloo ranks: every rank
runs an independent replica (own seed), the timed region is taken from the
slowest rank, the whole-job value adds the replicas' work, and the reference
arm runs on rank 0 alone."""
import argparse
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    # Rank r "took" 10 + 5 r ms: both ranks must report the slowest.
    ms = bench._max_over_ranks(10.0 + 5.0 * rank, dist, torch.device("cpu"))
    seed = bench._replica_seed(rank)
    ws, rk = bench._dist()
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, ms, seed, ws, rk))


def test_two_gloo_ranks_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]
    assert res[0][2] != res[1][2]                      # independent replicas
    assert [(r[3], r[4]) for r in res] == [(2, 0), (2, 1)]


def test_job_value_adds_the_replicas():
    import bench
    one = bench._job_tflops(1, 6e12, 10.0)
    assert one == pytest.approx(600.0)
    assert bench._job_tflops(2, 6e12, 10.0) == pytest.approx(2 * one)
    assert bench._job_tflops(2, 6e12, 20.0) == pytest.approx(one)  # slowest rank sets the time


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(argparse.Namespace(steps=1, warmup=0, ref_seconds=0.01))
    assert capsys.readouterr().out == ""
