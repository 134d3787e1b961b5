"""The host side of bench.py, on CPU: two gloo ranks, and the reference arm.

Under torchrun every rank runs an independent replica of the workload; the
job's step time is the largest over the ranks and its rate counts the units
of every replica.  The reference arm runs on rank 0 alone; the other ranks
leave without work or output, and rank 0 prints the contract's JSON line.
"""
import argparse
import contextlib
import io
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # per-rank step times: the slowest replica sets the job's time
        ms = bench.max_over_ranks(2.0 + 3.0 * rank)
        e2e = bench.max_over_ranks(7.5 if rank == 0 else 1.25)
        dist.barrier()
        out.put((rank, ms, e2e, bench.job_rate(dist.get_world_size(), 1000, ms / 1e3)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_replica():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    mp.start_processes(_rank_main, args=(world, port, q), nprocs=world, join=True,
                       start_method="spawn")
    got = sorted(q.get(timeout=60) for _ in range(world))
    for rank, ms, e2e, rate in got:
        assert ms == 5.0 and e2e == 7.5
        # 2 replicas x 1000 units in the slowest replica's 5 ms
        assert rate == pytest.approx(2 * 1000 / 5e-3)


def test_single_process_keeps_its_own_time():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_rate(1, 10, 2.0) == 5.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    import datagen
    args = argparse.Namespace(steps=1, warmup=0)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.run_reference(args, datagen.WORKLOADS["tiny_diag"])
    assert rc == 0 and buf.getvalue() == ""


def test_reference_arm_prints_the_contract_line(monkeypatch):
    """Rank 0 of the reference arm prints one JSON line with the bench's keys,
    the oracle's own throughput as value, cpu_baseline and e2e."""
    import json
    import datagen
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    # a small sample instead of the ~seconds-long calibration
    monkeypatch.setattr(bench, "cpu_sample_run", lambda wl, mix, s: (1.0, 512, 1, 0.01))
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.run_reference(argparse.Namespace(steps=2, warmup=1),
                                 datagen.WORKLOADS["tiny_diag"])
    assert rc == 0
    lines = buf.getvalue().strip().splitlines()
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and "512" in d["cpu_baseline"]["sample"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny_diag"
