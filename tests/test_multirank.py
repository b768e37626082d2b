"""The multi-rank bench path on CPU: two gloo ranks (127.0.0.1).

The path has no exchange step; under torchrun every rank scores its own
replica and bench.py reduces the timed region with a max over ranks.  These
tests run that reduction and the whole-job throughput on a real two-process
gloo group, and check that the reference arm does its work on rank 0 only.
"""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, lr = bench.dist_info()
        assert (ws, r, lr) == (world, rank, rank)
        bench.barrier(world)
        ms = 10.0 + 5.0 * rank                    # rank 1 is the slow one
        m = bench.max_over_ranks(ms, world, torch.device("cpu"))
        out[rank] = (m, bench.job_throughput(4096, 20, m, world))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_rank_time_reduction_and_throughput():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0] == out[1]
    m, v = out[0]
    assert m == 15.0
    assert v == pytest.approx(2 * 4096 * 20 / 0.015)


def test_single_rank_needs_no_group():
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.job_throughput(10, 2, 1000.0, 1) == 20.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class A:
        steps, warmup, workload, gpus = 3, 1, 1, 2
    assert bench.run_reference(A()) is None
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_the_contract_line(monkeypatch, capsys):
    """The reference arm (the float64 oracle on the host cores) prints one
    JSON line with the contract's keys, on the tiny workload here."""
    import json
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)

    class A:
        steps, warmup, workload, gpus = 2, 3, 0, 1
    bench.run_reference(A())
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 2
    assert line["config"]["workload"].startswith("tiny")
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_own_peak_of_block_scaled_lines():
    """Block-scaled lines are judged against the rate of their own MMAs:
    kind::mxf8f6f4 runs at twice the bf16 rate (4.5 against 2.25 PFLOP/s
    nominal), and the KL with a block-scaled teacher does half its flops at
    each rate, one after the other on the tensor pipe."""
    P = {"bf16_tflops": 1800.0, "bf16_tflops_sustained": 1600.0}
    assert bench.own_peak(P, "bf16") == 1800.0
    assert bench.own_peak(P, "mx") == 3600.0
    assert bench.own_peak(P, "mx", sustained=True) == 3200.0
    # time for F flops, half at b and half at 2b: F/2/b + F/2/(2b) = 3F/(4b)
    assert abs(bench.own_peak(P, "bf16+mx") - 2400.0) < 1e-9
    assert set(bench.PEAK_KIND) == {"bf16", "mx", "bf16+mx"}
