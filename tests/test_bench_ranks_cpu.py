"""The multi-GPU path of bench.py on the host: replicas (one per rank) that
share nothing but the timing -- the job's time is the slowest rank's, and
its rate counts every rank's work.  Run as two gloo ranks on the CPU."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [40.0, 55.5][rank]  # rank 1 is the slower replica
        total = bench.max_over_ranks(torch, dist, local_ms, "cpu")
        out[rank] = (total, bench.job_throughput(world, 1e9, 10, total))
    finally:
        dist.destroy_process_group()


def test_two_ranks_time_is_the_slowest_and_rate_counts_both():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 55.5
    # 2 ranks x 1e9 units x 10 steps over 55.5 ms, in giga-units per second
    assert out[0][1] == pytest.approx(2 * 10 / 55.5e-3)


def test_reference_arm_prints_only_on_rank_zero(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    from workloads import make_config
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup, gpus = 2, 1, 2

    bench.reference_arm(Args(), make_config("tiny"))  # returns at once, no oracle work
    assert capsys.readouterr().out == ""


def test_reference_arm_line_keeps_the_contract(monkeypatch, capsys):
    # the oracle timed as the reference arm: one JSON line with the keys the
    # driver reads, on the decode workload's metric and config
    import json
    sys.path.insert(0, ROOT)
    import bench
    from workloads import make_config
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setattr(bench, "REFERENCE_BUDGET_S", 0.5)

    class Args:
        steps, warmup, gpus = 2, 1, 1

    bench.reference_arm(Args(), make_config("llama-decode"))
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["metric"] == "decode KV-read GB/s" and line["unit"] == "GB/s"
    assert line["config"]["workload"] == "llama-decode" and line["value"] > 0 and line["higher_is_better"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
