"""The N > 1 host logic of bench.py on CPU: two gloo ranks (spawned
processes) agree on the max-over-ranks time and on the whole-job replica
rate; the CPU reference arm runs on rank 0 only."""
import argparse
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import multirank_worker  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_take_the_slowest_rank(tmp_path):
    pytest.importorskip("torch")
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=multirank_worker.bench_rank, args=(r, world, port, str(tmp_path)))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    for p in procs:
        if p.is_alive():
            p.kill()
            p.join()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    vals = [tuple(map(float, open(tmp_path / f"rank{r}.txt").read().split())) for r in range(world)]
    # rank 1 took 15 ms, rank 0 10 ms: both see 15 ms; 2 replicas x 1e9 units x 100 steps / 15 ms
    for ms_max, rate in vals:
        assert ms_max == 15.0
        assert rate == pytest.approx(2 * 1e9 * 100 / 0.015 / 1e9)


def test_job_rate_single_rank():
    assert bench.job_rate(1, 34799616, 1000, 20.0) == pytest.approx(34799616 * 1000 / 0.020 / 1e9)
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(steps=3, warmup=3, gpus=2, ref_seconds=1.0)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_the_contract_line(monkeypatch, capsys):
    """Rank 0 times the CPU oracle on a bounded sample and prints one JSON line
    with the reference arm's keys."""
    import json
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    args = argparse.Namespace(steps=3, warmup=3, gpus=1, ref_seconds=0.5)
    assert bench.run_reference(args) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "GB/s" and rec["value"] > 0
    assert rec["metric"] == bench.METRIC and rec["steps"] == 3 and rec["higher_is_better"] is True
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["value"] == rec["value"]
    assert rec["e2e"] == {"value": rec["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
