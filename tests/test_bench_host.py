"""bench.py host logic that needs no GPU: the single-GPU guard and the roofline arithmetic."""

import json
import os
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra, *argv):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *argv], env=env, capture_output=True,
                          text=True, timeout=120)


def test_more_than_one_process_is_refused_without_gpu_work():
    """Under torchrun with two ranks, rank 0 prints one 'unavailable' line and no rank runs the
    library (this container has no GPU: any device work would fail)."""
    r0 = _run({"RANK": "0", "WORLD_SIZE": "2", "LOCAL_RANK": "0"}, "--steps", "1", "--warmup", "0")
    assert r0.returncode == 0
    line = json.loads(r0.stdout.strip())
    assert line["n_gpus"] == 2 and "unavailable" in line
    r1 = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--steps", "1", "--warmup", "0")
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r2 = _run({}, "--gpus", "2")
    assert r2.returncode == 0 and "unavailable" in json.loads(r2.stdout.strip())


def test_reference_arm_on_a_non_zero_rank_exits_quietly():
    """Under torchrun only rank 0 runs the oracle arm; other ranks exit 0 and print nothing."""
    r = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--impl", "reference", "--steps", "1",
             "--warmup", "0")
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line_on_the_host():
    """The reference arm (the oracle on the host cores, no GPU) prints the contract's line: the
    metric, a positive value, a cpu_baseline of kind oracle and an e2e entry in the same unit."""
    r = _run({}, "--impl", "reference", "--steps", "1", "--warmup", "0", "--m", "64", "--cpu-rows", "4",
             "--cpu-cols", "32")
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["n_gpus"] == 1
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] >= 1 and line["cpu_baseline"]["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert line["config"]["M"] == 64 and "M=64" in line["config"]["workload"]


def test_roofline_time_takes_the_slower_bound():
    peak_tf, hbm = 3788.0, 6748.7
    # decode: weight stream dominates
    t = bench.roofline_time_s(1, 4096, 4096, False, peak_tf, hbm)
    assert t == pytest.approx((4096 * 4096 + 2 * 4096 + 4 + 2 * 4096) / (hbm * 1e9))
    # prefill: compute dominates
    t = bench.roofline_time_s(16384, 4096, 4096, True, peak_tf, hbm)
    assert t == pytest.approx(2.0 * 16384 * 4096 * 4096 / (peak_tf * 1e12))
