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


def test_roofline_time_takes_the_slower_bound():
    peak_tf, hbm = 3788.0, 6748.7
    # decode: weight stream dominates
    t = bench.roofline_time_s(1, 4096, 4096, False, peak_tf, hbm)
    assert t == pytest.approx((4096 * 4096 + 2 * 4096 + 4 + 2 * 4096) / (hbm * 1e9))
    # prefill: compute dominates
    t = bench.roofline_time_s(16384, 4096, 4096, True, peak_tf, hbm)
    assert t == pytest.approx(2.0 * 16384 * 4096 * 4096 / (peak_tf * 1e12))
