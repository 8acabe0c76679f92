"""Host logic of bench.py's N > 1 path (independent replicas, one per GPU), on CPU with the
gloo backend and two ranks: max-over-ranks timing and the whole-job rate."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = [2.0, 3.5][rank]  # rank 1 is the slower replica
        ms_max = bench.max_over_ranks(torch, ms_local, world, "cpu")
        dist.barrier()
        out[rank] = (ms_max, bench.replica_rate(1.0e12, world, ms_max))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_rate():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 3.5
    # two replicas, each 1e12 units of work, done when the slower (3.5 ms) is
    assert out[0][1] == pytest.approx(2 * 1.0e12 / 3.5e-3)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(torch, 1.25, 1) == 1.25
    assert bench.replica_rate(10.0, 1, 2.0) == pytest.approx(5000.0)


def test_reference_arm_on_a_non_zero_rank_exits_quietly():
    """Under torchrun only rank 0 runs the oracle arm; other ranks exit 0 and print nothing."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
