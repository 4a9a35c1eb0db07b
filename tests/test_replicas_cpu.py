"""The multi-GPU mode is replicas only: one independent replica per rank, no
collective on the data path; the bench takes the slowest rank's time and
sums the work.  These tests run that host-side logic as world_size-2 `gloo`
ranks on the CPU."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [5.0, 7.25][rank]
        ms = bench.max_over_ranks(torch, local_ms, dist, "cpu")
        value = bench.replica_value(world, 1.0e12, 10, ms)
        dist.barrier()
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    assert sorted(out.keys()) == [0, 1]
    for r in range(world):
        ms, value = out[r]
        assert ms == 7.25                       # every rank sees the max
        assert value == pytest.approx(2 * 1.0e12 * 10 / 7.25e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(torch, 3.5, None, "cpu") == 3.5
    assert bench.replica_value(1, 2.0e12, 4, 8.0) == pytest.approx(1000.0)  # 8e12 FLOP in 8 ms


def test_reference_arm_on_a_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert res.returncode == 0
    assert res.stdout.strip() == ""


def test_replicas_draw_distinct_inputs():
    import synth
    a, _ = synth.fprop_inputs(device="cpu", seed=2, M=128, N=128, K=128)
    b, _ = synth.fprop_inputs(device="cpu", seed=2 + 1000, M=128, N=128, K=128)
    assert not torch.equal(a, b)
