"""The N-rank path of the bench on CPU, with two gloo ranks.

The chain shards over independent rows with no exchange, so N GPUs run N
replicas: the only cross-rank steps are the barriers around the timed region
and the max over ranks of the time per step.  These tests run that host logic
in two real processes (gloo), and the reference arm under torchrun, where
rank 0 alone runs the oracle and prints the one JSON line."""
from __future__ import annotations

import argparse
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, per_rank_ms, flops, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    got_ws, got_rank, local = bench.dist_setup(argparse.Namespace(impl="reference"))
    try:
        bench.barrier(got_ws)
        ms = bench.max_over_ranks(per_rank_ms[rank], got_ws)
        bench.barrier(got_ws)
        out.put((got_rank, got_ws, local, ms, bench.whole_job_tflops(flops, ms, got_ws)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_all_work():
    ws, flops, per_rank_ms = 2, 3.0e12, [2.0, 5.0]
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    mp.start_processes(_rank, args=(ws, _free_port(), per_rank_ms, flops, out), nprocs=ws,
                       start_method="spawn", join=True)
    res = sorted(out.get() for _ in range(ws))
    assert [r[0] for r in res] == [0, 1]
    for rank, got_ws, local, ms, value in res:
        assert got_ws == ws and local == rank
        assert ms == max(per_rank_ms)
        # both ranks processed `flops` in the slowest rank's 5 ms: 2 * 3e12 / 5e-3 / 1e12
        assert value == pytest.approx(1200.0)


def test_whole_job_throughput_is_linear_in_ranks_at_fixed_step_time():
    one = bench.whole_job_tflops(1.0e12, 4.0, 1)
    assert one == pytest.approx(250.0)
    assert bench.whole_job_tflops(1.0e12, 4.0, 8) == pytest.approx(8 * one)


@pytest.mark.parametrize("kind,M,tile_m,expect", [
    ("gelu", 2048, 0, 256), ("gelu", 2048, 512, 256), ("gelu", 512, 0, 128),
    ("swiglu", 2048, 0, 128), ("swiglu", 2048, 512, 128), ("gelu", 2048, 128, 128),
    ("gelu", 2048, 256, 256)])
def test_replicas_use_no_cluster_multicast(kind, M, tile_m, expect):
    assert bench.replica_tile_m(2, tile_m, kind, M) == expect
    # one rank keeps whatever was asked, multicast tiles included
    assert bench.replica_tile_m(1, tile_m, kind, M) == tile_m


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    env = dict(os.environ, OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1", "--workload", "tiny"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [json.loads(s) for s in p.stdout.splitlines() if s.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
