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
import types

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


def _replica_rank(rank, ws, port, out):
    """One rank of an N-rank bench run, up to its plans: the environment torchrun
    gives it, then the binding (which picks the library build from WORLD_SIZE),
    then every plan desc the bench makes with ws ranks, resolved host-side."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    os.environ.pop("CS_CHAIN_LIBRARY", None)
    got_ws, _, _ = bench.dist_setup(argparse.Namespace(impl="reference"))  # gloo: no GPU here
    try:
        import cs_inputs
        import consumer_gemm_chain_gb300 as cs
        bench.check_replica_library(cs, got_ws)
        rec = {"lib": os.path.basename(cs.chain.LIB_PATH), "features": cs.cs_library_features(),
               "extras": bench.runs_extras(got_ws, False), "plans": [], "refused": []}
        cs.cs_tune_load()  # the bench's default: the shipped table, whose entries may name 512-row tiles
        for workload in ("gpt3", "llama", "stress", "tiny"):
            for M in sorted({cs_inputs.WORKLOADS[workload][4], 512, 1024, 2048}):
                for extra in ([], ["--tile-m", "512"], ["--tile-m", "256"], ["--policy", "stream"]):
                    args = bench.parse(["--workload", workload, "--M", str(M), "--gpus", str(got_ws)] + extra)
                    kind, H, F, dtype, _ = cs_inputs.WORKLOADS[workload]
                    inp = types.SimpleNamespace(kind=kind, H=H, F=F, dtype=dtype)
                    desc = bench.plan_desc(cs, args, inp, args.policy, M)
                    try:
                        q = cs.cs_chain_plan_info(desc, 152)
                        rec["plans"].append((workload, M, tuple(extra), q["tile_m"]))
                    except cs.CSError as e:
                        rec["refused"].append((workload, M, tuple(extra), e.status))
        out.put((rank, rec))
    finally:
        dist.destroy_process_group()


def test_replica_ranks_load_the_build_without_cluster_multicast():
    import __graft_entry__
    __graft_entry__._build_module().build()
    ws = 2
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    mp.start_processes(_replica_rank, args=(ws, _free_port(), out), nprocs=ws, start_method="spawn", join=True)
    res = dict(out.get() for _ in range(ws))
    assert sorted(res) == [0, 1]
    for rank, rec in res.items():
        assert rec["lib"] == "libcs_chain_nomc.so", rec["lib"]
        assert rec["features"] & 1 == 0  # CS_FEATURE_CLUSTER_MULTICAST
        assert rec["extras"] is False  # an N-rank run makes the headline plan only
        assert rec["plans"], "no plan resolved"
        # no plan of any workload resolves to 512-row (4-CTA multicast) tiles ...
        assert all(tm in (128, 256) for *_, tm in rec["plans"]), rec["plans"]
        # ... and asking for them is refused by the library, not silently changed
        assert rec["refused"] and all(extra == ("--tile-m", "512") and st == 2 for _, _, extra, st in rec["refused"])
        assert len(rec["refused"]) == len({(w, m) for w, m, _, _ in rec["plans"]})


def test_one_gpu_loads_the_full_build_and_keeps_its_tiles():
    import consumer_gemm_chain_gb300 as cs
    assert cs.chain.library_path({"WORLD_SIZE": "1"}).endswith("libcs_chain.so")
    assert cs.chain.library_path({}).endswith("libcs_chain.so")
    assert cs.chain.library_path({"WORLD_SIZE": "8"}).endswith("libcs_chain_nomc.so")
    assert cs.chain.library_path({"WORLD_SIZE": "8", "CS_CHAIN_LIBRARY": "full"}).endswith("libcs_chain.so")
    assert cs.chain.library_path({"CS_CHAIN_LIBRARY": "nomc"}).endswith("libcs_chain_nomc.so")
    with pytest.raises(ImportError):
        cs.chain.library_path({"CS_CHAIN_LIBRARY": "other"})
    assert bench.runs_extras(1, False) and not bench.runs_extras(1, True)
    if os.path.basename(cs.chain.LIB_PATH) == "libcs_chain.so":
        assert cs.cs_library_features() & cs.CS_FEATURE_CLUSTER_MULTICAST
        d = cs.cs_chain_desc_init(kind="gelu", M=2048, H=12288, F=6144, weight_layout="nk", tuned=-1)
        assert cs.cs_chain_plan_info(d, 152)["tile_m"] == 512


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
