"""Benchmark of the fused, tile-synchronised MLP chain on GB300.

Headline: TFLOP/s of one fused chain forward of the GPT-3 175B 8-way MLP shard
(X[2048,12288] -> W1[12288,6144] + b1, GeLU -> W2[6144,12288], fp16 in, fp32
accumulate), TileSync policy, inputs resident in HBM.  One "step" is one chain
forward (every step of the hot path: dispatch, producer GEMM + bias/GeLU
epilogue + release, consumer wait + GEMM + store).

Also reported on the same line: the roofline of the kernel, the two-kernel
stream-ordered control (plain and captured in a CUDA graph), the best
standalone GEMM times (this library's and cuBLAS through torch), the effective
sync overhead (chain time minus the best standalone GEMMs, after the Flux
summary's ECT idea), a sweep over M, an end-to-end number through the C ABI
with host buffers, and the fp64 CPU oracle timed on the host cores.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload gpt3|stress|llama]
                        [--M M] [--policy tile|row|strided|stream] [--quick] [--impl reference]
"""
from __future__ import annotations

import argparse
import contextlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def strip_comments(src: str) -> str:
    """C/C++ source without its comments and with runs of whitespace collapsed
    (string and character literals kept as written)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_sha():
    """sha256[:16] of what fixes the kernel's memory traffic apart from the
    schedule: the device code (comments removed) and the kernel configurations
    the host instantiates (ring depths and stage sizes)."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "consumer_gemm_chain_gb300", "csrc")
    for f in ("cs_kernel.cuh", "cs_ptx.cuh"):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(strip_comments(fh.read()).encode())
    with open(os.path.join(csrc, "cs_chain.cu"), encoding="utf-8") as fh:
        for m in re.finditer(r"constexpr int NS_\w+ = [^;]*;", strip_comments(fh.read())):
            h.update(m.group(0).encode())
    return h.hexdigest()[:16]


def schedule_sha(cs, desc, num_sms):
    """sha256[:16] of the dispatch order a plan of `desc` runs on num_sms SMs
    (tiles, K-splits, groups and their order: the rest of what fixes traffic)."""
    import hashlib
    import struct
    units = cs.cs_schedule_build(desc, num_sms)
    return hashlib.sha256(struct.pack(f"<{len(units)}I", *units)).hexdigest()[:16]


def measured_traffic(key, sched_sha):
    """DRAM bytes per launch recorded by ncu for this workload, while the kernel
    and the plan's schedule are still the ones the counters were taken with."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    rec = d.get("records", {}).get(key)
    if d.get("kernel_sha") != kernel_sha() or not rec or rec.get("schedule_sha") != sched_sha:
        return None
    return rec.get("bytes_per_launch")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="gpt3", choices=["gpt3", "stress", "llama", "tiny", "attn"])
    ap.add_argument("--M", type=int, default=None)
    ap.add_argument("--policy", default="tile", choices=["tile", "row", "strided", "stream"])
    ap.add_argument("--layout", default="nk", choices=["kn", "nk"],
                    help="weight storage: nk = [N, K] (torch.nn.Linear), kn = [K, N]")
    ap.add_argument("--lag", type=int, default=-1)
    ap.add_argument("--tile-n", type=int, default=0)
    ap.add_argument("--group-m", type=int, default=0)
    ap.add_argument("--tile-m", type=int, default=0)
    ap.add_argument("--split-k", type=int, default=0)
    ap.add_argument("--prefetch", type=int, default=0, help="L2 prefetch distance (0 auto, -1 off)")
    ap.add_argument("--raster", type=int, default=0,
                    help="0 auto, 1 column-major, 2 row-major in a group, 3 K-range-major split consumers")
    ap.add_argument("--pdl", type=int, default=0, help="programmatic dependent launch: 0 auto (on), 1 on, -1 off")
    ap.add_argument("--tuning", default="default",
                    help="tuning table for the plans' auto fields: 'default' (the package's table, when "
                         "present), 'none' (built-in rules only) or a path")
    ap.add_argument("--quick", action="store_true", help="headline kernel only (profiling runs)")
    ap.add_argument("--solo-vs-cublas", type=int, default=None, metavar="STAGE",
                    help="profiling aid: launch stage STAGE of the chain alone once, then the cuBLAS GEMM "
                         "of the same shape (via torch) once, and exit; no other kernel runs")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU-oracle sample time")
    return ap.parse_args(argv)


# ------------------------------------------------------------------ workload arithmetic
def chain_flops(kind, M, H, F):
    """Algorithmic flops of one chain forward (a multiply-add counts 2)."""
    if kind == "gelu":
        return 4.0 * M * H * F
    if kind == "swiglu":
        return 6.0 * M * H * F
    if kind == "attn":
        # QKV projection, Q K^T and P V over the causal half (key j <= query i),
        # output projection; F = heads x head_dim
        return 2.0 * M * H * 3 * F + 2.0 * M * (M + 1) * F + 2.0 * M * F * H
    raise ValueError(kind)


def chain_bytes(kind, M, H, F, esz=2):
    """Algorithmic HBM bytes of one chain forward: weights once, X, Y, bias, and
    every intermediate (H; for attention QKV and O) written once and read once."""
    if kind == "gelu":
        return esz * (2 * H * F + F + 2 * M * H + 2 * M * F)
    if kind == "swiglu":
        return esz * (3 * H * F + 2 * M * H + 2 * M * F)
    if kind == "attn":
        return esz * (4 * H * F + 2 * M * H + 2 * M * 3 * F + 2 * M * F)
    raise ValueError(kind)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.monotonic(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        """Median SM clock, max clock and throttle reasons of the samples taken
        inside [t0, t1]; with none inside (a timed region shorter than the
        sampling period), sm_mhz is None: samples of the idle GPU around the
        region would not show the clock under load."""
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        used = inside

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[0]) for s in used if num(s[0]) is not None]
        mx = [num(s[1]) for s in used if num(s[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in used:
            for name, v in zip(names, s[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        mx_all = [num(s[1]) for _, s in self.samples if num(s[1]) is not None]
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(mx) if mx else (max(mx_all) if mx_all else None),
               "reasons": sorted(reasons), "samples_in_timed_region": len(inside)}
        if not inside:
            out["note"] = "no clock sample fell inside the timed region (shorter than the 100 ms sampling period)"
        return out


# ------------------------------------------------------------------ timing helpers
def sampled_calls(steps, most=200):
    """{call index: event-pair slot} for at most `most` calls spread evenly over `steps`."""
    every = max(1, -(-steps // most))
    return {i: k for k, i in enumerate(range(0, steps, every))}


def time_loop(fn, steps, warmup, stream, finish=None):
    """Mean ms per call of fn over `steps` calls (after `warmup`), CUDA events on `stream`,
    plus the mean of per-call event pairs (the kernel's average launch duration) on up
    to 200 calls spread evenly over the timed region (the clock under the power cap
    drifts during it).  `finish` (if any) runs after the last call, before the end
    event (e.g. to make `stream` wait for work queued on other streams)."""
    import torch
    for _ in range(warmup):
        fn()
    if finish is not None:
        finish()
    torch.cuda.synchronize()
    slot = sampled_calls(steps)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in slot]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(steps):
        k = slot.get(i)
        if k is not None:
            ev[k][0].record(stream)
        fn()
        if k is not None:
            ev[k][1].record(stream)
    if finish is not None:
        finish()
    end.record(stream)
    torch.cuda.synchronize()
    total = start.elapsed_time(end) / steps
    per = statistics.mean(a.elapsed_time(b) for a, b in ev)
    return total, per


def warm_up(fn, warm_ms=100.0, min_calls=3):
    """Back-to-back calls of fn for at least warm_ms of device time.  Under the
    power cap the SM clock follows the power drawn over the last tens of
    milliseconds (measured: a fused chain timed right after the lighter
    two-kernel control ran 4-6 % faster than the same plan timed after another
    fused chain), so every timing starts from fn's own steady state."""
    import torch
    s = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n, spent = min_calls, 0.0
    while True:
        a.record(s)
        for _ in range(n):
            fn()
        b.record(s)
        torch.cuda.synchronize()
        spent += a.elapsed_time(b)
        if spent >= warm_ms:
            return
        n = min(2 * n, 4096)


def simple_time(fn, iters=100, warm_ms=100.0, repeats=3):
    """Median over `repeats` of the mean ms per call of fn over `iters` back-to-back
    calls (CUDA events on the current stream, after warm_up); the median keeps a
    momentary clock dip out of difference metrics such as the overhead."""
    import torch
    s = torch.cuda.current_stream()
    warm_up(fn, warm_ms)
    runs = []
    for _ in range(repeats):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(iters):
            fn()
        b.record(s)
        torch.cuda.synchronize()
        runs.append(a.elapsed_time(b) / iters)
    return statistics.median(runs)


def interleaved_times(fns, rounds=5):
    """Median ms per call of each fn, timed in interleaved rounds (all of them
    then see the same drift of the clock under the power cap); round r starts
    at the r-th fn, and each timing starts with its own warm_up."""
    names = list(fns)
    runs = {name: [] for name in names}
    for r in range(rounds):
        for i in range(len(names)):
            name = names[(r + i) % len(names)]
            runs[name].append(simple_time(fns[name], repeats=1))
    return {name: statistics.median(v) for name, v in runs.items()}


# ------------------------------------------------------------------ CPU oracle timing
def time_cpu_oracle(inp, target_s):
    """Time the fp64 oracle on a bounded row sample of the workload; returns
    (flop/s, rows, seconds, rows used, oracle output for those rows)."""
    import oracle
    rows = 8
    while True:
        t0 = time.perf_counter()
        Y = _oracle_rows(oracle, inp, list(range(rows)))
        dt = time.perf_counter() - t0
        if dt >= target_s or rows >= inp.M:
            break
        rows = min(inp.M, max(rows * 2, int(rows * target_s / max(dt, 1e-3) * 1.1)))
    fl = chain_flops(inp.kind, rows, inp.H, inp.F)
    return fl / dt, rows, dt, Y


def _oracle_rows(oracle, inp, rows):
    if inp.kind == "gelu":
        return oracle.mlp_gelu(inp.X[rows], inp.W1, inp.b1, inp.W2)
    if inp.kind == "attn":
        # causal: the first r output rows depend on the first r input rows only
        assert rows == list(range(len(rows)))
        return oracle.attention_chain(inp.X[: len(rows)], inp.Wqkv, inp.Wo, heads=inp.F // 128, head_dim=128)
    return oracle.mlp_swiglu(inp.X[rows], inp.Wg, inp.Wu, inp.W2)


def cpu_cores():
    """Host threads the oracle's BLAS may use: the CPUs this process may run on,
    capped by an explicit thread limit (torchrun sets OMP_NUM_THREADS=1)."""
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var, "")
        if v.isdigit() and int(v) > 0:
            return min(n, int(v))
    return n


# ------------------------------------------------------------------ distributed
def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    return ws, rank, local


def runs_extras(ws, quick):
    """The side measurements (controls, solo stages, cuBLAS, sweeps, the CPU
    oracle) run on one GPU only: an N-rank run times the headline chain alone."""
    return ws == 1 and not quick


def check_replica_library(cs, ws):
    """An N-rank run must have loaded the replica build (no TMA cluster
    multicast in it); the binding picks it from WORLD_SIZE."""
    if ws > 1 and cs.cs_library_features() & cs.CS_FEATURE_CLUSTER_MULTICAST:
        raise SystemExit(f"{ws} ranks but {os.path.basename(cs.chain.LIB_PATH)} has cluster multicast; "
                         "the replica build libcs_chain_nomc.so must be loaded")


def whole_job_tflops(flops_per_rank, ms_max, ws):
    """Whole-job throughput of N replicas: every rank does the same work, and the
    slowest rank's time per step bounds the job."""
    return ws * flops_per_rank / (ms_max * 1e-3) / 1e12


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, ws, device=None):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_tuning(cs, which):
    """Loads the tuning table the plans' auto fields come from; returns a record
    for the JSON line."""
    cs.cs_tune_clear()
    if which == "none":
        return {"table": None, "entries": 0}
    path = cs.chain.TUNE_TABLE if which == "default" else which
    if which == "default" and not os.path.exists(path):
        return {"table": None, "entries": 0}
    n = cs.cs_tune_load(path)
    return {"table": os.path.relpath(path, ROOT), "entries": n}


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    """The fp64 CPU oracle as the reference arm: same metric, workload and unit."""
    ws, rank, _ = dist_setup(args)
    try:
        if rank == 0:
            _reference_line(args)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


def _reference_line(args):
    import cs_inputs
    import oracle
    M = args.M or cs_inputs.WORKLOADS[args.workload][4]
    inp = cs_inputs.make_inputs(args.workload, M=M, seed=0)
    per_step = max(0.5, min(10.0, 60.0 / max(1, args.steps + args.warmup)))
    # size the row sample so one step is about `per_step` seconds
    fl, rows, dt, _ = time_cpu_oracle(inp, per_step)
    rows_list = list(range(rows))
    for _ in range(args.warmup):
        _oracle_rows(oracle, inp, rows_list)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_rows(oracle, inp, rows_list)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    value = chain_flops(inp.kind, rows, inp.H, inp.F) / dt / 1e12
    sample = f"first {rows} of {M} rows per step (rows are independent), numpy float64 BLAS"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload, M, inp, args.policy),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


METRIC = "MLP-chain TFLOP/s & % roofline vs M on 1 GB300; sync overhead vs best solo GEMMs"
STEADY_S = 1.5  # seconds of the steady-state timing beside a short timed region


def workload_config(name, M, inp, policy, layout="nk"):
    desc = {"gpt3": "GPT-3 175B 8-way TP MLP shard", "stress": "last-wave stress two-GEMM GeLU chain",
            "llama": "LLaMA 65.2B 8-way TP SwiGLU shard", "tiny": "tiny MLP chain",
            "attn": "GPT-3 attention shard (QKV GEMM, 12-head causal attention, output projection)"}[name]
    return {"workload": f"{desc}: X[{M},{inp.H}] -> F={inp.F} -> H={inp.H}, {str(inp.dtype).split('.')[-1]}, "
                        f"policy={policy}",
            "M": M, "H": inp.H, "F": inp.F, "policy": policy, "accumulate": "fp32",
            "weights": "[N, K] row-major (torch.nn.Linear)" if layout == "nk" else "[K, N] row-major",
            "l2": "inputs larger than L2 (weights alone exceed the 126 MB L2), no flush"}


# ------------------------------------------------------------------ our arm
def plan_desc(cs, args, inp, policy, M, pdl=None, tuned=0, out_release=0):
    """The desc of a plan of the bench's workload `inp` with M rows, the command
    line's choices applied."""
    extra = dict(heads=inp.F // 128, head_dim=128) if inp.kind == "attn" else {}
    return cs.cs_chain_desc_init(kind=inp.kind, M=M, H=inp.H, F=inp.F, dtype=inp.dtype, policy=policy,
                                 weight_layout=args.layout, lag=args.lag, tile_n=args.tile_n, group_m=args.group_m,
                                 tile_m=args.tile_m, split_k=args.split_k, prefetch=args.prefetch,
                                 raster=args.raster, pdl=args.pdl if pdl is None else pdl, tuned=tuned,
                                 out_release=out_release, **extra)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch

    import consumer_gemm_chain_gb300 as cs
    import cs_inputs

    ws, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    tuning = load_tuning(cs, args.tuning)
    device = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    M = args.M or cs_inputs.WORKLOADS[args.workload][4]
    inp = cs_inputs.make_inputs(args.workload, M=M, seed=0)
    kind = inp.kind
    lay = args.layout
    check_replica_library(cs, ws)

    def w(t):
        t = t if lay == "kn" else t.t().contiguous()
        return t.to(device)

    X = inp.X.to(device)
    dev = {"X": X}
    if kind == "gelu":
        dev.update(W1=w(inp.W1), b1=inp.b1.to(device), W2=w(inp.W2))
    elif kind == "swiglu":
        dev.update(Wg=w(inp.Wg), Wu=w(inp.Wu), W2=w(inp.W2))
    else:
        dev.update(Wqkv=w(inp.Wqkv), Wo=w(inp.Wo))
    Y = torch.empty_like(X)

    def make_plan(policy, MM=M, pdl=None, tuned=0, out_release=0):
        return cs.cs_chain_plan(plan_desc(cs, args, inp, policy, MM, pdl, tuned, out_release))

    plan = make_plan(args.policy)
    plan_info = cs.cs_chain_query(plan)
    stream = torch.cuda.current_stream()
    if args.solo_vs_cublas is not None:
        solo_vs_cublas(cs, torch, plan, plan_info, dev, Y, inp, lay, args.solo_vs_cublas)
        return

    def step():
        if kind == "attn":
            cs.cs_attn_chain_forward(plan, X, dev["Wqkv"], dev["Wo"], Y)
        else:
            cs.cs_mlp_forward(plan, Y=Y, **dev)

    flops = chain_flops(kind, M, inp.H, inp.F)
    nbytes = chain_bytes(kind, M, inp.H, inp.F)
    launches_per_step = 2 if args.policy == "stream" else 1

    # ---- headline timed region
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    # the warm-up steps run right before the timed ones (no idle gap between
    # them, in which the clock would rise above its level under load)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(ws)
    t_wall0 = time.monotonic()
    ms_total, ms_launch = time_loop(step, args.steps, 0, stream)
    t_wall1 = time.monotonic()
    barrier(ws)
    # A timed region shorter than a second is a burst: the SM clock has not yet
    # settled under the power cap.  Beside it, one GPU also times the same step
    # for at least STEADY_S seconds (reported apart; `value` stays the K steps).
    steady = None
    if ws == 1 and ms_total * args.steps < 1000.0 * STEADY_S and not args.quick:
        n_steady = max(args.steps, int(STEADY_S * 1e3 / max(ms_total, 1e-3)) + 1)
        t_s0 = time.monotonic()
        ms_s, ms_s_launch = time_loop(step, n_steady, 0, stream)
        t_s1 = time.monotonic()
        steady = {"value": flops / (ms_s * 1e-3) / 1e12, "unit": "TFLOP/s", "steps": n_steady, "ms_per_step": ms_s,
                  "launch_ms": ms_s_launch, "seconds": ms_s * n_steady / 1e3}
    if sampler:
        time.sleep(0.15)
        sampler.stop()
        if steady is not None:
            steady["clocks"] = sampler.summary(t_s0, t_s1)
    st = cs.cs_chain_status(plan)
    if st != cs.CS_OK:
        raise RuntimeError(f"device status {cs.STATUS_NAMES.get(st)}: {cs.cs_last_error_string()}")
    ms_step = max_over_ranks(ms_total, ws, device)
    value = whole_job_tflops(flops, ms_step, ws)

    timed_s = ms_total * args.steps / 1e3
    sustained = timed_s >= 1.0
    tc_peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]  # fp16 dense rate = bf16 rate
    hbm_peak = peaks["hbm_gbs"]
    achieved = flops / (ms_launch * 1e-3) / 1e12
    t_roof_ms = max(flops / (tc_peak * 1e12), nbytes / (hbm_peak * 1e9)) * 1e3
    bound = "tensor" if flops / (tc_peak * 1e12) >= nbytes / (hbm_peak * 1e9) else "hbm"
    if bound == "tensor":
        roof = {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": achieved / tc_peak}
    else:
        gbs = nbytes / (ms_launch * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak}
    traffic_key = f"{args.workload}_M{M}_{args.policy}_{lay}"
    roof.update({"traffic": measured_traffic(traffic_key, schedule_sha(cs, plan.desc, plan_info["num_sms"])),
                 "peak_source": f"{peak_src} ({'sustained' if sustained else 'burst'})",
                 "kernel": kernel_label(kind, M, plan_info),
                 "algorithmic_flops_per_launch": flops if launches_per_step == 1 else None,
                 "algorithmic_bytes_per_launch": nbytes if launches_per_step == 1 else None,
                 "launch_ms": ms_launch, "roofline_time_ms": t_roof_ms})

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16" if inp.dtype == torch.float16 else "bf16", "data": "synthetic",
        "config": dict(workload_config(args.workload, M, inp, args.policy, lay), parallelism=f"replicas{ws}",
                       tile_n=plan_info["tile_n"][:2], tile_m=plan_info["tile_m"], group_m=plan_info["group_m"],
                       lag=plan_info["lag"], pdl=args.pdl >= 0,
                       split_k=plan_info["split_k"][:plan_info["stages"]], raster=plan_info["raster"],
                       grid=plan_info["num_sms"], tuning=dict(tuning, entry=plan_info["tuned_entry"])),
        "roofline": roof, "gpu_launches": args.steps * launches_per_step,
    }
    if sampler:
        line["clocks"] = sampler.summary(t_wall0, t_wall1)
    if steady is not None:
        tc_s = peaks["bf16_tflops_sustained"]
        steady["roofline"] = {"achieved": flops / (steady["launch_ms"] * 1e-3) / 1e12, "peak": tc_s,
                              "frac": flops / (steady["launch_ms"] * 1e-3) / 1e12 / tc_s,
                              "peak_source": f"{peak_src} (sustained)"} if bound == "tensor" else None
        line["steady_state"] = steady

    # ---- end to end through the C ABI with host buffers
    Xh = inp.X.pin_memory()
    Yh = torch.empty(Y.shape, dtype=Y.dtype).pin_memory()

    # through the host-memory entry point: every step copies its X in and its Y
    # out (pinned buffers); the copies of consecutive steps overlap the kernels
    wts = {k: v for k, v in dev.items() if k != "X"}

    if kind == "attn":
        # the attention chain has no host-memory entry point: each step copies
        # X in, runs the chain and copies Y out on the stream, in series
        def e2e_step():
            X.copy_(Xh, non_blocking=True)
            step()
            Yh.copy_(Y, non_blocking=True)
        finish, api = None, "cs_attn_chain_forward with the X upload and Y read-back on the same stream"
    else:
        def e2e_step():
            cs.cs_mlp_forward_host(plan, X=Xh, Y=Yh, **wts)
        finish, api = (lambda: cs.cs_chain_host_join(plan, stream)), \
            "cs_mlp_forward_host (double-buffered copies on two copy streams)"

    e2e_ms, _ = time_loop(e2e_step, max(3, min(args.steps, 200)), 3, stream, finish=finish)
    e2e_ms = max_over_ranks(e2e_ms, ws, device)
    line["e2e"] = {"value": whole_job_tflops(flops, e2e_ms, ws), "unit": "TFLOP/s",
                   "h2d_bytes_per_step": Xh.numel() * Xh.element_size(),
                   "d2h_bytes_per_step": Yh.numel() * Yh.element_size(), "ms_per_step": e2e_ms, "api": api}

    if rank == 0 and runs_extras(ws, args.quick) and kind != "attn":
        line["extras"] = extras(cs, torch, inp, dev, Y, make_plan, plan, M, kind, peaks, stream)
        if args.workload == "gpt3":
            line["extras"]["other_configs"] = other_configs(cs, torch, peaks, lay)
        fl, rows, dt, Yref = time_cpu_oracle(inp, args.cpu_seconds)
        import oracle
        Yg = Yh[:rows] if rows <= Yh.shape[0] else Yh
        line["parity_rel_err_rows"] = oracle.rel_err(Yg[:rows], Yref)
        line["cpu_baseline"] = {"value": fl / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": f"first {rows} of {M} rows, {dt:.1f} s, numpy float64 BLAS"}
    cs.cs_chain_destroy(plan)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def solo_vs_cublas(cs, torch, plan, info, dev, Y, inp, lay, stage):
    """One launch of an MLP chain's stage alone and one of cuBLAS's GEMM of that
    stage's shape (stage 0 as addmm + GeLU), for an ncu capture of both kernels.
    The inputs are copied from the host, so no other kernel runs before them."""
    import torch.nn.functional as Fn
    if inp.kind != "gelu" or stage not in (0, 1):
        raise SystemExit("--solo-vs-cublas: stage 0 or 1 of a GeLU MLP workload")
    cs.cs_chain_forward_stage(plan, stage, Y=Y, **dev)
    t = (lambda w: w) if lay == "kn" else (lambda w: w.t())
    if stage == 0:
        Fn.gelu(torch.addmm(dev["b1"], dev["X"], t(dev["W1"])), approximate="tanh")
    else:
        Hbuf = torch.empty(inp.M, inp.F, dtype=inp.dtype, device=Y.device)
        torch.mm(Hbuf, t(dev["W2"]), out=Y)
    torch.cuda.synchronize()
    st = cs.cs_chain_status(plan)
    print(json.dumps({"solo_vs_cublas": stage, "M": inp.M, "tile_m": info["tile_m"], "tile_n": info["tile_n"][:2],
                      "status": cs.STATUS_NAMES.get(st)}))
    if st != cs.CS_OK:
        raise SystemExit(1)


def _union_len(iv, lo=None, hi=None):
    """Length of the union of intervals iv, clipped to [lo, hi]."""
    total, cur = 0, None
    for a, b in sorted(iv):
        if lo is not None:
            a, b = max(a, lo), min(b, hi)
            if b <= a:
                continue
        if cur is None or a > cur[1]:
            if cur is not None:
                total += cur[1] - cur[0]
            cur = [a, b]
        else:
            cur[1] = max(cur[1], b)
    return total + (cur[1] - cur[0] if cur else 0)


def sm_busy_stats(recs, n_sm):
    """Tensor-pipe occupancy of one kernel launch from its trace records (8
    integers: unit | index << 32, SM | ..., then ns at claim, dependencies
    published, first TMA load, last TMA load, accumulator complete, epilogue
    done).  An SM counts as busy while one of its units is between its first
    load and its accumulator (the mainloop: the span in which its MMAs run).
    The tail is the window from the moment the first SM has finished the
    mainloop of its last unit to the end of the launch: the last wave, in which
    SMs fall idle while others still work."""
    per_sm = {}
    t0 = min(r[2] for r in recs if r[2])
    t1 = max(r[7] for r in recs if r[7])
    for r in recs:
        if r[4] and r[6]:
            per_sm.setdefault(r[1] & 0xFFFF, []).append((r[4], r[6]))
    span = t1 - t0
    busy = sum(_union_len(iv) for iv in per_sm.values())
    # The tail is measured over the SMs that ran units: SMs that host no CTA
    # of a cluster shape (a GPC whose SM count is not a multiple of the
    # cluster size) are idle for the whole launch and are reported apart.
    used = len(per_sm)
    last = [max(b for _, b in iv) for iv in per_sm.values()]
    tail0 = min(last) if last else t1
    tail = t1 - tail0
    tail_busy = sum(_union_len(iv, tail0, t1) for iv in per_sm.values())
    return {"span_us": span / 1e3, "busy_frac": busy / (n_sm * span) if span else None,
            "busy_frac_used_sms": busy / (used * span) if span and used else None,
            "idle_sm_us": (n_sm * span - busy) / 1e3, "tail_us": tail / 1e3,
            "tail_busy_frac": tail_busy / (used * tail) if tail > 0 and used else None,
            "tail_idle_sm_us": (used * tail - tail_busy) / 1e3, "sms_used": used, "sms_unused": n_sm - used,
            "t_start": t0, "t_end": t1}


def traced_forward(cs, torch, plan, fwd):
    """Trace records of one forward of `plan` (fwd runs it)."""
    cs.cs_chain_debug_trace(plan, True)
    fwd()
    torch.cuda.synchronize()
    recs = cs.cs_chain_debug_read_trace(plan)
    cs.cs_chain_debug_trace(plan, False)
    return recs


def tail_stats(cs, torch, plan, fwd):
    """SM occupancy of one traced forward: per launch (one for a fused policy;
    the producer and the consumer launch of the two-kernel control) and for the
    whole forward, with the gap between the control's launches."""
    q = cs.cs_chain_query(plan)
    n_sm = q["num_sms"]
    recs = [r for r in traced_forward(cs, torch, plan, fwd) if r[2]]
    if q["policy"] != "stream":
        st = sm_busy_stats(recs, n_sm)
        st.pop("t_start"), st.pop("t_end")
        return {"launches": [st], "whole": st}
    by_stage = {}
    for r in recs:
        by_stage.setdefault(cs.decode_unit(r[0] & 0xFFFFFFFF)[0], []).append(r)
    launches = [sm_busy_stats(by_stage[s], n_sm) for s in sorted(by_stage)]
    whole = sm_busy_stats(recs, n_sm)
    gaps = [(b["t_start"] - a["t_end"]) / 1e3 for a, b in zip(launches, launches[1:])]
    for st in launches + [whole]:
        st.pop("t_start"), st.pop("t_end")
    whole["gaps_us"] = gaps
    return {"launches": launches, "whole": whole}


def rs_standin(cs, torch, make_plan, Y, dev, M, chunks=8):
    """Single-GPU stand-in for a GEMM + reduce-scatter fusion (Flux summary): the
    chain with its output released per 128-row block (desc.out_release), timed
    against the plain chain, and the per-unit timeline of one traced forward:
    when each of `chunks` row chunks of Y (one per destination rank) is complete,
    as a fraction of the kernel's span from the first unit claimed to the last
    tile stored.  A chunk-wise collective could send chunk r from then on."""
    fwd = lambda p: cs.cs_mlp_forward(p, Y=Y, **dev)  # noqa: E731
    with make_plan("tile") as p0, make_plan("tile", out_release=1) as p1:
        t = interleaved_times({"plain": lambda: fwd(p0), "out_release": lambda: fwd(p1)})
        cs.cs_chain_debug_trace(p1, True)
        fwd(p1)
        torch.cuda.synchronize()
        recs = cs.cs_chain_debug_read_trace(p1)
        q = cs.cs_chain_query(p1)
        cs.cs_chain_debug_trace(p1, False)
        st = cs.cs_chain_status(p1)
    if st != cs.CS_OK:
        return {"error": f"device status {cs.STATUS_NAMES.get(st)}"}
    rec = chunk_ready(recs, q["stages"] - 1, q["tile_m"], M, chunks, cs.decode_unit)
    rec.update({"chain_ms": t["plain"], "chain_out_release_ms": t["out_release"],
                "release_cost_frac": t["out_release"] / t["plain"] - 1.0})
    return rec


def chunk_ready(recs, last, tile_m, M, chunks, decode):
    """From trace records (8 integers: unit | index << 32, SM, then ns at claim,
    ..., epilogue done): the time each of `chunks` equal row chunks of the output
    is complete (its last tile of the last stage stored), as a fraction of the
    span from the first claim to the last epilogue."""
    ready = {}
    for r in recs:
        stage, m_tile, _, _ = decode(r[0] & 0xFFFFFFFF)
        if stage == last and r[7]:
            ready[m_tile] = max(ready.get(m_tile, 0), r[7])
    start = min(r[2] for r in recs if r[2])
    end = max(r[7] for r in recs if r[7])
    frac = []
    for c in range(chunks):
        lo, hi = c * M // chunks, (c + 1) * M // chunks
        tiles = range(lo // tile_m, (hi - 1) // tile_m + 1) if hi > lo else []
        frac.append(max(((ready[m] - start) / (end - start) for m in tiles), default=0.0))
    return {"chunks": chunks, "chunk_ready_frac": [round(f, 3) for f in frac],
            "overlap_window_frac": sum(1.0 - f for f in frac) / chunks, "kernel_span_us": (end - start) / 1e3}


def extras(cs, torch, inp, dev, Y, make_plan, plan, M, kind, peaks, stream):
    """Control, graph control, solo stages, cuBLAS solo GEMMs, sync overhead, M sweep."""
    import torch.nn.functional as Fn
    out = {}
    fwd = lambda p: cs.cs_mlp_forward(p, Y=Y, **dev)  # noqa: E731
    for pol in ("row", "strided", "stream"):
        with make_plan(pol) as p:
            out[f"{pol}_ms"] = simple_time(lambda: fwd(p))
    # without programmatic dependent launch: each launch waits for the previous
    # grid to finish before its CTAs start (the plain two-stream-kernel control)
    for pol in ("tile", "stream"):
        with make_plan(pol, pdl=-1) as p:
            out[f"{'chain' if pol == 'tile' else pol}_nopdl_ms"] = simple_time(lambda: fwd(p))
    # control captured in a CUDA graph (launch cost amortised)
    with make_plan("stream") as pc:
        fwd(pc)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fwd(pc)
        out["stream_graph_ms"] = simple_time(g.replay)
        ok = cs.cs_chain_status(pc)
        out["stream_graph_status"] = cs.STATUS_NAMES.get(ok)
        del g
    # best standalone GEMMs: this library's stage kernels and cuBLAS via torch.
    # The overhead is a difference of timings, so its terms are timed in
    # interleaved rounds (chain, stages, cuBLAS) and each takes its median:
    # all of them then see the same clock under the power cap.
    X = dev["X"]
    Hbuf = torch.empty(M, inp.F, dtype=inp.dtype, device=X.device)
    if kind == "gelu":
        W1 = dev["W1"] if plan.desc.weight_layout == 0 else dev["W1"].t()
        W2 = dev["W2"] if plan.desc.weight_layout == 0 else dev["W2"].t()
        cub1 = lambda: Fn.gelu(torch.addmm(dev["b1"], X, W1), approximate="tanh")  # noqa: E731
    else:
        Wg = dev["Wg"] if plan.desc.weight_layout == 0 else dev["Wg"].t()
        Wu = dev["Wu"] if plan.desc.weight_layout == 0 else dev["Wu"].t()
        W2 = dev["W2"] if plan.desc.weight_layout == 0 else dev["W2"].t()
        cub1 = lambda: Fn.silu(X @ Wg) * (X @ Wu)  # noqa: E731
    terms = {"chain": lambda: fwd(plan),
             "stage0": lambda: cs.cs_chain_forward_stage(plan, 0, Y=Y, **dev),
             "stage1": lambda: cs.cs_chain_forward_stage(plan, 1, Y=Y, **dev),
             "cublas0": cub1,
             "cublas1": lambda: torch.mm(Hbuf, W2, out=Y)}
    med = interleaved_times(terms)
    chain_ms = med["chain"]
    out["chain_ms"] = chain_ms
    solo = [med["stage0"], med["stage1"]]
    c1, c2 = med["cublas0"], med["cublas1"]
    out["solo_stage_ms"] = solo
    out["cublas_ms"] = [c1, c2]
    best = [min(solo[0], c1), min(solo[1], c2)]
    out["best_solo_ms"] = best
    out["sync_overhead_ms"] = chain_ms - sum(best)
    out["sync_overhead_frac"] = (chain_ms - sum(best)) / chain_ms
    out["beats_control"] = chain_ms < out["stream_ms"]
    try:
        out["reduce_scatter_standin"] = rs_standin(cs, torch, make_plan, Y, dev, M)
    except Exception as e:  # a side measurement that fails must not cost the bench line
        out["reduce_scatter_standin"] = {"error": repr(e)[:300]}
    # sweep over M (first M rows of the same draw)
    sweep = []
    tc, hbm = peaks["bf16_tflops"], peaks["hbm_gbs"]
    Ms = (1, 16, 64, 256, 512, 1024, 2048) if inp.H == 12288 else tuple(128 * b for b in range(1, 13))
    for m in Ms:
        if m > M:
            continue
        sub = {k: (v[:m].contiguous() if k == "X" else v) for k, v in dev.items()}
        Ym = torch.empty(m, inp.H, dtype=inp.dtype, device=X.device)
        rec = {"M": m}
        with contextlib.ExitStack() as es:
            fns = {}
            for pol, pdl, key, tuned in (("tile", None, "tile", 0), ("stream", None, "stream", 0),
                                         ("stream", -1, "stream_nopdl", 0), ("tile", None, "tile_builtin", -1)):
                p = es.enter_context(make_plan(pol, m, pdl, tuned))
                if key == "tile":
                    rec["plan"] = plan_record(cs.cs_chain_query(p))
                fns[key] = (lambda p=p: cs.cs_mlp_forward(p, Y=Ym, **sub))
            for key, ms in interleaved_times(fns).items():
                rec[f"{key}_us"] = ms * 1e3
        fl = chain_flops(kind, m, inp.H, inp.F)
        by = chain_bytes(kind, m, inp.H, inp.F)
        roof_ms = max(fl / (tc * 1e12), by / (hbm * 1e9)) * 1e3
        rec["tflops"] = fl / (rec["tile_us"] * 1e-6) / 1e12
        rec["roofline_frac"] = roof_ms / (rec["tile_us"] * 1e-3)
        rec["bound"] = "tensor" if fl / (tc * 1e12) >= by / (hbm * 1e9) else "hbm"
        rec["beats_control"] = rec["tile_us"] < rec["stream_us"]
        sweep.append(rec)
    out["sweep"] = sweep
    return out


def stream_k_remainder(q):
    """Tiles of the last stage left over after whole waves of a plan's units
    (0 when the plan splits its last stage or fills its waves)."""
    last = q["stages"] - 1
    if q["split_k"][last] != 1:
        return 0
    rem = sum(q["sched_units"][: q["stages"]]) % q["workers"]
    return rem if rem <= q["sched_units"][last] else 0


def kernel_label(kind, M, q):
    """The instantiation a plan launches (the library's configuration rules:
    up to 8 rows on single SMs, 11 stages of 17 KB or, with 256-wide B, 5 of
    33 KB; up to 32 rows 9 of 20 KB or 5 of 36 KB; 256-wide B otherwise 4
    stages of 48 KB; else 6 of 32 KB)."""
    wide_b = kind == "swiglu" or 256 in q["tile_n"][: q["stages"]]
    if kind == "attn":
        return f"cs_chain_kernel<6,32768,{q['tile_m'] // 128},1> (attention)"
    if q["tile_m"] == 512:
        return "cs_chain_kernel<6,32768,2,0,4> (4-CTA clusters)"
    if q["tile_m"] == 256:
        return "cs_chain_kernel<6,32768,2>"
    if M <= 8:
        return "cs_chain_kernel<5,33792,1,0,1,8>" if wide_b else "cs_chain_kernel<11,17408,1,0,1,8>"
    if M <= 32:
        return "cs_chain_kernel<5,36864,1,0,1,32>" if wide_b else "cs_chain_kernel<9,20480,1,0,1,32>"
    return "cs_chain_kernel<4,49152,1>" if wide_b else "cs_chain_kernel<6,32768,1>"


def plan_record(q):
    """Tile shape, K-splits, unit order and tuning entry of a plan, for the sweep records."""
    return {"tile_m": q["tile_m"], "tile_n": q["tile_n"][q["stages"] - 1], "split_k": max(q["split_k"]),
            "splits": q["split_k"][: q["stages"]], "raster": q["raster"], "sk_tiles": q["sk_tiles"],
            "tuned_entry": q["tuned_entry"]}


def _roof_frac(fl, by, us, peaks):
    tc, hbm = peaks["bf16_tflops"], peaks["hbm_gbs"]
    t_roof = max(fl / (tc * 1e12), by / (hbm * 1e9))
    return t_roof / (us * 1e-6), ("tensor" if fl / (tc * 1e12) >= by / (hbm * 1e9) else "hbm")


def other_configs(cs, torch, peaks, lay):
    """The other workloads of the sweep: LLaMA SwiGLU shard and the attention chain
    vs M (fused vs two-kernel control), and the last-wave stress sweep with every
    policy.  Rows of each M are the first M rows of the largest draw."""
    import cs_inputs
    dev_of = lambda t: (t if lay == "kn" else t.t().contiguous()).cuda()  # noqa: E731
    res = {}
    # LLaMA 65.2B 8-way SwiGLU shard, bf16
    inp = cs_inputs.make_inputs("llama", M=2048, seed=0)
    d = {"X": inp.X.cuda(), "Wg": dev_of(inp.Wg), "Wu": dev_of(inp.Wu), "W2": dev_of(inp.W2)}
    rows = []
    for m in cs_inputs.GPT3_M_SWEEP:
        sub = dict(d, X=d["X"][:m].contiguous())
        Ym = torch.empty(m, inp.H, dtype=inp.dtype, device="cuda")
        rec = {"M": m}
        with contextlib.ExitStack() as es:
            fns = {}
            for key, pol, tuned in (("tile", "tile", 0), ("stream", "stream", 0), ("tile_builtin", "tile", -1)):
                desc = cs.cs_chain_desc_init(kind="swiglu", M=m, H=inp.H, F=inp.F, dtype=inp.dtype, policy=pol,
                                             weight_layout=lay, tuned=tuned)
                p = es.enter_context(cs.cs_chain_plan(desc))
                if key == "tile":
                    rec["plan"] = plan_record(cs.cs_chain_query(p))
                fns[key] = (lambda p=p: cs.cs_mlp_forward(p, Y=Ym, **sub))
            for key, ms in interleaved_times(fns).items():
                rec[f"{key}_us"] = ms * 1e3
        fl = chain_flops("swiglu", m, inp.H, inp.F)
        rec["tflops"] = fl / (rec["tile_us"] * 1e-6) / 1e12
        rec["roofline_frac"], rec["bound"] = _roof_frac(fl, chain_bytes("swiglu", m, inp.H, inp.F), rec["tile_us"], peaks)
        rec["beats_control"] = rec["tile_us"] < rec["stream_us"]
        rows.append(rec)
    res["llama_swiglu"] = rows
    del d
    # attention chain of the GPT-3 shard (12 heads x 128, causal, seq = M), fp16
    inp = cs_inputs.make_inputs("attn", M=2048, seed=0)
    d = {"X": inp.X.cuda(), "Wqkv": dev_of(inp.Wqkv), "Wo": dev_of(inp.Wo)}
    rows = []
    for m in cs_inputs.GPT3_M_SWEEP:
        Xm = d["X"][:m].contiguous()
        Ym = torch.empty(m, inp.H, dtype=inp.dtype, device="cuda")
        rec = {"M": m}
        with contextlib.ExitStack() as es:
            fns = {}
            for key, pol, tuned in (("row", "row", 0), ("stream", "stream", 0), ("row_builtin", "row", -1)):
                desc = cs.cs_chain_desc_init(kind="attn", M=m, H=inp.H, F=inp.F, heads=inp.F // 128, head_dim=128,
                                             dtype=inp.dtype, policy=pol, weight_layout=lay, tuned=tuned)
                p = es.enter_context(cs.cs_chain_plan(desc))
                if key == "row":
                    rec["plan"] = plan_record(cs.cs_chain_query(p))
                fns[key] = (lambda p=p: cs.cs_attn_chain_forward(p, Xm, d["Wqkv"], d["Wo"], Ym))
            for key, ms in interleaved_times(fns).items():
                rec[f"{key}_us"] = ms * 1e3
        fl = chain_flops("attn", m, inp.H, inp.F)
        by = chain_bytes("attn", m, inp.H, inp.F)
        rec["tflops"] = fl / (rec["row_us"] * 1e-6) / 1e12
        rec["roofline_frac"], rec["bound"] = _roof_frac(fl, by, rec["row_us"], peaks)
        rec["beats_control"] = rec["row_us"] < rec["stream_us"]
        rows.append(rec)
    res["attention_chain"] = rows
    del d
    # last-wave stress sweep: two-GEMM GeLU chain, K = N = 8192, every policy
    inp = cs_inputs.make_inputs("stress", M=1536, seed=0)
    d = {"X": inp.X.cuda(), "W1": dev_of(inp.W1), "b1": inp.b1.cuda(), "W2": dev_of(inp.W2)}
    rows = []
    for m in cs_inputs.STRESS_M_SWEEP:
        sub = dict(d, X=d["X"][:m].contiguous())
        Ym = torch.empty(m, inp.H, dtype=inp.dtype, device="cuda")
        rec = {"M": m}
        with contextlib.ExitStack() as es:
            fns, plans = {}, {}
            for key, pol, tuned in (("tile", "tile", 0), ("row", "row", 0), ("strided", "strided", 0),
                                    ("stream", "stream", 0), ("tile_builtin", "tile", -1)):
                desc = cs.cs_chain_desc_init(kind="gelu", M=m, H=inp.H, F=inp.F, dtype=inp.dtype, policy=pol,
                                             weight_layout=lay, tuned=tuned)
                p = es.enter_context(cs.cs_chain_plan(desc))
                if key == "tile":
                    q = cs.cs_chain_query(p)
                    rec["plan"] = plan_record(q)
                fns[key] = (lambda p=p: cs.cs_mlp_forward(p, Y=Ym, **sub))
                plans[key] = p
            # Stream-K tail of the TileSync plan's tiles: the last stage's tiles
            # left over after whole waves, shared by one unit per resident worker
            sk = stream_k_remainder(q)
            if sk:
                dsk = cs.cs_chain_desc_init(kind="gelu", M=m, H=inp.H, F=inp.F, dtype=inp.dtype, policy="tile",
                                            weight_layout=lay, tile_m=q["tile_m"], tile_n=q["tile_n"][1],
                                            split_k=1, group_m=q["group_m"], sk_tiles=sk)
                p = es.enter_context(cs.cs_chain_plan(dsk))
                rec["stream_k_plan"] = {"sk_tiles": cs.cs_chain_query(p)["sk_tiles"],
                                        "sk_units": cs.cs_chain_query(p)["sk_units"]}
                fns["tile_sk"] = (lambda p=p: cs.cs_mlp_forward(p, Y=Ym, **sub))
            for key, ms in interleaved_times(fns).items():
                rec[f"{key}_us"] = ms * 1e3
            # SM occupancy of one traced forward of the fused chain and of the control
            try:
                rec["tail"] = {k: tail_stats(cs, torch, plans[k], fns[k]) for k in ("tile", "stream")}
            except Exception as e:  # a side measurement that fails must not cost the bench line
                rec["tail"] = {"error": repr(e)[:200]}
        workers = q["workers"]
        tiles0 = q["sched_units"][0]
        rec["stage0_units"], rec["workers"] = tiles0, workers
        rec["waves_remainder"] = [tiles0 // workers, tiles0 % workers]
        fl = chain_flops("gelu", m, inp.H, inp.F)
        best = min(rec["tile_us"], rec["row_us"], rec["strided_us"])
        rec["tflops_tile"] = fl / (rec["tile_us"] * 1e-6) / 1e12
        rec["roofline_frac_tile"], _ = _roof_frac(fl, chain_bytes("gelu", m, inp.H, inp.F), rec["tile_us"], peaks)
        rec["best_policy_vs_control"] = rec["stream_us"] / best
        if "tile_sk_us" in rec:
            rec["stream_k_vs_tile"] = rec["tile_us"] / rec["tile_sk_us"]
        rows.append(rec)
    res["stress"] = rows
    return res


if __name__ == "__main__":
    main()
