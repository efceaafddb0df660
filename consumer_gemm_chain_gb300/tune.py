"""Tuner for the plan's automatic choices: measures tile shape x K-split
candidates under every sync policy for a chain shape and a list of row counts
M, and writes the fastest per (M, policy) as a tuning table that
``cs_tune_load`` reads (Flux summary, idea I4: one kernel code base, tuned per
GPU and environment).

    python -m consumer_gemm_chain_gb300.tune --preset gpt3 [--M 1,16,...] [--out FILE] [--merge]
    python -m consumer_gemm_chain_gb300.tune --shape gelu,8192,4096,bf16 --layout kn --M 64,512,4096

Per M: every candidate runs under TileSync (RowSync for the attention chain),
and Stream-K tails of the last stage on the two fastest unsplit tile shapes;
up to 64 rows also the two fastest split tile shapes with the later stages'
units in K-range order (raster 3), with uniform splits and with more splits
for the first stage (split_k_first); the four fastest are timed again in
interleaved rounds, and the three fastest of those under every policy,
including the two-kernel control (so that the control, too, runs its best
tiles); the best
candidate of each policy is re-timed against the built-in rules in
interleaved rounds, and an entry is written per policy: the candidate's
choices if it wins by at least 2 %, else zeros (the built-in rules).  Each candidate's
output is checked against the built-in plan's output before it is timed.
Inputs are random device tensors of the shape (N(0, 0.02)); timing uses CUDA
events on the current stream, after warm-up, with weights larger than L2.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys

from . import chain as cs

PRESETS = {
    # name: (kind, H, F, dtype name, heads, default M list)
    "gpt3": ("gelu", 12288, 6144, "f16", 0, (1, 16, 64, 128, 256, 512, 1024, 2048)),
    "llama": ("swiglu", 8192, 2752, "bf16", 0, (1, 16, 64, 128, 256, 512, 1024, 2048)),
    "attn": ("attn", 12288, 1536, "f16", 12, (1, 16, 64, 128, 256, 512, 1024, 2048)),
    "stress": ("gelu", 8192, 8192, "f16", 0, tuple(128 * b for b in range(1, 13))),
}
MLP_TILES = ((128, 64), (128, 128), (128, 256), (256, 256), (512, 256))
ATTN_TILES = ((128, 128), (256, 256))
POLICIES = ("tile", "row", "strided", "stream")
ROUNDS = 5      # interleaved rounds of the final comparison
MARGIN = 0.02   # a tuned choice must beat the built-in rules by 2 %


def parse_shape(text):
    """KIND,H,F,DTYPE[,HEADS] -> (kind, H, F, dtype, heads) of a chain to tune."""
    parts = [p.strip() for p in text.split(",")]
    if len(parts) not in (4, 5):
        raise ValueError(f"--shape {text!r}: KIND,H,F,DTYPE[,HEADS]")
    kind, H, F, dtype = parts[0], int(parts[1]), int(parts[2]), parts[3]
    heads = int(parts[4]) if len(parts) == 5 else 0
    if kind not in ("gelu", "swiglu", "attn") or dtype not in ("f16", "bf16"):
        raise ValueError(f"--shape {text!r}: KIND is gelu, swiglu or attn; DTYPE f16 or bf16")
    if H < 8 or F < 8 or H % 8 or F % 8:
        raise ValueError(f"--shape {text!r}: H and F are positive multiples of 8")
    if kind == "attn" and heads * 128 != F:
        raise ValueError(f"--shape {text!r}: the attention chain needs HEADS with F = HEADS x 128")
    return kind, H, F, dtype, heads


def _inputs(torch, kind, M, H, F, dtype, dev, layout="nk", seed=0):
    g = torch.Generator(device=dev).manual_seed(seed)

    def r(*shape):
        return (torch.randn(*shape, generator=g, device=dev, dtype=torch.float32) * 0.02).to(dtype)

    def w(K, N):  # a weight of math shape [K, N] in the storage layout
        return r(N, K) if layout == "nk" else r(K, N)

    t = {"X": r(M, H)}
    if kind == "gelu":
        t.update(W1=w(H, F), b1=r(F), W2=w(F, H))
    elif kind == "swiglu":
        t.update(Wg=w(H, F), Wu=w(H, F), W2=w(F, H))
    else:
        t.update(Wqkv=w(H, 3 * F), Wo=w(F, H))
    return t


def _time(torch, fn, target_ms=12.0, warm_ms=60.0, repeats=1):
    """Mean us per call over about target_ms of back-to-back calls, after at
    least warm_ms of calls: under the power cap the SM clock follows the power
    drawn over the last tens of milliseconds, so the timing of a candidate must
    not start in the clock its predecessor left behind."""
    s = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n, spent, calls = 3, 0.0, 0
    while spent < warm_ms:
        a.record(s)
        for _ in range(n):
            fn()
        b.record(s)
        torch.cuda.synchronize()
        spent += a.elapsed_time(b)
        calls += n
        n = min(2 * n, 4096)
    iters = max(5, min(400, int(target_ms / max(spent / calls, 1e-3))))
    runs = []
    for _ in range(repeats):
        a.record(s)
        for _ in range(iters):
            fn()
        b.record(s)
        torch.cuda.synchronize()
        runs.append(a.elapsed_time(b) / iters * 1e3)
    return statistics.median(runs)


class Candidate:
    def __init__(self, kind, shape, policy, tile_m=0, tile_n=0, split_k=0, sk_tiles=0, sk_units=0,
                 split_k_first=0, raster=0, tuned=-1):
        self.key = (tile_m, tile_n, split_k, sk_tiles, sk_units, split_k_first, raster)
        self.policy = policy
        self.desc = cs.cs_chain_desc_init(kind=kind, M=shape["M"], H=shape["H"], F=shape["F"],
                                          dtype=shape["dtype"], policy=policy, weight_layout=shape["layout"],
                                          heads=shape["heads"] or 12, tile_m=tile_m, tile_n=tile_n,
                                          split_k=split_k, sk_tiles=sk_tiles if sk_tiles else -1,
                                          sk_units=sk_units, split_k_first=split_k_first, raster=raster,
                                          tuned=tuned)


def stream_k_candidates(info):
    """Stream-K tails worth timing for a plan of unsplit tiles: the last stage's
    tiles left over after whole waves of all the plan's units (the last wave),
    that remainder plus half a wave, each shared by one or two units per worker
    (the resident workers the plan reports)."""
    last = info["stages"] - 1
    if info["split_k"][last] != 1:
        return []
    w = info["workers"]
    total = sum(info["sched_units"][: info["stages"]])
    rem = total % w
    out = []
    for tiles in (rem, rem + w // 2):
        if 0 < tiles <= info["sched_units"][last]:
            out += [(tiles, w), (tiles, 2 * w)]
    return out


def k_range_combos(sp):
    """(split_k, split_k_first) pairs timed with the K-range order (raster 3) on
    a tile shape whose fastest split count is sp: uniform splits (0: the
    automatic rule), more splits for the first stage, and the first stage's
    splits with unsplit later stages (no reduction there; measured faster for
    the attention chain's short Wo GEMM at up to 16 rows), each pair once."""
    combos = [(s, 0) for s in (0, sp, 4, 6, 8)] + [(sp, f) for f in (2 * sp, 6, 8, 12) if f != sp]
    combos += [(1, f) for f in (sp, 2 * sp) if sp > 1]
    return list(dict.fromkeys(combos))


def plan_key(info):
    """What makes two plans the same candidate: the tile shape of every stage
    and the K-splits of every stage (tile_m alone does not tell 128 x 128 from
    128 x 256 tiles)."""
    return (info["tile_m"], tuple(info["tile_n"]), tuple(info["split_k"]))


def _forward(plan, kind, t, Y):
    if kind == "attn":
        return lambda: cs.cs_attn_chain_forward(plan, t["X"], t["Wqkv"], t["Wo"], Y)
    w = {k: v for k, v in t.items() if k != "X"}
    return lambda: cs.cs_mlp_forward(plan, t["X"], Y=Y, **w)


def _rel(torch, a, b):
    return float((a.float() - b.float()).abs().max() / b.float().abs().max().clamp_min(1e-30))


def tune_shape(torch, kind, H, F, dtype, heads, Ms, log=print, layout="nk", verbose=False):
    dev = torch.device("cuda", torch.cuda.current_device())
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    tiles = ATTN_TILES if kind == "attn" else MLP_TILES
    base = "row" if kind == "attn" else "tile"
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    entries = []
    for M in Ms:
        shape = {"M": M, "H": H, "F": F, "dtype": tdt, "heads": heads, "layout": layout}
        t = _inputs(torch, kind, M, H, F, tdt, dev, layout)
        Y = torch.empty(M, H, dtype=tdt, device=dev)
        splits = (1, 2, 3, 4) + ((6, 8, 12) if M <= 32 else ())

        def run(c):
            """(us, plan info) of one candidate; checks its status and its output
            against the built-in plan's."""
            with cs.cs_chain_plan(c.desc) as plan:
                info = cs.cs_chain_query(plan)
                fwd = _forward(plan, kind, t, Y)
                fwd()
                torch.cuda.synchronize()
                if cs.cs_chain_status(plan) != cs.CS_OK:
                    raise RuntimeError(f"M={M} {c.policy} {c.key}: device status {cs.cs_chain_status(plan)}")
                if ref is not None:
                    # both plans lie within 5e-3 of the exact chain (max-normalised),
                    # so within 1e-2 of each other; more means a broken candidate
                    err = _rel(torch, Y, ref)
                    if not err <= 1e-2:
                        raise RuntimeError(f"M={M} {c.policy} {c.key}: output differs from the built-in plan's "
                                           f"by {err:.2e}")
                us = _time(torch, fwd)
                if verbose:
                    log(f"  {kind} M={M:5d} {c.policy:8s} {c.key} splits {info['split_k'][:info['stages']]}: "
                        f"{us:8.2f} us")
                return us, info

        ref = None
        auto = Candidate(kind, shape, base)
        with cs.cs_chain_plan(auto.desc) as plan:
            _forward(plan, kind, t, Y)()
            torch.cuda.synchronize()
            ref = Y.clone()
        # 1: every tile shape x split under the base policy
        first, infos = {}, {}
        for tm, tn in tiles:
            for sp in splits:
                if sp > 4 and tm > 128:
                    continue  # many-way splits pay off only where single SMs stream the weights
                c = Candidate(kind, shape, base, tm, tn, sp)
                try:
                    us, info = run(c)
                except cs.CSError:
                    continue  # a shape this desc rejects
                # the last stage's tiles (SwiGLU producer tiles are always 128 wide)
                real = (info["tile_m"], info["tile_n"][info["stages"] - 1], max(info["split_k"]))
                if real != (tm, tn, sp):
                    continue  # clamped to another candidate (too few K-slices for the split)
                first[c.key] = us
                infos[c.key] = info
        # 1b: Stream-K tails on the two fastest unsplit tile shapes
        unsplit = sorted((k for k in first if k[2] == 1), key=first.get)[:2]
        for key in unsplit:
            for skt, sku in stream_k_candidates(infos[key]):
                c = Candidate(kind, shape, base, key[0], key[1], key[2], skt, sku)
                try:
                    us, info = run(c)
                except cs.CSError:
                    continue
                if info["sk_tiles"] == skt:
                    first[c.key] = us
        # 1c: at small M, the two fastest tile shapes with automatic K-splits for
        # the producers and a Stream-K last stage (all of its tiles shared out
        # over the resident workers)
        if M <= 256:
            shapes = []
            for key in sorted(first, key=first.get):
                if key[3] == 0 and key[:2] not in shapes:
                    shapes.append(key[:2])
            for tm, tn in shapes[:2]:
                info0 = infos[next(k for k in infos if k[:2] == (tm, tn))]
                last = info0["stages"] - 1
                skt = info0["n_tiles"][last] * -(-M // info0["tile_m"])
                c = Candidate(kind, shape, base, tm, tn, 0, skt, 0)
                try:
                    us, info = run(c)
                except cs.CSError:
                    continue
                if info["sk_tiles"] == skt:
                    first[c.key] = us
        # 1d: up to 64 rows, the two fastest split tile shapes with the later
        # stages' units in K-range order (raster 3), under uniform splits and
        # with more splits for the first stage: producers in several waves
        # finish their column tiles in turn, which K-range-major consumers use
        if M <= 64:
            shapes = []
            for key in sorted(first, key=first.get):
                if key[2] != 1 and key[3] == 0 and key[:2] not in [k[:2] for k in shapes]:
                    shapes.append(key)
            seen = set()
            for tm, tn, sp, *_ in shapes[:2]:
                for s, f in k_range_combos(sp):
                    c = Candidate(kind, shape, base, tm, tn, s, 0, 0, f, 3)
                    try:
                        us, info = run(c)
                    except cs.CSError:
                        continue
                    real = plan_key(info)
                    want_first = f or s
                    if real in seen or info["raster"] != 3 or (want_first and info["split_k"][0] != want_first):
                        continue  # clamped onto another candidate, or a repeat
                    seen.add(real)
                    first[c.key] = us
        # 2a: the four fastest again under the base policy, in interleaved
        # rounds (at small M single timings of near candidates differ by more
        # than their real gaps), keeping the three fastest medians
        top = sorted(first, key=first.get)[:4]
        again = {key: [] for key in top}
        for r in range(3):
            for i in range(len(top)):
                key = top[(r + i) % len(top)]
                again[key].append(run(Candidate(kind, shape, base, *key))[0])
        base_us = {key: statistics.median(v) for key, v in again.items()}
        top = sorted(top, key=base_us.get)[:3]
        # 2b: the three fastest under every policy (the control included)
        best = {}
        for pol in POLICIES:
            for key in top:
                us = base_us[key] if pol == base else run(Candidate(kind, shape, pol, *key))[0]
                if pol not in best or us < best[pol][1]:
                    best[pol] = (key, us)
        # 3: each policy's best against the built-in rules, interleaved rounds;
        # a candidate replaces the built-in rules only when it wins by MARGIN
        # (an entry of zeros keeps them: the timings of one configuration
        # spread by a few per cent under the power cap)
        finals = {pol: Candidate(kind, shape, pol, *best[pol][0]) for pol in POLICIES}
        builtin = {pol: Candidate(kind, shape, pol) for pol in POLICIES}
        times = {}
        order = [(pol, name, c) for pol in POLICIES for name, c in (("tuned", finals[pol]), ("builtin", builtin[pol]))]
        for r in range(ROUNDS):
            for i in range(len(order)):  # each round starts one place later
                pol, name, c = order[(r + i) % len(order)]
                times.setdefault((pol, name), []).append(run(c)[0])
        for pol in POLICIES:
            us = statistics.median(times[(pol, "tuned")])
            us_auto = statistics.median(times[(pol, "builtin")])
            if us < (1.0 - MARGIN) * us_auto:
                tm, tn, sp, skt, sku, spf, ras = finals[pol].key
            else:
                tm, tn, sp, skt, sku, spf, ras, us = 0, 0, 0, 0, 0, 0, 0, us_auto
            entry = {"kind": kind, "dtype": dtype, "H": H, "F": F, "M": M, "sms": sms, "layout": layout,
                     "policy": pol, "tile_m": tm, "tile_n": tn, "split_k": sp, "group_m": 0,
                     "us": round(us, 2), "builtin_us": round(us_auto, 2)}
            if skt:
                entry.update(sk_tiles=skt, sk_units=sku)
            if spf:
                entry.update(split_k_first=spf)
            if ras:
                entry.update(raster=ras)
            entries.append(entry)
            choice = (f"tile {tm}x{tn} split {sp:2d}" + (f" first {spf}" if spf else "") +
                      (f" raster {ras}" if ras else "") + (f" stream-K {skt}/{sku}" if skt else "")) if tm else \
                "built-in rules    "
            log(f"{kind} M={M:5d} {pol:8s} {choice}: {us:8.1f} us (built-in rules {us_auto:8.1f} us)")
        del t, Y, ref
        torch.cuda.empty_cache()
    return entries


def _key(e):
    return (e["kind"], e["dtype"], e["H"], e["F"], e["M"], e["sms"], e.get("layout", "any"), e.get("policy", "any"))


def write_table(path, entries, merge, device):
    old = []
    if merge and os.path.exists(path):
        with open(path) as f:
            old = json.load(f).get("entries", [])
    keys = {_key(e) for e in entries}
    merged = [e for e in old if _key(e) not in keys] + entries
    merged.sort(key=lambda e: (e["kind"], e["H"], e["F"], e["dtype"], e["M"], e.get("policy", "")))
    doc = {"format": "cs_chain_tuning", "version": 1, "device": device,
           "written_by": "python -m consumer_gemm_chain_gb300.tune", "entries": merged}
    os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
    with open(path, "w") as f:
        f.write("{\n")
        f.write(f'  "format": "cs_chain_tuning", "version": 1, "device": {json.dumps(device)},\n')
        f.write(f'  "written_by": {json.dumps(doc["written_by"])},\n  "entries": [\n')
        f.write(",\n".join("    " + json.dumps(e) for e in merged))
        f.write("\n  ]\n}\n")
    return len(merged)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--preset", action="append", default=[], choices=sorted(PRESETS))
    ap.add_argument("--shape", action="append", default=[], metavar="KIND,H,F,DTYPE[,HEADS]",
                    help="a chain shape of your own (its default M list is the presets' 1 .. 2048)")
    ap.add_argument("--layout", default="nk", choices=["nk", "kn"], help="weight storage layout")
    ap.add_argument("--M", default="", help="comma-separated row counts (default: the preset's list)")
    ap.add_argument("--out", default=cs.TUNE_TABLE)
    ap.add_argument("--merge", action="store_true", help="keep the file's entries for other shapes / M")
    ap.add_argument("--verbose", action="store_true", help="log every candidate's timing")
    args = ap.parse_args(argv)
    shapes = [PRESETS[name] for name in args.preset]
    try:
        shapes += [parse_shape(t) + (PRESETS["gpt3"][5],) for t in args.shape]
    except ValueError as e:
        ap.error(str(e))
    if not shapes:
        ap.error("give at least one --preset or --shape")
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("the tuner times kernels on a GPU; none is visible")
    props = torch.cuda.get_device_properties(0)
    device = {"name": props.name, "sms": props.multi_processor_count, "cc": f"{props.major}.{props.minor}"}
    entries = []
    n = 0
    for kind, H, F, dtype, heads, Ms in shapes:
        if args.M:
            Ms = tuple(int(v) for v in args.M.split(","))
        entries += tune_shape(torch, kind, H, F, dtype, heads, Ms, layout=args.layout, verbose=args.verbose,
                              log=lambda s: print(s, file=sys.stderr, flush=True))
        n = write_table(args.out, entries, args.merge, device)  # after every shape: keep what is measured
    print(json.dumps({"out": args.out, "entries": n}))


if __name__ == "__main__":
    main()
