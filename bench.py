"""Benchmark of the rolling-KV step: stream-steps/s (all layers) and decode-attention HBM GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mixed] [--impl ours|reference]

One step = the whole hot path for every active stream and every layer: begin
step (ring bookkeeping + RoPE angles), then per layer the exact re-base (exact
scheme), RoPE + append, and split-K decode attention with its merge.  The
timed steps replay CUDA graphs of `rkv_step` over inputs already resident in
HBM; the windows are full before timing starts (steady state).

The default workload is the largest batched one: mixed-clock serving, 256
streams with 80 / 120 / 160 ms clocks (windows 375 / 250 / 188) on a 40 ms
scheduler tick, 36 Qwen-shaped layers, exact re-base; one step is one tick.
The line also carries the Qwen-shaped decoder (36 layers, 64 streams) and the
voxtral-shaped decoder (26 layers, 16 streams, window 8192) as sub-records
with their own roofline.  Under torchrun every rank runs its own copy of the
workload (streams are independent: no collective on the data path) and
`value` sums all ranks' stream-steps over the slowest rank's time.

The reference arm (`--impl reference`) times the fp64 CPU oracle on this
host's cores, each step a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "stream-steps/sec (all layers) and decode-attn HBM GB/s as % of B300 peak"
UNIT = "stream-steps/s"
SCHEMES = {"offset": 0, "exact": 1, "on-read": 2}

# DRAM traffic (read + write bytes) of one all-layers decode-attention launch, from the committed
# ncu launch-list summary of the same command, valid only while the attention source's code is the
# one that was profiled: a different code digest (comments and white space left out) reports null.
TRAFFIC = [
    {"workload": "mixed", "layers": 36, "schemes": (0, 1), "attn_code_sha256_16": "d10556389b5bee13",
     "bytes_per_launch": 1131.00e6 + 13.58e6},   # the tick phase with the most active streams
    {"workload": "mixed", "layers": 36, "schemes": (2,), "attn_code_sha256_16": "d10556389b5bee13",
     "bytes_per_launch": 1131.25e6 + 13.41e6},   # the tick phase with the most active streams
    {"workload": "qwen", "layers": 36, "schemes": (0, 1), "attn_code_sha256_16": "d10556389b5bee13",
     "bytes_per_launch": 915.69e6 + 8.37e6},
    {"workload": "qwen", "layers": 36, "schemes": (2,), "attn_code_sha256_16": "d10556389b5bee13",
     "bytes_per_launch": 915.77e6 + 8.11e6},
    {"workload": "voxtral", "layers": 26, "schemes": (0,), "attn_code_sha256_16": "d10556389b5bee13",
     "bytes_per_launch": 13962.88e6 + 3.72e6},
    {"workload": "encoder", "layers": 32, "schemes": (0,), "attn_code_sha256_16": "d10556389b5bee13",
     "bytes_per_launch": 4037.93e6 + 10.59e6},
]
SCHEME_NAMES = {0: "offset-only", 1: "exact re-base", 2: "exact re-base applied on read"}


def bench_workload(args, **extra):
    """The workload a run measures.  A workload that re-bases exactly is run with the re-base applied
    on read unless --scheme says otherwise: the same outputs as the materialised re-base (every
    retained key re-rotated on every roll), which `schemes` reports beside it."""
    import synth
    over = dict(extra)
    if args.scheme:
        over["scheme"] = SCHEMES[args.scheme]
    if getattr(args, "kv_format", "f16") == "e4m3":
        over["kv_format"] = 1
    if args.layers:
        over["n_layers"] = args.layers
    wl = synth.workload(args.workload, **over)
    if not args.scheme and wl.scheme == 1:
        wl = synth.workload(args.workload, **dict(over, scheme=2))
    return wl, over


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default="mixed", choices=["tiny", "qwen", "voxtral", "encoder", "mixed"])
    p.add_argument("--scheme", default=None, choices=[None, "offset", "exact", "on-read"])
    p.add_argument("--kv-format", default="f16", choices=["f16", "e4m3"],
                   help="key/value store: fp16 keys and bf16 values, or the optional fp8 (e4m3) store "
                        "(lower precision: profiling and comparison runs, never the headline)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-baseline sample")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--inputs", type=int, default=4, help="distinct resident input sets cycled by the steps")
    p.add_argument("--layers", type=int, default=None, help="override the workload's layer count (profiling cases)")
    p.add_argument("--no-variants", dest="variants", action="store_false",
                   help="skip timing the workload under the other two schemes")
    p.add_argument("--no-flatness", dest="flatness", action="store_false",
                   help="skip the per-step time at five start offsets (Qwen-shaped workload)")
    p.add_argument("--no-sub", dest="sub", action="store_false",
                   help="skip the Qwen- and voxtral-shaped sub-records of the default run")
    p.add_argument("--no-per-layer", dest="per_layer", action="store_false",
                   help="skip the step made of per-layer calls")
    p.add_argument("--window-scan", action="store_true",
                   help="time one-layer decode-attention launches against the window length (Qwen-shaped "
                        "heads, 64 streams) and print that scan instead of the benchmark line")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def describe(wl, scheme_name):
    w = sorted(set(wl.windows().tolist()))
    return (f"{wl.name}: {wl.n_layers} layers, {wl.n_streams} streams, Hq={wl.n_q_heads} Hkv={wl.n_kv_heads} "
            f"d={wl.head_dim}, Q={wl.q_per_step}, W={'/'.join(map(str, w))}, {scheme_name}, "
            f"P0<{wl.p0_high or 1}, inputs N(0,1){' x 1/sqrt(d)' if wl.scale_inputs else ''} bf16")


def algorithmic_attn_bytes(wl, lens):
    """Bytes decode attention must move for one layer: K+V of the window, q in, out, lse (the fp8
    store: one byte per key and value element and a pair of float scales per token and kv head)."""
    Q, hq, hkv, d = wl.q_per_step, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    per_token = 2 * d + 8 if wl.kv_format == 1 else 2 * d * 2
    kv = sum(int(n) * hkv * per_token for n in lens)
    return kv + len(lens) * (Q * hq * d * 2 * 2 + Q * hq * 4)


def algorithmic_rebase_bytes(wl, act):
    """Bytes one exact re-base step moves: every retained key of every active stream, layer and
    kv head read as its pre-RoPE copy and written rotated (windows full: W - 1 retained keys)."""
    windows = wl.windows()
    return sum(wl.n_layers * wl.n_kv_heads * (int(windows[s]) - 1) * wl.head_dim * 2 * 2 for s in act)


def rebase_in_step(wl, m, variants, steps, peak):
    """The materialised exact re-base's share of the step, from two CUDA-event timings of this run:
    that scheme's step minus the offset-only step, which makes the same launches without the
    re-base (m: the materialised scheme's measurement, or the headline's whose variants hold it)."""
    off = variants.get(SCHEME_NAMES[0]) if variants else None
    if off is None:
        return None
    if wl.scheme == 1:
        ms_step = m["ms"] / steps
    elif SCHEME_NAMES[1] in variants:
        ms_step = variants[SCHEME_NAMES[1]]["ms_per_step"]
    else:
        return None
    plan = m["plan"]
    per_step_bytes = sum(algorithmic_rebase_bytes(wl, plan[i % len(plan)]) for i in range(steps)) / steps
    us = (ms_step - off["ms_per_step"]) * 1000.0
    if us <= 0:
        return None
    gbs = per_step_bytes / (us * 1e-6) / 1e9
    return {"kernel": f"rebase_kernel: exact re-base over all {wl.n_layers} layers in one launch",
            "us_per_step": us, "algorithmic_bytes_per_step": per_step_bytes, "achieved_gbs": gbs,
            "frac": gbs / peak, "how": "exact re-base step minus offset-only step (the same launches "
                                       "without the re-base), both timed with CUDA events in this run"}


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id  # nvidia-smi --id: the device's UUID ("GPU-...")
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            self.proc.wait(timeout=5)

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                        rows.append(parts)
        finally:
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(float(r[1]) for r in rows),
                "sm_max_mhz": max(float(r[2]) for r in rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit()) if rows else None,
                "reasons": reasons, "samples": len(rows)}


def code_digest(path):
    """sha256 (16 hex digits) of a C++/CUDA source with its comments and white space removed."""
    import hashlib
    import re
    with open(path, encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    text = re.sub(r"\s+", "", text)
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def profiled_traffic(wl):
    """ncu DRAM bytes per attention launch for this workload, or None (not profiled / kernel changed)."""
    try:
        digest = code_digest(os.path.join(ROOT, "rolling_kv_sliding_rkv_b300", "csrc", "rkv_attn.cu"))
    except OSError:
        return None
    for t in TRAFFIC:
        if (t["workload"] == wl.name and t["layers"] == wl.n_layers and wl.scheme in t["schemes"]
                and t["attn_code_sha256_16"] == digest):
            return t["bytes_per_launch"]
    return None


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6400.0, "fallback"


# ---------------------------------------------------------------- oracle legs

def _oracle_chunk(args):
    """Oracle evaluation of consecutive steps of one stream, all layers (runs in a worker process)."""
    name, stream, n0, n_steps, layers = args
    import synth
    from oracle.attention import attention_step
    wl = synth.workload(name)
    Q, hq, hkv, d = wl.q_per_step, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    w = int(wl.windows()[stream])
    p0 = int(wl.start_offsets()[stream])
    sc = wl.input_scale
    done = 0
    for i in range(n_steps):
        n_old = n0 + i * Q
        toks = list(range(max(0, n_old + Q - w), n_old + Q))
        for layer in layers:
            qb = synth.token_tensor(wl.seed, synth.TAG_Q, stream, layer, range(n_old, n_old + Q), hq, d, sc)
            kb = synth.token_tensor(wl.seed, synth.TAG_K, stream, layer, toks, hkv, d, sc)
            vb = synth.token_tensor(wl.seed, synth.TAG_V, stream, layer, toks, hkv, d, sc)
            attention_step(synth.bf16_bits_to_f64(qb), synth.bf16_bits_to_f64(kb), synth.bf16_bits_to_f64(vb),
                           toks, n_old, p0, w, 1.0 / math.sqrt(d), wl.rope_theta)
            done += 1
    return done


class OracleRunner:
    """The fp64 oracle on all host cores (spawned worker processes), timed in steps.

    A step is a bounded sample of the workload: batches of chunks, one chunk =
    `steps_per_chunk` consecutive full-window steps of one stream over a
    subset of layers, issued until the step's budget is spent.  Throughput is
    extrapolated from stream-layer-steps/s to stream-steps/s (all layers)."""

    def __init__(self, wl, steps_per_chunk=4):
        import multiprocessing as mp
        self.wl = wl
        self.cores = os.cpu_count() or 1
        self.steps_per_chunk = steps_per_chunk
        self.pool = mp.get_context("spawn").Pool(self.cores)
        w = int(wl.windows().max())
        self.n0 = (w // wl.q_per_step + 3) * wl.q_per_step     # steady state: window full
        self.layers = list(range(0, wl.n_layers, max(1, wl.n_layers // 4)))[:4]
        self.jobs = 0
        self.pool.map(_oracle_chunk, [(wl.name, 0, self.n0, 1, [0])] * self.cores)   # import + warm caches

    def step(self, budget_s):
        """One step: chunks until `budget_s` is spent (at least one batch); returns (layer-steps, seconds)."""
        wl = self.wl
        t0 = time.perf_counter()
        done = 0
        while True:
            batch = [(wl.name, (self.jobs + i) % wl.n_streams,
                      self.n0 + 64 * wl.q_per_step * ((self.jobs + i) // wl.n_streams),
                      self.steps_per_chunk, self.layers) for i in range(self.cores)]
            done += sum(self.pool.map(_oracle_chunk, batch))
            self.jobs += self.cores
            if time.perf_counter() - t0 >= budget_s:
                break
        return done, time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()

    def describe(self, done, elapsed, what=""):
        wl = self.wl
        return (f"{done} full-window stream-layer-steps ({len(self.layers)} of {wl.n_layers} layers, "
                f"{self.steps_per_chunk} consecutive steps per stream){what} in {elapsed:.1f} s on {self.cores} "
                f"spawned processes; value = stream-layer-steps/s / {wl.n_layers} layers (extrapolated)")


def oracle_timing(wl, budget_s):
    """The oracle's throughput on a bounded sample of about `budget_s` seconds (the cpu_baseline)."""
    r = OracleRunner(wl)
    try:
        done, elapsed = r.step(budget_s)
    finally:
        r.close()
    return {"value": done / elapsed / wl.n_layers, "unit": UNIT, "cores": r.cores, "kind": "oracle",
            "sample": r.describe(done, elapsed)}


def run_reference(args):
    import synth
    rank, world, _ = dist_env()
    if rank != 0:
        return
    wl, _ = bench_workload(args)
    # each step is a bounded sample: the whole run stays within about two minutes
    per_step = max(0.05, min(1.0, 110.0 / max(1, args.steps + args.warmup)))
    r = OracleRunner(wl)
    try:
        for _ in range(args.warmup):
            r.step(per_step)
        done = 0
        elapsed = 0.0
        for _ in range(args.steps):
            d, t = r.step(per_step)
            done += d
            elapsed += t
    finally:
        r.close()
    value = done / elapsed / wl.n_layers
    base = {"value": value, "unit": UNIT, "cores": r.cores, "kind": "oracle",
            "sample": r.describe(done, elapsed, f", {args.steps} timed steps of about {per_step:.2f} s each")}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * elapsed / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": describe(wl, SCHEME_NAMES[wl.scheme]),
                                            "parallelism": "replicas",
                                            "step": "a bounded sample of the workload's stream-layer-steps"},
            "cpu_baseline": base,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU leg

def aggregate(ms_local, stream_steps_local, world, device=None):
    """Whole-job figures over the ranks: the slowest rank's time and all ranks' stream-steps.

    Every rank runs its own streams (replicas: no exchange on the data path); the job is done
    when the slowest rank is, so value = (sum of stream-steps) / (max of times)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
        n = torch.tensor([float(stream_steps_local)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(n, op=dist.ReduceOp.SUM)
        ms, total = float(t.item()), float(n.item())
    else:
        ms, total = float(ms_local), float(stream_steps_local)
    return {"ms": ms, "stream_steps": total, "value": total / (ms / 1000.0)}


def step_phases(wl):
    """Active stream lists of one period of the workload's schedule (one list if every stream steps)."""
    if not wl.tick_ms:
        return [list(range(wl.n_streams))]
    periods = sorted({int(c) // wl.tick_ms for c in wl.stream_clocks()})
    period = 1
    for p in periods:
        period = period * p // math.gcd(period, p)
    return [wl.active_at_tick(t).tolist() for t in range(period)]


def measure(wl, args, dev, rank, world, timed=True, p0=None, attention=True, per_layer_step=False, churn=0):
    """Time the step of workload `wl` on this GPU; returns the figures of one JSON line.

    p0: start offset given to every stream (default: the workload's draws).
    per_layer_step: also time the same steps made of per-layer calls (begin step, then for each
    layer re-base, append and decode attention), one CUDA graph per step, as a model that runs
    other work between its layers must call them.
    churn: streams that leave per step, their slots taken at once by new streams with new start
    offsets (rkv_reset_streams from a device-side schedule the graphs walk through)."""
    import torch

    import rolling_kv_sliding_rkv_b300 as rkv
    import synth

    S, L, Q, hq, hkv, d = wl.n_streams, wl.n_layers, wl.q_per_step, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    windows = wl.windows()
    starts = wl.start_offsets().tolist() if p0 is None else [int(p0)] * S
    h = rkv.RollingKV(windows.tolist(), starts, device=dev, n_layers=L, n_streams=S,
                      n_q_heads=hq, n_kv_heads=hkv, head_dim=d, q_per_step=Q, scheme=wl.scheme,
                      rebase_interval=wl.rebase_interval, rope_theta=wl.rope_theta, kv_format=wl.kv_format)
    phases = [ph for ph in step_phases(wl)]
    # one resident input set (and one CUDA graph of a whole step) per phase; a single-phase
    # workload cycles through `--inputs` sets
    R = len(phases) if len(phases) > 1 else max(1, args.inputs)
    plan = [phases[r % len(phases)] for r in range(R)]
    sets = []
    for r, act in enumerate(plan):
        A = len(act)
        nq, nkv = L * A * Q * hq * d, L * A * Q * hkv * d
        bufs = {"q": torch.empty(max(nq, 8), dtype=torch.bfloat16, device=dev),
                "k": torch.empty(max(nkv, 8), dtype=torch.bfloat16, device=dev),
                "v": torch.empty(max(nkv, 8), dtype=torch.bfloat16, device=dev),
                "out": torch.empty(max(nq, 8), dtype=torch.bfloat16, device=dev),
                "lse": torch.empty(max(nq // d, 8), dtype=torch.float32, device=dev)}
        for tag, name in ((synth.TAG_Q, "q"), (synth.TAG_K, "k"), (synth.TAG_V, "v")):
            rkv.rkv_gen_tokens(wl.seed + 1000 * rank, tag, r, 0, 0, 1, bufs[name].numel(), wl.input_scale, bufs[name])
        sets.append(bufs)
    torch.cuda.synchronize()

    churn_state = None
    if churn:
        # a schedule of leave/join events: row t lists `churn` distinct slots and their new start
        # offsets; every step takes the next row (a device-side counter), so a replayed graph
        # resets different slots each time
        # (row t resets `churn` slots when t is a multiple of 12, none otherwise: with one slot per
        # 12 ticks each of 256 streams lives about two minutes, long enough to fill its window)
        T = 12 * 512
        t_idx = torch.arange(T * churn, dtype=torch.int64).view(T, churn)
        ids = (t_idx * 97 + 13) % S
        ids[torch.arange(T) % 12 != 0] = -1
        churn_state = {"ids": ids.to(torch.int32).to(dev),
                       "p0": ((t_idx * 1_000_003 + 7) % (2 ** 40)).to(dev),
                       "ctr": torch.zeros(1, dtype=torch.int64, device=dev),
                       "cur_ids": torch.empty(churn, dtype=torch.int32, device=dev),
                       "cur_p0": torch.empty(churn, dtype=torch.int64, device=dev), "T": T}

    def whole_step(act, b):
        if churn_state is not None:
            c = churn_state
            torch.index_select(c["ids"], 0, c["ctr"], out=c["cur_ids"].view(1, -1))
            torch.index_select(c["p0"], 0, c["ctr"], out=c["cur_p0"].view(1, -1))
            c["ctr"].add_(1).remainder_(c["T"])
            h.reset_streams(c["cur_ids"], c["cur_p0"])
        h.step(act, b["q"], b["k"], b["v"], b["out"], b["lse"])

    stream = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(stream):
        for r, act in enumerate(plan):   # eager warm-up of the capture stream
            if act:
                whole_step(act, sets[r])
        stream.synchronize()
        for r, act in enumerate(plan):
            if not act:
                graphs.append(None)
                continue
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                whole_step(act, sets[r])
            graphs.append(g)
    # begin step, re-base (materialised exact re-base), RoPE + append, decode attention: each one
    # launch over all layers
    launches_per_step = 1 + (1 if wl.scheme == 1 else 0) + 1 + 1 + (1 if churn else 0)

    # fill every window, then warm up: steady state before timing
    slowest = max(int(c) // max(wl.tick_ms, 1) for c in wl.stream_clocks()) if wl.tick_ms else 1
    fill = (int(windows.max()) // Q + 2) * slowest
    fill = (fill + R - 1) // R * R
    for i in range(fill + args.warmup):
        if graphs[i % R] is not None:
            graphs[i % R].replay()
    torch.cuda.synchronize()
    h.sync_status()
    free_before = torch.cuda.mem_get_info(dev)[0]

    cur = torch.cuda.current_stream()

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    out = {"h": h}
    if timed:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        sampler = ClockSampler(uuid if uuid.startswith("GPU-") else f"GPU-{uuid}")
        barrier()
        with sampler:
            ev0.record(cur)
            for i in range(args.steps):
                if graphs[i % R] is not None:
                    graphs[i % R].replay()
            ev1.record(cur)
            torch.cuda.synchronize()
        out["clocks"] = sampler.summary()
    else:
        barrier()
        ev0.record(cur)
        for i in range(args.steps):
            if graphs[i % R] is not None:
                graphs[i % R].replay()
        ev1.record(cur)
        torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    barrier()
    h.sync_status()
    job = aggregate(ms, sum(len(plan[i % R]) for i in range(args.steps)), world, dev)
    out.update(value=job["value"], ms=job["ms"], stream_steps=job["stream_steps"],
               launches=launches_per_step * sum(1 for i in range(args.steps) if graphs[i % R] is not None),
               free_bytes_delta=torch.cuda.mem_get_info(dev)[0] - free_before)

    if per_layer_step:
        def layer_calls(act, b, fused):
            A = len(act)
            h.begin_step(act)
            for layer in range(L):
                if wl.scheme in (1, 2):
                    h.rebase(layer)
                ql, kl, vl = b["q"][layer * A * Q * hq * d:], b["k"][layer * A * Q * hkv * d:], \
                    b["v"][layer * A * Q * hkv * d:]
                ol, ll = b["out"][layer * A * Q * hq * d:], b["lse"][layer * A * Q * hq:]
                if fused:
                    h.append_decode_attn(layer, ql, kl, vl, ol, ll)
                else:
                    h.append_rope(layer, kl, vl)
                    h.decode_attn(layer, ql, ol, ll)

        for fused in (False, True):
            lgraphs = []
            with torch.cuda.stream(stream):
                for r, act in enumerate(plan):
                    if act:
                        layer_calls(act, sets[r], fused)
                stream.synchronize()
                for r, act in enumerate(plan):
                    if not act:
                        lgraphs.append(None)
                        continue
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        layer_calls(act, sets[r], fused)
                    lgraphs.append(g)
            for i in range(args.warmup + R):
                if lgraphs[i % R] is not None:
                    lgraphs[i % R].replay()
            barrier()
            ev0.record(cur)
            for i in range(args.steps):
                if lgraphs[i % R] is not None:
                    lgraphs[i % R].replay()
            ev1.record(cur)
            torch.cuda.synchronize()
            lms = ev0.elapsed_time(ev1)
            h.sync_status()
            ljob = aggregate(lms, sum(len(plan[i % R]) for i in range(args.steps)), world, dev)
            rec = {"value": ljob["value"], "unit": UNIT, "ms_per_step": ljob["ms"] / args.steps,
                   "launches_per_step": 1 + L * ((1 if fused else 2) + (1 if wl.scheme == 1 else 0))}
            if fused:
                rec["how"] = ("the same per-layer calls with RoPE + append fused into the decode-attention "
                              "launch (rkv_append_decode_attn)")
                out["per_layer_step"]["fused_append"] = rec
            else:
                rec["how"] = ("the same steps as one CUDA graph of per-layer calls each: begin step, then for "
                              "every layer re-base (materialised exact re-base), RoPE + append and decode "
                              "attention, as a model that runs other work between its layers calls them")
                out["per_layer_step"] = rec
    if not attention:
        return out

    # decode attention alone: the all-layers launch the step makes (the dominant kernel), and,
    # for reference, per-layer launches as a model that interleaves other work would make them;
    # the phase with the most active streams, windows full
    r0 = max(range(R), key=lambda r: len(plan[r]))
    act = plan[r0]
    A = len(act)
    b = sets[r0]
    h.begin_step(act)
    for layer in range(L):
        if wl.scheme in (1, 2):
            h.rebase(layer)
        h.append_rope(layer, b["k"][layer * A * Q * hkv * d:], b["v"][layer * A * Q * hkv * d:])
    torch.cuda.synchronize()

    def time_graph(body, reps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            body()
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                body()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for _ in range(reps):
            g.replay()
        e1.record(cur)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    reps = max(5, min(200, args.steps // 2))
    attn_all_ms = time_graph(lambda: h.decode_attn_layers(0, L, b["q"], b["out"], b["lse"]), reps)

    def per_layer():
        for layer in range(L):
            h.decode_attn(layer, b["q"][layer * A * Q * hq * d:], b["out"][layer * A * Q * hq * d:],
                          b["lse"][layer * A * Q * hq:])
    attn_layer_ms = time_graph(per_layer, max(3, reps // 4)) / L
    lens = [int(windows[s]) for s in act]
    attn_bytes_layer = algorithmic_attn_bytes(wl, lens)
    out.update(attn_all_ms=attn_all_ms, attn_layer_ms=attn_layer_ms, attn_bytes_layer=attn_bytes_layer,
               attn_bytes=attn_bytes_layer * L, attn_streams=A, plan=plan)
    h.sync_status()   # closes nothing; the open step stays open until the handle is freed
    return out


def workload_figures(wl, scheme_name, m, peak, peak_kind, steps, world):
    """value, per-step time and the decode-attention roofline of one measured workload."""
    achieved = m["attn_bytes"] / (m["attn_all_ms"] / 1000.0) / 1e9
    achieved_layer = m["attn_bytes_layer"] / (m["attn_layer_ms"] / 1000.0) / 1e9
    A = len(step_phases(wl)[0]) if not wl.tick_ms else None
    fig = {"value": m["value"], "unit": UNIT, "ms_per_step": m["ms"] / steps,
           "config": {"workload": describe(wl, scheme_name),
                      "streams_per_gpu": A if A is not None else
                      f"{m['stream_steps'] / steps / world:.1f} active per 40 ms tick (of {wl.n_streams})",
                      "layers": wl.n_layers},
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                        "frac": achieved / peak, "traffic": profiled_traffic(wl),
                        "kernel": f"attn_kernel: decode attention over all {wl.n_layers} layers in one "
                                  "launch (as inside the timed step)",
                        "algorithmic_bytes_per_launch": m["attn_bytes"],
                        "avg_launch_us": m["attn_all_ms"] * 1000.0,
                        "streams_in_launch": m["attn_streams"],
                        "peak_kind": f"{peak_kind} (hbm_gbs, STREAM-style copy, burst)"},
           "decode_attn_gbs": achieved,
           "decode_attn_per_layer_launch": {"achieved_gbs": achieved_layer, "frac": achieved_layer / peak,
                                            "avg_launch_us": m["attn_layer_ms"] * 1000.0,
                                            "algorithmic_bytes_per_launch": m["attn_bytes_layer"]}}
    if "per_layer_step" in m:
        fig["value_per_layer_graph"] = m["per_layer_step"]["value"]
        fig["per_layer_step"] = m["per_layer_step"]
    return fig


def bench_line(wl, scheme_name, args, world, m, peak, peak_kind, variants=None, flat=None, e2e=None, cpu=None,
               subs=None):
    """The one JSON line of a run: the keys of the benchmark contract plus the roofline of the dominant kernel."""
    fig = workload_figures(wl, scheme_name, m, peak, peak_kind, args.steps, world)
    line = {"metric": METRIC, "value": fig["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": fig["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(fig["config"],
                           l2="per-step working set of KV pages > 126 MB L2; no flush between steps",
                           graph="one CUDA graph per step (per tick phase for mixed clocks), replayed",
                           parallelism="replicas" if world == 1 else f"replicas x{world}"),
            "roofline": fig["roofline"],
            "decode_attn_gbs": fig["decode_attn_gbs"],
            "decode_attn_per_layer_launch": fig["decode_attn_per_layer_launch"],
            "gpu_launches": m["launches"],
            "clocks": m.get("clocks")}
    for key in ("value_per_layer_graph", "per_layer_step"):
        if key in fig:
            line[key] = fig[key]
    if variants:
        line["schemes"] = variants
        rb = rebase_in_step(wl, m, variants, args.steps, peak)
        if rb is not None:
            line["rebase_in_step"] = rb
    if flat is not None:
        line["flatness"] = flat
    if subs:
        line["workloads"] = subs
    if e2e is not None:
        line["e2e"] = e2e
    if cpu is not None:
        line["cpu_baseline"] = cpu
    return line


def run_ours(args):
    import torch

    import synth

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl, over = bench_workload(args)
    scheme_name = SCHEME_NAMES[wl.scheme]
    m = measure(wl, args, dev, rank, world, per_layer_step=args.per_layer)
    h = m.pop("h")
    peak, peak_kind = measured_peak()

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(h, wl, m["plan"], args, dev)
    h.close()

    variants = {}
    if args.variants and rank == 0 and not args.scheme:
        todo = [(SCHEME_NAMES[sch], dict(over, scheme=sch)) for sch in SCHEMES.values() if sch != wl.scheme]
        if wl.scheme in (1, 2):   # chunked re-base: the materialised scheme re-basing once every 8 rolls
            todo.append(("exact re-base every 8 rolls", dict(over, scheme=1, rebase_interval=8)))
        if wl.scheme in (0, 2) and wl.n_q_heads // wl.n_kv_heads * wl.q_per_step <= 8:
            # the optional fp8 (e4m3) store: lower precision, so never the headline
            todo.append((f"{SCHEME_NAMES[wl.scheme]}, fp8 (e4m3) key/value store",
                         dict(over, scheme=wl.scheme, kv_format=1)))
        for label, vover in todo:
            vw = synth.workload(args.workload, **vover)
            vm = measure(vw, args, dev, rank, 1, timed=False, per_layer_step=args.per_layer)
            vm.pop("h").close()
            variants[label] = {
                "value": vm["value"], "unit": UNIT, "ms_per_step": vm["ms"] / args.steps,
                "decode_attn_gbs": vm["attn_bytes"] / (vm["attn_all_ms"] / 1000.0) / 1e9,
                "decode_attn_frac": vm["attn_bytes"] / (vm["attn_all_ms"] / 1000.0) / 1e9 / peak}
            if "per_layer_step" in vm:
                variants[label]["value_per_layer_graph"] = vm["per_layer_step"]["value"]
        if wl.tick_ms:
            # serving churn: one stream leaves and a new one joins in its slot every 12 ticks
            cm = measure(wl, args, dev, rank, 1, timed=False, attention=False, churn=1)
            cm.pop("h").close()
            variants[f"{SCHEME_NAMES[wl.scheme]}, one stream leaving and one joining every 12 ticks"] = {
                "value": cm["value"], "unit": UNIT, "ms_per_step": cm["ms"] / args.steps,
                "how": "each tick first runs rkv_reset_streams over the next row of a device-side schedule "
                       "(walked by the replayed graphs with a device counter); every 12th row resets one "
                       "slot to a new start offset, the others list no slot; a joining stream's window "
                       "starts empty and refills over its next W steps, so the tick moves fewer bytes"}

    def flatness(fw, free_delta):
        # cost per step must not depend on how far the streams are into their logical timelines
        offsets = [0, 540_000, 1_080_000, 2_000_000, 2 ** 31 + 5]
        per = []
        for p0 in offsets:
            fm = measure(fw, args, dev, rank, 1, timed=False, p0=p0, attention=False)
            fm.pop("h").close()
            per.append(fm["ms"] / args.steps)
        return {"p0": offsets, "ms_per_step": per, "spread": max(per) / min(per) - 1.0,
                "free_bytes_delta_over_timed_steps": free_delta}

    flat = None
    if args.flatness and rank == 0 and wl.name == "qwen" and not args.layers:
        flat = flatness(wl, m["free_bytes_delta"])

    # the other batched workloads, each with its own roofline (default run only)
    subs = {}
    if args.sub and rank == 0 and args.workload == "mixed" and not args.layers and not args.scheme:
        for name in ("qwen", "voxtral", "encoder"):
            sw, _ = bench_workload(argparse.Namespace(**dict(vars(args), workload=name)))
            sm = measure(sw, args, dev, rank, 1, timed=False, per_layer_step=args.per_layer)
            sm.pop("h").close()
            subs[name] = workload_figures(sw, SCHEME_NAMES[sw.scheme], sm, peak, peak_kind, args.steps, 1)
            subs[name]["free_bytes_delta_over_timed_steps"] = sm["free_bytes_delta"]
            if name == "qwen" and args.flatness:
                subs[name]["flatness"] = flatness(sw, sm["free_bytes_delta"])
        # the mixed-clock batch read the other way: every one of the 256 streams steps on every call
        # (no scheduler tick), 2.56 GB of windows per step
        import dataclasses
        sw = dataclasses.replace(wl, name="mixed_all_streams", tick_ms=0)
        sm = measure(sw, args, dev, rank, 1, timed=False, per_layer_step=args.per_layer)
        sm.pop("h").close()
        subs["mixed_all_streams"] = workload_figures(sw, SCHEME_NAMES[sw.scheme], sm, peak, peak_kind, args.steps, 1)
        subs["mixed_all_streams"]["free_bytes_delta_over_timed_steps"] = sm["free_bytes_delta"]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = oracle_timing(wl, args.cpu_seconds)

    if rank == 0:
        line = bench_line(wl, scheme_name, args, world, m, peak, peak_kind, variants, flat, e2e, cpu, subs)
        line["free_bytes_delta_over_timed_steps"] = m["free_bytes_delta"]
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def measure_e2e(h, wl, plan, args, dev):
    """Same metric through the public call with host buffers, every step: H2D of the step's inputs
    from pinned memory, rkv_step, D2H of the step's outputs.  The copies of neighbouring steps
    overlap the step's kernels (three CUDA streams, two device input/output sets), as a serving
    loop would run them."""
    import torch
    S, L, Q, hq, hkv, d = wl.n_streams, wl.n_layers, wl.q_per_step, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    A = max(len(p) for p in plan)
    nq, nkv = L * A * Q * hq * d, L * A * Q * hkv * d
    q_h = torch.randn(nq, dtype=torch.float32).mul_(wl.input_scale).to(torch.bfloat16).pin_memory()
    k_h = torch.randn(nkv, dtype=torch.float32).mul_(wl.input_scale).to(torch.bfloat16).pin_memory()
    v_h = torch.randn(nkv, dtype=torch.float32).mul_(wl.input_scale).to(torch.bfloat16).pin_memory()
    out_h = [torch.empty(nq, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    lse_h = [torch.empty(nq // d, dtype=torch.float32).pin_memory() for _ in range(2)]
    sets = [{"q": torch.empty(nq, dtype=torch.bfloat16, device=dev),
             "k": torch.empty(nkv, dtype=torch.bfloat16, device=dev),
             "v": torch.empty(nkv, dtype=torch.bfloat16, device=dev),
             "out": torch.empty(nq, dtype=torch.bfloat16, device=dev),
             "lse": torch.empty(nq // d, dtype=torch.float32, device=dev)} for _ in range(2)]
    steps = max(5, min(args.steps, 300))
    plan = [p for p in plan if p]
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("in", "run", "out")}
    bi = bo = n_ss = 0

    def one(i):
        nonlocal bi, bo, n_ss
        act = plan[i % len(plan)]
        a, b = len(act), sets[i % 2]
        n_q, n_kv = L * a * Q * hq * d, L * a * Q * hkv * d
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev["run"][i % 2])      # step i-2 has finished reading this set
            b["q"][:n_q].copy_(q_h[:n_q], non_blocking=True)
            b["k"][:n_kv].copy_(k_h[:n_kv], non_blocking=True)
            b["v"][:n_kv].copy_(v_h[:n_kv], non_blocking=True)
            ev["in"][i % 2].record(s_in)
        s_run.wait_event(ev["in"][i % 2])
        if i >= 2:
            s_run.wait_event(ev["out"][i % 2])         # step i-2's outputs have left this set
        h.step(act, b["q"], b["k"], b["v"], b["out"], b["lse"], stream=s_run)
        ev["run"][i % 2].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["run"][i % 2])
            out_h[i % 2][:n_q].copy_(b["out"][:n_q], non_blocking=True)
            lse_h[i % 2][:n_q // d].copy_(b["lse"][:n_q // d], non_blocking=True)
            ev["out"][i % 2].record(s_out)
        bi += (n_q + 2 * n_kv) * 2
        bo += n_q * 2 + (n_q // d) * 4
        n_ss += a

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    bi = bo = n_ss = 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(steps):
        one(i)
    s_in.wait_stream(s_out)
    s_in.wait_stream(s_run)
    e1.record(s_in)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    return {"value": n_ss / (ms / 1000.0), "unit": UNIT, "h2d_bytes_per_step": bi // steps,
            "d2h_bytes_per_step": bo // steps, "steps": steps,
            "call": "rkv_step on one stream, pinned-host H2D / D2H of every step's inputs and outputs on two "
                    "others, overlapping neighbouring steps (double-buffered)"}


def window_scan(args):
    """Per-layer decode-attention launch time against the window length: the intercept of a line
    through the points is the fixed cost of one launch, the slope the streaming bandwidth."""
    import torch

    import rolling_kv_sliding_rkv_b300 as rkv
    dev = torch.device("cuda")
    S, L, hq, hkv, d = 64, 36, 16, 2, 128
    points = []
    for W in (64, 128, 192, 256, 384, 512, 768):
        h = rkv.RollingKV([W] * S, [0] * S, device=dev, n_layers=L, n_streams=S, n_q_heads=hq, n_kv_heads=hkv,
                          head_dim=d, q_per_step=1, scheme=0, rope_theta=1e6)
        act = list(range(S))
        q = torch.randn(L * S * hq * d, device=dev).mul(0.088).to(torch.bfloat16)
        k = torch.randn(L * S * hkv * d, device=dev).mul(0.088).to(torch.bfloat16)
        v = torch.randn(L * S * hkv * d, device=dev).mul(0.088).to(torch.bfloat16)
        out = torch.empty_like(q)
        lse = torch.empty(L * S * hq, device=dev)
        for _ in range(W + 3):
            h.step(act, q, k, v, out, lse)
        h.begin_step(act)
        for layer in range(L):
            h.append_rope(layer, k[layer * S * hkv * d:], v[layer * S * hkv * d:])
        torch.cuda.synchronize()  # the capture stream does not wait for the default stream

        def body():
            for layer in range(L):
                h.decode_attn(layer, q[layer * S * hq * d:], out[layer * S * hq * d:], lse[layer * S * hq:])
        st = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(st):
            body()
            st.synchronize()
            with torch.cuda.graph(g, stream=st):
                body()
        for _ in range(5):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(max(5, args.steps)):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / max(5, args.steps) / L * 1000.0
        nbytes = S * (2 * W * hkv * d * 2 + hq * d * 2 * 2 + hq * 4)
        points.append({"window": W, "bytes_per_launch": nbytes, "us_per_launch": us})
        h.sync_status()
        h.close()
    xs = [p["bytes_per_launch"] for p in points]
    ys = [p["us_per_launch"] for p in points]
    mx, my = sum(xs) / len(xs), sum(ys) / len(ys)
    slope = sum((x - mx) * (y - my) for x, y in zip(xs, ys)) / sum((x - mx) ** 2 for x in xs)
    print(json.dumps({"scan": "one-layer decode attention launch against the window length",
                      "points": points, "fixed_us_per_launch": my - slope * mx,
                      "streaming_gbs": 1e-3 / slope}), flush=True)


def main():
    args = parse_args()
    if args.window_scan:
        window_scan(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
