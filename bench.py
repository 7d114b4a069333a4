"""Benchmark: one mixed decode step (5 sliding + 1 global layer) on GB300.

Workload (seeded, synthetic; shapes from the pages): 64 requests, 4 speculative
positions each, context lengths log-uniform in [512, 32768].  A step is the
whole hot path once: for each of 5 sliding layers, carat_ring_append of the 4
new K/V rows per request into its 1024-slot ring, then carat_swa_attention read
in place from the rotated rings; for the global layer, the append into the full
cache, then carat_global_verify_attention (8 heads x 4 positions = 32 rows per
KV head, masked key tail).

Metric: algorithmic HBM bytes of the step / step time (GB/s), plus us per call.
Every layer call streams > 400 MB, more than the 129 MB L2, so no L2 flush is
needed between steps.  Timed steps repeat the same step at fixed positions (same
work every step).

The line's `configs` key times the single-layer workloads one call at a time
(L2 flushed before each call; the attention call also with the kernel's code
put back in the caches by an untimed call on other, small data): the
single-request sliding decode (key count
1500), the batched sliding decode (56 requests), the single-request global
verify (6005 keys, 4 proposals) and the 8-request global verify sweeps (4 and
15 proposals), with the launch floor and the pages' unfused design of the
global verify as an ablation.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

With --impl reference the fp64 CPU oracle is timed instead, on a bounded
sample of the same workload (the reference arm).  Under torchrun (N > 1) every
rank runs an independent replica on its own GPU (the path has no exchange step:
requests are independent), and the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SWA decode + GQA verify attention: HBM GB/s (% of ~8 TB/s), µs/layer call"
WORKLOAD = "mixed_decode_step_b64_k4_5swa_1global"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = os.path.join(ROOT, "sliding_window_gqa_ring_gb300", "csrc")


# ---------------------------------------------------------------------------
# Algorithmic bytes (what the method must move at least once per call)
# ---------------------------------------------------------------------------

def sliding_call_bytes(w, b):
    """Bytes one request moves in one sliding layer.

    attention: the K and V rows of the union of its queries' windows (the
    step's own rows included), its queries and its fp32 outputs.  The fused
    append+attention call adds the new rows written into the ring; the
    separate append reads and writes them and also saves and reads back the
    displaced rows."""
    k, hkv, d, hq = w.proposal_count, w.kv_heads, w.head_dim, w.q_heads
    kc = int(w.key_counts[b])
    ctx = kc - k
    keys = kc - max(0, ctx - w.window + 1)            # positions [max(0,ctx-W+1), kc)
    row = hkv * d * 2
    attn = keys * row * 2 + k * hq * d * 2 + k * hq * d * 4
    disp = sum(1 for i in range(k - 1) if ctx - w.window + 1 + i >= 0)
    fused_writes = k * row * 2
    append = k * row * 2 * 2 + disp * row * 2 * 2
    return attn, fused_writes, append


def fp8_attention_bytes(w, b):
    """Algorithmic bytes of FP8 sliding attention for request b: the window's
    e4m3 K and V rows (1 byte per element), bf16 queries, fp32 outputs."""
    k, hkv, d, hq = w.proposal_count, w.kv_heads, w.head_dim, w.q_heads
    kc = int(w.key_counts[b])
    ctx = kc - k
    keys = kc - max(0, ctx - w.window + 1)
    return keys * hkv * d * 2 + k * hq * d * 2 + k * hq * d * 4


def global_call_bytes(w, b):
    k, hkv, d, hq = w.proposal_count, w.kv_heads, w.head_dim, w.q_heads
    kc = int(w.key_counts[b])
    row = hkv * d * 2
    attn = kc * row * 2 + k * hq * d * 2 + k * hq * d * 4
    return attn, k * row * 2, k * row * 2 * 2


def step_bytes(sliding, glob):
    def tot(fn, w, i):
        return sum(fn(w, b)[i] for b in range(w.batch))
    s_attn, s_wr, s_app = (tot(sliding_call_bytes, sliding, i) for i in range(3))
    g_attn, g_wr, g_app = (tot(global_call_bytes, glob, i) for i in range(3))
    return {
        # fused calls (the step as timed)
        "swa_call": s_attn + s_wr, "global_call": g_attn + g_wr,
        "step": sliding.layers * (s_attn + s_wr) + g_attn + g_wr,
        # separate calls (timed for comparison)
        "swa_append": s_app, "swa_attention": s_attn, "global_append": g_app,
        "global_attention": g_attn,
        "step_separate": sliding.layers * (s_attn + s_app) + g_attn + g_app,
    }


# ---------------------------------------------------------------------------
# Helpers
# ---------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for f in sorted(os.listdir(KERNEL_SOURCES)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(KERNEL_SOURCES, f), "rb") as fh:
                h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(call):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("source_hash") != kernel_source_hash():
        return None
    e = t.get("calls", {}).get(call)
    return None if e is None else e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def max_over_ranks(value, device="cpu"):
    """Max of a float over all ranks (no-op without torch.distributed).  The
    only collective of the benchmark: the path itself exchanges nothing."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(bytes_per_step, steps, ms_max, world):
    """Whole-job GB/s: every replica moved bytes_per_step per step, and the
    job took as long as the slowest replica."""
    return world * bytes_per_step * steps / (ms_max / 1e3) / 1e9


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---------------------------------------------------------------------------
# Oracle sample (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_jobs(sliding, glob, requests):
    """(bytes, args) of oracle calls covering the sampled requests: every
    sliding layer and the global layer of each.  Inputs come from the seeded
    generators, exactly as staged on the GPU."""
    from sliding_window_gqa_ring_gb300 import synth
    jobs = []
    for b in requests:
        for layer in range(sliding.layers):
            first, kh, vh = synth.last_rows(sliding, layer, b, sliding.window
                                            + sliding.proposal_count)
            q = synth.queries(sliding, layer, b)
            jobs.append((sliding_call_bytes(sliding, b)[0], ("swa", layer, b),
                         (q, kh, vh, first, int(sliding.context_lengths[b]), sliding.window,
                          sliding.scale)))
        kc = int(glob.key_counts[b])
        kh = synth.history(glob, 0, b, 0, kc, "k")
        vh = synth.history(glob, 0, b, 0, kc, "v")
        q = synth.queries(glob, 0, b)
        jobs.append((global_call_bytes(glob, b)[0], ("global", 0, b),
                     (q, kh, vh, 0, int(glob.context_lengths[b]), 0, glob.scale)))
    return jobs


def time_oracle(jobs, threads):
    import oracle
    orc = oracle.default()
    t0 = time.perf_counter()
    outs = orc.attention_batch([j[2] for j in jobs], threads=threads)
    dt = time.perf_counter() - t0
    return outs, dt


# ---------------------------------------------------------------------------
# Per-call timings of the single-layer workloads (configs 1-4)
# ---------------------------------------------------------------------------

def config_attention_bytes(w):
    """Algorithmic bytes of one attention call of workload w: each K/V row of
    every request's window (sliding) or key range (global) once, its queries
    and its fp32 outputs."""
    total = 0
    row = w.kv_heads * w.head_dim * 2
    for b in range(w.batch):
        kc = int(w.key_counts[b])
        keys = kc - max(0, kc - w.proposal_count - w.window + 1) if w.window else kc
        total += keys * row * 2 + w.proposal_count * w.q_heads * w.head_dim * (2 + 4)
    return total


def median_call_us(fn, reps, flush, stream, trimmed=None, warm=None):
    """Median over reps of one call timed with CUDA events on `stream`, with
    the L2 flushed (a write larger than L2) before each timed call.  CUDA event
    timestamps on this GPU come in steps of about 2 us, so the mean of the
    middle 80% of the samples (`trimmed`, a one-element list, if given) is
    also recorded: its resolution is finer than one step.  `warm`, if given,
    runs untimed between the flush and the call (a call of the same kernel on
    other, small data: the kernel's code is back in the caches, the timed
    call's data is not)."""
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        flush.zero_()
        if warm is not None:
            warm()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3)
    if trimmed is not None:
        ts = sorted(times)
        cut = len(ts) // 10
        mid = ts[cut:len(ts) - cut] or ts
        trimmed.append(sum(mid) / len(mid))
    return statistics.median(times)


def run_configs(dev, reps, peak, peak_kind, ablation_reps):
    """Configs 1-4 (the single-layer workloads): append alone, attention
    alone and the fused append+attention call, each the median of `reps`
    L2-flushed calls; the launch floor; and the unfused design of the pages as
    an ablation on the global workloads."""
    import torch

    from sliding_window_gqa_ring_gb300 import ablation, carat, engine, synth
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    ft = []
    floor1 = median_call_us(lambda: carat.carat_launch_floor(False), reps, flush, stream, ft)
    floor2 = median_call_us(lambda: carat.carat_launch_floor(True), reps, flush, stream, ft)
    rows = []

    def staged(w):
        if w.window:
            layer = engine.SlidingLayer(w.batch, window=w.window, q_heads=w.q_heads,
                                        kv_heads=w.kv_heads, head_dim=w.head_dim,
                                        max_proposals=w.proposal_count, scale=w.scale,
                                        device=dev)
            inp = engine.stage_sliding(w, 0, layer)
        else:
            layer = engine.GlobalLayer(w.batch, capacity=w.capacity, q_heads=w.q_heads,
                                       kv_heads=w.kv_heads, head_dim=w.head_dim,
                                       max_proposals=w.proposal_count, scale=w.scale,
                                       device=dev)
            inp = engine.stage_global(w, 0, layer, keep_history=False)
        inp.host.clear()
        return layer, inp

    for w in (synth.sliding_single(), synth.sliding_batched(), synth.global_single(),
              synth.global_sweep(4), synth.global_sweep(15)):
        layer, inp = staged(w)
        out = torch.empty(inp.queries.shape, dtype=torch.float32, device=dev)
        # the same shapes (so the same kernel and schedule) over 130 keys a
        # request, on memory of its own: its call before a timed one puts
        # the kernel's code back in the caches without the timed call's data
        ws = synth.small(w.name + "_warm", seed=w.seed + 7, batch=w.batch,
                         proposal_count=w.proposal_count, q_heads=w.q_heads,
                         kv_heads=w.kv_heads, head_dim=w.head_dim,
                         key_counts=[max(130, w.proposal_count)] * w.batch, window=w.window,
                         capacity=w.capacity, scale=w.scale)
        wlayer, winp = staged(ws)
        wlayer.append(winp.k_new, winp.v_new, winp.context_lengths)
        wout = torch.empty(winp.queries.shape, dtype=torch.float32, device=dev)

        def append():
            layer.append(inp.k_new, inp.v_new, inp.context_lengths)

        def attend():
            layer.attend(inp.queries, inp.context_lengths, out=out)

        def fused():
            layer.step(inp.queries, inp.k_new, inp.v_new, inp.context_lengths, out=out)

        append()
        n0 = carat.kernel_launches()
        attend()
        attn_launches = carat.kernel_launches() - n0
        def warm_attend():
            wlayer.attend(winp.queries, winp.context_lengths, out=wout)

        tm = []
        append_us = median_call_us(append, reps, flush, stream)
        attn_us = median_call_us(attend, reps, flush, stream, tm)
        fused_us = median_call_us(fused, reps, flush, stream, tm)
        attn_warm_us = median_call_us(attend, reps, flush, stream, tm, warm=warm_attend)
        nbytes = config_attention_bytes(w)
        floor = floor2 if attn_launches > 1 else floor1
        gbs = nbytes / (attn_us * 1e3)
        rows.append({"workload": w.name, "batch": w.batch, "proposal_count": w.proposal_count,
                     "attention_bytes": nbytes, "append_us": round(append_us, 2),
                     "attention_us": round(attn_us, 2), "fused_us": round(fused_us, 2),
                     "attention_us_trimmed_mean": round(tm[0], 2),
                     "fused_us_trimmed_mean": round(tm[1], 2),
                     "attention_gb_s": round(gbs, 1), "attention_frac": round(gbs / peak, 4),
                     "attention_us_code_warm": round(attn_warm_us, 2),
                     "attention_us_code_warm_trimmed_mean": round(tm[2], 2),
                     "attention_launches": attn_launches,
                     "attention_floor_us": round(floor, 2),
                     "attention_excess_over_floor_us": round(attn_us - floor, 2),
                     "attention_frac_excluding_floor": round(
                         nbytes / max(attn_us - floor, 1e-3) / 1e3 / peak, 4)})
        del layer, inp, out, wlayer, winp, wout
        torch.cuda.empty_cache()
    abl = []
    if ablation_reps > 0:
        for w in (synth.global_single(), synth.global_sweep(4), synth.global_sweep(15)):
            abl.append(ablation.measure(w, ablation_reps, flush))
            torch.cuda.empty_cache()
    return {"workloads": rows,
            "launch_floor_us": {"one_empty_launch": round(floor1, 2),
                                "empty_launch_then_dependent_launch": round(floor2, 2),
                                "trimmed_means": [round(x, 2) for x in ft]},
            "peak_gb_s": peak, "peak_source": f"{peak_kind} hbm_gbs",
            "timing": (f"median of {reps} calls, CUDA events on the launching stream, L2 "
                       "flushed (512 MB write) before every timed call; floor = the same "
                       "timing of carat_launch_floor (one empty launch, or two with the "
                       "second a programmatic dependent launch, matching the call's launch "
                       "count); attention_us_code_warm: the same, with an untimed call of "
                       "the same kernel on small data of its own between the flush and "
                       "the timed call (code in the caches, data not)"),
            "ablation_unfused_global_verify": abl}


# ---------------------------------------------------------------------------
# The GPU arm
# ---------------------------------------------------------------------------

def run_carat(args, world, rank, local):
    import torch

    from sliding_window_gqa_ring_gb300 import carat, engine, synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sliding, glob = synth.mixed_step()
    B, k = sliding.batch, sliding.proposal_count
    nbytes = step_bytes(sliding, glob)

    # --- stage the state: rings and caches written through carat_ring_append
    t_stage = time.perf_counter()
    sample = list(range(0, B, max(1, B // args.sample_requests))) if rank == 0 else []
    layers = []
    for li in range(sliding.layers):
        lay = engine.SlidingLayer(B, window=sliding.window, q_heads=sliding.q_heads,
                                  kv_heads=sliding.kv_heads, head_dim=sliding.head_dim,
                                  max_proposals=k, scale=sliding.scale, device=dev)
        inp = engine.stage_sliding(sliding, li, lay)
        if li > 0 or not args.fp8:
            inp.host["hist"] = {}          # layer 0's history sizes the FP8 scales
        layers.append((lay, inp))
    glay = engine.GlobalLayer(B, capacity=glob.capacity, q_heads=glob.q_heads,
                              kv_heads=glob.kv_heads, head_dim=glob.head_dim, max_proposals=k,
                              scale=glob.scale, device=dev)
    ginp = engine.stage_global(glob, 0, glay, keep_history=False)
    outs = [torch.empty(inp.queries.shape, dtype=torch.float32, device=dev) for _, inp in layers]
    gout = torch.empty(ginp.queries.shape, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    stage_s = time.perf_counter() - t_stage

    stream = torch.cuda.current_stream()
    dstep = engine.DecodeStep(
        [lay for lay, _ in layers] + [glay],
        [(inp.queries, inp.k_new, inp.v_new, inp.context_lengths) for _, inp in layers]
        + [(ginp.queries, ginp.k_new, ginp.v_new, ginp.context_lengths)],
        outs + [gout])

    def step():
        dstep.run()

    # --- first step: its outputs are checked against the oracle sample
    step()
    torch.cuda.synchronize()
    first_outs = [o.cpu().numpy() for o in outs]
    first_gout = gout.cpu().numpy()

    cpu_baseline = None
    parity = None
    if rank == 0 and args.cpu_baseline:
        jobs = oracle_jobs(sliding, glob, sample)
        threads = os.cpu_count() or 1
        refs, dt = time_oracle(jobs, threads)
        moved = sum(j[0] for j in jobs)
        worst = 0.0
        for (nb, (kind, li, b), _), ref in zip(jobs, refs):
            got = first_outs[li][b] if kind == "swa" else first_gout[b]
            worst = max(worst, float(np.abs(got - ref).max()))
        parity = {"requests": len(sample), "max_abs_err": worst, "gate": 2e-2,
                  "ok": worst <= 2e-2}
        cpu_baseline = {"value": moved / dt / 1e9, "unit": "GB/s", "cores": threads,
                        "kind": "oracle",
                        "sample": (f"fp64 C oracle, all 6 layers' attention for {len(sample)} of "
                                   f"{B} requests ({moved / 1e9:.3f} GB of algorithmic bytes), "
                                   f"{dt:.2f} s wall on {threads} threads")}

    # --- warm-up
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # --- timed region (uninstrumented): the step as a user runs it
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = carat.kernel_launches()
    with ClockSampler(local) as clk:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    launches = carat.kernel_launches() - launches0
    ms = max_over_ranks(e0.elapsed_time(e1), dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = clk.summary()
    ms_per_step = ms / args.steps
    value = replica_throughput(nbytes["step"], args.steps, ms, world)

    # --- a second timed region of the same steps with CUDA events around
    # every call (the records add a few us per call, so `value` comes from the
    # region above)
    nrep = min(args.steps, 300)

    def bracket(fn):
        a = torch.cuda.Event(enable_timing=True)
        bb = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        bb.record(stream)
        return a, bb

    marks = {"swa_call": [], "global_call": []}
    for _ in range(nrep):
        for (lay, inp), out in zip(layers, outs):
            marks["swa_call"].append(bracket(lambda: lay.step(
                inp.queries, inp.k_new, inp.v_new, inp.context_lengths, out=out)))
        marks["global_call"].append(bracket(lambda: glay.step(
            ginp.queries, ginp.k_new, ginp.v_new, ginp.context_lengths, out=gout)))
    torch.cuda.synchronize()
    per_call = {}
    for name, pairs in marks.items():
        mean_us = statistics.mean(a.elapsed_time(bb) * 1e3 for a, bb in pairs)
        per_call[name] = {"us": round(mean_us, 3), "gb_s": round(nbytes[name] / (mean_us * 1e3), 1),
                          "bytes": nbytes[name],
                          "launches_per_step": (sliding.layers if name.startswith("swa") else 1)}

    # --- the same calls back to back, one kind at a time, one event pair per
    # region: the mean launch duration of each kind without per-call records
    def region_us(fn, calls_per_rep):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        bb = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(nrep):
            fn()
        bb.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(bb) * 1e3 / (nrep * calls_per_rep)

    def all_sliding():
        for (lay, inp), out in zip(layers, outs):
            lay.step(inp.queries, inp.k_new, inp.v_new, inp.context_lengths, out=out)

    b2b = {"swa_call": region_us(all_sliding, sliding.layers),
           "global_call": region_us(lambda: glay.step(ginp.queries, ginp.k_new, ginp.v_new,
                                                      ginp.context_lengths, out=gout), 1)}
    per_call_b2b = {n: {"us": round(us, 3), "gb_s": round(nbytes[n] / (us * 1e3), 1)}
                    for n, us in b2b.items()}

    # --- the same step through the separate append and attention calls
    def step_separate():
        for (lay, inp), out in zip(layers, outs):
            lay.step(inp.queries, inp.k_new, inp.v_new, inp.context_lengths, out=out, fused=False)
        glay.step(ginp.queries, ginp.k_new, ginp.v_new, ginp.context_lengths, out=gout,
                  fused=False)

    for _ in range(3):
        step_separate()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(nrep):
        step_separate()
    e1.record(stream)
    torch.cuda.synchronize()
    sep_ms = e0.elapsed_time(e1) / nrep
    separate = {"ms_per_step": round(sep_ms, 4),
                "gb_s": round(nbytes["step_separate"] / (sep_ms * 1e6), 1),
                "step_bytes": nbytes["step_separate"],
                "calls": "carat_ring_append + carat_swa_attention (x5), carat_ring_append + "
                         "carat_global_verify_attention"}
    share = {n: per_call[n]["us"] * per_call[n]["launches_per_step"] for n in per_call}
    dominant = max(share, key=share.get)
    peak, peak_kind = measured_peaks()
    achieved = per_call_b2b[dominant]["gb_s"]
    roofline = {"bound": "hbm", "kernel": dominant, "achieved": achieved, "peak": peak,
                "peak_source": f"{peak_kind} hbm_gbs", "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": profiled_traffic(dominant),
                "algorithmic_bytes_per_launch": nbytes[dominant],
                "timing": ("mean launch duration of the fused append+attention call (one "
                           "kernel launch): CUDA events around a region of up to 300 x 5 "
                           "back-to-back sliding calls on the launching stream, divided by the "
                           "calls; per_call brackets every call in the step instead (records "
                           "included)")}

    # --- the same step with every cache in one shared pool: each sliding
    # layer's rings and the global layer's pages are allocated from one K and
    # one V pool by the library's allocator (pages of 512 KiB = a ring's 1/8)
    pooled = None
    if args.shared_pool:
        page_bytes = 128 * sliding.kv_heads * sliding.head_dim * 2
        g_rows = page_bytes // (glob.kv_heads * glob.head_dim * 2)
        g_pages = [-(-int(kc) // g_rows) for kc in glob.key_counts]
        npages = sliding.layers * B * 8 + sum(g_pages) + 8
        spool = engine.SharedPool(npages, page_bytes, 8, device=dev)
        p_layers, p_inputs = [], []
        for li in range(sliding.layers):
            ids = [spool.alloc.alloc_ring() for _ in range(B)]
            lay = engine.SlidingLayer(npages // 8, window=sliding.window, q_heads=sliding.q_heads,
                                      kv_heads=sliding.kv_heads, head_dim=sliding.head_dim,
                                      max_batch=B, max_proposals=k, scale=sliding.scale,
                                      device=dev, rings=spool.rings(sliding.window,
                                                                    sliding.kv_heads,
                                                                    sliding.head_dim))
            lay.ring_ids = torch.as_tensor(np.array(ids, np.int32), device=dev)
            pin = engine.stage_sliding(sliding, li, lay, ring_ids=ids)
            p_layers.append(lay)
            p_inputs.append((pin.queries, pin.k_new, pin.v_new, pin.context_lengths))
        table = np.zeros((B, max(g_pages)), np.int32)
        for b, n in enumerate(g_pages):
            table[b, :n] = spool.alloc.alloc_pages(n)
        pg = engine.PagedGlobalLayer(spool, torch.as_tensor(table, device=dev),
                                     q_heads=glob.q_heads, kv_heads=glob.kv_heads,
                                     head_dim=glob.head_dim, max_proposals=k, scale=glob.scale)
        pgin = engine.stage_global_paged(glob, 0, pg, keep_history=False)
        p_layers.append(pg)
        p_inputs.append((pgin.queries, pgin.k_new, pgin.v_new, pgin.context_lengths))
        pstep = engine.DecodeStep(p_layers, p_inputs)
        for _ in range(3):
            pstep.run()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(nrep):
            pstep.run()
        e1.record(stream)
        torch.cuda.synchronize()
        pool_ms = e0.elapsed_time(e1) / nrep
        pooled = {"ms_per_step": round(pool_ms, 4),
                  "gb_s": round(nbytes["step"] / (pool_ms * 1e6), 1),
                  "pool_pages": npages, "page_bytes": page_bytes,
                  "layout": "5 x 64 rings of 8 pages + paged global caches, one K and one V pool"}
        del pstep, p_layers, p_inputs, spool

    # --- FP8 (e4m3) rings for one sliding layer of the same step
    # ("gemma-cuda-hybrid", "Features" / "Server": the KV cache is FP8 e4m3):
    # append + attention and attention alone, per call; per-tensor scales
    # max|x| / 448 of the layer
    fp8 = None
    if args.fp8:
        hist = layers[0][1].host["hist"]
        kmax = max(float(np.abs(synth.bf16_to_float(hist[b][1])).max()) for b in range(B))
        vmax = max(float(np.abs(synth.bf16_to_float(hist[b][2])).max()) for b in range(B))
        layers[0][1].host["hist"] = {}
        f8 = engine.Fp8SlidingLayer(B, k_scale=kmax / 448.0, v_scale=vmax / 448.0,
                                    window=sliding.window, q_heads=sliding.q_heads,
                                    kv_heads=sliding.kv_heads, head_dim=sliding.head_dim,
                                    max_proposals=k, scale=sliding.scale, device=dev)
        f8in = engine.stage_sliding(sliding, 0, f8)
        f8out = torch.empty(f8in.queries.shape, dtype=torch.float32, device=dev)

        def f8_time(fn, reps):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) * 1e3 / reps

        reps = max(3, min(nrep, 300))
        f8.append(f8in.k_new, f8in.v_new, f8in.context_lengths)
        att_us = f8_time(lambda: f8.attend(f8in.queries, f8in.context_lengths, out=f8out), reps)
        both_us = f8_time(lambda: (f8.append(f8in.k_new, f8in.v_new, f8in.context_lengths),
                                   f8.attend(f8in.queries, f8in.context_lengths, out=f8out)), reps)
        att_bytes = sum(fp8_attention_bytes(sliding, b) for b in range(B))
        fp8 = {"attention_us": round(att_us, 3),
               "attention_gb_s": round(att_bytes / (att_us * 1e3), 1),
               "attention_bytes": att_bytes,
               "append_plus_attention_us": round(both_us, 3),
               "bf16_fused_call_us": per_call["swa_call"]["us"],
               "scales": {"k": kmax / 448.0, "v": vmax / 448.0},
               "layer": "sliding layer 0 of the step: e4m3 rings, bf16 queries, fp32 out"}
        del f8, f8in, f8out

    # --- the step replayed from a CUDA graph (one host launch per step)
    dstep.capture()
    for _ in range(3):
        dstep.replay()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(nrep):
        dstep.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    graph_ms = e0.elapsed_time(e1) / nrep
    graph = {"ms_per_step": round(graph_ms, 4),
             "gb_s": round(nbytes["step"] / (graph_ms * 1e6), 1)}

    # --- end to end through the public API with host buffers: every step
    # copies all layers' inputs from pinned host memory and every output back,
    # on a copy stream that overlaps them with the layers' compute
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu())  # noqa: E731
    h_in = [tuple(pin(x) for x in din) for din in dstep.inputs]
    h_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in dstep.outputs]
    h2d = sum(x.numel() * x.element_size() for hi in h_in for x in hi)
    d2h = sum(o.numel() * o.element_size() for o in h_out)

    def e2e_step():
        dstep.run_from_host(h_in, h_out)

    for _ in range(3):
        e2e_step()
    dstep.finish()
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 200))
    if world > 1:
        torch.distributed.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    dstep.finish()   # the last step's outputs are in host memory before e1
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    e2e_value = replica_throughput(nbytes["step"], e2e_steps, e2e_ms, world)

    # --- configs 1-4 (rank 0): per-call timings of the single-layer workloads,
    # under a clock record of their own
    configs = None
    if rank == 0 and args.configs:
        del dstep, layers, glay, ginp, outs, gout, h_in, h_out
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        with ClockSampler(local) as cclk:
            configs = run_configs(dev, args.config_reps, peak, peak_kind, args.ablation_reps)
        configs["clocks"] = cclk.summary()

    status = carat.carat_get_device_status(clear=True)
    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16; shapes of the pages' Gemma-4 layers)",
        "config": {"workload": WORKLOAD, "batch": B, "proposal_count": k,
                   "sliding_layers": sliding.layers, "global_layers": 1,
                   "window": sliding.window, "sliding_heads": "16 q / 8 kv x 256",
                   "global_heads": "16 q / 2 kv x 512", "global_capacity": glob.capacity,
                   "context_lengths": "log-uniform [512, 32768], seed 1006",
                   "mean_key_count": float(np.mean(glob.key_counts)),
                   "step_bytes": nbytes["step"],
                   "l2": "no flush: every layer call streams more than the 129 MB L2",
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline,
        "per_call": per_call,
        "per_call_back_to_back": per_call_b2b,
        "separate_calls": separate,
        "cuda_graph": graph,
        "shared_pool": pooled,
        "fp8_sliding": fp8,
        "configs": configs,
        "cpu_baseline": cpu_baseline,
        "parity_sample": parity,
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / e2e_steps, 4),
                "steps": e2e_steps,
                "how": "engine.DecodeStep.run_from_host: pinned host inputs of all 6 layers in, "
                       "all outputs out, on a copy-in and a copy-out stream into two sets of "
                       "device buffers that alternate between steps (the next step's inputs "
                       "stream in while this one computes); the timed region ends after the "
                       "last step's outputs are in host memory"},
        "gpu_launches": launches,
        "clocks": clocks,
        "device_status": status,
        "stage_seconds": round(stage_s, 1),
    }
    return line


# ---------------------------------------------------------------------------
# The reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args, world, rank):
    if rank != 0:
        return None
    from sliding_window_gqa_ring_gb300 import synth
    sliding, glob = synth.mixed_step()
    threads = os.cpu_count() or 1
    # one step = the oracle over a bounded slice of the step's work, sized so
    # the whole --warmup + --steps run stays within about a minute
    budget_s = 60.0 / max(1, args.steps + args.warmup)
    order = list(range(sliding.batch))
    jobs_all = oracle_jobs(sliding, glob, order[:threads])
    # estimate cost per job from bytes (global jobs dominate)
    _, t_one = time_oracle(jobs_all[:1], 1)
    per_byte = t_one / max(1, jobs_all[0][0])
    target_bytes = budget_s * threads / per_byte
    jobs, acc = [], 0
    for j in sorted(jobs_all, key=lambda j: j[0]):
        if acc + j[0] > target_bytes and jobs:
            break
        jobs.append(j)
        acc += j[0]
    for _ in range(args.warmup):
        time_oracle(jobs, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time_oracle(jobs, threads)
    dt = time.perf_counter() - t0
    moved = sum(j[0] for j in jobs) * args.steps
    value = moved / dt / 1e9
    sample = (f"fp64 C oracle, {len(jobs)} attention calls per step (one request-layer each, "
              f"{sum(j[0] for j in jobs) / 1e6:.1f} MB algorithmic) on {threads} threads")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "batch": sliding.batch,
                       "proposal_count": sliding.proposal_count},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["carat", "reference"], default="carat")
    ap.add_argument("--sample-requests", type=int, default=16,
                    help="requests the oracle recomputes for the CPU baseline / parity sample")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-fp8", dest="fp8", action="store_false",
                    help="skip the FP8 (e4m3) sliding-layer measurement")
    ap.add_argument("--no-shared-pool", dest="shared_pool", action="store_false",
                    help="skip timing the step with all caches in one shared pool")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip the per-call timings of the single-layer workloads")
    ap.add_argument("--config-reps", type=int, default=50,
                    help="L2-flushed calls per median in the single-layer timings")
    ap.add_argument("--ablation-reps", type=int, default=20,
                    help="repetitions per median of the unfused-design ablation (0: skip)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    line = run_carat(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
