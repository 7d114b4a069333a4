"""Per-call timings of the workloads other than the benchmark's mixed step.

    python -m sliding_window_gqa_ring_gb300.config_timing [--reps 50]

Workloads (``synth``): the single-request sliding decode (1 request, key count
1500, window 1024), the batched sliding decode (56 requests, key counts
uniform in [1024, 4096]), the single-request global verify (6005 keys, k = 4)
and the global verify sweeps (8 requests, k = 4 and k = 15, capacity 32768).
For each: the append alone (carat_ring_append), the attention alone
(carat_swa_attention / carat_global_verify_attention) and the fused
append+attention call, each the median of ``--reps`` CUDA-event timings with
L2 flushed (a 512 MB write) before every timed call.  Algorithmic bytes are the
attention's: each K/V row of a window or key range once, Q and the fp32 out;
GB/s and the fraction of the measured HBM copy rate (MEASURED_PEAKS.json)
follow.  Prints one JSON line per workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics

import torch

from . import engine, synth

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _peak():
    try:
        with open(os.path.join(_ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def _attention_bytes(w):
    total = 0
    row = w.kv_heads * w.head_dim * 2
    for b in range(w.batch):
        kc = int(w.key_counts[b])
        keys = kc - max(0, kc - w.proposal_count - w.window + 1) if w.window else kc
        total += keys * row * 2 + w.proposal_count * w.q_heads * w.head_dim * (2 + 4)
    return total


def _median_us(fn, reps, flush):
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3)
    return statistics.median(times)


def run(w, reps, flush, peak):
    if w.window:
        layer = engine.SlidingLayer(w.batch, window=w.window, q_heads=w.q_heads,
                                    kv_heads=w.kv_heads, head_dim=w.head_dim,
                                    max_proposals=w.proposal_count, scale=w.scale)
        inp = engine.stage_sliding(w, 0, layer)
    else:
        layer = engine.GlobalLayer(w.batch, capacity=w.capacity, q_heads=w.q_heads,
                                   kv_heads=w.kv_heads, head_dim=w.head_dim,
                                   max_proposals=w.proposal_count, scale=w.scale)
        inp = engine.stage_global(w, 0, layer, keep_history=False)
    out = torch.empty(inp.queries.shape, dtype=torch.float32, device=layer.device)
    append_us = _median_us(lambda: layer.append(inp.k_new, inp.v_new, inp.context_lengths),
                           reps, flush)
    attn_us = _median_us(lambda: layer.attend(inp.queries, inp.context_lengths, out=out),
                         reps, flush)
    fused_us = _median_us(lambda: layer.step(inp.queries, inp.k_new, inp.v_new,
                                             inp.context_lengths, out=out), reps, flush)
    nbytes = _attention_bytes(w)
    gbs = nbytes / (attn_us * 1e3)
    return {"workload": w.name, "batch": w.batch, "proposal_count": w.proposal_count,
            "attention_bytes": nbytes, "append_us": round(append_us, 2),
            "attention_us": round(attn_us, 2), "fused_append_attention_us": round(fused_us, 2),
            "attention_gb_s": round(gbs, 1), "attention_frac_of_peak": round(gbs / peak, 4),
            "l2": "flushed before every timed call (512 MB write)", "reps": reps}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--reps", type=int, default=50)
    args = ap.parse_args()
    peak, kind = _peak()
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    print(json.dumps({"peak_gb_s": peak, "peak_source": kind}), flush=True)
    for w in (synth.sliding_single(), synth.sliding_batched(), synth.global_single(),
              synth.global_sweep(4), synth.global_sweep(15)):
        print(json.dumps(run(w, args.reps, flush, peak)), flush=True)


if __name__ == "__main__":
    main()
