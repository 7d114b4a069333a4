"""Ablation: global verify attention as separate library steps, against the
fused kernel.

    python -m sliding_window_gqa_ring_gb300.ablation [--reps 50]

"Announcing Carat: An inference engine designed for Gemma 4" computes global
verify attention with separate library operations per request and keeps the
scores in device memory between them ("More FLOPs can be faster"); the rows
of those operations are the query heads of one KV head times the proposal
positions ("Doing it all in one kernel can be slower"); and the key dimension
is padded to a multiple of 64 with zero, masked rows so that the library picks
a tensor-core GEMM for the score product.  This module builds that unfused
design from its definition, for KV head c of request b with the rows r =
(position j, head h') and n keys (the key count, or it rounded up to 64):

    S = scale * Q_c K_c[0:n]^T        one GEMM per KV head, S stored in memory
    P = softmax(S masked)             key t hidden from row r when t > the
                                      position of r (causal; the padding too)
    O = P V_c[0:n]                    one GEMM per KV head

with cuBLAS GEMMs (torch.matmul), in one of two precisions:

  "bf16"  the pages' setting: the GEMMs read bf16 and write bf16, so S, P and
          O are rounded to bf16 between the steps (softmax in fp32);
  "fp32"  S, P and O kept in fp32 (the bf16 inputs widened exactly; fp32
          GEMMs).

It is a comparison, not part of the attention path: ``measure`` times it
next to carat_global_verify_attention on the same seeded inputs (CUDA
events, L2 flushed before every repetition), including the score GEMM alone
at the exact and at the padded key count.
"""
from __future__ import annotations

import argparse
import json
import statistics

import torch

from . import engine, synth


def unfused_verify(key_cache, value_cache, queries, key_counts, proposal_count, scale,
                   precision="bf16", pad64=False):
    """Global verify attention of every request as separate library steps.

    key_cache, value_cache: bf16 [B][capacity][Hkv][D] holding this step's
    rows; queries bf16 [B][k][Hq][D]; key_counts: host ints.  Returns fp32
    [B][k][Hq][D]."""
    batch, k, q_heads, head_dim = queries.shape
    capacity, kv_heads = key_cache.shape[1], key_cache.shape[2]
    g = q_heads // kv_heads
    dt = torch.bfloat16 if precision == "bf16" else torch.float32
    outs = []
    for b in range(batch):
        kc = int(key_counts[b])
        n = min(-(-kc // 64) * 64, capacity) if pad64 else kc
        first_q = kc - k                       # position of proposal 0
        # rows of KV head c: (position j, head h') -> [Hkv][k*g][D]
        q = queries[b].view(k, kv_heads, g, head_dim).transpose(0, 1)
        q = q.reshape(kv_heads, k * g, head_dim).to(dt)
        keys = key_cache[b, :n].transpose(0, 1).to(dt)        # [Hkv][n][D]
        vals = value_cache[b, :n].transpose(0, 1).to(dt)
        s = torch.matmul(q, keys.transpose(1, 2)).float() * scale
        row_pos = first_q + torch.arange(k, device=q.device).repeat_interleave(g)
        hidden = torch.arange(n, device=q.device)[None, :] > row_pos[:, None]
        p = torch.softmax(s.masked_fill(hidden[None], float("-inf")), dim=-1)
        o = torch.matmul(p.to(dt), vals).float()                # [Hkv][k*g][D]
        outs.append(o.view(kv_heads, k, g, head_dim).transpose(0, 1).reshape(k, q_heads,
                                                                             head_dim))
    return torch.stack(outs)


def _median_us(fn, reps, flush):
    times = []
    for r in range(reps + 3):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        if r >= 3:
            times.append(e0.elapsed_time(e1) * 1e3)
    return statistics.median(times)


def staged(w):
    """A global layer holding workload w's history and this step's rows."""
    layer = engine.GlobalLayer(w.batch, capacity=w.capacity, q_heads=w.q_heads,
                               kv_heads=w.kv_heads, head_dim=w.head_dim,
                               max_proposals=w.proposal_count, scale=w.scale)
    inp = engine.stage_global(w, 0, layer, keep_history=False)
    layer.append(inp.k_new, inp.v_new, inp.context_lengths)
    return layer, inp


def measure(w, reps, flush=None):
    """Times of the fused call and of the unfused design (bf16, exact and
    padded key counts) on workload w, and the score GEMM alone for its longest
    request at the exact and the padded key count."""
    layer, inp = staged(w)
    if flush is None:
        flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=layer.device)
    out = torch.empty(inp.queries.shape, dtype=torch.float32, device=layer.device)

    def fused():
        layer.attend(inp.queries, inp.context_lengths, out=out)

    def unfused(pad64):
        return unfused_verify(layer.key_cache, layer.value_cache, inp.queries, w.key_counts,
                              w.proposal_count, w.scale, "bf16", pad64)

    fused()
    exact, padded = unfused(False), unfused(True)
    torch.cuda.synchronize()
    diffs = {"fused_vs_unfused_bf16": float((out - exact).abs().max()),
             "padded_vs_exact": float((padded - exact).abs().max())}
    bmax = max(range(w.batch), key=lambda b: int(w.key_counts[b]))
    kc = int(w.key_counts[bmax])
    g = w.q_heads // w.kv_heads
    qm = inp.queries[bmax].view(w.proposal_count, w.kv_heads, g, w.head_dim).transpose(0, 1)
    qm = qm.reshape(w.kv_heads, w.proposal_count * g, w.head_dim).contiguous()
    kpad = min(-(-kc // 64) * 64, w.capacity)
    k_exact = layer.key_cache[bmax, :kc].permute(1, 2, 0)       # [Hkv][D][n]
    k_pad = layer.key_cache[bmax, :kpad].permute(1, 2, 0)
    res = {"workload": w.name, "batch": w.batch, "proposal_count": w.proposal_count,
           "fused_us": round(_median_us(fused, reps, flush), 2),
           "unfused_bf16_exact_us": round(_median_us(lambda: unfused(False), reps, flush), 1),
           "unfused_bf16_padded64_us": round(_median_us(lambda: unfused(True), reps, flush), 1),
           "score_gemm_keys": [kc, kpad],
           "score_gemm_exact_us": round(_median_us(lambda: torch.matmul(qm, k_exact), reps,
                                                   flush), 2),
           "score_gemm_padded64_us": round(_median_us(lambda: torch.matmul(qm, k_pad), reps,
                                                      flush), 2),
           "max_abs_diff": diffs, "reps": reps,
           "l2": "flushed before every repetition (512 MB write)"}
    del layer, inp, out
    return res


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--reps", type=int, default=50)
    args = ap.parse_args()
    for w in (synth.global_single(), synth.global_sweep(4), synth.global_sweep(15)):
        print(json.dumps(measure(w, args.reps)), flush=True)


if __name__ == "__main__":
    main()
