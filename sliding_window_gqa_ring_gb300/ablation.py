"""Ablation: the unfused three-pass global verify against the fused kernel.

    python -m sliding_window_gqa_ring_gb300.ablation [--reps 50]

"Announcing Carat: An inference engine designed for Gemma 4" computes global
verify attention as three library calls per request -- a bf16 QK^T GEMM into a
scores buffer in memory, a causal softmax over it, and a PV GEMM ("More FLOPs
can be faster") -- grouping the 8 query heads of a KV head with the proposal
positions into one 32-row matrix ("Doing it all in one kernel can be
slower"), and pads the key count to a multiple of 64 with a zero, masked
tail so the library picks a tensor-core GEMM.  This module runs that design
on this GPU (cuBLAS through torch.matmul, scores in HBM, padded or not) next
to carat_global_verify_attention on the same seeded inputs, checks that all
three agree, and prints one JSON line per workload with CUDA-event times
(median, L2 flushed before every repetition), including QK^T alone at the
exact and the padded key count.  Scores are materialised in bf16, as a GEMM
with bf16 output does; with 1% of keys scaled by 8 that rounding moves logits
visibly, which the max_abs_diff fields show.  It is a comparison, not part
of the attention path.
"""
from __future__ import annotations

import argparse
import json
import statistics

import torch

from . import engine, synth


def _three_pass(layer, inp, w, pad64):
    """Per request: scores = Q_rows . K^T (bf16 GEMM output, widened to fp32 in HBM),
    masked softmax, P (bf16) . V."""
    g = w.q_heads // w.kv_heads
    k = w.proposal_count
    outs = []
    for b in range(w.batch):
        kc = int(w.key_counts[b])
        n = ((kc + 63) // 64) * 64 if pad64 else kc
        n = min(n, w.capacity)
        ctx = kc - k
        # [Hkv, rows = k*g, D]: rows ordered (position j, head h') as in the tile
        q = inp.queries[b].view(k, w.kv_heads, g, w.head_dim).permute(1, 0, 2, 3)
        q = q.reshape(w.kv_heads, k * g, w.head_dim)
        kk = layer.key_cache[b, :n].permute(1, 0, 2)          # [Hkv, n, D]
        vv = layer.value_cache[b, :n].permute(1, 0, 2)
        scores = torch.matmul(q, kk.transpose(1, 2)).float() * w.scale   # qk_matmul
        pos = torch.arange(n, device=q.device)
        qpos = ctx + torch.arange(k, device=q.device).repeat_interleave(g)
        mask = pos[None, :] > qpos[:, None]                               # causal + padded tail
        p = torch.softmax(scores.masked_fill(mask[None], float("-inf")), dim=-1)  # causal_softmax
        o = torch.matmul(p.to(torch.bfloat16), vv)                        # pv_matmul
        o = o.float().reshape(w.kv_heads, k, g, w.head_dim).permute(1, 0, 2, 3)
        outs.append(o.reshape(k, w.q_heads, w.head_dim))
    return torch.stack(outs)


def _time(fn, reps, flush):
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


def run(w, reps):
    layer = engine.GlobalLayer(w.batch, capacity=w.capacity, q_heads=w.q_heads,
                               kv_heads=w.kv_heads, head_dim=w.head_dim,
                               max_proposals=w.proposal_count, scale=w.scale)
    inp = engine.stage_global(w, 0, layer, keep_history=False)
    layer.append(inp.k_new, inp.v_new, inp.context_lengths)
    out = torch.empty(inp.queries.shape, dtype=torch.float32, device=layer.device)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=layer.device)

    def fused():
        layer.attend(inp.queries, inp.context_lengths, out=out)

    fused()
    ref = out.clone()
    exact = _three_pass(layer, inp, w, pad64=False)
    padded = _three_pass(layer, inp, w, pad64=True)
    torch.cuda.synchronize()
    agree = {
        "fused_vs_three_pass": float((ref - exact).abs().max()),
        "padded_vs_exact": float((padded - exact).abs().max()),
    }
    # QK^T alone at the exact and the padded key count (the pages' 6,005 vs
    # 6,016 comparison), for the longest request of the workload
    bmax = int(max(range(w.batch), key=lambda b: int(w.key_counts[b])))
    kc = int(w.key_counts[bmax])
    g = w.q_heads // w.kv_heads
    qm = inp.queries[bmax].view(w.proposal_count, w.kv_heads, g, w.head_dim).permute(1, 0, 2, 3)
    qm = qm.reshape(w.kv_heads, w.proposal_count * g, w.head_dim).contiguous()
    kpad = min(((kc + 63) // 64) * 64, w.capacity)
    k_exact = layer.key_cache[bmax, :kc].permute(1, 2, 0)       # [Hkv, D, n]
    k_pad = layer.key_cache[bmax, :kpad].permute(1, 2, 0)
    t_qk_exact = _time(lambda: torch.matmul(qm, k_exact), reps, flush)
    t_qk_pad = _time(lambda: torch.matmul(qm, k_pad), reps, flush)
    t_fused = _time(fused, reps, flush)
    t_exact = _time(lambda: _three_pass(layer, inp, w, pad64=False), reps, flush)
    t_pad = _time(lambda: _three_pass(layer, inp, w, pad64=True), reps, flush)
    return {"workload": w.name, "batch": w.batch, "proposal_count": w.proposal_count,
            "key_counts": [int(x) for x in w.key_counts],
            "fused_tcgen05_us": round(t_fused, 1),
            "three_pass_exact_us": round(t_exact, 1),
            "three_pass_padded64_us": round(t_pad, 1),
            "qk_only_keys": [kc, kpad],
            "qk_only_exact_us": round(t_qk_exact, 1),
            "qk_only_padded64_us": round(t_qk_pad, 1),
            "max_abs_diff": agree}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--reps", type=int, default=50)
    args = ap.parse_args()
    for w in (synth.global_single(), synth.global_sweep(4), synth.global_sweep(15)):
        print(json.dumps(run(w, args.reps)), flush=True)


if __name__ == "__main__":
    main()
