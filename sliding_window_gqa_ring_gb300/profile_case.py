"""Run a few attention calls of one staged layer, for profiler captures.

    python -m sliding_window_gqa_ring_gb300.profile_case --case swa_mixed --calls 3

The layer is staged from the seeded workloads in ``synth`` (rings or caches
written with carat_ring_append), then the step's fused append+attention call
repeats ``--calls`` times (with ``--separate``: one carat_ring_append, then the
attention call alone repeats), so a profiler filtered on the attention kernel
sees exactly ``--calls`` launches.  Every case but global_mixed keeps a few
GB or less on the device; every case reads more than the 129 MB L2 per call.
"""
from __future__ import annotations

import argparse

import torch

from . import carat, engine, synth

CASES = {
    "swa_b1": lambda: synth.sliding_single(),
    "swa_b56": lambda: synth.sliding_batched(),
    "swa_mixed": lambda: synth.mixed_step()[0],
    "global_single": lambda: synth.global_single(),
    "global_sweep4": lambda: synth.global_sweep(4),
    "global_sweep15": lambda: synth.global_sweep(15),
    # the mixed step's global layer: about 9 GB of caches, for one-pass captures only
    "global_mixed": lambda: synth.mixed_step()[1],
    # the mixed step's sliding layer with FP8 e4m3 rings (append once, then the
    # attention call repeats)
    "swa_mixed_fp8": lambda: synth.mixed_step()[0],
}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--case", choices=sorted(CASES), required=True)
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--separate", action="store_true",
                    help="time carat_ring_append + the attention call instead of the fused call")
    args = ap.parse_args()
    w = CASES[args.case]()
    if args.case.endswith("_fp8"):
        # scales as a caller would calibrate them: max |x| / 448 over the layer
        probe = engine.SlidingLayer(w.batch, window=w.window, q_heads=w.q_heads,
                                    kv_heads=w.kv_heads, head_dim=w.head_dim,
                                    max_proposals=w.proposal_count, scale=w.scale)
        hist = engine.stage_sliding(w, 0, probe).host["hist"]
        kmax = max(float(abs(synth.bf16_to_float(h[1])).max()) for h in hist.values())
        vmax = max(float(abs(synth.bf16_to_float(h[2])).max()) for h in hist.values())
        del probe
        layer = engine.Fp8SlidingLayer(w.batch, k_scale=kmax / 448.0, v_scale=vmax / 448.0,
                                       window=w.window, q_heads=w.q_heads, kv_heads=w.kv_heads,
                                       head_dim=w.head_dim, max_proposals=w.proposal_count,
                                       scale=w.scale)
        inp = engine.stage_sliding(w, 0, layer)
        out = torch.empty(inp.queries.shape, dtype=torch.float32, device=layer.device)
        layer.append(inp.k_new, inp.v_new, inp.context_lengths)
        for _ in range(args.calls):
            layer.attend(inp.queries, inp.context_lengths, out=out)
        torch.cuda.synchronize()
        status = carat.carat_get_device_status(clear=True)
        print(f"{args.case}: {args.calls} calls, device status {status:#x}")
        if status:
            raise SystemExit(1)
        return
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
    if args.separate:
        layer.append(inp.k_new, inp.v_new, inp.context_lengths)
        for _ in range(args.calls):
            layer.attend(inp.queries, inp.context_lengths, out=out)
    else:
        for _ in range(args.calls):
            layer.step(inp.queries, inp.k_new, inp.v_new, inp.context_lengths, out=out)
    torch.cuda.synchronize()
    status = carat.carat_get_device_status(clear=True)
    print(f"{args.case}: {args.calls} calls, device status {status:#x}")
    if status:
        raise SystemExit(1)


if __name__ == "__main__":
    main()
