"""The benchmark's algorithmic byte counts, against a direct count.

bench.py divides algorithmic bytes by time.  Here those counts are rebuilt
from the definition, position by position: query j of a request (position
context_length + j) sees the positions of its window (sliding: the last
`window` positions up to its own) or every position up to its own (global);
the call must read each visible K and V row once (Hkv x D bf16 each), its
queries once (bf16) and write its outputs once (fp32); a fused append also
writes the step's k new K and V rows.
"""
import random

import numpy as np
import pytest

import bench
from sliding_window_gqa_ring_gb300 import synth


def direct(w, fused):
    row = w.kv_heads * w.head_dim * 2
    total = 0
    for b in range(w.batch):
        kc = int(w.key_counts[b])
        ctx = kc - w.proposal_count
        seen = set()
        for j in range(w.proposal_count):
            pos = ctx + j
            lo = max(0, pos - w.window + 1) if w.window else 0
            seen.update(range(lo, pos + 1))
        total += len(seen) * row * 2
        total += w.proposal_count * w.q_heads * w.head_dim * (2 + 4)
        if fused:
            total += w.proposal_count * row * 2
    return total


def random_workload(rng, sliding):
    k = rng.choice([1, 2, 4, 15, 16])
    batch = rng.randint(1, 6)
    window = rng.choice([256, 1024]) if sliding else 0
    kcs = [rng.randint(k, 5000) for _ in range(batch)]
    return synth.small("bytes", seed=1, batch=batch, proposal_count=k, q_heads=16,
                       kv_heads=rng.choice([2, 8]), head_dim=rng.choice([256, 512]),
                       key_counts=kcs, window=window, capacity=0 if sliding else 8192)


@pytest.mark.parametrize("seed", range(40))
def test_call_bytes_match_a_direct_count(seed):
    rng = random.Random(seed)
    for sliding in (True, False):
        w = random_workload(rng, sliding)
        fn = bench.sliding_call_bytes if sliding else bench.global_call_bytes
        attn = sum(fn(w, b)[0] for b in range(w.batch))
        fused_writes = sum(fn(w, b)[1] for b in range(w.batch))
        assert attn == direct(w, False)
        assert attn + fused_writes == direct(w, True)
        assert bench.config_attention_bytes(w) == direct(w, False)


def test_mixed_step_bytes():
    sliding, glob = synth.mixed_step()
    nb = bench.step_bytes(sliding, glob)
    assert nb["swa_call"] == direct(sliding, True) == 524918784
    assert nb["global_call"] == direct(glob, True)
    assert nb["step"] == sliding.layers * nb["swa_call"] + nb["global_call"]


def test_workload_configs_bytes():
    # the single-layer workloads the bench's configs block times
    for w in (synth.sliding_single(), synth.sliding_batched(), synth.global_single(),
              synth.global_sweep(4), synth.global_sweep(15)):
        assert bench.config_attention_bytes(w) == direct(w, False)
    assert np.isclose(bench.config_attention_bytes(synth.sliding_single()) / 1e6, 8.41, atol=0.01)
