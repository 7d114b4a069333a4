"""Seeded synthetic inputs shaped like the pages' workloads.

This module holds no attention or ring arithmetic: it only draws numbers and
describes shapes.  Both the CUDA path (through the tests and the benchmark) and
the fp64 oracle receive the arrays it produces, so neither side's inputs come
from the other.

Recipe (every value reproducible from the seed alone):
  * Values are fp32 draws from ``numpy.random.default_rng(...).standard_normal``
    rounded to bf16 with round-to-nearest-even, returned as uint16 bit patterns.
  * Each request's K/V history is drawn in blocks of ``BLOCK`` positions; block
    ``i`` of tensor ``name`` of request ``b`` in layer ``layer`` comes from the
    generator seeded with ``[seed, layer, b, TENSOR_ID[name], i]``.  A position
    therefore has the same value however much of the history a caller asks for.
  * Queries come from the generator seeded with ``[seed, layer, b, TENSOR_ID['q']]``.
  * Optional K pre-scaling (``k_prescale``) multiplies the fp32 draw before
    rounding; optional outlier rows (``outlier_fraction``, ``outlier_gain``)
    multiply a seeded fraction of K rows (per position and KV head) before
    rounding, to stress the softmax range.

The five workloads follow the shapes of the pages (Gemma-4 sliding layers:
8 KV heads x 256, window 1024; global layers: 2 KV heads x 512, 16 query heads;
4- and 15-position speculative verify).  ``key_count`` is the number of keys a
request holds after this step's tokens are appended; ``context_length`` is the
number held before (``key_count - proposal_count``).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

BLOCK = 64
TENSOR_ID = {"q": 1, "k": 2, "v": 3, "outlier": 4, "lengths": 5}


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round to nearest, ties to even) as uint16 bit patterns.

    Inputs are finite normal draws, so no NaN handling is needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_to_float(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    batch: int
    proposal_count: int
    q_heads: int
    kv_heads: int
    head_dim: int
    key_counts: np.ndarray          # int64 [batch], keys after this step's append
    scale: float
    window: int = 0                 # ring slots for sliding layers (0: global layer)
    capacity: int = 0               # cache rows per request for global layers
    k_prescale: float = 1.0
    outlier_fraction: float = 0.0
    outlier_gain: float = 1.0
    layers: int = 1
    description: str = ""

    @property
    def context_lengths(self) -> np.ndarray:
        return (self.key_counts - self.proposal_count).astype(np.int64)

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads


def _rng(*key) -> np.random.Generator:
    return np.random.default_rng([int(k) for k in key])


def queries(w: Workload, layer: int, b: int) -> np.ndarray:
    """uint16 [proposal_count][q_heads][head_dim]."""
    g = _rng(w.seed, layer, b, TENSOR_ID["q"])
    x = g.standard_normal((w.proposal_count, w.q_heads, w.head_dim), dtype=np.float32)
    return bf16_bits(x)


def history(w: Workload, layer: int, b: int, first: int, stop: int, which: str) -> np.ndarray:
    """uint16 [stop-first][kv_heads][head_dim]: rows for positions first..stop-1."""
    if not 0 <= first <= stop:
        raise ValueError("bad position range")
    rows = stop - first
    out = np.empty((rows, w.kv_heads, w.head_dim), dtype=np.uint16)
    blk0, blk1 = first // BLOCK, (stop + BLOCK - 1) // BLOCK
    for blk in range(blk0, blk1):
        g = _rng(w.seed, layer, b, TENSOR_ID[which], blk)
        x = g.standard_normal((BLOCK, w.kv_heads, w.head_dim), dtype=np.float32)
        if which == "k":
            if w.k_prescale != 1.0:
                x *= np.float32(w.k_prescale)
            if w.outlier_fraction > 0.0:
                go = _rng(w.seed, layer, b, TENSOR_ID["outlier"], blk)
                hit = go.random((BLOCK, w.kv_heads)) < w.outlier_fraction
                x[hit] *= np.float32(w.outlier_gain)
        lo = max(first, blk * BLOCK)
        hi = min(stop, (blk + 1) * BLOCK)
        out[lo - first:hi - first] = bf16_bits(x[lo - blk * BLOCK:hi - blk * BLOCK])
    return out


def last_rows(w: Workload, layer: int, b: int, rows: int):
    """The last `rows` positions of request b's history (fewer if it is shorter).

    Returns (first_position, k_hist, v_hist).
    """
    stop = int(w.key_counts[b])
    first = max(0, stop - rows)
    return first, history(w, layer, b, first, stop, "k"), history(w, layer, b, first, stop, "v")


# ---------------------------------------------------------------------------
# The five workloads.
# ---------------------------------------------------------------------------

def sliding_single(seed: int = 1001) -> Workload:
    """One request, key count 1500 (the ring has wrapped; next write slot 476),
    8 KV heads x 256, 16 query heads, 1 query at position 1499; K drawn N(0,1)
    then scaled by 1/sqrt(256) before rounding, softmax scale 1."""
    return Workload(name="swa_decode_b1_s1500", seed=seed, batch=1, proposal_count=1,
                    q_heads=16, kv_heads=8, head_dim=256,
                    key_counts=np.array([1500], dtype=np.int64), scale=1.0, window=1024,
                    k_prescale=1.0 / math.sqrt(256.0),
                    description="sliding-window decode, 1 request, 1500 keys, window 1024")


def sliding_batched(seed: int = 1002, batch: int = 56) -> Workload:
    """56 requests, key counts uniform in [1024, 4096], 1 new token each."""
    g = _rng(seed, 0, 0, TENSOR_ID["lengths"])
    kc = g.integers(1024, 4096, size=batch, endpoint=True).astype(np.int64)
    return Workload(name="swa_decode_b56", seed=seed, batch=batch, proposal_count=1,
                    q_heads=16, kv_heads=8, head_dim=256, key_counts=kc,
                    scale=1.0 / math.sqrt(256.0), window=1024,
                    description="sliding-window decode, 56 requests, keys U[1024,4096]")


def global_single(seed: int = 1003) -> Workload:
    """One request, 6001 cached + 4 proposal keys = 6005, cache capacity 8192."""
    return Workload(name="global_verify_b1_k4_s6005", seed=seed, batch=1, proposal_count=4,
                    q_heads=16, kv_heads=2, head_dim=512,
                    key_counts=np.array([6005], dtype=np.int64),
                    scale=1.0 / math.sqrt(512.0), capacity=8192,
                    description="global verify, 1 request, 4 proposals, 6005 keys")


def global_sweep(proposal_count: int = 4, seed: int | None = None) -> Workload:
    """8 requests: key counts {1024, 4093, 6005, 6016, 12289, 32768} and two
    uniform draws in [1, 32768] (raised to at least proposal_count); 1% of K rows
    scaled by 8 before rounding; capacity 32768."""
    if seed is None:
        seed = 1004 if proposal_count == 4 else 1005
    g = _rng(seed, 0, 0, TENSOR_ID["lengths"])
    extra = g.integers(1, 32768, size=2, endpoint=True)
    kc = np.array([1024, 4093, 6005, 6016, 12289, 32768, *extra], dtype=np.int64)
    kc = np.maximum(kc, proposal_count)
    return Workload(name=f"global_verify_b8_k{proposal_count}", seed=seed, batch=8,
                    proposal_count=proposal_count, q_heads=16, kv_heads=2, head_dim=512,
                    key_counts=kc, scale=1.0 / math.sqrt(512.0), capacity=32768,
                    outlier_fraction=0.01, outlier_gain=8.0,
                    description=f"global verify sweep, 8 requests, {proposal_count} proposals")


MIXED_SLIDING_LAYERS = 5


def mixed_step(seed: int = 1006, batch: int = 64):
    """Mixed decode step: 64 requests, 4 speculative positions, context lengths
    log-uniform in [512, 32768]; 5 sliding layers (own rings) + 1 global layer
    (cache capacity 32832).  Returns (sliding workload, global workload) that
    share the key counts."""
    g = _rng(seed, 0, 0, TENSOR_ID["lengths"])
    ctx = np.floor(np.exp(g.uniform(math.log(512.0), math.log(32768.0), size=batch)))
    ctx = np.clip(ctx, 512, 32768).astype(np.int64)
    k = 4
    kc = ctx + k
    sliding = Workload(name="mixed_step_sliding", seed=seed, batch=batch, proposal_count=k,
                       q_heads=16, kv_heads=8, head_dim=256, key_counts=kc,
                       scale=1.0 / math.sqrt(256.0), window=1024,
                       layers=MIXED_SLIDING_LAYERS,
                       description="mixed step, sliding layers")
    glob = Workload(name="mixed_step_global", seed=seed + 100, batch=batch, proposal_count=k,
                    q_heads=16, kv_heads=2, head_dim=512, key_counts=kc,
                    scale=1.0 / math.sqrt(512.0), capacity=32832, layers=1,
                    description="mixed step, global layer")
    return sliding, glob


def small(name: str, *, seed: int, batch: int, proposal_count: int, q_heads: int,
          kv_heads: int, head_dim: int, key_counts, window: int = 0, capacity: int = 0,
          scale: float | None = None, outlier_fraction: float = 0.0) -> Workload:
    """A custom small workload for parity tests."""
    return Workload(name=name, seed=seed, batch=batch, proposal_count=proposal_count,
                    q_heads=q_heads, kv_heads=kv_heads, head_dim=head_dim,
                    key_counts=np.asarray(key_counts, dtype=np.int64),
                    scale=(1.0 / math.sqrt(head_dim)) if scale is None else scale,
                    window=window, capacity=capacity, outlier_fraction=outlier_fraction,
                    outlier_gain=8.0 if outlier_fraction else 1.0)
