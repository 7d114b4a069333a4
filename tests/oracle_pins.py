"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises ``AssertionError``
if the oracle disagrees with

  * a library routine that computes the same definition
    (``torch.nn.functional.scaled_dot_product_attention`` in float64 on CPU),
  * a closed form (one key, uniform weights, two keys, a saturated softmax),
  * an invariant the pages state (a common reordering of K and V inside the
    window, zero-filled masked tails, causality, window >= context being global
    attention, grouped heads = repeated KV heads, ring = rotated linear window),
  * or a value the pages print (``tests/golden/pages_worked_values.json``).

The same functions run against deliberately broken builds of the oracle in
``test_oracle_mutations.py``, to show that a plausible mistake in the oracle
fails at least one of them.  This module has no ``test_`` prefix so pytest does
not collect it by itself.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

from sliding_window_gqa_ring_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_worked_values.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _rand_bf16(rng, shape, scale=1.0):
    return synth.bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(scale))


def _val(bits):
    return synth.bf16_to_float(bits).astype(np.float64)


def _const_bits(values):
    """Exactly representable small values -> bf16 bits."""
    return synth.bf16_bits(np.asarray(values, dtype=np.float32))


def _sdpa_reference(q, k_hist, v_hist, hist_base, context_length, window, scale):
    """Library route: float64 scaled_dot_product_attention with an explicit mask.

    q: [k][Hq][D]; history [L][Hkv][D].  The boolean mask marks, for query j at
    position context_length + j, the history rows inside its window.
    """
    kq, hq, d = q.shape
    length, hkv, _ = k_hist.shape
    qt = torch.from_numpy(_val(q)).permute(1, 0, 2).unsqueeze(0)          # [1,Hq,k,D]
    kt = torch.from_numpy(_val(k_hist)).permute(1, 0, 2).unsqueeze(0)     # [1,Hkv,L,D]
    vt = torch.from_numpy(_val(v_hist)).permute(1, 0, 2).unsqueeze(0)
    pos = hist_base + torch.arange(length)
    mask = torch.zeros(kq, length, dtype=torch.bool)
    for j in range(kq):
        p = context_length + j
        lo = 0 if window <= 0 else max(0, p - window + 1)
        mask[j] = (pos >= lo) & (pos <= p)
    try:
        out = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, attn_mask=mask, scale=scale, enable_gqa=True)
    except TypeError:  # older torch without enable_gqa
        g = hq // hkv
        out = torch.nn.functional.scaled_dot_product_attention(
            qt, kt.repeat_interleave(g, dim=1), vt.repeat_interleave(g, dim=1),
            attn_mask=mask, scale=scale)
    return out.squeeze(0).permute(1, 0, 2).numpy()


def pin_sdpa_sliding(orc):
    """Sliding window (small ring): oracle == float64 SDPA with a window mask."""
    rng = np.random.default_rng(11)
    for (window, key_count, k, hq, hkv, d) in [(8, 29, 3, 4, 2, 16), (8, 5, 2, 4, 2, 8),
                                               (16, 40, 4, 8, 2, 32), (6, 6, 1, 2, 1, 8)]:
        ctx = key_count - k
        q = _rand_bf16(rng, (k, hq, d))
        kh = _rand_bf16(rng, (key_count, hkv, d))
        vh = _rand_bf16(rng, (key_count, hkv, d))
        scale = 1.0 / math.sqrt(d)
        got = orc.attention_request(q, kh, vh, 0, ctx, window, scale)
        ref = _sdpa_reference(q, kh, vh, 0, ctx, window, scale)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def pin_sdpa_global(orc):
    """Global causal verify: oracle == float64 SDPA with a causal mask, incl. GQA."""
    rng = np.random.default_rng(12)
    for (key_count, k, hq, hkv, d) in [(37, 4, 16, 2, 16), (15, 15, 8, 2, 8), (70, 4, 8, 2, 64)]:
        ctx = key_count - k
        q = _rand_bf16(rng, (k, hq, d))
        kh = _rand_bf16(rng, (key_count, hkv, d), scale=3.0)
        vh = _rand_bf16(rng, (key_count, hkv, d))
        scale = 1.0 / math.sqrt(d)
        got = orc.attention_request(q, kh, vh, 0, ctx, 0, scale)
        ref = _sdpa_reference(q, kh, vh, 0, ctx, 0, scale)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def pin_single_key(orc):
    """Closed form: with one visible key the output is exactly that key's V row."""
    rng = np.random.default_rng(13)
    q = _rand_bf16(rng, (1, 2, 8))
    kh = _rand_bf16(rng, (1, 1, 8))
    vh = _rand_bf16(rng, (1, 1, 8))
    got = orc.attention_request(q, kh, vh, 0, 0, 1024, 0.7)
    for h in range(2):
        assert np.array_equal(got[0, h], _val(vh[0, 0])), "single key must return V_0"


def pin_uniform_window_golden(orc):
    """Closed form + printed value: with scale 0 every visible key has the same
    weight, so the output is the mean of V over the window.  V columns mark
    positions, which pins the window to exactly [476, 1499] for a query at 1499
    with a 1024-slot window."""
    gold = _golden()["sliding_window_positions"]
    p, window = gold["query_position"], gold["window"]
    first, last = gold["first_position"], gold["last_position"]
    n = p + 1
    v = np.zeros((n, 1, 8), dtype=np.float32)
    v[:first, 0, 0] = 1.0                 # everything before the window
    v[first, 0, 1] = 1.0                  # first position inside
    v[last, 0, 2] = 1.0                   # the query's own position
    v[:, 0, 3] = 1.0                      # normaliser
    v[first:last + 1, 0, 4] = 1.0         # the whole window
    if first > 0:
        v[first - 1, 0, 5] = 1.0          # just outside
    vh = _const_bits(v)
    kh = _const_bits(np.ones((n, 1, 8), dtype=np.float32))
    q = _const_bits(np.ones((1, 1, 8), dtype=np.float32))
    got = orc.attention_request(q, kh, vh, 0, p, window, 0.0)[0, 0]
    count = last - first + 1
    assert count == window
    expect = np.array([0.0, 1.0 / count, 1.0 / count, 1.0, 1.0, 0.0, 0.0, 0.0])
    np.testing.assert_allclose(got, expect, rtol=0, atol=1e-15)
    assert orc.window_first(p, window) == first


def pin_two_keys(orc):
    """Closed form: two keys with scores s0, s1 give
    sigmoid(s0 - s1) * V0 + sigmoid(s1 - s0) * V1."""
    q = _const_bits(np.array([[[2.0, 0, 0, 0]]], dtype=np.float32))
    kh = _const_bits(np.array([[[1.5, 0, 0, 0]], [[-0.5, 0, 0, 0]]], dtype=np.float32))
    vh = _const_bits(np.array([[[1.0, 2.0, -3.0, 0.25]], [[-1.0, 4.0, 5.0, 0.5]]],
                              dtype=np.float32))
    scale = 0.75
    s0, s1 = scale * 2.0 * 1.5, scale * 2.0 * -0.5
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    expect = w0 * _val(vh[0, 0]) + w1 * _val(vh[1, 0])
    got = orc.attention_request(q, kh, vh, 0, 1, 0, scale)[0, 0]
    np.testing.assert_allclose(got, expect, rtol=1e-14, atol=0)


def pin_saturated(orc):
    """Closed form: a score 1000 above all others takes all the weight, even
    with large scores (no overflow)."""
    q = _const_bits(np.array([[[32.0, 0, 0, 0]]], dtype=np.float32))
    kh = _const_bits(np.array([[[0.0, 0, 0, 0]], [[40.0, 0, 0, 0]], [[8.0, 0, 0, 0]]],
                              dtype=np.float32))
    vh = _const_bits(np.array([[[1, 1, 1, 1]], [[3, -2, 0.5, 7]], [[9, 9, 9, 9]]],
                              dtype=np.float32))
    got = orc.attention_request(q, kh, vh, 0, 2, 0, 1.0)[0, 0]   # scores 0, 1280, 256
    assert np.array_equal(got, _val(vh[1, 0])), got


def pin_permutation_invariance(orc):
    """Invariant (Gaudi page, 'Our approach'): attention does not change under a
    common reordering of K and V.  Reordering the rows inside one query's window
    leaves its output unchanged; this is why a rotated ring can be read in
    place."""
    rng = np.random.default_rng(14)
    window, n, d = 16, 40, 32
    q = _rand_bf16(rng, (1, 4, d))
    kh = _rand_bf16(rng, (n, 2, d))
    vh = _rand_bf16(rng, (n, 2, d))
    p = n - 1
    lo = p - window + 1
    base = orc.attention_request(q, kh, vh, 0, p, window, 0.3)
    for shift in (1, 5, 15):
        perm = np.arange(n)
        perm[lo:] = lo + np.roll(np.arange(window), shift)   # a cyclic shift, like a ring
        got = orc.attention_request(q, kh[perm], vh[perm], 0, p, window, 0.3)
        np.testing.assert_allclose(got, base, rtol=1e-13, atol=1e-15)
    perm = np.arange(n)
    perm[lo:] = lo + rng.permutation(window)
    got = orc.attention_request(q, kh[perm], vh[perm], 0, p, window, 0.3)
    np.testing.assert_allclose(got, base, rtol=1e-13, atol=1e-15)
    # Negative control: moving a row across the window edge does change it.
    perm = np.arange(n)
    perm[lo - 1], perm[lo] = perm[lo], perm[lo - 1]
    got = orc.attention_request(q, kh[perm], vh[perm], 0, p, window, 0.3)
    assert not np.allclose(got, base, rtol=1e-9, atol=0)


def pin_padded_tail(orc):
    """Invariant + printed value (Carat, 'More FLOPs can be faster'): 6005 keys
    padded with zero rows to 6016 (11 masked columns) give the same output;
    unmasking the zero rows would change it."""
    gold = _golden()["padded_tail"]
    kc, padded = gold["key_count"], gold["padded_key_count"]
    assert padded - kc == gold["masked_columns"]
    assert padded % gold["multiple"] == 0 and padded - gold["multiple"] < kc
    rng = np.random.default_rng(15)
    d, k = 8, 4
    q = _rand_bf16(rng, (k, 8, d))
    kh = _rand_bf16(rng, (kc, 1, d))
    vh = _rand_bf16(rng, (kc, 1, d))
    kp = np.concatenate([kh, np.zeros((padded - kc, 1, d), np.uint16)])
    vp = np.concatenate([vh, np.zeros((padded - kc, 1, d), np.uint16)])
    ctx = orc.key_count(kc, -k)         # = kc - k via the key-count rule
    assert ctx == kc - k
    a = orc.attention_request(q, kh, vh, 0, ctx, 0, 0.5)
    b = orc.attention_request(q, kp, vp, 0, ctx, 0, 0.5)
    assert np.array_equal(a, b)
    # Negative control: treating the zero tail as visible keys changes the rows.
    c = orc.attention_request(q, kp, vp, 0, padded - k, 0, 0.5)
    assert not np.allclose(c[-1], a[-1], rtol=1e-6, atol=0)


def pin_causal(orc):
    """Invariant (Carat: a query looks at no key later than its own position):
    changing K/V after position p leaves query p's row unchanged, and changing
    a key it does see changes it."""
    rng = np.random.default_rng(16)
    k, n, d = 4, 25, 16
    ctx = n - k
    q = _rand_bf16(rng, (k, 8, d))
    kh = _rand_bf16(rng, (n, 2, d))
    vh = _rand_bf16(rng, (n, 2, d))
    base = orc.attention_request(q, kh, vh, 0, ctx, 0, 0.25)
    for j in range(k - 1):
        p = ctx + j
        k2, v2 = kh.copy(), vh.copy()
        k2[p + 1:] = _rand_bf16(rng, k2[p + 1:].shape)
        v2[p + 1:] = _rand_bf16(rng, v2[p + 1:].shape)
        got = orc.attention_request(q, k2, v2, 0, ctx, 0, 0.25)
        assert np.array_equal(got[:j + 1], base[:j + 1])
        assert not np.allclose(got[j + 1:], base[j + 1:])
        v3 = vh.copy()
        v3[p] = _rand_bf16(rng, v3[p].shape)
        got = orc.attention_request(q, kh, v3, 0, ctx, 0, 0.25)
        assert not np.allclose(got[j], base[j])


def pin_window_covers_context(orc):
    """Invariant: a sliding window at least as long as the context is global
    attention (same output, bit for bit)."""
    rng = np.random.default_rng(17)
    for (n, k) in [(30, 1), (30, 4), (1024, 4)]:
        q = _rand_bf16(rng, (k, 4, 16))
        kh = _rand_bf16(rng, (n, 2, 16))
        vh = _rand_bf16(rng, (n, 2, 16))
        g = orc.attention_request(q, kh, vh, 0, n - k, 0, 0.25)
        s = orc.attention_request(q, kh, vh, 0, n - k, 1024, 0.25)
        assert np.array_equal(g, s)
    # and a window shorter than the context is not
    q = _rand_bf16(rng, (1, 4, 16))
    kh = _rand_bf16(rng, (40, 2, 16))
    vh = _rand_bf16(rng, (40, 2, 16))
    g = orc.attention_request(q, kh, vh, 0, 39, 0, 0.25)
    s = orc.attention_request(q, kh, vh, 0, 39, 8, 0.25)
    assert not np.allclose(g, s)


def pin_gqa_repeat(orc):
    """Invariant: grouped heads equal ungrouped attention on KV heads repeated
    for each query head of their group (contiguous groups: head h -> h // g)."""
    rng = np.random.default_rng(18)
    hq, hkv, d, n, k = 16, 2, 16, 33, 4
    q = _rand_bf16(rng, (k, hq, d))
    kh = _rand_bf16(rng, (n, hkv, d))
    vh = _rand_bf16(rng, (n, hkv, d))
    grouped = orc.attention_request(q, kh, vh, 0, n - k, 0, 0.25)
    rep_k = np.repeat(kh, hq // hkv, axis=1)
    rep_v = np.repeat(vh, hq // hkv, axis=1)
    flat = orc.attention_request(q, rep_k, rep_v, 0, n - k, 0, 0.25)
    assert np.array_equal(grouped, flat)
    # and the same for a sliding window
    grouped = orc.attention_request(q, kh, vh, 0, n - k, 8, 0.25)
    flat = orc.attention_request(q, rep_k, rep_v, 0, n - k, 8, 0.25)
    assert np.array_equal(grouped, flat)


def pin_row_matches_request(orc):
    """The single-row entry point gives the same row as the whole-request one."""
    rng = np.random.default_rng(19)
    hq, hkv, d, n, k = 8, 2, 16, 50, 3
    q = _rand_bf16(rng, (k, hq, d))
    kh = _rand_bf16(rng, (n, hkv, d))
    vh = _rand_bf16(rng, (n, hkv, d))
    for window in (0, 8):
        full = orc.attention_request(q, kh[10:], vh[10:], 10, n - k, 8 if window else 0, 0.3) \
            if window else orc.attention_request(q, kh, vh, 0, n - k, 0, 0.3)
        for j in range(k):
            for h in range(hq):
                if window:
                    row = orc.attention_row(q[j, h], kh[10:], vh[10:], 10, h // (hq // hkv),
                                            n - k + j, 8, 0.3)
                else:
                    row = orc.attention_row(q[j, h], kh, vh, 0, h // (hq // hkv),
                                            n - k + j, 0, 0.3)
                assert np.array_equal(row, full[j, h])


def pin_ring_golden(orc):
    """Printed values: slot = position mod window (1500 -> 476 for 1024 slots)
    and key_count = context_length + proposal_count (6001 + 4 = 6005)."""
    gold = _golden()
    for e in gold["ring_slot"]:
        assert orc.ring_slot(e["position"], e["window"]) == e["slot"], e
    for e in gold["key_count"]:
        assert orc.key_count(e["context_length"], e["proposal_count"]) == e["key_count"], e


def pin_ring_is_rotated_window(orc):
    """Invariant (Gaudi page, 'Our approach'): the ring is the linear window
    rotated by the head, so rolling it by the head slot recovers the last
    `window` rows of the linear history in order; a ring that has not wrapped
    holds the whole history from slot 0."""
    rng = np.random.default_rng(20)
    window = 8
    for n in (3, 8, 13, 21, 64):
        hist = _rand_bf16(rng, (n, 2, 4))
        ring, valid = orc.ring_expected(hist, 0, n, window)
        if n < window:
            assert valid[:n].all() and not valid[n:].any()
            assert np.array_equal(ring[:n], hist)
        else:
            assert valid.all()
            head = n % window
            assert np.array_equal(np.roll(ring, -head, axis=0), hist[n - window:])


def pin_displaced_covers_windows(orc):
    """After k tokens are appended, every position a query of the step needs is
    either still in the ring or among the displaced rows, and the displaced rows
    are exactly the ones the ring lost."""
    rng = np.random.default_rng(21)
    window = 8
    for (ctx, k) in [(20, 4), (9, 4), (7, 4), (30, 8), (5, 2), (40, 1)]:
        n = ctx + k
        kh = _rand_bf16(rng, (n, 1, 4))
        vh = _rand_bf16(rng, (n, 1, 4))
        ring_k, valid = orc.ring_expected(kh, 0, n, window)
        ring_v, _ = orc.ring_expected(vh, 0, n, window)
        disp, dvalid = orc.displaced_expected(kh, vh, 0, ctx, k, window)
        assert disp.shape[0] == k - 1
        for j in range(k):
            p = ctx + j
            for t in range(max(0, p - window + 1), p + 1):
                in_ring = (valid[t % window] and np.array_equal(ring_k[t % window], kh[t])
                           and t >= n - window)
                hits = [i for i in range(k - 1) if dvalid[i]
                        and np.array_equal(disp[i, 0], kh[t]) and np.array_equal(disp[i, 1], vh[t])]
                assert in_ring or hits, (ctx, k, j, t)
                if in_ring:
                    assert np.array_equal(ring_v[t % window], vh[t])
        lost = [t for t in range(max(0, ctx - window + 1), ctx) if t < n - window]
        assert sum(dvalid) == len(lost)


# ---------------------------------------------------------------------------
# FP8 (e4m3) KV cache ("gemma-cuda-hybrid", "Features" / "Server": the KV
# cache is stored as FP8 e4m3; "Limitations": it is lossy)
# ---------------------------------------------------------------------------

def _torch_e4m3_value(codes):
    """Library route: PyTorch's float8_e4m3fn reinterpretation of the bytes."""
    t = torch.from_numpy(np.asarray(codes, dtype=np.uint8).copy())
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _torch_e4m3_code(values_f32):
    """Library route: PyTorch's float32 -> float8_e4m3fn conversion (round to
    nearest even; used only for values inside the finite range)."""
    t = torch.from_numpy(np.asarray(values_f32, dtype=np.float32).copy())
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def pin_e4m3_format_values(orc):
    """Values the e4m3 format fixes: 1.0 = 0x38, the largest finite 448 =
    0x7e, the smallest normal 2^-6 = 0x08, the smallest subnormal 2^-9 = 0x01,
    the largest subnormal 7 * 2^-9 = 0x07, NaN = 0x7f, sign in bit 7; and the
    decoded value of every code agrees with PyTorch's float8_e4m3fn."""
    known = {0x00: 0.0, 0x38: 1.0, 0xB8: -1.0, 0x7E: 448.0, 0xFE: -448.0, 0x08: 2.0 ** -6,
             0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x40: 2.0, 0x3C: 1.5, 0x77: 240.0}
    for c, v in known.items():
        assert orc.e4m3_decode([c])[0] == v, (hex(c), v)
    assert np.isnan(orc.e4m3_decode([0x7F, 0xFF])).all()
    codes = np.arange(256, dtype=np.uint8)
    mine = orc.e4m3_decode(codes)
    lib = _torch_e4m3_value(codes)
    both_nan = np.isnan(mine) & np.isnan(lib)
    assert np.array_equal(mine[~both_nan], lib[~both_nan])
    assert both_nan.sum() == 2


def pin_e4m3_rounding(orc):
    """Encoding rounds to the nearest value with ties to the even code (as
    PyTorch's conversion does inside the finite range), saturates beyond 448,
    and every finite code round-trips."""
    assert list(orc.e4m3_encode([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, -1.0625])) == \
        [0x38, 0x3A, 0x00, 0x02, 0xB8]
    assert list(orc.e4m3_encode([449.0, 464.0, 1e9, -500.0, 447.0])) == [0x7E, 0x7E, 0x7E, 0xFE,
                                                                        0x7E]
    rng = np.random.default_rng(30)
    x = np.concatenate([rng.standard_normal(3000) * 8, rng.standard_normal(1000) * 0.01,
                        rng.uniform(-448, 448, 1000)]).astype(np.float32)
    assert np.array_equal(orc.e4m3_encode(x.astype(np.float64)), _torch_e4m3_code(x))
    codes = np.arange(256, dtype=np.uint8)
    vals = orc.e4m3_decode(codes)
    fin = ~np.isnan(vals)
    assert np.array_equal(orc.e4m3_encode(vals[fin]), codes[fin])


def pin_quantize_bf16(orc):
    """FP8 cache codes: with scale 1 (or a power of two, where the product is
    exact) they are the e4m3 codes of the scaled values; with any scale they
    equal PyTorch's float32 product by float32(1/scale) converted to
    float8_e4m3fn (inside the finite range)."""
    rng = np.random.default_rng(31)
    bits = _rand_bf16(rng, (4000,), scale=3.0)
    vals = _val(bits)
    assert np.array_equal(orc.quantize_bf16(bits, 1.0), orc.e4m3_encode(vals))
    assert np.array_equal(orc.quantize_bf16(bits, 0.25), orc.e4m3_encode(vals * 4.0))
    for scale in (0.0123, 0.37, 1.7):
        inv = np.float32(1.0) / np.float32(scale)
        prod = (synth.bf16_to_float(bits).astype(np.float32) * inv).astype(np.float32)
        inside = np.abs(prod) < 448
        mine = orc.quantize_bf16(bits, scale)
        assert np.array_equal(mine[inside], _torch_e4m3_code(prod[inside]))
        assert (mine[~inside] & 0x7F == 0x7E).all()


def pin_attention_f64(orc):
    """The float64-history attention equals the bf16 one on bf16-exact values
    and PyTorch's float64 scaled_dot_product_attention on dequantised FP8
    values."""
    rng = np.random.default_rng(32)
    q = _rand_bf16(rng, (3, 4, 8))
    kh = _rand_bf16(rng, (20, 2, 8))
    vh = _rand_bf16(rng, (20, 2, 8))
    a = orc.attention_request(q, kh, vh, 0, 17, 8, 0.35)
    b = orc.attention_request_f64(q, _val(kh), _val(vh), 0, 17, 8, 0.35)
    assert np.array_equal(a, b)
    kd = orc.dequantize(orc.quantize_bf16(kh, 0.05), 0.05)
    vd = orc.dequantize(orc.quantize_bf16(vh, 0.02), 0.02)
    got = orc.attention_request_f64(q, kd, vd, 0, 17, 8, 0.35)
    kq, hq, d = q.shape
    qt = torch.from_numpy(_val(q)).permute(1, 0, 2).unsqueeze(0)
    kt = torch.from_numpy(kd).permute(1, 0, 2).unsqueeze(0).repeat_interleave(2, dim=1)
    vt = torch.from_numpy(vd).permute(1, 0, 2).unsqueeze(0).repeat_interleave(2, dim=1)
    mask = torch.zeros(kq, 20, dtype=torch.bool)
    for j in range(kq):
        p = 17 + j
        mask[j, max(0, p - 7):p + 1] = True
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=0.35)
    ref = ref.squeeze(0).permute(1, 0, 2).numpy()
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def pin_ring_bytes_match_rows(orc):
    """The byte-row ring and displaced rows place whole rows exactly as the
    bf16 versions do (checked on the same data viewed as bytes)."""
    rng = np.random.default_rng(33)
    window = 8
    for (ctx, k) in [(20, 4), (5, 3), (13, 1)]:
        n = ctx + k
        kh = _rand_bf16(rng, (n, 2, 4))
        vh = _rand_bf16(rng, (n, 2, 4))
        ring16, valid16 = orc.ring_expected(kh, 0, n, window)
        ring8, valid8 = orc.ring_expected_bytes(kh.view(np.uint8), 0, n, window)
        assert np.array_equal(valid16, valid8)
        assert np.array_equal(ring16.view(np.uint8)[valid16], ring8[valid8])
        d16, dv16 = orc.displaced_expected(kh, vh, 0, ctx, k, window)
        d8, dv8 = orc.displaced_expected_bytes(kh.view(np.uint8), vh.view(np.uint8), 0, ctx, k,
                                               window)
        assert np.array_equal(dv16, dv8)
        assert np.array_equal(d16.view(np.uint8)[dv16], d8[dv8])


ALL_PINS = [
    pin_sdpa_sliding, pin_sdpa_global, pin_single_key, pin_uniform_window_golden,
    pin_two_keys, pin_saturated, pin_permutation_invariance, pin_padded_tail, pin_causal,
    pin_window_covers_context, pin_gqa_repeat, pin_row_matches_request, pin_ring_golden,
    pin_ring_is_rotated_window, pin_displaced_covers_windows, pin_e4m3_format_values,
    pin_e4m3_rounding, pin_quantize_bf16, pin_attention_f64, pin_ring_bytes_match_rows,
]
