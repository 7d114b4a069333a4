"""GPU parity of the FP8 (e4m3) ring variant against the fp64 oracle.

"gemma-cuda-hybrid" ("Features" / "Server") stores the KV cache as FP8 e4m3;
its "Limitations" call that lossy, outside the bit-exact comparison.  Here:

  * the appended e4m3 bytes (rings and displaced rows) equal the oracle's
    quantiser bit for bit (integer work: exact);
  * the attention output equals the oracle's attention of the DEQUANTISED
    history (e4m3 value x scale) within the same tolerance as the bf16 path
    (gpu_harness): the kernel widens K and V to f16 exactly, converts each
    query row to f16 after a power-of-two scale (exact for every element
    within 2^-28 of the row's largest) and rounds P to f16, so its arithmetic
    error stays within the bf16 path's;
  * the FP8 output differs from the oracle's attention of the UNQUANTISED
    bf16 history by about what the oracle itself computes for the
    quantisation (the test's own tolerance: the oracle's quantisation effect
    plus the gate above).

Scales are the calibration a caller would use: max |x| / 448 over the data,
one per tensor.
"""
import concurrent.futures
import os

import numpy as np
import pytest
import torch

from gpu_harness import GATE_ABS, assert_close
from sliding_window_gqa_ring_gb300 import carat, engine, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    carat.library()
    carat.carat_get_device_status(clear=True)
    yield
    assert carat.carat_get_device_status(clear=True) == 0


def _amax_scale(w, kind):
    """Per-tensor scale max|x| / 448 over every row the workload uses."""
    m = 0.0
    for b in range(w.batch):
        first = max(0, int(w.key_counts[b]) - w.window - w.proposal_count)
        rows = synth.history(w, 0, b, first, int(w.key_counts[b]), kind)
        m = max(m, float(np.abs(synth.bf16_to_float(rows)).max()))
    return m / 448.0


def _run(orc, w, check_displaced=True):
    ks, vs = _amax_scale(w, "k"), _amax_scale(w, "v")
    layer = engine.Fp8SlidingLayer(w.batch, k_scale=ks, v_scale=vs, window=w.window,
                                   q_heads=w.q_heads, kv_heads=w.kv_heads, head_dim=w.head_dim,
                                   max_proposals=w.proposal_count, scale=w.scale)
    inp = engine.stage_sliding(w, 0, layer)
    out = layer.step(inp.queries, inp.k_new, inp.v_new, inp.context_lengths)
    torch.cuda.synchronize()
    out_h = out.cpu().numpy()
    k_ring = layer.k_ring.cpu().numpy()
    v_ring = layer.v_ring.cpu().numpy()
    disp = layer.displaced.cpu().numpy()
    worst_quant, worst_vs_bf16 = 0.0, 0.0

    def oracle_pair(b):
        # attention of the dequantised and of the unquantised history
        first, kh, vh = inp.host["hist"][b]
        ctx = int(w.context_lengths[b])
        kq, vq = orc.quantize_bf16(kh, ks), orc.quantize_bf16(vh, vs)
        q = inp.host["q"][b]
        ref = orc.attention_request_f64(q, orc.dequantize(kq, ks), orc.dequantize(vq, vs), first,
                                        ctx, w.window, w.scale)
        return kq, vq, ref, orc.attention_request(q, kh, vh, first, ctx, w.window, w.scale)

    with concurrent.futures.ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as pool:
        refs = list(pool.map(oracle_pair, range(w.batch)))
    for b in range(w.batch):
        first, kh, vh = inp.host["hist"][b]
        ctx, kc = int(w.context_lengths[b]), int(w.key_counts[b])
        kq, vq, ref, unq = refs[b]
        exp_k, valid = orc.ring_expected_bytes(kq, first, kc, w.window)
        exp_v, _ = orc.ring_expected_bytes(vq, first, kc, w.window)
        assert np.array_equal(k_ring[b][valid], exp_k[valid]), f"{w.name}: K ring bytes, request {b}"
        assert np.array_equal(v_ring[b][valid], exp_v[valid]), f"{w.name}: V ring bytes, request {b}"
        if check_displaced and w.proposal_count > 1:
            exp_d, dvalid = orc.displaced_expected_bytes(kq, vq, first, ctx, w.proposal_count,
                                                         w.window)
            assert np.array_equal(disp[b][:w.proposal_count - 1][dvalid], exp_d[dvalid]), \
                f"{w.name}: displaced bytes, request {b}"
        assert_close(out_h[b], ref, f"{w.name} (dequantised) request {b}")
        quant = float(np.abs(ref - unq).max())
        vs_bf16 = float(np.abs(out_h[b] - unq).max())
        assert vs_bf16 <= quant + GATE_ABS, (w.name, b, vs_bf16, quant)
        worst_quant = max(worst_quant, quant)
        worst_vs_bf16 = max(worst_vs_bf16, vs_bf16)
    return layer, inp, worst_quant, worst_vs_bf16


def test_fp8_sliding_single_request(orc):
    _run(orc, synth.sliding_single())


def test_fp8_sliding_batched(orc):
    _run(orc, synth.sliding_batched())


def test_fp8_mixed_step_sliding_layer(orc):
    w = synth.mixed_step()[0]
    # every request's attention against the oracle would take minutes on the
    # host: a contiguous subset of 12 of the 64 requests (96 units, fewer than
    # the 152 CTAs: the stream-K schedule) is compared; test_fp8_sliding_batched
    # and test_fp8_unit_queue_skips_rejected_requests cover the unit queue
    sub = synth.small("fp8_mixed_sub", seed=w.seed, batch=12, proposal_count=w.proposal_count,
                      q_heads=w.q_heads, kv_heads=w.kv_heads, head_dim=w.head_dim,
                      key_counts=w.key_counts[:12], window=w.window)
    _run(orc, sub)


def test_fp8_unit_queue_skips_rejected_requests(orc):
    """24 requests x 8 KV heads = 192 units over 152 persistent CTAs that take
    whole units from the work counter.  Requests rejected on the device (a
    negative context length, a ring id out of range) put no unit in the queue,
    get NaN outputs and set the status bits; every other request comes out bit
    for bit as in a call where all requests are valid, which matches the
    oracle."""
    kcs = [100 + 173 * i for i in range(24)]          # rings not full, full, wrapped
    w = synth.small("fp8_queue", seed=5400, batch=24, proposal_count=4, q_heads=16, kv_heads=8,
                    head_dim=256, key_counts=kcs, window=1024)
    layer, inp, _, _ = _run(orc, w)                   # every request against the oracle
    ref = layer.attend(inp.queries, inp.context_lengths).cpu().numpy()
    torch.cuda.synchronize()
    assert carat.carat_get_device_status(clear=True) == 0
    bad_ctx = inp.context_lengths.clone()
    bad_ctx[[3, 17]] = -5
    ids = torch.arange(24, dtype=torch.int32, device="cuda")
    ids[[0, 8, 23]] = 99                              # 24 rings: out of range
    out = layer.attend(inp.queries, bad_ctx, ring_ids=ids).cpu().numpy()
    status = carat.carat_get_device_status(clear=True)
    assert status & carat.CARAT_DEV_BAD_CONTEXT and status & carat.CARAT_DEV_BAD_CACHE_ID
    assert not status & carat.CARAT_DEV_TIMEOUT
    for b in range(24):
        if b in (0, 3, 8, 17, 23):
            assert np.isnan(out[b]).all(), b
        else:
            assert np.array_equal(out[b], ref[b]), b
    # the next call on the same workspace starts the counter afresh
    again = layer.attend(inp.queries, inp.context_lengths).cpu().numpy()
    assert np.array_equal(again, ref)
    assert carat.carat_get_device_status(clear=True) == 0


FP8_EDGES = {
    # (batch, k, key counts): empty-ish rings, ring not yet full, exactly full,
    # wrapped, 16 proposals (32-row tiles), a single proposal
    "decode_k1": (5, 1, [1, 100, 1023, 1024, 5000]),
    "verify_k4": (6, 4, [4, 130, 1027, 1028, 2049, 70000]),
    "verify_k16": (3, 16, [16, 1040, 3000]),
}


@pytest.mark.parametrize("case", sorted(FP8_EDGES))
def test_fp8_edges(orc, case):
    batch, k, kcs = FP8_EDGES[case]
    w = synth.small(f"fp8_{case}", seed=5300 + k, batch=batch, proposal_count=k, q_heads=16,
                    kv_heads=8, head_dim=256, key_counts=kcs, window=1024)
    _run(orc, w)


def test_fp8_rollback_restores_bytes(orc):
    """After a k=4 FP8 append, rolling back to accepted[b] rows leaves the
    rings as the oracle's rings for key count context + accepted."""
    w = synth.small("fp8_rollback", seed=5400, batch=4, proposal_count=4, q_heads=16,
                    kv_heads=8, head_dim=256, key_counts=[1030, 2050, 1500, 900], window=1024)
    layer, inp, _, _ = _run(orc, w)
    accepted = torch.tensor([0, 1, 3, 2], dtype=torch.int32, device="cuda")
    layer.rollback(inp.context_lengths, accepted, w.proposal_count)
    torch.cuda.synchronize()
    k_ring = layer.k_ring.cpu().numpy()
    for b in range(w.batch):
        first, kh, vh = inp.host["hist"][b]
        ctx = int(w.context_lengths[b])
        kept = ctx + int(accepted[b])
        kq = orc.quantize_bf16(kh, layer.k_scale)
        exp_k, valid = orc.ring_expected_bytes(kq, first, kept, w.window)
        # every slot the next query (position `kept`, window [kept - window + 1,
        # kept]) can see matches; other slots are never read again
        for slot in np.nonzero(valid)[0]:
            pos_newest = kept - 1 - ((kept - 1 - slot) % w.window)
            if pos_newest >= kept - w.window + 1:
                assert np.array_equal(k_ring[b][slot], exp_k[slot]), (b, slot)


def test_fp8_unsupported_head_dim_is_rejected():
    q = torch.zeros((1, 1, 4, 512), dtype=torch.bfloat16, device="cuda")
    ring = torch.zeros((1, 1024, 2, 512), dtype=torch.uint8, device="cuda")
    ctx = torch.full((1,), 10, dtype=torch.int32, device="cuda")
    out = torch.empty((1, 1, 4, 512), dtype=torch.float32, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(carat.CaratError) as e:
        carat.carat_swa_attention_fp8(out, q, ring, ring, ctx, scale=0.04, k_scale=0.01,
                                      v_scale=0.01, workspace=ws)
    assert e.value.status == carat.CARAT_ERR_UNSUPPORTED
