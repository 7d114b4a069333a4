"""Repeated calls: the same inputs give the same outputs, bit for bit, call
after call, with the device status word clear.  Covers the schedules whose
state lives across a launch or between launches of one workspace: the FP8
unit queue's work counter (cleared by each launch's last CTA), bf16 unit mode
with the row sums kept per lane, and the stream-K global verify with its
merge launch."""
import numpy as np
import pytest
import torch

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


def _repeat(call, ref, n):
    out = torch.empty_like(ref)
    for i in range(n):
        call(out)
        if i % 25 == 24:
            torch.cuda.synchronize()
            assert torch.equal(out, ref), f"call {i} differs from the first"
    torch.cuda.synchronize()
    assert carat.carat_get_device_status(clear=True) == 0


def test_fp8_unit_queue_repeats():
    # 24 requests x 8 KV heads = 192 units over 152 persistent CTAs
    w = synth.small("rep_fp8", seed=5600, batch=24, proposal_count=4, q_heads=16, kv_heads=8,
                    head_dim=256, key_counts=[200 + 150 * i for i in range(24)], window=1024)
    layer = engine.Fp8SlidingLayer(24, k_scale=0.0126, v_scale=0.013, window=1024,
                                   max_proposals=4, scale=w.scale)
    inp = engine.stage_sliding(w, 0, layer)
    layer.append(inp.k_new, inp.v_new, inp.context_lengths)
    ref = layer.attend(inp.queries, inp.context_lengths).clone()
    _repeat(lambda o: layer.attend(inp.queries, inp.context_lengths, out=o), ref, 500)


def test_bf16_unit_mode_repeats():
    # 40 requests x 8 KV heads = 320 units over 304 CTA slots, fused calls
    w = synth.small("rep_bf16", seed=5700, batch=40, proposal_count=4, q_heads=16, kv_heads=8,
                    head_dim=256, key_counts=[300 + 97 * i for i in range(40)], window=1024)
    layer = engine.SlidingLayer(40, window=1024, max_proposals=4, scale=w.scale)
    inp = engine.stage_sliding(w, 0, layer)
    layer.append(inp.k_new, inp.v_new, inp.context_lengths)
    ref = layer.attend(inp.queries, inp.context_lengths).clone()
    _repeat(lambda o: layer.attend(inp.queries, inp.context_lengths, out=o), ref, 500)


def test_global_stream_k_repeats():
    w = synth.global_sweep(4)
    layer = engine.GlobalLayer(w.batch, capacity=w.capacity, max_proposals=w.proposal_count,
                               scale=w.scale)
    inp = engine.stage_global(w, 0, layer, keep_history=False)
    layer.append(inp.k_new, inp.v_new, inp.context_lengths)
    ref = layer.attend(inp.queries, inp.context_lengths).clone()
    assert np.isfinite(ref.cpu().numpy()).all()
    _repeat(lambda o: layer.attend(inp.queries, inp.context_lengths, out=o), ref, 200)
