"""Speculative-verify rollback on the rings (GPU, through the C ABI).

A verify step appends k proposals and attends; the sampler keeps the first
`accepted` of them.  carat_ring_rollback restores the rejected rows' slots;
the ring must then equal, byte for byte, the ring after appending only the
accepted rows (the oracle's expected ring for that key count), and the next
step -- appending the tokens that really follow -- must match the oracle on
the corrected history.  Both the fused and the separate append save the
displaced rows the rollback needs.
"""
import numpy as np
import pytest
import torch

from gpu_harness import assert_close, bits
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


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "separate"])
@pytest.mark.parametrize("window", [1024, 200])
def test_rollback_then_next_step(orc, fused, window):
    k = 4
    kcs = [9, 700, 1024, 1026, 1030, 3000, window + 2, 5000]
    w = synth.small("rb", seed=7000 + window, batch=len(kcs), proposal_count=k, q_heads=16,
                    kv_heads=8, head_dim=256, key_counts=kcs, window=window)
    layer = engine.SlidingLayer(w.batch, window=window, max_proposals=k, scale=w.scale,
                                fill=float("nan"))
    inp = engine.stage_sliding(w, 0, layer)
    layer.step(inp.queries, inp.k_new, inp.v_new, inp.context_lengths, fused=fused)
    accepted = np.array([1, 2, 3, 4, 1, 2, 3, 1], dtype=np.int32)
    acc_t = torch.as_tensor(accepted, device="cuda")
    layer.rollback(inp.context_lengths, acc_t, k)
    torch.cuda.synchronize()
    ctx = w.context_lengths
    k_ring, v_ring = bits(layer.k_ring), bits(layer.v_ring)
    # the corrected history: accepted proposals, then different "true" tokens
    w2 = synth.small("rb_true", seed=8000 + window, batch=len(kcs), proposal_count=k,
                     q_heads=16, kv_heads=8, head_dim=256, key_counts=kcs, window=window)
    new_ctx = (ctx + accepted).astype(np.int64)
    hist, kn, vn = [], [], []
    for b in range(w.batch):
        first, kh, vh = inp.host["hist"][b]
        keep = int(new_ctx[b]) - first                   # rows [first, new_ctx) survive
        kc_ring, valid = orc.ring_expected(kh[:keep], first, int(new_ctx[b]), window)
        vc_ring, _ = orc.ring_expected(vh[:keep], first, int(new_ctx[b]), window)
        assert np.array_equal(k_ring[b][valid], kc_ring[valid]), f"K ring after rollback, req {b}"
        assert np.array_equal(v_ring[b][valid], vc_ring[valid]), f"V ring after rollback, req {b}"
        tk = synth.history(w2, 0, b, int(new_ctx[b]), int(new_ctx[b]) + k, "k")
        tv = synth.history(w2, 0, b, int(new_ctx[b]), int(new_ctx[b]) + k, "v")
        hist.append((first, np.concatenate([kh[:keep], tk]), np.concatenate([vh[:keep], tv])))
        kn.append(tk)
        vn.append(tv)
    q2 = np.stack([synth.queries(w2, 0, b) for b in range(w.batch)])
    out = layer.step(engine._bf16_tensor(q2, "cuda"), engine._bf16_tensor(np.stack(kn), "cuda"),
                     engine._bf16_tensor(np.stack(vn), "cuda"), engine._i32(new_ctx, "cuda"),
                     fused=fused)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    refs = orc.attention_batch([(q2[b], hist[b][1], hist[b][2], hist[b][0], int(new_ctx[b]),
                                 window, w.scale) for b in range(w.batch)])
    for b, ref in enumerate(refs):
        assert_close(o[b], ref, f"next step after rollback, request {b}")


def test_rollback_rejects_bad_accept_counts():
    layer = engine.SlidingLayer(2, window=64, max_proposals=4)
    ctx = torch.tensor([100, 200], dtype=torch.int32, device="cuda")
    carat.carat_get_device_status(clear=True)
    layer.rollback(ctx, torch.tensor([5, -1], dtype=torch.int32, device="cuda"), 4)
    torch.cuda.synchronize()
    assert carat.carat_get_device_status(clear=True) & carat.CARAT_DEV_BAD_CONTEXT
    with pytest.raises(carat.CaratError):
        layer.rollback(ctx, torch.tensor([1, 1], dtype=torch.int32, device="cuda"), 1)
