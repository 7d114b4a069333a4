"""The allocation-free sliding-window attention entry point.

carat_swa_attention_noalloc serves callers that cannot allocate device memory
(a plugin inside a runtime that owns all GPU memory, or a loop that must never
call cudaMalloc): it uses a fixed scratch array inside the library instead of a
caller workspace.  These tests call it through the C ABI twice in a row (the
second call finds the first call's partial results still in the shared
scratch) and require each output to equal, bit for bit, that of
carat_swa_attention (the entry point that takes a workspace: same kernel, same
plan), and to match the fp64 oracle within the GPU parity tolerance.  This
file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from gpu_harness import assert_close
from sliding_window_gqa_ring_gb300 import carat, engine, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    carat.library()


def _staged(w):
    layer = engine.SlidingLayer(w.batch, window=w.window, q_heads=w.q_heads, kv_heads=w.kv_heads,
                                head_dim=w.head_dim, max_proposals=w.proposal_count,
                                scale=w.scale)
    inp = engine.stage_sliding(w, 0, layer)
    layer.append(inp.k_new, inp.v_new, inp.context_lengths)
    return layer, inp


@pytest.mark.parametrize("which", ["decode_b1", "verify_k4"])
def test_noalloc_matches_workspace_entry_point(orc, which):
    if which == "decode_b1":
        w = synth.sliding_single()
    else:
        w = synth.small("noalloc_k4", seed=5100, batch=12, proposal_count=4, q_heads=16,
                        kv_heads=8, head_dim=256, key_counts=[5, 700, 1023, 1024, 1027, 1028,
                                                              2000, 4096, 9000, 64, 300, 1500],
                        window=1024)
    layer, inp = _staged(w)
    need = carat.swa_workspace_bytes(w.batch, w.proposal_count, w.q_heads, w.kv_heads,
                                     w.head_dim, w.window)
    assert 0 < need <= carat.noalloc_scratch_bytes()
    ref = layer.attend(inp.queries, inp.context_lengths)
    outs = []
    for _ in range(2):
        out = torch.full(inp.queries.shape, float("nan"), dtype=torch.float32, device="cuda")
        carat.carat_swa_attention_noalloc(out, inp.queries, layer.k_ring, layer.v_ring,
                                          inp.context_lengths, scale=layer.scale,
                                          displaced=layer.displaced)
        outs.append(out)
    torch.cuda.synchronize()
    r = ref.cpu().numpy()
    for out in outs:
        np.testing.assert_array_equal(out.cpu().numpy(), r, err_msg=f"noalloc {which}")
    jobs = []
    for b in range(w.batch):
        first, kh, vh = inp.host["hist"][b]
        jobs.append((inp.host["q"][b], kh, vh, first, int(w.context_lengths[b]), w.window,
                     w.scale))
    got = outs[1].cpu().numpy()
    for b, expect in enumerate(orc.attention_batch(jobs)):
        assert_close(got[b], expect, f"noalloc {which} request {b} vs oracle")
    assert carat.carat_get_device_status(clear=True) == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # 16 proposals x 8 query heads per KV head at head_dim 512 take 64-row
    # tiles: two partial slots of 64 x 512 floats for each of a GB300's 152
    # CTAs is about 40 MB of scratch, more than the array holds.
    need = carat.swa_workspace_bytes(8, 16, 16, 2, 512, 1024)
    assert need > carat.noalloc_scratch_bytes()
    q = torch.zeros((8, 16, 16, 512), dtype=torch.bfloat16, device="cuda")
    ring = torch.zeros((8, 1024, 2, 512), dtype=torch.bfloat16, device="cuda")
    disp = torch.zeros((8, 15, 2, 2, 512), dtype=torch.bfloat16, device="cuda")
    ctx = torch.full((8,), 2000, dtype=torch.int32, device="cuda")
    out = torch.empty((8, 16, 16, 512), dtype=torch.float32, device="cuda")
    before = carat.kernel_launches()
    with pytest.raises(carat.CaratError) as e:
        carat.carat_swa_attention_noalloc(out, q, ring, ring, ctx, scale=0.044, displaced=disp)
    assert e.value.status == carat.CARAT_ERR_WORKSPACE
    assert carat.kernel_launches() == before
