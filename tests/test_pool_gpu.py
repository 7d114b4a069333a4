"""Rings and global pages in one shared pool (GPU, through the C ABI).

Two sliding layers' rings and one global layer's pages are allocated from
the same K and V pools by the library's allocator; the fused steps must match
the oracle, the rings must hold the expected bytes, and every page row the
global layer wrote must hold its history row."""
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


def test_shared_pool_rings_and_pages(orc):
    k = 4
    kcs = [6, 900, 1030, 2600, 5000]
    B = len(kcs)
    # page = 128 sliding rows (8 x 256 bf16) = 256 global rows (2 x 512 bf16) = 512 KiB
    page_bytes = 128 * 8 * 256 * 2
    pool = engine.SharedPool(num_pages=128, page_bytes=page_bytes, pages_per_ring=8,
                             fill=float("nan"))
    sw = synth.small("pool_swa", seed=7100, batch=B, proposal_count=k, q_heads=16, kv_heads=8,
                     head_dim=256, key_counts=kcs, window=1024)
    gw = synth.small("pool_glob", seed=7200, batch=B, proposal_count=k, q_heads=16, kv_heads=2,
                     head_dim=512, key_counts=kcs, capacity=0)
    # interleave allocations the way requests arrive: rings and pages mixed
    ring_ids = [[], []]
    page_lists = []
    for b in range(B):
        for layer in range(2):
            r = pool.alloc.alloc_ring()
            assert r >= 0
            ring_ids[layer].append(r)
        pages = pool.alloc.alloc_pages(-(-kcs[b] // 256))
        assert pages is not None
        page_lists.append(pages)
    max_pages = max(len(p) for p in page_lists)
    table = np.full((B, max_pages), -1, np.int32)
    for b, pages in enumerate(page_lists):
        table[b, :len(pages)] = pages[::-1]           # pages need not be in order
    page_table = torch.as_tensor(table, device="cuda")
    st = pool.alloc.stats()
    assert st["rings"] == 2 * B and st["pages"] == sum(len(p) for p in page_lists)

    outs, checks = [], []
    for layer in range(2):
        lay = engine.SlidingLayer(pool.num_pages // 8, window=1024, max_batch=B, max_proposals=k,
                                  scale=sw.scale, rings=pool.rings(1024, 8, 256))
        ids = torch.as_tensor(np.array(ring_ids[layer], np.int32), device="cuda")
        inp = engine.stage_sliding(sw, layer, lay, ring_ids=ring_ids[layer])
        out = lay.step(inp.queries, inp.k_new, inp.v_new, inp.context_lengths, ring_ids=ids)
        outs.append(out)
        checks.append(("swa", lay, inp, ring_ids[layer]))
    g = engine.PagedGlobalLayer(pool, page_table, max_proposals=k, scale=gw.scale)
    ginp = engine.stage_global_paged(gw, 0, g)
    gout = g.step(ginp.queries, ginp.k_new, ginp.v_new, ginp.context_lengths)
    torch.cuda.synchronize()

    for (kind, lay, inp, ids), out in zip(checks, outs):
        o = out.cpu().numpy()
        kr, vr = bits(lay.k_ring), bits(lay.v_ring)
        for b in range(B):
            first, kh, vh = inp.host["hist"][b]
            ref = orc.attention_request(inp.host["q"][b], kh, vh, first, int(sw.context_lengths[b]),
                                        1024, sw.scale)
            assert_close(o[b], ref, f"pooled ring layer, request {b}")
            exp_k, valid = orc.ring_expected(kh, first, kcs[b], 1024)
            exp_v, _ = orc.ring_expected(vh, first, kcs[b], 1024)
            assert np.array_equal(kr[ids[b]][valid], exp_k[valid])
            assert np.array_equal(vr[ids[b]][valid], exp_v[valid])
    go = gout.cpu().numpy()
    kp, vp = bits(g.key_pages), bits(g.value_pages)
    for b in range(B):
        _, kh, vh = ginp.host["hist"][b]
        ref = orc.attention_request(ginp.host["q"][b], kh, vh, 0, int(gw.context_lengths[b]), 0,
                                    gw.scale)
        assert_close(go[b], ref, f"paged global layer, request {b}")
        t = np.arange(kcs[b])
        rows_k = kp[table[b, t // 256], t % 256]
        rows_v = vp[table[b, t // 256], t % 256]
        assert np.array_equal(rows_k, kh) and np.array_equal(rows_v, vh)
