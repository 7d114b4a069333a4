"""The multi-layer decode step (engine.DecodeStep): eager launches, a CUDA
graph replay and the host-to-host path with overlapped copies give the same
outputs, and they match the oracle on the first step."""
import numpy as np
import pytest
import torch

from gpu_harness import assert_close
from sliding_window_gqa_ring_gb300 import carat, engine, synth

pytestmark = pytest.mark.gpu


def _build():
    sw = synth.small("step_swa", seed=6001, batch=6, proposal_count=4, q_heads=16, kv_heads=8,
                     head_dim=256, key_counts=[9, 700, 1024, 1030, 3000, 5000], window=1024)
    gw = synth.small("step_glob", seed=6002, batch=6, proposal_count=4, q_heads=16, kv_heads=2,
                     head_dim=512, key_counts=[9, 700, 1024, 1030, 3000, 5000], capacity=5120)
    layers, inputs, hists = [], [], []
    for li in range(2):
        lay = engine.SlidingLayer(sw.batch, window=1024, max_proposals=4, scale=sw.scale)
        inp = engine.stage_sliding(sw, li, lay)
        layers.append(lay)
        inputs.append((inp.queries, inp.k_new, inp.v_new, inp.context_lengths))
        hists.append(("swa", sw, inp.host))
    g = engine.GlobalLayer(gw.batch, capacity=gw.capacity, max_proposals=4, scale=gw.scale)
    ginp = engine.stage_global(gw, 0, g)
    layers.append(g)
    inputs.append((ginp.queries, ginp.k_new, ginp.v_new, ginp.context_lengths))
    hists.append(("global", gw, ginp.host))
    return engine.DecodeStep(layers, inputs), hists


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    carat.library()


def test_eager_graph_and_host_paths_agree(orc):
    step, hists = _build()
    first = [o.clone() for o in step.run()]
    torch.cuda.synchronize()
    # first step against the oracle
    for out, (kind, w, host) in zip(first, hists):
        o = out.cpu().numpy()
        for b in range(w.batch):
            first_pos, kh, vh = host["hist"][b]
            ref = orc.attention_request(host["q"][b], kh, vh, first_pos,
                                        int(w.context_lengths[b]),
                                        w.window if kind == "swa" else 0, w.scale)
            assert_close(o[b], ref, f"{kind} request {b}")
    # repeated steps: the same kernels on the same (already appended) state
    eager = [o.clone() for o in step.run()]
    step.capture()
    replayed = [o.clone() for o in step.replay()]
    h_in = [tuple(x.cpu().pin_memory() for x in din) for din in step.inputs]
    # three host-path steps back to back: both device staging sets, and the
    # first set again once its previous outputs have been copied out
    h_outs = [[torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in step.outputs]
              for _ in range(3)]
    for h_out in h_outs:
        step.run_from_host(h_in, h_out)
    step.finish()
    torch.cuda.synchronize()
    for h_out in h_outs:
        for a, b_, c in zip(eager, replayed, h_out):
            assert torch.equal(a, b_)
            assert torch.equal(a.cpu(), c)
    # and the device path after the host path
    again = [o.clone() for o in step.run()]
    torch.cuda.synchronize()
    for a, d in zip(eager, again):
        assert torch.equal(a, d)
    assert carat.carat_get_device_status(clear=True) == 0
