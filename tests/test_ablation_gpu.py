"""The unfused global verify (the pages' separate-steps design, used as an
ablation) against the fp64 oracle.

"fp32" keeps scores, weights and outputs in fp32: it must meet the same gate
and implementation bound as the fused kernel.  "bf16" is the pages' setting
(GEMMs that write bf16).  Its bound follows from the roundings it makes, for a
request whose visible scores satisfy |s| <= S and values |v| <= V:
  * each score is rounded to bf16: |ds| <= u*S, u = 2^-8 (8 significant bits,
    round to nearest);
  * a softmax of scores moved by at most d changes every weight by a factor in
    [e^-2d, e^2d];
  * each weight is rounded to bf16 (factor 1 +- u), then the output (1 +- u).
So |O - o| <= E*V*(1 + u) + u*|o| with E = e^(2uS)*(1 + u) - 1, plus the fp32
accumulation slack of the fused kernel's bound (4e-3).
"""
import math

import numpy as np
import pytest
import torch

from gpu_harness import IMPL_ABS, assert_close
from sliding_window_gqa_ring_gb300 import ablation, synth

pytestmark = pytest.mark.gpu

U_BF16 = 2.0 ** -8


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


_CASES = {}


def _case(orc, name):
    """Staged layer, inputs, oracle outputs and per-request (S, V) of a workload."""
    if name not in _CASES:
        w = synth.global_single() if name == "global_single" else synth.global_sweep(4)
        layer, inp = ablation.staged(w)
        jobs, bounds = [], []
        for b in range(w.batch):
            kc = int(w.key_counts[b])
            kh = synth.history(w, 0, b, 0, kc, "k")
            vh = synth.history(w, 0, b, 0, kc, "v")
            q = inp.host["q"][b]
            jobs.append((q, kh, vh, 0, int(w.context_lengths[b]), 0, w.scale))
            # largest |score| over every row and key (the visible ones are among them)
            qf = synth.bf16_to_float(q).astype(np.float64)          # [k][Hq][D]
            kf = synth.bf16_to_float(kh).astype(np.float64)         # [n][Hkv][D]
            g = w.q_heads // w.kv_heads
            smax = 0.0
            for c in range(w.kv_heads):
                rows = qf[:, c * g:(c + 1) * g, :].reshape(-1, w.head_dim)
                smax = max(smax, float(np.abs(rows @ kf[:, c, :].T).max()) * w.scale)
            vmax = float(np.abs(synth.bf16_to_float(vh)).max())
            bounds.append((smax, vmax))
        _CASES[name] = (w, layer, inp, orc.attention_batch(jobs), bounds)
    return _CASES[name]


@pytest.mark.parametrize("pad64", [False, True], ids=["exact", "padded64"])
@pytest.mark.parametrize("name", ["global_single", "global_sweep_k4"])
def test_unfused_fp32_matches_oracle(orc, name, pad64):
    w, layer, inp, refs, _ = _case(orc, name)
    out = ablation.unfused_verify(layer.key_cache, layer.value_cache, inp.queries, w.key_counts,
                                  w.proposal_count, w.scale, "fp32", pad64).cpu().numpy()
    for b, ref in enumerate(refs):
        assert_close(out[b], ref, f"unfused fp32 {name} request {b}")


@pytest.mark.parametrize("pad64", [False, True], ids=["exact", "padded64"])
@pytest.mark.parametrize("name", ["global_single", "global_sweep_k4"])
def test_unfused_bf16_within_its_rounding_bound(orc, name, pad64):
    w, layer, inp, refs, bounds = _case(orc, name)
    out = ablation.unfused_verify(layer.key_cache, layer.value_cache, inp.queries, w.key_counts,
                                  w.proposal_count, w.scale, "bf16", pad64).cpu().numpy()
    for b, ref in enumerate(refs):
        smax, vmax = bounds[b]
        e = math.exp(2 * U_BF16 * smax) * (1 + U_BF16) - 1
        bound = e * vmax * (1 + U_BF16) + U_BF16 * np.abs(ref) + IMPL_ABS
        diff = np.abs(out[b].astype(np.float64) - ref)
        assert np.isfinite(out[b]).all()
        assert (diff <= bound).all(), (f"unfused bf16 {name} request {b}: worst excess "
                                       f"{float((diff - bound).max()):.3e}")
