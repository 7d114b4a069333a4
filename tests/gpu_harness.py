"""Shared helpers for the GPU parity tests (not collected by pytest).

Comparison rule for fp32 attention outputs (bf16 inputs):
  * the gate: elementwise |gpu - oracle| <= 2e-2 and normwise
    max|gpu - oracle| / max|oracle| <= 2e-2;
  * and an implementation bound derived from the kernels' arithmetic
    (fp32 accumulation, P rounded to bf16 for the tensor-core PV product, the
    SFU exp2): |gpu - oracle| <= IMPL_ABS + IMPL_REL * |oracle|.  The gate alone
    could hide a single missing key in a 1024-key window, so the structured
    window-probe tests also check edges at 1e-5.
"""
from __future__ import annotations

import numpy as np
import torch

GATE_ABS = 2e-2
GATE_REL = 2e-2
IMPL_ABS = 4e-3
IMPL_REL = 1e-2


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns on the host."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str = "", impl_abs=IMPL_ABS,
                 impl_rel=IMPL_REL):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), f"{what}: non-finite GPU output"
    diff = np.abs(gpu - ref)
    max_abs = float(diff.max()) if diff.size else 0.0
    scale = float(np.abs(ref).max()) if ref.size else 1.0
    normwise = max_abs / max(scale, 1e-30)
    assert max_abs <= GATE_ABS, f"{what}: max abs err {max_abs:.3e} > {GATE_ABS}"
    assert normwise <= GATE_REL, f"{what}: normwise rel err {normwise:.3e} > {GATE_REL}"
    bound = impl_abs + impl_rel * np.abs(ref)
    bad = diff > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond the implementation bound; "
                           f"worst {max_abs:.3e}")
    return max_abs, normwise
