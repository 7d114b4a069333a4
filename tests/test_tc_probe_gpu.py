"""Self-check of the tensor-core primitives (TMA swizzled loads, tcgen05.mma
descriptors for K-major and MN-major operands, hand-swizzled operands, TMEM
loads and stores) against torch matmuls.  Layout checks of the hardware
operations the attention kernel is built from, on in-bounds inputs."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def probe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sliding_window_gqa_ring_gb300 import build
    lib = ctypes.CDLL(build.build_probe())
    lib.tc_probe_run.restype = ctypes.c_int
    lib.tc_probe_run.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                 ctypes.c_void_p]
    return lib


@pytest.mark.parametrize("n", [16, 32, 64])
def test_kmajor_qk_product(probe, n):
    g = torch.Generator().manual_seed(n)
    a = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    b = torch.randn(n, 128, generator=g).to(torch.bfloat16).cuda()
    out = torch.full((2, 128, n), float("nan"), device="cuda")
    rc = probe.tc_probe_run(1, n, a.data_ptr(), b.data_ptr(), out.data_ptr())
    assert rc == 0
    ref = a.float() @ b.float().T
    torch.testing.assert_close(out[0], ref, rtol=1e-4, atol=1e-3)
    torch.testing.assert_close(out[1], 2 * ref, rtol=1e-4, atol=2e-3)


@pytest.mark.parametrize("n", [16, 32, 64])
def test_mnmajor_pv_product(probe, n):
    g = torch.Generator().manual_seed(100 + n)
    v = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()   # [keys][d]
    p = torch.rand(n, 128, generator=g).to(torch.bfloat16).cuda()      # [rows][keys]
    out = torch.full((2, 128, n), float("nan"), device="cuda")
    rc = probe.tc_probe_run(2, n, v.data_ptr(), p.data_ptr(), out.data_ptr())
    assert rc == 0
    ref = v.float().T @ p.float().T                                     # [d][rows]
    torch.testing.assert_close(out[0], ref, rtol=1e-4, atol=1e-3)
    torch.testing.assert_close(out[1], 2 * ref, rtol=1e-4, atol=2e-3)
