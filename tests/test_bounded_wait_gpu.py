"""The bounded waits of the library's kernels give up without faulting.

Every wait on a barrier phase in the kernels is bounded: when it runs out the
kernel sets CARAT_DEV_TIMEOUT in the device status word, stops, and returns,
so the CUDA context stays usable and the host learns of it.  Here a one-thread
kernel waits, with the same helper and a short limit, on a barrier phase that
nothing completes (no fault, no hang: the wait ends by itself), then the test
checks the status bit, that it clears, and that an attention call afterwards
still matches the oracle.
"""
import time

import pytest
import torch

from sliding_window_gqa_ring_gb300 import carat, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    carat.library()
    carat.carat_get_device_status(clear=True)


def test_limit_out_of_range_rejected():
    for bad in (0, 999_999, 10_000_000_001):
        with pytest.raises(carat.CaratError):
            carat.carat_check_bounded_wait(bad)


def test_bounded_wait_gives_up_and_context_stays_usable(orc):
    from test_parity_gpu import _run_sliding
    assert carat.carat_get_device_status(clear=True) == 0
    t0 = time.perf_counter()
    carat.carat_check_bounded_wait(20_000_000)   # 20 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    status = carat.carat_get_device_status(clear=True)
    assert status & carat.CARAT_DEV_TIMEOUT, status
    assert elapsed >= 0.02, elapsed           # it waited at least the limit
    assert elapsed < 20.0, elapsed            # and then gave up
    assert carat.carat_get_device_status(clear=True) == 0
    # the context is still usable: a sliding-window call matches the oracle
    _run_sliding(orc, synth.sliding_single(), fused=False)
    assert carat.carat_get_device_status(clear=True) == 0
