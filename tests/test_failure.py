"""Failure detection without a GPU fault: every wait in the kernels is bounded; when one
runs out the kernel records the error in the cache's device error word and returns, and
the host reads it with kv_device_error.  kv_debug_wait_timeout runs that path on its own
(a bounded wait on a barrier that nothing completes), so the test needs no broken kernel
and leaves the context usable.
"""
import pytest

from harness import Scenario

pytestmark = pytest.mark.gpu


def test_timed_out_wait_is_reported_and_the_cache_stays_usable():
    import torch
    import kv_cache_incremental_gb300 as kvi
    sc = Scenario(B=2, max_len=64, Hq=4, Hk=2, D=64, W=8, kinds=[1, 0], seed=7)
    sc.step([5, 3], C=5, check_state=True)
    assert sc.cache.device_error() == 0
    sc.cache.debug_wait_timeout(4096)
    torch.cuda.synchronize()
    assert sc.cache.device_error() == 1   # reported once, then cleared
    assert sc.cache.device_error() == 0
    sc.step([1, 1], C=1, check_state=True)   # later work runs and is checked
    sc.step([7, 0], C=7, check_state=True)
    assert sc.cache.device_error() == 0
    for bad in (0, (1 << 20) + 1):
        with pytest.raises(kvi.KVError):
            sc.cache.debug_wait_timeout(bad)
