"""The bounded-wait error path on the GPU, with no fault and no hang.

Every wait inside a CTA of this library is bounded; a wait that runs out
records PKV_DEVERR_TIMEOUT in the device error word and the CTA returns.
pkv_wait_selftest makes such a wait run out on purpose (one CTA waits, with a
short limit, on an mbarrier phase that nothing completes), so the path is
tested without stalling a real pipeline: the host reads the code, the word is
cleared, and the context stays usable for the next call.
"""
import time

import numpy as np
import pytest

import paged_kv_cache_11_gb300 as pkv
from paged_kv_cache_11_gb300 import workload as W
from tests.step_helpers import gpu_step, max_abs_err, oracle_step, to_bits

pytestmark = pytest.mark.gpu
TIMEOUT = 5  # PKV_DEVERR_TIMEOUT


def test_wait_runs_out_and_is_reported(gpu):
    assert pkv.check_device_error() == 0
    t0 = time.perf_counter()
    pkv.wait_selftest(50_000)  # 50 ms
    assert pkv.check_device_error() == TIMEOUT
    elapsed = time.perf_counter() - t0
    assert 0.045 <= elapsed < 5.0, elapsed  # the wait lasted its limit, and no longer than a bounded wait can
    assert pkv.check_device_error() == 0  # read and cleared


def test_context_usable_after_a_timeout(gpu):
    pkv.wait_selftest(10_000)
    assert pkv.check_device_error() == TIMEOUT
    wl = W.make_workload("tiny")
    wl.poison()
    kc, vc, out = gpu_step(wl, gpu)
    okc, ovc, ref = oracle_step(wl)
    assert np.array_equal(to_bits(kc), okc) and np.array_equal(to_bits(vc), ovc)
    assert max_abs_err(out, ref) <= 5e-3
    assert pkv.check_device_error() == 0


def test_limit_out_of_range_launches_nothing(gpu):
    n = pkv.launch_count()
    for bad in (0, -1, 2_000_001):
        with pytest.raises(pkv.PagedKVError):
            pkv.wait_selftest(bad)
    assert pkv.launch_count() == n
    assert pkv.check_device_error() == 0
