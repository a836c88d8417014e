"""Failure detection without a GPU fault: a bounded wait that runs out is
reported through the device status word and the context stays usable.

The library's kernels wait on mbarriers for their bulk copies with a time
limit; the self-test entry point runs the same bounded wait on a phase that
nothing completes (a flag that nothing sets), with a 50 ms limit."""
import time

import numpy as np
import pytest

import oracle
import workloads as W
from tests.gpu_helpers import assert_parity, to_dev, to_host

pytestmark = pytest.mark.gpu

SEG_ERR_DEVICE_TIMEOUT = 5


def test_wait_that_runs_out_is_reported_and_the_device_keeps_working():
    import torch
    import segmented_reduction_csr_gb300 as sr
    assert sr.device_status() == 0                       # clean before
    t0 = time.perf_counter()
    sr.selftest_wait_timeout(50)
    assert sr.device_status() == SEG_ERR_DEVICE_TIMEOUT  # synchronises, reads and clears
    elapsed = time.perf_counter() - t0
    assert 0.04 <= elapsed < 5.0, elapsed                # the wait gave up after its limit
    assert sr.device_status() == 0                       # cleared by the read
    # the context is usable: a reduction right after is correct
    w = W.make("tiny")
    r = sr.seg_reduce(to_dev(w.values["f32"]), to_dev(w.offsets), "max")
    assert_parity(w.values["f32"], w.offsets, "max", to_host(r[0]), to_host(r[1]), where="after timeout")
    assert sr.device_status() == 0
    torch.cuda.synchronize()


def test_selftest_rejects_bad_limits():
    import segmented_reduction_csr_gb300 as sr
    with pytest.raises(sr.SegReduceError):
        sr.selftest_wait_timeout(0)
    with pytest.raises(sr.SegReduceError):
        sr.selftest_wait_timeout(20000)
