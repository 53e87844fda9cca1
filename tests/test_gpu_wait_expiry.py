"""The bounded-wait failure path of the pipeline kernels, made to run out on
purpose in the permitted way: one warp waits on an mbarrier phase that nothing
completes, with a short bound and nothing in flight (pa_check_bounded_wait).

The wait must give up after its bound (not hang), every lane must agree on the
outcome, the kernel must report PA_DEVERR_WAIT through the device error word,
and the context must stay usable: a decode right after it runs clean and
matches the oracle."""
import numpy as np
import pytest
import torch

import workloads
from gpu_cases import assert_close, gpu_decode, oracle_decode, pa_mod, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    return pa_mod()


@pytest.mark.parametrize("limit_ns", [20_000, 1_000_000, 20_000_000])
def test_a_wait_that_nothing_completes_gives_up_and_reports(pa, limit_ns):
    assert pa.get_device_error() == 0
    report = torch.full((4,), -1, dtype=torch.int64, device="cuda")
    pa.check_bounded_wait(limit_ns, report)
    bits = pa.get_device_error()                    # synchronises; the kernel has returned
    assert bits == pa.PA_DEVERR_WAIT
    seen, gave_up, agreed, waited = report.cpu().tolist()
    assert seen == 1                                # a completed phase is still seen
    assert gave_up == 32 and agreed == 1            # every lane gave up, the warp agreed
    assert waited >= limit_ns                       # not before its bound ...
    assert waited < limit_ns + 200_000_000          # ... and not long after it
    assert pa.get_device_error() == 0               # reading cleared the word


def test_the_context_stays_usable_after_an_expired_wait(pa):
    pa.check_bounded_wait(100_000)
    assert pa.get_device_error() == pa.PA_DEVERR_WAIT
    w = workloads.make_decode("after_wait", 77, np.array([1, 300, 900], np.int32), 16, 4, 128, 16, "bf16")
    out, _, _ = gpu_decode(w)
    assert pa.get_device_error() == 0
    assert_close(to_f64(out), oracle_decode(w, range(w.num_seqs)), "bf16", "decode after an expired wait")


def test_bounds_outside_the_accepted_range_are_refused(pa):
    for bad in (0, 999, 1_000_000_001):
        with pytest.raises(pa.PagedAttnError):
            pa.check_bounded_wait(bad)
    assert pa.get_device_error() == 0
