"""The bounded pipeline wait gives up, reports MARS_DEV_TIMEOUT and leaves the
context usable (include/mars.h: mars_selftest_wait_timeout).

The kernel runs the same wait helper the library's kernels use on a barrier
that needs two arrivals; the test withholds the second one.  Nothing
asynchronous targets that barrier, so nothing is in flight when the wait gives
up, and the kernel frees the tensor memory it holds before it returns.
"""
import numpy as np
import pytest
import torch

import token_decoding_gb300 as mars
from token_decoding_gb300 import _lib, synth

pytestmark = pytest.mark.gpu


def run(withhold, limit):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ns = torch.zeros(1, dtype=torch.int64, device="cuda")
    _lib.selftest_wait_timeout(withhold, limit, status, ns)
    torch.cuda.synchronize()
    return int(status.item()), int(ns.item())


def test_withheld_arrival_times_out_and_reports():
    st, ns = run(True, 2000)
    assert st & mars.MARS_DEV_TIMEOUT
    per_poll = ns / 2000
    print(f"2000 polls gave up after {ns} ns ({per_poll:.0f} ns per poll)")
    assert ns > 0


def test_arrival_in_time_reports_nothing():
    st, _ = run(False, 2000)
    assert st == 0


def test_context_is_usable_after_a_timeout():
    """After the wait gave up, an ordinary call on the same context still runs and is right."""
    st, _ = run(True, 500)
    assert st & mars.MARS_DEV_TIMEOUT
    import oracle
    from tests.gpu_util import ATTN_TOL, bf16_to_f64, dev_bf16, max_abs

    s = synth.TINY_TRAIN
    q, k, v = synth.train_inputs(s)
    o = mars.train_attn(dev_bf16(q), dev_bf16(k), dev_bf16(v), s.L, s.B)
    torch.cuda.synchronize()
    o_ref, _ = oracle.train_attn(q.f64, k.f64, v.f64, s.L, s.B, s.D ** -0.5)
    assert max_abs(bf16_to_f64(o), o_ref) <= ATTN_TOL


def test_limit_out_of_range_is_rejected_on_the_host():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for bad in (0, (1 << 20) + 1):
        with pytest.raises(mars.MarsError) as e:
            _lib.selftest_wait_timeout(True, bad, status)
        assert e.value.code == _lib.MARS_ERR_INVALID_ARG
    assert int(status.item()) == 0
