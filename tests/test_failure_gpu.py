"""Failure detection without a GPU fault: every pipeline wait of the library is bounded
(about a second), and a wait that gives up sets PFA_DEVERR_TIMEOUT in the device error
word and records where, instead of trapping. pfa_wait_probe makes such a wait run out
on purpose (an mbarrier nothing completes); the test reads the status back, clears it,
and checks that the device still runs the attention path correctly."""
import time

import pytest
import torch

import precision_flash_attention_gb300 as pfa
from precision_flash_attention_gb300 import _lib, inputs

from gpu_helpers import assert_bwd_close, assert_fwd_close, oracle_full, run_gpu

pytestmark = pytest.mark.gpu

PFA_DEVERR_TIMEOUT = _lib.DEVERR_TIMEOUT   # checked against include/pfa.h by the ABI tests


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    pfa.device_error(clear=True)


def test_bounded_wait_gives_up_and_reports():
    try:
        t0 = time.perf_counter()
        pfa.wait_probe()
        err = pfa.device_error()            # synchronises: the probe has finished
        elapsed = time.perf_counter() - t0
        site = pfa.device_error_site()
        assert err & PFA_DEVERR_TIMEOUT, err
        assert site is not None and site["kernel"] == "wait_probe", site
        assert not site["drain"] and site["parity"] == 0 and site["barrier_offset"] == 0
        assert site["block"] == 0
        assert 0.5 < elapsed < 30.0, elapsed   # the wait budget is about a second
    finally:
        pfa.device_error(clear=True)
    assert pfa.device_error() == 0 and pfa.device_error_site() is None


def test_device_stays_usable_after_a_timeout():
    pfa.wait_probe()
    assert pfa.device_error(clear=True) & PFA_DEVERR_TIMEOUT
    t = inputs.make("tiny", seed=0)
    got = run_gpu(t, causal=True, scale=0.125, fix_mode=1)
    ref = oracle_full(t, causal=True, scale=0.125, fix_mode=1)
    assert_fwd_close(got, ref, "after a timeout")
    assert_bwd_close(got, ref, "after a timeout")
