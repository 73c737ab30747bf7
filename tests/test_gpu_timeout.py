"""The bounded device-side wait of the tensor-core weight passes.

Those passes wait on mbarriers for their TMA copies and MMAs; a wait that
runs out of time sets a device flag, the kernel frees its tensor memory and
returns, and the host reports ES_ERR_TIMEOUT.  es_wait_selftest runs one
such wait on a barrier that a second thread arrives at late or never, so the
failure path is exercised without faulting, trapping or hanging the GPU;
the device stays usable afterwards.
"""
import pytest
import torch

from layer_drafting_draft_b300.easyspec import (ES_ERR_ARG, ES_ERR_TIMEOUT, ES_OK, es_accept_resample,
                                                es_wait_selftest)

pytestmark = pytest.mark.gpu


def test_wait_gives_up_when_nothing_arrives():
    assert es_wait_selftest(20_000_000, -1) == ES_ERR_TIMEOUT


def test_wait_returns_when_the_arrival_comes_in_time():
    assert es_wait_selftest(500_000_000, 1_000_000) == ES_OK


def test_arrival_after_the_limit_is_a_timeout():
    assert es_wait_selftest(5_000_000, 100_000_000) == ES_ERR_TIMEOUT


def test_limits_out_of_range_are_refused():
    assert es_wait_selftest(0, -1) == ES_ERR_ARG
    assert es_wait_selftest(3_000_000_000, -1) == ES_ERR_ARG


def test_device_usable_after_a_timeout():
    assert es_wait_selftest(10_000_000, -1) == ES_ERR_TIMEOUT
    p = torch.softmax(torch.randn(1, 3, 64, device="cuda"), -1)
    q = torch.softmax(torch.randn(1, 2, 64, device="cuda"), -1)
    d = torch.argmax(q, -1).to(torch.int32).contiguous()
    n, tok = es_accept_resample(p, q, d, None, True)
    torch.cuda.synchronize()
    assert 0 <= int(n[0]) <= 2
