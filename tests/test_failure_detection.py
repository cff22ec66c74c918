"""Failure detection of the kernels, exercised without faulting the GPU.

Every wait inside the kernels is bounded: a wait that expires raises the CTA's
abort flag (so the other roles stop waiting too), records
GQA_ERR_DEVICE_TIMEOUT in a device status word and returns, leaving the CUDA
context usable.  The device self-test makes a wait run out on purpose (an
mbarrier that nothing arrives on, with a short budget) and checks the status,
the timing of both waiters and that ordinary calls still work afterwards.
"""
import ctypes

import pytest
import torch

import oracle
import causal_grouped_query_gqa_b300 as gq
from causal_grouped_query_gqa_b300.inputs import make_inputs
from parity_util import check_close, to64


def test_selftest_rejects_bad_arguments():
    """Needs no GPU: argument checks come before any device work."""
    el = (ctypes.c_ulonglong * 2)()
    ok = (ctypes.c_int * 2)()
    assert gq.gqa_attn_selftest_timeout(20, None, ok) == gq.GQA_ERR_NULL
    assert gq.gqa_attn_selftest_timeout(20, el, None) == gq.GQA_ERR_NULL
    assert gq.gqa_attn_selftest_timeout(0, el, ok) == gq.GQA_ERR_SHAPE
    assert gq.gqa_attn_selftest_timeout(5000, el, ok) == gq.GQA_ERR_SHAPE


@pytest.mark.gpu
@pytest.mark.parametrize("budget_ms", [10, 50])
def test_expired_wait_is_reported_and_the_context_survives(budget_ms):
    assert gq.gqa_attn_last_device_status() == gq.GQA_OK
    rc, elapsed, returned = gq.selftest_timeout(budget_ms)
    assert rc == gq.GQA_ERR_DEVICE_TIMEOUT, gq.gqa_attn_strerror(rc)
    assert returned == [0, 0]  # neither wait claimed success
    budget_ns = budget_ms * 1_000_000
    # the short wait expired after its budget (plus at most a few suspensions)
    assert budget_ns <= elapsed[0] < budget_ns + 20_000_000, elapsed
    # the 2 s wait left through the CTA abort flag, right after the first
    assert elapsed[1] < elapsed[0] + 10_000_000, elapsed
    # the status word was read and cleared, and ordinary calls still work
    assert gq.gqa_attn_last_device_status() == gq.GQA_OK
    q, k, v = (t.cuda() for t in make_inputs(1, 4, 2, 300, seed=3))
    o, lse = gq.fwd(q, k, v)
    torch.cuda.synchronize()
    assert gq.gqa_attn_last_device_status() == gq.GQA_OK
    ro, _ = oracle.attn_fwd(to64(q), to64(k), to64(v))
    check_close("O after the self-test", to64(o), ro)
