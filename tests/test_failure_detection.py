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


def _stall_lib():
    """The failure-detection test build of the library (a separate module with
    its own device status word): CTA 0 of each kernel never gets one of its
    loads, and every wait gives up after 100 ms."""
    from causal_grouped_query_gqa_b300 import build as gbuild
    path = gbuild.build_stall_test()
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.gqa_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp]
    lib.gqa_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                 i, i, i, i, i, i, i, i, f, vp, sz, vp]
    lib.gqa_attn_bwd_workspace_size.argtypes = [i, i, i, i, i]
    lib.gqa_attn_bwd_workspace_size.restype = sz
    lib.gqa_attn_last_device_status.argtypes = [vp]
    lib.gqa_attn_fwd_yarn.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f,
                                      f, f, i, f, f, i, i, vp, sz, vp]
    lib.gqa_attn_fwd_yarn_workspace_size.argtypes = [i, i, i, i, i, i]
    lib.gqa_attn_fwd_yarn_workspace_size.restype = sz
    lib.gqa_attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, f, f, vp]
    return lib


@pytest.mark.gpu
@pytest.mark.parametrize("window,n_sink", [(0, 0), (200, 64)])
def test_production_kernels_leave_through_the_abort_path(window, n_sink):
    """A load that never lands: the forward and the backward must each end
    (every role leaves through its bounded waits and the CTA abort flag, TMEM
    is freed), report GQA_ERR_DEVICE_TIMEOUT, and leave the context usable."""
    import time
    lib = _stall_lib()
    B, H, G, S, d, scale = 1, 4, 2, 700, 64, 0.125
    q, k, v, do = (t.cuda() for t in make_inputs(B, H, G, S, seed=9, with_grad=True))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(lib.gqa_attn_bwd_workspace_size(B, H, G, S, d), dtype=torch.uint8,
                     device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    p = lambda t: t.data_ptr()
    assert lib.gqa_attn_last_device_status(st) == gq.GQA_OK
    t0 = time.perf_counter()
    assert lib.gqa_attn_fwd(p(q), p(k), p(v), p(o), p(lse), B, H, G, S, d, 1, window, n_sink,
                            scale, st) == gq.GQA_OK
    assert lib.gqa_attn_last_device_status(st) == gq.GQA_ERR_DEVICE_TIMEOUT
    assert lib.gqa_attn_bwd(p(q), p(k), p(v), p(o), p(do), p(lse), p(dq), p(dk), p(dv), B, H, G,
                            S, d, 1, window, n_sink, scale, p(ws), ws.numel(),
                            st) == gq.GQA_OK
    assert lib.gqa_attn_last_device_status(st) == gq.GQA_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 10.0  # bounded waits of 100 ms, a few in sequence
    # the context is intact: the regular library computes correct results
    o2, lse2 = gq.fwd(q, k, v, window=window, n_sink=n_sink, scale=scale)
    dq2, dk2, dv2 = gq.bwd(q, k, v, o2, do, lse2, window=window, n_sink=n_sink, scale=scale)
    torch.cuda.synchronize()
    assert gq.gqa_attn_last_device_status() == gq.GQA_OK
    ro, _ = oracle.attn_fwd(to64(q), to64(k), to64(v), window=window, n_sink=n_sink, scale=scale)
    rq, rk, rv = oracle.attn_bwd(to64(q), to64(k), to64(v), to64(do), window=window,
                                 n_sink=n_sink, scale=scale)
    check_close("O after the aborted launches", to64(o2), ro)
    check_close("dQ after the aborted launches", to64(dq2), rq)
    check_close("dK after the aborted launches", to64(dk2), rk)
    check_close("dV after the aborted launches", to64(dv2), rv)


@pytest.mark.gpu
def test_yarn_and_fp8_forwards_leave_through_the_abort_path():
    """The same missing load in the rotary forward (both modes: rotated inputs,
    and the query-rotation barriers of the fused mode; with the score bound)
    and in the fp8 instantiation, whose tiles' transaction counts differ: no
    role may be kept waiting."""
    lib = _stall_lib()
    B, H, G, S, d, scale = 1, 6, 2, 700, 64, 0.125
    q, k, v = (t.cuda() for t in make_inputs(B, H, G, S, seed=19))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    p = lambda t: t.data_ptr()
    assert lib.gqa_attn_last_device_status(st) == gq.GQA_OK
    for mode in (gq.GQA_ROPE_PREPASS, gq.GQA_ROPE_FUSED):
        ws = torch.empty(lib.gqa_attn_fwd_yarn_workspace_size(B, H, G, S, d, mode),
                         dtype=torch.uint8, device="cuda")
        assert lib.gqa_attn_fwd_yarn(p(q), p(k), p(v), p(o), p(lse), B, H, G, S, d, 1, 0, 0, scale,
                                     10000.0, 32.0, 6400, 1.0, 32.0, 1, mode, p(ws), ws.numel(),
                                     st) == gq.GQA_OK
        assert lib.gqa_attn_last_device_status(st) == gq.GQA_ERR_DEVICE_TIMEOUT
    q8 = (q.float() * 64).to(torch.float8_e4m3fn).view(torch.uint8)
    k8 = (k.float() * 64).to(torch.float8_e4m3fn).view(torch.uint8)
    assert lib.gqa_attn_fwd_fp8(p(q8), p(k8), p(v), p(o), p(lse), B, H, G, S, d, 1, 0, 0, scale,
                                1 / 64, 1 / 64, st) == gq.GQA_OK
    assert lib.gqa_attn_last_device_status(st) == gq.GQA_ERR_DEVICE_TIMEOUT
    # the context is intact
    o2, _ = gq.fwd_yarn(q, k, v)
    torch.cuda.synchronize()
    assert gq.gqa_attn_last_device_status() == gq.GQA_OK
    ro, _ = oracle.attn_fwd_yarn(to64(q), to64(k), to64(v))
    check_close("YaRN O after the aborted launches", to64(o2), ro)
