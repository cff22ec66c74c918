"""Run-time index checks of the kernels (the debug build compiled with
GQA_DEVICE_CHECKS): TMA tile coordinates, query/key ranges and the global
store offsets of O, LSE, dK, dV and the dQ reduction are checked on every
access, a violation would report GQA_ERR_DEVICE_BOUNDS and skip the access.
Small odd shapes -- ragged tails, odd heads per kv head, multi-query, windows
and sinks across tile edges, more units than SMs -- must run clean and still
match the oracle.  (The checks stand in for a memory checker.)"""
import ctypes

import pytest
import torch

import oracle
import causal_grouped_query_gqa_b300 as gq
from causal_grouped_query_gqa_b300.inputs import make_inputs
from parity_util import check_close, to64

pytestmark = pytest.mark.gpu

SHAPES = [  # B, H, G, S, causal, window, n_sink
    (1, 2, 1, 1, 1, 0, 0),
    (1, 3, 1, 127, 1, 0, 0),
    (2, 6, 2, 129, 1, 0, 0),
    (1, 8, 1, 300, 1, 0, 0),
    (1, 4, 2, 513, 0, 0, 0),
    (1, 4, 2, 777, 1, 129, 300),
    (2, 6, 2, 1000, 1, 100, 130),
    (3, 6, 2, 1536, 1, 0, 0),
]


@pytest.fixture(scope="module")
def checked():
    from causal_grouped_query_gqa_b300 import build as gbuild
    lib = ctypes.CDLL(gbuild.build_checked())
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


@pytest.mark.parametrize("B,H,G,S,causal,window,n_sink", SHAPES)
def test_checked_build_runs_clean(checked, B, H, G, S, causal, window, n_sink):
    d, scale = 64, 0.125
    q, k, v, do = (t.cuda() for t in make_inputs(B, H, G, S, seed=S, with_grad=True))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(checked.gqa_attn_bwd_workspace_size(B, H, G, S, d), dtype=torch.uint8,
                     device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    p = lambda t: t.data_ptr()
    assert checked.gqa_attn_fwd(p(q), p(k), p(v), p(o), p(lse), B, H, G, S, d, causal, window,
                                n_sink, scale, st) == gq.GQA_OK
    assert checked.gqa_attn_bwd(p(q), p(k), p(v), p(o), p(do), p(lse), p(dq), p(dk), p(dv), B,
                                H, G, S, d, causal, window, n_sink, scale, p(ws), ws.numel(),
                                st) == gq.GQA_OK
    assert checked.gqa_attn_last_device_status(st) == gq.GQA_OK
    kw = dict(causal=bool(causal), window=window, n_sink=n_sink, scale=scale)
    ro, _ = oracle.attn_fwd(to64(q), to64(k), to64(v), **kw)
    rq, rk, rv = oracle.attn_bwd(to64(q), to64(k), to64(v), to64(do), **kw)
    check_close("O", to64(o), ro)
    check_close("dQ", to64(dq), rq)
    check_close("dK", to64(dk), rk)
    check_close("dV", to64(dv), rv)


@pytest.mark.parametrize("B,H,G,S,causal,window,n_sink", [SHAPES[1], SHAPES[5], SHAPES[7]])
def test_checked_build_yarn_and_fp8(checked, B, H, G, S, causal, window, n_sink):
    """The rotary and fp8 forwards under the index checks: clean, and equal to
    the oracle (rotated-and-rounded q, k; decoded E4M3 q, k)."""
    d, scale = 64, 0.125
    q, k, v = make_inputs(B, H, G, S, seed=S + 1)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    p = lambda t: t.data_ptr()
    kw = dict(causal=bool(causal), window=window, n_sink=n_sink, scale=scale)
    ro, _ = oracle.attn_fwd_yarn(to64(q), to64(k), to64(v), **kw)
    for mode in (gq.GQA_ROPE_PREPASS, gq.GQA_ROPE_FUSED):
        ws = torch.empty(checked.gqa_attn_fwd_yarn_workspace_size(B, H, G, S, d, mode),
                         dtype=torch.uint8, device="cuda")
        assert checked.gqa_attn_fwd_yarn(p(qd), p(kd), p(vd), p(o), p(lse), B, H, G, S, d, causal,
                                         window, n_sink, scale, 10000.0, 32.0, 6400, 1.0, 32.0, 1,
                                         mode, p(ws), ws.numel(), st) == gq.GQA_OK
        assert checked.gqa_attn_last_device_status(st) == gq.GQA_OK
        check_close(f"O (YaRN, rope_mode {mode})", to64(o), ro)
    q8 = (q.float() * 64).to(torch.float8_e4m3fn).view(torch.uint8)
    k8 = (k.float() * 64).to(torch.float8_e4m3fn).view(torch.uint8)
    assert checked.gqa_attn_fwd_fp8(p(q8.cuda()), p(k8.cuda()), p(vd), p(o), p(lse), B, H, G, S, d,
                                    causal, window, n_sink, scale, 1 / 64, 1 / 64, st) == gq.GQA_OK
    assert checked.gqa_attn_last_device_status(st) == gq.GQA_OK
    ro, _ = oracle.attn_fwd_fp8(q8.numpy(), k8.numpy(), to64(v), 1 / 64, 1 / 64, **kw)
    check_close("O (fp8)", to64(o), ro)
