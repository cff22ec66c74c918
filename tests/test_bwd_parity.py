"""GPU backward vs the float64 oracle through the C ABI.

The GPU backward consumes the GPU forward's O and LSE (as a caller would);
the oracle recomputes its own exact P from q, k, v."""
import numpy as np
import pytest
import torch

import oracle
import causal_grouped_query_gqa_b300 as gq
from causal_grouped_query_gqa_b300.inputs import WORKLOADS, make_inputs
from parity_util import check_close, to64

pytestmark = pytest.mark.gpu


def _gpu_fwd_bwd(q, k, v, do, **kw):
    q, k, v, do = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = gq.fwd(q, k, v, **kw)
    dq, dk, dv = gq.bwd(q, k, v, o, do, lse, **kw)
    torch.cuda.synchronize()
    assert gq.gqa_attn_last_device_status() == gq.GQA_OK
    return dq, dk, dv


def _run_full(B, H, G, S, causal=True, window=0, n_sink=0, seed=0, scale=None):
    q, k, v, do = make_inputs(B, H, G, S, seed=seed, with_grad=True)
    kw = dict(causal=causal, window=window, n_sink=n_sink, scale=scale)
    dq, dk, dv = _gpu_fwd_bwd(q, k, v, do, **kw)
    rq, rk, rv = oracle.attn_bwd(to64(q), to64(k), to64(v), to64(do), **kw)
    check_close("dQ", to64(dq), rq)
    check_close("dK", to64(dk), rk)
    check_close("dV", to64(dv), rv)


def test_tiny_workload():
    w = WORKLOADS["tiny_b1_h4_g2_s128"]
    _run_full(w.B, w.H, w.G, w.S)


@pytest.mark.parametrize("B,H,G,S", [
    (1, 2, 1, 1),
    (1, 2, 1, 127),
    (1, 2, 1, 129),
    (2, 4, 2, 300),
    (1, 3, 1, 256),     # R = 3
    (1, 2, 2, 384),     # H == G
    (1, 8, 1, 520),     # multi-query: dK/dV summed over 8 heads
])
def test_causal(B, H, G, S):
    _run_full(B, H, G, S)


@pytest.mark.parametrize("S", [64, 200, 513])
def test_full_attention(S):
    _run_full(1, 4, 2, S, causal=False)


@pytest.mark.parametrize("S,window,n_sink", [
    (700, 256, 64),
    (900, 100, 130),
    (640, 1, 0),
    (640, 200, 0),
    (500, 600, 5),
    (1000, 128, 128),
    (777, 129, 300),
    (300, 50, 1000),
])
def test_window_sinks(S, window, n_sink):
    _run_full(1, 4, 2, S, window=window, n_sink=n_sink)


def test_scale_not_default():
    """A non-default scale (logit std about 1.6) reaches dS, dQ and dK: the
    oracle at the stated tolerance."""
    _run_full(1, 4, 2, 300, scale=0.2)


def test_large_logits_against_rounding_model():
    """Scale 0.37 (logit std about 3).  There the method itself, with D taken on
    the bf16 O the forward hands over and bf16 dS operands, is farther than 2e-2
    from the exact gradients (tests/test_grad_precision.py pins that on the
    CPU), so the stated bound cannot apply.  The backward is checked against the
    float64 model of its own roundings fed the same O instead: within half a
    bf16 ulp of the output plus the fp32 noise of the scores and sums."""
    from bwd_rounding_model import model_bwd_group
    B, H, G, S, scale = 1, 4, 2, 300, 0.37
    q, k, v, do = make_inputs(B, H, G, S, seed=0, with_grad=True)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = gq.fwd(qd, kd, vd, scale=scale)
    dq, dk, dv = gq.bwd(qd, kd, vd, o, dod, lse, scale=scale)
    torch.cuda.synchronize()
    assert gq.gqa_attn_last_device_status() == gq.GQA_OK
    R = H // G
    for g in range(G):
        hs = slice(g * R, (g + 1) * R)
        m = model_bwd_group(to64(q[0, hs]), to64(k[0, g]), to64(v[0, g]), to64(do[0, hs]), scale,
                            o=to64(o[0, hs]), p_round="f16_rowscaled")
        for name, got, ref in zip(("dQ", "dK", "dV"), (dq[0, hs], dk[0, g], dv[0, g]), m):
            err = np.abs(to64(got) - ref)
            e = np.floor(np.log2(np.maximum(np.abs(ref), 1e-30)))
            assert (err <= 0.5 * np.exp2(e - 7) + 4e-3).all(), (name, g, float(err.max()))


def test_caller_workspace_and_null_workspace_agree():
    q, k, v, do = [t.cuda() for t in make_inputs(1, 4, 2, 333, seed=5, with_grad=True)]
    o, lse = gq.fwd(q, k, v)
    a = gq.bwd(q, k, v, o, do, lse)
    B, H, G, S, d = 1, 4, 2, 333, 64
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    rc = gq.gqa_attn_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, G, S, d, 1, 0, 0, 0.125,
                         None, 0, None)
    assert rc == gq.GQA_OK
    torch.cuda.synchronize()
    assert torch.equal(a[1], dk) and torch.equal(a[2], dv)
    assert (a[0].float() - dq.float()).abs().max().item() <= 2e-2


def test_bwd_workload_sampled_groups():
    """The full backward workload (bench launch), checked on two whole kv groups."""
    w = WORKLOADS["bwd_b4_h32_g8_s4096"]
    q, k, v, do = make_inputs(w.B, w.H, w.G, w.S, seed=0, with_grad=True)
    dq, dk, dv = _gpu_fwd_bwd(q, k, v, do)
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    R = w.H // w.G
    for b, g in [(0, 0), (w.B - 1, w.G - 1)]:
        rq, rk, rv = oracle.attn_bwd_group(to64(q[b:b + 1]), to64(k[b:b + 1]), to64(v[b:b + 1]),
                                           to64(do[b:b + 1]), 0, g)
        check_close(f"dK[b{b},g{g}]", to64(dk[b, g]), rk)
        check_close(f"dV[b{b},g{g}]", to64(dv[b, g]), rv)
        check_close(f"dQ[b{b},g{g}]", to64(dq[b, g * R:(g + 1) * R]), rq)


def test_wide_workload_bwd_groups():
    """B1 H128 G16 S8192: the backward of the benchmark's default step, checked
    on the first and last kv groups whole (dQ of their 8 heads, dK, dV)."""
    w = WORKLOADS["wide_b1_h128_g16_s8192"]
    q, k, v, do = make_inputs(w.B, w.H, w.G, w.S, seed=0, with_grad=True)
    dq, dk, dv = _gpu_fwd_bwd(q, k, v, do)
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    R = w.H // w.G
    for g in (0, w.G - 1):
        heads = slice(g * R, (g + 1) * R)
        rq, rk, rv = oracle.attn_bwd_group(to64(q[:, heads]), to64(k[:, g:g + 1]),
                                           to64(v[:, g:g + 1]), to64(do[:, heads]), 0, 0)
        check_close(f"dK[g{g}]", to64(dk[0, g]), rk)
        check_close(f"dV[g{g}]", to64(dv[0, g]), rv)
        check_close(f"dQ[g{g}]", to64(dq[0, heads]), rq)


def test_window_bwd_long_context_sampled():
    """Window + sink backward at S = 32768 (one kv group of the window workload's
    shape with fewer heads), checked on the whole group."""
    B, H, G, S, W, ns = 1, 4, 2, 32768, 4096, 128
    q, k, v, do = make_inputs(B, H, G, S, seed=1, with_grad=True)
    dq, dk, dv = _gpu_fwd_bwd(q, k, v, do, window=W, n_sink=ns)
    rq, rk, rv = oracle.attn_bwd_group(to64(q), to64(k), to64(v), to64(do), 0, 1,
                                       window=W, n_sink=ns)
    check_close("dK", to64(dk[0, 1]), rk)
    check_close("dV", to64(dv[0, 1]), rv)
    check_close("dQ", to64(dq[0, 2:4]), rq)


def test_window_workload_bwd_group():
    """B1 H128 G16 S32768, window 4096 + 128 sinks: the backward as the
    benchmark launches it (the 16 sink key tiles ahead of the one-kv-head
    batches), checked on the last kv group whole (dQ of its 8 heads, dK, dV)."""
    w = WORKLOADS["window_b1_h128_g16_s32768_w4096_sink128"]
    q, k, v, do = make_inputs(w.B, w.H, w.G, w.S, seed=0, with_grad=True)
    kw = dict(window=w.window, n_sink=w.n_sink)
    dq, dk, dv = _gpu_fwd_bwd(q, k, v, do, **kw)
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    R, g = w.H // w.G, w.G - 1
    heads = slice(g * R, (g + 1) * R)
    rq, rk, rv = oracle.attn_bwd_group(to64(q[:, heads]), to64(k[:, g:g + 1]), to64(v[:, g:g + 1]),
                                       to64(do[:, heads]), 0, 0, **kw)
    check_close("dK", to64(dk[0, g]), rk)
    check_close("dV", to64(dv[0, g]), rv)
    check_close("dQ", to64(dq[0, heads]), rq)


def test_model_workload_bwd_tail():
    """The model-spec mask (window 65536, 2048 sinks) at S = 204800: full
    forward and backward on the GPU, checked on the last kv group: dQ of the
    last 512 query rows (their window edge and the sinks are both in play) and
    dK, dV of the last 512 keys, every visible query of which is among those
    rows, so the oracle's restricted sums are complete there."""
    w = WORKLOADS["model_b1_h128_g16_s204800_w65536_sink2048"]
    q, k, v, do = make_inputs(w.B, w.H, w.G, w.S, seed=0, with_grad=True)
    kw = dict(window=w.window, n_sink=w.n_sink)
    dq, dk, dv = _gpu_fwd_bwd(q, k, v, do, **kw)
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    R, g, n = w.H // w.G, w.G - 1, 512
    i0 = w.S - n
    heads = slice(g * R, (g + 1) * R)
    rq, rk, rv = oracle.attn_bwd_group_rows(to64(q[:, heads]), to64(k[:, g:g + 1]),
                                            to64(v[:, g:g + 1]), to64(do[:, heads]), 0, 0,
                                            i0, w.S, **kw)
    check_close("dQ(last rows)", to64(dq[0, heads, i0:]), rq[:, i0:])
    check_close("dK(last keys)", to64(dk[0, g, i0:]), rk[i0:])
    check_close("dV(last keys)", to64(dv[0, g, i0:]), rv[i0:])


def test_uneven_cta_batches():
    """B4 H64 G4 S4096: 16 kv heads run in CTA batches of 5, 5 and 6 (the order of
    bwd_order.cuh).  Checked on a kv head of the first batch and one of the last:
    dQ of 256 middle rows (every key tile before them contributes, from many
    CTAs) and of the last 256 rows, dK and dV of the last 256 keys (all of their
    visible queries are among those rows)."""
    B, H, G, S = 4, 64, 4, 4096
    q, k, v, do = make_inputs(B, H, G, S, seed=5, with_grad=True)
    dq, dk, dv = _gpu_fwd_bwd(q, k, v, do)
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    R, n = H // G, 256
    for b, g in [(0, 1), (B - 1, G - 1)]:
        heads = slice(g * R, (g + 1) * R)
        args = (to64(q[b:b + 1, heads]), to64(k[b:b + 1, g:g + 1]), to64(v[b:b + 1, g:g + 1]),
                to64(do[b:b + 1, heads]), 0, 0)
        i0 = S // 2
        rq, _, _ = oracle.attn_bwd_group_rows(*args, i0, i0 + n)
        check_close(f"dQ(middle rows)[b{b},g{g}]", to64(dq[b, heads, i0:i0 + n]), rq[:, i0:i0 + n])
        i0 = S - n
        rq, rk, rv = oracle.attn_bwd_group_rows(*args, i0, S)
        check_close(f"dQ(last rows)[b{b},g{g}]", to64(dq[b, heads, i0:]), rq[:, i0:])
        check_close(f"dK(last keys)[b{b},g{g}]", to64(dk[b, g, i0:]), rk[i0:])
        check_close(f"dV(last keys)[b{b},g{g}]", to64(dv[b, g, i0:]), rv[i0:])


def test_repeat_dk_dv_deterministic():
    q, k, v, do = [t.cuda() for t in make_inputs(1, 8, 2, 700, seed=4, with_grad=True)]
    o, lse = gq.fwd(q, k, v, window=200, n_sink=50)
    a = gq.bwd(q, k, v, o, do, lse, window=200, n_sink=50)
    b = gq.bwd(q, k, v, o, do, lse, window=200, n_sink=50)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
