"""Precision of the backward's gradients before and after the bf16 output rounding.

The stated tolerance (max |err| 2e-2, mean |err| 2e-3 on dQ, dK, dV against the
float64 oracle) is checked here on the gradients as the kernels accumulate
them, before they are rounded to bf16: a test build of the library
(libgqa_attn_fp32grad.so, -DGQA_FP32_GRAD_OUT) writes dq, dk and dv as fp32.

The CPU tests pin the float64 model of the backward's own roundings
(bwd_rounding_model.py) to the oracle and record what it predicts: on the
stated workloads (scale 1/8) every gradient is well inside 2e-2 before the
output rounding; at a logit spread of about 3 (scale 0.37) the method itself,
with D taken on the bf16 O that the forward hands over and bf16 dS operands,
errs by about 0.03-0.04 even with exact P, so no tolerance of 2e-2 can hold
there for any backward that takes a bf16 O.  The GPU test at that scale
therefore checks the kernel against the model (the kernel adds no error of
its own) and the model against the oracle within the distance it predicts.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from causal_grouped_query_gqa_b300.inputs import WORKLOADS, make_inputs
from bwd_rounding_model import model_bwd_group
from parity_util import MAX_ABS, MEAN_ABS, check_close

# The 16-bit format of the P operand of dV += P^T dO in the CUDA backward.
KERNEL_P_OPERAND = "f16_rowscaled"


def _group(q, k, v, do, b, g):
    R = q.shape[1] // k.shape[1]
    f = lambda t: t.to(torch.float64).numpy()
    return (f(q[b, g * R:(g + 1) * R]), f(k[b, g]), f(v[b, g]), f(do[b, g * R:(g + 1) * R]))


def _err(a, b):
    e = np.abs(np.asarray(a) - np.asarray(b))
    return float(e.max()), float(e.mean())


# ------------------------------------------------------------- CPU: the model

def test_model_without_rounding_is_the_oracle():
    """With no rounding anywhere the model computes the method: it matches the
    oracle's backward to float64 precision (window and sinks included)."""
    q, k, v, do = make_inputs(1, 4, 2, 200, seed=3, with_grad=True)
    for kw in (dict(), dict(window=37, n_sink=5)):
        rq, rk, rv = oracle.attn_bwd_group(q.double().numpy(), k.double().numpy(),
                                           v.double().numpy(), do.double().numpy(), 0, 1, **kw)
        mq, mk, mv = model_bwd_group(*_group(q, k, v, do, 0, 1), 0.125, o_round="none",
                                     p_round="none", ds_round="none", **kw)
        for a, b in ((mq, rq), (mk, rk), (mv, rv)):
            assert _err(a, b)[0] < 1e-10


def test_model_stated_scale_within_tolerance():
    """Scale 1/8 (every stated workload): the kernel's roundings keep each
    gradient within 2e-2 / 2e-3 before the bf16 output rounding (one kv group
    of the 4x32x8x4096 backward workload)."""
    w = WORKLOADS["bwd_b4_h32_g8_s4096"]
    q, k, v, do = make_inputs(w.B, w.H, w.G, w.S, seed=0, with_grad=True)
    gq_, gk, gv, gdo = _group(q, k, v, do, 0, 0)
    rq, rk, rv = oracle.attn_bwd_group(gq_[None], gk[None, None], gv[None, None], gdo[None], 0, 0)
    mq, mk, mv = model_bwd_group(gq_, gk, gv, gdo, w.scale, p_round=KERNEL_P_OPERAND)
    for name, a, b in (("dQ", mq, rq), ("dK", mk, rk), ("dV", mv, rv)):
        mx, mean = _err(a, b)
        assert mx <= MAX_ABS and mean <= MEAN_ABS, (name, mx, mean)


def test_model_large_logits_floor():
    """Scale 0.37 (logit std about 3): with D from the bf16 O the method errs
    beyond 2e-2 in dQ or dK even when P and dS are not rounded at all, so the
    2e-2 bound is out of reach there for a backward fed a bf16 O."""
    q, k, v, do = make_inputs(1, 4, 2, 300, seed=0, with_grad=True)
    grp = _group(q, k, v, do, 0, 0)
    rq, rk, rv = oracle.attn_bwd_group(grp[0][None], grp[1][None, None], grp[2][None, None],
                                       grp[3][None], 0, 0, scale=0.37)
    mq, mk, _ = model_bwd_group(*grp, 0.37, p_round="none", ds_round="none")
    assert max(_err(mq, rq)[0], _err(mk, rk)[0]) > MAX_ABS
    # with an exact D, the bf16 dS operand alone already takes dQ / dK close to it
    mq2, mk2, _ = model_bwd_group(*grp, 0.37, o_round="none", p_round="none")
    assert max(_err(mq2, rq)[0], _err(mk2, rk)[0]) > 0.75 * MAX_ABS


# ------------------------------------------------- GPU: fp32 gradient outputs

@pytest.fixture(scope="module")
def fp32lib():
    from causal_grouped_query_gqa_b300 import build as gbuild
    lib = ctypes.CDLL(gbuild.build_fp32_grad())
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.gqa_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp]
    lib.gqa_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                 i, i, i, i, i, i, i, i, f, vp, sz, vp]
    lib.gqa_attn_bwd_workspace_size.argtypes = [i, i, i, i, i]
    lib.gqa_attn_bwd_workspace_size.restype = sz
    lib.gqa_attn_last_device_status.argtypes = [vp]
    return lib


def _fp32_grads(lib, q, k, v, do, *, causal=True, window=0, n_sink=0, scale=0.125):
    B, H, S, d = q.shape
    G = k.shape[1]
    q, k, v, do = (t.cuda() for t in (q, k, v, do))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    dq = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    dk = torch.empty(k.shape, dtype=torch.float32, device="cuda")
    dv = torch.empty(v.shape, dtype=torch.float32, device="cuda")
    ws = torch.empty(lib.gqa_attn_bwd_workspace_size(B, H, G, S, d), dtype=torch.uint8,
                     device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    p = lambda t: t.data_ptr()
    assert lib.gqa_attn_fwd(p(q), p(k), p(v), p(o), p(lse), B, H, G, S, d, int(causal), window,
                            n_sink, scale, st) == 0
    assert lib.gqa_attn_bwd(p(q), p(k), p(v), p(o), p(do), p(lse), p(dq), p(dk), p(dv), B, H, G,
                            S, d, int(causal), window, n_sink, scale, p(ws), ws.numel(), st) == 0
    assert lib.gqa_attn_last_device_status(st) == 0
    f = lambda t: t.to("cpu", torch.float64).numpy()
    _fp32_grads.last_o = f(o)
    return f(dq), f(dk), f(dv)


def _check_fp32(tag, got, ref):
    for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
        check_close(f"{name} fp32 {tag}", a, b, max_abs=MAX_ABS, mean_abs=MEAN_ABS, bf16_out=False)


@pytest.mark.gpu
def test_fp32_gradients_tiny(fp32lib):
    w = WORKLOADS["tiny_b1_h4_g2_s128"]
    q, k, v, do = make_inputs(w.B, w.H, w.G, w.S, seed=0, with_grad=True)
    got = _fp32_grads(fp32lib, q, k, v, do)
    f = lambda t: t.double().numpy()
    _check_fp32("tiny", got, oracle.attn_bwd(f(q), f(k), f(v), f(do)))


@pytest.mark.gpu
@pytest.mark.parametrize("S,window,n_sink,causal", [
    (300, 0, 0, True), (777, 129, 300, True), (513, 0, 0, False), (1000, 100, 130, True)])
def test_fp32_gradients_small_shapes(fp32lib, S, window, n_sink, causal):
    q, k, v, do = make_inputs(1, 6, 2, S, seed=S, with_grad=True)
    got = _fp32_grads(fp32lib, q, k, v, do, causal=causal, window=window, n_sink=n_sink)
    f = lambda t: t.double().numpy()
    _check_fp32(f"S{S}", got, oracle.attn_bwd(f(q), f(k), f(v), f(do), causal=causal,
                                              window=window, n_sink=n_sink))


@pytest.mark.gpu
@pytest.mark.parametrize("name,groups", [
    ("bwd_b4_h32_g8_s4096", [(0, 0), (3, 7)]),
    ("wide_b1_h128_g16_s8192", [(0, 0), (0, 15)]),
])
def test_fp32_gradients_workload_groups(fp32lib, name, groups):
    """The stated backward workload and the benchmark's default shape: whole
    kv groups (dQ of their R heads, dK, dV) at plain 2e-2 / 2e-3."""
    w = WORKLOADS[name]
    q, k, v, do = make_inputs(w.B, w.H, w.G, w.S, seed=0, with_grad=True)
    dq, dk, dv = _fp32_grads(fp32lib, q, k, v, do, scale=w.scale)
    R = w.H // w.G
    for b, g in groups:
        gq_, gk, gv, gdo = _group(q, k, v, do, b, g)
        ref = oracle.attn_bwd_group(gq_[None], gk[None, None], gv[None, None], gdo[None], 0, 0)
        _check_fp32(f"{name} b{b} g{g}", (dq[b, g * R:(g + 1) * R], dk[b, g], dv[b, g]), ref)


@pytest.mark.gpu
def test_fp32_gradients_long_window_group(fp32lib):
    """Window 4096 + 128 sinks at S = 32768, one whole kv group."""
    B, H, G, S, W, ns = 1, 4, 2, 32768, 4096, 128
    q, k, v, do = make_inputs(B, H, G, S, seed=1, with_grad=True)
    dq, dk, dv = _fp32_grads(fp32lib, q, k, v, do, window=W, n_sink=ns)
    gq_, gk, gv, gdo = _group(q, k, v, do, 0, 1)
    ref = oracle.attn_bwd_group(gq_[None], gk[None, None], gv[None, None], gdo[None], 0, 0,
                                window=W, n_sink=ns)
    _check_fp32("window", (dq[0, 2:4], dk[0, 1], dv[0, 1]), ref)


@pytest.mark.gpu
def test_fp32_gradients_large_logits(fp32lib):
    """Scale 0.37: the kernel's fp32 gradients equal the rounding model's, fed
    the O the forward actually handed over (within the fp32 noise of the scores
    and sums), and the model's distance from the oracle is the method's own
    (see test_model_large_logits_floor)."""
    q, k, v, do = make_inputs(1, 4, 2, 300, seed=0, with_grad=True)
    dq, dk, dv = _fp32_grads(fp32lib, q, k, v, do, scale=0.37)
    o = _fp32_grads.last_o
    for g in range(2):
        grp = _group(q, k, v, do, 0, g)
        mq, mk, mv = model_bwd_group(*grp, 0.37, p_round=KERNEL_P_OPERAND,
                                     o=o[0, 2 * g:2 * g + 2])
        got = (dq[0, 2 * g:2 * g + 2], dk[0, g], dv[0, g])
        for name, a, b in zip(("dQ", "dK", "dV"), got, (mq, mk, mv)):
            mx, mean = _err(a, b)
            assert mx <= 4e-3 and mean <= 2e-4, (name, g, mx, mean)
        ref = oracle.attn_bwd_group(grp[0][None], grp[1][None, None], grp[2][None, None],
                                    grp[3][None], 0, 0, scale=0.37)
        for name, a, m, r in zip(("dQ", "dK", "dV"), got, (mq, mk, mv), ref):
            # the kernel is no farther from the oracle than the model, up to fp32 noise
            assert _err(a, r)[0] <= _err(m, r)[0] + 4e-3, name
