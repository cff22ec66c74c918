"""Pins for the float64 oracle, none of which asks the oracle to check itself.

Each test ties the oracle to something fixed outside it: the worked example of
"nx_f32_gqa_gate.nx source" (tests T0-T4, by closed form and by the page's own
central differences), hand-enumerated mask sets, closed forms for equal scores,
float64 finite differences, and torch's CPU scaled-dot-product attention with
autograd as an independent library computation.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _p5_tensors():
    ex = _load("p5_worked_example.json")
    Q = np.array(ex["Q"])[None, None]
    K = np.array(ex["K"])[None, None]
    V = np.array(ex["V"])[None, None]
    return ex, Q, K, V


# ---------------------------------------------------------------- page 5 ---

def test_p5_forward_closed_form():
    """T0/T1: attn[0] = [1], out[0] = V[0]; attn[1] = softmax([0, 1/sqrt2])."""
    _, Q, K, V = _p5_tensors()
    o, lse = oracle.attn_fwd(Q, K, V, causal=True, scale=1 / math.sqrt(2))
    a1 = math.exp(1 / math.sqrt(2))
    a = np.array([1.0, a1]) / (1.0 + a1)             # attn[1], sums to 1 (T0)
    assert abs(a.sum() - 1.0) < 1e-15
    np.testing.assert_allclose(o[0, 0, 0], [1.0, 2.0], rtol=0, atol=1e-14)        # T1
    np.testing.assert_allclose(o[0, 0, 1], a[0] * np.array([1, 2]) + a[1] * np.array([3, 4]),
                               rtol=0, atol=1e-14)
    np.testing.assert_allclose(o[0, 0, 1], [2.339523, 3.339523], atol=1e-6)
    # row 0 sees only key 0: LSE_0 = s_00 = (Q0.K0)/sqrt2; row 1: ln(e^0 + e^(1/sqrt2))
    np.testing.assert_allclose(lse[0, 0], [1 / math.sqrt(2), math.log(1.0 + a1)], atol=1e-14)


def test_p5_gradients_closed_form_and_page_gradcheck():
    """T3/T4: L = out[1][0]; dL/dV[j][0] = attn[1][j]; dL/dQ[1] = +-sqrt2*a0*a1."""
    ex, Q, K, V = _p5_tensors()
    scale = 1 / math.sqrt(2)
    dO = np.zeros_like(Q)
    dO[0, 0, 1, 0] = 1.0                                   # L = out[1][0]
    dq, dk, dv = oracle.attn_bwd(Q, K, V, dO, causal=True, scale=scale)
    a1 = math.exp(1 / math.sqrt(2))
    a0, a1 = 1 / (1 + a1), a1 / (1 + a1)
    np.testing.assert_allclose(dv[0, 0, :, 0], [a0, a1], atol=1e-14)            # T3
    np.testing.assert_allclose(dv[0, 0, :, 1], [0, 0], atol=1e-14)
    s = math.sqrt(2) * a0 * a1
    np.testing.assert_allclose(dq[0, 0, 1], [-s, s], atol=1e-14)                # T4
    np.testing.assert_allclose(dq[0, 0, 1], [-0.312797, 0.312797], atol=1e-6)
    np.testing.assert_allclose(dq[0, 0, 0], [0, 0], atol=1e-14)   # row 0: one key, softmax flat

    # The page's own check: central differences with h = 0.01, tolerance 0.03.
    h, tol = ex["h"], ex["tol"]

    def L(Qx, Vx):
        return oracle.attn_fwd(Qx, K, Vx, causal=True, scale=scale)[0][0, 0, 1, 0]

    Vp, Vm = V.copy(), V.copy()
    Vp[0, 0, 0, 0] += h
    Vm[0, 0, 0, 0] -= h
    assert abs((L(Q, Vp) - L(Q, Vm)) / (2 * h) - dv[0, 0, 0, 0]) <= tol
    Qp, Qm = Q.copy(), Q.copy()
    Qp[0, 0, 1, 0] += h
    Qm[0, 0, 1, 0] -= h
    assert abs((L(Qp, V) - L(Qm, V)) / (2 * h) - dq[0, 0, 1, 0]) <= tol


def test_p5_gqa_head_map():
    """T2: H=4, G=2 -> heads {0,1} read kv0 and {2,3} read kv1."""
    rng = np.random.default_rng(1)
    S, d = 6, 4
    q = rng.standard_normal((1, 4, S, d))
    k = rng.standard_normal((1, 2, S, d))
    v = rng.standard_normal((1, 2, S, d))
    o, lse = oracle.attn_fwd(q, k, v, causal=True)
    for h, g in [(0, 0), (1, 0), (2, 1), (3, 1)]:
        oh, lh = oracle.attn_fwd(q[:, h:h + 1], k[:, g:g + 1], v[:, g:g + 1], causal=True)
        np.testing.assert_array_equal(o[0, h], oh[0, 0])
        np.testing.assert_array_equal(lse[0, h], lh[0, 0])
        other = 1 - g
        oo, _ = oracle.attn_fwd(q[:, h:h + 1], k[:, other:other + 1], v[:, other:other + 1])
        assert np.abs(o[0, h] - oo[0, 0]).max() > 1e-3


def test_causal_row0_is_v0():
    """T1 for every head of a GQA problem: out[b,h,0] == v[b,h/(H/G),0]."""
    rng = np.random.default_rng(2)
    B, H, G, S, d = 2, 6, 3, 7, 5
    q = rng.standard_normal((B, H, S, d))
    k = rng.standard_normal((B, G, S, d))
    v = rng.standard_normal((B, G, S, d))
    o, _ = oracle.attn_fwd(q, k, v, causal=True, window=3, n_sink=1)
    for b in range(B):
        for h in range(H):
            np.testing.assert_allclose(o[b, h, 0], v[b, h // (H // G), 0], atol=1e-15)


# ------------------------------------------------------------------ mask ---

def _equal_score_check(S, causal, window, n_sink, vis_sets):
    """q = 0 makes every score 0, so each row averages V over its visible keys.

    With V = identity rows, out[i, j] = 1/|vis(i)| on the visible set and 0 off
    it, and LSE_i = ln |vis(i)|: the mask and the normalisation in closed form.
    """
    d = 64
    assert S <= d
    q = np.zeros((1, 1, S, d))
    k = np.random.default_rng(3).standard_normal((1, 1, S, d))
    v = np.zeros((1, 1, S, d))
    v[0, 0, np.arange(S), np.arange(S)] = 1.0
    o, lse = oracle.attn_fwd(q, k, v, causal=causal, window=window, n_sink=n_sink)
    for i in range(S):
        want = np.zeros(d)
        want[list(vis_sets[i])] = 1.0 / len(vis_sets[i])
        np.testing.assert_allclose(o[0, 0, i], want, atol=1e-15, err_msg=f"row {i}")
        assert abs(o[0, 0, i].sum() - 1.0) < 1e-14                 # T0
        assert abs(lse[0, 0, i] - math.log(len(vis_sets[i]))) < 1e-14


@pytest.mark.parametrize("fixture", ["window_sink_mask_w4_s2.json", "window_sink_mask_w1_s5.json"])
def test_window_sink_mask_literal_sets(fixture):
    m = _load(fixture)
    _equal_score_check(m["S"], True, m["window"], m["n_sink"], m["visible"])
    for i, row in enumerate(m["visible"]):
        for j in range(m["S"]):
            assert oracle.visible(i, j, causal=True, window=m["window"],
                                  n_sink=m["n_sink"]) == (j in row)


def test_causal_and_full_masks_literal():
    S = 5
    _equal_score_check(S, True, 0, 0, [list(range(i + 1)) for i in range(S)])
    _equal_score_check(S, False, 0, 0, [list(range(S)) for _ in range(S)])
    # window >= S is plain causal; sinks without a window are ignored
    _equal_score_check(S, True, S, 3, [list(range(i + 1)) for i in range(S)])
    _equal_score_check(S, True, 0, 3, [list(range(i + 1)) for i in range(S)])
    # no sinks: pure window of 2
    _equal_score_check(S, True, 2, 0, [[0], [0, 1], [1, 2], [2, 3], [3, 4]])
    # more sinks than tokens: plain causal
    _equal_score_check(S, True, 1, 9, [list(range(i + 1)) for i in range(S)])


def test_equal_keys_closed_form_backward():
    """All keys equal -> scores equal in a row -> P uniform on the visible set,
    dQ = scale * sum_j dS_ij k = 0 (dS sums to zero), dK_j = scale*sum_i dS_ij q_i
    and dV_j = sum_{h,i} dO_i / |vis(i)|."""
    rng = np.random.default_rng(4)
    B, H, G, S, d = 1, 4, 2, 9, 3
    W, ns = 3, 2
    q = rng.standard_normal((B, H, S, d))
    kvec = rng.standard_normal(d)
    k = np.broadcast_to(kvec, (B, G, S, d)).copy()
    v = rng.standard_normal((B, G, S, d))
    dO = rng.standard_normal((B, H, S, d))
    dq, dk, dv = oracle.attn_bwd(q, k, v, dO, causal=True, window=W, n_sink=ns)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)
    vis = [[j for j in range(S) if (j <= i and (j > i - W or j < ns))] for i in range(S)]
    R = H // G
    want_dv = np.zeros((G, S, d))
    want_dk = np.zeros((G, S, d))
    for h in range(H):
        g = h // R
        for i in range(S):
            n = len(vis[i])
            # dP_ij = dO_i . v_j, D_i = mean over visible j, dS_ij = (dP_ij - D_i)/n
            dp = {j: dO[0, h, i] @ v[0, g, j] for j in vis[i]}
            D = sum(dp.values()) / n
            for j in vis[i]:
                want_dv[g, j] += dO[0, h, i] / n
                want_dk[g, j] += (dp[j] - D) / n * q[0, h, i] / math.sqrt(d)
    np.testing.assert_allclose(dv[0], want_dv, atol=1e-13)
    np.testing.assert_allclose(dk[0], want_dk, atol=1e-13)


# --------------------------------------------------- independent library ---

def _torch_reference(q, k, v, causal, window, n_sink, scale, dO):
    """torch CPU float64 SDPA (math path) with an explicit boolean mask and the
    kv heads repeated per query head; gradients by autograd."""
    B, H, S, d = q.shape
    G = k.shape[1]
    i = torch.arange(S)[:, None]
    j = torch.arange(S)[None, :]
    mask = torch.ones(S, S, dtype=torch.bool)
    if causal:
        mask &= j <= i
        if window > 0:
            mask &= (j > i - window) | (j < n_sink)
    qt = torch.tensor(q, requires_grad=True)
    kt = torch.tensor(k, requires_grad=True)
    vt = torch.tensor(v, requires_grad=True)
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt.repeat_interleave(H // G, dim=1), vt.repeat_interleave(H // G, dim=1),
        attn_mask=mask, scale=scale)
    o.backward(torch.tensor(dO))
    s = torch.einsum("bhid,bhjd->bhij", qt.detach(), kt.detach().repeat_interleave(H // G, 1))
    lse = torch.logsumexp((s * scale).masked_fill(~mask, float("-inf")), dim=-1)
    return (o.detach().numpy(), lse.numpy(), qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy())


@pytest.mark.parametrize("B,H,G,S,d,causal,window,n_sink", [
    (1, 4, 2, 16, 8, True, 0, 0),
    (2, 6, 2, 13, 5, True, 4, 2),
    (1, 3, 3, 11, 4, True, 3, 0),
    (1, 4, 1, 9, 6, False, 0, 0),
    (1, 2, 1, 10, 4, True, 1, 3),
    (1, 8, 2, 21, 7, True, 6, 6),
])
def test_against_torch_sdpa_float64(B, H, G, S, d, causal, window, n_sink):
    rng = np.random.default_rng(5 + S)
    q = rng.standard_normal((B, H, S, d))
    k = rng.standard_normal((B, G, S, d))
    v = rng.standard_normal((B, G, S, d))
    dO = rng.standard_normal((B, H, S, d))
    scale = 0.37
    o, lse = oracle.attn_fwd(q, k, v, causal=causal, window=window, n_sink=n_sink, scale=scale)
    dq, dk, dv = oracle.attn_bwd(q, k, v, dO, causal=causal, window=window, n_sink=n_sink,
                                 scale=scale)
    to, tl, tdq, tdk, tdv = _torch_reference(q, k, v, causal, window, n_sink, scale, dO)
    np.testing.assert_allclose(o, to, atol=1e-12)
    np.testing.assert_allclose(lse, tl, atol=1e-12)
    np.testing.assert_allclose(dq, tdq, atol=1e-12)
    np.testing.assert_allclose(dk, tdk, atol=1e-12)
    np.testing.assert_allclose(dv, tdv, atol=1e-12)


def test_finite_differences_float64():
    """Central differences (h = 1e-6) of L = sum(O * W) against the oracle's
    analytic dq, dk, dv on a tiny GQA window/sink problem."""
    rng = np.random.default_rng(6)
    B, H, G, S, d = 1, 2, 1, 6, 3
    kw = dict(causal=True, window=3, n_sink=1, scale=0.7)
    q = rng.standard_normal((B, H, S, d))
    k = rng.standard_normal((B, G, S, d))
    v = rng.standard_normal((B, G, S, d))
    W = rng.standard_normal((B, H, S, d))
    dq, dk, dv = oracle.attn_bwd(q, k, v, W, **kw)

    def L(q, k, v):
        return float((oracle.attn_fwd(q, k, v, **kw)[0] * W).sum())

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name], args_m[name] = xp, xm
            fd[idx] = (L(**args_p) - L(**args_m)) / (2 * h)
        np.testing.assert_allclose(g, fd, atol=1e-7, err_msg=name)


def test_rows_and_group_entry_points_match_full():
    rng = np.random.default_rng(7)
    B, H, G, S, d = 2, 4, 2, 10, 4
    kw = dict(causal=True, window=4, n_sink=2)
    q = rng.standard_normal((B, H, S, d))
    k = rng.standard_normal((B, G, S, d))
    v = rng.standard_normal((B, G, S, d))
    dO = rng.standard_normal((B, H, S, d))
    o, lse = oracle.attn_fwd(q, k, v, **kw)
    rows = [(1, 3, 9), (0, 0, 0), (1, 2, 5)]
    orow, lrow = oracle.attn_fwd_rows(q, k, v, rows, **kw)
    for t, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(orow[t], o[b, h, i])
        assert lrow[t] == lse[b, h, i]
    dq, dk, dv = oracle.attn_bwd(q, k, v, dO, **kw)
    gq, gk, gv = oracle.attn_bwd_group(q, k, v, dO, 1, 1, **kw)
    np.testing.assert_allclose(gq, dq[1, 2:4], atol=1e-15)
    np.testing.assert_allclose(gk, dk[1, 1], atol=1e-15)
    np.testing.assert_allclose(gv, dv[1, 1], atol=1e-15)


def test_row_range_backward_sums_to_group():
    """Row ranges partition the group's backward: dq rows match, dk/dv add up."""
    rng = np.random.default_rng(8)
    B, H, G, S, d = 1, 4, 2, 12, 3
    kw = dict(causal=True, window=5, n_sink=2)
    q, dO = rng.standard_normal((B, H, S, d)), rng.standard_normal((B, H, S, d))
    k, v = rng.standard_normal((B, G, S, d)), rng.standard_normal((B, G, S, d))
    gq_, gk, gv = oracle.attn_bwd_group(q, k, v, dO, 0, 1, **kw)
    a = oracle.attn_bwd_group_rows(q, k, v, dO, 0, 1, 0, 7, **kw)
    c = oracle.attn_bwd_group_rows(q, k, v, dO, 0, 1, 7, S, **kw)
    np.testing.assert_allclose(a[1] + c[1], gk, atol=1e-14)
    np.testing.assert_allclose(a[2] + c[2], gv, atol=1e-14)
    np.testing.assert_allclose(a[0][:, :7], gq_[:, :7], atol=1e-15)
    np.testing.assert_allclose(c[0][:, 7:], gq_[:, 7:], atol=1e-15)
    assert oracle.num_threads() >= 1
