"""GPU forward vs the float64 oracle, element by element, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import causal_grouped_query_gqa_b300 as gq
from causal_grouped_query_gqa_b300.inputs import WORKLOADS, make_inputs
from parity_util import LSE_ABS, check_close, sample_rows, to64

pytestmark = pytest.mark.gpu


def _run_full(B, H, G, S, causal=True, window=0, n_sink=0, seed=0, scale=None,
              score_bound=None):
    q, k, v = make_inputs(B, H, G, S, seed=seed)
    o, lse = gq.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, window=window, n_sink=n_sink,
                    scale=scale, score_bound=score_bound)
    torch.cuda.synchronize()
    assert gq.gqa_attn_last_device_status() == gq.GQA_OK
    ro, rl = oracle.attn_fwd(to64(q), to64(k), to64(v), causal=causal, window=window,
                             n_sink=n_sink, scale=scale)
    check_close("O", to64(o), ro)
    check_close("LSE", to64(lse), rl, max_abs=LSE_ABS, mean_abs=None, bf16_out=False)


@pytest.mark.parametrize("B,H,G,S", [
    (1, 4, 2, 128),      # the tiny workload
    (1, 4, 2, 1),        # one token
    (1, 2, 1, 127),      # one partial tile
    (1, 2, 1, 129),      # a full tile and a 1-row tail
    (2, 4, 2, 300),      # several tiles and a ragged tail
    (1, 3, 1, 256),      # odd heads per kv head: the last pair has one head
    (1, 6, 2, 200),      # R = 3
    (1, 2, 2, 384),      # H == G (plain multi-head)
    (1, 8, 1, 520),      # R = 8, multi-query
])
@pytest.mark.parametrize("score_bound", [False, True], ids=["plain", "bound"])
def test_causal(B, H, G, S, score_bound):
    _run_full(B, H, G, S, score_bound=score_bound)


@pytest.mark.parametrize("S", [64, 200, 513])
def test_full_attention(S):
    _run_full(1, 4, 2, S, causal=False)


@pytest.mark.parametrize("S,window,n_sink", [
    (700, 256, 64),     # sink tile + window tiles
    (900, 100, 130),    # more sinks than the window, window inside a tile
    (640, 1, 0),        # each row sees only itself
    (640, 200, 0),      # pure window
    (500, 600, 5),      # window longer than the sequence: plain causal
    (1000, 128, 128),   # tile-aligned window and sinks
    (777, 129, 300),    # sinks spanning three tiles
    (300, 50, 1000),    # more sinks than keys: every key is a sink, plain causal
])
@pytest.mark.parametrize("score_bound", [False, True], ids=["plain", "bound"])
def test_window_sinks(S, window, n_sink, score_bound):
    _run_full(1, 4, 2, S, window=window, n_sink=n_sink, score_bound=score_bound)


@pytest.mark.parametrize("score_bound", [False, True], ids=["plain", "bound"])
def test_scale_not_default(score_bound):
    _run_full(1, 4, 2, 300, scale=0.37, score_bound=score_bound)


@pytest.mark.parametrize("B,H,G,S,window,n_sink", [
    (4, 6, 2, 2048, 0, 0),       # 256 units: each CTA of the persistent grid walks
                                 # several, two-head and one-head pairs mixed (R = 3)
    (2, 12, 4, 1536, 300, 70),   # the same with a window and sinks (192 units)
    (3, 16, 2, 1100, 0, 0),      # R = 8, ragged tail, 216 units
])
@pytest.mark.parametrize("score_bound", [False, True], ids=["plain", "bound"])
def test_persistent_grid_many_units(B, H, G, S, window, n_sink, score_bound):
    """More work units than SMs, so every CTA carries its barrier phases, Q
    buffers and O accumulators from one unit to the next."""
    _run_full(B, H, G, S, window=window, n_sink=n_sink, score_bound=score_bound)


def test_gqa_workload_full():
    w = WORKLOADS["gqa_b2_h32_g8_s2048"]
    _run_full(w.B, w.H, w.G, w.S)


def _run_sampled(w, n_rows=48, extra=(), groups=(), score_bound=None):
    """Full-size launch (the benchmark's), checked on whole kv groups (every
    row of their R query heads), on sampled rows of the other heads, and on
    properties that hold at any size."""
    q, k, v = make_inputs(w.B, w.H, w.G, w.S, seed=0)
    o, lse = gq.fwd(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, window=w.window,
                    n_sink=w.n_sink, scale=w.scale, score_bound=score_bound)
    torch.cuda.synchronize()
    assert gq.gqa_attn_last_device_status() == gq.GQA_OK
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    # T1 at full size: row 0 of every head is exactly v[g, 0]
    R = w.H // w.G
    v_rep = v.cuda().repeat_interleave(R, dim=1)
    assert torch.equal(o[:, :, 0], v_rep[:, :, 0])
    mask = dict(causal=w.causal, window=w.window, n_sink=w.n_sink, scale=w.scale)
    for b, g in groups:
        heads = slice(g * R, (g + 1) * R)
        ro, rl = oracle.attn_fwd(to64(q[b:b + 1, heads]), to64(k[b:b + 1, g:g + 1]),
                                 to64(v[b:b + 1, g:g + 1]), **mask)
        check_close(f"O[b{b},g{g}]", to64(o[b:b + 1, heads]), ro)
        check_close(f"LSE[b{b},g{g}]", to64(lse[b:b + 1, heads]), rl, max_abs=LSE_ABS,
                    mean_abs=None, bf16_out=False)
    rows = sample_rows(w.B, w.H, w.S, n_rows, extra=[(0, w.H - 1, w.S - 1), *extra])
    got_o = np.stack([to64(o[b, h, i]) for b, h, i in rows])
    got_l = np.array([float(lse[b, h, i]) for b, h, i in rows])
    ref_o = np.zeros_like(got_o)
    ref_l = np.zeros_like(got_l)
    by_head = {}
    for t, (b, h, i) in enumerate(rows):
        by_head.setdefault((b, h), []).append((t, i))
    for (b, h), items in by_head.items():
        g = h // R
        qs = to64(q[b:b + 1, h:h + 1])
        ks = to64(k[b:b + 1, g:g + 1])
        vs = to64(v[b:b + 1, g:g + 1])
        ro, rl = oracle.attn_fwd_rows(qs, ks, vs, [(0, 0, i) for _, i in items], **mask)
        for (t, _), a, c in zip(items, ro, rl):
            ref_o[t] = a
            ref_l[t] = c
    check_close("O(sampled)", got_o, ref_o)
    check_close("LSE(sampled)", got_l, ref_l, max_abs=LSE_ABS, mean_abs=None, bf16_out=False)


@pytest.mark.parametrize("score_bound", [False, True], ids=["plain", "bound"])
def test_wide_workload_groups(score_bound):
    """B1 H128 G16 S8192 (the benchmark's forward): the first and last kv
    groups whole (8 heads x 8192 rows each), through both forward paths."""
    w = WORKLOADS["wide_b1_h128_g16_s8192"]
    _run_sampled(w, groups=[(0, 0), (0, w.G - 1)], score_bound=score_bound)


def test_window_workload_group():
    """B1 H128 G16 S32768, window 4096 + 128 sinks: the last kv group whole
    (8 heads x 32768 rows), plus sampled rows of the others."""
    w = WORKLOADS["window_b1_h128_g16_s32768_w4096_sink128"]
    _run_sampled(w, groups=[(0, w.G - 1)])


def test_model_workload_sampled():
    """The model-spec mask at S = 204800: rows around the window edge (65536)
    and the sink boundary, plus the sampled ones."""
    w = WORKLOADS["model_b1_h128_g16_s204800_w65536_sink2048"]
    edges = [w.n_sink - 1, w.n_sink, w.window - 1, w.window, w.window + 1,
             w.window + w.n_sink - 1, w.window + w.n_sink, w.S - 1]
    _run_sampled(w, extra=[(0, (7 * t) % w.H, i) for t, i in enumerate(edges)])


def test_repeat_is_deterministic():
    q, k, v = make_inputs(1, 8, 2, 1000, seed=3)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = gq.fwd(q, k, v, window=300, n_sink=17)
    o2, l2 = gq.fwd(q, k, v, window=300, n_sink=17)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ---------------------------------------------------------------- score bound
# gqa_attn_fwd_ws (gq.fwd with score_bound=True, and gq.fwd's default on large
# problems): a key-norm pre-pass, then the forward kernel in which a query head
# whose 128 rows' score bounds U_i = |q_i| max_j |k_j| scale log2(e) are all
# <= 64 runs its unit against the fixed reference U_i - 32 without row maxima.
# The tests above cover that path on their inputs (the "bound" cases); these pin
# the pre-pass, the plain entry point and the heads that keep the exact step.

def _oracle_check(q, k, v, o, lse, **mask):
    ro, rl = oracle.attn_fwd(to64(q), to64(k), to64(v), **mask)
    check_close("O", to64(o), ro)
    check_close("LSE", to64(lse), rl, max_abs=LSE_ABS, mean_abs=None, bf16_out=False)


@pytest.mark.parametrize("S", [777, 20, 4100])
def test_key_norm_prepass_record(S):
    """The workspace holds, per kv head, 32 partial maxima: each the largest
    |k_j|^2 of its slice of ceil(S / 32) keys, 0 for an empty slice (float64
    reference from the same bf16 keys)."""
    B, H, G, P = 2, 8, 4, 32
    q, k, v = make_inputs(B, H, G, S, seed=5)
    ws = torch.full((gq.gqa_attn_fwd_workspace_size(B, H, G, S, 64),), 0xff, dtype=torch.uint8,
                    device="cuda")
    gq.fwd(q.cuda(), k.cuda(), v.cuda(), workspace=ws, score_bound=True)
    torch.cuda.synchronize()
    rec = ws.view(torch.float32).view(B * G, P).cpu().numpy().astype(np.float64)
    ref = (to64(k) ** 2).sum(-1).reshape(B * G, S)
    per = -(-S // P)
    parts = np.array([[ref[bg, p * per:(p + 1) * per].max() if p * per < S else 0.0
                       for p in range(P)] for bg in range(B * G)])
    np.testing.assert_allclose(rec, parts, rtol=1e-5)


@pytest.mark.parametrize("window,n_sink", [(0, 0), (200, 33)])
def test_plain_entry_point(window, n_sink):
    """gqa_attn_fwd (one launch, the online maximum everywhere) against the
    oracle and against the score-bound entry point."""
    B, H, G, S = 2, 4, 2, 700
    q, k, v = [t.cuda() for t in make_inputs(B, H, G, S, seed=7)]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    assert gq.gqa_attn_fwd(q, k, v, o, lse, B, H, G, S, 64, 1, window, n_sink, 0.125) == gq.GQA_OK
    o2, l2 = gq.fwd(q, k, v, window=window, n_sink=n_sink, score_bound=True)
    torch.cuda.synchronize()
    assert gq.gqa_attn_last_device_status() == gq.GQA_OK
    _oracle_check(q, k, v, o, lse, window=window, n_sink=n_sink)
    check_close("O(ws vs plain)", to64(o2), to64(o))
    check_close("LSE(ws vs plain)", to64(l2), to64(lse), max_abs=LSE_ABS, mean_abs=None,
                bf16_out=False)


def test_score_bound_mixed_warps():
    """Rows 0..31 of every 128-row block have 8x larger queries (bound > 64):
    the other warps of the same heads would qualify, and the head's vote sends
    all four warps down the exact step together."""
    B, H, G, S = 1, 4, 2, 1100
    q, k, v = make_inputs(B, H, G, S, seed=11)
    q[:, :, torch.arange(S) % 128 < 32] *= 8  # exact in bf16
    o, lse = gq.fwd(q.cuda(), k.cuda(), v.cuda(), score_bound=True)
    torch.cuda.synchronize()
    assert gq.gqa_attn_last_device_status() == gq.GQA_OK
    _oracle_check(q, k, v, o, lse)


@pytest.mark.parametrize("window,n_sink", [(0, 0), (300, 70)])
def test_score_bound_loose_everywhere(window, n_sink):
    """One key per kv head with 8x the norm makes every row's bound exceed 64:
    the whole forward keeps the exact step (large scores, peaked rows)."""
    B, H, G, S = 1, 4, 2, 900
    q, k, v = make_inputs(B, H, G, S, seed=13)
    k[:, :, S // 3] *= 8  # exact in bf16
    o, lse = gq.fwd(q.cuda(), k.cuda(), v.cuda(), window=window, n_sink=n_sink,
                    score_bound=True)
    torch.cuda.synchronize()
    assert gq.gqa_attn_last_device_status() == gq.GQA_OK
    _oracle_check(q, k, v, o, lse, window=window, n_sink=n_sink)


def test_score_bound_growing_keys():
    """Key norms growing 1x..4x along the sequence: bounds near the 64 limit
    (some warps on each side) and row maxima that keep rising after the first
    tile, which the fixed reference must absorb."""
    B, H, G, S = 1, 2, 1, 1024
    q, k, v = make_inputs(B, H, G, S, seed=17)
    ramp = 1.0 + 3.0 * torch.arange(S, dtype=torch.float32) / S
    k = (k.float() * ramp[None, None, :, None]).to(torch.bfloat16)
    o, lse = gq.fwd(q.cuda(), k.cuda(), v.cuda(), score_bound=True)
    torch.cuda.synchronize()
    assert gq.gqa_attn_last_device_status() == gq.GQA_OK
    _oracle_check(q, k, v, o, lse)


def test_score_bound_tiny_queries():
    """Queries near zero: the bound is tiny, the reference about -32, and every
    term close to 2^32 (uniform weights); O is the mean of the visible values."""
    B, H, G, S = 1, 2, 1, 600
    q, k, v = make_inputs(B, H, G, S, seed=19)
    q = (q.float() * 2.0 ** -20).to(torch.bfloat16)
    o, lse = gq.fwd(q.cuda(), k.cuda(), v.cuda(), score_bound=True)
    torch.cuda.synchronize()
    assert gq.gqa_attn_last_device_status() == gq.GQA_OK
    _oracle_check(q, k, v, o, lse)


@pytest.mark.parametrize("window,n_sink", [(0, 0), (300, 70)])
def test_score_bound_persistent_varying_norms(window, n_sink):
    """R = 3 (every other unit has one head) and more units than SMs, with the
    queries of every other 128-row block scaled 8x: the bound decisions differ
    from unit to unit, so each head must read its own unit's Q tile and record
    (one Q barrier per head; a phase left over from an earlier unit must not
    pass for the current one)."""
    B, H, G, S = 4, 6, 2, 2048
    q, k, v = make_inputs(B, H, G, S, seed=23)
    q[:, :, (torch.arange(S) // 128) % 2 == 0] *= 8  # exact in bf16
    o, lse = gq.fwd(q.cuda(), k.cuda(), v.cuda(), window=window, n_sink=n_sink, score_bound=True)
    torch.cuda.synchronize()
    assert gq.gqa_attn_last_device_status() == gq.GQA_OK
    _oracle_check(q, k, v, o, lse, window=window, n_sink=n_sink)
