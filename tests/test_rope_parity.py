"""GPU forward with YaRN rotary embeddings (gqa_attn_fwd_yarn) vs the float64
oracle, through the C ABI.

The oracle rotates q and k exactly (YaRN frequencies and temperature, YaRN
paper section 3), rounds the rotated tensors once to bf16 -- what a bf16 model
hands to its attention -- and attends in float64.  Both modes of the library
are checked: q and k rotated in a pre-pass into its workspace (the forward
then runs on them), and the fused mode, where the forward kernel rotates each
query tile in shared memory as it lands."""
import numpy as np
import pytest
import torch

import oracle
import causal_grouped_query_gqa_b300 as gq
from causal_grouped_query_gqa_b300.inputs import WORKLOADS, make_inputs
from parity_util import LSE_ABS, check_close, to64

pytestmark = pytest.mark.gpu

DEFAULT = dict(base=10000.0, factor=32.0, orig_ctx=6400, alpha=1.0, beta=32.0)


MODES = pytest.mark.parametrize("mode", [0, 1], ids=["prepass", "fused"])


def _gpu(q, k, v, rope, score_bound=None, mode=0, **mask):
    o, lse = gq.fwd_yarn(q.cuda(), k.cuda(), v.cuda(), rope_base=rope["base"],
                         rope_factor=rope["factor"], rope_orig_ctx=rope["orig_ctx"],
                         rope_alpha=rope["alpha"], rope_beta=rope["beta"],
                         score_bound=score_bound, rope_mode=mode, **mask)
    torch.cuda.synchronize()
    assert gq.gqa_attn_last_device_status() == gq.GQA_OK
    return o, lse


@pytest.mark.parametrize("B,H,G,S,causal,window,n_sink", [
    (1, 4, 2, 128, True, 0, 0),
    (2, 4, 2, 300, True, 0, 0),
    (1, 6, 2, 777, True, 129, 300),
    (1, 4, 2, 513, False, 0, 0),
    (1, 8, 1, 520, True, 0, 0),
    (4, 6, 2, 2048, True, 0, 0),      # more units than SMs: rotations carried across units
])
@pytest.mark.parametrize("score_bound", [False, True], ids=["plain", "bound"])
@MODES
def test_yarn_forward(B, H, G, S, causal, window, n_sink, score_bound, mode):
    q, k, v = make_inputs(B, H, G, S, seed=S)
    mask = dict(causal=causal, window=window, n_sink=n_sink)
    o, lse = _gpu(q, k, v, DEFAULT, score_bound=score_bound, mode=mode, **mask)
    ro, rl = oracle.attn_fwd_yarn(to64(q), to64(k), to64(v), **DEFAULT, **mask)
    check_close("O", to64(o), ro)
    check_close("LSE", to64(lse), rl, max_abs=LSE_ABS, mean_abs=None, bf16_out=False)


@pytest.mark.parametrize("rope", [
    dict(base=10000.0, factor=1.0, orig_ctx=4096, alpha=1.0, beta=32.0),     # plain RoPE
    dict(base=500000.0, factor=8.0, orig_ctx=8192, alpha=1.0, beta=32.0),
    dict(base=10000.0, factor=32.0, orig_ctx=6400, alpha=2.0, beta=16.0),
])
@MODES
def test_yarn_parameters(rope, mode):
    q, k, v = make_inputs(1, 4, 2, 1000, seed=7)
    o, lse = _gpu(q, k, v, rope, mode=mode)
    ro, rl = oracle.attn_fwd_yarn(to64(q), to64(k), to64(v), **rope)
    check_close("O", to64(o), ro)
    check_close("LSE", to64(lse), rl, max_abs=LSE_ABS, mean_abs=None, bf16_out=False)


def test_rotated_rows_in_workspace():
    """The pre-pass leaves bf16(rot(k)) at the start of the workspace and
    bf16(rot(q)) at its end (after the table and the key-norm record): equal to
    the oracle's rounded rotation except for rare one-ulp ties decided by the
    fp32 rounding of the rotation (at most 1e-3 of the elements)."""
    B, H, G, S = 1, 4, 2, 3000
    q, k, v = make_inputs(B, H, G, S, seed=9)
    ws = torch.zeros(gq.gqa_attn_fwd_yarn_workspace_size(B, H, G, S, 64, gq.GQA_ROPE_PREPASS),
                     dtype=torch.uint8, device="cuda")
    gq.fwd_yarn(q.cuda(), k.cuda(), v.cuda(), workspace=ws)
    torch.cuda.synchronize()
    nq, nk = B * H * S * 64 * 2, B * G * S * 64 * 2
    assert ws.numel() == nk + S * 32 * 8 + B * G * 128 + nq
    got_k = ws[:nk].view(torch.bfloat16).view(B, G, S, 64).to(torch.float64).cpu().numpy()
    got_q = ws[ws.numel() - nq:].view(torch.bfloat16).view(B, H, S, 64).to(torch.float64).cpu().numpy()
    ref_q, ref_k = oracle.yarn_rotated(to64(q), to64(k), **DEFAULT)
    for got, ref in ((got_q, ref_q), (got_k, ref_k)):
        diff = np.abs(got - ref)
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
        assert (diff <= ulp * 1.0001).all()
        assert (diff > 0).mean() <= 1e-3


@pytest.mark.parametrize("score_bound", [False, True], ids=["plain", "bound"])
@MODES
def test_wide_workload_group(score_bound, mode):
    """B1 H128 G16 S8192 with YaRN: the last kv group whole (8 heads x 8192 rows)."""
    w = WORKLOADS["wide_b1_h128_g16_s8192"]
    q, k, v = make_inputs(w.B, w.H, w.G, w.S, seed=0)
    o, lse = _gpu(q, k, v, DEFAULT, score_bound=score_bound, mode=mode)
    R, g = w.H // w.G, w.G - 1
    hs = slice(g * R, (g + 1) * R)
    ro, rl = oracle.attn_fwd_yarn(to64(q[:, hs]), to64(k[:, g:g + 1]), to64(v[:, g:g + 1]),
                                  **DEFAULT)
    check_close("O", to64(o[:, hs]), ro)
    check_close("LSE", to64(lse[:, hs]), rl, max_abs=LSE_ABS, mean_abs=None, bf16_out=False)


@MODES
def test_long_positions_model_mask(mode):
    """Positions up to 204799 (angles far beyond 2 pi: the table's reduction),
    the model-spec mask (window 65536, 2048 sinks), one kv group of 8 heads;
    rows sampled around the window and sink edges and at the end."""
    B, H, G, S, W, ns = 1, 8, 1, 204800, 65536, 2048
    q, k, v = make_inputs(B, H, G, S, seed=21)
    o, lse = _gpu(q, k, v, DEFAULT, mode=mode, window=W, n_sink=ns)
    qr, kr = oracle.yarn_rotated(to64(q), to64(k), **DEFAULT)
    ms = oracle.yarn_mscale(DEFAULT["factor"])
    rows = [(0, h, i) for h, i in [(0, 0), (1, ns - 1), (2, ns), (3, W - 1), (4, W), (5, W + ns),
                                    (6, 150001), (7, S - 1), (0, S - 2), (5, 131072)]]
    ro, rl = oracle.attn_fwd_rows(qr, kr, to64(v), rows, window=W, n_sink=ns,
                                  scale=0.125 * ms * ms)
    got_o = np.stack([to64(o[b, h, i]) for b, h, i in rows])
    got_l = np.array([float(lse[b, h, i]) for b, h, i in rows])
    check_close("O", got_o, ro)
    check_close("LSE", got_l, rl, max_abs=LSE_ABS, mean_abs=None, bf16_out=False)
