"""The forward and backward captured in a CUDA graph and replayed: with
caller-provided workspaces the library allocates nothing on these paths,
launches only on the stream it is given, and keeps no host-side state between
calls, so a captured step replays with new inputs to the same results as eager
calls (forward, dK, dV bit-identical; dQ sums partials in L2 in a varying
order)."""
import pytest
import torch

import causal_grouped_query_gqa_b300 as gq
from causal_grouped_query_gqa_b300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fwd_ws", [False, True])
def test_graph_replay_matches_eager(fwd_ws):
    B, H, G, S, W, NS, d, scale = 1, 8, 2, 1000, 300, 64, 64, 0.125
    q, k, v, do = (t.cuda() for t in make_inputs(B, H, G, S, seed=21, with_grad=True))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(gq.gqa_attn_bwd_workspace_size(B, H, G, S, d), dtype=torch.uint8,
                     device="cuda")
    fws = torch.empty(gq.gqa_attn_fwd_workspace_size(B, H, G, S, d), dtype=torch.uint8,
                      device="cuda")

    def forward(q_, k_, v_, o_, lse_, stream):
        if fwd_ws:  # key-norm pre-pass + score-bound forward
            return gq.gqa_attn_fwd_ws(q_, k_, v_, o_, lse_, B, H, G, S, d, 1, W, NS, scale, fws,
                                      fws.numel(), stream)
        return gq.gqa_attn_fwd(q_, k_, v_, o_, lse_, B, H, G, S, d, 1, W, NS, scale, stream)

    def step(stream):
        assert forward(q, k, v, o, lse, stream) == gq.GQA_OK
        rc = gq.gqa_attn_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, G, S, d, 1, W, NS, scale,
                             ws, ws.numel(), stream)
        assert rc == gq.GQA_OK

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step(s)  # one-time set-up (kernel attributes, driver entry points) outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    for seed in (22, 23):
        new = make_inputs(B, H, G, S, seed=seed, with_grad=True)
        for dst, src in zip((q, k, v, do), new):
            dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        assert gq.gqa_attn_last_device_status() == gq.GQA_OK
        got = [t.clone() for t in (o, lse, dq, dk, dv)]
        ro, rl = torch.empty_like(o), torch.empty_like(lse)
        assert forward(q, k, v, ro, rl, None) == gq.GQA_OK
        rq, rk, rv = gq.bwd(q, k, v, ro, do, rl, window=W, n_sink=NS, scale=scale)
        torch.cuda.synchronize()
        assert torch.equal(got[0], ro) and torch.equal(got[1], rl)
        assert torch.equal(got[3], rk) and torch.equal(got[4], rv)
        assert (got[2].float() - rq.float()).abs().max().item() <= 2e-2


@pytest.mark.parametrize("kind", ["yarn", "yarn_fused", "fp8"])
def test_graph_replay_yarn_and_fp8(kind):
    """The rotary forward (both modes: table, rotation, forward) and the fp8
    forward captured and replayed with new inputs: bit-identical to eager calls."""
    B, H, G, S, d, scale = 1, 8, 2, 1000, 64, 0.125
    q, k, v = (t.cuda() for t in make_inputs(B, H, G, S, seed=31))
    q8 = torch.empty(q.shape, dtype=torch.uint8, device="cuda")
    k8 = torch.empty(k.shape, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    mode = gq.GQA_ROPE_FUSED if kind == "yarn_fused" else gq.GQA_ROPE_PREPASS
    yws = torch.empty(gq.gqa_attn_fwd_yarn_workspace_size(B, H, G, S, d, mode), dtype=torch.uint8,
                      device="cuda")

    def forward(o_, lse_, stream):
        if kind.startswith("yarn"):
            return gq.gqa_attn_fwd_yarn(q, k, v, o_, lse_, B, H, G, S, d, 1, 0, 0, scale, 10000.0,
                                        32.0, 6400, 1.0, 32.0, 1, mode, yws, yws.numel(), stream)
        return gq.gqa_attn_fwd_fp8(q8, k8, v, o_, lse_, B, H, G, S, d, 1, 0, 0, scale, 1 / 64,
                                   1 / 64, stream)

    def step(stream):
        if kind == "fp8":
            assert gq.gqa_attn_quantize_e4m3(q, q8, q.numel(), 64.0, stream) == gq.GQA_OK
            assert gq.gqa_attn_quantize_e4m3(k, k8, k.numel(), 64.0, stream) == gq.GQA_OK
        assert forward(o, lse, stream) == gq.GQA_OK

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    for seed in (32, 33):
        new = make_inputs(B, H, G, S, seed=seed)
        for dst, src in zip((q, k, v), new):
            dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        assert gq.gqa_attn_last_device_status() == gq.GQA_OK
        got = (o.clone(), lse.clone())
        ro, rl = torch.empty_like(o), torch.empty_like(lse)
        assert forward(ro, rl, None) == gq.GQA_OK
        torch.cuda.synchronize()
        assert torch.equal(got[0], ro) and torch.equal(got[1], rl)
