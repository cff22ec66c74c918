"""GPU fp8 forward (gqa_attn_fwd_fp8: E4M3 queries and keys, tcgen05
kind::f8f6f4 Q K^T, bf16 P.V) vs the float64 oracle, through the C ABI.

Inputs: seeded bf16 q, k, v (the shared recipe); q and k quantised on the HOST
with torch's CPU float32 -> float8_e4m3fn cast (round to nearest even) at
per-tensor scales, so the same bytes go to the GPU and -- decoded exactly by
the oracle's own E4M3 decoder -- to the oracle.  The stated tolerances then
hold unchanged: the only fp8 step is the representation of q and k, which
both sides share.  The library's own quantisation kernel is checked against
the same host cast, byte for byte."""
import numpy as np
import pytest
import torch

import oracle
import causal_grouped_query_gqa_b300 as gq
from causal_grouped_query_gqa_b300.inputs import WORKLOADS, make_inputs
from parity_util import LSE_ABS, check_close, to64

pytestmark = pytest.mark.gpu


def _host_quantize(x):
    """(bytes uint8, dequantisation scale): inv = 440 / max|x| keeps every
    product below 448, where the host cast and the kernel's saturating one agree."""
    xf = x.float()
    inv = torch.tensor(440.0 / float(xf.abs().max()), dtype=torch.float32)
    b = (xf * inv).to(torch.float8_e4m3fn).view(torch.uint8)
    return b, float(1.0 / inv.double()), float(inv)


def _run(B, H, G, S, causal=True, window=0, n_sink=0, seed=0, heads=None):
    q, k, v = make_inputs(B, H, G, S, seed=seed)
    q8, qs, _ = _host_quantize(q)
    k8, ks, _ = _host_quantize(k)
    # the scales as the fp32 values the GPU receives
    qs, ks = float(np.float32(qs)), float(np.float32(ks))
    o, lse = gq.fwd_fp8(q8.cuda(), k8.cuda(), v.cuda(), qs, ks, causal=causal, window=window,
                        n_sink=n_sink)
    torch.cuda.synchronize()
    assert gq.gqa_attn_last_device_status() == gq.GQA_OK
    mask = dict(causal=causal, window=window, n_sink=n_sink)
    if heads is None:
        ro, rl = oracle.attn_fwd_fp8(q8.numpy(), k8.numpy(), to64(v), qs, ks, **mask)
        check_close("O", to64(o), ro)
        check_close("LSE", to64(lse), rl, max_abs=LSE_ABS, mean_abs=None, bf16_out=False)
    else:
        b, g = heads
        R = H // G
        hs = slice(g * R, (g + 1) * R)
        ro, rl = oracle.attn_fwd_fp8(q8[b:b + 1, hs].numpy(), k8[b:b + 1, g:g + 1].numpy(),
                                     to64(v[b:b + 1, g:g + 1]), qs, ks, **mask)
        check_close("O", to64(o[b:b + 1, hs]), ro)
        check_close("LSE", to64(lse[b:b + 1, hs]), rl, max_abs=LSE_ABS, mean_abs=None,
                    bf16_out=False)


@pytest.mark.parametrize("B,H,G,S,causal,window,n_sink", [
    (1, 4, 2, 128, True, 0, 0),
    (2, 4, 2, 300, True, 0, 0),
    (1, 6, 2, 777, True, 129, 300),
    (1, 4, 2, 513, False, 0, 0),
    (1, 8, 1, 520, True, 0, 0),
    (4, 6, 2, 2048, True, 0, 0),      # more units than SMs
])
def test_fp8_forward(B, H, G, S, causal, window, n_sink):
    _run(B, H, G, S, causal, window, n_sink, seed=S)


def test_fp8_wide_workload_group():
    """B1 H128 G16 S8192 in fp8: the last kv group whole."""
    w = WORKLOADS["wide_b1_h128_g16_s8192"]
    _run(w.B, w.H, w.G, w.S, heads=(0, w.G - 1))


def test_quantize_kernel_matches_host_cast():
    x = make_inputs(1, 3, 1, 1000, seed=31)[0]
    _, _, inv = _host_quantize(x)
    ref, _, _ = _host_quantize(x)
    got = gq.quantize_e4m3(x.cuda(), inv)
    torch.cuda.synchronize()
    assert torch.equal(got.cpu(), ref)
    # saturation: the kernel clamps to +-448 (0x7E / 0xFE) instead of NaN
    big = torch.tensor([1e6, -1e6] + [0.0] * 14, dtype=torch.bfloat16)
    sat = gq.quantize_e4m3(big.cuda(), 1.0).cpu()
    assert sat[0].item() == 0x7E and sat[1].item() == 0xFE
