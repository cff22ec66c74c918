"""gqa_attn_bwd_noalloc: the backward for callers that cannot allocate.

Some callers cannot call cudaMalloc at the moment they run the backward (a
plug-in inside a framework that owns all device memory and hands it no scratch,
a latency-critical path that must not enter the allocator).
For them the library offers one entry point that uses a fixed scratch array the
library keeps in device memory instead of a caller-provided workspace.  These
tests check, through the C ABI, that it gives the same results as the regular
entry point and as the float64 oracle on two calls in a row, and that it
refuses problems larger than its scratch before launching anything.  This file is named to be collected last.
"""
import pytest
import torch

import oracle
import causal_grouped_query_gqa_b300 as gq
from causal_grouped_query_gqa_b300.inputs import make_inputs
from parity_util import check_close, to64

FAKE = 0x10000  # aligned non-null address; never dereferenced (rejected before launch)


def test_noalloc_rejects_problems_beyond_its_scratch():
    """Needs no GPU: the size check comes before any device work."""
    B, H, G, S = 1, 256, 16, 65536
    assert gq.gqa_attn_bwd_workspace_size(B, H, G, S, 64) > gq.GQA_NOALLOC_SCRATCH_BYTES
    rc = gq.gqa_attn_bwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                 B, H, G, S, 64, 1, 0, 0, 0.125, 0)
    assert rc == gq.GQA_ERR_TOO_LARGE
    assert "scratch" in gq.gqa_attn_strerror(rc)
    # argument checks are the same as the regular backward's
    assert gq.gqa_attn_bwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                   1, 4, 2, 128, 32, 1, 0, 0, 0.125, 0) == gq.GQA_ERR_HEADDIM


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,G,S,window,n_sink", [
    (1, 4, 2, 333, 0, 0),
    (2, 8, 2, 700, 200, 64),
])
def test_noalloc_matches_regular_backward_twice(B, H, G, S, window, n_sink):
    """Two calls in a row on different inputs (values a call left behind in the
    shared scratch would show in the next one).  Each call must match the
    regular backward -- dK and dV bit for bit (same kernels, sums in the same
    order), dQ within the tolerance (its fp32 reduce-adds may land in any
    order) -- and the float64 oracle."""
    kw = dict(window=window, n_sink=n_sink)
    for call, seed in enumerate((11, 12)):
        q_h, k_h, v_h, do_h = make_inputs(B, H, G, S, seed=seed, with_grad=True)
        q, k, v, do = (t.cuda() for t in (q_h, k_h, v_h, do_h))
        o, lse = gq.fwd(q, k, v, **kw)
        ref_dq, ref_dk, ref_dv = gq.bwd(q, k, v, o, do, lse, **kw)
        torch.cuda.synchronize()
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        rc = gq.gqa_attn_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, B, H, G, S, 64, 1,
                                     window, n_sink, 0.125, None)
        assert rc == gq.GQA_OK, gq.gqa_attn_strerror(rc)
        torch.cuda.synchronize()
        assert gq.gqa_attn_last_device_status() == gq.GQA_OK
        assert torch.equal(dk, ref_dk), f"dK call {call}"
        assert torch.equal(dv, ref_dv), f"dV call {call}"
        check_close(f"dQ call {call} vs gqa_attn_bwd", to64(dq), to64(ref_dq))
        rq, rk, rv = oracle.attn_bwd(to64(q_h), to64(k_h), to64(v_h), to64(do_h), **kw)
        check_close(f"dQ call {call}", to64(dq), rq)
        check_close(f"dK call {call}", to64(dk), rk)
        check_close(f"dV call {call}", to64(dv), rv)
