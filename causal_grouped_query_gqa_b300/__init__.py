"""libgqa_attn Python binding: causal grouped-query attention on one B300.

The compute path is the C-ABI library ``libgqa_attn.so`` (hand-written CUDA for
sm_103a, declared in ``include/gqa_attn.h``).  This module only marshals
arguments: torch provides device memory and the current stream, and every step
of the attention runs in the library's kernels.  There is no fallback: if the
library is missing or cannot be loaded, every call raises.

Low-level calls (same names and argument order as the C header):
    gqa_attn_fwd(q, k, v, o, lse, B, H, G, S, d, causal, window, n_sink, scale, stream)
    gqa_attn_fwd_ws(q, k, v, o, lse, B, H, G, S, d, causal, window, n_sink, scale,
                    workspace, workspace_bytes, stream)   (score-bound forward)
    gqa_attn_fwd_workspace_size(B, H, G, S, d)
    gqa_attn_fwd_yarn(q, k, v, o, lse, B, H, G, S, d, causal, window, n_sink, scale, rope_base,
                      rope_factor, rope_orig_ctx, rope_alpha, rope_beta, score_bound,
                      rope_mode, workspace, workspace_bytes, stream)
                      (YaRN rotary embeddings on q and k; rope_mode GQA_ROPE_PREPASS or
                      GQA_ROPE_FUSED)
    gqa_attn_fwd_yarn_workspace_size(B, H, G, S, d, rope_mode)
    gqa_attn_fwd_fp8(q8, k8, v, o, lse, B, H, G, S, d, causal, window, n_sink, scale, q_scale,
                     k_scale, stream)   (E4M3 queries and keys, tcgen05 kind::f8f6f4 Q K^T)
    gqa_attn_quantize_e4m3(x, out, n, inv_scale, stream)   (bf16 -> E4M3 bytes)
    gqa_attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, G, S, d, causal, window,
                 n_sink, scale, workspace, workspace_bytes, stream)
    gqa_attn_bwd_workspace_size(B, H, G, S, d)
    gqa_attn_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, H, G, S, d, causal, window,
                         n_sink, scale, stream)   (fixed library-held scratch, no allocation)
    gqa_attn_strerror(status), gqa_attn_last_device_status(stream)
    gqa_attn_timing_enable(on), gqa_attn_timing_collect(buf)  (per-kernel CUDA-event times)
Tensor helpers: ``fwd(q, k, v, ...)`` (picks the score-bound entry point for
problems of at least SCORE_BOUND_MIN_FLOPS causal FLOPs, the plain one below)
``fwd_yarn(q, k, v, ...)``, ``fwd_fp8(q8, k8, v, q_scale, k_scale, ...)``,
``quantize_e4m3(x, inv_scale)`` and ``bwd(q, k, v, o, dout, lse, ...)``.
"""
from __future__ import annotations

from ._lib import (GQA_ERR_ALIGN, GQA_ERR_CUDA, GQA_ERR_DEVICE_TIMEOUT, GQA_ERR_HEADDIM,
                   GQA_ERR_DEVICE_BOUNDS, GQA_ERR_MASK, GQA_ERR_NULL, GQA_ERR_SCALE,
                   GQA_ERR_SHAPE, GQA_ERR_TOO_LARGE, GQA_ERR_ROPE, GQA_ROPE_PREPASS, GQA_ROPE_FUSED, YARN_DEFAULTS,
                   fwd_yarn, gqa_attn_fwd_yarn, gqa_attn_fwd_yarn_workspace_size,
                   fwd_fp8, gqa_attn_fwd_fp8, gqa_attn_quantize_e4m3, quantize_e4m3,
                   GQA_ERR_WORKSPACE, GQA_NOALLOC_SCRATCH_BYTES, GQA_OK, SCORE_BOUND_MIN_FLOPS,
                   GqaError, bwd, fwd, visible_pairs,
                   gqa_attn_bwd, gqa_attn_bwd_noalloc,
                   gqa_attn_bwd_workspace_size, gqa_attn_fwd, gqa_attn_fwd_workspace_size,
                   gqa_attn_fwd_ws, gqa_attn_last_device_status,
                   gqa_attn_last_error_detail, gqa_attn_selftest_timeout, gqa_attn_strerror, gqa_attn_timing_collect, gqa_attn_timing_enable,
                   lib_path, load_library, selftest_timeout, timing_buffer)

__all__ = [
    "fwd", "bwd", "fwd_yarn", "fwd_fp8", "gqa_attn_fwd_fp8", "gqa_attn_quantize_e4m3",
    "quantize_e4m3", "gqa_attn_fwd_yarn", "gqa_attn_fwd_yarn_workspace_size",
    "GQA_ERR_ROPE", "GQA_ROPE_PREPASS", "GQA_ROPE_FUSED", "YARN_DEFAULTS", "visible_pairs", "SCORE_BOUND_MIN_FLOPS", "gqa_attn_fwd", "gqa_attn_fwd_ws", "gqa_attn_fwd_workspace_size",
    "gqa_attn_bwd", "gqa_attn_bwd_noalloc",
    "gqa_attn_bwd_workspace_size", "GQA_ERR_TOO_LARGE", "GQA_ERR_DEVICE_BOUNDS", "GQA_NOALLOC_SCRATCH_BYTES",
    "gqa_attn_strerror", "gqa_attn_last_error_detail", "gqa_attn_last_device_status",
    "gqa_attn_selftest_timeout", "selftest_timeout", "gqa_attn_timing_enable",
    "gqa_attn_timing_collect", "timing_buffer", "load_library", "lib_path", "GqaError",
    "GQA_OK", "GQA_ERR_NULL", "GQA_ERR_SHAPE", "GQA_ERR_HEADDIM", "GQA_ERR_ALIGN",
    "GQA_ERR_MASK", "GQA_ERR_SCALE", "GQA_ERR_WORKSPACE", "GQA_ERR_CUDA",
    "GQA_ERR_DEVICE_TIMEOUT",
]
