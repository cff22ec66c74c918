"""ctypes marshalling for libgqa_attn.so (see include/gqa_attn.h for the contract)."""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libgqa_attn.so")
_lock = threading.Lock()
_lib = None

GQA_OK = 0
GQA_ERR_NULL = -1
GQA_ERR_SHAPE = -2
GQA_ERR_HEADDIM = -3
GQA_ERR_ALIGN = -4
GQA_ERR_MASK = -5
GQA_ERR_SCALE = -6
GQA_ERR_WORKSPACE = -7
GQA_ERR_CUDA = -8
GQA_ERR_DEVICE_TIMEOUT = -9
GQA_ERR_TOO_LARGE = -10
GQA_ERR_DEVICE_BOUNDS = -11
GQA_ERR_ROPE = -12
# gqa_attn_fwd_yarn rope_mode: rotate q and k before the forward / query tiles inside it
GQA_ROPE_PREPASS = 0
GQA_ROPE_FUSED = 1
GQA_NOALLOC_SCRATCH_BYTES = 64 << 20


class GqaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {gqa_attn_strerror(status)} (status {status})"
        if status == GQA_ERR_CUDA:
            detail = gqa_attn_last_error_detail()
            if detail:
                msg += f" -- {detail}"
        super().__init__(msg)


def lib_path() -> str:
    return _LIB_PATH


def load_library():
    """Loads the in-tree CUDA library; raises if it is absent (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with "
                "`python -m causal_grouped_query_gqa_b300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.gqa_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp]
        lib.gqa_attn_fwd.restype = i
        lib.gqa_attn_fwd_ws.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp, sz, vp]
        lib.gqa_attn_fwd_ws.restype = i
        lib.gqa_attn_fwd_workspace_size.argtypes = [i, i, i, i, i]
        lib.gqa_attn_fwd_workspace_size.restype = sz
        lib.gqa_attn_fwd_yarn.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f,
                                          f, f, i, f, f, i, i, vp, sz, vp]
        lib.gqa_attn_fwd_yarn.restype = i
        lib.gqa_attn_fwd_yarn_workspace_size.argtypes = [i, i, i, i, i, i]
        lib.gqa_attn_fwd_yarn_workspace_size.restype = sz
        lib.gqa_attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, f, f, vp]
        lib.gqa_attn_fwd_fp8.restype = i
        lib.gqa_attn_quantize_e4m3.argtypes = [vp, vp, ctypes.c_longlong, f, vp]
        lib.gqa_attn_quantize_e4m3.restype = i
        lib.gqa_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                     i, i, i, i, i, i, i, i, f, vp, sz, vp]
        lib.gqa_attn_bwd.restype = i
        lib.gqa_attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                             i, i, i, i, i, i, i, i, f, vp]
        lib.gqa_attn_bwd_noalloc.restype = i
        lib.gqa_attn_bwd_workspace_size.argtypes = [i, i, i, i, i]
        lib.gqa_attn_bwd_workspace_size.restype = sz
        lib.gqa_attn_strerror.argtypes = [i]
        lib.gqa_attn_strerror.restype = ctypes.c_char_p
        lib.gqa_attn_last_error_detail.argtypes = []
        lib.gqa_attn_last_error_detail.restype = ctypes.c_char_p
        lib.gqa_attn_last_device_status.argtypes = [vp]
        lib.gqa_attn_last_device_status.restype = i
        lib.gqa_attn_selftest_timeout.argtypes = [ctypes.c_uint,
                                                  ctypes.POINTER(ctypes.c_ulonglong),
                                                  ctypes.POINTER(ctypes.c_int), vp]
        lib.gqa_attn_selftest_timeout.restype = i
        lib.gqa_attn_timing_enable.argtypes = [i]
        lib.gqa_attn_timing_enable.restype = i
        lib.gqa_attn_timing_collect.argtypes = [ctypes.POINTER(ctypes.c_float), i]
        lib.gqa_attn_timing_collect.restype = i
        _lib = lib
        return lib


def _p(x):
    """Device address of a tensor (or an int address / None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------- C-ABI mirrors ---

def gqa_attn_fwd(q, k, v, o, lse, B, H, G, S, d, causal, window, n_sink, scale, stream=None):
    return load_library().gqa_attn_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, G, S, d,
                                       int(causal), int(window), int(n_sink), float(scale),
                                       _stream(stream))


def gqa_attn_fwd_ws(q, k, v, o, lse, B, H, G, S, d, causal, window, n_sink, scale, workspace,
                    workspace_bytes, stream=None):
    return load_library().gqa_attn_fwd_ws(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, G, S, d,
                                          int(causal), int(window), int(n_sink), float(scale),
                                          _p(workspace), int(workspace_bytes), _stream(stream))


def gqa_attn_fwd_workspace_size(B, H, G, S, d):
    return load_library().gqa_attn_fwd_workspace_size(B, H, G, S, d)


def gqa_attn_fwd_yarn(q, k, v, o, lse, B, H, G, S, d, causal, window, n_sink, scale, rope_base,
                      rope_factor, rope_orig_ctx, rope_alpha, rope_beta, score_bound, rope_mode,
                      workspace, workspace_bytes, stream=None):
    return load_library().gqa_attn_fwd_yarn(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, G, S, d,
                                            int(causal), int(window), int(n_sink), float(scale),
                                            float(rope_base), float(rope_factor),
                                            int(rope_orig_ctx), float(rope_alpha),
                                            float(rope_beta), int(bool(score_bound)),
                                            int(rope_mode), _p(workspace), int(workspace_bytes),
                                            _stream(stream))


def gqa_attn_fwd_fp8(q8, k8, v, o, lse, B, H, G, S, d, causal, window, n_sink, scale, q_scale,
                     k_scale, stream=None):
    return load_library().gqa_attn_fwd_fp8(_p(q8), _p(k8), _p(v), _p(o), _p(lse), B, H, G, S, d,
                                           int(causal), int(window), int(n_sink), float(scale),
                                           float(q_scale), float(k_scale), _stream(stream))


def gqa_attn_quantize_e4m3(x, out, n, inv_scale, stream=None):
    return load_library().gqa_attn_quantize_e4m3(_p(x), _p(out), int(n), float(inv_scale),
                                                 _stream(stream))


def gqa_attn_fwd_yarn_workspace_size(B, H, G, S, d, rope_mode=0):
    return load_library().gqa_attn_fwd_yarn_workspace_size(B, H, G, S, d, int(rope_mode))


def gqa_attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, G, S, d, causal, window, n_sink,
                 scale, workspace, workspace_bytes, stream=None):
    return load_library().gqa_attn_bwd(_p(q), _p(k), _p(v), _p(o), _p(dout), _p(lse), _p(dq),
                                       _p(dk), _p(dv), B, H, G, S, d, int(causal), int(window),
                                       int(n_sink), float(scale), _p(workspace),
                                       int(workspace_bytes), _stream(stream))


def gqa_attn_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, H, G, S, d, causal, window,
                         n_sink, scale, stream=None):
    return load_library().gqa_attn_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(dout), _p(lse),
                                               _p(dq), _p(dk), _p(dv), B, H, G, S, d, int(causal),
                                               int(window), int(n_sink), float(scale),
                                               _stream(stream))


def gqa_attn_bwd_workspace_size(B, H, G, S, d):
    return load_library().gqa_attn_bwd_workspace_size(B, H, G, S, d)


def gqa_attn_strerror(status: int) -> str:
    return load_library().gqa_attn_strerror(int(status)).decode()


def gqa_attn_last_error_detail() -> str:
    return load_library().gqa_attn_last_error_detail().decode()


def gqa_attn_last_device_status(stream=None) -> int:
    return load_library().gqa_attn_last_device_status(_stream(stream))


def gqa_attn_selftest_timeout(budget_ms: int, elapsed_ns=None, returned_ok=None, stream=0) -> int:
    """C-ABI mirror; elapsed_ns / returned_ok may be ctypes arrays or None."""
    return load_library().gqa_attn_selftest_timeout(int(budget_ms), elapsed_ns, returned_ok,
                                                    _stream(stream))


def selftest_timeout(budget_ms: int = 20, stream=None):
    """Runs the device self-test of the bounded waits; returns (status,
    [elapsed ns of the two waiters], [whether each wait reported success])."""
    el = (ctypes.c_ulonglong * 2)()
    ok = (ctypes.c_int * 2)()
    rc = gqa_attn_selftest_timeout(budget_ms, el, ok, stream)
    return rc, [int(x) for x in el], [int(x) for x in ok]


GQA_KERNEL_COUNT = 6  # fwd, bwd prep, bwd main, bwd dq convert, fwd key norms, rotary pre-pass


def gqa_attn_timing_enable(on: bool) -> int:
    return load_library().gqa_attn_timing_enable(int(bool(on)))


def timing_buffer():
    return (ctypes.c_float * GQA_KERNEL_COUNT)()


def gqa_attn_timing_collect(buf=None):
    """Durations (ms) of the last launch of each kernel since the previous collect
    (-1 where a kernel did not run); fills and returns `buf`."""
    buf = timing_buffer() if buf is None else buf
    rc = load_library().gqa_attn_timing_collect(buf, len(buf))
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_timing_collect")
    return buf


# --------------------------------------------------------- tensor helpers ---

def _check(t, shape, dtype, name):
    import torch
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: expected contiguous CUDA {dtype} {tuple(shape)}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device}")
    return torch


def visible_pairs(S: int, causal=True, window=0, n_sink=0) -> int:
    """Visible (query, key) pairs of one head under the mask (closed form)."""
    if not causal:
        return S * S
    if window <= 0 or window >= S:
        return S * (S + 1) // 2
    in_window = window * (window + 1) // 2 + (S - window) * window
    older = S - window  # rows with keys before their window: 1 .. S - window such keys
    ns = min(max(n_sink, 0), older)
    sinks = ns * (ns + 1) // 2 + (older - ns) * ns
    return in_window + sinks


# Smallest forward, in causal FLOPs, for which the score bound is taken by
# default: below it the key-norm pre-pass costs about what the bound saves.
SCORE_BOUND_MIN_FLOPS = 1 << 36


def fwd(q, k, v, *, causal=True, window=0, n_sink=0, scale=None, out=None, lse=None,
        workspace=None, score_bound=None, stream=None):
    """o, lse = fwd(q [B,H,S,64] bf16, k/v [B,G,S,64] bf16) on the current CUDA stream.

    score_bound: True runs gqa_attn_fwd_ws (key-norm pre-pass, then the forward
    with the score bound; `workspace` is allocated when not given), False runs
    gqa_attn_fwd; None takes the bound when the forward has at least
    SCORE_BOUND_MIN_FLOPS causal FLOPs.  Both give the same result contract."""
    import torch
    B, H, S, d = q.shape
    G = k.shape[1]
    _check(q, (B, H, S, d), torch.bfloat16, "q")
    _check(k, (B, G, S, d), torch.bfloat16, "k")
    _check(v, (B, G, S, d), torch.bfloat16, "v")
    scale = 1.0 / d ** 0.5 if scale is None else scale
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None else lse
    if score_bound is None:
        flops = 4 * d * B * H * visible_pairs(S, causal, window, n_sink)
        score_bound = flops >= SCORE_BOUND_MIN_FLOPS
    if not score_bound:
        rc = gqa_attn_fwd(q, k, v, o, l, B, H, G, S, d, causal, window, n_sink, scale, stream)
        if rc != GQA_OK:
            raise GqaError(rc, "gqa_attn_fwd")
        return o, l
    need = gqa_attn_fwd_workspace_size(B, H, G, S, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    rc = gqa_attn_fwd_ws(q, k, v, o, l, B, H, G, S, d, causal, window, n_sink, scale, workspace,
                         workspace.numel() * workspace.element_size(), stream)
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_fwd_ws")
    return o, l


# YaRN parameters of the model-spec workload: factor 32 over an original
# context of 204800 / 32 tokens, RoFormer's base 10^4 and the paper's ramp
# bounds alpha = 1, beta = 32 (the pages give only the factor and the length).
YARN_DEFAULTS = dict(rope_base=10000.0, rope_factor=32.0, rope_orig_ctx=6400, rope_alpha=1.0,
                     rope_beta=32.0)


def fwd_yarn(q, k, v, *, causal=True, window=0, n_sink=0, scale=None, rope_base=10000.0,
             rope_factor=32.0, rope_orig_ctx=6400, rope_alpha=1.0, rope_beta=32.0,
             out=None, lse=None, workspace=None, score_bound=None, rope_mode=GQA_ROPE_PREPASS,
             stream=None):
    """o, lse = fwd_yarn(q, k, v) with YaRN rotary embeddings on q and k
    (gqa_attn_fwd_yarn; `workspace` is allocated when not given; score_bound as
    in fwd(): None takes it for problems of at least SCORE_BOUND_MIN_FLOPS;
    rope_mode GQA_ROPE_PREPASS rotates q and k before the forward,
    GQA_ROPE_FUSED turns the query tiles inside it, with no rotated-query
    workspace)."""
    import torch
    B, H, S, d = q.shape
    G = k.shape[1]
    _check(q, (B, H, S, d), torch.bfloat16, "q")
    _check(k, (B, G, S, d), torch.bfloat16, "k")
    _check(v, (B, G, S, d), torch.bfloat16, "v")
    scale = 1.0 / d ** 0.5 if scale is None else scale
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None else lse
    need = gqa_attn_fwd_yarn_workspace_size(B, H, G, S, d, rope_mode)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if score_bound is None:
        score_bound = 4 * d * B * H * visible_pairs(S, causal, window, n_sink) >= SCORE_BOUND_MIN_FLOPS
    rc = gqa_attn_fwd_yarn(q, k, v, o, l, B, H, G, S, d, causal, window, n_sink, scale, rope_base,
                           rope_factor, rope_orig_ctx, rope_alpha, rope_beta, score_bound,
                           rope_mode, workspace, workspace.numel() * workspace.element_size(),
                           stream)
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_fwd_yarn")
    return o, l


def quantize_e4m3(x, inv_scale, *, stream=None):
    """E4M3 bytes of a bf16 CUDA tensor: round(x * inv_scale), saturating
    (gqa_attn_quantize_e4m3); returns a uint8 tensor of the same shape."""
    import torch
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous() or x.numel() % 16:
        raise ValueError("quantize_e4m3: contiguous CUDA bf16 tensor with a multiple of 16 elements")
    out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    rc = gqa_attn_quantize_e4m3(x, out, x.numel(), inv_scale, stream)
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_quantize_e4m3")
    return out


def fwd_fp8(q8, k8, v, q_scale, k_scale, *, causal=True, window=0, n_sink=0, scale=None,
            out=None, lse=None, stream=None):
    """o, lse = fwd_fp8(q8 [B,H,S,64] uint8, k8 [B,G,S,64] uint8 (E4M3 bytes), v
    [B,G,S,64] bf16, q_scale, k_scale): attention over decode(q8) * q_scale and
    decode(k8) * k_scale (gqa_attn_fwd_fp8)."""
    import torch
    B, H, S, d = q8.shape
    G = k8.shape[1]
    _check(q8, (B, H, S, d), torch.uint8, "q8")
    _check(k8, (B, G, S, d), torch.uint8, "k8")
    _check(v, (B, G, S, d), torch.bfloat16, "v")
    scale = 1.0 / d ** 0.5 if scale is None else scale
    o = torch.empty((B, H, S, d), dtype=torch.bfloat16, device=v.device) if out is None else out
    l = torch.empty((B, H, S), dtype=torch.float32, device=v.device) if lse is None else lse
    rc = gqa_attn_fwd_fp8(q8, k8, v, o, l, B, H, G, S, d, causal, window, n_sink, scale, q_scale,
                          k_scale, stream)
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_fwd_fp8")
    return o, l


def bwd(q, k, v, o, dout, lse, *, causal=True, window=0, n_sink=0, scale=None,
        workspace=None, stream=None):
    """dq, dk, dv = bwd(q, k, v, o, dout, lse) (o and lse from fwd)."""
    import torch
    B, H, S, d = q.shape
    G = k.shape[1]
    _check(q, (B, H, S, d), torch.bfloat16, "q")
    _check(k, (B, G, S, d), torch.bfloat16, "k")
    _check(v, (B, G, S, d), torch.bfloat16, "v")
    _check(o, (B, H, S, d), torch.bfloat16, "o")
    _check(dout, (B, H, S, d), torch.bfloat16, "dout")
    _check(lse, (B, H, S), torch.float32, "lse")
    scale = 1.0 / d ** 0.5 if scale is None else scale
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    need = gqa_attn_bwd_workspace_size(B, H, G, S, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    rc = gqa_attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, G, S, d, causal, window, n_sink,
                      scale, workspace, workspace.numel() * workspace.element_size(), stream)
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_bwd")
    return dq, dk, dv
