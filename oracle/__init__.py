"""Float64 CPU oracle for causal grouped-query attention (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never calls it and shares no code with it.

The arithmetic lives in ``gqa_oracle.c`` (plain C, float64, OpenMP); this
module only compiles it with gcc on first use and marshals numpy arrays.
What it computes is stated in the C file's header: the definition printed in
"nx_f32_gqa_gate.nx source" (scores, causal mask, softmax, attn.V, the GQA
head map of test T2, the softmax backward of test T4) plus the window/sink
mask and the backward named in "SnapKitty Transformer 8B", and the YaRN
rotary embedding that page names, written from the YaRN paper (section 3).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgqa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH, defines=()) -> str:
    """Compile the oracle with gcc (-O2, no fast-math, OpenMP).  Returns the .so path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           *[f"-D{d}" for d in defines], src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    lp = ctypes.POINTER(ctypes.c_long)
    i, d = ctypes.c_int, ctypes.c_double
    lib.oracle_visible.argtypes = [ctypes.c_long, ctypes.c_long, i, i, i]
    lib.oracle_visible.restype = i
    lib.oracle_attn_fwd.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i, i, i, d]
    lib.oracle_attn_fwd.restype = None
    lib.oracle_attn_fwd_rows.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i, i, i, d, lp, i]
    lib.oracle_attn_fwd_rows.restype = None
    lib.oracle_attn_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, i, i, i, d]
    lib.oracle_attn_bwd.restype = None
    lib.oracle_attn_bwd_group.argtypes = [dp, dp, dp, dp, dp, dp, dp,
                                          i, i, i, i, i, i, i, i, d, i, i]
    lib.oracle_attn_bwd_group.restype = None
    lib.oracle_attn_bwd_group_rows.argtypes = [dp, dp, dp, dp, dp, dp, dp,
                                               i, i, i, i, i, i, i, i, d, i, i,
                                               ctypes.c_long, ctypes.c_long]
    lib.oracle_attn_bwd_group_rows.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i
    lib.oracle_yarn_freqs.argtypes = [i, d, d, d, d, d, dp]
    lib.oracle_yarn_freqs.restype = None
    lib.oracle_yarn_mscale.argtypes = [d]
    lib.oracle_yarn_mscale.restype = d
    lib.oracle_rope_rotate.argtypes = [dp, dp, lp, ctypes.c_long, i, dp]
    lib.oracle_rope_rotate.restype = None
    lib.oracle_round_bf16.argtypes = [dp, ctypes.c_long]
    lib.oracle_round_bf16.restype = None
    lib.oracle_decode_e4m3.argtypes = [ctypes.c_ubyte]
    lib.oracle_decode_e4m3.restype = d
    lib.oracle_decode_e4m3_array.argtypes = [ctypes.POINTER(ctypes.c_ubyte), dp, ctypes.c_long, d]
    lib.oracle_decode_e4m3_array.restype = None
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; a custom path loads a variant."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shape(q, k):
    B, H, S, d = q.shape
    Bk, G, Sk, dk = k.shape
    assert (B, S, d) == (Bk, Sk, dk) and H % G == 0, "q [B,H,S,d] / k,v [B,G,S,d] with H % G == 0"
    return B, H, G, S, d


def attn_fwd(q, k, v, *, causal=True, window=0, n_sink=0, scale=None, lib=None):
    """Full forward.  q [B,H,S,d], k/v [B,G,S,d] -> (o [B,H,S,d], lse [B,H,S]) in float64."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, G, S, d = _shape(q, k)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    o = np.zeros((B, H, S, d))
    lse = np.zeros((B, H, S))
    lib.oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                        B, H, G, S, d, int(causal), int(window), int(n_sink), scale)
    return o, lse


def attn_fwd_rows(q, k, v, rows, *, causal=True, window=0, n_sink=0, scale=None, lib=None):
    """Forward on sampled rows (b, h, i) only -> (o_rows [n,d], lse_rows [n])."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, G, S, d = _shape(q, k)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    n = rows.shape[0]
    o = np.zeros((n, d))
    lse = np.zeros(n)
    lib.oracle_attn_fwd_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                             B, H, G, S, d, int(causal), int(window), int(n_sink), scale,
                             rows.ctypes.data_as(ctypes.POINTER(ctypes.c_long)), n)
    return o, lse


def attn_bwd(q, k, v, dO, *, causal=True, window=0, n_sink=0, scale=None, lib=None):
    """Full backward (exact P recomputed by the oracle) -> (dq, dk, dv) in float64."""
    lib = lib or load()
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, H, G, S, d = _shape(q, k)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    dq = np.zeros((B, H, S, d))
    dk = np.zeros((B, G, S, d))
    dv = np.zeros((B, G, S, d))
    lib.oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv),
                        B, H, G, S, d, int(causal), int(window), int(n_sink), scale)
    return dq, dk, dv


def attn_bwd_group(q, k, v, dO, b, g, *, causal=True, window=0, n_sink=0, scale=None, lib=None):
    """Backward of one kv group -> (dq of its R heads [R,S,d], dk [S,d], dv [S,d])."""
    lib = lib or load()
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, H, G, S, d = _shape(q, k)
    R = H // G
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    dq = np.zeros((R, S, d))
    dk = np.zeros((S, d))
    dv = np.zeros((S, d))
    lib.oracle_attn_bwd_group(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv),
                              B, H, G, S, d, int(causal), int(window), int(n_sink), scale,
                              int(b), int(g))
    return dq, dk, dv


def attn_bwd_group_rows(q, k, v, dO, b, g, i_begin, i_end, *, causal=True, window=0,
                        n_sink=0, scale=None, lib=None):
    """Backward of one kv group restricted to query rows [i_begin, i_end): the
    dq of those rows and their contributions to dk, dv (a bounded sample)."""
    lib = lib or load()
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, H, G, S, d = _shape(q, k)
    R = H // G
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    dq = np.zeros((R, S, d))
    dk = np.zeros((S, d))
    dv = np.zeros((S, d))
    lib.oracle_attn_bwd_group_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dq), _ptr(dk),
                                   _ptr(dv), B, H, G, S, d, int(causal), int(window),
                                   int(n_sink), scale, int(b), int(g), int(i_begin), int(i_end))
    return dq, dk, dv


def num_threads(lib=None) -> int:
    return int((lib or load()).oracle_num_threads())


def visible(i: int, j: int, *, causal=True, window=0, n_sink=0, lib=None) -> bool:
    lib = lib or load()
    return bool(lib.oracle_visible(int(i), int(j), int(causal), int(window), int(n_sink)))


# ------------------------------------------------------------------ YaRN RoPE

def yarn_freqs(d=64, base=10000.0, factor=32.0, orig_ctx=6400, alpha=1.0, beta=32.0, lib=None):
    """Per-pair rotation frequencies h_i (YaRN, NTK-by-parts) -> [d/2] float64."""
    lib = lib or load()
    f = np.zeros(d // 2)
    lib.oracle_yarn_freqs(int(d), float(base), float(factor), float(orig_ctx), float(alpha),
                          float(beta), _ptr(f))
    return f


def yarn_mscale(factor, lib=None) -> float:
    """sqrt(1/t) of YaRN's attention temperature: 0.1 ln(s) + 1."""
    return float((lib or load()).oracle_yarn_mscale(float(factor)))


def rope_rotate(x, freqs, positions=None, lib=None):
    """Rotates x [..., S, d] (positions 0..S-1 along the second-last axis unless
    given) by the per-pair frequencies; returns float64 of the same shape."""
    lib = lib or load()
    x = _f64(x)
    S, d = x.shape[-2], x.shape[-1]
    rows = x.reshape(-1, d)
    pos = np.ascontiguousarray(np.tile(np.arange(S) if positions is None
                                       else np.asarray(positions), rows.shape[0] // S)
                               .astype(np.int64))
    out = np.zeros_like(rows)
    f = _f64(freqs)
    lib.oracle_rope_rotate(_ptr(rows), _ptr(out), pos.ctypes.data_as(ctypes.POINTER(ctypes.c_long)),
                           rows.shape[0], d, _ptr(f))
    return out.reshape(x.shape)


def round_bf16(x, lib=None):
    """Nearest bf16 (ties to even) of each value, as float64."""
    lib = lib or load()
    y = _f64(x).copy()
    lib.oracle_round_bf16(_ptr(y), y.size)
    return y


def yarn_rotated(q, k, *, base=10000.0, factor=32.0, orig_ctx=6400, alpha=1.0, beta=32.0,
                 rounded=True, lib=None):
    """rot(q), rot(k) at positions 0..S-1, rounded once to bf16 when `rounded`
    (the tensors a bf16 model hands to attention after its rotary embedding)."""
    lib = lib or load()
    f = yarn_freqs(q.shape[-1], base, factor, orig_ctx, alpha, beta, lib=lib)
    qr, kr = rope_rotate(q, f, lib=lib), rope_rotate(k, f, lib=lib)
    if rounded:
        qr, kr = round_bf16(qr, lib=lib), round_bf16(kr, lib=lib)
    return qr, kr


def attn_fwd_yarn(q, k, v, *, base=10000.0, factor=32.0, orig_ctx=6400, alpha=1.0, beta=32.0,
                  causal=True, window=0, n_sink=0, scale=None, rounded=True, lib=None):
    """Forward with YaRN rotary embeddings on q and k (positions 0..S-1) and the
    attention temperature: attn_fwd(rot(q), rot(k), v, scale * (0.1 ln s + 1)^2),
    the rotated q and k rounded once to bf16 unless `rounded` is False."""
    lib = lib or load()
    d = q.shape[-1]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    ms = yarn_mscale(factor, lib=lib)
    qr, kr = yarn_rotated(q, k, base=base, factor=factor, orig_ctx=orig_ctx, alpha=alpha,
                          beta=beta, rounded=rounded, lib=lib)
    return attn_fwd(qr, kr, v, causal=causal, window=window, n_sink=n_sink, scale=scale * ms * ms,
                    lib=lib)


# ------------------------------------------------------------------ FP8 E4M3

def decode_e4m3(x, scale=1.0, lib=None):
    """Exact float64 values of OCP E4M3 bytes (uint8 array) times `scale`."""
    lib = lib or load()
    b = np.ascontiguousarray(np.asarray(x, dtype=np.uint8))
    out = np.zeros(b.shape, dtype=np.float64)
    lib.oracle_decode_e4m3_array(b.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)), _ptr(out),
                                 b.size, float(scale))
    return out


def attn_fwd_fp8(q8, k8, v, q_scale, k_scale, *, causal=True, window=0, n_sink=0, scale=None,
                 lib=None):
    """Forward on fp8 queries and keys: attn_fwd(decode(q8) * q_scale,
    decode(k8) * k_scale, v) with v as given (float64 of the bf16 values)."""
    lib = lib or load()
    q = decode_e4m3(q8, q_scale, lib=lib)
    k = decode_e4m3(k8, k_scale, lib=lib)
    return attn_fwd(q, k, v, causal=causal, window=window, n_sink=n_sink, scale=scale, lib=lib)
