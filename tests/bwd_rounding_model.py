"""A float64 model of the roundings the CUDA backward performs (test helper).

The oracle computes the method exactly.  The CUDA backward computes the same
method with its operands rounded as the hardware path needs them:
  * D_i = rowsum(dO_i * O_i) is taken on the forward's output O as the caller
    passes it: rounded to bf16 (page "SnapKitty Transformer 8B", section
    "Protected Inventions": D from dO and the saved O);
  * the tensor-core operands: P for dV += P^T dO (fp16, scaled per row as the
    kernel does), and dS = P (dP - D) for dK += dS^T Q and dQ = dS K (bf16),
    each rounded once;
  * everything else (scores, dP, the sums) in fp32 or better.
This module evaluates exactly that in float64 (numpy), for one kv group, so
that a test can tell the error the method's roundings cause from any error of
the kernel: the model with no operand rounding equals the oracle, and the
GPU's fp32 gradients equal the model with the kernel's roundings.

It shares no code with the CUDA library and is not the oracle: it is only
used to explain the distance between the two.
"""
from __future__ import annotations

import numpy as np


def round_bf16(x):
    """Round to the nearest bf16 (ties to even), returned as float64."""
    x32 = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    b = x32.view(np.uint32).astype(np.uint64)
    b = (b + (((b >> 16) & 1) + 0x7FFF)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def round_f16(x):
    """Round to the nearest IEEE fp16 (ties to even, with subnormals)."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def _ident(x):
    return np.asarray(x, dtype=np.float64)


ROUNDINGS = {"bf16": round_bf16, "f16": round_f16, "none": _ident}


def row_exponent(m):
    """e with 2^e * m in [2^14, 2^15) for m = max |x| of a row (float32 m),
    clamped to [-120, 120]; rows of zeros (or subnormals) take 120."""
    m = np.asarray(m, dtype=np.float32).astype(np.float64)
    _, ex = np.frexp(m)                      # m = f * 2^ex, f in [0.5, 1)
    e = np.where(m >= np.float64(np.finfo(np.float32).tiny), 15 - ex, 120)
    return np.clip(e, -120, 120).astype(np.int64)


def p_operand_rowscaled_f16(P, do_rows, E):
    """The CUDA backward's P operand of dV += P^T dO: P' = P 2^(E - e_i) rounded
    to fp16 (e_i the row exponent of dO_i, E the minimum over the kv group),
    scaled back; with dO' = dO 2^e_i exact, P'^T dO' = 2^E (P-as-rounded)^T dO."""
    e = row_exponent(np.abs(do_rows).max(axis=1))[:, None]
    return round_f16(P * np.exp2(E - e)) * np.exp2(e - E)


def visible_mask(S, causal=True, window=0, n_sink=0):
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    if not causal:
        return np.ones((S, S), dtype=bool)
    m = j <= i
    if window > 0:
        m &= (j > i - window) | (j < n_sink)
    return m


def model_bwd_group(q, k, v, do, scale, *, causal=True, window=0, n_sink=0, o=None,
                    o_round="bf16", p_round="bf16", ds_round="bf16"):
    """Backward of one kv group under the given roundings.

    q, do: [R, S, d]; k, v: [S, d] (float64 holding the bf16 inputs).
    o: the forward output the backward is handed ([R, S, d]); when None, the
    exact output rounded by `o_round`.  p_round: "bf16", "f16", "none", or
    "f16_rowscaled" (the scheme of p_operand_rowscaled_f16).
    Returns (dq [R,S,d], dk [S,d], dv [S,d]) in float64."""
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    R, S, d = q.shape
    mask = visible_mask(S, causal, window, n_sink)
    ro, rs = ROUNDINGS[o_round], ROUNDINGS[ds_round]
    if p_round == "f16_rowscaled":
        E = int(row_exponent(np.abs(do).max(axis=2)).min())
        rp = lambda P, h: p_operand_rowscaled_f16(P, do[h], E)
    else:
        rp = lambda P, h: ROUNDINGS[p_round](P)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(R):
        s = np.where(mask, scale * (q[h] @ k.T), -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        P = e / e.sum(axis=1, keepdims=True)
        O = ro(P @ v) if o is None else np.asarray(o[h], dtype=np.float64)
        D = (do[h] * O).sum(axis=1, keepdims=True)
        dP = do[h] @ v.T
        dS = rs(P * (dP - D))
        dq[h] = scale * (dS @ k)
        dk += scale * (dS.T @ q[h])
        dv += rp(P, h).T @ do[h]
    return dq, dk, dv
