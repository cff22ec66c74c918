"""Shared helpers of the GPU parity tests: tolerances and comparisons against
the float64 oracle.

Tolerances (stated for the path: bf16 in, fp32 accumulate):
  O, dQ, dK, dV : max |gpu - oracle| <= 2e-2 and mean |gpu - oracle| <= 2e-3
  LSE           : max |gpu - oracle| <= 1e-3
Reading for bf16 outputs with |oracle| >= 8: there half a bf16 ulp (0.031 and
up) alone exceeds 2e-2, so such an element is accepted within
max(2e-2, ulp_bf16(|oracle|) / 2 + 1e-3); every element with |oracle| < 8 is
held to the plain 2e-2.  The gradients before the bf16 rounding are held to
the plain 2e-2 everywhere (tests/test_grad_precision.py, fp32-output build).
"""
from __future__ import annotations

import numpy as np
import torch

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def _bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    # bf16 has 8 significant bits: ulp(x) = 2^(floor(log2|x|) - 7)
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    return 0.5 * np.exp2(e - 7)


def check_close(name: str, got, ref, *, max_abs=MAX_ABS, mean_abs=MEAN_ABS, bf16_out=True):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    err = np.abs(got - ref)
    bound = np.full(ref.shape, float(max_abs))
    big = np.zeros(ref.shape, dtype=bool)
    if bf16_out:
        big = np.abs(ref) >= 8.0
        bound[big] = np.maximum(max_abs, _bf16_half_ulp(ref[big]) + 1e-3)
    over_small = int((err[~big] > max_abs).sum())
    over_big = int((err[big] > max_abs).sum())
    worst = np.unravel_index(np.argmax(err - bound), err.shape) if err.size else None
    msg = (f"{name}: max_err={err.max() if err.size else 0:.3e} mean_err="
           f"{err.mean() if err.size else 0:.3e} max|ref|={np.abs(ref).max() if ref.size else 0:.3f}"
           f" n_over_{max_abs:g}: |ref|<8 {over_small}, |ref|>=8 {over_big} worst_at={worst}")
    assert over_small == 0, msg
    assert (err <= bound).all(), msg
    if mean_abs is not None and err.size:
        assert err.mean() <= mean_abs, msg
    return msg


def sample_rows(B, H, S, n, seed=0, extra=()):
    """(b, h, i) rows: first/last rows, tile edges and random ones."""
    rng = np.random.default_rng(seed)
    cand = {0, S - 1, min(127, S - 1), min(128, S - 1), S // 2, max(0, S - 129)}
    rows = set()
    for i in cand:
        rows.add((int(rng.integers(B)), int(rng.integers(H)), int(i)))
    while len(rows) < n:
        rows.add((int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(S))))
    rows |= set(extra)
    return sorted(rows)
