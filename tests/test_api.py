"""Host-side checks of the C ABI: the library loads without a GPU, exports every
symbol include/gqa_attn.h declares, and rejects bad arguments before touching
the device (so these calls are safe on a machine with no GPU)."""
import ctypes
import os
import re

import pytest

import causal_grouped_query_gqa_b300 as gq
from causal_grouped_query_gqa_b300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gq.load_library()


def _declared_symbols():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names |= set(re.findall(r"GQA_API\s+[\w\s\*]*?\b(gqa_\w+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_symbols()
    assert {"gqa_attn_fwd", "gqa_attn_fwd_ws", "gqa_attn_fwd_workspace_size",
            "gqa_attn_bwd", "gqa_attn_bwd_workspace_size",
            "gqa_attn_strerror", "gqa_attn_last_device_status"} <= names
    raw = ctypes.CDLL(gq.lib_path())
    for n in sorted(names):
        assert hasattr(raw, n), f"{n} declared but not exported"


def test_strerror(lib):
    for code in range(0, -13, -1):
        s = gq.gqa_attn_strerror(code)
        assert isinstance(s, str) and s and s != "unknown status"
    assert gq.gqa_attn_strerror(12345) == "unknown status"


def test_workspace_size(lib):
    B, H, G, S = 4, 32, 8, 4096
    # fp32 dQ accumulator, two fp32 row arrays, an fp16 copy of dout, one int per kv group
    assert gq.gqa_attn_bwd_workspace_size(B, H, G, S, 64) == (
        B * H * S * 64 * 4 + 2 * B * H * S * 4 + B * H * S * 64 * 2 + -(-B * G * 4 // 16) * 16)
    # row arrays are padded to a multiple of 128 rows
    assert gq.gqa_attn_bwd_workspace_size(1, 2, 1, 130, 64) == (
        2 * 130 * 64 * 4 + 2 * 2 * 256 * 4 + 2 * 130 * 64 * 2 + 16)
    assert gq.gqa_attn_bwd_workspace_size(B, H, G, S, 128) == 0
    assert gq.gqa_attn_bwd_workspace_size(1, 3, 2, 10, 64) == 0
    assert gq.gqa_attn_bwd_workspace_size(0, 4, 2, 10, 64) == 0
    # forward: one 128-byte record (32 fp32 partial maxima of |k|^2) per kv head
    assert gq.gqa_attn_fwd_workspace_size(B, H, G, S, 64) == B * G * 128
    assert gq.gqa_attn_fwd_workspace_size(1, 3, 2, 10, 64) == 0
    assert gq.gqa_attn_fwd_workspace_size(B, H, G, S, 128) == 0


FAKE = 0x10000  # a 16-byte-aligned non-null address that is never dereferenced


def _fwd(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=4, G=2, S=128, d=64,
             causal=1, window=0, n_sink=0, scale=0.125, stream=0)
    a.update(kw)
    return gq.gqa_attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["G"],
                           a["S"], a["d"], a["causal"], a["window"], a["n_sink"], a["scale"],
                           a["stream"])


def _fwd_ws(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=4, G=2, S=128, d=64,
             causal=1, window=0, n_sink=0, scale=0.125, ws=FAKE, wsb=1 << 20, stream=0)
    a.update(kw)
    return gq.gqa_attn_fwd_ws(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["G"],
                              a["S"], a["d"], a["causal"], a["window"], a["n_sink"], a["scale"],
                              a["ws"], a["wsb"], a["stream"])


def _bwd(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, dout=FAKE, lse=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
             B=1, H=4, G=2, S=128, d=64, causal=1, window=0, n_sink=0, scale=0.125,
             ws=FAKE, wsb=1 << 30, stream=0)
    a.update(kw)
    return gq.gqa_attn_bwd(a["q"], a["k"], a["v"], a["o"], a["dout"], a["lse"], a["dq"], a["dk"],
                           a["dv"], a["B"], a["H"], a["G"], a["S"], a["d"], a["causal"],
                           a["window"], a["n_sink"], a["scale"], a["ws"], a["wsb"], a["stream"])


def _fwd_yarn(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=4, G=2, S=128, d=64,
             causal=1, window=0, n_sink=0, scale=0.125, base=10000.0, factor=32.0, L=6400,
             alpha=1.0, beta=32.0, sb=1, mode=0, ws=FAKE, wsb=1 << 24, stream=0)
    a.update(kw)
    return gq.gqa_attn_fwd_yarn(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["G"],
                                a["S"], a["d"], a["causal"], a["window"], a["n_sink"], a["scale"],
                                a["base"], a["factor"], a["L"], a["alpha"], a["beta"], a["sb"],
                                a["mode"], a["ws"], a["wsb"], a["stream"])


def _fwd_fp8(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=4, G=2, S=128, d=64,
             causal=1, window=0, n_sink=0, scale=0.125, qs=0.01, ks=0.01, stream=0)
    a.update(kw)
    return gq.gqa_attn_fwd_fp8(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["G"],
                               a["S"], a["d"], a["causal"], a["window"], a["n_sink"], a["scale"],
                               a["qs"], a["ks"], a["stream"])


@pytest.mark.parametrize("call", [_fwd, _fwd_ws, _fwd_yarn, _fwd_fp8, _bwd])
def test_argument_errors(lib, call):
    assert call(B=0) == gq.GQA_ERR_SHAPE
    assert call(S=0) == gq.GQA_ERR_SHAPE
    assert call(S=-5) == gq.GQA_ERR_SHAPE
    assert call(H=5, G=2) == gq.GQA_ERR_SHAPE
    assert call(G=0) == gq.GQA_ERR_SHAPE
    assert call(d=128) == gq.GQA_ERR_HEADDIM
    assert call(d=32) == gq.GQA_ERR_HEADDIM
    assert call(causal=0, window=16) == gq.GQA_ERR_MASK
    assert call(n_sink=-1, window=16) == gq.GQA_ERR_MASK
    assert call(scale=0.0) == gq.GQA_ERR_SCALE
    assert call(scale=-1.0) == gq.GQA_ERR_SCALE
    assert call(scale=float("inf")) == gq.GQA_ERR_SCALE
    assert call(scale=float("nan")) == gq.GQA_ERR_SCALE
    assert call(q=None) == gq.GQA_ERR_NULL
    assert call(k=FAKE + 8) == gq.GQA_ERR_ALIGN
    assert call(v=FAKE + 2) == gq.GQA_ERR_ALIGN


def test_fwd_specific_errors(lib):
    assert _fwd(lse=None) == gq.GQA_ERR_NULL
    assert _fwd(o=FAKE + 4) == gq.GQA_ERR_ALIGN


def test_fwd_ws_specific_errors(lib):
    assert _fwd_ws(ws=None) == gq.GQA_ERR_NULL
    assert _fwd_ws(ws=FAKE + 4) == gq.GQA_ERR_ALIGN
    assert _fwd_ws(wsb=1 * 2 * 16 - 1) == gq.GQA_ERR_WORKSPACE
    assert _fwd_ws(lse=None) == gq.GQA_ERR_NULL


def test_fwd_yarn_specific_errors(lib):
    assert _fwd_yarn(base=1.0) == gq.GQA_ERR_ROPE
    assert _fwd_yarn(factor=0.5) == gq.GQA_ERR_ROPE
    assert _fwd_yarn(L=0) == gq.GQA_ERR_ROPE
    assert _fwd_yarn(alpha=32.0, beta=32.0) == gq.GQA_ERR_ROPE
    assert _fwd_yarn(alpha=-1.0) == gq.GQA_ERR_ROPE
    assert _fwd_yarn(base=float("nan")) == gq.GQA_ERR_ROPE
    assert _fwd_yarn(ws=None) == gq.GQA_ERR_NULL
    assert _fwd_yarn(ws=FAKE + 4) == gq.GQA_ERR_ALIGN
    assert _fwd_yarn(mode=2) == gq.GQA_ERR_ROPE
    assert _fwd_yarn(mode=-1) == gq.GQA_ERR_ROPE
    # rotated keys (bf16), the (cos, sin) table, the key-norm record and, in the
    # pre-pass mode, the rotated queries (bf16)
    fused = gq.gqa_attn_fwd_yarn_workspace_size(1, 4, 2, 128, 64, gq.GQA_ROPE_FUSED)
    assert fused == 1 * 2 * 128 * 64 * 2 + 128 * 32 * 8 + 1 * 2 * 128
    need = gq.gqa_attn_fwd_yarn_workspace_size(1, 4, 2, 128, 64, gq.GQA_ROPE_PREPASS)
    assert need == fused + 1 * 4 * 128 * 64 * 2
    assert _fwd_yarn(wsb=need - 1) == gq.GQA_ERR_WORKSPACE
    assert _fwd_yarn(mode=1, wsb=fused - 1) == gq.GQA_ERR_WORKSPACE
    assert gq.gqa_attn_fwd_yarn_workspace_size(1, 3, 2, 128, 64, 0) == 0
    assert gq.gqa_attn_fwd_yarn_workspace_size(1, 4, 2, 128, 64, 2) == 0


def test_fp8_specific_errors(lib):
    assert _fwd_fp8(qs=0.0) == gq.GQA_ERR_SCALE
    assert _fwd_fp8(ks=float("inf")) == gq.GQA_ERR_SCALE
    assert _fwd_fp8(qs=1e-30, ks=1e-30) == gq.GQA_ERR_SCALE
    assert _fwd_fp8(lse=None) == gq.GQA_ERR_NULL
    q = gq.gqa_attn_quantize_e4m3
    assert q(None, FAKE, 16, 1.0, 0) == gq.GQA_ERR_NULL
    assert q(FAKE, FAKE, 15, 1.0, 0) == gq.GQA_ERR_SHAPE
    assert q(FAKE, FAKE, 0, 1.0, 0) == gq.GQA_ERR_SHAPE
    assert q(FAKE + 2, FAKE, 16, 1.0, 0) == gq.GQA_ERR_ALIGN
    assert q(FAKE, FAKE, 16, 0.0, 0) == gq.GQA_ERR_SCALE


def test_bwd_specific_errors(lib):
    assert _bwd(dq=None) == gq.GQA_ERR_NULL
    assert _bwd(dout=None) == gq.GQA_ERR_NULL
    assert _bwd(dv=FAKE + 8) == gq.GQA_ERR_ALIGN
    assert _bwd(wsb=16) == gq.GQA_ERR_WORKSPACE
    assert _bwd(ws=FAKE + 4) == gq.GQA_ERR_ALIGN


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    import causal_grouped_query_gqa_b300._lib as L
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L, "_LIB_PATH", str(tmp_path / "libgqa_attn.so"))
    with pytest.raises(RuntimeError, match="missing"):
        L.load_library()


def test_cuda_failure_names_the_failing_call(lib):
    """Without a GPU, valid arguments reach the first CUDA call, which fails; the
    status is GQA_ERR_CUDA and the detail names the call and CUDA's reason."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("needs a host without a usable GPU")
    assert _fwd() == gq.GQA_ERR_CUDA
    detail = gq.gqa_attn_last_error_detail()
    assert detail.startswith("cudaGetDevice: ") and "cudaError" in detail
    with pytest.raises(gq.GqaError, match="cudaGetDevice"):
        raise gq.GqaError(gq.GQA_ERR_CUDA, "gqa_attn_fwd")
