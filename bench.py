#!/usr/bin/env python3
"""Benchmark of libgqa_attn: causal grouped-query attention, forward + backward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one pass of the whole path over one synthetic batch: the forward
(O, LSE) and the backward (dQ, dK, dV) for the same inputs, both through the
C ABI.  The default workload is B=1, H=128, G=16, S=8192, d=64, causal: the
shape at which the forward / backward targets are stated (S >= 8192).  Work is
counted as causal FLOPs: 4*d per visible (query, key) pair per head for the
forward and 2.5x that (10*d) for the backward.  The value is TFLOPS over the
whole job (all ranks), timed with CUDA events on the launching stream, L2
flushed (1 GiB written, which also keeps the GPU busy while the host
enqueues the step) before every timed step.

Also reported on the same JSON line: the roofline of the dominant kernel
(its own CUDA-event time inside the timed steps), the end-to-end number
through the same API with host buffers (H2D of the inputs and D2H of all
outputs inside the timed region), SM clocks sampled during the timed region,
and the float64 CPU oracle timed on a bounded sample of the same workload.

--impl reference times that oracle alone (the only reference this project
has: the pages ship no runnable implementation), on the same workload, metric
and unit.  Under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOPS (causal FLOPs) and % of B300 BF16 tensor peak"
KERNEL_NAMES = ["gqa_fwd_kernel", "bwd_prep_kernel", "bwd_main_kernel", "bwd_dq_convert_kernel",
                "fwd_knorm_kernel", "rope_table_and_rotation"]
N_KERNELS = len(KERNEL_NAMES)
L2_FLUSH_BYTES = 1 << 30


# ------------------------------------------------------------ FLOP counting ---

def visible_pairs(S: int, causal: bool, window: int, n_sink: int) -> int:
    """Number of visible (query, key) pairs of one head under the mask."""
    if not causal:
        return S * S
    total = 0
    if window <= 0:
        return S * (S + 1) // 2
    for i in range(S):
        in_window = min(i + 1, window)
        older = max(0, i + 1 - window)       # keys before the window start
        total += in_window + min(n_sink, older)
    return total


def step_flops(w, with_bwd: bool):
    pairs = visible_pairs(w.S, w.causal, w.window, w.n_sink) * w.B * w.H
    fwd = 4 * w.d * pairs
    bwd = 10 * w.d * pairs if with_bwd else 0
    return fwd, bwd


def fwd_bytes(w):
    """Algorithmic HBM bytes of one forward: Q, K, V, O (bf16) and LSE (fp32)."""
    return 2 * w.d * w.S * w.B * (2 * w.H + 2 * w.G) + 4 * w.B * w.H * w.S


def bwd_bytes(w):
    """Algorithmic HBM bytes of one backward: Q, K, V, O, dO, dQ, dK, dV (bf16),
    LSE, D (fp32) and one fp32 write + read of the dQ accumulator."""
    rows_h = w.B * w.H * w.S
    rows_g = w.B * w.G * w.S
    return 2 * w.d * (4 * rows_h + 4 * rows_g) + 8 * rows_h + 8 * w.d * rows_h


# ------------------------------------------------------------------- helpers ---

def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "hbm_gbs": 6400.0,
                "source": "fallback"}


def source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "causal_grouped_query_gqa_b300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        e = rec[kernel][workload]
        if e.get("source_hash") == source_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks / throttle reasons while it runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.out = None

    def summary(self):
        if not self.out:
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- our arm ---

class Problem:
    """Device tensors of one workload and the calls of one step (through the C ABI)."""

    def __init__(self, w, dev, seed, with_bwd, yarn=False, fp8=False, outliers=False, yarn_mode=0):
        import torch
        import causal_grouped_query_gqa_b300 as gq
        from causal_grouped_query_gqa_b300.inputs import make_inputs
        self.w, self.dev, self.with_bwd = w, dev, with_bwd
        B, H, G, S, d = w.B, w.H, w.G, w.S, w.d
        self.host = make_inputs(B, H, G, S, seed=seed, with_grad=True)
        if outliers:  # rows 0..31 of every 128-row block 8x larger: a quarter of the warps
            # then exceed the score bound and take the exact step (8x is exact in bf16)
            self.host[0][:, :, torch.arange(S) % 128 < 32] *= 8
        self.ins = tuple(t.to(dev) for t in self.host)
        q = self.ins[0]
        self.outs = (torch.empty_like(q), torch.empty((B, H, S), dtype=torch.float32, device=dev),
                     torch.empty_like(q), torch.empty_like(self.ins[1]),
                     torch.empty_like(self.ins[2]))
        self.ws_bytes = gq.gqa_attn_bwd_workspace_size(B, H, G, S, d)
        self.ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=dev)
        self.fws_bytes = gq.gqa_attn_fwd_workspace_size(B, H, G, S, d)
        self.fws = torch.empty(max(self.fws_bytes, 16), dtype=torch.uint8, device=dev)
        # the forward entry point the library's own fwd() picks for this size
        fwd_f, _ = step_flops(w, False)
        self.score_bound = fwd_f >= gq.SCORE_BOUND_MIN_FLOPS
        # the fp8 forward: q and k quantised once to E4M3 (before any timing)
        self.fp8 = fp8
        if fp8:
            self.score_bound = False
            self.q8, self.k8 = torch.empty_like(q, dtype=torch.uint8), torch.empty_like(
                self.ins[1], dtype=torch.uint8)
            self.fp8_scales = []
            for src, dst in ((q, self.q8), (self.ins[1], self.k8)):
                inv = 440.0 / float(src.float().abs().max())
                dst.copy_(gq.quantize_e4m3(src, inv))
                self.fp8_scales.append(1.0 / inv)
        # the YaRN forward (rotary embeddings on q and k) instead of the plain one
        self.yarn = yarn
        if yarn:
            self.yarn_mode = yarn_mode  # rotate q and k in a pre-pass (0) or q inside the forward (1)
            self.yws_bytes = gq.gqa_attn_fwd_yarn_workspace_size(B, H, G, S, d, yarn_mode)
            self.yws = torch.empty(max(self.yws_bytes, 16), dtype=torch.uint8, device=dev)

    def step_on(self, ins, outs, strm, score_bound=None):
        import causal_grouped_query_gqa_b300 as gq
        w = self.w
        B, H, G, S, d = w.B, w.H, w.G, w.S, w.d
        q_, k_, v_, do_ = ins
        o_, lse_, dq_, dk_, dv_ = outs
        bound = self.score_bound if score_bound is None else score_bound
        if self.fp8:
            rc = gq.gqa_attn_fwd_fp8(self.q8, self.k8, v_, o_, lse_, B, H, G, S, d, w.causal,
                                     w.window, w.n_sink, w.scale, self.fp8_scales[0],
                                     self.fp8_scales[1], strm)
        elif self.yarn:
            y = gq.YARN_DEFAULTS
            rc = gq.gqa_attn_fwd_yarn(q_, k_, v_, o_, lse_, B, H, G, S, d, w.causal, w.window,
                                      w.n_sink, w.scale, y["rope_base"], y["rope_factor"],
                                      y["rope_orig_ctx"], y["rope_alpha"], y["rope_beta"],
                                      bound, self.yarn_mode, self.yws, self.yws_bytes, strm)
        elif bound:
            rc = gq.gqa_attn_fwd_ws(q_, k_, v_, o_, lse_, B, H, G, S, d, w.causal, w.window,
                                    w.n_sink, w.scale, self.fws, self.fws_bytes, strm)
        else:
            rc = gq.gqa_attn_fwd(q_, k_, v_, o_, lse_, B, H, G, S, d, w.causal, w.window,
                                 w.n_sink, w.scale, strm)
        if rc != gq.GQA_OK:
            raise gq.GqaError(rc, "forward")
        if self.with_bwd:
            rc = gq.gqa_attn_bwd(q_, k_, v_, o_, do_, lse_, dq_, dk_, dv_, B, H, G, S, d,
                                 w.causal, w.window, w.n_sink, w.scale, self.ws, self.ws_bytes,
                                 strm)
            if rc != gq.GQA_OK:
                raise gq.GqaError(rc, "gqa_attn_bwd")

    def launches_per_step(self, score_bound=None):
        bound = self.score_bound if score_bound is None else score_bound
        fwd_launches = 1 + (1 if bound and not self.fp8 else 0) + (2 if self.yarn else 0)
        return fwd_launches + (4 if self.with_bwd else 0)


def timed_steps(pb, steps, warmup, flush, stream, world, score_bound=None, clocks=False):
    """Times `steps` steps of `pb` with CUDA events on `stream`, L2 flushed before
    each step outside the events.  Returns (total ms, per-kernel ms lists, clocks)."""
    import torch
    import causal_grouped_query_gqa_b300 as gq

    def step():
        pb.step_on(pb.ins, pb.outs, stream, score_bound)

    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if gq.gqa_attn_last_device_status() != gq.GQA_OK:
        raise SystemExit("device status error during warm-up")
    gq.gqa_attn_timing_enable(1)
    kms = gq.timing_buffer()
    kernel_ms = [[] for _ in range(N_KERNELS)]
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    _barrier(world)
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device()) if clocks else None
    if sampler:
        sampler.__enter__()
    try:
        for s_i in range(steps):
            flush.zero_()
            ev[s_i][0].record(stream)
            step()
            ev[s_i][1].record(stream)
            gq.gqa_attn_timing_collect(kms)
            for kid in range(N_KERNELS):
                if kms[kid] >= 0:
                    kernel_ms[kid].append(float(kms[kid]))
        torch.cuda.synchronize()
    finally:
        if sampler:
            sampler.__exit__(None, None, None)
    gq.gqa_attn_timing_enable(0)
    _barrier(world)
    if gq.gqa_attn_last_device_status() != gq.GQA_OK:
        raise SystemExit("device status error in the timed region")
    total = sum(a.elapsed_time(b) for a, b in ev)
    return total, kernel_ms, (sampler.summary() if sampler else None)


def tensor_roofline(kernel, flops, ms, peaks, workload):
    achieved = flops / (ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
            "traffic": recorded_traffic(kernel, workload), "kernel": kernel,
            "peak_source": f"{peaks['source']} burst bf16 (MEASURED_PEAKS.json)",
            "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4)}


def summarize(w, pb, kernel_ms, total_ms, steps, world, peaks, workload):
    fwd_f, bwd_f = step_flops(w, pb.with_bwd)
    avg = {kid: kernels_ms_avg(kernel_ms, kid) for kid in range(N_KERNELS)}
    fwd_ms = avg[0] + avg[4] + avg[5]
    bwd_ms = avg[1] + avg[2] + avg[3]
    tot = [sum(x) for x in kernel_ms]
    dom = max(range(N_KERNELS), key=lambda kid: tot[kid])
    dom_flops = {0: fwd_f, 2: bwd_f}.get(dom)
    if dom_flops:
        roofline = tensor_roofline(KERNEL_NAMES[dom], dom_flops, avg[dom], peaks, workload)
    else:
        nbytes = bwd_bytes(w)
        achieved = nbytes / (avg[dom] * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "traffic": None, "kernel": KERNEL_NAMES[dom]}
    out = {
        "value": round(job_throughput(fwd_f + bwd_f, steps, total_ms, world), 2),
        "ms_per_step": round(total_ms / steps, 4),
        "fwd_tflops": round(fwd_f / (fwd_ms * 1e-3) / 1e12, 2) if fwd_ms > 0 else None,
        "bwd_tflops": round(bwd_f / (bwd_ms * 1e-3) / 1e12, 2) if pb.with_bwd and bwd_ms > 0
        else None,
        "fwd_score_bound": pb.score_bound,
        "kernel_us": {KERNEL_NAMES[kid]: round(avg[kid] * 1e3, 1)
                      for kid in range(N_KERNELS) if kernel_ms[kid]},
        "roofline": roofline,
    }
    if avg[0] > 0:
        fb = fwd_bytes(w)
        gbs = fb / (avg[0] * 1e-3) / 1e9
        out["fwd_hbm"] = {"achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                          "frac": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": fb,
                          "kernel": "gqa_fwd_kernel"}
    for kid, nbytes in ((4, knorm_bytes(w)), (1, prep_bytes(w)), (3, convert_bytes(w)),
                       (5, rope_bytes(w, getattr(pb, "yarn_mode", 0)))):
        if avg[kid] > 0:
            gbs = nbytes / (avg[kid] * 1e-3) / 1e9
            out.setdefault("hbm_kernels", {})[KERNEL_NAMES[kid]] = {
                "achieved": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4),
                "algorithmic_bytes": nbytes, "unit": "GB/s"}
    return out


def run_ours(args, w, rank, world, local_rank):
    import torch
    import causal_grouped_query_gqa_b300 as gq
    from causal_grouped_query_gqa_b300.inputs import WORKLOADS

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the library has no CPU path)")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    gq.load_library()
    with_bwd = args.step == "fwd+bwd" or (
        args.step == "auto" and (w.backward or args.workload == DEFAULT_WORKLOAD))
    # each rank owns its own shard of independent problems (different seeds)
    pb = Problem(w, dev, seed=rank, with_bwd=with_bwd)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    peaks = measured_peaks()

    total_ms, kernel_ms, clocks = timed_steps(pb, args.steps, args.warmup, flush, stream, world,
                                              clocks=True)
    total_ms = _max_over_ranks(total_ms, world)
    main = summarize(w, pb, kernel_ms, total_ms, args.steps, world, peaks, args.workload)

    # the plain forward (gqa_attn_fwd: the online maximum on every tile, any input)
    fwd_only = Problem.__new__(Problem)
    fwd_only.__dict__.update(pb.__dict__)
    fwd_only.with_bwd = False
    p_ms, p_kernel, _ = timed_steps(fwd_only, args.steps, args.warmup, flush, stream, world,
                                    score_bound=False)
    fwd_f, bwd_f = step_flops(w, with_bwd)
    plain_ms = kernels_ms_avg(p_kernel, 0)
    fwd_plain = {"tflops": round(fwd_f / (plain_ms * 1e-3) / 1e12, 2),
                 "kernel_us": round(plain_ms * 1e3, 1),
                 "frac": round(fwd_f / (plain_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                 "entry": "gqa_attn_fwd"}

    # ---- end to end through the same calls, host buffers
    e2e = run_e2e(args, dev, pb, world=world, flops_step=fwd_f + bwd_f)

    out = {
        "metric": METRIC, "value": main["value"], "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": main["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (bf16 iid N(0,1), torch CPU generator, seed = rank)",
        "config": {"workload": args.workload, "B": w.B, "H": w.H, "G": w.G, "S": w.S, "d": w.d,
                   "causal": w.causal, "window": w.window, "n_sink": w.n_sink,
                   "step": "fwd+bwd" if with_bwd else "fwd",
                   "l2": "flushed before every timed step (1 GiB write, outside the events)",
                   "parallelism": f"replicas over ranks ({world}), no collective"},
        "pct_of_peak": round(100 * main["value"] / world / peaks["bf16_tflops"], 2),
        "fwd_tflops": main["fwd_tflops"], "bwd_tflops": main["bwd_tflops"],
        "fwd_score_bound": main["fwd_score_bound"],
        "fwd_plain_tflops": fwd_plain["tflops"], "fwd_plain": fwd_plain,
        "kernel_us": main["kernel_us"],
        "roofline": main["roofline"],
        "hbm_kernels": main.get("hbm_kernels"),
        "e2e": e2e,
        "gpu_launches": pb.launches_per_step() * args.steps,
        "clocks": clocks,
    }

    # ---- the other stated workloads, a few steps each (rank 0, after the timed region)
    if rank == 0 and not args.no_extra and args.workload == DEFAULT_WORKLOAD:
        extras = {}
        for name, step in EXTRA_WORKLOADS:
            ew = WORKLOADS[name]
            epb = Problem(ew, dev, seed=0, with_bwd=(step == "fwd+bwd"),
                          yarn=step.startswith("fwd_yarn"), fp8=(step == "fwd_fp8"),
                          outliers=step.startswith("fwd_outliers"),
                          yarn_mode=1 if step == "fwd_yarn_fused" else 0)
            if step == "fwd_outliers_plain":
                epb.score_bound = False
            e_steps = max(3, min(args.steps, 10))
            e_ms, e_kernel, e_clk = timed_steps(epb, e_steps, 3, flush, stream, 1, clocks=True)
            res = summarize(ew, epb, e_kernel, e_ms, e_steps, 1, peaks, name)
            res.update({"step": step, "steps": e_steps, "clocks": e_clk,
                        "config": {"B": ew.B, "H": ew.H, "G": ew.G, "S": ew.S,
                                   "window": ew.window, "n_sink": ew.n_sink}})
            extras[extra_key(name, step, extras)] = res
            del epb
            torch.cuda.empty_cache()
        out["extra_workloads"] = extras
    return out


EXTRA_STEPS = ("fwd", "fwd+bwd", "fwd_yarn", "fwd_yarn_fused", "fwd_fp8", "fwd_outliers",
               "fwd_outliers_plain")


def extra_key(name, step, taken):
    """Key of an extra workload's entry in the JSON line: the workload's name,
    a suffix for the variant steps, and the step itself when the plain key is
    already taken by the same workload measured with another step."""
    key = name + {"fwd_yarn": "+yarn", "fwd_yarn_fused": "+yarn_fused", "fwd_fp8": "+fp8",
                  "fwd_outliers": "+outlier_rows",
                  "fwd_outliers_plain": "+outlier_rows_plain"}.get(step, "")
    if key in taken:
        key = name + "+" + step.replace("+", "_")
    return key


# The stated workloads besides the default one, measured in the same run
# (the default line's value is unaffected).
EXTRA_WORKLOADS = [
    ("gqa_b2_h32_g8_s2048", "fwd"),
    ("window_b1_h128_g16_s32768_w4096_sink128", "fwd"),
    ("bwd_b4_h32_g8_s4096", "fwd+bwd"),
    ("window_b1_h128_g16_s32768_w4096_sink128", "fwd+bwd"),  # the window + sink backward at S = 32768
    ("model_b1_h128_g16_s204800_w65536_sink2048", "fwd+bwd"),  # the model's mask at S = 204800
    ("wide_b1_h128_g16_s8192", "fwd_yarn"),   # YaRN rotary forward (table, q and k rotation, forward)
    ("wide_b1_h128_g16_s8192", "fwd_yarn_fused"),  # the same, query tiles rotated inside the forward
    ("wide_b1_h128_g16_s8192", "fwd_fp8"),    # E4M3 queries and keys (quantised before timing)
    ("wide_b1_h128_g16_s8192", "fwd_outliers"),  # score bound with a quarter of the warps exact
    ("wide_b1_h128_g16_s8192", "fwd_outliers_plain"),  # the same input through gqa_attn_fwd
]


def knorm_bytes(w):
    """Key-norm pre-pass: reads K, writes one 128-byte record per kv head."""
    return 2 * w.d * w.S * w.B * w.G + 128 * w.B * w.G


def rope_bytes(w, mode=0):
    """Rotary pre-pass: writes the (cos, sin) table ([S][32] float2), reads k and,
    in the pre-pass mode (0), q (bf16) and writes their rotations (bf16); the
    fused mode (1) rotates q inside the forward."""
    heads = w.H + w.G if mode == 0 else w.G
    return 8 * 32 * w.S + 2 * 2 * w.d * w.S * w.B * heads


def prep_bytes(w):
    """Backward prep and shift: read O, dO (bf16) and LSE; write D and LSE2
    (fp32), the fp16 copy of dO, and clear the fp32 dQ accumulator; then read and
    write LSE2 once more."""
    rows = w.B * w.H * w.S
    return 2 * 2 * w.d * rows + 4 * rows + 8 * rows + 4 * w.d * rows + 2 * w.d * rows + 8 * rows


def convert_bytes(w):
    """dQ convert: reads the fp32 accumulator, writes bf16 dQ."""
    rows = w.B * w.H * w.S
    return 6 * w.d * rows


def kernels_ms_avg(kernel_ms, kid):
    x = kernel_ms[kid]
    return sum(x) / len(x) if x else 0.0


def run_e2e(args, dev, pb, world, flops_step):
    """Same step with the inputs copied from pinned host memory and every output
    copied back, all inside the timed region.  Copies and compute run on three
    streams (upload, compute, download) over two sets of device tensors, so the
    upload of step i+1 and the download of step i-1 overlap the compute of
    step i, as a training or serving loop would arrange them."""
    import torch
    with_bwd = pb.with_bwd
    dev_in, dev_out, host = pb.ins, pb.outs, pb.host
    n_in = 4 if with_bwd else 3
    n_out = 5 if with_bwd else 2
    sets = [(list(dev_in), list(dev_out)),
            ([torch.empty_like(t) for t in dev_in], [torch.empty_like(t) for t in dev_out])]
    ins = [t.pin_memory() for t in host[:n_in]]
    outs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dev_out[:n_out]]
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = sum(t.numel() * t.element_size() for t in outs)
    s_up, s_cmp, s_down = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event(enable_timing=False)
    in_ready, cmp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def e2e_step(i):
        b = i & 1
        d_in, d_out = sets[b]
        with torch.cuda.stream(s_up):
            s_up.wait_event(cmp_done[b])  # step i-2 has finished reading this input set
            for dst, src in zip(d_in[:n_in], ins):
                dst.copy_(src, non_blocking=True)
            in_ready[b].record(s_up)
        s_cmp.wait_event(in_ready[b])
        s_cmp.wait_event(out_done[b])  # step i-2's outputs of this set are downloaded
        pb.step_on(d_in, d_out, s_cmp)
        cmp_done[b].record(s_cmp)
        with torch.cuda.stream(s_down):
            s_down.wait_event(cmp_done[b])
            for dst, src in zip(outs, d_out[:n_out]):
                dst.copy_(src, non_blocking=True)
            out_done[b].record(s_down)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    n = args.steps
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize()
    a.record(s_up)
    for i in range(n):
        e2e_step(i)
    b.record(s_down)
    torch.cuda.synchronize()
    ms = _max_over_ranks(a.elapsed_time(b), world)
    val = job_throughput(flops_step, n, ms, world)
    return {"value": round(val, 2), "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms / n, 4),
            "overlap": "upload, compute and download on three streams, two device tensor sets"}


# ------------------------------------------------------- reference (oracle) ---

def oracle_sample(w, target_s: float, seed: int = 0):
    """Times the float64 oracle on a bounded sample of the workload: the last
    rows of every query head of kv group (b=0, g=0), forward and backward,
    sized for about `target_s` seconds.  Returns (counted FLOPs, seconds, text)."""
    import numpy as np
    import oracle
    import torch
    from causal_grouped_query_gqa_b300.inputs import make_inputs

    q, k, v, do = make_inputs(1, w.H // w.G, 1, w.S, w.d, seed=seed, with_grad=True)
    q, k, v, do = (t.to(torch.float64).numpy() for t in (q, k, v, do))
    R = w.H // w.G

    def pairs_of(i0, i1):
        return sum(_row_pairs(i, w) for i in range(i0, i1))

    # calibrate on a few rows, then size the sample
    n0 = min(w.S, 8)
    t0 = time.perf_counter()
    oracle.attn_fwd_rows(q, k, v, [(0, h, i) for h in range(R) for i in range(w.S - n0, w.S)],
                         causal=w.causal, window=w.window, n_sink=w.n_sink, scale=w.scale)
    oracle.attn_bwd_group_rows(q, k, v, do, 0, 0, w.S - n0, w.S, causal=w.causal,
                               window=w.window, n_sink=w.n_sink, scale=w.scale)
    dt0 = max(time.perf_counter() - t0, 1e-4)
    n_rows = int(min(w.S, max(n0, n0 * target_s / dt0)))
    i0 = w.S - n_rows
    t0 = time.perf_counter()
    oracle.attn_fwd_rows(q, k, v, [(0, h, i) for h in range(R) for i in range(i0, w.S)],
                         causal=w.causal, window=w.window, n_sink=w.n_sink, scale=w.scale)
    oracle.attn_bwd_group_rows(q, k, v, do, 0, 0, i0, w.S, causal=w.causal, window=w.window,
                               n_sink=w.n_sink, scale=w.scale)
    secs = time.perf_counter() - t0
    flops = 14 * w.d * R * pairs_of(i0, w.S)
    text = (f"kv group (b=0, g=0): its {R} query heads, query rows {i0}..{w.S - 1} of {w.S}, "
            f"forward + backward, float64 oracle")
    return flops, secs, text, oracle.num_threads()


def _row_pairs(i, w):
    if not w.causal:
        return w.S
    if w.window <= 0:
        return i + 1
    return min(i + 1, w.window) + min(w.n_sink, max(0, i + 1 - w.window))


def run_reference(args, w):
    per_step = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, per_step)
    fl, secs, text, cores = 0, 0.0, "", 1
    for _ in range(args.steps):
        f, s, text, cores = oracle_sample(w, per_step)
        fl += f
        secs += s
    value = fl / secs / 1e12
    return {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (bf16 iid N(0,1) widened to float64)",
        "config": {"workload": args.workload, "B": w.B, "H": w.H, "G": w.G, "S": w.S, "d": w.d,
                   "causal": w.causal, "window": w.window, "n_sink": w.n_sink,
                   "step": "fwd+bwd on a bounded sample"},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": text},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# -------------------------------------------------------------- distributed ---

def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _init_dist(world, use_cuda):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("nccl" if use_cuda else "gloo")


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x: float, world: int) -> float:
    """Slowest rank's time: the job's time (timing reduction only, no data path)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank_step: float, steps: int, max_ms: float, world: int) -> float:
    """Whole-job TFLOPS: the work of every rank divided by the slowest rank's time."""
    return world * flops_per_rank_step * steps / (max_ms * 1e-3) / 1e12


DEFAULT_WORKLOAD = "wide_b1_h128_g16_s8192"


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--step", choices=["auto", "fwd", "fwd+bwd"], default="auto",
                    help="what one step runs; auto: fwd+bwd on the default workload and on "
                         "workloads stated with a backward, else fwd")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip timing the oracle (profiling runs only)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other stated workloads (profiling runs only)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from causal_grouped_query_gqa_b300.inputs import WORKLOADS
    if args.workload not in WORKLOADS:
        ap.error(f"unknown workload {args.workload}; one of {sorted(WORKLOADS)}")
    w = WORKLOADS[args.workload]
    world, rank, local = _dist_env()

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, w)), flush=True)
        return 0

    _init_dist(world, use_cuda=True)
    out = run_ours(args, w, rank, world, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            fl, secs, text, cores = oracle_sample(w, 15.0)
            out["cpu_baseline"] = {"value": fl / secs / 1e12, "unit": "TFLOPS", "cores": cores,
                                   "kind": "oracle", "sample": text}
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
