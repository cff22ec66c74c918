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
flushed (256 MB written) before every timed step.

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
                "fwd_knorm_kernel"]
N_KERNELS = len(KERNEL_NAMES)
L2_FLUSH_BYTES = 256 << 20


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

def run_ours(args, w, rank, world, local_rank):
    import torch
    import causal_grouped_query_gqa_b300 as gq
    from causal_grouped_query_gqa_b300.inputs import make_inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the library has no CPU path)")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    gq.load_library()
    with_bwd = args.step == "fwd+bwd" or (
        args.step == "auto" and (w.backward or args.workload == DEFAULT_WORKLOAD))
    B, H, G, S, d = w.B, w.H, w.G, w.S, w.d
    kw = dict(causal=w.causal, window=w.window, n_sink=w.n_sink, scale=w.scale)

    # each rank owns its own shard of independent problems (different seeds)
    q_h, k_h, v_h, do_h = make_inputs(B, H, G, S, seed=rank, with_grad=True)
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = gq.gqa_attn_bwd_workspace_size(B, H, G, S, d)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    fws_bytes = gq.gqa_attn_fwd_workspace_size(B, H, G, S, d)
    fws = torch.empty(max(fws_bytes, 16), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step_on(ins, outs, strm):
        q_, k_, v_, do_ = ins
        o_, lse_, dq_, dk_, dv_ = outs
        rc = gq.gqa_attn_fwd_ws(q_, k_, v_, o_, lse_, B, H, G, S, d, w.causal, w.window,
                                w.n_sink, w.scale, fws, fws_bytes, strm)
        if rc != gq.GQA_OK:
            raise gq.GqaError(rc, "gqa_attn_fwd_ws")
        if with_bwd:
            rc = gq.gqa_attn_bwd(q_, k_, v_, o_, do_, lse_, dq_, dk_, dv_, B, H, G, S, d,
                                 w.causal, w.window, w.n_sink, w.scale, ws, ws_bytes, strm)
            if rc != gq.GQA_OK:
                raise gq.GqaError(rc, "gqa_attn_bwd")

    def step():
        step_on((q, k, v, do), (o, lse, dq, dk, dv), stream)

    launches_per_step = 2 + (3 if with_bwd else 0)  # key norms + forward, prep + main + convert
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if gq.gqa_attn_last_device_status() != gq.GQA_OK:
        raise SystemExit("device status error during warm-up")

    # ---- timed region: per-step events, kernel events from the library hooks
    gq.gqa_attn_timing_enable(1)
    kms = gq.timing_buffer()
    kernel_ms = [[] for _ in range(N_KERNELS)]
    step_ms = []
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    _barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        for s_i in range(args.steps):
            flush.zero_()
            ev[s_i][0].record(stream)
            step()
            ev[s_i][1].record(stream)
            gq.gqa_attn_timing_collect(kms)
            for kid in range(N_KERNELS):
                if kms[kid] >= 0:
                    kernel_ms[kid].append(float(kms[kid]))
        torch.cuda.synchronize()
    gq.gqa_attn_timing_enable(0)
    _barrier(world)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    if gq.gqa_attn_last_device_status() != gq.GQA_OK:
        raise SystemExit("device status error in the timed region")
    local_total_ms = sum(step_ms)
    total_ms = _max_over_ranks(local_total_ms, world)

    fwd_f, bwd_f = step_flops(w, with_bwd)
    flops_step = fwd_f + bwd_f
    value = job_throughput(flops_step, args.steps, total_ms, world)
    peaks = measured_peaks()

    # ---- dominant kernel roofline
    tot = [sum(x) for x in kernel_ms]
    dom = max(range(N_KERNELS), key=lambda kid: tot[kid])
    dom_avg_ms = tot[dom] / max(1, len(kernel_ms[dom]))
    dom_flops = {0: fwd_f, 2: bwd_f}.get(dom)
    if dom_flops:
        achieved = dom_flops / (dom_avg_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(achieved, 2),
                    "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": round(achieved / peaks["bf16_tflops"], 4),
                    "traffic": recorded_traffic(KERNEL_NAMES[dom], args.workload),
                    "kernel": KERNEL_NAMES[dom],
                    "peak_source": f"{peaks['source']} burst bf16 (MEASURED_PEAKS.json)",
                    "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4)}
    else:
        nbytes = bwd_bytes(w)
        achieved = nbytes / (dom_avg_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "traffic": None, "kernel": KERNEL_NAMES[dom]}
    kernels = {KERNEL_NAMES[kid]: round(tot[kid] / max(1, len(kernel_ms[kid])) * 1e3, 1)
               for kid in range(N_KERNELS) if kernel_ms[kid]}

    # ---- end to end through the same calls, host buffers
    e2e = run_e2e(args, dev, with_bwd, dev_in=(q, k, v, do), dev_out=(o, lse, dq, dk, dv),
                  host=(q_h, k_h, v_h, do_h), step_on=step_on, world=world, flops_step=flops_step)

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (bf16 iid N(0,1), torch CPU generator, seed = rank)",
        "config": {"workload": args.workload, "B": B, "H": H, "G": G, "S": S, "d": d,
                   "causal": w.causal, "window": w.window, "n_sink": w.n_sink,
                   "step": "fwd+bwd" if with_bwd else "fwd",
                   "l2": "flushed before every timed step (256 MB write, outside the events)",
                   "parallelism": f"replicas over ranks ({world}), no collective"},
        "pct_of_peak": round(100 * value / world / peaks["bf16_tflops"], 2),
        "fwd_tflops": round(fwd_f / (sum(kernels_ms_avg(kernel_ms, k) for k in (0, 4)) * 1e-3)
                            / 1e12, 2)
        if kernel_ms[0] else None,
        "bwd_tflops": round(bwd_f / (sum(kernels_ms_avg(kernel_ms, k) for k in (1, 2, 3)) * 1e-3)
                            / 1e12, 2) if with_bwd and kernel_ms[2] else None,
        "kernel_us": kernels,
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
    }
    return out


def kernels_ms_avg(kernel_ms, kid):
    x = kernel_ms[kid]
    return sum(x) / len(x) if x else 0.0


def run_e2e(args, dev, with_bwd, dev_in, dev_out, host, step_on, world, flops_step):
    """Same step with the inputs copied from pinned host memory and every output
    copied back, all inside the timed region.  Copies and compute run on three
    streams (upload, compute, download) over two sets of device tensors, so the
    upload of step i+1 and the download of step i-1 overlap the compute of
    step i, as a training or serving loop would arrange them."""
    import torch
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
        step_on(d_in, d_out, s_cmp)
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
