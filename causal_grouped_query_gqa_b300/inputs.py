"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic, so both the CUDA path and the float64 oracle can be fed
from it without sharing any of the method.

Recipe (the workloads are stated as "bf16 iid N(0,1), seed 0"):
  * a CPU ``torch.Generator`` seeded with ``seed``;
  * float32 standard normals drawn in the fixed order q, k, v, dO;
  * each cast to bfloat16 (round to nearest even).
The same bf16 tensors go to the GPU, and their exact float64 widening goes to
the oracle.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    """One attention problem: sizes and mask parameters."""
    name: str
    B: int
    H: int
    G: int
    S: int
    d: int = 64
    causal: bool = True
    window: int = 0
    n_sink: int = 0
    backward: bool = False

    @property
    def scale(self) -> float:
        return 1.0 / float(self.d) ** 0.5


# The workloads the library is measured and checked on: five stated ones, and
# the model-spec mask (window 65536, 2048 sinks) at its longest context.
WORKLOADS = {
    "tiny_b1_h4_g2_s128": Workload("tiny_b1_h4_g2_s128", 1, 4, 2, 128, backward=True),
    "gqa_b2_h32_g8_s2048": Workload("gqa_b2_h32_g8_s2048", 2, 32, 8, 2048),
    "wide_b1_h128_g16_s8192": Workload("wide_b1_h128_g16_s8192", 1, 128, 16, 8192),
    "window_b1_h128_g16_s32768_w4096_sink128": Workload(
        "window_b1_h128_g16_s32768_w4096_sink128", 1, 128, 16, 32768, window=4096, n_sink=128),
    "bwd_b4_h32_g8_s4096": Workload("bwd_b4_h32_g8_s4096", 4, 32, 8, 4096, backward=True),
    "model_b1_h128_g16_s204800_w65536_sink2048": Workload(
        "model_b1_h128_g16_s204800_w65536_sink2048", 1, 128, 16, 204800, window=65536,
        n_sink=2048, backward=True),
}


def make_inputs(B: int, H: int, G: int, S: int, d: int = 64, *, seed: int = 0,
                with_grad: bool = False, device: str | torch.device = "cpu"):
    """Draw q [B,H,S,d], k,v [B,G,S,d] (and dO [B,H,S,d]) as bf16, in that order."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    q = torch.randn((B, H, S, d), generator=gen, dtype=torch.float32)
    k = torch.randn((B, G, S, d), generator=gen, dtype=torch.float32)
    v = torch.randn((B, G, S, d), generator=gen, dtype=torch.float32)
    out = [q, k, v]
    if with_grad:
        out.append(torch.randn((B, H, S, d), generator=gen, dtype=torch.float32))
    return tuple(t.to(torch.bfloat16).to(device) for t in out)
