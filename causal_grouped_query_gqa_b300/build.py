"""Builds libgqa_attn.so in-tree with nvcc for sm_103a.

    python -m causal_grouped_query_gqa_b300.build [--force]

The library is plain CUDA C++ with an extern "C" interface (include/gqa_attn.h);
the CUDA runtime is linked statically, and the driver's tensor-map encoder is
fetched at run time, so the .so loads on a machine without a GPU.
"""
from __future__ import annotations

import argparse
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libgqa_attn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_cmd(out: str = LIB, extra=()):
    return ["nvcc", *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
            "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
            "-I", os.path.join(ROOT, "include"), *extra,
            os.path.join(CSRC, "gqa_attn_api.cu"), "-o", out, "-cudart", "static"]


def sources():
    return glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h")) + [os.path.abspath(__file__)]


def build(force: bool = False, verbose: bool = False, out: str = LIB, extra=()) -> str:
    if not force and os.path.exists(out):
        newest = max(os.path.getmtime(s) for s in sources())
        if os.path.getmtime(out) >= newest:
            return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = nvcc_cmd(tmp, extra)
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


# Failure-detection test build: CTA 0's producers skip one load and every wait
# gives up after 100 ms (see GQA_INJECT_STALL in the kernels).  Used only by
# tests/test_failure_detection.py; never loaded by the package.
STALL_TEST_LIB = os.path.join(PKG, "libgqa_attn_stalltest.so")
STALL_TEST_FLAGS = ("-DGQA_INJECT_STALL", "-DGQA_WAIT_BUDGET_NS=100000000ull")


def build_stall_test(force: bool = False, verbose: bool = False) -> str:
    return build(force=force, verbose=verbose, out=STALL_TEST_LIB, extra=STALL_TEST_FLAGS)


# Debug build with the kernels' run-time index checks (GQA_DEVICE_CHECKS): a
# violated check reports GQA_ERR_DEVICE_BOUNDS instead of touching memory.
# Used only by tests/test_device_checks.py.
CHECKED_LIB = os.path.join(PKG, "libgqa_attn_checked.so")


def build_checked(force: bool = False, verbose: bool = False) -> str:
    return build(force=force, verbose=verbose, out=CHECKED_LIB, extra=("-DGQA_DEVICE_CHECKS",))


# Test build whose backward writes dq, dk and dv as fp32 (GQA_FP32_GRAD_OUT):
# the gradients before the final bf16 rounding, for the tolerance tests of
# tests/test_grad_precision.py.  Never loaded by the package.
FP32_GRAD_LIB = os.path.join(PKG, "libgqa_attn_fp32grad.so")


def build_fp32_grad(force: bool = False, verbose: bool = False) -> str:
    return build(force=force, verbose=verbose, out=FP32_GRAD_LIB, extra=("-DGQA_FP32_GRAD_OUT",))


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--test-libs", action="store_true",
                    help="also build the failure-detection, index-check and fp32-gradient test libraries")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose))
    if a.test_libs:
        print(build_stall_test(force=a.force, verbose=a.verbose))
        print(build_checked(force=a.force, verbose=a.verbose))
        print(build_fp32_grad(force=a.force, verbose=a.verbose))
    sys.exit(0)
