"""Host logic of bench.py that needs no GPU: FLOP counting against the oracle's
mask, and the multi-rank timing reduction on 2 gloo ranks (CPU)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench
import oracle
from causal_grouped_query_gqa_b300.inputs import WORKLOADS


@pytest.mark.parametrize("S,causal,window,n_sink", [
    (50, True, 0, 0), (50, False, 0, 0), (60, True, 7, 3), (60, True, 1, 0), (40, True, 8, 20),
])
def test_visible_pairs_matches_mask(S, causal, window, n_sink):
    brute = sum(oracle.visible(i, j, causal=causal, window=window, n_sink=n_sink)
                for i in range(S) for j in range(S))
    assert bench.visible_pairs(S, causal, window, n_sink) == brute


def test_workload_flops():
    w = WORKLOADS["wide_b1_h128_g16_s8192"]
    fwd, bwd = bench.step_flops(w, True)
    assert fwd == 4 * 64 * 128 * 8192 * 8193 // 2
    assert bwd == 2.5 * fwd
    w4 = WORKLOADS["window_b1_h128_g16_s32768_w4096_sink128"]
    assert abs(bench.step_flops(w4, False)[0] / 4.2432e12 - 1) < 1e-4


def test_extra_workloads_are_known_and_keyed_apart():
    """Every extra workload of the bench line names a stated workload and a
    step the bench knows, and no two share a key in the JSON line."""
    keys = {}
    for name, step in bench.EXTRA_WORKLOADS:
        assert name in WORKLOADS and step in bench.EXTRA_STEPS
        keys[bench.extra_key(name, step, keys)] = (name, step)
    assert len(keys) == len(bench.EXTRA_WORKLOADS)
    assert keys["window_b1_h128_g16_s32768_w4096_sink128"][1] == "fwd"
    assert keys["window_b1_h128_g16_s32768_w4096_sink128+fwd_bwd"][1] == "fwd+bwd"


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench._barrier(world)
    slowest = bench._max_over_ranks(times[rank], world)
    out[rank] = slowest
    dist.destroy_process_group()


def test_two_rank_timing_reduction_gloo():
    world, port = 2, _free_port()
    times = [12.5, 20.0]
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, port, times, out), nprocs=world,
                       start_method="spawn", join=True)
    assert out[0] == out[1] == 20.0
    # every rank's work over the slowest rank's time
    v = bench.job_throughput(1e12, 10, out[0], world)
    assert abs(v - 2 * 1e12 * 10 / 0.020 / 1e12) < 1e-9
