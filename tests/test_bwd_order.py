"""The backward's CTA order (csrc/bwd_order.cuh), checked on the host.

A host program built from the header alone enumerates every CTA of a launch
and prints its (key tile, kv head) unit; the order must visit every unit once,
run the sink key tiles of a windowed mask first (key-tile-major over every kv
head), keep each batch of kv heads contiguous, and run each batch
key-tile-major.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "causal_grouped_query_gqa_b300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <cstdlib>
#include "bwd_order.cuh"
int main(int argc, char **argv) {
  const int B = atoi(argv[1]), G = atoi(argv[2]), R = atoi(argv[3]), S = atoi(argv[4]);
  const int sms = atoi(argv[5]), window = atoi(argv[6]), n_sink = atoi(argv[7]);
  const int nk = (S + 127) / 128;
  const int nf = gqa::bwd::front_tiles(nk, window, n_sink, 128);
  int n_small, bp;
  gqa::bwd::cta_order(B, G, R, S, nk, nf, sms, n_small, bp);
  printf("%d %d %d\n", n_small, bp, nf);
  for (int u = 0; u < nk * B * G; ++u) {
    int kb, pair;
    gqa::bwd::cta_unit(u, nk, nf, B * G, n_small, bp, kb, pair);
    printf("%d %d\n", kb, pair);
  }
  return 0;
}
"""


@pytest.fixture(scope="module")
def order_exe(tmp_path_factory):
    if shutil.which("nvcc") is None:
        pytest.skip("nvcc not found")
    d = tmp_path_factory.mktemp("order")
    src = d / "order.cu"
    src.write_text(PROGRAM)
    exe = d / "order"
    subprocess.run(["nvcc", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    return str(exe)


def _order(exe, B, G, R, S, sms=148, window=0, n_sink=0, front=False):
    out = subprocess.run([exe, str(B), str(G), str(R), str(S), str(sms), str(window), str(n_sink)],
                         check=True, capture_output=True, text=True).stdout.split("\n")
    n_small, bp, nf = map(int, out[0].split())
    units = [tuple(map(int, line.split())) for line in out[1:] if line]
    return (n_small, bp, units, nf) if front else (n_small, bp, units)


@pytest.mark.parametrize("B,G,R,S", [
    (1, 16, 8, 8192),    # 4 batches of 4 kv heads
    (4, 8, 4, 4096),     # 2 batches of 16
    (2, 8, 4, 2048),     # one batch: the whole launch key-tile-major
    (1, 16, 8, 32768),   # one kv head a batch
    (1, 1, 8, 130),      # a single kv head, ragged key tiles
    (3, 5, 2, 1000),     # uneven batch sizes
    (7, 3, 16, 20000),
    (1, 16, 8, 204800),  # the longest stated sequence
    (4, 4, 16, 4096),    # batches of 5, 5 and 6
])
def test_order_is_a_bijection_in_key_tile_major_batches(order_exe, B, G, R, S):
    n_small, bp, units = _order(order_exe, B, G, R, S)
    nk, pairs = -(-S // 128), B * G
    assert len(units) == nk * pairs
    assert sorted(units) == [(kb, p) for kb in range(nk) for p in range(pairs)]
    sizes = [bp] * n_small + [bp + 1] * ((pairs - n_small * bp) // (bp + 1))
    assert sum(sizes) == pairs and n_small >= 1 and bp >= 1
    pos = 0
    first = 0
    for sz in sizes:
        batch = units[pos:pos + sz * nk]
        # the batch covers pairs [first, first + sz), key tile by key tile
        assert [kb for kb, _ in batch] == [kb for kb in range(nk) for _ in range(sz)]
        assert [p for _, p in batch] == list(range(first, first + sz)) * nk
        pos += sz * nk
        first += sz
    assert pos == len(units)


def test_batch_sizes_follow_the_row_budget(order_exe):
    """About 136 MiB of Q, dO and dQ rows a batch (R * S * 512 bytes a kv head),
    no fewer than 1.5 * SMs / (key tiles + 1) kv heads, at most all of them."""
    assert _order(order_exe, 1, 16, 8, 8192)[:2] == (4, 4)      # 33.5 MB a head
    assert _order(order_exe, 4, 8, 4, 4096)[:2] == (2, 16)      # 8.4 MB a head
    assert _order(order_exe, 1, 16, 8, 32768)[:2] == (16, 1)    # 134 MB a head
    assert _order(order_exe, 2, 8, 4, 2048)[:2] == (1, 16)      # all in one batch
    # 16 kv heads of 33.5 MB: the budget allows 4, 32 key tiles ask for
    # ceil(222 / 33) = 7, so 3 batches: 5, 5, 6 (the GPU parity test's shape)
    assert _order(order_exe, 4, 4, 16, 4096)[:2] == (2, 5)
    # the floor: 8 kv heads of 268 MB each at S = 65536 would be one a batch by
    # the budget; 512 key tiles ask for ceil(1.5 * 148 / 513) = 1 -- unchanged
    assert _order(order_exe, 1, 8, 8, 65536)[:2] == (8, 1)
    # many query heads on a short sequence: 67 MB a kv head allows 2 by the
    # budget, but 16 key tiles ask for ceil(1.5 * 148 / 17) = 14, so the 16
    # kv heads go in 2 batches of 8
    assert _order(order_exe, 1, 16, 64, 2048)[:2] == (2, 8)
    # the floor on uneven sizes: 268 MB a kv head, 8 key tiles -> at least
    # ceil(222 / 9) = 25 of the 64, so 3 batches: 21, 21, 22
    assert _order(order_exe, 1, 64, 512, 1024)[:2] == (2, 21)


@pytest.mark.parametrize("B,G,R,S,window,n_sink,nf", [
    (1, 16, 8, 32768, 4096, 128, 1),       # the window workload: key tile 0 holds the 128 sinks
    (1, 16, 8, 204800, 65536, 2048, 16),   # the model's mask: 16 sink key tiles a kv head
    (2, 3, 4, 1000, 300, 200, 2),          # sinks ending inside the second key tile
    (1, 2, 4, 300, 100, 1000, 3),          # sinks past the sequence: every key tile in front
    (1, 16, 8, 8192, 4096, 0, 0),          # a window without sinks: no front
    (1, 16, 8, 8192, 0, 64, 0),            # sinks without a window are plain causal keys
])
def test_sink_key_tiles_run_first(order_exe, B, G, R, S, window, n_sink, nf):
    n_small, bp, units, got_nf = _order(order_exe, B, G, R, S, window=window, n_sink=n_sink,
                                        front=True)
    nk, pairs = -(-S // 128), B * G
    assert got_nf == nf
    assert len(units) == nk * pairs
    assert sorted(units) == [(kb, p) for kb in range(nk) for p in range(pairs)]
    # the front: key tiles 0 .. nf-1 of every kv head, key tile by key tile
    assert units[:nf * pairs] == [(kb, p) for kb in range(nf) for p in range(pairs)]
    rest, nk2 = units[nf * pairs:], nk - nf
    if nk2 == 0:
        assert not rest
        return
    sizes = [bp] * n_small + [bp + 1] * ((pairs - n_small * bp) // (bp + 1))
    assert sum(sizes) == pairs
    pos = first = 0
    for sz in sizes:
        batch = rest[pos:pos + sz * nk2]
        assert [kb for kb, _ in batch] == [kb for kb in range(nf, nk) for _ in range(sz)]
        assert [p for _, p in batch] == list(range(first, first + sz)) * nk2
        pos += sz * nk2
        first += sz
    assert pos == len(rest)
