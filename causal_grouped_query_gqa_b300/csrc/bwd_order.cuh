// bwd_order.cuh -- the order in which the backward's CTAs take their work units.
//
// A unit is one key tile kb of one kv head (a (b, g) pair, index b * G + g):
// the CTA accumulates dK, dV of those 128 keys over every query row of the
// pair's R query heads that sees them, reading those rows' Q and dO and
// reducing into their fp32 dQ accumulator rows.  A pair's key tiles thus
// share about R * S * 512 bytes of rows (dQ 256 B, Q 128 B, dO 128 B a row).
//
// Ordered key-tile-major over every pair, each wave of CTAs sweeps all pairs'
// rows, and the 126 MB L2 keeps none of them from one key tile's wave to the
// next: on B1 H128 G16 S8192 that order moved 3.3 GB through DRAM per launch,
// against 0.6 GB of operands and gradients.  So the pairs are split into
// batches of about kOrderBudget bytes of rows and each batch runs
// key-tile-major (the heaviest key tiles, with the most query tiles, first).
// Batch sizes differ by at most one, the larger batches last: the heaviest
// key tiles of the last batch still have to end with the other CTAs, which
// asks for at least about 1.5 * SMs / (key tiles + 1) pairs in it (the share
// of one pair's work that falls on an SM, against one key tile's work).
//
// With a window, the key tiles that hold sinks are seen by every later query,
// not by a window's worth: at S = 32768, window 4096, 128 sinks, key tile 0
// has 256 query tiles against 33 for the others.  Left at the head of their
// pair's batch, the last pair's sink tiles would start near the end of the
// launch and run on alone (a batch of one pair there lasts about a fifth of
// such a tile).  They stream through all of their pair's rows whatever the
// order, so they gain nothing from the batches: the sink key tiles of every
// pair run first, key-tile-major, and the batches cover the other key tiles.
//
// Host and device code, with no other dependency, so that a host program can
// check the order on its own.
#pragma once

namespace gqa {
namespace bwd {

constexpr double kOrderBudget = 136.0 * 1024 * 1024;

// Key tiles that run ahead of the batches: those holding sinks when the mask
// has a window (window > 0 only with causal masking), else none.
__host__ __device__ inline int front_tiles(int n_ktiles, int window, int n_sink, int tile_keys) {
  if (window <= 0 || n_sink <= 0) return 0;
  const long long t = (static_cast<long long>(n_sink) + tile_keys - 1) / tile_keys;
  return t < n_ktiles ? static_cast<int>(t) : n_ktiles;
}

// Batches of the B * G pairs over the key tiles after the n_front first ones:
// n_small batches of batch_pairs pairs, then the rest of batch_pairs + 1.
__host__ __device__ inline void cta_order(int B, int G, int R, int S, int n_ktiles, int n_front,
                                          int sm_count, int &n_small, int &batch_pairs) {
  const int pairs = B * G;
  n_ktiles -= n_front;
  long long m = static_cast<long long>(kOrderBudget / (static_cast<double>(R) * S * 512.0));
  const long long m_tail = (3LL * sm_count + 2LL * (n_ktiles + 1) - 1) / (2LL * (n_ktiles + 1));
  m = m < m_tail ? m_tail : m;
  m = m < 1 ? 1 : (m > pairs ? pairs : m);
  const int nb = static_cast<int>((pairs + m - 1) / m);
  batch_pairs = pairs / nb;
  n_small = nb - pairs % nb;
}

// CTA u (0 <= u < n_ktiles * pairs) -> key tile kb and pair: first the
// n_front key tiles of every pair, key-tile-major, then the batches.
__host__ __device__ inline void cta_unit(int u, int n_ktiles, int n_front, int pairs, int n_small,
                                         int batch_pairs, int &kb, int &pair) {
  if (u < n_front * pairs) {
    kb = u / pairs;
    pair = u % pairs;
    return;
  }
  u -= n_front * pairs;
  n_ktiles -= n_front;
  const int q = batch_pairs;
  const int small = n_small * q * n_ktiles;  // CTAs of the small batches
  int v, sz, base;
  if (u < small) {
    const int bi = u / (q * n_ktiles);
    v = u - bi * q * n_ktiles;
    sz = q;
    base = bi * q;
  } else {
    const int u2 = u - small;
    const int bi = u2 / ((q + 1) * n_ktiles);
    v = u2 - bi * (q + 1) * n_ktiles;
    sz = q + 1;
    base = n_small * q + bi * (q + 1);
  }
  kb = n_front + v / sz;
  pair = base + v % sz;
}

}  // namespace bwd
}  // namespace gqa
