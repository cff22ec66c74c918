// fwd_kernel.cuh -- forward of causal grouped-query attention on sm_103a.
//
// Computes, for each query row i of head h (kv head g = h / (H/G)):
//   o_i = softmax_j(scale * q_i . k_j, visible j) . V,   lse_i = ln sum_j exp(scale * q_i . k_j)
// ("nx_f32_gqa_gate.nx source": scores, causal mask, softmax, attn.V and the
// head map of test T2; "SnapKitty Transformer 8B": online softmax over K/V
// tiles, sliding window and attention sinks.)
//
// Work unit = (batch b, kv head g, 128-row query block qb) x two query heads of
// g.  Both heads read every K/V tile the CTA loads, so each tile crosses
// HBM/L2 once per pair of heads.  Only key tiles with at least one visible key
// are visited (sink tiles, then the window / causal range), and the elementwise
// mask runs only on tiles that straddle a mask boundary.
//
// The grid is persistent: one CTA per SM walks the unit list (heaviest query
// blocks first, in zig-zag rounds of one unit per CTA).  Every barrier phase is
// counted across units, so the producer loads the next unit's Q and K/V while
// the current one finishes, each head's next Q K^T starts as soon as its S
// buffer is free, and its first P.V waits only until the epilogue has read O;
// the CTA launch, barrier and TMEM set-up and the cold loads are paid once per
// SM instead of once per unit.
//
// Roles (384 threads):
//   warp 0        TMA producer: each unit's Q tiles, then K and V tiles through
//                 an NSTAGE-deep shared-memory ring (full/empty mbarriers).
//   warp 2        allocates / frees the 512 TMEM columns; its lane 0 issues
//                 S_t = Q_t K^T into TMEM for both heads.
//   warps 1, 3    one thread each issues O_t += P_t V for query head t, with
//                 P_t read from TMEM (A operand in TMEM).
//                 Three issuing threads keep the tensor pipe fed while any of
//                 them waits on a barrier (an mbarrier hand-off costs about as
//                 much as three MMAs, and the tensor queue is only a few deep),
//                 and the next tile's S never waits behind this tile's P.V in
//                 program order.
//   warps 4..7    softmax + O correction + epilogue of head 0 (one row per thread)
//   warps 8..11   the same for head 1
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,320) O1 [320,384)
//               P0 [384,448) P1 [448,512) (bf16 pairs).
// Because P has its own columns, S_t(j+1) = Q_t K_{j+1}^T is issued as soon as
// the softmax of head t has read S_t(j) into registers; only the P store and
// the O correction wait for P_t V_j to finish, and each head's softmax of
// tile j+1 overlaps the other head's products.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include <type_traits>

#include "device_checks.cuh"
#include "rope_kernels.cuh"
#include "sm100_ptx.cuh"
#include "trace.cuh"

namespace gqa {
namespace fwd {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per tile
constexpr int HD = 64;   // head dimension
constexpr int NSTAGE = 3;
constexpr int TILE_BYTES = BM * HD * 2;  // 16 KB, 128-byte rows
constexpr int NTHREADS = 384;
// Registers per thread after the split: warps 0-3 (producer, MMA, TMEM alloc)
// drop to kRegsControl, the two softmax warpgroups rise to kRegsSoftmax.
constexpr int kRegsControl = 72;
constexpr int kRegsSoftmax = 208;
// the launch allocation must cover the split (checked on the host)
constexpr int kMinLaunchRegs = (128 * kRegsControl + 256 * kRegsSoftmax + NTHREADS - 1) / NTHREADS;
constexpr uint32_t TMEM_COLS = 512;
// A row keeps its running max until a tile's max exceeds it by more than this
// (base-2 units), so P stays below 2^8 and O is rescaled only rarely; the
// result is exact because O and l are normalised with the same running max.
constexpr float kRescaleThreshold = 8.0f;
// Score bound (gqa_attn_fwd_ws only): |s_ij| * scale * log2(e) <= U_i =
// |q_i| * max_j |k_j| * scale * log2(e) (Cauchy-Schwarz), with max_j |k_j|^2 over
// the kv head from fwd_knorm_kernel.  A head whose 128 rows all have U_i <=
// kBoundMax runs the whole unit against the fixed reference m_i = U_i -
// kFastSlack and takes no row maxima: every term 2^(s * sl2 - m_i) lies in
// [2^(kFastSlack - 2 U_i), 2^kFastSlack], so none overflows and the largest of
// a row stays above 2^(kFastSlack - 2 kBoundMax) = 2^-96; the result is the same
// softmax, normalised by the same reference in O and l.
constexpr float kFastSlack = 32.0f;
constexpr float kBoundMax = 64.0f;
// partial maxima of |k_j|^2 per kv head: one 128-byte record (many CTAs per kv
// head keep the pre-pass's loads spread over every SM)
constexpr int kKnParts = 32;
static_assert(kKnParts % 4 == 0, "score_bound reads the record as float4");
__device__ __forceinline__ uint32_t col_s(int t) { return static_cast<uint32_t>(t) * 128u; }
__device__ __forceinline__ uint32_t col_o(int t) { return 256u + static_cast<uint32_t>(t) * 64u; }
__device__ __forceinline__ uint32_t col_p(int t) { return 384u + static_cast<uint32_t>(t) * 64u; }

constexpr int SM_Q = 0;
constexpr int SM_K = SM_Q + 2 * TILE_BYTES;
constexpr int SM_V = SM_K + NSTAGE * TILE_BYTES;
constexpr int SM_BARS = SM_V + NSTAGE * TILE_BYTES;

struct Bars {
  alignas(16) float kn[2][2][kKnParts];  // |k_j|^2 record per head and slot (a head's units
                                         // alternate slots)
  uint64_t q_full[2];  // head t's Q tile (and its |k|^2 record) landed (TMA transaction
                       // bytes).  One barrier per head: head 1 sits out the single-head
                       // units, and counting its own phases keeps it from mistaking an
                       // older completed phase for the one it waits on
  uint64_t q_empty;    // every Q K^T of the unit finished: Q may be reloaded
  uint64_t kv_full[NSTAGE];   // K and V tile landed (TMA transaction bytes)
  uint64_t kv_empty[NSTAGE];  // every head's products with the tile finished (the
                              // QK issuer and both P.V issuers, always 3 arrivals)
  uint64_t s_full[2];  // S_t ready (MMA commit)
  uint64_t s_free[2];  // S_t read into registers (128 softmax threads)
  uint64_t p_full[2];  // P_t stored and O_t corrected (128 softmax threads)
  uint64_t o_done[2];  // P_t V finished (MMA commit)
  uint64_t o_full[2];  // every product of head t in the unit finished (MMA commit)
  uint64_t o_empty[2]; // the epilogue read O_t: the next unit may overwrite it (128 threads)
  uint64_t qk_done;    // every S product finished (QK issuer commit, abort drain)
  uint64_t pv_done[2]; // every P.V product of head t finished (abort drain)
  uint64_t turn[2];    // ping-pong of the exp2 sections: turn[t] opens head t's
                       // section (arrived by the other head's 128 threads)
  uint64_t q_ready[2]; // rotary embedding only: head t's Q tile rotated in place
                       // (128 softmax threads of head t, once per unit)
  uint64_t vote_bar[2];  // score bound: head t's four warps have cast their vote
  int vote[2][2];        // score bound: AND of head t's warp votes, two alternating slots
  uint32_t tmem_base;
  AbortState abort;
};

constexpr int SMEM_BYTES = 1024 /* alignment slack */ + SM_BARS + static_cast<int>(sizeof(Bars));

struct Params {
  int B, H, G, S, R;
  int causal, window, n_sink;
  float scale_log2;  // scale * log2(e): scores are kept in the base-2 domain
  int n_qblocks;
  int n_pairs;  // ceil(R / 2) head pairs per kv head
  int n_units;  // n_qblocks * B * G * n_pairs
  const float *kn2;  // [B*G][kKnParts] partial maxima of |k_j|^2, or null (no score bound)
  const float2 *rope_tab;  // rotary embedding: [S][32] (cos, sin) per position and pair
  __nv_bfloat16 *o;
  float *lse;
  int *status;
};

enum : int { kTimeoutCode = -9 };

// Key tiles a query block visits: [0, n_sink_tiles) then [wlo, hi].
struct KvRange {
  int n_sink_tiles;
  int wlo;
  int count;
  __device__ __forceinline__ int tile(int idx) const {
    return idx < n_sink_tiles ? idx : wlo + (idx - n_sink_tiles);
  }
};

__device__ __forceinline__ KvRange kv_range(int qb, const Params &p) {
  const int nkb = (p.S + BN - 1) / BN;
  KvRange r;
  r.n_sink_tiles = 0;
  r.wlo = 0;
  if (!p.causal) {
    r.count = nkb;
    return r;
  }
  const int i0 = qb * BM;
  const int hi = min((i0 + BM - 1) / BN, nkb - 1);
  if (p.window <= 0) {
    r.count = hi + 1;
    return r;
  }
  const int lo_key = i0 - p.window + 1;  // oldest key any row of the block sees in-window
  const int wlo = lo_key <= 0 ? 0 : lo_key / BN;
  const int nst = min((p.n_sink + BN - 1) / BN, wlo);
  r.n_sink_tiles = nst;
  r.wlo = wlo;
  r.count = nst + hi - wlo + 1;
  return r;
}

// The n lowest bits set (n clamped to [0, 32]).
__device__ __forceinline__ uint32_t low_bits(int n) {
  return n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : (1u << n) - 1u);
}

// True when some (row, key) pair of the tile is masked, so the elementwise
// mask must run.
__device__ __forceinline__ bool tile_needs_mask(int qb, int kb, const Params &p) {
  const int i0 = qb * BM, j0 = kb * BN, j1 = j0 + BN - 1;
  if (j1 >= p.S) return true;
  if (!p.causal) return false;
  if (j1 > i0) return true;
  if (p.window > 0) {
    const bool all_in_window = j0 > i0 + BM - 1 - p.window;
    const bool all_sinks = j1 < p.n_sink;
    if (!all_in_window && !all_sinks) return true;
  }
  return false;
}

// One work unit, heaviest (latest) query blocks first.
struct Unit {
  int qb, b, g, h0;
  bool two;  // both heads of the pair exist (R odd leaves a single last head)
};

__device__ __forceinline__ Unit unit_of(int u, const Params &p) {
  const int per_qb = p.B * p.G * p.n_pairs;
  const int rem = u % per_qb;
  Unit un;
  un.qb = p.n_qblocks - 1 - u / per_qb;
  un.b = rem / (p.G * p.n_pairs);
  un.g = (rem / p.n_pairs) % p.G;
  const int pair = rem % p.n_pairs;
  un.h0 = un.g * p.R + 2 * pair;
  un.two = (2 * pair + 1) < p.R;
  return un;
}

__device__ __forceinline__ int kvz_of(const Unit &un, const Params &p) { return un.b * p.G + un.g; }

// U_i of the score bound, in base-2 units: sqrt(|q_i|^2 * max_j |k_j|^2) * sl2,
// widened by 2^-10 relative and absolute for the rounding of the norms and of
// the MMA's fp32 sums.  qrow: row r of a Q tile in shared memory (128-byte
// swizzle: 16-byte chunk c at c ^ (r & 7), read in that order so that the
// eight rows r..r+7 of a load hit eight different chunks of the banks).
__device__ __forceinline__ float score_bound(const uint8_t *qrow, int r, const float *kn, float sl2) {
  uint64_t acc = 0ull;  // fp32 pair (0.0f bits)
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 w = *reinterpret_cast<const uint4 *>(qrow + ((c ^ (r & 7)) << 4));
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint64_t x = f32x2(__uint_as_float(ws[e] << 16), __uint_as_float(ws[e] & 0xffff0000u));
      acc = fma_f32x2(x, x, acc);
    }
  }
  float qa, qb;
  f32x2_split(acc, qa, qb);
  float4 m4 = reinterpret_cast<const float4 *>(kn)[0];
#pragma unroll
  for (int c = 1; c < kKnParts / 4; ++c) {
    const float4 x = reinterpret_cast<const float4 *>(kn)[c];
    m4 = make_float4(fmaxf(m4.x, x.x), fmaxf(m4.y, x.y), fmaxf(m4.z, x.z), fmaxf(m4.w, x.w));
  }
  const float kmax2 = fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w));
  return sqrtf((qa + qb) * kmax2) * sl2 * (1.f + 0x1p-10f) + 0x1p-10f;
}

// The k-th unit of this CTA, or -1 when none is left.  Rounds of gridDim.x
// units alternate direction (CTA c takes unit c of even rounds and unit
// grid - 1 - c of odd ones): unit sizes shrink along the heaviest-first list,
// and the zig-zag evens out what a plain stride leaves to the first CTAs.
__device__ __forceinline__ int unit_at(int k, const Params &p) {
  const int base = k * static_cast<int>(gridDim.x);
  if (base >= p.n_units) return -1;
  const int c = (k & 1) ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x);
  return base + c < p.n_units ? base + c : -1;
}

// kRope: the query tiles are turned by the rotary embedding (rope_kernels.cuh)
// in shared memory before their first Q K^T; the keys arrive already rotated.
// kFp8: queries and keys are OCP E4M3 bytes (64-byte rows, 64-byte swizzle,
// 8 KB tiles in the 16 KB slots); S = Q K^T runs as tcgen05.mma
// kind::f8f6f4 (K = 32 per instruction) and the two per-tensor scales are
// folded into scale_log2 on the host.  P.V stays bf16.
template <bool kRope, bool kFp8>
__global__ void __launch_bounds__(NTHREADS, 1)
    gqa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled tiles, by pointer arithmetic on the
  // __shared__ array so that accesses stay shared-space (ld/st.shared).
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars *bars = reinterpret_cast<Bars *>(smem + SM_BARS);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // bytes of one Q or K tile as loaded (fp8 rows are half as long)
  constexpr uint32_t kQTileBytes = kFp8 ? TILE_BYTES / 2 : TILE_BYTES;
  static_assert(!(kFp8 && kRope), "the fp8 forward takes no rotary embedding");

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full[0], 1);
    mbar_init(&bars->q_full[1], 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 3);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->s_free[t], 128);
      mbar_init(&bars->p_full[t], 128);
      mbar_init(&bars->o_done[t], 1);
      mbar_init(&bars->o_full[t], 1);
      mbar_init(&bars->o_empty[t], 128);
      mbar_init(&bars->turn[t], 128);
      mbar_init(&bars->pv_done[t], 1);
      mbar_init(&bars->q_ready[t], 128);
      mbar_init(&bars->vote_bar[t], 128);
      bars->vote[t][0] = 1;
      bars->vote[t][1] = 1;
    }
    mbar_init(&bars->qk_done, 1);
    bars->abort.flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&bars->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = bars->tmem_base;
  AbortState *ab = &bars->abort;
  if (threadIdx.x == 0) GQA_TRACE_EVENT(0, 14, 0);

  if (warp < 4) {
  setmaxnreg_dec<kRegsControl>();
  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int gt = 0;       // K/V tiles issued (all units): ring stage and phase
      int q_loads[2] = {0, 0};  // Q tiles issued per head (all units)
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int u = unit_at(k, p);
        if (u < 0) break;
        const Unit un = unit_of(u, p);
        const KvRange kr = kv_range(un.qb, p);
        // the previous unit's Q K^T products must have read Q
        if (k > 0 && !mbar_wait(&bars->q_empty, (k - 1) & 1, ab, p.status, kTimeoutCode)) break;
        const int qrow = un.qb * BM, qz = un.b * p.H + un.h0;
        GQA_REPORT(p.status, un.qb >= 0 && un.qb < p.n_qblocks && kr.count >= 1 &&
                                qz + (un.two ? 1 : 0) < p.B * p.H);
        for (int t = 0; t < (un.two ? 2 : 1); ++t) {
          mbar_arrive_expect_tx(&bars->q_full[t], kQTileBytes + (p.kn2 ? kKnParts * 4 : 0));
          tma_load_3d(smem + SM_Q + t * TILE_BYTES, &tm_q, &bars->q_full[t], 0, qrow, qz + t);
          if (p.kn2)  // the kv head's |k|^2 record, for the softmax's score bound
            bulk_load(&bars->kn[t][q_loads[t] & 1][0],
                      p.kn2 + static_cast<size_t>(kvz_of(un, p)) * kKnParts, kKnParts * 4,
                      &bars->q_full[t]);
          ++q_loads[t];
        }
        const int kvz = un.b * p.G + un.g;
        for (int it = 0; it < kr.count; ++it, ++gt) {
          const int st = gt % NSTAGE;
          const int kb = kr.tile(it);
          if (!mbar_wait(&bars->kv_empty[st], ((gt / NSTAGE) & 1) ^ 1, ab, p.status, kTimeoutCode)) {
            ok = false;
            break;
          }
          GQA_TRACE_EVENT(0, 0, k == 0 ? it : kTraceSteps);
#ifdef GQA_INJECT_STALL
          // failure-detection test build only: CTA 0 never loads one K/V tile
          // of its first unit, so every role must leave through the bounded
          // waits and the abort flag
          if (blockIdx.x == 0 && k == 0 && it == min(1, kr.count - 1)) continue;
#endif
          GQA_REPORT(p.status, kb >= 0 && kb * BN < p.S && kvz < p.B * p.G);
          mbar_arrive_expect_tx(&bars->kv_full[st], kQTileBytes + TILE_BYTES);
          tma_load_3d(smem + SM_K + st * TILE_BYTES, &tm_k, &bars->kv_full[st], 0, kb * BN, kvz);
          tma_load_3d(smem + SM_V + st * TILE_BYTES, &tm_v, &bars->kv_full[st], 0, kb * BN, kvz);
          GQA_TRACE_EVENT(0, 1, k == 0 ? it : kTraceSteps);
        }
      }
      // Exit drain: every copy this CTA issued must have landed before the CTA
      // leaves (no-op on the normal path, where the consumers already saw them).
      for (int t = 0; t < 2; ++t)
        if (q_loads[t] > 0) mbar_wait_drain(&bars->q_full[t], (q_loads[t] - 1) & 1);
      for (int x = max(0, gt - NSTAGE); x < gt; ++x)
        mbar_wait_drain(&bars->kv_full[x % NSTAGE], (x / NSTAGE) & 1);
    }
  } else if (warp == 2 && lane == 0) {
    // ================================================================ QK issuer
    const uint32_t idesc_qk = kFp8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN, false, false);
    const uint32_t q_addr0 = smem_u32(smem + SM_Q);
    const uint32_t k_addr0 = smem_u32(smem + SM_K);
    int gt = 0;             // K/V tiles consumed (all units)
    int ts[2] = {0, 0};     // S products issued per head (all units)
    int qf[2] = {0, 0};     // Q tiles consumed per head (all units)
    int qr[2] = {0, 0};     // rotated Q tiles consumed per head (rotary embedding)
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = unit_at(k, p);
      if (u < 0) break;
      const Unit un = unit_of(u, p);
      const int n = kv_range(un.qb, p).count;
      for (int it = 0; it < n; ++it, ++gt) {
        const int st = gt % NSTAGE;
        if (!mbar_wait(&bars->kv_full[st], (gt / NSTAGE) & 1, ab, p.status, kTimeoutCode)) { ok = false; break; }
        for (int t = 0; t < (un.two ? 2 : 1); ++t) {
          // the softmax must have read S_t of head t's previous tile
          if (ts[t] > 0 && !mbar_wait(&bars->s_free[t], (ts[t] - 1) & 1, ab, p.status, kTimeoutCode)) {
            ok = false;
            break;
          }
          if (it == 0) {  // the unit's first product of head t needs its Q tile
            if (!mbar_wait(&bars->q_full[t], qf[t] & 1, ab, p.status, kTimeoutCode)) {
              ok = false;
              break;
            }
            ++qf[t];
          }
          if constexpr (kRope) {
            // and, with the rotary embedding, that tile turned
            if (it == 0) {
              if (!mbar_wait(&bars->q_ready[t], qr[t] & 1, ab, p.status, kTimeoutCode)) {
                ok = false;
                break;
              }
              ++qr[t];
            }
          }
          GQA_TRACE_EVENT(0, t == 0 ? 22 : 23, k == 0 ? it : kTraceSteps);  // S_t issue starts
          tc_fence_after_sync();
          if constexpr (kFp8) {
            const uint64_t ad = sdesc_sw64(q_addr0 + t * TILE_BYTES, 16, 512);
            const uint64_t bd = sdesc_sw64(k_addr0 + st * TILE_BYTES, 16, 512);
#pragma unroll
            for (int ks = 0; ks < HD / 32; ++ks)  // K step 32 bytes inside the 64-B row
              mma_f8_ss(tbase + col_s(t), ad + 2 * ks, bd + 2 * ks, idesc_qk, ks > 0);
          } else {
            const uint64_t ad = sdesc_sw128(q_addr0 + t * TILE_BYTES, 16, 1024);
            const uint64_t bd = sdesc_sw128(k_addr0 + st * TILE_BYTES, 16, 1024);
#pragma unroll
            for (int ks = 0; ks < HD / 16; ++ks)  // K step 16 bf16 = 32 B inside the 128-B row
              mma_bf16_ss(tbase + col_s(t), ad + 2 * ks, bd + 2 * ks, idesc_qk, ks > 0);
          }
          mma_commit(&bars->s_full[t]);
          ++ts[t];
        }
        if (!ok) break;
        GQA_TRACE_EVENT(0, 21, k == 0 ? it : kTraceSteps);
        mma_commit(&bars->kv_empty[st]);  // K read
      }
      if (!ok) break;
      mma_commit(&bars->q_empty);  // this unit's Q read
    }
    mma_commit(&bars->qk_done);
    if (!ok) mbar_wait_drain(&bars->qk_done, 0);
  } else if ((warp == 1 || warp == 3) && lane == 0) {
    // ================================================================ P.V issuers
    const int t = warp == 1 ? 0 : 1;  // the query head this thread serves
    const uint32_t idesc_pv = idesc_bf16_f32(BM, HD, false, true);
    const uint32_t v_addr0 = smem_u32(smem + SM_V);
    const uint32_t d_o = tbase + col_o(t), a_p = tbase + col_p(t);
    int gt = 0;  // K/V tiles seen (all units)
    int tp = 0;  // P.V products of this head (all units)
    int uo = 0;  // units of this head whose O was released
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = unit_at(k, p);
      if (u < 0) break;
      const Unit un = unit_of(u, p);
      const int n = kv_range(un.qb, p).count;
      const bool mine = t == 0 || un.two;
      for (int it = 0; it < n; ++it, ++gt) {
        const int st = gt % NSTAGE;
        // V landed (the softmax of the tile has started, so its K did too);
        // for a single-head unit the absent head still releases the stage,
        // after it was filled for this use
        if (!mbar_wait(&bars->kv_full[st], (gt / NSTAGE) & 1, ab, p.status, kTimeoutCode)) { ok = false; break; }
        if (!mine) {
          mbar_arrive(&bars->kv_empty[st]);
          continue;
        }
        // the previous unit's epilogue must have read O_t before it is overwritten
        if (it == 0 && uo > 0 && !mbar_wait(&bars->o_empty[t], (uo - 1) & 1, ab, p.status, kTimeoutCode)) {
          ok = false;
          break;
        }
        if (!mbar_wait(&bars->p_full[t], tp & 1, ab, p.status, kTimeoutCode)) { ok = false; break; }
        if (t == 0) GQA_TRACE_EVENT(0, 2, k == 0 ? it : kTraceSteps); else GQA_TRACE_EVENT(0, 4, k == 0 ? it : kTraceSteps);
        tc_fence_after_sync();
        const uint64_t bd = sdesc_sw128(v_addr0 + st * TILE_BYTES, TILE_BYTES, 1024);
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)  // 16 keys = two 8-row groups = 2048 B
          mma_bf16_ts(d_o, a_p + ks * 8, bd + (ks * 2048 >> 4), idesc_pv, (it > 0 || ks > 0) ? 1u : 0u);
        mma_commit(&bars->o_done[t]);
        mma_commit(&bars->kv_empty[st]);  // V read by this head
        ++tp;
        if (t == 0) GQA_TRACE_EVENT(0, 3, k == 0 ? it : kTraceSteps); else GQA_TRACE_EVENT(0, 5, k == 0 ? it : kTraceSteps);
      }
      if (!ok) break;
      if (mine) {
        mma_commit(&bars->o_full[t]);  // releases this head's epilogue of the unit
        ++uo;
      }
    }
    // lets this thread wait, on the abort path, until its products are done
    // before TMEM is freed
    mma_commit(&bars->pv_done[t]);
    if (!ok) mbar_wait_drain(&bars->pv_done[t], 0);
  }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // ================================================================ softmax
    const int t = (warp - 4) >> 2;
    const int lane_base = 32 * (warp & 3);
    const int r = lane_base + lane;  // row of the tile this thread owns
    const float sl2 = p.scale_log2;
    const uint32_t lane_off = static_cast<uint32_t>(lane_base) << 16;
    const uint32_t t_s = tbase + lane_off + col_s(t);
    const uint32_t t_o = tbase + lane_off + col_o(t);
    const uint32_t t_p = tbase + lane_off + col_p(t);
    const uint64_t sl2x2 = f32x2(sl2, sl2);
    // The waits below are per thread, without a warp vote (a vote on each of
    // them cost 3-4 % of the forward): the warp is converged at every wait and
    // inside the wait loop, so its lanes execute each try_wait, abort-flag load
    // and clock read as one instruction and take the same branch; the result
    // is warp-uniform before the warp-collective tcgen05.ld/st that follow.
    int ts = 0;  // tiles of this head (all units): S, P and O-done phases
    int uo = 0;  // units of this head: O-full / O-empty phases
    int tt = 0;  // tiles of two-head units: ping-pong phases (same count in both heads)
    int uq = 0;  // Q tiles of this head (all units): Q-full phases and record slots
    int uv = 0;  // score-bound votes of this head: vote phases and slots
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = unit_at(k, p);
      if (u < 0) break;
      const Unit un = unit_of(u, p);
      if (t == 1 && !un.two) continue;
      const int qk = uq++;  // this head's Q tile count: phase of q_full[t], record slot
      const KvRange kr = kv_range(un.qb, p);
      const int n = kr.count;
      const int qb = un.qb;
      const int i = qb * BM + r;  // query index
      // mask bounds: key j visible iff j <= hi && (j > lo || j < ns)
      const int hi = p.causal ? min(i, p.S - 1) : p.S - 1;
      const bool win = p.causal && p.window > 0;
      const int lo = win ? i - p.window : -1;
      const int ns = win ? p.n_sink : 0;

      if constexpr (kRope) {
        // turn this row of head t's Q tile (position i) before any Q K^T reads it
        if (!mbar_wait(&bars->q_full[t], qk & 1, ab, p.status, kTimeoutCode)) { ok = false; break; }
        if (i < p.S)
          rope::rope_rotate_smem_row(smem + SM_Q + t * TILE_BYTES + r * 128, r,
                                     p.rope_tab + static_cast<size_t>(i) * rope::kPairs);
        fence_proxy_async_smem();
        mbar_arrive(&bars->q_ready[t]);
      }
      float m_run = -CUDART_INF_F;  // running max of scaled scores, base-2 units
      float l_run = 0.f;            // running sum of 2^(s - m_run)
      // Score bound (kBoundMax): decided for the head's 128 rows together
      // (all four warps) before the unit's first tile: a head whose warps mixed
      // the two steps measured about 50 % slower than one on the exact step
      // throughout.  Units of one key tile keep the exact step: their Q may be
      // reloaded as soon as their only Q K^T is done, before this read could
      // happen.
      bool fast = false;
      if (p.kn2 != nullptr && n >= 2) {
        // Q and the record landed with q_full[t] (phase qk); they stay until
        // every Q K^T of the unit is done, and the last one (tile n - 1 >= 1)
        // waits for this thread's release of S of tile n - 2 >= 0.
        if (!mbar_wait(&bars->q_full[t], qk & 1, ab, p.status, kTimeoutCode)) { ok = false; break; }
        const float bound = score_bound(smem + SM_Q + t * TILE_BYTES + r * 128, r, &bars->kn[t][qk & 1][0], sl2);
        // each warp ANDs its vote into the slot, then the 128 threads meet on an
        // mbarrier (a bounded wait, so an abort cannot leave a thread behind)
        const int slot = uv & 1;
        if (!__all_sync(0xffffffffu, bound <= kBoundMax) && lane == 0) atomicAnd(&bars->vote[t][slot], 0);
        mbar_arrive(&bars->vote_bar[t]);
        if (!mbar_wait(&bars->vote_bar[t], uv & 1, ab, p.status, kTimeoutCode)) { ok = false; break; }
        ++uv;
        fast = *reinterpret_cast<volatile int *>(&bars->vote[t][slot]) != 0;
        // every thread of the head has read the other slot (its previous vote)
        // before arriving here: reset it for the head's next vote
        if (r == 0) bars->vote[t][slot ^ 1] = 1;
        if (fast) m_run = bound - kFastSlack;
      }
      // One key tile of the unit.  kFast: the warp runs against the score
      // bound's fixed reference and takes no row maxima.  Two instantiations,
      // chosen once per unit, so the steady-state loop carries no max code.
      // Returns false on abort.
      int it = 0;
      auto tile = [&](auto fast_tag) -> bool {
        constexpr bool kFast = decltype(fast_tag)::value;
        const int kb = kr.tile(it);
        const int step = k == 0 ? it : kTraceSteps;  // trace the first unit only
        (void)step;
        if (!mbar_wait(&bars->s_full[t], ts & 1, ab, p.status, kTimeoutCode)) return false;
        if (lane == 0 && (warp == 4 || warp == 8)) GQA_TRACE_EVENT(0, warp == 4 ? 6 : 10, step);
        tc_fence_after_sync();
        uint32_t s0[32], s1[32], s2[32], s3[32];
        tmem_ld_32x32b_x32(t_s + 0, s0);
        tmem_ld_32x32b_x32(t_s + 32, s1);
        tmem_ld_32x32b_x32(t_s + 64, s2);
        tmem_ld_32x32b_x32(t_s + 96, s3);
        tmem_wait_ld();
        reg_fence(s0);
        reg_fence(s1);
        reg_fence(s2);
        reg_fence(s3);
        // S_t is in registers: the next Q_t K^T may overwrite it
        tc_fence_before_sync();
        mbar_arrive(&bars->s_free[t]);
        if (lane == 0 && warp == 4) GQA_TRACE_EVENT(0, 7, step);
        float s[BN];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          s[c] = __uint_as_float(s0[c]);
          s[32 + c] = __uint_as_float(s1[c]);
          s[64 + c] = __uint_as_float(s2[c]);
          s[96 + c] = __uint_as_float(s3[c]);
        }
        if (tile_needs_mask(qb, kb, p)) {
          // Visibility of the tile's 128 keys as 4 words of bits, from three
          // bounds (built with a few integer operations per word), then one
          // bit test and select per score.  A boolean expression per key
          // compiled to a far slower sequence on this path.
          const int j0 = kb * BN;
          uint32_t vb[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int base = j0 + 32 * w;
            vb[w] = low_bits(hi - base + 1) & (~low_bits(lo - base + 1) | low_bits(ns - base));
          }
#pragma unroll
          for (int c = 0; c < BN; ++c) s[c] = ((vb[c >> 5] >> (c & 31)) & 1u) ? s[c] : -CUDART_INF_F;
        }
        // row max: 4 independent chains of 3-input max over elements 8..127,
        // seeded with elements 0..7 (not needed against a bound's reference)
        bool need = false;  // O and l are rescaled by alpha
        float m_new = m_run, alpha = 1.f;
        if constexpr (!kFast) {
          float mx4[4];
#pragma unroll
          for (int a = 0; a < 4; ++a) mx4[a] = fmaxf(s[2 * a], s[2 * a + 1]);
#pragma unroll
          for (int c = 8; c < BN; c += 8) {
#pragma unroll
            for (int a = 0; a < 4; ++a) mx4[a] = max3f(mx4[a], s[c + 2 * a], s[c + 2 * a + 1]);
          }
          const float mx = fmaxf(max3f(mx4[0], mx4[1], mx4[2]), mx4[3]);
          const float m_tile = mx * sl2;
          // lazy rescale: keep the running max unless this tile exceeds it by > threshold
          need = m_tile > m_run + kRescaleThreshold;
          m_new = need ? m_tile : m_run;
        }
        const float m_use = (m_new == -CUDART_INF_F) ? 0.f : m_new;
        if constexpr (!kFast) alpha = need ? ex2_approx(m_run - m_use) : 1.f;
        const uint64_t negm = f32x2(-m_use, -m_use);
        if (lane == 0 && warp == 4) GQA_TRACE_EVENT(0, 16, step);
        // Ping-pong: the two heads take turns on the exp2 section (MUFU-bound), so
        // each runs at the full MUFU rate while the other head's products keep
        // the tensor pipe busy.  Head 0 goes first in every tile.
        if (un.two) {
          const bool wait_turn = (t == 1) || tt > 0;
          const uint32_t par = t == 0 ? ((tt - 1) & 1) : (tt & 1);
          if (wait_turn && !mbar_wait(&bars->turn[t], par, ab, p.status, kTimeoutCode)) return false;
        }
        if (lane == 0 && warp == 4) GQA_TRACE_EVENT(0, 17, step);
        uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};  // four chains of fp32 pairs (0.0f bits)
        uint32_t pk[BN / 2];
#pragma unroll
        for (int c2 = 0; c2 < BN / 2; ++c2) {
          const uint64_t x = fma_f32x2(f32x2(s[2 * c2], s[2 * c2 + 1]), sl2x2, negm);
          float x0, x1;
          f32x2_split(x, x0, x1);
          const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
          sum2[c2 & 3] = add_f32x2(sum2[c2 & 3], f32x2(e0, e1));
          pk[c2] = pack_bf16x2(e0, e1);
        }
        if (lane == 0 && warp == 4) GQA_TRACE_EVENT(0, 18, step);
        if (un.two) {
          mbar_arrive(&bars->turn[1 - t]);
          ++tt;
        }
        float sa, sb, sc, sd;
        f32x2_split(add_f32x2(sum2[0], sum2[1]), sa, sb);
        f32x2_split(add_f32x2(sum2[2], sum2[3]), sc, sd);
        const float sum = (sa + sb) + (sc + sd);
        if (lane == 0 && warp == 4) GQA_TRACE_EVENT(0, 8, step);
        // P_t V of the previous tile must be finished before P_t is overwritten
        // and O_t rescaled.  (Before a unit's first tile the previous unit's
        // epilogue already waited for all of its products.)
        if (it > 0) {
          if (!mbar_wait(&bars->o_done[t], (ts - 1) & 1, ab, p.status, kTimeoutCode)) return false;
          tc_fence_after_sync();
          if (!kFast && __any_sync(0xffffffffu, need)) {
            uint32_t o0[32], o1[32];
            tmem_ld_32x32b_x32(t_o + 0, o0);
            tmem_ld_32x32b_x32(t_o + 32, o1);
            tmem_wait_ld();
            reg_fence(o0);
            reg_fence(o1);
            const uint64_t a2 = f32x2(alpha, alpha);
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              float x0, x1;
              f32x2_split(mul_f32x2(f32x2(__uint_as_float(o0[c]), __uint_as_float(o0[c + 1])), a2), x0, x1);
              o0[c] = __float_as_uint(x0);
              o0[c + 1] = __float_as_uint(x1);
              f32x2_split(mul_f32x2(f32x2(__uint_as_float(o1[c]), __uint_as_float(o1[c + 1])), a2), x0, x1);
              o1[c] = __float_as_uint(x0);
              o1[c + 1] = __float_as_uint(x1);
            }
            tmem_st_32x32b_x32(t_o + 0, o0);
            tmem_st_32x32b_x32(t_o + 32, o1);
          }
        }
        {
          uint32_t p0[32], p1[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            p0[c] = pk[c];
            p1[c] = pk[32 + c];
          }
          tmem_st_32x32b_x32(t_p + 0, p0);
          tmem_st_32x32b_x32(t_p + 32, p1);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        if (lane == 0 && (warp == 4 || warp == 8)) GQA_TRACE_EVENT(0, warp == 4 ? 9 : 11, step);
        mbar_arrive(&bars->p_full[t]);
        l_run = l_run * alpha + sum;
        m_run = m_new;
        return true;
      };
      if (fast) {
        for (; ok && it < n; ++it, ++ts) ok = tile(std::true_type{});
      } else {
        for (; ok && it < n; ++it, ++ts) ok = tile(std::false_type{});
      }
      if (!ok) break;
      // ---- epilogue of the unit: O_t / l -> bf16, LSE
      if (!mbar_wait(&bars->o_full[t], uo & 1, ab, p.status, kTimeoutCode)) { ok = false; break; }
      if (lane == 0 && warp == 4 && k == 0) GQA_TRACE_EVENT(0, 12, 0);
      tc_fence_after_sync();
      uint32_t o0[32], o1[32];
      tmem_ld_32x32b_x32(t_o + 0, o0);
      tmem_ld_32x32b_x32(t_o + 32, o1);
      tmem_wait_ld();
      reg_fence(o0);
      reg_fence(o1);
      // O_t is in registers: the next unit's first P.V may overwrite it
      tc_fence_before_sync();
      mbar_arrive(&bars->o_empty[t]);
      ++uo;
      const int h = un.h0 + t;
      const size_t row = (static_cast<size_t>(un.b) * p.H + h) * p.S + i;
      if (i < p.S && GQA_CHECK(p.status, h < p.H && row < static_cast<size_t>(p.B) * p.H * p.S)) {
        const float inv_l = 1.f / l_run;
        uint4 *dst = reinterpret_cast<uint4 *>(p.o + row * HD);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(o0[8 * c + 0]) * inv_l, __uint_as_float(o0[8 * c + 1]) * inv_l);
          w.y = pack_bf16x2(__uint_as_float(o0[8 * c + 2]) * inv_l, __uint_as_float(o0[8 * c + 3]) * inv_l);
          w.z = pack_bf16x2(__uint_as_float(o0[8 * c + 4]) * inv_l, __uint_as_float(o0[8 * c + 5]) * inv_l);
          w.w = pack_bf16x2(__uint_as_float(o0[8 * c + 6]) * inv_l, __uint_as_float(o0[8 * c + 7]) * inv_l);
          dst[c] = w;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(o1[8 * c + 0]) * inv_l, __uint_as_float(o1[8 * c + 1]) * inv_l);
          w.y = pack_bf16x2(__uint_as_float(o1[8 * c + 2]) * inv_l, __uint_as_float(o1[8 * c + 3]) * inv_l);
          w.z = pack_bf16x2(__uint_as_float(o1[8 * c + 4]) * inv_l, __uint_as_float(o1[8 * c + 5]) * inv_l);
          w.w = pack_bf16x2(__uint_as_float(o1[8 * c + 6]) * inv_l, __uint_as_float(o1[8 * c + 7]) * inv_l);
          dst[4 + c] = w;
        }
        // natural-log LSE of the scaled scores: (m + log2 l) * ln 2
        p.lse[row] = (m_run + __log2f(l_run)) * 0.69314718055994530942f;
      }
      if (lane == 0 && warp == 4 && k == 0) GQA_TRACE_EVENT(0, 13, 0);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0) GQA_TRACE_EVENT(0, 15, 0);
  if (warp == 2) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, TMEM_COLS);
  }
}

// Pre-pass of the score bound: for each kv head bg = b * G + g,
// kn2[bg * kKnParts + part] = max |k_j|^2 over the keys of slice `part` of
// [0, S) (fp32 sums of the squared bf16 elements; 0 for an empty slice).  One
// CTA per (kv head, slice); 8 lanes per key row (16 bytes each), 32 rows per
// pass of the CTA, and kKnormUnroll passes' loads issued before any is used,
// so each thread keeps several 16-byte loads in flight.  fmaxf drops NaN rows
// (their scores are NaN whatever the reference); an infinite row gives an
// infinite bound, hence the exact step.
constexpr int kKnormThreads = 256;
constexpr int kKnormUnroll = 8;  // 256 rows (32 KB) per CTA pass: one slice of S = 8192 at once
__global__ void __launch_bounds__(kKnormThreads)
    fwd_knorm_kernel(const __nv_bfloat16 *__restrict__ k, int S, float *__restrict__ kn2) {
  constexpr int kRowsPerPass = kKnormThreads / 8;
  const int bg = blockIdx.x / kKnParts, part = blockIdx.x % kKnParts;
  const int per = (S + kKnParts - 1) / kKnParts;
  const int r0 = min(S, part * per), r1 = min(S, r0 + per);
  const uint4 *rows = reinterpret_cast<const uint4 *>(k + static_cast<size_t>(bg) * S * HD);
  const int sub = threadIdx.x >> 3, ch = threadIdx.x & 7;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float m = 0.f;
  // the loop bound is uniform in the block, so every lane reaches the shuffles
  for (int rb = r0; rb < r1; rb += kRowsPerPass * kKnormUnroll) {
    uint4 w[kKnormUnroll];
#pragma unroll
    for (int u = 0; u < kKnormUnroll; ++u) {
      const int row = rb + kRowsPerPass * u + sub;
      w[u] = row < r1 ? __ldg(rows + static_cast<size_t>(row) * (HD / 8) + ch) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kKnormUnroll; ++u) {
      const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
      float sq = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = __uint_as_float(ws[e] << 16), hi = __uint_as_float(ws[e] & 0xffff0000u);
        sq = fmaf(lo, lo, fmaf(hi, hi, sq));
      }
      sq += __shfl_xor_sync(0xffffffffu, sq, 1);
      sq += __shfl_xor_sync(0xffffffffu, sq, 2);
      sq += __shfl_xor_sync(0xffffffffu, sq, 4);
      m = fmaxf(m, sq);
    }
  }
#pragma unroll
  for (int o = 8; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float wmax[kKnormThreads / 32];
  if (lane == 0) wmax[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = wmax[0];
#pragma unroll
    for (int x = 1; x < kKnormThreads / 32; ++x) b = fmaxf(b, wmax[x]);
    kn2[blockIdx.x] = b;
  }
}

}  // namespace fwd
}  // namespace gqa
