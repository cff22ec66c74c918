// bwd_kernels.cuh -- backward of causal grouped-query attention on sm_103a.
//
// Given dO = dL/dO, with P recomputed from the forward's saved LSE
// ("SnapKitty Transformer 8B", section "Protected Inventions": S/P
// recomputation from the saved row statistics, dP = dO.V^T,
// dS = P * (dP - D), dQ reduced across query tiles; the softmax backward
// ds_j = a_j (g_j - sum_k a_k g_k) of "nx_f32_gqa_gate.nx source", test T4):
//
//   D_i   = sum_c dO_ic O_ic                         (= sum_j P_ij dP_ij)
//   P_ij  = exp(scale q_i.k_j - LSE_i),  dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - D_i)
//   dQ_i  = scale sum_j dS_ij k_j
//   dK_j  = scale sum_{h in group} sum_i dS_ij q_i,    dV_j = sum_{h in group} sum_i P_ij dO_i
//
// Four launches on the caller's stream (after clearing one int per kv group):
//   prep   per query row i: the power of two 2^e_i that brings max_c |dO_ic|
//          into [2^14, 2^15); an fp16 copy dO' = dO * 2^e_i (exact: fp16 holds
//          every bf16 value within 2^29 of the row's largest); D' = 2^e_i D
//          (fp32); LSE * log2(e) + e_i (fp32); E_g = min_i e_i over kv group g;
//          the fp32 dQ accumulator cleared;
//   shift  LSE * log2(e) + e_i - E_g, so that the recomputed probabilities come
//          out as P' = P 2^(E_g - e_i) <= P;
//   main   one CTA per (b, kv head g, 128-key tile): V' = V 2^ev_j in fp16 in
//          shared memory (one power of two per key row, taken once); then for
//          each of the R query heads of g and each query tile that sees the key
//          tile (a "step"), on tcgen05:
//            S^T  = K Q^T  (bf16)      dP''^T = V' dO'^T  (fp16)   (TMEM, fp32)
//            P'^T (fp16) -> TMEM; dS' = P' (dP'' 2^-ev_j - D') = 2^E_g dS
//            (bf16) -> shared memory, which serves as dS'^T (K-major) for dK
//            and as dS' (MN-major) for dQ
//            dV  += P'^T dO' (fp16)   dK  += dS'^T Q (bf16)   (TMEM, fp32, whole CTA life)
//            dQ   = dS' K (bf16)       -> fp32 TMA reduce-add into the accumulator
//          (every accumulator holds 2^E_g times its gradient; the epilogues
//          take the power of two back out exactly).  The fp16 P' and dO' give
//          the dV product 11-bit operands where bf16 would give 8;
//          S^T, dP^T of step n+1 are issued as soon as the P/dS warps have read
//          all of step n into registers, so those warps overlap step n's dV, dK,
//          dQ; three issuing threads (S^T and dP^T; dV and dK; dQ) keep a
//          step's dQ, which waits for the drain, from holding back the rest;
//          P^T and dS are handed over separately (dV starts while dS is still
//          being written) and freed separately (after dV, after dK and dQ).
//          dS alternates between two shared-memory tiles by step, so each half
//          of a row is stored as soon as it is computed: the tile being written
//          was last read by the products of step n - 2, long finished, while
//          step n - 1's dK and dQ still read the other one.
//          dK, dV are summed over the group's heads inside the CTA
//          (deterministic) and written once as bf16;
//   convert dQ = bf16(scale * 2^-E_g * accumulator).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include <cstddef>
#include <cstdint>

#include "bwd_order.cuh"
#include "device_checks.cuh"
#include "error_detail.cuh"
#include "sm100_ptx.cuh"
#include "timing.cuh"
#include "trace.cuh"

namespace gqa {
namespace bwd {

constexpr int BQ = 128;  // query rows per tile
constexpr int BK = 128;  // keys per CTA
constexpr int HD = 64;
constexpr int TILE_BYTES = 128 * HD * 2;  // 16 KB bf16 tile, 128-byte rows
constexpr int NSTAGE = 3;                 // Q/dO ring depth
constexpr int NTHREADS = 512;
// Registers per thread after the split: warps 0-3 (producer, three MMA
// issuers, TMEM alloc), the two P/dS warpgroups (which hold a whole step's
// S^T and dP^T rows), the dQ drain warpgroup.
constexpr int kRegsControl = 56;
constexpr int kRegsSoftmax = 184;
constexpr int kRegsDrain = 80;
// the launch allocation must cover the split (checked on the host)
constexpr int kMinLaunchRegs =
    (128 * (kRegsControl + kRegsDrain) + 256 * kRegsSoftmax + NTHREADS - 1) / NTHREADS;
constexpr uint32_t TMEM_COLS = 512;
// TMEM columns
constexpr uint32_t C_S = 0;     // S^T (128 fp32)
constexpr uint32_t C_DP = 128;  // dP^T (128 fp32)
constexpr uint32_t C_PT = 256;  // P^T (64 columns of bf16 pairs: 128 queries)
constexpr uint32_t C_DV = 320;  // dV accumulator (64 fp32)
constexpr uint32_t C_DK = 384;  // dK accumulator (64 fp32)
constexpr uint32_t C_DQ = 448;  // dQ tile (64 fp32)

// shared memory map (offsets from a 1024-aligned base)
constexpr int SM_K = 0;
constexpr int SM_V = SM_K + TILE_BYTES;
constexpr int SM_Q = SM_V + TILE_BYTES;                 // NSTAGE tiles
constexpr int SM_DO = SM_Q + NSTAGE * TILE_BYTES;       // NSTAGE tiles
constexpr int DS_BYTES = 2 * TILE_BYTES;                 // one dS tile: two 64-query halves
constexpr int SM_DS = SM_DO + NSTAGE * TILE_BYTES;      // two dS tiles, alternating by step
constexpr int SM_DQ = SM_DS + 2 * DS_BYTES;             // 16 KB fp32 dQ staging (32 columns)
constexpr int SM_VEC = SM_DQ + TILE_BYTES;              // NSTAGE x (LSE2[128], D[128]) fp32
constexpr int SM_BARS = SM_VEC + NSTAGE * 2 * BQ * 4;

struct Bars {
  uint64_t kv_full;
  uint64_t v_ready;   // V' (fp16) written over V in shared memory (128 threads of P/dS group 0)
  uint64_t qdo_full[NSTAGE];
  uint64_t qdo_empty[NSTAGE];
  uint64_t st_full;   // S^T, dP^T of the step ready (issuer A commit)
  uint64_t st_free;   // S^T, dP^T read into registers (256 P/dS threads)
  uint64_t pt_ready;  // P^T stored in TMEM (256 P/dS threads)
  uint64_t ds_ready;  // dS stored in shared memory (256 P/dS threads)
  uint64_t pt_free;   // dV of the step finished: P^T may be overwritten (issuer B commit)
  uint64_t ds_free[2];  // dK and dQ finished with dS tile t (issuer B and C commits, steps t, t+2, ...)
  uint64_t dq_full;   // dQ tile ready (issuer C commit)
  uint64_t dq_free;   // dQ tile read out (128 drain threads)
  uint64_t a_done;    // every product of issuer A finished
  uint64_t dkv_done;  // every product of issuer B finished
  uint64_t q_done;    // every product of issuer C finished
  uint32_t tmem_base;
  AbortState abort;
};

constexpr int SMEM_BYTES = 1024 + SM_BARS + static_cast<int>(sizeof(Bars));
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

struct Problem {
  int B, H, G, S;
  int causal, window, n_sink;
  float scale;
};

// Element type of the dq, dk and dv outputs.  A test build of the library
// (-DGQA_FP32_GRAD_OUT) writes them as fp32, straight from the fp32
// accumulators, so that tests can measure the error of the gradients before
// the final bf16 rounding; release builds write bf16.
#ifdef GQA_FP32_GRAD_OUT
using GradOut = float;
#else
using GradOut = __nv_bfloat16;
#endif

// Stores 8 consecutive gradient elements a[0..7] * f at dst.
__device__ __forceinline__ void store_grad8(GradOut *dst, const uint32_t *a, float f) {
#ifdef GQA_FP32_GRAD_OUT
  float4 *d = reinterpret_cast<float4 *>(dst);
  d[0] = make_float4(__uint_as_float(a[0]) * f, __uint_as_float(a[1]) * f,
                     __uint_as_float(a[2]) * f, __uint_as_float(a[3]) * f);
  d[1] = make_float4(__uint_as_float(a[4]) * f, __uint_as_float(a[5]) * f,
                     __uint_as_float(a[6]) * f, __uint_as_float(a[7]) * f);
#else
  uint4 w;
  w.x = pack_bf16x2(__uint_as_float(a[0]) * f, __uint_as_float(a[1]) * f);
  w.y = pack_bf16x2(__uint_as_float(a[2]) * f, __uint_as_float(a[3]) * f);
  w.z = pack_bf16x2(__uint_as_float(a[4]) * f, __uint_as_float(a[5]) * f);
  w.w = pack_bf16x2(__uint_as_float(a[6]) * f, __uint_as_float(a[7]) * f);
  *reinterpret_cast<uint4 *>(dst) = w;
#endif
}

struct MainParams {
  int B, H, G, S, R, S_pad;
  int causal, window, n_sink;
  float scale;
  float scale_log2;
  int n_ktiles;
  int n_front;      // CTA order (bwd_order.cuh): the first n_front key tiles of every kv head first,
  int n_small;      // then batches of the others: the first n_small batches hold
  int batch_pairs;  // batch_pairs kv heads, the others batch_pairs + 1
  const float *lse2;  // [B*H][S_pad]  LSE log2(e) + e_i - E_g
  const float *delta; // [B*H][S_pad]  D' = 2^e_i D
  const int *emin;    // [B*G]         E_g
  GradOut *dk;
  GradOut *dv;
  int *status;
};

enum : int { kTimeoutCode = -9 };


__host__ __device__ inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Scratch of one backward call, carved from the caller's workspace (every
// piece starts on a 16-byte boundary):
//   dq_acc  fp32 [B*H][S][64]     lse2, delta  fp32 [B*H][S_pad]
//   dout_h  fp16 [B*H][S][64]     emin  int32 [B*G] (rounded up to 16 bytes)
struct Workspace {
  float *dq_acc;
  float *lse2;
  float *delta;
  __half *dout_h;
  int *emin;
};

inline size_t workspace_bytes(int B, int H, int G, int S) {
  const size_t rows = static_cast<size_t>(B) * H * S;
  const size_t rows_pad = static_cast<size_t>(B) * H * round_up(S, BQ);
  const size_t groups = (static_cast<size_t>(B) * G * sizeof(int) + 15) / 16 * 16;
  return rows * HD * sizeof(float) + 2 * rows_pad * sizeof(float) + rows * HD * sizeof(__half) +
         groups;
}

inline Workspace carve_workspace(void *ws, int B, int H, int S) {
  const size_t rows = static_cast<size_t>(B) * H * S;
  const size_t rows_pad = static_cast<size_t>(B) * H * round_up(S, BQ);
  Workspace w;
  w.dq_acc = static_cast<float *>(ws);
  w.lse2 = w.dq_acc + rows * HD;
  w.delta = w.lse2 + rows_pad;
  w.dout_h = reinterpret_cast<__half *>(w.delta + rows_pad);
  w.emin = reinterpret_cast<int *>(w.dout_h + rows * HD);
  return w;
}

// The row exponent e with 2^e * m in [2^14, 2^15) for a finite normal m =
// max |x| of a row, clamped to [-kEClamp, kEClamp]; rows of zeros (and of
// subnormals) take the largest shift.  2^e is then exact in fp32 and the
// scaled row fits fp16 without overflow.
constexpr int kEClamp = 120;
__device__ __forceinline__ int row_exponent(float m) {
  const int be = (__float_as_int(m) >> 23) & 0xff;
  const int e = be == 0 ? kEClamp : 141 - be;  // 14 - (be - 127)
  return max(-kEClamp, min(kEClamp, e));
}

// Query tiles [qlo, qhi] that see at least one key of key tile kb.
__device__ __forceinline__ void q_range(int kb, const MainParams &p, int &qlo, int &qhi) {
  const int nq = (p.S + BQ - 1) / BQ;
  if (!p.causal) {
    qlo = 0;
    qhi = nq - 1;
    return;
  }
  const int j0 = kb * BK, j1 = min(j0 + BK - 1, p.S - 1);
  qlo = j0 / BQ;
  if (p.window > 0 && j0 >= p.n_sink) {
    const long long last = static_cast<long long>(j1) + p.window - 1;  // newest query seeing j1
    qhi = static_cast<int>(min(static_cast<long long>(nq - 1), last / BQ));
  } else {
    qhi = nq - 1;
  }
}

// True when some (query, key) pair of the tile pair is masked.
__device__ __forceinline__ bool pair_needs_mask(int qb, int kb, const MainParams &p) {
  const int i0 = qb * BQ, i1 = i0 + BQ - 1, j0 = kb * BK, j1 = j0 + BK - 1;
  if (i1 >= p.S || j1 >= p.S) return true;
  if (!p.causal) return false;
  if (j1 > i0) return true;
  if (p.window > 0) {
    const bool all_in_window = j0 > i1 - p.window;
    const bool all_sinks = j1 < p.n_sink;
    if (!all_in_window && !all_sinks) return true;
  }
  return false;
}

// ------------------------------------------------------------------- prep

// Per row r of [B*H][S_pad] (rows past S: D' = LSE2 = 0, no dO' row):
//   e_r = row_exponent(max_c |dO_rc|),  dO'_r = fp16(dO_r 2^e_r),
//   D'_r = 2^e_r rowsum(dO_r * O_r),  LSE2_r = LSE_r log2(e) + e_r,
//   E_g = min e_r over the rows of kv group g (emin cleared to a large value
//   before the launch), and the fp32 dQ accumulator rows cleared.
// Each block takes one contiguous range of rows (a multiple of 64); eight
// lanes share one 128-byte row, so a warp covers eight rows per pass (two
// groups of four whose loads are all issued before either is used).  Eight
// consecutive rows always lie in one (b, h), so a warp folds its rows' e into
// one running minimum per kv group and flushes it with one atomicMin when the
// group changes.
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16 *__restrict__ o,
                                                       const __nv_bfloat16 *__restrict__ dout,
                                                       const float *__restrict__ lse,
                                                       float *__restrict__ lse2,
                                                       float *__restrict__ delta,
                                                       float *__restrict__ dq_acc,
                                                       __half *__restrict__ dout_h,
                                                       int *__restrict__ emin,
                                                       long long rows_pad, int S, int S_pad,
                                                       int H, int G, int R) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int sub = lane >> 3;  // row within a group of four
  const int ch = lane & 7;    // 16-byte chunk of the row
  const long long per_block =
      ((rows_pad + gridDim.x - 1) / gridDim.x + 63) / 64 * 64;
  const long long r_begin = static_cast<long long>(blockIdx.x) * per_block;
  const long long r_end = min(rows_pad, r_begin + per_block);
  int cur_g = -1, cur_min = 0x7fffffff;
  for (long long r0 = r_begin + warp * 8; r0 < r_end; r0 += 64) {  // warp-uniform bound
    const long long bh = r0 / S_pad;
    const int grp = static_cast<int>(bh / H) * G + static_cast<int>(bh % H) / R;
    long long src[2];
    uint4 a[2], c[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int i = static_cast<int>(r0 + 4 * u + sub - bh * S_pad);
      src[u] = -1;
      a[u] = c[u] = make_uint4(0, 0, 0, 0);
      if (i < S) {
        src[u] = bh * S + i;
        a[u] = reinterpret_cast<const uint4 *>(o + src[u] * HD)[ch];
        c[u] = reinterpret_cast<const uint4 *>(dout + src[u] * HD)[ch];
      }
    }
    int e_min = 0x7fffffff;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const long long r = r0 + 4 * u + sub;
      float acc = 0.f, m = 0.f;
      float y[8];
      const __nv_bfloat162 *a2 = reinterpret_cast<const __nv_bfloat162 *>(&a[u]);
      const __nv_bfloat162 *c2 = reinterpret_cast<const __nv_bfloat162 *>(&c[u]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(a2[e]);
        const float2 d = __bfloat1622float2(c2[e]);
        acc = fmaf(x.x, d.x, acc);
        acc = fmaf(x.y, d.y, acc);
        m = fmaxf(m, fmaxf(fabsf(d.x), fabsf(d.y)));
        y[2 * e] = d.x;
        y[2 * e + 1] = d.y;
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 4);
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
      const int er = row_exponent(m);
      const float sc = exp2i(er);
      if (src[u] >= 0) {
        float4 *z = reinterpret_cast<float4 *>(dq_acc + src[u] * HD) + 2 * ch;
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        uint4 hw;
        hw.x = pack_f16x2(y[0] * sc, y[1] * sc);
        hw.y = pack_f16x2(y[2] * sc, y[3] * sc);
        hw.z = pack_f16x2(y[4] * sc, y[5] * sc);
        hw.w = pack_f16x2(y[6] * sc, y[7] * sc);
        reinterpret_cast<uint4 *>(dout_h + src[u] * HD)[ch] = hw;
        e_min = min(e_min, er);
      }
      if (r < rows_pad && ch == 0) {
        delta[r] = src[u] >= 0 ? acc * sc : 0.f;
        lse2[r] = src[u] >= 0 ? fmaf(lse[src[u]], 1.4426950408889634f, static_cast<float>(er)) : 0.f;
      }
    }
    // the warp's eight rows: one minimum
#pragma unroll
    for (int o2 = 8; o2 < 32; o2 <<= 1) e_min = min(e_min, __shfl_xor_sync(0xffffffffu, e_min, o2));
    if (grp != cur_g) {
      if (lane == 0 && cur_g >= 0 && cur_min != 0x7fffffff) atomicMin(emin + cur_g, cur_min);
      cur_g = grp;
      cur_min = e_min;
    } else {
      cur_min = min(cur_min, e_min);
    }
  }
  if (lane == 0 && cur_g >= 0 && cur_min != 0x7fffffff) atomicMin(emin + cur_g, cur_min);
}

// LSE2_r -= E_g for every row r of [B*H][S_pad] (four rows per thread and
// pass; S_pad is a multiple of 4, so the four share one (b, h)).
__global__ void __launch_bounds__(256) bwd_shift_kernel(float *__restrict__ lse2,
                                                        const int *__restrict__ emin,
                                                        long long n4, int S_pad, int H, int G,
                                                        int R) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < n4;
       e += stride) {
    const long long bh = 4 * e / S_pad;
    const int grp = static_cast<int>(bh / H) * G + static_cast<int>(bh % H) / R;
    const float E = static_cast<float>(emin[grp]);
    float4 x = reinterpret_cast<float4 *>(lse2)[e];
    x.x -= E;
    x.y -= E;
    x.z -= E;
    x.w -= E;
    reinterpret_cast<float4 *>(lse2)[e] = x;
  }
}

// ---------------------------------------------------------------- convert

// dq = bf16(scale * 2^-E_g * dq_acc), eight elements (an eighth of a row) per
// thread and pass.
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float *__restrict__ dq_acc,
                                                             GradOut *__restrict__ dq,
                                                             const int *__restrict__ emin,
                                                             long long n8, float scale, int S,
                                                             int H, int G, int R) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < n8;
       e += stride) {
    const long long bh = (e >> 3) / S;
    const int grp = static_cast<int>(bh / H) * G + static_cast<int>(bh % H) / R;
    const float f = scale * exp2i(-emin[grp]);
    const uint4 a = reinterpret_cast<const uint4 *>(dq_acc)[2 * e];
    const uint4 b = reinterpret_cast<const uint4 *>(dq_acc)[2 * e + 1];
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    store_grad8(dq + 8 * e, v, f);
  }
}

// ------------------------------------------------------------------- main

// The n lowest bits set (n clamped to [0, 32]).
__device__ __forceinline__ uint32_t low_bits(int n) {
  return n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : (1u << n) - 1u);
}

// Visibility of query columns [cb, cb+32) of the tile for key row j, one bit
// per column.  For a fixed key the visible queries of a tile form one range
// [c_lo, c_hi) of columns: causality bounds it below (i >= j), the window
// above (i < j + window, unless j is a sink), and the sequence end above.
__device__ __forceinline__ uint32_t visible_bits(int cb, int i0, int j, const MainParams &p) {
  if (j >= p.S) return 0u;
  const int c_lo = p.causal ? j - i0 : 0;
  int c_hi = p.S - i0;
  if (p.causal && p.window > 0 && j >= p.n_sink) c_hi = min(c_hi, j - i0 + min(p.window, p.S));
  return low_bits(c_hi - cb) & ~low_bits(c_lo - cb);
}

// P and dS of 32 query columns [cb, cb+32) for this thread's key row; `vbits`
// holds their visibility when the tile pair needs the mask.
// P' goes out as fp16 pairs (pp), dS' = P' (dP'' cv - D') as bf16 pairs (pd);
// cv = 2^-ev_j takes this key row's V scale out of dP''.
__device__ __forceinline__ void p_ds_chunk(const uint32_t (&sr)[32], const uint32_t (&dr)[32],
                                           const float *lse2, const float *dlt, int cb,
                                           uint32_t vbits, bool masked, float sl2, float cv,
                                           uint32_t (&pp)[16], uint32_t (&pd)[16]) {
  // sub-chunks of 8 query columns: two broadcast 16-byte shared loads for the
  // 8 LSE2 and two for the 8 D values, so few values are live at once
#pragma unroll
  for (int sc = 0; sc < 4; ++sc) {
    const float4 la = reinterpret_cast<const float4 *>(lse2 + cb)[2 * sc];
    const float4 lb = reinterpret_cast<const float4 *>(lse2 + cb)[2 * sc + 1];
    const float4 da = reinterpret_cast<const float4 *>(dlt + cb)[2 * sc];
    const float4 db = reinterpret_cast<const float4 *>(dlt + cb)[2 * sc + 1];
    const float l8[8] = {la.x, la.y, la.z, la.w, lb.x, lb.y, lb.z, lb.w};
    const float d8[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
    float pv[8], dv[8];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      float x0, x1;
      f32x2_split(fma_f32x2(f32x2(__uint_as_float(sr[8 * sc + e]), __uint_as_float(sr[8 * sc + e + 1])),
                            f32x2(sl2, sl2), f32x2(-l8[e], -l8[e + 1])),
                  x0, x1);
      pv[e] = ex2_approx(x0);
      pv[e + 1] = ex2_approx(x1);
    }
    if (masked) {
#pragma unroll
      for (int e = 0; e < 8; ++e) pv[e] = ((vbits >> (8 * sc + e)) & 1u) ? pv[e] : 0.f;
    }
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      float y0, y1;
      f32x2_split(mul_f32x2(f32x2(pv[e], pv[e + 1]),
                            fma_f32x2(f32x2(__uint_as_float(dr[8 * sc + e]), __uint_as_float(dr[8 * sc + e + 1])),
                                      f32x2(cv, cv), f32x2(-d8[e], -d8[e + 1]))),
                  y0, y1);
      dv[e] = y0;
      dv[e + 1] = y1;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      pp[4 * sc + e] = pack_f16x2(pv[2 * e], pv[2 * e + 1]);
      pd[4 * sc + e] = pack_bf16x2(dv[2 * e], dv[2 * e + 1]);
    }
  }
}

__global__ void __launch_bounds__(NTHREADS, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const MainParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled tiles, by pointer arithmetic on the
  // __shared__ array so that accesses stay shared-space (ld/st.shared).
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars *bars = reinterpret_cast<Bars *>(smem + SM_BARS);
  float *vec = reinterpret_cast<float *>(smem + SM_VEC);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // work unit (cta_unit): batches of kv heads, key tiles with the most query
  // tiles first in each
  int kb, pair;
  cta_unit(static_cast<int>(blockIdx.x), p.n_ktiles, p.n_front, p.B * p.G, p.n_small, p.batch_pairs,
           kb, pair);
  const int b = pair / p.G;
  const int g = pair % p.G;
  int qlo, qhi;
  q_range(kb, p, qlo, qhi);
  const int nqt = qhi - qlo + 1;
  const int nsteps = p.R * nqt;  // (head, query tile) steps, heads outer

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->v_ready, 128);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&bars->qdo_full[s], 1);
      mbar_init(&bars->qdo_empty[s], 1);
    }
    mbar_init(&bars->st_full, 1);
    mbar_init(&bars->st_free, 256);
    mbar_init(&bars->pt_ready, 256);
    mbar_init(&bars->ds_ready, 256);
    mbar_init(&bars->pt_free, 1);
    mbar_init(&bars->ds_free[0], 2);
    mbar_init(&bars->ds_free[1], 2);
    mbar_init(&bars->q_done, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, 128);
    mbar_init(&bars->a_done, 1);
    mbar_init(&bars->dkv_done, 1);
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
  if (threadIdx.x == 0) GQA_TRACE_EVENT(1, 15, 0);

  if (warp < 4) {
    setmaxnreg_dec<kRegsControl>();
    if (warp == 0 && lane == 0) {
      // ========================================================== producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      const int kvz = b * p.G + g;
      GQA_REPORT(p.status, kb >= 0 && kb * BK < p.S && kvz < p.B * p.G && qlo <= qhi);
      mbar_arrive_expect_tx(&bars->kv_full, 2 * TILE_BYTES);
      tma_load_3d(smem + SM_K, &tm_k, &bars->kv_full, 0, kb * BK, kvz);
      tma_load_3d(smem + SM_V, &tm_v, &bars->kv_full, 0, kb * BK, kvz);
      int issued = 0;
      for (int n = 0; n < nsteps; ++n) {
        const int st = n % NSTAGE;
        const uint32_t ph = (n / NSTAGE) & 1;
        const int h = g * p.R + n / nqt;
        const int qb = qlo + n % nqt;
        const int bh = b * p.H + h;
        if (!mbar_wait<true>(&bars->qdo_empty[st], ph ^ 1, ab, p.status, kTimeoutCode)) break;
        GQA_TRACE_EVENT(1, 0, n);
#ifdef GQA_INJECT_STALL
        // failure-detection test build only: CTA 0 never loads one step's Q/dO
        if (blockIdx.x == 0 && n == min(1, nsteps - 1)) {
          issued = n + 1;
          continue;
        }
#endif
        GQA_REPORT(p.status, h < p.H && qb >= 0 && qb * BQ < p.S &&
                                static_cast<size_t>(bh) * p.S_pad + (qb + 1) * BQ <=
                                    static_cast<size_t>(p.B) * p.H * p.S_pad);
        mbar_arrive_expect_tx(&bars->qdo_full[st], 2 * TILE_BYTES + 2 * BQ * 4);
        tma_load_3d(smem + SM_Q + st * TILE_BYTES, &tm_q, &bars->qdo_full[st], 0, qb * BQ, bh);
        tma_load_3d(smem + SM_DO + st * TILE_BYTES, &tm_do, &bars->qdo_full[st], 0, qb * BQ, bh);
        const size_t voff = static_cast<size_t>(bh) * p.S_pad + static_cast<size_t>(qb) * BQ;
        bulk_load(vec + st * 2 * BQ, p.lse2 + voff, BQ * 4, &bars->qdo_full[st]);
        bulk_load(vec + st * 2 * BQ + BQ, p.delta + voff, BQ * 4, &bars->qdo_full[st]);
        GQA_TRACE_EVENT(1, 1, n);
        issued = n + 1;
      }
      mbar_wait_drain(&bars->kv_full, 0);
      for (int n = max(0, issued - NSTAGE); n < issued; ++n)
        mbar_wait_drain(&bars->qdo_full[n % NSTAGE], (n / NSTAGE) & 1);
    } else if (warp == 1 && lane == 0) {
      // ================================================= issuer A: S^T, dP^T
      const uint32_t id_nn = idesc_bf16_f32(128, 128, false, false);    // S^T: K, Q bf16
      const uint32_t id_nn16 = idesc_fp16_f32(128, 128, false, false);  // dP''^T: V', dO' fp16
      const uint64_t k_kmaj = sdesc_sw128(smem_u32(smem + SM_K), 16, 1024);
      const uint64_t v_kmaj = sdesc_sw128(smem_u32(smem + SM_V), 16, 1024);
      const uint32_t q_addr = smem_u32(smem + SM_Q);
      const uint32_t do_addr = smem_u32(smem + SM_DO);
      bool ok = mbar_wait<true>(&bars->kv_full, 0, ab, p.status, kTimeoutCode);
      for (int n = 0; ok && n < nsteps; ++n) {
        const int st = n % NSTAGE;
        GQA_TRACE_EVENT(1, 21, n);  // issuer A starts waiting for the step's Q and dO
        if (!mbar_wait<true>(&bars->qdo_full[st], (n / NSTAGE) & 1, ab, p.status, kTimeoutCode)) { ok = false; break; }
        GQA_TRACE_EVENT(1, 22, n);
        // V' (fp16) must be in place before the first dP''^T
        if (n == 0 && !mbar_wait<true>(&bars->v_ready, 0, ab, p.status, kTimeoutCode)) { ok = false; break; }
        // the P/dS warps must have read the previous step's S^T and dP^T
        if (n > 0 && !mbar_wait<true>(&bars->st_free, (n - 1) & 1, ab, p.status, kTimeoutCode)) { ok = false; break; }
        GQA_TRACE_EVENT(1, 2, n);
        tc_fence_after_sync();
        const uint64_t q_kmaj = sdesc_sw128(q_addr + st * TILE_BYTES, 16, 1024);
        const uint64_t do_kmaj = sdesc_sw128(do_addr + st * TILE_BYTES, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks)
          mma_bf16_ss(tbase + C_S, k_kmaj + 2 * ks, q_kmaj + 2 * ks, id_nn, ks > 0);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks)
          mma_bf16_ss(tbase + C_DP, v_kmaj + 2 * ks, do_kmaj + 2 * ks, id_nn16, ks > 0);
        mma_commit(&bars->st_full);
        GQA_TRACE_EVENT(1, 3, n);
#ifdef GQA_TRACE
        // trace builds: the time this step's S^T and dP^T are complete, seen by
        // the issuing thread itself (its next wait comes after that anyway)
        if (mbar_wait<true>(&bars->st_full, n & 1, ab, p.status, kTimeoutCode)) GQA_TRACE_EVENT(1, 32, n);
#endif
      }
      mma_commit(&bars->a_done);
      if (!ok) mbar_wait_drain(&bars->a_done, 0);
    } else if (warp == 3 && lane == 0) {
      // ============================================ issuer B: dV, dK
      const uint32_t id_dv = idesc_fp16_f32(128, 64, false, true);  // dV: P'^T, dO' fp16
      const uint32_t id_dk = idesc_bf16_f32(128, 64, false, true);  // dK: dS'^T, Q bf16
      const uint32_t q_addr = smem_u32(smem + SM_Q);
      const uint32_t do_addr = smem_u32(smem + SM_DO);
      const uint32_t ds_addr = smem_u32(smem + SM_DS);
      bool ok = true;
      for (int n = 0; n < nsteps; ++n) {
        const int st = n % NSTAGE;
        const uint64_t q_mn = sdesc_sw128(q_addr + st * TILE_BYTES, TILE_BYTES, 1024);
        const uint32_t ds_t = ds_addr + (n & 1) * DS_BYTES;  // this step's dS tile
        const uint64_t do_mn = sdesc_sw128(do_addr + st * TILE_BYTES, TILE_BYTES, 1024);
        GQA_TRACE_EVENT(1, 20, n);  // issuer B starts waiting for the step's P^T
        if (!mbar_wait<true>(&bars->pt_ready, n & 1, ab, p.status, kTimeoutCode)) { ok = false; break; }
        GQA_TRACE_EVENT(1, 4, n);
        tc_fence_after_sync();
        // dV += P^T dO: P^T from TMEM (16 queries = 8 packed columns per step)
#pragma unroll
        for (int ks = 0; ks < BQ / 16; ++ks)
          mma_bf16_ts(tbase + C_DV, tbase + C_PT + ks * 8, do_mn + ks * 128, id_dv, (n > 0 || ks > 0));
        mma_commit(&bars->pt_free);
        if (!mbar_wait<true>(&bars->ds_ready, n & 1, ab, p.status, kTimeoutCode)) { ok = false; break; }
        tc_fence_after_sync();
        // dK += dS^T Q: dS^T is the shared dS tile read K-major (queries 0-63 in
        // the first 16 KB half, 64-127 in the second; 32 B per 16 queries)
#pragma unroll
        for (int ks = 0; ks < BQ / 16; ++ks) {
          const uint64_t a = sdesc_sw128(ds_t + (ks >> 2) * TILE_BYTES + (ks & 3) * 32, 16, 1024);
          mma_bf16_ss(tbase + C_DK, a, q_mn + ks * 128, id_dk, (n > 0 || ks > 0));
        }
        mma_commit(&bars->qdo_empty[st]);
        mma_commit(&bars->ds_free[n & 1]);
        GQA_TRACE_EVENT(1, 23, n);
      }
      mma_commit(&bars->dkv_done);
      if (!ok) mbar_wait_drain(&bars->dkv_done, 0);
    } else if (warp == 2 && lane == 0) {
      // ============================================ issuer C: dQ
      // On its own thread, so that a step's dQ, which waits for the drain to
      // have read the previous tile, never holds back the next step's dV and dK
      // (one issuer for all three left the tensor pipe idle between steps).
      const uint32_t id_dq = idesc_bf16_f32(128, 64, true, true);  // dQ: dS', K bf16
      const uint32_t ds_addr = smem_u32(smem + SM_DS);
      const uint64_t k_mn = sdesc_sw128(smem_u32(smem + SM_K), TILE_BYTES, 1024);
      bool ok = true;
      for (int n = 0; n < nsteps; ++n) {
        const uint64_t ds_mn = sdesc_sw128(ds_addr + (n & 1) * DS_BYTES, TILE_BYTES, 1024);  // LBO: next 64-query half
        // dS of the step is written (which implies K has landed: S^T read it)
        if (!mbar_wait<true>(&bars->ds_ready, n & 1, ab, p.status, kTimeoutCode)) { ok = false; break; }
        // the drain has read the previous dQ tile out of TMEM
        if (n > 0 && !mbar_wait<true>(&bars->dq_free, (n - 1) & 1, ab, p.status, kTimeoutCode)) { ok = false; break; }
        GQA_TRACE_EVENT(1, 5, n);
        tc_fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks)  // 16 keys = 2048 B of the MN-major operands
          mma_bf16_ss(tbase + C_DQ, ds_mn + ks * 128, k_mn + ks * 128, id_dq, ks > 0);
        mma_commit(&bars->dq_full);
        mma_commit(&bars->ds_free[n & 1]);
        GQA_TRACE_EVENT(1, 6, n);
      }
      mma_commit(&bars->q_done);
      if (!ok) mbar_wait_drain(&bars->q_done, 0);
    }
  } else if (warp < 12) {
    setmaxnreg_inc<kRegsSoftmax>();
    // ============================================================ P / dS
    const int wg = (warp - 4) >> 2;         // query columns 64*wg .. 64*wg+63
    const int lane_base = 32 * (warp & 3);
    const int r = lane_base + lane;         // key row of the tile
    const int j = kb * BK + r;              // key index
    const float sl2 = p.scale_log2;
    const uint32_t lane_off = static_cast<uint32_t>(lane_base) << 16;
    // this thread's key row of its group's 64-query half of a dS tile; chunk c
    // of 8 queries sits at (c ^ (r & 7)) (128-byte swizzle)
    uint8_t *ds_row0 = smem + SM_DS + wg * TILE_BYTES + r * 128;
    // V' = fp16(V 2^ev) in place, one key row per thread: both groups read the
    // row and take cv = 2^-ev, group 0 writes it back once every P/dS thread
    // has read (a barrier every one of the 256 threads reaches, also on abort).
    float cv = 1.f;
    bool ok = mbar_wait_warp<true>(&bars->kv_full, 0, ab, p.status, kTimeoutCode);
    {
      uint8_t *vrow = smem + SM_V + r * 128;  // 16-byte chunk c at (c ^ (r & 7))
      uint4 vv[8];
      float m = 0.f;
      if (ok) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          vv[c] = *reinterpret_cast<const uint4 *>(vrow + ((c ^ (r & 7)) << 4));
          const uint32_t w4[4] = {vv[c].x, vv[c].y, vv[c].z, vv[c].w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w4[e] << 16)),
                               fabsf(__uint_as_float(w4[e] & 0xffff0000u))));
        }
      }
      const int ev = row_exponent(m);
      cv = exp2i(-ev);
      ok = named_bar_and(2, 256, ok);
      if (ok && wg == 0) {
        const float sc = exp2i(ev);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t w4[4] = {vv[c].x, vv[c].y, vv[c].z, vv[c].w};
          uint32_t h4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            h4[e] = pack_f16x2(__uint_as_float(w4[e] << 16) * sc,
                               __uint_as_float(w4[e] & 0xffff0000u) * sc);
          *reinterpret_cast<uint4 *>(vrow + ((c ^ (r & 7)) << 4)) = make_uint4(h4[0], h4[1], h4[2], h4[3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars->v_ready);
      }
    }
    for (int n = 0; ok && n < nsteps; ++n) {
      const int st = n % NSTAGE;
      const int qb = qlo + n % nqt;
      const int i0 = qb * BQ;
      const float *lse2 = vec + st * 2 * BQ;
      const float *dlt = lse2 + BQ;
      if (warp == 4 && lane == 0) GQA_TRACE_EVENT(1, 34, n);
      if (!mbar_wait_warp<true>(&bars->st_full, n & 1, ab, p.status, kTimeoutCode)) { ok = false; break; }
      if (warp == 4 && lane == 0) GQA_TRACE_EVENT(1, 8, n);
      tc_fence_after_sync();
      const bool masked = pair_needs_mask(qb, kb, p);
      uint32_t pp0[16], pd0[16], pp1[16], pd1[16];
      uint32_t sr0[32], dr0[32], sr1[32], dr1[32];
      // the whole step's S^T and dP^T rows into registers first, so that the
      // next step's two products may start while this step is computed
      tmem_ld_32x32b_x32(tbase + lane_off + C_S + 64 * wg, sr0);
      tmem_ld_32x32b_x32(tbase + lane_off + C_DP + 64 * wg, dr0);
      tmem_ld_32x32b_x32(tbase + lane_off + C_S + 64 * wg + 32, sr1);
      tmem_ld_32x32b_x32(tbase + lane_off + C_DP + 64 * wg + 32, dr1);
      tmem_wait_ld();
      reg_fence(sr0);
      reg_fence(dr0);
      reg_fence(sr1);
      reg_fence(dr1);
      tc_fence_before_sync();
      mbar_arrive(&bars->st_free);
      if (warp == 4 && lane == 0) GQA_TRACE_EVENT(1, 9, n);
      p_ds_chunk(sr0, dr0, lse2, dlt, 64 * wg, masked ? visible_bits(64 * wg, i0, j, p) : 0u,
                 masked, sl2, cv, pp0, pd0);
#ifdef GQA_TRACE
      reg_fence(pd0);  // the chunk's results exist before the time is taken
#endif
      if (warp == 4 && lane == 0) GQA_TRACE_EVENT(1, 17, n);
      // dS goes to the step's tile as soon as each half of the row is computed:
      // the tile was last read by the dK and dQ products of step n - 2
      uint8_t *ds_row = ds_row0 + (n & 1) * DS_BYTES;
      if (n >= 2 && !mbar_wait_warp<true>(&bars->ds_free[n & 1], ((n >> 1) - 1) & 1, ab, p.status, kTimeoutCode)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8)
        *reinterpret_cast<uint4 *>(ds_row + ((q8 ^ (r & 7)) << 4)) =
            make_uint4(pd0[4 * q8], pd0[4 * q8 + 1], pd0[4 * q8 + 2], pd0[4 * q8 + 3]);
      if (warp == 4 && lane == 0) GQA_TRACE_EVENT(1, 18, n);
      p_ds_chunk(sr1, dr1, lse2, dlt, 64 * wg + 32,
                 masked ? visible_bits(64 * wg + 32, i0, j, p) : 0u, masked, sl2, cv, pp1, pd1);
#ifdef GQA_TRACE
      reg_fence(pd1);
#endif
      if (warp == 4 && lane == 0) GQA_TRACE_EVENT(1, 19, n);
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8)
        *reinterpret_cast<uint4 *>(ds_row + (((4 + q8) ^ (r & 7)) << 4)) =
            make_uint4(pd1[4 * q8], pd1[4 * q8 + 1], pd1[4 * q8 + 2], pd1[4 * q8 + 3]);
      // the previous step's dV must be done with P^T
      if (n > 0) {
        if (!mbar_wait_warp<true>(&bars->pt_free, (n - 1) & 1, ab, p.status, kTimeoutCode)) { ok = false; break; }
        tc_fence_after_sync();
      }
      if (warp == 4 && lane == 0) GQA_TRACE_EVENT(1, 10, n);
      // P^T: this group's 64 queries are packed columns 32*wg .. 32*wg+31
      tmem_st_32x32b_x16(tbase + lane_off + C_PT + 32 * wg, pp0);
      tmem_st_32x32b_x16(tbase + lane_off + C_PT + 32 * wg + 16, pp1);
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(&bars->pt_ready);
      // the dS stores above become visible to the tensor core's operand reads
      fence_proxy_async_smem();
      if (lane == 0 && (warp == 4 || warp == 8)) GQA_TRACE_EVENT(1, warp == 4 ? 11 : 7, n);
      if (lane == 0) GQA_TRACE_EVENT(1, 20 + warp, n);  // every P/dS warp's hand-over (events 24-31)
      mbar_arrive(&bars->ds_ready);
      if (warp == 4 && lane == 0) GQA_TRACE_EVENT(1, 33, n);
    }
    // epilogue: group 0 writes dV, group 1 writes dK (x scale), one key row per thread
    if (ok && mbar_wait_warp<true>(&bars->dkv_done, 0, ab, p.status, kTimeoutCode)) {
      tc_fence_after_sync();
      uint32_t a0[32], a1[32];
      const uint32_t col = wg == 0 ? C_DV : C_DK;
      tmem_ld_32x32b_x32(tbase + lane_off + col, a0);
      tmem_ld_32x32b_x32(tbase + lane_off + col + 32, a1);
      tmem_wait_ld();
      reg_fence(a0);
      reg_fence(a1);
      if (j < p.S && GQA_CHECK(p.status, b < p.B && g < p.G)) {
        // the accumulators hold 2^E_g times the gradients
        const float unscale = exp2i(-p.emin[b * p.G + g]);
        const float f = wg == 0 ? unscale : p.scale * unscale;
        GradOut *dst = (wg == 0 ? p.dv : p.dk) + ((static_cast<size_t>(b) * p.G + g) * p.S + j) * HD;
#pragma unroll
        for (int c = 0; c < 4; ++c) store_grad8(dst + 8 * c, a0 + 8 * c, f);
#pragma unroll
        for (int c = 0; c < 4; ++c) store_grad8(dst + 32 + 8 * c, a1 + 8 * c, f);
      }
    }
  } else {
    setmaxnreg_dec<kRegsDrain>();
    // ============================================================ dQ drain
    const int lane_base = 32 * (warp & 3);
    const int r = lane_base + lane;  // query row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(lane_base) << 16;
    const bool leader = (warp == 12 && lane == 0);
    uint8_t *stg = smem + SM_DQ + r * 128;
    for (int n = 0; n < nsteps; ++n) {
      const int h = g * p.R + n / nqt;
      const int qb = qlo + n % nqt;
      // The four drain warps meet at named barriers below, so they decide
      // together whether to go on: one warp must never leave while the others
      // wait there for it.
      if (!named_bar_and(1, 128, mbar_wait<true>(&bars->dq_full, n & 1, ab, p.status, kTimeoutCode)))
        break;
      if (leader) GQA_TRACE_EVENT(1, 12, n);
      tc_fence_after_sync();
      uint32_t a0[32], a1[32];
      tmem_ld_32x32b_x32(tbase + lane_off + C_DQ, a0);
      tmem_ld_32x32b_x32(tbase + lane_off + C_DQ + 32, a1);
      tmem_wait_ld();
      reg_fence(a0);
      reg_fence(a1);
      tc_fence_before_sync();
      mbar_arrive(&bars->dq_free);
      // Two passes through the 16 KB staging box, 32 fp32 columns each: [128
      // rows][32 fp32] with the 128-byte swizzle (16-B chunk c of row r at
      // c ^ (r & 7)), then a TMA reduce-add into the fp32 dQ accumulator.
      const bool do_reduce = GQA_CHECK(p.status, h < p.H && qb * BQ < p.S);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t *a = half == 0 ? a0 : a1;
        // the staging box was last read by the previous pass's reduce
        if (leader) bulk_wait_group_read<0>();
        if (leader) GQA_TRACE_EVENT(1, half == 0 ? 13 : 16, n);
        named_bar_sync(1, 128);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4 *>(stg + ((c ^ (r & 7)) << 4)) =
              make_uint4(a[4 * c], a[4 * c + 1], a[4 * c + 2], a[4 * c + 3]);
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (leader && do_reduce) {
          tma_reduce_add_3d(&tm_dq, smem + SM_DQ, 32 * half, qb * BQ, b * p.H + h);
          bulk_commit_group();
        }
      }
      if (leader) GQA_TRACE_EVENT(1, 14, n);
    }
    if (leader) bulk_wait_group_all();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0) GQA_TRACE_EVENT(1, 15, 1);
  if (warp == 2) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, TMEM_COLS);
  }
}

// ------------------------------------------------------------------- host

inline int configure_kernels() {
  if (cuda_failed(cudaFuncSetAttribute(bwd_main_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES),
                  "cudaFuncSetAttribute(backward shared memory)"))
    return -1;
  // the main kernel rebalances registers between warpgroups (setmaxnreg); that
  // is only safe when the compiled launch allocation covers the split
  cudaFuncAttributes fa{};
  if (cuda_failed(cudaFuncGetAttributes(&fa, bwd_main_kernel), "cudaFuncGetAttributes(backward)"))
    return -1;
  if (fa.numRegs < kMinLaunchRegs) {
    set_error_detail("backward kernel compiled with fewer registers than its warpgroup split needs");
    return -1;
  }
  return 0;
}

inline int encode_3d(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap *map,
                     CUtensorMapDataType dt, int esize, const void *base, uint64_t inner,
                     uint64_t rows, uint64_t outer, uint32_t box_inner, uint32_t box_rows) {
  cuuint64_t dims[3] = {inner, rows, outer};
  cuuint64_t strides[2] = {inner * esize, rows * inner * esize};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? 0
             : -1;
}

// Launches prep, shift, main and convert on `st` (after clearing E).
// Returns 0, -2 (sizes the kernels cannot index) or -8 (CUDA failure).
inline int launch(const Problem &pr, const void *q, const void *k, const void *v, const void *o,
                  const void *dout, const float *lse, void *dq, void *dk, void *dv, void *ws,
                  int *status, int sm_count, PFN_cuTensorMapEncodeTiled_v12000 enc,
                  cudaStream_t st) {
  const int B = pr.B, H = pr.H, G = pr.G, S = pr.S, R = H / G;
  const int S_pad = round_up(S, BQ);
  // every size check comes before the first launch
  const long long units = static_cast<long long>((S + BK - 1) / BK) * B * G;
  if (units > 0x7fffffffLL) return -2;
  const long long rows = static_cast<long long>(B) * H * S;
  const long long rows_pad = static_cast<long long>(B) * H * S_pad;
  const Workspace w = carve_workspace(ws, B, H, S);

  CUtensorMap tq, tk, tv, tdo, tdq;
  if (encode_3d(enc, &tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q, HD, S,
                static_cast<uint64_t>(B) * H, HD, BQ) ||
      encode_3d(enc, &tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k, HD, S,
                static_cast<uint64_t>(B) * G, HD, BK) ||
      encode_3d(enc, &tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, v, HD, S,
                static_cast<uint64_t>(B) * G, HD, BK) ||
      encode_3d(enc, &tdo, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, w.dout_h, HD, S,
                static_cast<uint64_t>(B) * H, HD, BQ) ||
      encode_3d(enc, &tdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, w.dq_acc, HD, S,
                static_cast<uint64_t>(B) * H, 32, BQ)) {
    set_error_detail("cuTensorMapEncodeTiled rejected a backward tensor map");
    return -8;
  }

  // E_g starts above any row exponent (0x7f7f7f7f), so atomicMin takes the first value
  if (cuda_failed(cudaMemsetAsync(w.emin, 0x7f, static_cast<size_t>(B) * G * sizeof(int), st),
                  "cudaMemsetAsync(backward group exponents)"))
    return -8;
  {
    long long blocks = (rows_pad + 63) / 64;
    blocks = blocks < 1 ? 1 : (blocks > 8LL * sm_count ? 8LL * sm_count : blocks);
    timing_begin(1, st);
    bwd_prep_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(o), static_cast<const __nv_bfloat16 *>(dout), lse,
        w.lse2, w.delta, w.dq_acc, w.dout_h, w.emin, rows_pad, S, S_pad, H, G, R);
    if (cuda_failed(cudaGetLastError(), "launch of the backward prep kernel")) return -8;
    const long long n4 = rows_pad / 4;
    long long sblocks = (n4 + 255) / 256;
    sblocks = sblocks < 1 ? 1 : (sblocks > 4LL * sm_count ? 4LL * sm_count : sblocks);
    bwd_shift_kernel<<<static_cast<unsigned>(sblocks), 256, 0, st>>>(w.lse2, w.emin, n4, S_pad,
                                                                      H, G, R);
    timing_end(1, st);
    if (cuda_failed(cudaGetLastError(), "launch of the backward shift kernel")) return -8;
  }
  {
    MainParams p{};
    p.B = B;
    p.H = H;
    p.G = G;
    p.S = S;
    p.R = R;
    p.S_pad = S_pad;
    p.causal = pr.causal;
    p.window = pr.window;
    p.n_sink = pr.n_sink;
    p.scale = pr.scale;
    p.scale_log2 = pr.scale * 1.4426950408889634f;
    p.n_ktiles = (S + BK - 1) / BK;
    p.n_front = p.causal ? front_tiles(p.n_ktiles, p.window, p.n_sink, BK) : 0;
    cta_order(B, G, R, S, p.n_ktiles, p.n_front, sm_count, p.n_small, p.batch_pairs);
    p.lse2 = w.lse2;
    p.delta = w.delta;
    p.emin = w.emin;
    p.dk = static_cast<GradOut *>(dk);
    p.dv = static_cast<GradOut *>(dv);
    p.status = status;
    timing_begin(2, st);
    bwd_main_kernel<<<static_cast<unsigned>(units), NTHREADS, SMEM_BYTES, st>>>(tq, tk, tv, tdo,
                                                                               tdq, p);
    timing_end(2, st);
    if (cuda_failed(cudaGetLastError(), "launch of the backward main kernel")) return -8;
  }
  {
    const long long n8 = rows * HD / 8;
    long long blocks = (n8 + 255) / 256;
    blocks = blocks < 1 ? 1 : (blocks > 8LL * sm_count ? 8LL * sm_count : blocks);
    timing_begin(3, st);
    bwd_dq_convert_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        w.dq_acc, static_cast<GradOut *>(dq), w.emin, n8, pr.scale, S, H, G, R);
    timing_end(3, st);
    if (cuda_failed(cudaGetLastError(), "launch of the dQ convert kernel")) return -8;
  }
  return 0;
}

}  // namespace bwd
}  // namespace gqa
