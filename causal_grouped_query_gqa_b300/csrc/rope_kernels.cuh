// rope_kernels.cuh -- YaRN rotary position embedding for the forward.
//
// "SnapKitty Transformer 8B" (model specification table, section "Protected
// Inventions") rotates queries and keys with YaRN-scaled rotary embeddings
// (32x factor, 204800-token sequences).  The frequencies follow the YaRN paper
// (Peng et al. 2023, section 3, "NTK-by-parts"): for pair i of the head
// dimension, theta_i = base^(-2i/d), r_i = L theta_i / (2 pi) with L the
// original context length, gamma = clamp((r_i - alpha) / (beta - alpha), 0, 1),
// h_i = (1 - gamma) theta_i / s + gamma theta_i; the pair (x_2i, x_2i+1) of a
// row at position m turns by m h_i (RoFormer's rotation, adjacent pairs).  The
// paper's attention temperature sqrt(1/t) = 0.1 ln s + 1 multiplies the
// scaled scores by (0.1 ln s + 1)^2; the launch folds it into the softmax
// scale.
//
// Kernels (on the caller's stream, into the caller's workspace):
//   rope_table_kernel   cos / sin of m h_i for every position m < S and pair
//                       i < 32 ([S][32] float2); the angle is reduced modulo
//                       2 pi in fp64 (m h_i / pi in fp64, minus the nearest
//                       even integer) before an fp32 sincospif, so positions
//                       up to 2^24 keep full fp32 accuracy;
//   rope_rotate_kernel  the rotated keys [B*G][S][64] in bf16 (one rounding)
//                       and, in the pre-pass mode, the rotated queries
//                       [B*H][S][64] as well, in one launch.
// In the fused mode the forward kernel rotates each query tile in shared
// memory as it lands (rope_rotate_smem_row, fwd_kernel.cuh kRope), which
// needs no query-sized workspace; the pre-pass mode measured faster.
#pragma once

#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "sm100_ptx.cuh"

namespace gqa {
namespace rope {

constexpr int kPairs = 32;  // d / 2 for d = 64

// h_i / pi for the 32 pairs, computed on the host in double.
struct Freqs {
  double h_over_pi[kPairs];
};

// YaRN frequencies (double precision, host).  Returns false for parameters the
// definition does not cover (base <= 1, factor < 1, L <= 0, not 0 <= alpha < beta).
inline bool yarn_freqs(double base, double factor, double orig_ctx, double alpha, double beta,
                       Freqs *out) {
  if (!(base > 1.0) || !(factor >= 1.0) || !(orig_ctx > 0.0) || !(alpha >= 0.0) ||
      !(beta > alpha) || !std::isfinite(base) || !std::isfinite(factor) ||
      !std::isfinite(beta))
    return false;
  const double pi = std::acos(-1.0);
  for (int i = 0; i < kPairs; ++i) {
    const double theta = std::pow(base, -2.0 * i / (2.0 * kPairs));
    const double r = orig_ctx * theta / (2.0 * pi);  // L / wavelength
    const double gamma = r < alpha ? 0.0 : (r > beta ? 1.0 : (r - alpha) / (beta - alpha));
    const double h = (1.0 - gamma) * theta / factor + gamma * theta;
    out->h_over_pi[i] = h / pi;
  }
  return true;
}

// (0.1 ln s + 1)^2: the factor YaRN's temperature puts on the scaled scores.
inline double yarn_score_factor(double factor) {
  const double m = 0.1 * std::log(factor) + 1.0;
  return m * m;
}

// tab[m * 32 + i] = (cos m h_i, sin m h_i) for m < S.
__global__ void __launch_bounds__(256) rope_table_kernel(const Freqs f, int S,
                                                         float2 *__restrict__ tab) {
  const long long n = static_cast<long long>(S) * kPairs;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
       e += stride) {
    const int m = static_cast<int>(e / kPairs), i = static_cast<int>(e % kPairs);
    const double x = static_cast<double>(m) * f.h_over_pi[i];  // angle / pi
    const double t = x - 2.0 * rint(0.5 * x);                  // in [-1, 1], same angle
    float s, c;
    sincospif(static_cast<float>(t), &s, &c);
    tab[e] = make_float2(c, s);
  }
}

// One rotated 16-byte chunk (4 pairs) of a row at position m.
__device__ __forceinline__ uint4 rope_rotate_chunk(const uint4 w, const float2 *__restrict__ tab_m,
                                                   int ch) {
  const float4 *t4 = reinterpret_cast<const float4 *>(tab_m + 4 * ch);
  const float4 cs01 = __ldg(t4), cs23 = __ldg(t4 + 1);  // (c0, s0, c1, s1), (c2, s2, c3, s3)
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
  const float cs[8] = {cs01.x, cs01.y, cs01.z, cs01.w, cs23.x, cs23.y, cs23.z, cs23.w};
  uint32_t out[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const float x0 = __uint_as_float(in[p] << 16), x1 = __uint_as_float(in[p] & 0xffff0000u);
    const float c = cs[2 * p], s = cs[2 * p + 1];
    out[p] = pack_bf16x2(x0 * c - x1 * s, x0 * s + x1 * c);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// q_rot, k_rot = rotations of q's and k's rows (row r of a head sits at
// position r % S): chunks [0, n_q) are q's, [n_q, n_q + n_k) k's; 8 chunks a
// row, one chunk per thread and pass.
__global__ void __launch_bounds__(256) rope_rotate_kernel(const __nv_bfloat16 *__restrict__ q,
                                                          __nv_bfloat16 *__restrict__ q_rot,
                                                          long long n_q,
                                                          const __nv_bfloat16 *__restrict__ k,
                                                          __nv_bfloat16 *__restrict__ k_rot,
                                                          long long n_k,
                                                          const float2 *__restrict__ tab, int S) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < n_q + n_k;
       e += stride) {
    const bool is_q = e < n_q;
    const long long c = is_q ? e : e - n_q;
    const uint4 *src = reinterpret_cast<const uint4 *>(is_q ? q : k);
    uint4 *dst = reinterpret_cast<uint4 *>(is_q ? q_rot : k_rot);
    const int m = static_cast<int>((c >> 3) % S);
    dst[c] = rope_rotate_chunk(__ldcs(src + c), tab + static_cast<size_t>(m) * kPairs,
                               static_cast<int>(c & 7));
  }
}

// Rotates one 128-byte bf16 row (64 elements; 128-byte swizzle: 16-byte chunk c
// at c ^ (r & 7)) in shared memory by the table row of its position.
__device__ __forceinline__ void rope_rotate_smem_row(uint8_t *row, int r,
                                                     const float2 *__restrict__ tab_m) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint4 *p = reinterpret_cast<uint4 *>(row + ((c ^ (r & 7)) << 4));
    *p = rope_rotate_chunk(*p, tab_m, c);
  }
}

}  // namespace rope
}  // namespace gqa
