// quantize_kernel.cuh -- bf16 -> OCP E4M3 bytes with one per-tensor scale, the
// input format of the fp8 forward (gqa_attn_fwd_fp8).  out = e4m3(x * inv_scale),
// round to nearest even, saturating to +-448 (NaN stays NaN); the value an
// output byte stands for is decode(byte) / inv_scale.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "sm100_ptx.cuh"

namespace gqa {

// 16 elements (one 16-byte output store) per thread and pass.
__global__ void __launch_bounds__(256) quantize_e4m3_kernel(const __nv_bfloat16 *__restrict__ x,
                                                            uint8_t *__restrict__ out,
                                                            long long n16, float inv_scale) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < n16;
       e += stride) {
    const uint4 a = reinterpret_cast<const uint4 *>(x)[2 * e];
    const uint4 b = reinterpret_cast<const uint4 *>(x)[2 * e + 1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = pack_e4m3x2(__uint_as_float(w[2 * i] << 16) * inv_scale,
                                      __uint_as_float(w[2 * i] & 0xffff0000u) * inv_scale);
      const uint32_t hi = pack_e4m3x2(__uint_as_float(w[2 * i + 1] << 16) * inv_scale,
                                      __uint_as_float(w[2 * i + 1] & 0xffff0000u) * inv_scale);
      o[i] = lo | (hi << 16);
    }
    reinterpret_cast<uint4 *>(out)[e] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace gqa
