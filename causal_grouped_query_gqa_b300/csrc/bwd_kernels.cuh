// bwd_kernels.cuh -- backward of causal grouped-query attention (in progress).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstddef>

namespace gqa {
namespace bwd {

struct Problem {
  int B, H, G, S;
  int causal, window, n_sink;
  float scale;
};

inline size_t workspace_bytes(int B, int H, int S) {
  const size_t rows = static_cast<size_t>(B) * H * S;
  return rows * 64 * sizeof(float) + rows * sizeof(float);
}

inline int configure_kernels() { return 0; }

inline int launch(const Problem &, const void *, const void *, const void *, const void *,
                  const void *, const float *, void *, void *, void *, void *, int *,
                  PFN_cuTensorMapEncodeTiled_v12000, cudaStream_t) {
  return -8;
}

}  // namespace bwd
}  // namespace gqa
