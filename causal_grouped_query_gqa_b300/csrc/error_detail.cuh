// error_detail.cuh -- the text behind GQA_ERR_CUDA: which call failed and the
// CUDA runtime's description of why, kept per host thread and returned by
// gqa_attn_last_error_detail().
#pragma once

#include <cuda_runtime.h>

#include <cstdio>

namespace gqa {

inline char *error_detail_buffer() {
  static thread_local char buf[256] = "";
  return buf;
}

// Records a failed CUDA call; returns true when `e` is an error.
inline bool cuda_failed(cudaError_t e, const char *where) {
  if (e == cudaSuccess) return false;
  std::snprintf(error_detail_buffer(), 256, "%s: %s (%s)", where, cudaGetErrorString(e),
                cudaGetErrorName(e));
  return true;
}

// Records a failure that has no CUDA error code.
inline void set_error_detail(const char *what) { std::snprintf(error_detail_buffer(), 256, "%s", what); }

}  // namespace gqa
