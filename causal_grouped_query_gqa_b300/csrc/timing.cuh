// timing.cuh -- optional CUDA-event bracketing of every kernel launch, on the
// launch stream itself (the profiling aid behind gqa_attn_timing_*).  The
// library is a single translation unit, so this state is private to it.
#pragma once

#include <cuda_runtime.h>

namespace gqa {

constexpr int kNumKernelIds = 6;  // fwd, bwd prep, bwd main, bwd dq convert, fwd key norms,
                                   // rotary pre-pass

struct TimingState {
  bool on = false;
  int device = -1;
  cudaEvent_t start[kNumKernelIds] = {};
  cudaEvent_t stop[kNumKernelIds] = {};
  bool recorded[kNumKernelIds] = {};
};

inline TimingState &timing_state() {
  static TimingState s;
  return s;
}

inline void timing_begin(int id, cudaStream_t st) {
  TimingState &t = timing_state();
  if (t.on) cudaEventRecord(t.start[id], st);
}

inline void timing_end(int id, cudaStream_t st) {
  TimingState &t = timing_state();
  if (t.on) {
    cudaEventRecord(t.stop[id], st);
    t.recorded[id] = true;
  }
}

}  // namespace gqa
