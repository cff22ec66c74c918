// trace.cuh -- optional per-role pipeline timeline (compiled only with
// -DGQA_TRACE): selected threads record clock64() at named events of the
// first kTraceSteps steps of the first kTraceCtas CTAs of each kernel, and
// gqa_attn_trace_read() copies the table out.  Without GQA_TRACE every
// GQA_TRACE_EVENT is an empty statement.
#pragma once

#include <cstdint>

namespace gqa {
constexpr int kTraceKernels = 2;  // 0 forward, 1 backward main
constexpr int kTraceCtas = 4;
constexpr int kTraceEvents = 40;
constexpr int kTraceSteps = 128;
}  // namespace gqa

#ifdef GQA_TRACE
__device__ unsigned long long g_gqa_trace[gqa::kTraceKernels][gqa::kTraceCtas][gqa::kTraceEvents]
                                         [gqa::kTraceSteps];
#define GQA_TRACE_EVENT(kernel, ev, step)                                                    \
  do {                                                                                       \
    if (blockIdx.x < gqa::kTraceCtas && (step) < gqa::kTraceSteps)                          \
      g_gqa_trace[kernel][blockIdx.x][ev][step] = static_cast<unsigned long long>(clock64()); \
  } while (0)
#else
#define GQA_TRACE_EVENT(kernel, ev, step) \
  do {                                    \
  } while (0)
#endif
