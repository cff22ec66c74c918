// device_checks.cuh -- run-time checks of the kernels' index and address
// invariants, compiled only into a debug build (-DGQA_DEVICE_CHECKS): a
// violated check records GQA_ERR_DEVICE_BOUNDS in the device status word
// (first error wins) and the guarded global access is skipped, so nothing
// traps.  Release builds compile every check to `true`.  This stands in for a
// memory checker, which this hardware's tool set does not offer here.
#pragma once

namespace gqa {

constexpr int kBoundsCode = -11;  // GQA_ERR_DEVICE_BOUNDS

__device__ __forceinline__ bool device_check(int *status, bool cond) {
  if (!cond && status) atomicCAS(status, 0, kBoundsCode);
  return cond;
}

}  // namespace gqa

// GQA_CHECK(status, cond) guards an access: `if (GQA_CHECK(...)) access;`.
// GQA_REPORT(status, cond) only records a violation (for accesses that are
// safe anyway, such as TMA loads, whose out-of-range parts read as zeros).
#ifdef GQA_DEVICE_CHECKS
#define GQA_CHECK(status, cond) (::gqa::device_check((status), (cond)))
#define GQA_REPORT(status, cond) static_cast<void>(::gqa::device_check((status), (cond)))
#else
#define GQA_CHECK(status, cond) (true)
#define GQA_REPORT(status, cond) \
  do {                           \
  } while (0)
#endif
