// gqa_attn_api.cu -- the C ABI of libgqa_attn (declared in include/gqa_attn.h):
// argument checks, TMA tensor-map encoding and kernel launches.  No torch types
// and no allocation on the forward path; every step of the computation runs in
// the kernels of fwd_kernel.cuh and bwd_kernels.cuh.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/gqa_attn.h"
#include "error_detail.cuh"
#include "timing.cuh"
#include "trace.cuh"
#include "bwd_kernels.cuh"
#include "fwd_kernel.cuh"
#include "quantize_kernel.cuh"
#include "rope_kernels.cuh"
#include "selftest_kernel.cuh"

namespace {

// Device status word: kernels set it (first error wins) when a bounded wait
// expires; gqa_attn_last_device_status() reads and clears it.
__device__ int g_device_status;

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  int sm_count = 0;
  int *status = nullptr;  // device address of g_device_status
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int device_state(DeviceState **out) {
  int dev = 0;
  if (gqa::cuda_failed(cudaGetDevice(&dev), "cudaGetDevice")) return GQA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) {
    gqa::set_error_detail("device ordinal beyond the library's per-device table");
    return GQA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState &st = g_dev[dev];
  if (!st.ready) {
    if (!g_encode) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q{};
      if (gqa::cuda_failed(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                            cudaEnableDefault, &q),
                           "cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)"))
        return GQA_ERR_CUDA;
      if (q != cudaDriverEntryPointSuccess || fn == nullptr) {
        gqa::set_error_detail("the driver does not provide cuTensorMapEncodeTiled");
        return GQA_ERR_CUDA;
      }
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (gqa::cuda_failed(cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev),
                         "cudaDeviceGetAttribute(MultiProcessorCount)"))
      return GQA_ERR_CUDA;
    if (gqa::cuda_failed(
            cudaGetSymbolAddress(reinterpret_cast<void **>(&st.status), g_device_status),
            "cudaGetSymbolAddress(device status word)"))
      return GQA_ERR_CUDA;
    for (auto kern : {gqa::fwd::gqa_fwd_kernel<false, false>, gqa::fwd::gqa_fwd_kernel<true, false>,
                      gqa::fwd::gqa_fwd_kernel<false, true>}) {
      if (gqa::cuda_failed(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                gqa::fwd::SMEM_BYTES),
                           "cudaFuncSetAttribute(forward shared memory)"))
        return GQA_ERR_CUDA;
      // The forward rebalances registers between warpgroups (setmaxnreg); that
      // is only safe when the compiled launch allocation covers the split.
      cudaFuncAttributes fa{};
      if (gqa::cuda_failed(cudaFuncGetAttributes(&fa, kern), "cudaFuncGetAttributes(forward)"))
        return GQA_ERR_CUDA;
      if (fa.numRegs < gqa::fwd::kMinLaunchRegs) {
        gqa::set_error_detail("forward kernel compiled with fewer registers than its warpgroup split needs");
        return GQA_ERR_CUDA;
      }
    }
    int rc = gqa::bwd::configure_kernels();
    if (rc != 0) return GQA_ERR_CUDA;  // detail recorded by configure_kernels
    st.ready = true;
  }
  *out = &st;
  return GQA_OK;
}

// 3-D bf16 tensor map over [outer][rows][64] with a box of [1][box_rows][64],
// 128-byte swizzle; rows past `rows` read as zeros.
int make_tmap_bf16(CUtensorMap *map, const void *base, uint64_t outer, uint64_t rows,
                   uint32_t box_rows) {
  cuuint64_t dims[3] = {64, rows, outer};
  cuuint64_t strides[2] = {64 * 2, rows * 64 * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    gqa::set_error_detail("cuTensorMapEncodeTiled rejected a bf16 tensor map");
    return GQA_ERR_CUDA;
  }
  return GQA_OK;
}

// 3-D E4M3 (byte) tensor map over [outer][rows][64] with a box of
// [1][box_rows][64]: 64-byte rows, 64-byte swizzle; rows past `rows` read as zeros.
int make_tmap_e4m3(CUtensorMap *map, const void *base, uint64_t outer, uint64_t rows,
                   uint32_t box_rows) {
  cuuint64_t dims[3] = {64, rows, outer};
  cuuint64_t strides[2] = {64, rows * 64};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    gqa::set_error_detail("cuTensorMapEncodeTiled rejected an fp8 tensor map");
    return GQA_ERR_CUDA;
  }
  return GQA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_common(int B, int H, int G, int S, int d, int causal, int window, int n_sink,
                 float scale) {
  if (B <= 0 || H <= 0 || G <= 0 || S <= 0) return GQA_ERR_SHAPE;
  if (H % G != 0) return GQA_ERR_SHAPE;
  // element counts must fit the kernels' int64 offsets and TMA's 32-bit dims
  const uint64_t rows_q = static_cast<uint64_t>(B) * H;
  if (rows_q > 0x7fffffffull || static_cast<uint64_t>(S) * 64ull * 2ull * rows_q > (1ull << 46))
    return GQA_ERR_SHAPE;
  if (d != 64) return GQA_ERR_HEADDIM;
  if (n_sink < 0) return GQA_ERR_MASK;
  if (!causal && window > 0) return GQA_ERR_MASK;
  if (!(std::isfinite(scale) && scale > 0.f)) return GQA_ERR_SCALE;
  return GQA_OK;
}

// Scratch of gqa_attn_bwd_noalloc, for callers that cannot allocate: one
// fixed array per device the library is loaded on.  Host code must not use the
// symbol as an address; its device address is looked up once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GQA_NOALLOC_SCRATCH_BYTES];

struct NoAllocState {
  bool ready = false;
  void *scratch = nullptr;  // device address of g_noalloc_scratch on this device
};
NoAllocState g_noalloc[kMaxDevices];

}  // namespace

extern "C" {

const char *gqa_attn_strerror(int status) {
  switch (status) {
    case GQA_OK: return "ok";
    case GQA_ERR_NULL: return "a required pointer is NULL";
    case GQA_ERR_SHAPE: return "invalid sizes (B, H, G, S must be positive, H % G == 0)";
    case GQA_ERR_HEADDIM: return "unsupported head dimension (only d = 64)";
    case GQA_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case GQA_ERR_MASK: return "invalid mask (window > 0 needs causal; n_sink >= 0)";
    case GQA_ERR_SCALE: return "scale must be finite and positive";
    case GQA_ERR_WORKSPACE: return "workspace too small";
    case GQA_ERR_CUDA: return "CUDA call or kernel launch failed";
    case GQA_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
    case GQA_ERR_TOO_LARGE: return "problem needs more scratch than gqa_attn_bwd_noalloc holds";
    case GQA_ERR_DEVICE_BOUNDS: return "a kernel's run-time index check failed (debug build)";
    case GQA_ERR_ROPE: return "invalid rotary embedding parameters (base > 1, factor >= 1, original context > 0, 0 <= alpha < beta)";
    default: return "unknown status";
  }
}

namespace {

// The forward launch shared by the entry points; kn2 (the score-bound record
// that fwd_knorm_kernel writes first, on the same stream) may be null, and so
// may rope_tab (the rotary table: with it the kernel rotates each query tile;
// k is then already rotated).  fp8: q and k
// are E4M3 bytes and `scale` already carries their two dequantisation scales.
int launch_forward(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                   int G, int S, int causal, int window, int n_sink, float scale, float *kn2,
                   const float2 *rope_tab, cudaStream_t st, bool fp8 = false) {
  DeviceState *ds = nullptr;
  int rc = device_state(&ds);
  if (rc != GQA_OK) return rc;

  using namespace gqa::fwd;
  CUtensorMap tq, tk, tv;
  if (fp8) {
    if (make_tmap_e4m3(&tq, q, static_cast<uint64_t>(B) * H, S, BM) != GQA_OK ||
        make_tmap_e4m3(&tk, k, static_cast<uint64_t>(B) * G, S, BN) != GQA_OK)
      return GQA_ERR_CUDA;
  } else if (make_tmap_bf16(&tq, q, static_cast<uint64_t>(B) * H, S, BM) != GQA_OK ||
             make_tmap_bf16(&tk, k, static_cast<uint64_t>(B) * G, S, BN) != GQA_OK) {
    return GQA_ERR_CUDA;
  }
  if (make_tmap_bf16(&tv, v, static_cast<uint64_t>(B) * G, S, BN) != GQA_OK) return GQA_ERR_CUDA;

  Params p{};
  p.B = B;
  p.H = H;
  p.G = G;
  p.S = S;
  p.R = H / G;
  p.causal = causal ? 1 : 0;
  p.window = (causal && window > 0) ? window : 0;
  p.n_sink = p.window > 0 ? n_sink : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.n_qblocks = (S + BM - 1) / BM;
  p.n_pairs = (p.R + 1) / 2;
  p.kn2 = kn2;
  p.rope_tab = rope_tab;
  p.o = static_cast<__nv_bfloat16 *>(o);
  p.lse = lse;
  p.status = ds->status;
  const long long units = static_cast<long long>(p.n_qblocks) * B * G * p.n_pairs;
  if (units > 0x7fffffffLL) return GQA_ERR_SHAPE;
  p.n_units = static_cast<int>(units);
  // persistent grid: one CTA per SM (the kernel's shared memory and TMEM allow one)
  const int grid = static_cast<int>(units < ds->sm_count ? units : ds->sm_count);

  if (kn2) {
    const long long blocks = static_cast<long long>(B) * G * kKnParts;
    if (blocks > 0x7fffffffLL) return GQA_ERR_SHAPE;
    gqa::timing_begin(GQA_KERNEL_FWD_KNORM, st);
    fwd_knorm_kernel<<<static_cast<unsigned>(blocks), kKnormThreads, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(k), S, kn2);
    gqa::timing_end(GQA_KERNEL_FWD_KNORM, st);
    if (gqa::cuda_failed(cudaGetLastError(), "launch of the forward's key-norm kernel"))
      return GQA_ERR_CUDA;
  }
  gqa::timing_begin(GQA_KERNEL_FWD, st);
  if (fp8)
    gqa_fwd_kernel<false, true><<<static_cast<unsigned>(grid), NTHREADS, SMEM_BYTES, st>>>(tq, tk, tv, p);
  else if (rope_tab)
    gqa_fwd_kernel<true, false><<<static_cast<unsigned>(grid), NTHREADS, SMEM_BYTES, st>>>(tq, tk, tv, p);
  else
    gqa_fwd_kernel<false, false><<<static_cast<unsigned>(grid), NTHREADS, SMEM_BYTES, st>>>(tq, tk, tv, p);
  gqa::timing_end(GQA_KERNEL_FWD, st);
  return gqa::cuda_failed(cudaGetLastError(), "launch of the forward kernel") ? GQA_ERR_CUDA
                                                                               : GQA_OK;
}

}  // namespace

int gqa_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                 int G, int S, int d, int causal, int window, int n_sink, float scale,
                 void *stream) {
  int rc = check_common(B, H, G, S, d, causal, window, n_sink, scale);
  if (rc != GQA_OK) return rc;
  if (!q || !k || !v || !o || !lse) return GQA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return GQA_ERR_ALIGN;
  return launch_forward(q, k, v, o, lse, B, H, G, S, causal, window, n_sink, scale, nullptr,
                        nullptr, static_cast<cudaStream_t>(stream));
}

size_t gqa_attn_fwd_workspace_size(int B, int H, int G, int S, int d) {
  if (check_common(B, H, G, S, d, 1, 0, 0, 1.f) != GQA_OK) return 0;
  return static_cast<size_t>(B) * G * gqa::fwd::kKnParts * sizeof(float);
}

int gqa_attn_fwd_ws(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                    int G, int S, int d, int causal, int window, int n_sink, float scale,
                    void *workspace, size_t workspace_bytes, void *stream) {
  int rc = check_common(B, H, G, S, d, causal, window, n_sink, scale);
  if (rc != GQA_OK) return rc;
  if (!q || !k || !v || !o || !lse || !workspace) return GQA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(workspace))
    return GQA_ERR_ALIGN;
  if (workspace_bytes < gqa_attn_fwd_workspace_size(B, H, G, S, d)) return GQA_ERR_WORKSPACE;
  return launch_forward(q, k, v, o, lse, B, H, G, S, causal, window, n_sink, scale,
                        static_cast<float *>(workspace), nullptr, static_cast<cudaStream_t>(stream));
}

int gqa_attn_fwd_fp8(const void *q8, const void *k8, const void *v, void *o, float *lse, int B,
                     int H, int G, int S, int d, int causal, int window, int n_sink, float scale,
                     float q_scale, float k_scale, void *stream) {
  int rc = check_common(B, H, G, S, d, causal, window, n_sink, scale);
  if (rc != GQA_OK) return rc;
  if (!(std::isfinite(q_scale) && q_scale > 0.f && std::isfinite(k_scale) && k_scale > 0.f))
    return GQA_ERR_SCALE;
  const double folded = static_cast<double>(scale) * q_scale * k_scale;
  if (!(folded < 3.0e38 && folded > 1.0e-37)) return GQA_ERR_SCALE;
  if (!q8 || !k8 || !v || !o || !lse) return GQA_ERR_NULL;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return GQA_ERR_ALIGN;
  return launch_forward(q8, k8, v, o, lse, B, H, G, S, causal, window, n_sink,
                        static_cast<float>(folded), nullptr, nullptr,
                        static_cast<cudaStream_t>(stream), true);
}

int gqa_attn_quantize_e4m3(const void *x, void *out, long long n, float inv_scale, void *stream) {
  if (!x || !out) return GQA_ERR_NULL;
  if (n <= 0 || (n & 15) != 0) return GQA_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(out)) return GQA_ERR_ALIGN;
  if (!(std::isfinite(inv_scale) && inv_scale > 0.f)) return GQA_ERR_SCALE;
  DeviceState *ds = nullptr;
  int rc = device_state(&ds);
  if (rc != GQA_OK) return rc;
  const long long n16 = n / 16;
  long long blocks = (n16 + 255) / 256;
  blocks = blocks < 1 ? 1 : (blocks > 8LL * ds->sm_count ? 8LL * ds->sm_count : blocks);
  gqa::quantize_e4m3_kernel<<<static_cast<unsigned>(blocks), 256, 0,
                              static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16 *>(x), static_cast<uint8_t *>(out), n16, inv_scale);
  return gqa::cuda_failed(cudaGetLastError(), "launch of the fp8 quantisation kernel")
             ? GQA_ERR_CUDA
             : GQA_OK;
}

size_t gqa_attn_fwd_yarn_workspace_size(int B, int H, int G, int S, int d, int rope_mode) {
  if (check_common(B, H, G, S, d, 1, 0, 0, 1.f) != GQA_OK) return 0;
  if (rope_mode != GQA_ROPE_PREPASS && rope_mode != GQA_ROPE_FUSED) return 0;
  // k_rot, the (cos, sin) table, the key-norm record, then (pre-pass) q_rot;
  // every part a multiple of 16 bytes
  const size_t krot = static_cast<size_t>(B) * G * S * 64 * 2;
  const size_t tab = static_cast<size_t>(S) * gqa::rope::kPairs * sizeof(float2);
  const size_t kn = static_cast<size_t>(B) * G * gqa::fwd::kKnParts * sizeof(float);
  const size_t qrot = rope_mode == GQA_ROPE_PREPASS ? static_cast<size_t>(B) * H * S * 64 * 2 : 0;
  return krot + tab + kn + qrot;
}

int gqa_attn_fwd_yarn(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                      int H, int G, int S, int d, int causal, int window, int n_sink, float scale,
                      float rope_base, float rope_factor, int rope_orig_ctx, float rope_alpha,
                      float rope_beta, int score_bound, int rope_mode, void *workspace,
                      size_t workspace_bytes, void *stream) {
  int rc = check_common(B, H, G, S, d, causal, window, n_sink, scale);
  if (rc != GQA_OK) return rc;
  gqa::rope::Freqs f;
  if (!gqa::rope::yarn_freqs(rope_base, rope_factor, rope_orig_ctx, rope_alpha, rope_beta, &f) ||
      (rope_mode != GQA_ROPE_PREPASS && rope_mode != GQA_ROPE_FUSED))
    return GQA_ERR_ROPE;
  if (!q || !k || !v || !o || !lse || !workspace) return GQA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(workspace))
    return GQA_ERR_ALIGN;
  if (workspace_bytes < gqa_attn_fwd_yarn_workspace_size(B, H, G, S, d, rope_mode))
    return GQA_ERR_WORKSPACE;
  const double tempered = static_cast<double>(scale) * gqa::rope::yarn_score_factor(rope_factor);
  if (!(tempered < 3.0e38)) return GQA_ERR_SCALE;
  DeviceState *ds = nullptr;
  if ((rc = device_state(&ds)) != GQA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool prepass = rope_mode == GQA_ROPE_PREPASS;
  char *wp = static_cast<char *>(workspace);
  __nv_bfloat16 *k_rot = reinterpret_cast<__nv_bfloat16 *>(wp);
  wp += static_cast<size_t>(B) * G * S * 64 * 2;
  float2 *tab = reinterpret_cast<float2 *>(wp);
  wp += static_cast<size_t>(S) * gqa::rope::kPairs * sizeof(float2);
  float *kn2 = score_bound ? reinterpret_cast<float *>(wp) : nullptr;
  wp += static_cast<size_t>(B) * G * gqa::fwd::kKnParts * sizeof(float);
  __nv_bfloat16 *q_rot = prepass ? reinterpret_cast<__nv_bfloat16 *>(wp) : nullptr;
  gqa::timing_begin(GQA_KERNEL_ROPE, st);
  {
    const long long n = static_cast<long long>(S) * gqa::rope::kPairs;
    long long blocks = (n + 255) / 256;
    blocks = blocks > 4LL * ds->sm_count ? 4LL * ds->sm_count : blocks;
    gqa::rope::rope_table_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(f, S, tab);
    if (gqa::cuda_failed(cudaGetLastError(), "launch of the rotary table kernel")) return GQA_ERR_CUDA;
  }
  {
    const long long nq = prepass ? static_cast<long long>(B) * H * S * 8 : 0;
    const long long nk = static_cast<long long>(B) * G * S * 8;
    long long blocks = (nq + nk + 255) / 256;
    blocks = blocks > 8LL * ds->sm_count ? 8LL * ds->sm_count : blocks;
    gqa::rope::rope_rotate_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(q), q_rot, nq, static_cast<const __nv_bfloat16 *>(k),
        k_rot, nk, tab, S);
    gqa::timing_end(GQA_KERNEL_ROPE, st);
    if (gqa::cuda_failed(cudaGetLastError(), "launch of the rotation kernel")) return GQA_ERR_CUDA;
  }
  // pre-pass: the plain forward on rotated q and k; fused: the forward turns
  // each query tile by the table itself
  return launch_forward(prepass ? static_cast<const void *>(q_rot) : q, k_rot, v, o, lse, B, H, G,
                        S, causal, window, n_sink, static_cast<float>(tempered), kn2,
                        prepass ? nullptr : tab, st);
}

size_t gqa_attn_bwd_workspace_size(int B, int H, int G, int S, int d) {
  if (check_common(B, H, G, S, d, 1, 0, 0, 1.f) != GQA_OK) return 0;
  return gqa::bwd::workspace_bytes(B, H, G, S);
}

int gqa_attn_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
                 const float *lse, void *dq, void *dk, void *dv, int B, int H, int G, int S, int d,
                 int causal, int window, int n_sink, float scale, void *workspace,
                 size_t workspace_bytes, void *stream) {
  int rc = check_common(B, H, G, S, d, causal, window, n_sink, scale);
  if (rc != GQA_OK) return rc;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return GQA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (workspace && !aligned16(workspace)))
    return GQA_ERR_ALIGN;
  const size_t need = gqa::bwd::workspace_bytes(B, H, G, S);
  if (workspace && workspace_bytes < need) return GQA_ERR_WORKSPACE;
  DeviceState *ds = nullptr;
  if ((rc = device_state(&ds)) != GQA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void *ws = workspace;
  if (!ws) {
    if (gqa::cuda_failed(cudaMallocAsync(&ws, need, st), "cudaMallocAsync(backward workspace)"))
      return GQA_ERR_CUDA;
  }
  gqa::bwd::Problem pr{};
  pr.B = B;
  pr.H = H;
  pr.G = G;
  pr.S = S;
  pr.causal = causal ? 1 : 0;
  pr.window = (causal && window > 0) ? window : 0;
  pr.n_sink = pr.window > 0 ? n_sink : 0;
  pr.scale = scale;
  rc = gqa::bwd::launch(pr, q, k, v, o, dout, lse, dq, dk, dv, ws, ds->status, ds->sm_count,
                        g_encode, st);
  if (rc == -2) rc = GQA_ERR_SHAPE;
  else if (rc != 0) rc = GQA_ERR_CUDA;
  if (!workspace) {
    if (gqa::cuda_failed(cudaFreeAsync(ws, st), "cudaFreeAsync(backward workspace)") &&
        rc == GQA_OK)
      rc = GQA_ERR_CUDA;
  }
  return rc;
}

int gqa_attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                         const void *dout, const float *lse, void *dq, void *dk, void *dv, int B,
                         int H, int G, int S, int d, int causal, int window, int n_sink,
                         float scale, void *stream) {
  int rc = check_common(B, H, G, S, d, causal, window, n_sink, scale);
  if (rc != GQA_OK) return rc;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return GQA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return GQA_ERR_ALIGN;
  if (gqa::bwd::workspace_bytes(B, H, G, S) > GQA_NOALLOC_SCRATCH_BYTES) return GQA_ERR_TOO_LARGE;
  DeviceState *ds = nullptr;
  if ((rc = device_state(&ds)) != GQA_OK) return rc;
  int dev = 0;
  if (gqa::cuda_failed(cudaGetDevice(&dev), "cudaGetDevice")) return GQA_ERR_CUDA;
  void *scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    NoAllocState &na = g_noalloc[dev];
    if (!na.ready) {
      // once per device, with that device current
      if (gqa::cuda_failed(cudaGetSymbolAddress(&na.scratch, g_noalloc_scratch),
                           "cudaGetSymbolAddress(static backward scratch)"))
        return GQA_ERR_CUDA;
      na.ready = true;
    }
    scratch = na.scratch;
  }
  gqa::bwd::Problem pr{};
  pr.B = B;
  pr.H = H;
  pr.G = G;
  pr.S = S;
  pr.causal = causal ? 1 : 0;
  pr.window = (causal && window > 0) ? window : 0;
  pr.n_sink = pr.window > 0 ? n_sink : 0;
  pr.scale = scale;
  rc = gqa::bwd::launch(pr, q, k, v, o, dout, lse, dq, dk, dv, scratch, ds->status, ds->sm_count,
                        g_encode, static_cast<cudaStream_t>(stream));
  if (rc == -2) return GQA_ERR_SHAPE;
  return rc == 0 ? GQA_OK : GQA_ERR_CUDA;
}

const char *gqa_attn_last_error_detail(void) { return gqa::error_detail_buffer(); }

int gqa_attn_timing_enable(int on) {
  gqa::TimingState &t = gqa::timing_state();
  if (on) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
    if (t.device != dev) {
      for (int i = 0; i < gqa::kNumKernelIds; ++i) {
        if (cudaEventCreate(&t.start[i]) != cudaSuccess ||
            cudaEventCreate(&t.stop[i]) != cudaSuccess)
          return GQA_ERR_CUDA;
        t.recorded[i] = false;
      }
      t.device = dev;
    }
  }
  t.on = on != 0;
  return GQA_OK;
}

int gqa_attn_timing_collect(float *ms, int n) {
  if (!ms) return GQA_ERR_NULL;
  gqa::TimingState &t = gqa::timing_state();
  int rc = GQA_OK;
  for (int i = 0; i < gqa::kNumKernelIds && i < n; ++i) {
    ms[i] = -1.f;
    if (t.device >= 0 && t.recorded[i]) {
      if (cudaEventSynchronize(t.stop[i]) != cudaSuccess ||
          cudaEventElapsedTime(&ms[i], t.start[i], t.stop[i]) != cudaSuccess) {
        ms[i] = -1.f;
        rc = GQA_ERR_CUDA;
      }
      t.recorded[i] = false;
    }
  }
  return rc;
}

#ifdef GQA_TRACE
// Trace builds only (not part of the public header): copies the clock64 event
// table [kernel][cta][event][step] (unsigned 64-bit) to host memory.
GQA_API int gqa_attn_trace_read(void *host, size_t bytes) {
  if (!host || bytes < sizeof(g_gqa_trace)) return GQA_ERR_NULL;
  if (cudaDeviceSynchronize() != cudaSuccess) return GQA_ERR_CUDA;
  return cudaMemcpyFromSymbol(host, g_gqa_trace, sizeof(g_gqa_trace)) == cudaSuccess
             ? GQA_OK
             : GQA_ERR_CUDA;
}
#endif

int gqa_attn_selftest_timeout(unsigned budget_ms, unsigned long long *elapsed_ns,
                              int *returned_ok, void *stream) {
  if (!elapsed_ns || !returned_ok) return GQA_ERR_NULL;
  if (budget_ms == 0 || budget_ms > 1000) return GQA_ERR_SHAPE;
  DeviceState *ds = nullptr;
  int rc = device_state(&ds);
  if (rc != GQA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // start from a clear status word, so the result is this kernel's own
  if (gqa::cuda_failed(cudaStreamSynchronize(st), "cudaStreamSynchronize")) return GQA_ERR_CUDA;
  const int zero = 0;
  if (gqa::cuda_failed(cudaMemcpy(ds->status, &zero, sizeof(int), cudaMemcpyHostToDevice),
                       "cudaMemcpy(clear device status)"))
    return GQA_ERR_CUDA;
  gqa::selftest::selftest_wait_kernel<<<1, 64, 0, st>>>(
      ds->status, static_cast<uint64_t>(budget_ms) * 1000000ull);
  if (gqa::cuda_failed(cudaGetLastError(), "launch of the self-test kernel")) return GQA_ERR_CUDA;
  if (gqa::cuda_failed(cudaStreamSynchronize(st), "cudaStreamSynchronize(self-test)"))
    return GQA_ERR_CUDA;
  if (gqa::cuda_failed(cudaMemcpyFromSymbol(elapsed_ns, gqa::selftest::g_selftest_elapsed_ns,
                                            2 * sizeof(unsigned long long)),
                       "cudaMemcpyFromSymbol(self-test times)") ||
      gqa::cuda_failed(cudaMemcpyFromSymbol(returned_ok, gqa::selftest::g_selftest_returned,
                                            2 * sizeof(int)),
                       "cudaMemcpyFromSymbol(self-test results)"))
    return GQA_ERR_CUDA;
  return gqa_attn_last_device_status(stream);
}

int gqa_attn_last_device_status(void *stream) {
  DeviceState *ds = nullptr;
  if (device_state(&ds) != GQA_OK) return GQA_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GQA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, ds->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GQA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(ds->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return GQA_ERR_CUDA;
  return v;
}

}  // extern "C"
