/*
 * gqa_attn.h -- C ABI of libgqa_attn: exact causal scaled-dot-product attention
 * with grouped-query K/V sharing, an optional sliding window plus always-visible
 * leading sink tokens, and its backward pass, on one NVIDIA B300 (sm_103a).
 *
 * The operation (from "nx_f32_gqa_gate.nx source", header comment and tests T0-T5,
 * and "SnapKitty Transformer 8B", sections "FlashAttention Inference" and
 * "Protected Inventions"):
 *
 *   for batch b, query head h (kv head g = h / (H/G)), query row i:
 *     s_ij  = scale * q[b,h,i,:] . k[b,g,j,:]            for every visible j
 *     P_ij  = exp(s_ij - max_j s_ij) / sum_j exp(s_ij - max_j s_ij)
 *     o[b,h,i,:] = sum_j P_ij v[b,g,j,:]
 *     lse[b,h,i] = ln sum_j exp(s_ij)                    (natural log)
 *
 *   visible(i, j) = (!causal || j <= i) &&
 *                   (window <= 0 || j > i - window || j < n_sink)
 *
 *   so with causal and window = W > 0 a query sees the W most recent keys
 *   (itself included) plus the keys j < n_sink that are not in its future.
 *   window <= 0 disables the window; n_sink is then ignored.  A window
 *   without causal masking is rejected (GQA_ERR_MASK).
 *
 * Conventions shared by every call:
 *   - Tensors are DEVICE pointers owned by the caller, dense and row-major:
 *       q, o, dout, dq : [B][H][S][d] bf16      k, v, dk, dv : [B][G][S][d] bf16
 *       lse            : [B][H][S]    fp32
 *     each aligned to 16 bytes.  Only d = 64 is implemented.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *     is asynchronous on that stream; the return value covers argument checks
 *     and launch errors only.  A kernel that gives up a bounded wait records
 *     GQA_ERR_DEVICE_TIMEOUT in a device status word read by
 *     gqa_attn_last_device_status().
 *   - Calls are C: no exceptions, 0 on success, a negative gqa_status on error.
 *     Nothing is launched when an argument check fails.
 *   - The calls use the GPU that is current on the calling thread.
 */
#ifndef GQA_ATTN_H_
#define GQA_ATTN_H_

#include <stddef.h>

#if defined(__GNUC__)
#define GQA_API __attribute__((visibility("default")))
#else
#define GQA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GQA_OK = 0,
    GQA_ERR_NULL = -1,           /* a required pointer is NULL */
    GQA_ERR_SHAPE = -2,          /* B, H, G or S not positive, H % G != 0, or a size overflows */
    GQA_ERR_HEADDIM = -3,        /* d != 64 */
    GQA_ERR_ALIGN = -4,          /* a pointer is not 16-byte aligned */
    GQA_ERR_MASK = -5,           /* window > 0 without causal, or n_sink < 0 */
    GQA_ERR_SCALE = -6,          /* scale not finite or not positive */
    GQA_ERR_WORKSPACE = -7,      /* workspace smaller than gqa_attn_bwd_workspace_size() */
    GQA_ERR_CUDA = -8,           /* a CUDA runtime/driver call or a launch failed */
    GQA_ERR_DEVICE_TIMEOUT = -9, /* a kernel gave up a bounded wait (device status) */
    GQA_ERR_TOO_LARGE = -10,     /* needs more than the fixed scratch of gqa_attn_bwd_noalloc */
    GQA_ERR_DEVICE_BOUNDS = -11, /* a run-time index check of a debug build failed (device status;
                                    only libraries built with -DGQA_DEVICE_CHECKS report it) */
    GQA_ERR_ROPE = -12           /* rotary embedding parameters outside the definition */
} gqa_status;

/*
 * Forward.  Writes o [B][H][S][d] bf16 and lse [B][H][S] fp32 (natural log of the
 * softmax denominator of the scaled scores; it is what gqa_attn_bwd needs).
 * Inputs q [B][H][S][d], k and v [B][G][S][d] are bf16; products accumulate in
 * fp32.  Page: "SnapKitty Transformer 8B", section "FlashAttention Inference"
 * (flash_attention_fwd(Q, K, V, causal, sliding_window, num_sinks) on
 * [batch, heads, seq_len, head_dim] tensors), with the GQA head map of
 * "nx_f32_gqa_gate.nx source", test T2.
 */
GQA_API int gqa_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                 int B, int H, int G, int S, int d,
                 int causal, int window, int n_sink, float scale, void *stream);

/*
 * Bytes of scratch that gqa_attn_fwd_ws needs: B * G records of 32 fp32 partial
 * maxima of |k_j|^2 (128 bytes per kv head).  Returns 0 for invalid sizes.
 */
GQA_API size_t gqa_attn_fwd_workspace_size(int B, int H, int G, int S, int d);

/*
 * Forward with a score bound: the result contract of gqa_attn_fwd (the same
 * definition in the same precision), in two launches on `stream`.  A first
 * kernel writes into `workspace` the largest squared norm of each kv head's key
 * rows (32 partial maxima per kv head).  Every scaled score of query row i is
 * at most U_i = |q_i| * max_j |k_j| * scale * log2(e) in magnitude
 * (Cauchy-Schwarz, base-2 units); a query head whose 128 rows of a work unit
 * all have U_i <= 64 computes the unit's key tiles against the fixed reference
 * U_i - 32 instead of a running row maximum (every term 2^(s - reference) then
 * lies in [2^-96, 2^32]), and heads with larger bounds keep the online maximum of
 * "SnapKitty Transformer 8B", section "FlashAttention Inference".  The bound is
 * this library's.
 * Input range: the fp32 sums of O then hold up to S * 2^32 * max|v|, so the
 * result equals gqa_attn_fwd's while max|v| < 2^(95 - log2 S) (2^77 at
 * S = 204800); gqa_attn_fwd keeps terms below 2^8 and allows max|v| up to
 * 2^(119 - log2 S).  Use gqa_attn_fwd for values beyond the first limit.
 * workspace: device memory of at least gqa_attn_fwd_workspace_size() bytes,
 * 16-byte aligned, owned by the caller and not used by any other call running
 * at the same time.  Errors: as gqa_attn_fwd, plus GQA_ERR_NULL for a null
 * workspace and GQA_ERR_WORKSPACE for a short one.
 */
GQA_API int gqa_attn_fwd_ws(const void *q, const void *k, const void *v, void *o, float *lse,
                    int B, int H, int G, int S, int d,
                    int causal, int window, int n_sink, float scale,
                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * Forward with YaRN rotary position embeddings on q and k.  Page: "SnapKitty
 * Transformer 8B", model specification table ("YaRN RoPE 32x factor") and
 * section "Protected Inventions" (YaRN-scaled RoPE for 204800-token sequences,
 * applied inside the attention kernels).  The pages give no formula; the one
 * used is the YaRN paper's (Peng et al. 2023, section 3) on RoFormer's
 * rotation:
 *   theta_i = rope_base^(-2i/d), r_i = rope_orig_ctx * theta_i / (2 pi),
 *   gamma_i = clamp((r_i - rope_alpha) / (rope_beta - rope_alpha), 0, 1),
 *   h_i     = (1 - gamma_i) theta_i / rope_factor + gamma_i theta_i,
 * and the pair (x[2i], x[2i+1]) of query row i and key row j (positions i and
 * j, 0-based) turns by position * h_i.  The paper's attention temperature
 * multiplies the scaled scores by (0.1 ln rope_factor + 1)^2:
 *   s_ij = scale * (0.1 ln rope_factor + 1)^2 * rot(q_i) . rot(k_j),
 * and o, lse are those of these scores (lse is their natural-log normaliser).
 * The rotated rows are rounded once to bf16 before the products.  Mask, layouts
 * and errors as gqa_attn_fwd, plus GQA_ERR_ROPE when rope_base <= 1,
 * rope_factor < 1, rope_orig_ctx <= 0, not 0 <= rope_alpha < rope_beta or
 * rope_mode is neither GQA_ROPE_PREPASS nor GQA_ROPE_FUSED, and
 * GQA_ERR_NULL / GQA_ERR_WORKSPACE for a missing or short workspace.
 * score_bound: 0 takes the online maximum on every tile as gqa_attn_fwd does;
 * non-zero takes the score bound of gqa_attn_fwd_ws on the rotated queries and
 * keys (one more launch: the key-norm pre-pass on the rotated keys; same input
 * range note as gqa_attn_fwd_ws).
 * rope_mode: GQA_ROPE_PREPASS rotates q and k in one launch before the forward,
 * which then runs as gqa_attn_fwd on the rotated tensors (the faster mode);
 * GQA_ROPE_FUSED rotates only k beforehand and turns each query tile in
 * shared memory inside the forward kernel, right after it lands and before
 * its first Q K^T, so the workspace holds no rotated queries.  The two modes
 * compute the same bf16-rounded rotations.
 * workspace: device memory of at least
 * gqa_attn_fwd_yarn_workspace_size(B, H, G, S, d, rope_mode) bytes, 16-byte
 * aligned, owned by the caller and not used by any other call running at the
 * same time: the rotated keys [B][G][S][d] bf16, a [S][d/2] table of
 * (cos, sin) fp32 pairs, the key-norm record (B * G * 128 bytes) and, with
 * GQA_ROPE_PREPASS, the rotated queries [B][H][S][d] bf16, in that order; the
 * size function returns 0 for arguments the call rejects.
 */
enum { GQA_ROPE_PREPASS = 0, GQA_ROPE_FUSED = 1 };
GQA_API size_t gqa_attn_fwd_yarn_workspace_size(int B, int H, int G, int S, int d, int rope_mode);
GQA_API int gqa_attn_fwd_yarn(const void *q, const void *k, const void *v, void *o, float *lse,
                      int B, int H, int G, int S, int d,
                      int causal, int window, int n_sink, float scale,
                      float rope_base, float rope_factor, int rope_orig_ctx,
                      float rope_alpha, float rope_beta, int score_bound, int rope_mode,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * Forward on FP8 queries and keys.  Page: "SnapKitty Transformer 8B", section
 * "Protected Inventions" (a forward "with FP8 computation"; the pages name no
 * format).  q8 [B][H][S][d] and k8 [B][G][S][d] are OCP E4M3 bytes (1 sign, 4
 * exponent bits with bias 7, 3 mantissa bits; S.1111.111 is NaN), standing for
 * decode(byte) * q_scale and decode(byte) * k_scale; v [B][G][S][d] is bf16.
 * S = Q K^T runs on the tensor cores as tcgen05.mma kind::f8f6f4 with fp32
 * accumulation, the scores are scale * q_scale * k_scale * q8 . k8, and P.V is
 * the bf16 product of gqa_attn_fwd, so o and lse are those of gqa_attn_fwd on
 * the decoded queries and keys.  q8, k8 16-byte aligned.  Errors as
 * gqa_attn_fwd, plus GQA_ERR_SCALE when q_scale or k_scale is not finite and
 * positive or scale * q_scale * k_scale leaves the fp32 range.
 */
GQA_API int gqa_attn_fwd_fp8(const void *q8, const void *k8, const void *v, void *o, float *lse,
                     int B, int H, int G, int S, int d,
                     int causal, int window, int n_sink, float scale,
                     float q_scale, float k_scale, void *stream);

/*
 * Quantisation to the fp8 forward's input format: out[i] = E4M3(x[i] *
 * inv_scale) for n bf16 values x (device), round to nearest even, saturating
 * to +-448 (NaN stays NaN); byte out[i] then stands for decode(out[i]) /
 * inv_scale.  n a positive multiple of 16; x and out 16-byte aligned.  No page
 * describes this call: it prepares inputs for gqa_attn_fwd_fp8.
 */
GQA_API int gqa_attn_quantize_e4m3(const void *x, void *out, long long n, float inv_scale,
                                   void *stream);

/*
 * Bytes of scratch that gqa_attn_bwd needs for these sizes: an fp32 dq
 * accumulator [B][H][S][d]; two fp32 row arrays [B][H][S_pad] with
 * S_pad = S rounded up to a multiple of 128 (lse * log2(e) and the row term
 * D = rowsum(dout * o), both carrying the row's power-of-two scale below); an
 * fp16 copy of dout [B][H][S][d], each row scaled by a power of two; one int32
 * per kv head (B * G, rounded up to 16 bytes).  Returns 0 for invalid sizes.
 */
GQA_API size_t gqa_attn_bwd_workspace_size(int B, int H, int G, int S, int d);

/*
 * Backward.  Given q, k, v, the forward's o and lse, and dout = dL/do, writes
 * dq [B][H][S][d], dk and dv [B][G][S][d] (bf16; fp32 accumulation).  dk and dv
 * are summed over the H/G query heads that share each kv head.
 * Page: "SnapKitty Transformer 8B", section "Protected Inventions" (backward with
 * P recomputed from the saved row statistics, dP = dO.V^T, dS = P * (dP - D),
 * D = rowsum(dO * O), dQ reduced across query tiles), and the softmax backward
 * of "nx_f32_gqa_gate.nx source", test T4.
 * Operand precision of the tensor-core products: S = q.k^T, dK and dQ take
 * bf16 operands (q, k and dS = P * (dP - D) rounded once); dP = dout.v^T and
 * dV = P^T.dout take fp16 operands: each dout row and each v row is scaled by
 * the power of two that brings its largest element into [2^14, 2^15) (exact for
 * every bf16 value within 2^29 of that element) and P by the matching power of
 * two, so P reaches the dV product with 11 significant bits instead of 8.
 * D is taken on the o passed in, as stated above.
 * workspace: device memory of at least gqa_attn_bwd_workspace_size() bytes,
 * 16-byte aligned, owned by the caller and not used by any other call running at
 * the same time.  When workspace is NULL the call takes it with cudaMallocAsync
 * on `stream` and frees it with cudaFreeAsync before returning.
 * The call has no other effect on o, lse, q, k, v or dout.
 */
GQA_API int gqa_attn_bwd(const void *q, const void *k, const void *v, const void *o,
                 const void *dout, const float *lse,
                 void *dq, void *dk, void *dv,
                 int B, int H, int G, int S, int d,
                 int causal, int window, int n_sink, float scale,
                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward that allocates nothing.  Same computation, arguments and results as
 * gqa_attn_bwd, without the workspace: its scratch (the fp32 dq accumulator and
 * the two row arrays) lives in a fixed array of GQA_NOALLOC_SCRATCH_BYTES that
 * the library keeps in device memory; every GPU that loads the library holds
 * that array until the process exits.
 * It is meant for callers that cannot call cudaMalloc (or any allocator) when
 * they run the backward: plug-ins that run inside a host framework that owns all
 * device memory and hands them no scratch; real-time or latency-critical paths
 * that must never enter the allocator.  The pages have
 * no counterpart of this call.
 *   - A problem whose scratch (gqa_attn_bwd_workspace_size) exceeds
 *     GQA_NOALLOC_SCRATCH_BYTES is rejected with GQA_ERR_TOO_LARGE before
 *     anything is launched (64 MiB holds about 170,000 query rows, B*H*S).
 *   - The first call on a device looks up the device address of the array with
 *     that device current; make that first call before any stream capture.
 *   - All calls on a device share the one array, which keeps whatever the last
 *     call left in it; each call clears what it needs zeroed.  Calls that may
 *     run at the same time on the GPU (different streams without ordering)
 *     race on the array and corrupt each other's results.
 *   - Calls no cudaMalloc, cudaMallocAsync, cudaFree or allocating library
 *     routine.
 */
#define GQA_NOALLOC_SCRATCH_BYTES (64u << 20)
GQA_API int gqa_attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                 const void *dout, const float *lse,
                 void *dq, void *dk, void *dv,
                 int B, int H, int G, int S, int d,
                 int causal, int window, int n_sink, float scale, void *stream);

/* Static text for a gqa_status value (never NULL). */
GQA_API const char *gqa_attn_strerror(int status);

/*
 * After a call returned GQA_ERR_CUDA: which CUDA call (or set-up step) failed
 * and the CUDA runtime's description of the error, e.g.
 * "launch of the forward kernel: too many resources requested for launch
 * (cudaErrorLaunchOutOfResources)".  Kept per host thread, overwritten by the
 * next failure on that thread, never cleared by a success; the pointer stays
 * valid for the life of the thread.  Empty string if nothing failed yet.
 */
GQA_API const char *gqa_attn_last_error_detail(void);

/*
 * Synchronises `stream`, then returns and clears the device status word that
 * kernels set when a bounded wait expires: GQA_OK or GQA_ERR_DEVICE_TIMEOUT
 * (GQA_ERR_CUDA if the synchronisation itself failed).
 */
GQA_API int gqa_attn_last_device_status(void *stream);

/*
 * Self-test of the failure detection, on the device, without faulting it.
 * Launches one CTA on `stream` whose two waiting threads wait on mbarriers
 * that nothing ever arrives on: the first gives up after `budget_ms`
 * (1..1000), raises the CTA abort flag and records GQA_ERR_DEVICE_TIMEOUT; the
 * second waits with the kernels' normal 2 s budget and must leave through the
 * abort flag within about 1 ms of the first.  Synchronises `stream`.
 * elapsed_ns[2] (host) receives each thread's wait in nanoseconds and
 * returned_ok[2] (host) whether each wait reported success (expected 0, 0).
 * Returns the device status word read (and cleared) afterwards, which is
 * GQA_ERR_DEVICE_TIMEOUT when detection works; GQA_ERR_NULL / GQA_ERR_SHAPE
 * for bad arguments, GQA_ERR_CUDA if a CUDA call failed.  The CUDA context
 * stays usable: nothing traps, faults or hangs.
 */
GQA_API int gqa_attn_selftest_timeout(unsigned budget_ms, unsigned long long *elapsed_ns,
                                      int *returned_ok, void *stream);

/*
 * Kernel timing (a profiling aid, not thread-safe).  While enabled, every
 * kernel the library launches is bracketed by CUDA events recorded on its own
 * launch stream.  gqa_attn_timing_collect() waits for the events of the last
 * launch of each kernel and writes its duration in milliseconds to ms[id]
 * (-1 when that kernel has not run since the previous collect), for
 * id < min(n, GQA_KERNEL_COUNT).  No page describes this; it backs the
 * per-kernel roofline the benchmark reports.
 */
typedef enum {
    GQA_KERNEL_FWD = 0,       /* forward (one launch per gqa_attn_fwd) */
    GQA_KERNEL_BWD_PREP = 1,  /* backward: D, fp16 dout, dq accumulator cleared, LSE shift */
    GQA_KERNEL_BWD_MAIN = 2,  /* backward: dk, dv and the dq accumulation */
    GQA_KERNEL_BWD_DQ = 3,    /* backward: dq accumulator -> bf16 dq */
    GQA_KERNEL_FWD_KNORM = 4, /* gqa_attn_fwd_ws: key-norm maxima for the score bound */
    GQA_KERNEL_ROPE = 5,      /* gqa_attn_fwd_yarn: rotary table and the q / k rotation */
    GQA_KERNEL_COUNT = 6
} gqa_kernel_id;

GQA_API int gqa_attn_timing_enable(int on);
GQA_API int gqa_attn_timing_collect(float *ms, int n);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H_ */
