/*
 * farn.h - fused rank-sum + residual add + RMSNorm on one GB300 (sm_103a).
 *
 * The operation is the contract of FlagTree pull request "[TLERaw] Add
 * NVSHMEM allreduce RMSNorm tutorial" (Summary):
 *
 *     reduced      = sum over ranks r = 0..W-1 of x[r]
 *     residual_out = reduced + residual
 *     norm_out     = RMSNorm(residual_out, weight, eps)
 *
 * with the epilogue of its Implementation section 3 (residual add, then
 * RMSNorm with FP32 accumulation) fused into the same kernel.  On one GPU
 * the W partials of the page's all-reduce are W bf16 tensors that already
 * sit in this GPU's memory; the library reads them through a pointer array,
 * so there is no collective and no cross-GPU traffic.
 *
 * Arithmetic (element (t,h); f() widens bf16 to fp32 exactly, bf16()
 * rounds fp32 to nearest even):
 *     reduced[t,h]      = bf16(f(x[0]) + f(x[1]) + ... + f(x[W-1]))   fp32, rank order
 *     residual_out[t,h] = bf16(f(reduced[t,h]) + f(residual[t,h]))
 *     rstd[t]           = 1 / sqrt(sum_h f(residual_out[t,h])^2 / H + eps)
 *     norm_out[t,h]     = bf16((f(residual_out[t,h]) * rstd[t]) * f(weight[h]))
 * reduced and residual_out are exact functions of the inputs (bit for bit
 * the same on every launch configuration); norm_out depends on the
 * summation order of the row's sum of squares and may differ by one bf16
 * ulp between launch configurations.
 *
 * Layout: every [T,H] tensor is row-major and contiguous (row t starts at
 * element t*H), bf16 (2-byte IEEE bfloat16 patterns).  weight is [H].
 * All tensor pointers are DEVICE pointers on the context's device, owned
 * by the caller; the library keeps none of them after a call returns.
 * The fast kernels need every pointer 16-byte aligned and H a multiple
 * of 8; other shapes and alignments are served by a slower kernel.
 *
 * Errors: every entry point returns FARN_OK (0) or a negative farn_status.
 * On an error nothing is launched and no output is written.
 * Launch-time CUDA errors are reported; errors of the asynchronous kernel
 * itself surface at the caller's next synchronisation, as usual in CUDA.
 */
#ifndef FARN_H_
#define FARN_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Largest number of rank partials one call accepts. */
#define FARN_MAX_W 32

typedef enum {
    FARN_OK = 0,
    FARN_ERR_INVALID_ARG = -1,  /* null pointer, W/T/H/eps out of range     */
    FARN_ERR_UNSUPPORTED = -2,  /* shape the library cannot launch           */
    FARN_ERR_ALIAS = -3,        /* an output overlaps an input or an output  */
    FARN_ERR_CUDA = -4,         /* CUDA runtime error (launch, device query) */
    FARN_ERR_NOMEM = -5         /* host allocation of the context failed     */
} farn_status;

/* Element types of the partials (farn_forward_typed). */
typedef enum {
    FARN_BF16 = 0,   /* bfloat16, 2 bytes */
    FARN_F32 = 1     /* IEEE binary32, 4 bytes */
} farn_dtype;

/* Opaque per-device context: device properties and kernel attributes
 * queried once.  Immutable after farn_create; one context may serve any
 * number of streams and host threads at once. */
typedef struct farn_ctx farn_ctx;

/* Create a context for CUDA device `device` (this is the one-time set-up
 * that the page's host side does at initialisation, Implementation
 * section 4, "host-side C ABI"; there is no communicator to bootstrap).
 * Queries the SM count and cluster limits, sets kernel attributes and
 * allocates one 256-byte device block (the status word of the TMA-staged
 * kernel, see farn_device_status).  The caller's current device is left
 * as it was.  The environment is read here and only here: FARN_VARIANT,
 * FARN_CLUSTER, FARN_VPT, FARN_PDL, FARN_SMALL_T, FARN_BULK,
 * FARN_BULK_CTAS, FARN_STAGE, FARN_STAGE_R, FARN_STAGE_CTAS,
 * FARN_STAGE_MIN_T and FARN_STAGE_MIN_MB override the kernel choice (tests
 * and sweeps); FARN_FAULT_INJECT injects a fault for the tests: "create"
 * fails this call, "launch" makes every launch of the context fail before
 * anything is enqueued, "stall" makes CTA 0 of every TMA-staged launch
 * wait out its time limit and report it in the status word.
 * Returns FARN_ERR_INVALID_ARG if out is NULL or device < 0 or not a device
 * of this process, FARN_ERR_CUDA if the device cannot be queried (or
 * FARN_FAULT_INJECT=create), FARN_ERR_NOMEM. */
int farn_create(farn_ctx **out, int device);

/* The fused operator on `stream` (asynchronous; the call does not wait
 * for the GPU).
 *   partials     host array of W device pointers, partials[r] -> x[r],
 *                bf16 [T,H]; the array itself is read during the call only.
 *   W            1 .. FARN_MAX_W
 *   residual     bf16 [T,H]
 *   weight       bf16 [H]
 *   eps          finite, >= 0 (fp32; added to the mean square inside sqrt)
 *   T            rows (tokens), >= 0; T == 0 returns FARN_OK and launches
 *                nothing (the tensor pointers may then be NULL, as the data
 *                pointers of empty tensors are)
 *   H            hidden size (row length), >= 1
 *   reduced_out, residual_out, norm_out   bf16 [T,H] outputs
 *   stream       CUDA stream (0 = legacy default stream)
 * Outputs may not overlap each other or any input, with one exception:
 * residual_out may be exactly residual (in-place residual update).
 * Returns FARN_ERR_INVALID_ARG (ctx or a pointer NULL, W, T, H or eps out
 * of range, T*H*2 bytes overflowing), FARN_ERR_ALIAS, FARN_ERR_UNSUPPORTED,
 * or FARN_ERR_CUDA if the launch failed. */
int farn_forward(const farn_ctx *ctx,
                 const void *const *partials, int W,
                 const void *residual, const void *weight, float eps,
                 int64_t T, int64_t H,
                 void *reduced_out, void *residual_out, void *norm_out,
                 cudaStream_t stream);

/* farn_forward with the partials in `partial_dtype` (a farn_dtype):
 * FARN_BF16 is exactly farn_forward; FARN_F32 takes fp32 partials [T,H]
 * (for example the fp32 output of a GEMM epilogue, before any rounding)
 * and sums their own fp32 values in rank order, rounding once to bf16 --
 * the "FP32 accumulation where required" of the page's Implementation
 * section 3.  residual, weight and the three outputs stay bf16; everything
 * else (layout, ownership, aliasing, errors) is as for farn_forward, with
 * each fp32 partial occupying T*H*4 bytes.  Returns FARN_ERR_INVALID_ARG
 * for an unknown dtype. */
int farn_forward_typed(const farn_ctx *ctx,
                       const void *const *partials, int partial_dtype, int W,
                       const void *residual, const void *weight, float eps,
                       int64_t T, int64_t H,
                       void *reduced_out, void *residual_out, void *norm_out,
                       cudaStream_t stream);

/* The argument checks of farn_forward alone, on the host: no CUDA call, no
 * launch, pointers are only compared, never dereferenced.  Returns what
 * farn_forward would return before launching. */
int farn_check_args(const void *const *partials, int W,
                    const void *residual, const void *weight, float eps,
                    int64_t T, int64_t H,
                    const void *reduced_out, const void *residual_out,
                    const void *norm_out);

/* Read and clear the context's device status word (blocking: waits for
 * the device).  0 means every wait of the TMA-staged kernel completed; a
 * non-zero value has one bit per kind of wait that gave up after its time
 * limit (2 s): 1 a consumer waiting for a staged segment, 2 the producer
 * waiting for a free stage, 4 a consumer in the row reduction, 8 the
 * producer draining its copies.  The kernel that gave up left its outputs
 * incomplete.  The TMA-staged kernel runs where farn_plan /
 * farn_plan_moe_combine report variant 3, and in every
 * farn_forward_noalloc call.  Returns FARN_ERR_INVALID_ARG or FARN_ERR_CUDA
 * on failure. */
int farn_device_status(const farn_ctx *ctx, int *status);

/* Release a context (NULL is accepted).  Returns FARN_OK. */
int farn_destroy(farn_ctx *ctx);

/* Text for a farn_status value (never NULL). */
const char *farn_status_string(int status);

/* Which kernel variant farn_forward would launch for this shape and these
 * pointers, without launching: 0 row (one CTA per row; decode sizes, and
 * long calls with a bf16 norm_out of W < 8 bf16 partials or of 8..11 with
 * H <= 5120, or with an FP8 / NVFP4 output of one or two partials or of
 * W < 8 with H <= 5120), 1 cluster (a cluster of CTAs splits each row; fewer than 16
 * rows), 2 generic (any H or alignment), 3 bulk (persistent CTAs whose
 * producer warp stages column segments of every input row in shared memory
 * with TMA bulk copies; rows of at most 16384 elements; calls of W >= 12
 * bf16 partials from 256 rows, long calls of 8..11 with 5120 < H < 8192,
 * or any call when enabled), 4 stage (persistent CTAs whose threads stage their own
 * vectors in shared memory with cp.async; the other long calls: 8..11
 * partials with H >= 8192, and the FP8 / NVFP4 outputs of W >= 3 partials
 * with H > 5120 or of W >= 8).
 * *cluster_size receives the CTAs per row (1 for row and generic),
 * *threads the threads per CTA.  Returns a farn_status. */
int farn_plan(const farn_ctx *ctx, int W, int64_t T, int64_t H,
              const void *const *partials, const void *residual,
              const void *weight, const void *reduced_out,
              const void *residual_out, const void *norm_out,
              int *variant, int *cluster_size, int *threads);

/* farn_forward_noalloc - the fused operator for callers that cannot
 * allocate device memory.  (No counterpart in the paper: the page's host
 * side allocates a symmetric workspace; this entry point exists for
 * callers that must not call cudaMalloc, e.g. code running inside another
 * framework's plugin or allocator interface, where every device allocation
 * has to go through that framework.)
 *
 * Same arithmetic, arguments, layout and error checks as farn_forward, but
 * without a context: `device` names the CUDA device that owns the tensors.
 * It always runs the TMA-staged kernel and allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library call.  The kernel's only
 * memory beyond the caller's tensors is a 4-byte status word kept in a
 * fixed 256-byte array that this library places in every GPU's memory for
 * the life of the process; a call needs that one word whatever T, H and W
 * are.  Every shape with 16-byte aligned tensors, H % 8 == 0 and
 * H <= 16384 is taken, for any W <= FARN_MAX_W; other shapes (tensors not
 * 16-byte aligned, H % 8 != 0, rows longer than 16384 elements) return
 * FARN_ERR_UNSUPPORTED.
 *
 * The first call on a device sets that device up (finds the array's device
 * address, reads the device limits, sets the kernels' shared-memory
 * attribute); make that first call before any stream capture.  Every call
 * clears the status word on `stream` before launching; the word is shared
 * by all calls on the device, so calls that overlap on the GPU (different
 * streams, no ordering between them) race on it.
 *
 * status_out: optional host pointer.  When non-NULL the call waits for the
 * kernel to finish and stores the status word there (0 = every wait
 * completed; bits as in farn_device_status).  When NULL the call is
 * asynchronous like farn_forward.
 * Returns FARN_OK, FARN_ERR_INVALID_ARG (as farn_forward, or device out of
 * range), FARN_ERR_ALIAS, FARN_ERR_UNSUPPORTED or FARN_ERR_CUDA. */
int farn_forward_noalloc(int device,
                         const void *const *partials, int W,
                         const void *residual, const void *weight, float eps,
                         int64_t T, int64_t H,
                         void *reduced_out, void *residual_out, void *norm_out,
                         cudaStream_t stream, int *status_out);

/* farn_forward_typed plus an FP8 copy of norm_out for the next layer's
 * GEMM.  (The page does not describe this output; it extends the fused
 * epilogue by one step.)  Per row t:
 *     amax         = max over h of |norm_out[t,h]|   (the bf16 values; NaN ignored)
 *     row_scale[t] = amax / 448, or 1 if amax is 0   (fp32; norm ~ q * scale)
 *     norm_q[t,h]  = E4M3(norm_out[t,h] * inv),  inv = 448 / amax (fp32), or 1
 * E4M3 is the OCP 8-bit float with 4 exponent and 3 fraction bits (largest
 * finite 448, no infinities); the conversion rounds to nearest even and
 * saturates larger magnitudes (and infinities) to +-448; NaN stays NaN.
 *   norm_q     uint8 [T,H] (E4M3 patterns), 16-byte aligned for the fast
 *              kernels
 *   row_scale  float [T]
 *   norm_out   bf16 [T,H], or NULL to skip writing it (it is still computed)
 * The other arguments, checks and errors are those of farn_forward_typed;
 * norm_q and row_scale take part in the aliasing checks. */
int farn_forward_quant(const farn_ctx *ctx,
                       const void *const *partials, int partial_dtype, int W,
                       const void *residual, const void *weight, float eps,
                       int64_t T, int64_t H,
                       void *reduced_out, void *residual_out, void *norm_out,
                       void *norm_q, float *row_scale,
                       cudaStream_t stream);

/* farn_forward_typed plus an NVFP4 copy of norm_out, the 4-bit input of a
 * block-scaled GEMM.  (Not described by the page either.)  Each block of 16
 * consecutive elements of a row, b = h / 16, shares one E4M3 scale under
 * the fp32 tensor scale g = tensor_scale (a calibrated input: a fused
 * kernel cannot see the whole tensor before it writes its first block):
 *     amax            = max of |norm_out| over the block (NaN ignored)
 *     block_scale[t,b] = E4M3((amax / 6) * g)            (saturating)
 *     inv             = g / value(block_scale[t,b])      (fp32 division)
 *     code[t,h]       = E2M1(norm_out[t,h] * inv)
 * E2M1 has 1 sign, 2 exponent and 1 fraction bit (magnitudes 0, 0.5, 1,
 * 1.5, 2, 3, 4, 6); the conversion rounds to nearest even and saturates
 * larger magnitudes and infinities to +-6; a NaN element is written as +6
 * (code 7); a block whose scale is 0 gets all-zero codes.  The value a code
 * stands for is value(code) * value(block_scale) / g.
 *   norm_fp4     uint8 [T, H/2]: codes of elements 2i (low nibble) and
 *                2i+1 (high nibble) in byte i; 4-byte aligned for the
 *                fast kernels
 *   block_scale  uint8 [T, H/16] (E4M3 patterns, row-major, no swizzle)
 *   tensor_scale finite, > 0
 *   norm_out     bf16 [T,H], or NULL to skip writing it
 *   H            a multiple of 16
 * The other arguments, checks and errors are those of farn_forward_typed
 * (FARN_ERR_INVALID_ARG also for H % 16 != 0 or a bad tensor_scale);
 * norm_fp4 and block_scale take part in the aliasing checks. */
int farn_forward_nvfp4(const farn_ctx *ctx,
                       const void *const *partials, int partial_dtype, int W,
                       const void *residual, const void *weight, float eps,
                       int64_t T, int64_t H, float tensor_scale,
                       void *reduced_out, void *residual_out, void *norm_out,
                       void *norm_fp4, void *block_scale,
                       cudaStream_t stream);

/* farn_moe_combine - the MoE "local y reduce" fused with the same
 * residual add + RMSNorm.  (The page names the per-token reduction of
 * expert outputs but defines neither its weights nor its layout; this is
 * the plain reading.)  For each token t and column h:
 *     reduced[t,h] = bf16(acc),  acc = -0; for k = 0..K-1, slot s = index[t*K+k]
 *                    in [0, n_slots):  acc = acc + gates[t*K+k] * f(expert_out[s,h])
 * with the product and the sum each rounded to fp32 (no fused multiply-add),
 * k in order; slots outside [0, n_slots) (e.g. -1 for a dropped expert) are
 * skipped, and are never read.  residual_out and norm_out then follow as in
 * farn_forward.
 *   expert_out  bf16 [n_slots, H], one row per (token, expert) assignment
 *   index       int32 [T, K] (4-byte aligned), gates fp32 [T, K] (4-byte aligned)
 *   K           1 .. FARN_MAX_W
 * Other arguments, layouts, ownership, in-place residual_out and errors as
 * for farn_forward; outputs may not overlap expert_out, index or gates. */
int farn_moe_combine(const farn_ctx *ctx,
                     const void *expert_out, int64_t n_slots,
                     const int32_t *index, const float *gates, int K,
                     const void *residual, const void *weight, float eps,
                     int64_t T, int64_t H,
                     void *reduced_out, void *residual_out, void *norm_out,
                     cudaStream_t stream);

/* Which kernel farn_moe_combine would launch for this shape and these
 * pointers, without launching: 2 generic (any H or alignment), 3 bulk
 * (persistent CTAs that gather the rows into shared memory with TMA bulk
 * copies; long inputs with rows of more than 3072 elements, or 5120 below
 * 8 experts, that fit two segments of at most 512 consumer threads or more
 * segments of 256), 4 stage (persistent CTAs that gather the rows into
 * shared memory with cp.async; the other long inputs with such rows),
 * 5 combine (one CTA per row; shorter inputs and shorter rows).  *threads receives the threads per CTA (at most 544 for bulk: one
 * producer warp and the consumers; at most 512 otherwise).  Returns a farn_status (FARN_ERR_INVALID_ARG for a bad shape or a
 * NULL pointer; aliasing is not checked). */
int farn_plan_moe_combine(const farn_ctx *ctx, int K, int64_t T, int64_t H,
                          const void *expert_out, const void *residual,
                          const void *weight, const void *reduced_out,
                          const void *residual_out, const void *norm_out,
                          int *variant, int *threads);

/* Flags of farn_plan_typed. */
#define FARN_PLAN_FP8_OUT 1   /* the call also writes the FP8 norm output */
#define FARN_PLAN_NVFP4_OUT 2 /* the call also writes the NVFP4 norm output */

/* farn_plan for partials of type `partial_dtype` (a farn_dtype), for a
 * farn_forward_typed call (flags 0), a farn_forward_quant call
 * (FARN_PLAN_FP8_OUT) or a farn_forward_nvfp4 call (FARN_PLAN_NVFP4_OUT);
 * with either flag norm_out may be NULL.  Only shape, dtype,
 * flags and pointer alignment matter; aliasing is not checked.  Returns
 * FARN_ERR_INVALID_ARG for a bad shape, dtype, flag or NULL pointer. */
int farn_plan_typed(const farn_ctx *ctx, int partial_dtype, int flags, int W,
                    int64_t T, int64_t H,
                    const void *const *partials, const void *residual,
                    const void *weight, const void *reduced_out,
                    const void *residual_out, const void *norm_out,
                    int *variant, int *cluster_size, int *threads);

#ifdef __cplusplus
}
#endif

#endif /* FARN_H_ */
