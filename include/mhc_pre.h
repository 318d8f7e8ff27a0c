/*
 * mhc_pre.h -- C ABI of the GB300 (sm_103a) mHC pre-mapping forward.
 *
 * The operation (per token t of T; n residual streams of width D; K = n*D):
 *
 *   invRms      = (mean_k x[t,k]^2 + normEps)^(-1/2)            raw x, k < n*D
 *   hMix[t,:]   = (x[t,:] (.) gamma) . phi^T                     phi [R, K] fp32
 *   w           = hMix * invRms, split [pre n | post n | res n*n]
 *   hPre        = sigmoid(alpha0*pre  + bias[0:n])  + hcEps
 *   hPost       = 2*sigmoid(alpha1*post + bias[n:2n])   (+ hcEps, two-gate only)
 *   H           = alpha2*res + bias[2n:], reshaped row-major to [n, n]
 *   comb        = Sinkhorn(H): softmax over each row + hcEps, then a column
 *                 normalisation, then (row, column) x (numIters - 1); every
 *                 normalisation divides by (sum + hcEps)
 *   y[t,d]      = bf16( sum_i m_i * x[t,i,d] ),  m = pre_mix[t] if given else hPre
 *
 * Sources: "CANN ops-transformer 中 aclnnMhcPreV2 算子接口全解析：MHC 架构 H
 * 投影矩阵与 hIn 计算实战指南" §三 (formula), §四 (two-phase call), §5.1-§5.4
 * (tensors, optional output group, status codes), §7.3 (n in {4,6,8}, D
 * multiple of 16, two-gate shapes); "CANN ops-transformer 算子详解：
 * aclnnMhcPreSinkhorn 接口与 MhcPreSinkhorn 实现剖析" §3.2 (Sinkhorn), §5.1
 * (sumOut / normOut shapes), §6 (status codes); "CANN HcPre 融合算子解析：
 * custom.npu_hc_pre 与 npu_hc_pre_v2 实战指南" (pre_mix).
 *
 * Conventions
 *  - Every tensor pointer in mhc_pre_args is a DEVICE pointer owned by the
 *    caller, dense and row-major (no strides).  x and y must be 16-byte
 *    aligned, the workspace 256-byte aligned, fp32 tensors 4-byte aligned.
 *  - The handle owns host-side configuration only.  It holds no device
 *    memory and may be used from one host thread at a time.
 *  - mhc_pre_run validates on the host, then enqueues kernels on `stream`
 *    and returns without waiting.  Results are deterministic: the same
 *    inputs give bit-identical outputs, run after run.
 *  - Nothing here falls back to the CPU.  If the device is not an sm_103
 *    part, mhc_pre_run returns MHC_ERR_RUNTIME.
 */
#ifndef MHC_PRE_H
#define MHC_PRE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MHC_API __attribute__((visibility("default")))
#else
#define MHC_API
#endif

/* Status codes, numerically equal to the aclnn codes the pages list. */
typedef int32_t mhc_status_t;
#define MHC_OK                0
#define MHC_ERR_NULLPTR       161001  /* a required pointer is NULL            */
#define MHC_ERR_PARAM_INVALID 161002  /* shape, mode, alignment or group error  */
#define MHC_ERR_RUNTIME       361001  /* CUDA launch / device-side failure      */

/* Precision of the projection (opImplMode on the MhcPreV2 page, §二). */
#define MHC_IMPL_FP32 0   /* phi used at full fp32 precision (exact products)   */
#define MHC_IMPL_TF32 1   /* phi truncated toward zero to 10 mantissa bits
                             (the pages' HF32 mode); x (bf16) is exact in both */

typedef struct mhc_pre_s *mhc_pre_t;

/* Element type of x and y (bf16 x is what every page's example uses; fp16 is
 * the other type the MhcPreSinkhorn page lists for x). */
#define MHC_DTYPE_BF16 0
#define MHC_DTYPE_FP16 1

/* Which fused forward kernel runs (mhc_pre_config.kernel).  AUTO lets the
 * library choose by shape; the others force one, for benchmarks and tests.
 * Every kernel computes the same results within the stated tolerances. */
#define MHC_KERNEL_AUTO    0
#define MHC_KERNEL_CLUSTER 1   /* 64-token tiles shared by a thread-block cluster   */
#define MHC_KERNEL_GRID    2   /* every SM on a few tiles (small T, bf16 x)         */
#define MHC_KERNEL_RESIDENT 3  /* cluster kernel keeping the last chunks of x in
                                  tensor memory for y (n = 4)                        */

/* Fixed per handle.  Defaults (mhc_pre_config_default): n = 4, D = 0 (must be
 * set), alpha_len = 3, num_iters = 20, norm_eps = hc_eps = 1e-6,
 * impl_mode = MHC_IMPL_FP32, need_backward = 0, batch_consistent = 0,
 * x_dtype = MHC_DTYPE_BF16, and every launch-choice field 0 (automatic).
 *
 * Launch choice (kernel .. gw_x_lead): 0 means "let the library choose";
 * a non-zero value fixes one choice of kernel or launch shape, for
 * benchmarks and tests.  None of them changes what is computed.  A forced
 * choice that does not fit the shape or device makes mhc_pre_run return
 * MHC_ERR_PARAM_INVALID.  The library reads no environment variable.
 *
 * batch_consistent (the Sinkhorn page's §8.1 "Batch 一致性", off by default
 * there too): every token's outputs are bitwise the same whatever T and
 * whatever other tokens share the call.  The forward then always runs the
 * 64-token cluster kernel at cluster size 2 (the reduction of a token over
 * its n*D columns is split the same way for every T), which can be slower
 * for small T.  With it off the cluster size follows T and the last bits of
 * a token's results may change with T (still deterministic for a given T:
 * the default is a fixed reduction order, as the pages require). */
typedef struct {
    int64_t n;              /* residual streams: 4, 6 or 8                          */
    int64_t D;              /* stream width: 16 <= D <= 16384, D % 16 == 0          */
    int32_t alpha_len;      /* 3 (pre/post/res) or 2 (no residual path)             */
    int32_t num_iters;      /* Sinkhorn iterations, 1..100 (pages: 20)              */
    double  norm_eps;       /* RMS epsilon, > 0 not required                        */
    double  hc_eps;         /* gate / Sinkhorn epsilon                              */
    int32_t impl_mode;      /* MHC_IMPL_FP32 or MHC_IMPL_TF32                       */
    int32_t need_backward;  /* 1: also write inv_rms, h_mix, sum_out, norm_out      */
    int32_t batch_consistent; /* 1: results per token independent of T (see above)  */
    int32_t x_dtype;        /* MHC_DTYPE_BF16 (x and y bf16) or MHC_DTYPE_FP16 (x and
                               y fp16; n = 4; the backward takes bf16 only). fp16
                               x runs the projection on fp16 planes of phi . gamma,
                               so every |phi . gamma| must be <= 65504: a larger
                               one sets bit 3 of the device error word, which
                               mhc_pre_status reports                              */
    int32_t kernel;         /* MHC_KERNEL_AUTO / _CLUSTER / _GRID / _RESIDENT (grid:
                               bf16 x; grid and resident: not batch_consistent)    */
    int32_t cluster;        /* cluster kernel: CTAs per cluster, 1, 2, 4, 8 or 16   */
    int32_t x_stages;       /* cluster kernel: deepest x ring tried, 2..8           */
    int32_t w_stages;       /* cluster kernel: deepest phi-plane ring tried, 2..8   */
    int32_t gw_groups;      /* grid-wide kernel: CTA groups, 1 or 2                 */
    int32_t gw_x_stages;    /* grid-wide kernel: deepest x ring tried, 2..8         */
    int32_t gw_x_lead;      /* grid-wide kernel: tiles its loads may run ahead of
                               its own y, 1..15                                     */
    int32_t tm_buffers;     /* resident kernel: tensor-memory chunk buffers, 1 or 2
                               (2: alternate tiles use their own, so a tile does
                               not wait for the previous one's y)                  */
} mhc_pre_config;

/* Per call.  R = n*n + 2n (alpha_len 3) or 2n (alpha_len 2); I = num_iters. */
typedef struct {
    int64_t      T;         /* tokens; 0 returns MHC_OK at once (pointers unchecked)  */
    const void  *x;         /* [T, n, D] of x_dtype (bf16 or fp16)     required       */
    const float *phi;       /* fp32 [R, n*D]                           required       */
    const float *alpha;     /* fp32 [alpha_len]                        required       */
    const float *bias;      /* fp32 [R]                                required       */
    const float *gamma;     /* fp32 [n, D] or NULL (no scaling)                       */
    const float *pre_mix;   /* fp32 [T, n] or NULL (y weights = hPre)                 */
    void        *y;         /* [T, D] of x_dtype                       required       */
    float       *h_post;    /* fp32 [T, n]                             required       */
    float       *h_res;     /* fp32 [T, n, n] comb after Sinkhorn; required when
                               alpha_len == 3; optional (filled with 0) when 2        */
    float       *h_pre;     /* fp32 [T, n]; required when need_backward or pre_mix,
                               else optional                                         */
    float       *inv_rms;   /* fp32 [T]          } need_backward == 1: all required  */
    float       *h_mix;     /* fp32 [T, R]       } (sum_out / norm_out only when     */
    float       *sum_out;   /* fp32 [2I, T, n]   }  alpha_len == 3);                  */
    float       *norm_out;  /* fp32 [2I, T, n, n]} need_backward == 0: all NULL       */
    void        *workspace;       /* device scratch, >= mhc_pre_workspace_size bytes   */
    size_t       workspace_bytes; /* its size                                          */
    const void  *weights;   /* NULL, or phi (.) gamma prepared by
                               mhc_pre_prepare_weights with this handle: the run
                               then uses it and neither reads phi nor gamma (they
                               may be NULL) nor launches the preparation          */
} mhc_pre_args;

/* Fill *cfg with the defaults listed above.  NULL cfg is ignored. */
MHC_API void mhc_pre_config_default(mhc_pre_config *cfg);

/* Validate cfg and create a handle.  MHC_ERR_NULLPTR if out or cfg is NULL;
 * MHC_ERR_PARAM_INVALID for a value outside the ranges above (the handle is
 * then not created and *out is set to NULL). */
MHC_API mhc_status_t mhc_pre_create(mhc_pre_t *out, const mhc_pre_config *cfg);

/* Bytes of device workspace a call with T tokens needs (first phase of the
 * pages' two-phase call).  Depends on the handle's shape and mode and on T;
 * T == 0 gives 0.  MHC_ERR_NULLPTR / MHC_ERR_PARAM_INVALID (T < 0). */
MHC_API mhc_status_t mhc_pre_workspace_size(mhc_pre_t h, int64_t T, size_t *bytes);

/* Weights phase, for calls that reuse one phi and gamma (the decode steps of
 * a layer): the projection's weight side, phi (.) gamma split into the
 * precision planes the tensor cores read, depends on phi, gamma and the
 * handle's n, D, alpha_len, impl_mode and x_dtype only.  mhc_pre_weights_size
 * gives the bytes of that form (a 256-byte header, then the planes);
 * mhc_pre_prepare_weights writes it into `weights` (a caller-owned device
 * buffer, 256-byte aligned, at least that size) on `stream`.  A run given
 * args->weights then skips its own preparation launch: one copy of the
 * 256-byte header into the workspace and one kernel.  The buffer stays
 * valid until phi or gamma change; it must come from a handle with the same
 * n, D, alpha_len, impl_mode and x_dtype.  fp16 x: an entry of phi (.) gamma
 * beyond fp16's range is recorded in the buffer's header and reported by
 * mhc_pre_status after each run that uses it.  The pages' operator
 * re-derives nothing per call either: its weight-side tiling is fixed at
 * set-up (the MhcPreV2 page, §十).  MHC_ERR_NULLPTR for a NULL handle,
 * bytes, phi or weights; MHC_ERR_PARAM_INVALID for misalignment or a small
 * buffer; MHC_ERR_RUNTIME if the launch fails. */
MHC_API mhc_status_t mhc_pre_weights_size(mhc_pre_t h, size_t *bytes);
MHC_API mhc_status_t mhc_pre_prepare_weights(mhc_pre_t h, const float *phi, const float *gamma, void *weights,
                                             size_t weights_bytes, void *stream);

/* Second phase: check args, then enqueue the forward on `stream` (a
 * cudaStream_t; NULL = legacy default stream).  Host-side checks return
 * before anything is enqueued:
 *   MHC_ERR_NULLPTR        a required pointer is NULL;
 *   MHC_ERR_PARAM_INVALID  T < 0, an optional-group violation, a pointer
 *                          not aligned as stated, or workspace too small;
 *   MHC_ERR_RUNTIME        no usable sm_103 device, or a launch failed.
 * Device-side waits are bounded; a wait that gives up sets an error word in
 * the workspace that mhc_pre_status reports. */
MHC_API mhc_status_t mhc_pre_run(mhc_pre_t h, const mhc_pre_args *args, void *stream);

/* Synchronise `stream`, then report MHC_ERR_RUNTIME if a CUDA error is
 * pending or the last run's device error word is set; else MHC_OK.  The
 * word is read from `workspace` when it is given.  With workspace NULL it is
 * read from the library's fixed scratch array if the handle's last run was
 * mhc_pre_run_noalloc, and not read at all otherwise. */
MHC_API mhc_status_t mhc_pre_status(mhc_pre_t h, const void *workspace, void *stream);

/* Optional timing hooks.  When set, mhc_pre_run records `before` on its
 * stream just before it launches the fused forward kernel and `after` just
 * after (both cudaEvent_t; pass NULL, NULL to clear); mhc_pre_backward_run
 * (mhc_pre_backward.h) does the same around its contraction kernel.  This
 * lets a caller time that kernel alone, with CUDA events on the stream it
 * runs on.  The events are borrowed, not owned.  MHC_ERR_NULLPTR if h is
 * NULL. */
MHC_API mhc_status_t mhc_pre_set_profile_events(mhc_pre_t h, void *before, void *after);

/* Device wait limit and a test of the give-up path.  Every wait inside the
 * forward kernels is bounded: after wait_limit_us microseconds (0 restores
 * the default, 2 s; at most 10 s) it gives up, sets the device error word and
 * the kernel winds down, so that mhc_pre_status reports MHC_ERR_RUNTIME and
 * the CUDA context stays usable (the status codes of the MhcPreSinkhorn page,
 * §6).  withhold_last_x_copy = 1 makes the next runs on this handle leave out
 * one copy of x -- the last one the first CTA would issue -- so that the
 * waits on it give up: a host-requested test of that path which faults
 * nothing (no copy is left in flight, every other wait still ends).  Those
 * runs' outputs are then incomplete.  Set it back to 0 for normal runs.
 * Applies to the fused forward kernels of mhc_pre_run and
 * mhc_pre_run_noalloc and to the contraction kernel of mhc_pre_backward_run
 * (there the first CTA leaves out the copies of its last tile).
 * MHC_ERR_NULLPTR if h is NULL; MHC_ERR_PARAM_INVALID for a value outside
 * these ranges. */
MHC_API mhc_status_t mhc_pre_set_wait_test(mhc_pre_t h, uint32_t wait_limit_us, int32_t withhold_last_x_copy);

/* Launch shape chosen by the last successful mhc_pre_run on this handle:
 * CTAs per cluster (0 for the grid-wide kernel), grid size in CTAs, x-ring
 * depth, and phi-ring depth (cluster kernels) or group count (grid-wide).
 * After mhc_pre_backward_run: 1, the contraction kernel's grid, its stage
 * count, and the token-stage block count.  All zero before the first run.
 * Any output pointer may be NULL. */
MHC_API mhc_status_t mhc_pre_last_launch(mhc_pre_t h, int32_t *cluster, int32_t *grid,
                                         int32_t *stages, int32_t *ystages);

/* Name of the fused kernel the last successful mhc_pre_run on this handle
 * launched, or "bw_main_kernel" after mhc_pre_backward_run ("" before the
 * first run, or for a NULL handle).  The string is
 * static and owned by the library.  A diagnostic for benchmarks and tests;
 * the pages have no counterpart. */
MHC_API const char *mhc_pre_last_kernel(mhc_pre_t h);

/* Same forward as mhc_pre_run, for callers that cannot allocate device memory
 * at all -- for instance code running under an allocator lock, a host
 * runtime with no device allocator of its own, or a stream that is not
 * allowed to block on cudaMalloc/cudaFree.  It takes no workspace:
 * args->workspace must be NULL and args->workspace_bytes 0.  Instead the
 * library keeps one fixed scratch array of MHC_PRE_STATIC_SCRATCH_BYTES in
 * device memory (a file-scope __device__ variable, so every GPU that loads the
 * library holds it until the process exits).  This entry point itself
 * allocates nothing: it calls no cudaMalloc, cudaFree or allocating library
 * routine.
 *  - The first call on each device looks up the array's device address with
 *    that device current; make that first call before any stream capture.
 *  - A call whose mhc_pre_workspace_size exceeds the array is rejected with
 *    MHC_ERR_PARAM_INVALID (mhc_pre_last_error says by how much).
 *  - Every call shares the one array, and each run rewrites all of it that it
 *    uses (the error word is cleared at the start of every run), so calls
 *    whose work overlaps on the GPU (different streams, no ordering between
 *    them) race on it: serialise them.
 *  - The device error word lives in that array; check a run with
 *    mhc_pre_status(h, NULL, stream), which reads it from there (a wait
 *    that gave up, or an fp16 weight out of range, gives MHC_ERR_RUNTIME
 *    as it does after mhc_pre_run).
 *  - The array's address is cached per device together with the CUDA
 *    context it was looked up in; if the context changes (for instance
 *    after cudaDeviceReset) the next call looks it up again.
 * This entry point is a property of this library; the pages' operator has no
 * counterpart.  Other arguments and status codes as mhc_pre_run. */
#define MHC_PRE_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
MHC_API mhc_status_t mhc_pre_run_noalloc(mhc_pre_t h, const mhc_pre_args *args, void *stream);

/* Release the handle (NULL is ignored). */
MHC_API void mhc_pre_destroy(mhc_pre_t h);

/* Static description of a status code. */
MHC_API const char *mhc_pre_status_string(mhc_status_t s);

/* Text of the last validation failure on this host thread ("" if none). */
MHC_API const char *mhc_pre_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MHC_PRE_H */
