/*
 * mhc_post.h -- C ABI of the mHC post-mapping (hc_post) on sm_103a.
 *
 * Operation ("CANN HcPre 融合算子解析：mHC 结构前处理 custom.npu_hc_pre 与
 * npu_hc_pre_v2 实战指南", mHC section: hc_pre does the pre-processing, hc_post
 * the post-processing), per token t, output stream j and column d:
 *
 *     out[t][j][d] = post[t][j] * x[t][d] + sum_i comb[t][i][j] * residual[t][i][d]
 *
 * post is the pre-mapping's hPost and comb its Sinkhorn output (h_res); x is
 * the layer output (the F of F(hIn)), residual the n streams that entered the
 * layer.  The page prints the sum over the axis that would scale each stream
 * by its own row sum of comb; the stream mixing above is taken instead.
 * Accumulation is fp32; the result is rounded to bf16 (RN-even).
 *
 * Status codes are those of mhc_pre.h.
 */
#ifndef MHC_POST_H_
#define MHC_POST_H_

#include "mhc_pre.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Enqueue the post-mapping on `stream` (a cudaStream_t, NULL = legacy
 * default stream); asynchronous.
 *
 *   T         tokens (>= 0; T == 0 returns MHC_OK and launches nothing,
 *             pointers may then be NULL)
 *   n         streams, 1..8
 *   D         hidden width, a multiple of 8, >= 8
 *   x         device bf16 [T][D], 16-byte aligned
 *   residual  device bf16 [T][n][D], 16-byte aligned
 *   post      device fp32 [T][n], 4-byte aligned
 *   comb      device fp32 [T][n][n] (row i = input stream, column j = output
 *             stream), 4-byte aligned
 *   out       device bf16 [T][n][D], 16-byte aligned; must not overlap the
 *             inputs
 *
 * All tensors are contiguous and owned by the caller.  Returns
 * MHC_ERR_NULLPTR for a NULL tensor with T > 0, MHC_ERR_PARAM_INVALID for a
 * bad n, D, T or alignment, MHC_ERR_RUNTIME if the launch fails;
 * mhc_pre_last_error() then describes the problem.  No device-side waits:
 * the kernel cannot hang. */
MHC_API mhc_status_t mhc_post_run(int64_t T, int64_t n, int64_t D, const void *x, const void *residual,
                                  const float *post, const float *comb, void *out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MHC_POST_H_ */
