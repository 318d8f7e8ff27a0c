/*
 * mhc_pre_stages.h -- the composite route of the mHC pre-mapping: the
 * forward as three separate operations, a debug aid next to the fused
 * mhc_pre_run.
 *
 * "CANN HcPre 融合算子解析：mHC 结构前处理 custom.npu_hc_pre 与 npu_hc_pre_v2
 * 实战指南" (功能说明与计算流程; 融合路由策略) splits the pre-processing into
 * an RMS-reciprocal operator, the mixing projection and a Sinkhorn operator
 * that takes the mixes and the reciprocal, the split route being the slower
 * fallback of the fused operator.  Here:
 *
 *   mhc_pre_inv_rms_run   invRms[t] = (mean over n*D of x[t]^2 + norm_eps)^-1/2
 *   mhc_pre_mixes_run     mixes[t][r] = sum_k x[t][k] gamma[k] phi[r][k]
 *                         (the hMix of the forward: before invRms)
 *   mhc_pre_sinkhorn_run  from mixes and invRms: the gates, the Sinkhorn mix
 *                         and y = sum_i w_i x[t][i], with every output of
 *                         mhc_pre_run (inv_rms / h_mix, when requested, are
 *                         copies of the inputs)
 *
 * The three in order give the outputs of mhc_pre_run up to fp32 rounding
 * order (the mixes are fp32 CUDA-core sums, not tensor-core plane products:
 * impl_mode is not applied).  All run on the handle's n, D, alpha_len,
 * num_iters, eps and x_dtype; all pointers are device pointers to contiguous
 * tensors owned by the caller; every call is asynchronous on `stream` and
 * returns the status codes of mhc_pre.h (T == 0: MHC_OK, nothing launched).
 * No workspace, no device-side waits.
 */
#ifndef MHC_PRE_STAGES_H_
#define MHC_PRE_STAGES_H_

#include "mhc_pre.h"

#ifdef __cplusplus
extern "C" {
#endif

/* x [T, n, D] (x_dtype), 16-byte aligned; inv_rms fp32 [T]. */
MHC_API mhc_status_t mhc_pre_inv_rms_run(mhc_pre_t h, int64_t T, const void *x, float *inv_rms, void *stream);

/* x [T, n, D] (x_dtype), 16-byte aligned; phi fp32 [R, n*D]; gamma fp32
 * [n, D] or NULL; mixes fp32 [T, R]. */
MHC_API mhc_status_t mhc_pre_mixes_run(mhc_pre_t h, int64_t T, const void *x, const float *phi,
                                       const float *gamma, float *mixes, void *stream);

/* args as for mhc_pre_run (its x, alpha, bias, pre_mix and outputs are used;
 * phi, gamma and the workspace are not), mixes fp32 [T, R] and inv_rms fp32
 * [T] from the two calls above. */
MHC_API mhc_status_t mhc_pre_sinkhorn_run(mhc_pre_t h, const mhc_pre_args *args, const float *mixes,
                                          const float *inv_rms, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MHC_PRE_STAGES_H_ */
