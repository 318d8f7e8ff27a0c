/*
 * mhc_pre_backward.h -- C ABI of the backward of the mHC pre-mapping with
 * Sinkhorn on sm_103a.
 *
 * Operation ("CANN ops-transformer 算子解析：MhcPreBackward 反向梯度算子实现与
 * aclnn 调用指南", §一, §三 3.1-3.8, §8.1-8.2; the Sinkhorn variant's saved
 * sums and matrices, "aclnnMhcPreSinkhorn 接口与 MhcPreSinkhorn 实现剖析"
 * §3.2, §5.1, §10): given the forward's inputs x, phi, alpha, gamma, its
 * saved intermediates invRms, hMix, hPre, hPost (and, for the Sinkhorn form,
 * sumOut and normOut) and the upstream gradients of y (grad_h_in), hPost and
 * the residual mix, form the gradients of the forward with respect to x,
 * phi, alpha, bias and gamma:
 *
 *   0  (Sinkhorn form) carry grad_h_res back through the 2*numIters saved
 *      normalisation steps and the row softmax to the res logits;
 *   3.1 H_pre_grad[i] = sum_d grad_h_in[d] x[i][d];  gx3[i][d] = grad_h_in[d] hPre[i]
 *   3.2 pre gate:  g = H_pre_grad s (1 - s), s = hPre - hcEps
 *   3.3 post gate: g = grad_h_post hPost (1 - hPost / 2)
 *   3.4 res map:   g = grad of the logits
 *   3.5 G = [alpha0 g_pre, alpha1 g_post, alpha2 g_res] * invRms;
 *       inv_rms_grad = sum_r [alpha g]_r hMix_r
 *   3.6 grad_phi = G^T (x . gamma);  x_rs_grad = G phi
 *   3.7 grad_gamma = sum_t x . x_rs_grad;
 *       grad_x = gx3 + gamma . x_rs_grad - inv_rms_grad invRms^3 / (nD) * x
 *   3.8 grad_x += grad_x_post (when given)
 * grad_alpha[c] and grad_bias[r] are the token sums of the gate gradients
 * times the pre-alpha terms, and of the gate gradients themselves.  The RMS
 * term uses raw x and grad_alpha[2] the pre-alpha res term hMix_res invRms,
 * because the outputs are the gradients of the forward (the page's printed
 * symbols there are read as garbled).
 *
 * Precision: fp32 mode (impl_mode 0) forms both contractions on the tensor
 * cores from exact three-plane bf16 splits of G and of phi . gamma (products
 * up to combined order 2^-16 kept), fp32 accumulation; tf32 mode (1) first
 * truncates G and phi . gamma to 10 mantissa bits (the pages' HF32) and
 * splits them in two planes.  grad_x is rounded once to bf16 (RN-even); the
 * other outputs are fp32.  Token sums run in a fixed order: results are
 * bitwise reproducible for a given T and device.
 *
 * Scope: three-gate handles only (alpha_len 3: gradAlpha has 3 entries), n
 * = 4, D a multiple of 64, y formed from hPre (no pre_mix).  Other handles
 * get MHC_ERR_PARAM_INVALID from both calls below.
 */
#ifndef MHC_PRE_BACKWARD_H_
#define MHC_PRE_BACKWARD_H_

#include "mhc_pre.h"

#ifdef __cplusplus
extern "C" {
#endif

/* All pointers are device pointers to contiguous tensors owned by the caller;
 * bf16 tensors and the workspace must be 16-byte aligned, fp32 ones 4-byte. */
typedef struct {
  int64_t T;                 /* tokens; 0 => MHC_OK, nothing launched */
  const void *x;             /* bf16 [T, n, D] (the forward's input) */
  const float *phi;          /* [n*n + 2n, n*D] */
  const float *alpha;        /* [3] */
  const float *gamma;        /* [n, D] or NULL (then grad_gamma must be NULL) */
  const void *grad_h_in;     /* bf16 [T, D], gradient of y */
  const float *grad_h_post;  /* [T, n] */
  const float *grad_h_res;   /* [T, n, n]: gradient of the Sinkhorn output when
                                sum_out/norm_out are given, else of the res logits */
  const float *inv_rms;      /* [T]        saved by the forward */
  const float *h_mix;        /* [T, R]     saved by the forward (before invRms) */
  const float *h_pre;        /* [T, n]     saved by the forward */
  const float *h_post;       /* [T, n]     the forward's output */
  const float *sum_out;      /* [2I, T, n]    or NULL } both or neither */
  const float *norm_out;     /* [2I, T, n, n] or NULL } */
  const void *grad_x_post;   /* bf16 [T, n, D] or NULL */
  void *grad_x;              /* bf16 [T, n, D], written */
  float *grad_phi;           /* [R, n*D], written */
  float *grad_alpha;         /* [3], written */
  float *grad_bias;          /* [R], written */
  float *grad_gamma;         /* [n, D], written; required iff gamma is given */
  void *workspace;           /* device scratch, mhc_pre_backward_workspace_size bytes */
  size_t workspace_bytes;
} mhc_pre_bwd_args;

/* First phase: device scratch bytes the backward needs for T tokens (0 for
 * T == 0).  The first 4 bytes hold the device error word that
 * mhc_pre_status reads.  MHC_ERR_PARAM_INVALID for a handle outside the
 * scope above. */
MHC_API mhc_status_t mhc_pre_backward_workspace_size(mhc_pre_t h, int64_t T, size_t *bytes);

/* Second phase: validate, then enqueue five kernels on `stream` (a
 * cudaStream_t, NULL = legacy default): the phi . gamma planes, the row dot
 * products grad_h_in . x (stage 3.1), the per-token stage (3.2-3.5 and the
 * Sinkhorn backward), the contraction kernel (3.6-3.8 and the per-unit
 * partial sums of grad_phi) and the fixed-order reductions.  Asynchronous;
 * the inputs must stay valid until the stream
 * reaches the end of this call.  MHC_ERR_NULLPTR for a missing required
 * pointer, MHC_ERR_PARAM_INVALID for a shape, alignment, optional-group or
 * workspace-size problem, MHC_ERR_RUNTIME for a launch failure
 * (mhc_pre_last_error() says which).  Device waits are bounded: one that
 * gives up sets the error word and the kernels return; mhc_pre_status(h,
 * workspace, stream) reports it. */
MHC_API mhc_status_t mhc_pre_backward_run(mhc_pre_t h, const mhc_pre_bwd_args *a, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MHC_PRE_BACKWARD_H_ */
