// mhc_common.cuh -- shared device code and launch plumbing of the sm_103a
// mHC pre-mapping forward library.
//
// The per-token epilogue below follows "CANN ops-transformer 中 aclnnMhcPreV2
// 算子接口全解析" §三 (scale by invRms, split pre/post/res, sigmoid gates,
// affine residual logits) and "CANN ops-transformer 算子详解：aclnnMhcPreSinkhorn
// 接口与 MhcPreSinkhorn 实现剖析" §3.2 (Sinkhorn: row softmax + eps, a column
// step, then (row, column) x (numIters - 1), each dividing by sum + eps).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mhc {

// Device error word bits (written into the first 4 bytes of the workspace).
enum : uint32_t {
  kErrWaitTimeout = 1u << 0,   // an mbarrier wait gave up
  kErrClusterWait = 1u << 1,   // a cluster exchange wait gave up
};

// Workspace layout: [0, 256) header (error word at 0), then the phi planes.
constexpr size_t kWsHeader = 256;

struct EpiParams {
  int T;
  int n, D, R, alpha_len, num_iters;
  float norm_eps, hc_eps;
  const float* bias;           // [R]
  const float* pre_mix;        // [T, n] or null
  __nv_bfloat16* y;            // [T, D]
  float* h_post;               // [T, n]
  float* h_res;                // [T, n, n] or null
  float* h_pre;                // [T, n] or null
  float* inv_rms;              // [T] or null
  float* h_mix;                // [T, R] or null
  float* sum_out;              // [2I, T, n] or null
  float* norm_out;             // [2I, T, n, n] or null
  const float* alpha;          // device alpha (read by kernels)
};

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + expf(-z)); }

// Gates and Sinkhorn for one token held by one thread.  mix[RR] is the
// projection before the RMS scale (hMix), ssq the sum of squares over the
// n*D elements.  Writes every per-token output when `write` is set and fills
// coef[NS] with the weights of y (pre_mix row or hPre).  RR = NS*NS + 2*NS
// selects the three-gate form, RR = 2*NS the two-gate form (no Sinkhorn).
template <int NS, int RR>
__device__ __forceinline__ void token_epilogue(const EpiParams& p, int t, const float (&mix)[RR],
                                               float ssq, bool write, float (&coef)[NS]) {
  constexpr int NN = NS * NS;
  constexpr bool kThree = (RR == NN + 2 * NS);
  static_assert(kThree || RR == 2 * NS, "R must be n*n+2n or 2n");
  const float K = (float)(NS * p.D);
  const float inv_rms = 1.0f / sqrtf(ssq / K + p.norm_eps);
  const float hc_eps = p.hc_eps;
  const float a0 = __ldg(p.alpha), a1 = __ldg(p.alpha + 1);

  if (write) {
    if (p.inv_rms) p.inv_rms[t] = inv_rms;
    if (p.h_mix) {
#pragma unroll
      for (int r = 0; r < RR; ++r) p.h_mix[(size_t)t * RR + r] = mix[r];
    }
  }
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    float pre = sigmoidf_(a0 * (mix[i] * inv_rms) + __ldg(p.bias + i)) + hc_eps;
    float post = 2.0f * sigmoidf_(a1 * (mix[NS + i] * inv_rms) + __ldg(p.bias + NS + i));
    if (!kThree) post += hc_eps;
    coef[i] = pre;
    if (write) {
      p.h_post[(size_t)t * NS + i] = post;
      if (p.h_pre) p.h_pre[(size_t)t * NS + i] = pre;
    }
  }
  if (p.pre_mix) {
#pragma unroll
    for (int i = 0; i < NS; ++i) coef[i] = __ldg(p.pre_mix + (size_t)t * NS + i);
  }

  if constexpr (!kThree) {
    if (write && p.h_res) {
#pragma unroll
      for (int e = 0; e < NN; ++e) p.h_res[(size_t)t * NN + e] = 0.0f;
    }
    return;
  } else {
    const float a2 = __ldg(p.alpha + 2);
    float P[NN];
#pragma unroll
    for (int e = 0; e < NN; ++e)
      P[e] = a2 * (mix[2 * NS + e] * inv_rms) + __ldg(p.bias + 2 * NS + e);

    const size_t Tn = (size_t)p.T * NS, Tnn = (size_t)p.T * NN;
    const bool wb = write && (p.sum_out != nullptr);
    // Step 0: softmax over each row (row maximum subtracted), then + eps.
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      float m = P[i * NS];
#pragma unroll
      for (int j = 1; j < NS; ++j) m = fmaxf(m, P[i * NS + j]);
      float s = 0.0f;
#pragma unroll
      for (int j = 0; j < NS; ++j) {
        P[i * NS + j] = expf(P[i * NS + j] - m);
        s += P[i * NS + j];
      }
      const float rs = 1.0f / s;
#pragma unroll
      for (int j = 0; j < NS; ++j) P[i * NS + j] = fmaf(P[i * NS + j], rs, hc_eps);
      if (wb) p.sum_out[(size_t)t * NS + i] = s;
    }
    if (wb) {
#pragma unroll
      for (int e = 0; e < NN; ++e) p.norm_out[(size_t)t * NN + e] = P[e];
    }
    // Steps 1 .. 2I-1: odd steps divide columns, even steps rows, by sum + eps.
    const int steps = 2 * p.num_iters;
    for (int k = 1; k < steps; ++k) {
      if (k & 1) {
#pragma unroll
        for (int j = 0; j < NS; ++j) {
          float s = 0.0f;
#pragma unroll
          for (int i = 0; i < NS; ++i) s += P[i * NS + j];
          s += hc_eps;
          const float rs = 1.0f / s;
#pragma unroll
          for (int i = 0; i < NS; ++i) P[i * NS + j] *= rs;
          if (wb) p.sum_out[k * Tn + (size_t)t * NS + j] = s;
        }
      } else {
#pragma unroll
        for (int i = 0; i < NS; ++i) {
          float s = 0.0f;
#pragma unroll
          for (int j = 0; j < NS; ++j) s += P[i * NS + j];
          s += hc_eps;
          const float rs = 1.0f / s;
#pragma unroll
          for (int j = 0; j < NS; ++j) P[i * NS + j] *= rs;
          if (wb) p.sum_out[k * Tn + (size_t)t * NS + i] = s;
        }
      }
      if (wb) {
#pragma unroll
        for (int e = 0; e < NN; ++e) p.norm_out[k * Tnn + (size_t)t * NN + e] = P[e];
      }
    }
    if (write && p.h_res) {
#pragma unroll
      for (int e = 0; e < NN; ++e) p.h_res[(size_t)t * NN + e] = P[e];
    }
  }
}

// y[t, d0 .. d0+8) = bf16(sum_i coef[i] * x[t, i, d0 .. d0+8)), one 16-byte
// vector per stream, accumulated in fp32 in stream order.
template <int NS>
__device__ __forceinline__ void weighted_sum8(const __nv_bfloat16* __restrict__ x_tok, int D, int d0,
                                              const float* coef, __nv_bfloat16* __restrict__ y_dst) {
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    uint4 v = __ldg(reinterpret_cast<const uint4*>(x_tok + (size_t)i * D + d0));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float2 f = __bfloat1622float2(h[q]);
      acc[2 * q] = fmaf(coef[i], f.x, acc[2 * q]);
      acc[2 * q + 1] = fmaf(coef[i], f.y, acc[2 * q + 1]);
    }
  }
  uint4 out;
  __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(&out);
#pragma unroll
  for (int q = 0; q < 4; ++q) o[q] = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
  *reinterpret_cast<uint4*>(y_dst + d0) = out;
}

// ---------------------------------------------------------------------------
// Host-side launch descriptions shared by the API translation unit and the
// kernel translation units.
// ---------------------------------------------------------------------------
struct PlaneParams {
  const float* phi;        // [R, K]
  const float* gamma;      // [K] or null
  __nv_bfloat16* planes;   // [NP, K]
  int R, K, NP, P;         // P = 3 (fp32) or 2 (tf32)
  int tf32;
  uint32_t* err_word;
};

cudaError_t launch_prepare_planes(const PlaneParams& pp, cudaStream_t s);

struct TcLaunch {
  EpiParams epi;
  const void* x;           // bf16 [T, n, D] (for the y pass)
  CUtensorMap tmap_x;      // 3-D: (D, n, T), box (64, 1, 128), 128B swizzle
  CUtensorMap tmap_w;      // 3-D: (D, n, NP), box (64, 1, NP), 128B swizzle
  int NP, P;
  int cluster;             // CTAs per token tile (split over d-chunks)
  int grid;                // CTAs (multiple of cluster)
  int stages;
  size_t smem_bytes;
  uint32_t* err_word;
};

// Resolved by the kernel translation unit for the given (n, R, P).
cudaError_t launch_tc_forward(const TcLaunch& L, cudaStream_t s);
// Largest dynamic shared memory per CTA the kernel for this shape may use and
// the number of clusters of the given size that fit at once (0: unsupported).
cudaError_t tc_forward_occupancy(int n, int R, int P, size_t smem_bytes, int cluster,
                                 int* max_clusters);

constexpr int kTileM = 128;        // tokens per MMA tile (TMEM lanes)
constexpr int kChunkK = 64;        // bf16 elements per 128-byte swizzle row
constexpr int kThreads = 256;      // 8 warps: TMA, MMA, 2 x sum-of-squares, 4 x epilogue

}  // namespace mhc
