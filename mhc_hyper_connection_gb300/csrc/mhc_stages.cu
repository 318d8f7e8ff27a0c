// mhc_stages.cu -- the composite route of the mHC pre-mapping: three
// separate launches instead of the fused kernel.
//
// "CANN HcPre 融合算子解析：mHC 结构前处理 custom.npu_hc_pre 与 npu_hc_pre_v2
// 实战指南" (功能说明与计算流程, 融合路由策略) splits the pre-processing into
// an RMS-reciprocal operator, the mixing projection, and a Sinkhorn operator
// that takes the mixes and the reciprocal; the fused operator is the fast
// path and the split one the fallback.  Here the split route is a debug aid:
// each stage can be checked on its own, and the route as a whole against
// the fused kernel.  Plain CUDA-core kernels:
//
//  * inv_rms: one warp per token, 16-byte loads, fp32 sum of squares.
//  * mixes:   mixes[t][r] = sum_k x[t][k] gamma[k] phi[r][k] (not scaled by
//             invRms), 64 tokens x all R rows per CTA, K in 64-column steps
//             staged in shared memory; each thread forms 2 tokens x 3 rows.
//  * sinkhorn: one warp per token: lane 0 forms the gates and the Sinkhorn
//             mix from the mixes and invRms, all lanes form y.
#include "mhc_ptx.cuh"

namespace mhc {
namespace {

template <bool F16>
__global__ void __launch_bounds__(256) stage_inv_rms_kernel(StageLaunch L) {
  using X = XType<F16>;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, nw = (gridDim.x * blockDim.x) >> 5;
  const int nv = L.n * L.D / 8;
  for (int t = gw; t < L.T; t += nw) {
    const uint4* row = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(L.x) + (size_t)t * L.n * L.D * 2);
    float acc = 0.0f;
    for (int v0 = lane; v0 < nv; v0 += 32 * 4) {
      uint4 q[4];
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (v0 + 32 * b < nv) q[b] = __ldg(row + v0 + 32 * b);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        if (v0 + 32 * b >= nv) continue;
        const typename X::T2* h2 = reinterpret_cast<const typename X::T2*>(&q[b]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = X::to_f2(h2[e]);
          acc = fmaf(f.x, f.x, acc);
          acc = fmaf(f.y, f.y, acc);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) L.inv_rms[t] = __frsqrt_rn(acc / (float)(L.n * L.D) + L.norm_eps);
  }
}

constexpr int kMixTok = 64, kMixK = 64, kMixRowsPerWarp = 3, kMixWarps = 8;   // 8 warps x 3 rows = 24

template <bool F16>
__global__ void __launch_bounds__(kMixWarps * 32) stage_mixes_kernel(StageLaunch L) {
  using X = XType<F16>;
  __shared__ float xs[kMixTok][kMixK + 1];         // x . gamma, padded rows (no bank conflicts)
  __shared__ float ps[kMixRowsPerWarp * kMixWarps][kMixK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = L.n * L.D;
  const int t0 = blockIdx.x * kMixTok;
  for (int r0 = 0; r0 < L.R; r0 += kMixRowsPerWarp * kMixWarps) {
    float acc[2][kMixRowsPerWarp] = {};
    for (int k0 = 0; k0 < K; k0 += kMixK) {
      __syncthreads();
      // stage x . gamma [64 tokens][64 columns] and phi [24 rows][64 columns]
      for (int e = threadIdx.x; e < kMixTok * kMixK / 2; e += blockDim.x) {
        const int tt = e / (kMixK / 2), kk = 2 * (e % (kMixK / 2));
        float2 f = make_float2(0.0f, 0.0f);
        if (t0 + tt < L.T && k0 + kk < K) {
          const typename X::T2 v = *reinterpret_cast<const typename X::T2*>(
              static_cast<const uint8_t*>(L.x) + ((size_t)(t0 + tt) * K + k0 + kk) * 2);
          f = X::to_f2(v);
          if (L.gamma) {
            f.x *= __ldg(L.gamma + k0 + kk);
            f.y *= __ldg(L.gamma + k0 + kk + 1);
          }
        }
        xs[tt][kk] = f.x;
        xs[tt][kk + 1] = f.y;
      }
      for (int e = threadIdx.x; e < kMixRowsPerWarp * kMixWarps * kMixK; e += blockDim.x) {
        const int rr = e / kMixK, kk = e % kMixK;
        ps[rr][kk] = (r0 + rr < L.R && k0 + kk < K) ? __ldg(L.phi + (size_t)(r0 + rr) * K + k0 + kk) : 0.0f;
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < kMixK; ++kk) {
        const float xa = xs[lane][kk], xb = xs[lane + 32][kk];
#pragma unroll
        for (int j = 0; j < kMixRowsPerWarp; ++j) {
          const float pv = ps[warp * kMixRowsPerWarp + j][kk];
          acc[0][j] = fmaf(xa, pv, acc[0][j]);
          acc[1][j] = fmaf(xb, pv, acc[1][j]);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = t0 + lane + 32 * h;
#pragma unroll
      for (int j = 0; j < kMixRowsPerWarp; ++j) {
        const int r = r0 + warp * kMixRowsPerWarp + j;
        if (t < L.T && r < L.R) L.mixes[(size_t)t * L.R + r] = acc[h][j];
      }
    }
  }
}

template <int NS, int RR, bool F16>
__global__ void __launch_bounds__(256) stage_sinkhorn_kernel(EpiParams ep, const void* x, const float* mixes,
                                                             const float* inv_rms) {
  using X = XType<F16>;
  constexpr bool kThree = (RR == NS * NS + 2 * NS);
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, nw = (gridDim.x * blockDim.x) >> 5;
  const int nvd = ep.D / 8;                        // 16-byte vectors per stream row
  for (int t = gw; t < ep.T; t += nw) {
    float coef[NS] = {};
    if (lane == 0) {
      float mix[RR];
#pragma unroll
      for (int r = 0; r < RR; ++r) mix[r] = __ldg(mixes + (size_t)t * RR + r);
      const float ir = __ldg(inv_rms + t);
      token_gates_r<NS, RR>(ep, t, mix, ir, true, coef);
      float H[NS * NS];
      residual_logits<NS, RR>(ep, mix, ir, H);
      token_sinkhorn<NS, kThree>(ep, t, H, true);
    }
#pragma unroll
    for (int i = 0; i < NS; ++i) coef[i] = __shfl_sync(0xffffffffu, coef[i], 0);
    const uint8_t* xr = static_cast<const uint8_t*>(x) + (size_t)t * NS * ep.D * 2;
    uint8_t* yr = reinterpret_cast<uint8_t*>(ep.y) + (size_t)t * ep.D * 2;
    for (int v = lane; v < nvd; v += 32) {
      float a[8] = {};
#pragma unroll
      for (int i = 0; i < NS; ++i) {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(xr + (size_t)i * ep.D * 2) + v);
        const typename X::T2* h2 = reinterpret_cast<const typename X::T2*>(&q);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = X::to_f2(h2[e]);
          a[2 * e] = fmaf(coef[i], f.x, a[2 * e]);
          a[2 * e + 1] = fmaf(coef[i], f.y, a[2 * e + 1]);
        }
      }
      uint4 o;
      typename X::T2* ob = reinterpret_cast<typename X::T2*>(&o);
#pragma unroll
      for (int e = 0; e < 4; ++e) ob[e] = X::from_f2(a[2 * e], a[2 * e + 1]);
      reinterpret_cast<uint4*>(yr)[v] = o;
    }
  }
}

int grid_for(const void* kernel, int threads, long long work_warps) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0);
  long long g = (long long)sms * (per_sm > 0 ? per_sm : 1);
  const long long need = (work_warps * 32 + threads - 1) / threads;
  if (g > need) g = need;
  return (int)(g > 0 ? g : 1);
}

}  // namespace

cudaError_t launch_stage_inv_rms(const StageLaunch& L, cudaStream_t s) {
  const void* k = L.fp16 ? reinterpret_cast<const void*>(&stage_inv_rms_kernel<true>)
                         : reinterpret_cast<const void*>(&stage_inv_rms_kernel<false>);
  const int grid = grid_for(k, 256, L.T);
  if (L.fp16) stage_inv_rms_kernel<true><<<grid, 256, 0, s>>>(L);
  else stage_inv_rms_kernel<false><<<grid, 256, 0, s>>>(L);
  return cudaGetLastError();
}

cudaError_t launch_stage_mixes(const StageLaunch& L, cudaStream_t s) {
  const int grid = (L.T + kMixTok - 1) / kMixTok;
  if (L.fp16) stage_mixes_kernel<true><<<grid, kMixWarps * 32, 0, s>>>(L);
  else stage_mixes_kernel<false><<<grid, kMixWarps * 32, 0, s>>>(L);
  return cudaGetLastError();
}

cudaError_t launch_stage_sinkhorn(const EpiParams& ep, const void* x, const float* mixes, const float* inv_rms,
                                  int fp16, cudaStream_t s) {
  const void* k = nullptr;
#define MHC_SK(NS_, RR_)                                                                         \
  if (ep.n == NS_ && ep.R == RR_)                                                                \
    k = fp16 ? reinterpret_cast<const void*>(&stage_sinkhorn_kernel<NS_, RR_, true>)             \
             : reinterpret_cast<const void*>(&stage_sinkhorn_kernel<NS_, RR_, false>);
  MHC_SK(4, 24) MHC_SK(4, 8) MHC_SK(6, 48) MHC_SK(6, 12) MHC_SK(8, 80) MHC_SK(8, 16)
#undef MHC_SK
  if (!k) return cudaErrorInvalidValue;
  const int grid = grid_for(k, 256, ep.T);
  EpiParams p = ep;
  void* args[] = {&p, const_cast<void**>(&x), const_cast<float**>(&mixes), const_cast<float**>(&inv_rms)};
  return cudaLaunchKernel(k, dim3(grid), dim3(256), args, 0, s);
}

}  // namespace mhc
