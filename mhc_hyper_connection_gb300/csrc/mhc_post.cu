// mhc_post.cu -- the mHC post-mapping (hc_post) on sm_103a.
//
// What is computed follows "CANN HcPre 融合算子解析：mHC 结构前处理
// custom.npu_hc_pre 与 npu_hc_pre_v2 实战指南" (mHC section, hc_post):
//     out[t][j][d] = post[t][j] * x[t][d] + sum_i comb[t][i][j] * residual[t][i][d]
// with the streams mixed by comb (the printed reduction axis would only
// scale each stream by its row sum).
//
// A pure streaming op: per token it reads 2D + 2nD bytes and writes 2nD,
// against (n + n^2) coefficients.  One warp takes a token at a time (grid
// stride over tokens, no block-wide barrier); each lane forms all n outputs
// of a few 16-byte column vectors, issuing all their n + 1 loads each before
// any arithmetic; fp32 accumulation, RN-even bf16 rounding.  Loads of x and
// residual are marked evict-first (read once), as are the stores.
#include "mhc_ptx.cuh"

namespace mhc {
namespace {

constexpr int kPostThreads = 256;

// One warp per token (grid stride over tokens, no block-wide barrier): each
// lane loads the token's n + n^2 coefficients through the read-only cache
// (the same addresses across the warp), then forms all n outputs of kV
// 16-byte column vectors per pass with all their loads in flight.
template <int NS>
__global__ void __launch_bounds__(kPostThreads)
    mhc_post_kernel(int T, int D, const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ res,
                    const float* __restrict__ post, const float* __restrict__ comb, __nv_bfloat16* __restrict__ out) {
  constexpr int kV = NS <= 4 ? 4 : 2;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * kPostThreads + threadIdx.x) >> 5, nw = (gridDim.x * kPostThreads) >> 5;
  const int nv = D >> 3;                      // 16-byte vectors per row
  const uint64_t once = policy_evict_first();
  for (int t = gw; t < T; t += nw) {
    float pc[NS], cm[NS * NS];
#pragma unroll
    for (int j = 0; j < NS; ++j) pc[j] = __ldg(post + (size_t)t * NS + j);
#pragma unroll
    for (int e = 0; e < NS * NS; ++e) cm[e] = __ldg(comb + (size_t)t * NS * NS + e);
    const __nv_bfloat16* xt = x + (size_t)t * D;
    const __nv_bfloat16* rt = res + (size_t)t * NS * D;
    __nv_bfloat16* ot = out + (size_t)t * NS * D;
    for (int v0 = lane; v0 < nv; v0 += 32 * kV) {
      uint4 xv[kV], rv[kV][NS];
#pragma unroll
      for (int q = 0; q < kV; ++q) {
        const int v = v0 + q * 32;
        if (v < nv) {
          xv[q] = ld_global_v4_hint(xt + (size_t)v * 8, once);
#pragma unroll
          for (int i = 0; i < NS; ++i) rv[q][i] = ld_global_v4_hint(rt + (size_t)i * D + (size_t)v * 8, once);
        }
      }
#pragma unroll
      for (int q = 0; q < kV; ++q) {
        const int v = v0 + q * 32;
        if (v >= nv) continue;
#pragma unroll
        for (int j = 0; j < NS; ++j) {
          float acc[8];
          const __nv_bfloat162* hx = reinterpret_cast<const __nv_bfloat162*>(&xv[q]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(hx[e]);
            acc[2 * e] = pc[j] * f.x;
            acc[2 * e + 1] = pc[j] * f.y;
          }
#pragma unroll
          for (int i = 0; i < NS; ++i) {
            const float c = cm[i * NS + j];
            const __nv_bfloat162* hr = reinterpret_cast<const __nv_bfloat162*>(&rv[q][i]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(hr[e]);
              acc[2 * e] = fmaf(c, f.x, acc[2 * e]);
              acc[2 * e + 1] = fmaf(c, f.y, acc[2 * e + 1]);
            }
          }
          uint4 o;
          __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
          for (int e = 0; e < 4; ++e) ob[e] = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
          st_global_v4_hint(ot + (size_t)j * D + (size_t)v * 8, o, once);
        }
      }
    }
  }
}

template <int NS>
cudaError_t launch_ns(const PostLaunch& L, cudaStream_t s) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mhc_post_kernel<NS>, kPostThreads, 0)) !=
      cudaSuccess)
    return e;
  long long grid = (long long)sms * (per_sm > 0 ? per_sm : 1);
  const long long need = (L.T * 32 + kPostThreads - 1) / kPostThreads;   // one warp per token
  if (grid > need) grid = need;
  mhc_post_kernel<NS><<<(int)grid, kPostThreads, 0, s>>>(
      (int)L.T, (int)L.D, static_cast<const __nv_bfloat16*>(L.x), static_cast<const __nv_bfloat16*>(L.residual),
      L.post, L.comb, static_cast<__nv_bfloat16*>(L.out));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_post(const PostLaunch& L, cudaStream_t s) {
  switch (L.n) {
    case 1: return launch_ns<1>(L, s);
    case 2: return launch_ns<2>(L, s);
    case 3: return launch_ns<3>(L, s);
    case 4: return launch_ns<4>(L, s);
    case 5: return launch_ns<5>(L, s);
    case 6: return launch_ns<6>(L, s);
    case 7: return launch_ns<7>(L, s);
    case 8: return launch_ns<8>(L, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mhc
