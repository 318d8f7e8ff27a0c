// mhc_pre_aux.cu -- the phi-plane preparation kernel and the CUDA-core
// forward used for small token counts and as the diagnostic variant.
//
// Precision planes.  The projection runs on bf16 tensor cores with x (bf16,
// exact) as one operand and phi' = phi (.) gamma split into bf16 planes as the
// other: phi' = hi + mid + lo exactly (three planes, 24 significant bits,
// "fp32" mode), or phi' truncated toward zero to 11 significant bits and split
// hi + lo exactly (two planes, the pages' HF32 mode -- "CANN HcPre 融合算子解析"
// 精度验证, to_hf32; "aclnnMhcPreV2 算子接口全解析" §二 opImplMode).  Each
// bf16 x bf16 product is exact in fp32, so the only rounding left is the fp32
// accumulation.
#include "mhc_common.cuh"

namespace mhc {

__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

__global__ void __launch_bounds__(256) prepare_planes_kernel(PlaneParams pp) {
  if (blockIdx.x == 0 && threadIdx.x < kHdrWords && pp.err_word) pp.err_word[threadIdx.x] = 0u;
  const long long total = (long long)pp.nch * pp.n * pp.RB * 64;
  const int K = pp.n * pp.D;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    // Element idx of the swizzled image: block (chunk j, stream i), row r,
    // stored 16-byte piece e >> 3, which holds the row's logical piece
    // (e >> 3) ^ (r & 7).
    const int e = (int)(idx & 63);
    const long long brow = idx >> 6;
    const int r = (int)(brow % pp.RB);
    const long long blk = brow / pp.RB;
    const int i = (int)(blk % pp.n);
    const int j = (int)(blk / pp.n);
    const int d = j * 64 + ((((e >> 3) ^ (r & 7)) << 3) | (e & 7));
    const int plane = r / pp.R;
    const int rr = r - plane * pp.R;
    float out = 0.0f;
    if (plane < pp.P && d < pp.D) {
      const int k = i * pp.D + d;
      float v = __ldg(pp.phi + (size_t)rr * K + k);
      if (pp.gamma) v = v * __ldg(pp.gamma + k);
      if (pp.tf32) v = __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
      const float hi = bf16_round(v);
      const float rem = v - hi;           // exact: the rounding error of hi
      if (plane == 0) {
        out = hi;
      } else {
        const float mid = bf16_round(rem);
        out = (plane == 1) ? mid : bf16_round(rem - mid);   // rem - mid exact
      }
    }
    pp.planes[idx] = __float2bfloat16_rn(out);  // exact: out already bf16
  }
}

cudaError_t launch_prepare_planes(const PlaneParams& pp, cudaStream_t s) {
  const long long total = (long long)pp.nch * pp.n * pp.RB * 64;
  int blocks = (int)((total + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  prepare_planes_kernel<<<blocks, 256, 0, s>>>(pp);
  return cudaGetLastError();
}

}  // namespace mhc
