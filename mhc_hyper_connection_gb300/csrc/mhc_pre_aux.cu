// mhc_pre_aux.cu -- the phi-plane preparation kernel of the forward.
//
// Precision planes.  The projection runs on the tensor cores with x (exact)
// as one operand and phi' = phi (.) gamma split into planes of x's type as
// the other.  bf16 x: phi' = hi + mid + lo exactly (three bf16 planes, 24
// significant bits, "fp32" mode), or phi' truncated toward zero to 11
// significant bits and split hi + lo exactly (two planes, the pages' HF32
// mode -- "CANN HcPre 融合算子解析" 精度验证, to_hf32; "aclnnMhcPreV2 算子接口
// 全解析" §二 opImplMode).  fp16 x (an MMA takes one operand type): fp16
// planes, each scaled into fp16's range, phi' = h0 + h1 2^-11 + h2 2^-22.
// Every product of two planes' elements is exact in fp32, so the only
// rounding left is the fp32 accumulation.
#include "mhc_common.cuh"

namespace mhc {

__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

__global__ void __launch_bounds__(256) prepare_planes_kernel(PlaneParams pp) {
  // bf16 planes: this kernel zeroes the header.  fp16 planes: the header was
  // zeroed before the launch, since blocks here may raise the range error.
  if (!pp.fp16 && blockIdx.x == 0 && threadIdx.x < kHdrWords && pp.err_word) pp.err_word[threadIdx.x] = 0u;
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
      if (pp.fp16) {
        // v = h0 + h1 2^-11 + h2 2^-22, each h an fp16 value (11 significant
        // bits each, so exact for an fp32 v inside fp16's range)
        if (plane == 0 && !(fabsf(v) <= 65504.0f) && pp.err_word) atomicOr(pp.err_word, kErrPlaneRange);
        const float h0 = __half2float(__float2half_rn(v));
        const float r1 = v - h0;                                   // exact
        const float h1 = __half2float(__float2half_rn(r1 * 2048.0f));
        out = plane == 0 ? h0 : plane == 1 ? h1 : __half2float(__float2half_rn((r1 - h1 * (1.0f / 2048.0f)) * 4194304.0f));
      } else {
        const float hi = bf16_round(v);
        const float rem = v - hi;           // exact: the rounding error of hi
        if (plane == 0) {
          out = hi;
        } else {
          const float mid = bf16_round(rem);
          out = (plane == 1) ? mid : bf16_round(rem - mid);   // rem - mid exact
        }
      }
    }
    if (pp.fp16) reinterpret_cast<__half*>(pp.planes)[idx] = __float2half_rn(out);   // exact
    else pp.planes[idx] = __float2bfloat16_rn(out);  // exact: out already bf16
  }
}

cudaError_t launch_prepare_planes(const PlaneParams& pp, cudaStream_t s) {
  if (pp.fp16 && pp.err_word) {
    const cudaError_t e = cudaMemsetAsync(pp.err_word, 0, kHdrWords * sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
  }
  const long long total = (long long)pp.nch * pp.n * pp.RB * 64;
  int blocks = (int)((total + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  prepare_planes_kernel<<<blocks, 256, 0, s>>>(pp);
  return cudaGetLastError();
}

}  // namespace mhc
