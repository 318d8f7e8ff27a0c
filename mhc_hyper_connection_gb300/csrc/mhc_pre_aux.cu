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

// Plane `plane` of v (see the file comment), as the float value it stores.
__device__ __forceinline__ float plane_value(const PlaneParams& pp, float v, int plane) {
  if (pp.tf32) v = __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
  if (pp.fp16) {
    // v = h0 + h1 2^-11 + h2 2^-22, each h an fp16 value (11 significant
    // bits each, so exact for an fp32 v inside fp16's range)
    const float h0 = __half2float(__float2half_rn(v));
    if (plane == 0) return h0;
    const float r1 = v - h0;                                   // exact
    const float h1 = __half2float(__float2half_rn(r1 * 2048.0f));
    return plane == 1 ? h1 : __half2float(__float2half_rn((r1 - h1 * (1.0f / 2048.0f)) * 4194304.0f));
  }
  const float hi = bf16_round(v);
  if (plane == 0) return hi;
  const float rem = v - hi;                                    // exact: the rounding error of hi
  const float mid = bf16_round(rem);
  return plane == 1 ? mid : bf16_round(rem - mid);             // rem - mid exact
}

// One thread per stored 16-byte piece of the swizzled image: block (chunk j,
// stream i), row r, stored piece e, which holds the row's logical piece
// e ^ (r & 7) -- eight consecutive columns d0 .. d0+7 (D is a multiple of
// 16, so a piece is wholly inside or wholly past D).
__global__ void __launch_bounds__(256) prepare_planes_kernel(PlaneParams pp) {
  // bf16 planes: this kernel zeroes the header.  fp16 planes: the header was
  // zeroed before the launch, since blocks here may raise the range error.
  if (!pp.fp16 && blockIdx.x == 0 && threadIdx.x < kHdrWords && pp.err_word) pp.err_word[threadIdx.x] = 0u;
  const long long pieces = (long long)pp.nch * pp.n * pp.RB * 8;
  const int K = pp.n * pp.D;
  for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < pieces;
       q += (long long)gridDim.x * blockDim.x) {
    const int e = (int)(q & 7);
    const long long brow = q >> 3;
    const int r = (int)(brow % pp.RB);
    const long long blk = brow / pp.RB;
    const int i = (int)(blk % pp.n);
    const int j = (int)(blk / pp.n);
    const int d0 = j * 64 + ((e ^ (r & 7)) << 3);
    const int plane = r / pp.R;
    const int rr = r - plane * pp.R;
    float out[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) out[c] = 0.0f;
    if (plane < pp.P && d0 < pp.D) {
      const int k = i * pp.D + d0;
      const float4* src = reinterpret_cast<const float4*>(pp.phi + (size_t)rr * K + k);
      float v[8];
      if (pp.vec16) {                                  // phi and gamma 16-byte aligned
        const float4 a = __ldg(src), b = __ldg(src + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) v[c] = __ldg(reinterpret_cast<const float*>(src) + c);
      }
      if (pp.gamma) {
#pragma unroll
        for (int c = 0; c < 8; ++c) v[c] *= __ldg(pp.gamma + k + c);
      }
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        if (pp.fp16 && plane == 0 && !(fabsf(v[c]) <= 65504.0f) && pp.err_word) atomicOr(pp.err_word, kErrPlaneRange);
        out[c] = plane_value(pp, v[c], plane);
      }
    }
    uint4 o;
    if (pp.fp16) {
      __half2* h = reinterpret_cast<__half2*>(&o);
#pragma unroll
      for (int c = 0; c < 4; ++c) h[c] = __floats2half2_rn(out[2 * c], out[2 * c + 1]);   // exact
    } else {
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int c = 0; c < 4; ++c) h[c] = __floats2bfloat162_rn(out[2 * c], out[2 * c + 1]);   // exact
    }
    reinterpret_cast<uint4*>(pp.planes)[q] = o;
  }
}

cudaError_t launch_prepare_planes(const PlaneParams& pp, cudaStream_t s) {
  if (pp.fp16 && pp.err_word) {
    const cudaError_t e = cudaMemsetAsync(pp.err_word, 0, kHdrWords * sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
  }
  const long long total = (long long)pp.nch * pp.n * pp.RB * 8;   // 16-byte pieces
  int blocks = (int)((total + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  prepare_planes_kernel<<<blocks, 256, 0, s>>>(pp);
  return cudaGetLastError();
}

}  // namespace mhc
