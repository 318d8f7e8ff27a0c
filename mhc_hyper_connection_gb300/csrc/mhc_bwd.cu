// mhc_bwd.cu -- the sm_103a backward of the mHC pre-mapping with Sinkhorn
// (n = 4, three gates).
//
// What is computed follows "CANN ops-transformer 算子解析：MhcPreBackward 反向
// 梯度算子实现与 aclnn 调用指南" §三 3.1-3.8 (the outputs are the gradients of
// the forward, §一), with the Sinkhorn variant's saved sums and matrices of
// "aclnnMhcPreSinkhorn 接口与 MhcPreSinkhorn 实现剖析" §3.2 carried back first.
// How it is laid out on the GPU is this file's own design:
//
//  * Row dot (one CTA per SM): H_pre_grad = grad_h_in . x over the whole
//    row (the only full-row reduction of the backward), whole token rows
//    brought in by bulk copy.
//  * Token stage (one half-warp per token): the Sinkhorn backward on 16
//    lanes from the saved steps, the gate backward, and
//    G = H_mix_grad with the RMS factor c = -inv_rms_grad invRms^3 / (nD).
//    G goes out as exact bf16 planes in a per-64-token tile record laid out
//    for the tensor core, next to hPre and c of the tile's tokens.
//  * Main kernel (one CTA per SM): the work units are (64-column slab of all
//    four streams, one of nq contiguous chunks of the 64-token tiles); CTA b
//    takes units b, b + grid, ...  With grid a multiple of nq, the CTAs that
//    share b mod nq sweep the same tokens at the same time over different
//    slabs, so together they read whole rows of x (DRAM-page friendly).
//    Per tile, TMA brings x [4][64 tokens][64], grad_h_in
//    [64 tokens][64] and the tile record; tcgen05 forms
//      - G phi' (phi' = phi . gamma in planes, resident per slab; in fp32
//        mode planes 0 and 1 are read from tensor memory) as D1[k][token]
//        in TMEM (M = 128 columns k of two streams, N = 64 tokens, K = the
//        24 gate rows per plane product), then
//      - x^T G accumulated in TMEM across the run's tiles of one slab
//        (M = 128 columns k, N = P * 32 plane rows, K = 16 tokens per step).
//    Sixteen epilogue warps (32 tokens of one M-group each) form
//    grad_x = hPre grad_h_in + D1 + c x (+ grad_x_post) in fp32, round it
//    to bf16 and store it from registers; the slot goes back to the
//    producer once they and the tile's MMAs are done with it.  At the end
//    of a unit eight of them write x^T G, summed over the planes, to the
//    unit's partial buffer.
//  * Final kernel: grad_phi = gamma . sum(x^T G), grad_gamma = sum_r phi .
//    sum(x^T G), summing a slab's units in chunk order; grad_alpha and
//    grad_bias from the token stage's per-warp partials in warp order.
//  * Every wait is bounded; a wait that gives up sets the error word and the
//    kernel winds down.
#include "mhc_ptx.cuh"

namespace mhc {
namespace {

__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// Plane `plane` of the exact split v = hi + mid + lo (three planes), or of
// v truncated to 10 mantissa bits and split hi + lo (two planes).
__device__ __forceinline__ float plane_part(float v, int plane, int tf32) {
  if (tf32) v = __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
  const float hi = bf16_round(v);
  if (plane == 0) return hi;
  const float rem = v - hi;               // exact
  const float mid = bf16_round(rem);
  if (plane == 1) return mid;
  return bf16_round(rem - mid);           // rem - mid exact
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Byte offset of element (row, col) (col < 64) in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return (uint32_t)(row * 128 + ((((col >> 3) ^ (row & 7)) << 4) | ((col & 7) << 1)));
}

// The backward's launches after the first are programmatic dependents of
// the one before (their launch and set-up overlap its tail): each kernel
// lets its dependent launch as soon as all of its own CTAs run, and waits
// for its predecessor's grid (complete, memory visible) before it reads
// anything.  Without the launch attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// =================================================================== planes
// One thread per stored 16-byte piece: eight consecutive columns of one
// plane row (D is a multiple of 64 here, so every piece is inside D).
__global__ void __launch_bounds__(256) bw_planes_kernel(BwPlaneParams pp) {
  pdl_trigger();
  if (blockIdx.x == 0 && threadIdx.x < kHdrWords && pp.hdr) pp.hdr[threadIdx.x] = 0u;
  const int rows = pp.P * kBwRp;                        // rows of one stream block
  const long long pieces = (long long)pp.nslab * kBwNS * rows * 8;
  const int K = kBwNS * pp.D;
  for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < pieces;
       q += (long long)gridDim.x * blockDim.x) {
    const int e = (int)(q & 7);
    const long long grow = q >> 3;
    const int rr = (int)(grow % rows);                  // row in the stream block
    const long long blk = grow / rows;
    const int i = (int)(blk % kBwNS);
    const int j = (int)(blk / kBwNS);
    const int plane = rr / kBwRp, r = rr % kBwRp;
    const int d0 = j * 64 + ((e ^ (rr & 7)) << 3);
    float out[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) out[c] = 0.0f;
    if (r < kBwR) {
      const int k = i * pp.D + d0;
      const float4* src = reinterpret_cast<const float4*>(pp.phi + (size_t)r * K + k);
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
      for (int c = 0; c < 8; ++c) out[c] = plane_part(v[c], plane, pp.tf32);
    }
    uint4 o;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int c = 0; c < 4; ++c) h[c] = __floats2bfloat162_rn(out[2 * c], out[2 * c + 1]);   // exact
    reinterpret_cast<uint4*>(pp.planes)[q] = o;
  }
}

// ================================================================== row dot
// H_pre_grad[t][i] = sum_d grad_h_in[t][d] x[t][i][d] (stage 3.1).  Token
// rows of x (n*D contiguous) and grad_h_in (D contiguous) arrive whole by
// bulk copy into a ring of shared-memory stages (tps tokens each); eight
// warps form the four dot products of each token, reduced in a fixed order.
constexpr int kRdWarps = 8;
constexpr int kRdThreads = (kRdWarps + 1) * 32;   // + one producer warp
constexpr int kRdMaxStages = 4;

struct RdTail {
  uint64_t full[kRdMaxStages], empty[kRdMaxStages];
  uint32_t abort;
  float red[2][kRdWarps][kBwNS];
};

__global__ void __launch_bounds__(kRdThreads, 1) bw_rowdot_kernel(BwRowdotParams p) {
  constexpr int NS = kBwNS;
  extern __shared__ __align__(128) uint8_t rd_smem[];
  const size_t xrow = (size_t)NS * p.D * 2, grow = (size_t)p.D * 2;
  const size_t stage_bytes = (size_t)p.tps * (xrow + grow);
  RdTail* tail = reinterpret_cast<RdTail*>(rd_smem + (size_t)p.stages * stage_bytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = (p.T + p.tps - 1) / p.tps;
  Ctl ctl{&tail->abort, p.err};
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&tail->full[s], 1);
      mbar_init(&tail->empty[s], kRdWarps);
    }
    tail->abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (warp == kRdWarps) {
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();
      int s = 0;
      uint32_t ph = 0;
      long long iss = 0;
      for (int gi = blockIdx.x; gi < ngroups; gi += gridDim.x) {
        const int t0 = gi * p.tps, cnt = min(p.tps, p.T - t0);
        if (!wait_bar<false>(&tail->empty[s], ph ^ 1u, ctl, kErrWaitTimeout)) break;
        uint8_t* st = rd_smem + (size_t)s * stage_bytes;
        mbar_expect_tx(&tail->full[s], (uint32_t)((size_t)cnt * (xrow + grow)));
        bulk_load_hint(st, p.x + (size_t)t0 * NS * p.D, (uint32_t)((size_t)cnt * xrow), &tail->full[s], keep);
        bulk_load_hint(st + (size_t)p.tps * xrow, p.g_in + (size_t)t0 * p.D, (uint32_t)((size_t)cnt * grow),
                       &tail->full[s], keep);
        ++iss;
        if (++s == p.stages) { s = 0; ph ^= 1u; }
      }
      for (long long q = 0; q < (iss < p.stages ? iss : p.stages); ++q) {
        if (--s < 0) { s = p.stages - 1; ph ^= 1u; }
        mbar_drain(&tail->full[s], ph);
      }
    }
    return;
  }
  const int nv = p.D >> 3;                 // 16-byte vectors per stream row
  int s = 0, par = 0;
  uint32_t ph = 0;
  for (int gi = blockIdx.x; gi < ngroups; gi += gridDim.x) {
    const int t0 = gi * p.tps, cnt = min(p.tps, p.T - t0);
    // all compute warps leave together (they meet at a named barrier below)
    if (!role_all<1, kRdWarps * 32>(wait_bar<false>(&tail->full[s], ph, ctl, kErrWaitTimeout))) break;
    const uint8_t* st = rd_smem + (size_t)s * stage_bytes;
    for (int k = 0; k < cnt; ++k, par ^= 1) {
      const uint4* xs = reinterpret_cast<const uint4*>(st + (size_t)k * xrow);
      const uint4* gs = reinterpret_cast<const uint4*>(st + (size_t)p.tps * xrow + (size_t)k * grow);
      float acc[NS] = {0.0f, 0.0f, 0.0f, 0.0f};
      for (int v = threadIdx.x; v < nv; v += kRdWarps * 32) {
        const uint4 gv = gs[v];
        const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
        for (int i = 0; i < NS; ++i) {
          const uint4 xv = xs[(size_t)i * nv + v];
          const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&xv);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 gf = __bfloat1622float2(g2[e]), xf = __bfloat1622float2(x2[e]);
            acc[i] = fmaf(gf.x, xf.x, acc[i]);
            acc[i] = fmaf(gf.y, xf.y, acc[i]);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < NS; ++i) acc[i] = warp_sum(acc[i]);
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < NS; ++i) tail->red[par][warp][i] = acc[i];
      }
      role_sync<1, kRdWarps * 32>();
      if (threadIdx.x < NS) {
        float tot = 0.0f;
#pragma unroll
        for (int w = 0; w < kRdWarps; ++w) tot += tail->red[par][w][threadIdx.x];
        p.hg[(size_t)(t0 + k) * NS + threadIdx.x] = tot;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tail->empty[s]);
    if (++s == p.stages) { s = 0; ph ^= 1u; }
  }
}

// =============================================================== token stage
constexpr int kSinkChunk = 20;   // saved Sinkhorn steps staged per round and token

// 16-byte global -> shared copy that bypasses the registers (completes at
// cp_async_wait_all of the issuing thread).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// One token per half-warp (two per warp, so twice the tokens in flight):
// lane hl = i*4 + j of the half holds the Sinkhorn element (i, j) and gate
// rows hl and hl + 16.  Both halves run every shuffle (all of them stay
// inside a half); a padding token of the last tile runs the same code on
// zeros and writes zero G planes.
__global__ void __launch_bounds__(kBwTokenWarps * 32) bw_token_kernel(BwTokenParams p) {
  constexpr int NS = kBwNS, R = kBwR, NN = NS * NS;
  static_assert(NN == 16 && R <= 32, "the half-warp layout is for n = 4");
  __shared__ __align__(16) float stage[kBwTokenWarps][2][kSinkChunk][NN + NS];
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, hl = lane & 15;
  const int gw = blockIdx.x * kBwTokenWarps + warp;
  const int nw = gridDim.x * kBwTokenWarps;
  const int Tpad = p.ntiles * kBwTile;
  const float a0 = __ldg(p.alpha), a1 = __ldg(p.alpha + 1), a2 = __ldg(p.alpha + 2);
  const float eps = p.hc_eps;
  const int rec_bytes = bw_tile_rec_bytes(p.P);
  const int r0 = hl, r1 = hl + 16;                      // this lane's gate rows
  float acc_b0 = 0.0f, acc_b1 = 0.0f, acc_a0 = 0.0f, acc_a1 = 0.0f;   // partial sums per row
  float (*st)[NN + NS] = stage[warp][half];

  for (int tb = 2 * gw; tb < Tpad; tb += 2 * nw) {      // warp-uniform (Tpad is a multiple of 64)
    const int t = tb + half;
    const bool valid = t < p.T;
    const int tv = valid ? t : 0;                       // a token that exists, for loads
    uint8_t* rec = p.tiles + (size_t)(t / kBwTile) * rec_bytes;
    const int col = t % kBwTile;
    float* scal = reinterpret_cast<float*>(rec + p.P * kBwPlaneBytes) + col * 2;
    // ---- 3.1: H_pre_grad[i], from the row-dot kernel
    const float4 hg4 = __ldg(reinterpret_cast<const float4*>(p.hg) + tv);
    const float hg[NS] = {hg4.x, hg4.y, hg4.z, hg4.w};
    const float ir = __ldg(p.inv_rms + tv);
    const float hm0 = __ldg(p.h_mix + (size_t)tv * R + r0);
    const float hm1 = r1 < R ? __ldg(p.h_mix + (size_t)tv * R + r1) : 0.0f;

    // ---- Sinkhorn backward (element (i, j) = lane hl of the half)
    float g = valid ? __ldg(p.g_res + (size_t)tv * NN + hl) : 0.0f;
    if (p.norm_out) {
      for (int kh = 2 * p.num_iters - 1; kh >= 1; kh -= kSinkChunk) {
        const int klo = max(1, kh - kSinkChunk + 1);
        const int cnt = kh - klo + 1;
        __syncwarp();
        // the chunk's saved matrices and sums of this half's token: with
        // 16-byte aligned tensors all of them at once as asynchronous copies
        // (four pieces of a step's matrix and one of its sums), else eight
        // loads in flight per lane (sums of a padding token read as 1)
        const int nm = cnt * NN, ntot = nm + cnt * NS;
        constexpr int kBatch = 8;
        if (p.saved16 && valid) {
          for (int q = hl; q < cnt * 5; q += 16) {
            const int s = q / 5, part = q - 5 * s;
            const float* src = part < 4 ? p.norm_out + ((size_t)(klo + s) * p.T + tv) * NN + part * 4
                                        : p.sum_out + ((size_t)(klo + s) * p.T + tv) * NS;
            cp_async16(&st[s][part * 4], src);
          }
          cp_async_wait_all();
        } else
        for (int e0 = hl; e0 < ntot; e0 += 16 * kBatch) {
          float v[kBatch];
#pragma unroll
          for (int j = 0; j < kBatch; ++j) {
            const int e = e0 + 16 * j;
            v[j] = 0.0f;
            if (e < nm) {
              if (valid) v[j] = __ldg(p.norm_out + ((size_t)(klo + e / NN) * p.T + tv) * NN + e % NN);
            } else if (e < ntot) {
              v[j] = valid ? __ldg(p.sum_out + ((size_t)(klo + (e - nm) / NS) * p.T + tv) * NS + (e - nm) % NS) : 1.0f;
            }
          }
#pragma unroll
          for (int j = 0; j < kBatch; ++j) {
            const int e = e0 + 16 * j;
            if (e < nm) st[e / NN][e % NN] = v[j];
            else if (e < ntot) st[(e - nm) / NS][NN + (e - nm) % NS] = v[j];
          }
        }
        __syncwarp();
        for (int k = kh; k >= klo; --k) {
          const float* row = st[k - klo];
          const float prod = g * row[hl];
          float dot, sv;
          if (k & 1) {            // column step: sum over i, divide by column sum j
            dot = prod + __shfl_xor_sync(0xffffffffu, prod, 4);
            dot += __shfl_xor_sync(0xffffffffu, dot, 8);
            sv = row[NN + (hl & 3)];
          } else {                // row step: sum over j, divide by row sum i
            dot = prod + __shfl_xor_sync(0xffffffffu, prod, 1);
            dot += __shfl_xor_sync(0xffffffffu, dot, 2);
            sv = row[NN + (hl >> 2)];
          }
          g = __fdividef(g - dot, sv);     // sv is a sum plus eps: >= eps, well inside the fast range
        }
      }
      // the row softmax (+ eps): S = normOut[0] - eps
      const float S = valid ? __ldg(p.norm_out + (size_t)tv * NN + hl) - eps : 0.0f;
      const float prod = g * S;
      float dot = prod + __shfl_xor_sync(0xffffffffu, prod, 1);
      dot += __shfl_xor_sync(0xffffffffu, dot, 2);
      g = S * (g - dot);
    }
    // res logit gradients of rows r0 (hl >= 8: element hl - 8) and r1 (element hl + 8)
    const float gres0 = __shfl_sync(0xffffffffu, g, (half << 4) + ((hl - 8) & 15));
    const float gres1 = __shfl_sync(0xffffffffu, g, (half << 4) + ((hl + 8) & 15));

    // ---- gates (3.2-3.4) of rows r0, r1
    float b0 = 0.0f, gt0 = 0.0f, b1 = 0.0f, gt1 = 0.0f;
    if (r0 < NS) {
      const float sg = __ldg(p.h_pre + (size_t)tv * NS + r0) - eps;
      float hh = hg[0];
#pragma unroll
      for (int i = 1; i < NS; ++i) hh = (r0 == i) ? hg[i] : hh;
      b0 = hh * sg * (1.0f - sg);
      gt0 = b0 * a0;
    } else if (r0 < 2 * NS) {
      const float hp = __ldg(p.h_post + (size_t)tv * NS + r0 - NS);
      b0 = __ldg(p.g_post + (size_t)tv * NS + r0 - NS) * hp * (1.0f - 0.5f * hp);
      gt0 = b0 * a1;
    } else {
      b0 = gres0;
      gt0 = b0 * a2;
    }
    if (r1 < R) {
      b1 = gres1;
      gt1 = b1 * a2;
    }
    if (!valid) b0 = gt0 = b1 = gt1 = 0.0f;
    acc_b0 += b0;
    acc_b1 += b1;
    acc_a0 += b0 * (hm0 * ir);
    acc_a1 += b1 * (hm1 * ir);
    // ---- 3.5: G = [alpha g] invRms; inv_rms_grad = sum [alpha g] hMix (over the half)
    float irg = gt0 * hm0 + gt1 * hm1;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) irg += __shfl_xor_sync(0xffffffffu, irg, o);
    const float G0 = gt0 * ir, G1 = gt1 * ir;
    const float c = valid ? -(irg * ir * ir * ir) / (float)(NS * p.D) : 0.0f;
    for (int pl = 0; pl < p.P; ++pl) {
      *reinterpret_cast<__nv_bfloat16*>(rec + pl * kBwPlaneBytes + swz(r0, col)) =
          __float2bfloat16_rn(plane_part(G0, pl, p.tf32));
      *reinterpret_cast<__nv_bfloat16*>(rec + pl * kBwPlaneBytes + swz(r1, col)) =
          __float2bfloat16_rn(plane_part(G1, pl, p.tf32));
    }
    // per stream i, per token: (hPre_i, RMS factor) -- [i][token] pairs
    if (hl < 2 * NS) {
      const float hp = valid ? __ldg(p.h_pre + (size_t)tv * NS + (hl >> 1)) : 0.0f;
      scal[(hl >> 1) * (2 * kBwTile) + (hl & 1)] = (hl & 1) ? c : hp;
    }
  }
  // ---- this warp's partial sums: [0, R) bias, R .. R+2 alpha by segment
  const float bs0 = acc_b0 + __shfl_xor_sync(0xffffffffu, acc_b0, 16);   // rows 0..15
  const float bs1 = acc_b1 + __shfl_xor_sync(0xffffffffu, acc_b1, 16);   // rows 16..31
  const float seg0 = warp_sum(hl < NS ? acc_a0 : 0.0f);
  const float seg1 = warp_sum((hl >= NS && hl < 2 * NS) ? acc_a0 : 0.0f);
  const float seg2 = warp_sum((hl >= 2 * NS ? acc_a0 : 0.0f) + acc_a1);
  const float hi_rows = __shfl_sync(0xffffffffu, bs1, lane & 15);
  float* out = p.partials + (size_t)gw * 32;
  float v = lane < 16 ? bs0 : (lane < R ? hi_rows : 0.0f);
  if (lane == R) v = seg0;
  if (lane == R + 1) v = seg1;
  if (lane == R + 2) v = seg2;
  out[lane] = v;
}

// ================================================================ main kernel
// Warps: 0 TMA producer, 1 MMA issuer (and TMEM owner), 2..17 epilogue.
// Epilogue warp e works on TMEM lane quarter (warp % 4), M-group (e >> 3)
// and token half ((e >> 2) & 1) of each tile.
constexpr int kWarpProd = 0, kWarpMma = 1, kWarpEpi0 = 2;
constexpr int kEpiWarps = 16;
constexpr int kMainThreads = (kWarpEpi0 + kEpiWarps) * 32;
constexpr int kMaxStages = 4;
constexpr int kXBytes = kBwNS * kBwTile * 128;    // x tile of all streams (32 KB)
constexpr int kGinBytes = kBwTile * 128;          // grad_h_in tile (8 KB)
constexpr int kGroups = kBwNS / 2;                // M = 128 columns = two streams
constexpr int kHalf = kBwTile / 2;                // tokens per epilogue warp
// Tiles of L2 prefetch ahead of the copy.  0: with grad_x stored from
// registers the kernel no longer waits on its loads, and prefetching 1 / 2
// / 3 / 4 tiles ahead measured 0.4 / 0.6 / 0.8 / 12% slower than none.
#ifndef MHC_BW_PREFETCH
#define MHC_BW_PREFETCH 0
#endif
constexpr int kPrefetch = MHC_BW_PREFETCH;

struct MainTail {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t a_full, a_free, at_full;
  uint64_t d1_full[2], d1_empty[2];
  uint64_t mt_full, mt_empty;
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t abort;
};
static_assert(sizeof(MainTail) <= kBwTailBytes, "barrier block outgrew its reservation");

// Plane products of G phi' as (G plane, phi' plane).  Three planes keep the
// six of combined order up to 2^-16 (hi.hi, hi.mid, mid.hi, hi.lo, lo.hi,
// mid.mid); two planes the first three (hi.hi, hi.lo, lo.hi).
__device__ __forceinline__ void product_planes(int q, int& gp, int& pp) {
  const int g3[6] = {0, 0, 1, 0, 2, 1}, p3[6] = {0, 1, 0, 2, 0, 1};
  gp = g3[q];
  pp = p3[q];
}

template <int P, bool kGxp>
__global__ void __launch_bounds__(kMainThreads, 1)
    bw_main_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_gin,
                   const __grid_constant__ CUtensorMap tmap_gxp, const __nv_bfloat16* __restrict__ planes,
                   const uint8_t* __restrict__ tiles, float* __restrict__ pieces, __nv_bfloat16* __restrict__ gx,
                   uint32_t* err, int T, int D, int ntiles, int nslab, int nq, int stages, WaitTest wt) {
  constexpr int kABlk = P * kBwPlaneBytes;            // one stream's block of the phi' slab
  constexpr int kABytes = kBwNS * kABlk;
  constexpr int kRec = bw_tile_rec_bytes(P);
  constexpr int kMtCols = bw_mt_cols(P);              // N of x^T G
  constexpr int kNQ = P == 3 ? 6 : 3;                 // plane products of G phi'
  constexpr int kMtCol0 = 2 * kGroups * kBwTile;      // after two D1 buffers
  // fp32 mode (three planes) reads phi' planes 0 and 1 from tensor memory
  // (five of the six plane products), which relieves the shared-memory
  // port that the epilogue and the other operands share; with two planes
  // (tf32 mode) the shared slab measured faster.
  constexpr bool kTmA = P == 3;
  constexpr int kAtCol0 = kMtCol0 + kGroups * kMtCols;  // phi' planes 0 and 1 as tensor-memory A operands
  constexpr int kAtCols = 2 * kBwRp / 2;              // two planes of 32 rows, two bf16 per column
  constexpr uint32_t kTmemCols = 512;
  constexpr int kStageBytes = bw_stage_bytes(P, kGxp);
  // stage layout: x | grad_x_post (optional) | grad_h_in | tile record
  constexpr int offGxp = kXBytes;
  constexpr int offGin = kXBytes * (kGxp ? 2 : 1);
  constexpr int offRec = offGin + kGinBytes;
  static_assert(kAtCol0 + kGroups * kAtCols <= (int)kTmemCols, "TMEM budget");

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sStage = smem + kABytes;
  MainTail* tail = reinterpret_cast<MainTail*>(sStage + (size_t)stages * kStageBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Work units u = slab * nq + chunk (chunk: a contiguous nq-th of the token
  // tiles), CTA b taking u = b, b + grid, ...; a unit is one run of x^T G.
  const int nunits = nslab * nq;
  Ctl ctl{&tail->abort, err, wt.wait_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&tail->full[s], 1);
      mbar_init(&tail->empty[s], kEpiWarps + 1);    // the epilogue warps + the MMAs that read the slot
    }
    mbar_init(&tail->a_full, 1);
    mbar_init(&tail->a_free, 1);
    mbar_init(&tail->at_full, 4);                  // one filling warp per TMEM lane quarter
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tail->d1_full[b], 1);
      mbar_init(&tail->d1_empty[b], kEpiWarps);
    }
    mbar_init(&tail->mt_full, 1);
    mbar_init(&tail->mt_empty, kEpiWarps / 2);
    mbar_init(&tail->mma_done, 1);
    tail->abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_gin);
    if (kGxp) tma_prefetch_desc(&tmap_gxp);
  }
  if (warp == kWarpMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tail->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tail->tmem_base;
  pdl_trigger();
  pdl_wait();                                    // tile records and planes are the earlier launches'

  if (warp == kWarpProd) {
    // ===================================================== TMA producer
    if (lane == 0) {
      const uint64_t once = policy_evict_first();
      const uint64_t keep = policy_evict_last();
      int s = 0;
      uint32_t ph = 0;
      long long iss = 0;
      int piece = 0;
      bool ok = true, a_pending = false;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const int slab = u / nq, chunk = u % nq;
        const int t0 = (int)((long long)chunk * ntiles / nq), t1 = (int)((long long)(chunk + 1) * ntiles / nq);
        if (t0 == t1) continue;
        if (piece > 0 && !wait_bar_sleep(&tail->a_free, (uint32_t)(piece - 1) & 1u, ctl, kErrWaitTimeout)) break;
        mbar_expect_tx(&tail->a_full, (uint32_t)kABytes);
        bulk_load_hint(sA, planes + (size_t)slab * (kABytes / 2), (uint32_t)kABytes, &tail->a_full, keep);
        a_pending = true;
        ++piece;
        for (int tile = t0; tile < t1; ++tile) {
          // L2 prefetch of the tile kPrefetch ahead: its later copy hits L2
          if (kPrefetch > 0 && tile + kPrefetch < t1) {
            const int pt = tile + kPrefetch;
            tma_prefetch_l2_4d(&tmap_x, 0, pt * kBwTile, slab, 0);
            if (kGxp) tma_prefetch_l2_4d(&tmap_gxp, 0, pt * kBwTile, slab, 0);
            tma_prefetch_l2_3d(&tmap_gin, 0, pt * kBwTile, slab);
            bulk_prefetch_l2(tiles + (size_t)pt * kRec, (uint32_t)kRec);
          }
          if (!wait_bar_sleep(&tail->empty[s], ph ^ 1u, ctl, kErrWaitTimeout)) { ok = false; break; }
          // test hook: CTA 0 issues nothing for its last tile, so the waits
          // on that stage give up (no copy is left in flight)
          if (wt.withhold_x && blockIdx.x == 0 && tile == t1 - 1 && u + (int)gridDim.x >= nunits) {
            ok = false;
            break;
          }
          uint8_t* st = sStage + (size_t)s * kStageBytes;
          mbar_expect_tx(&tail->full[s], (uint32_t)kStageBytes);
          tma_load_4d_hint(st, &tmap_x, &tail->full[s], 0, tile * kBwTile, slab, 0, once);
          if (kGxp) tma_load_4d_hint(st + offGxp, &tmap_gxp, &tail->full[s], 0, tile * kBwTile, slab, 0, once);
          tma_load_3d_hint(st + offGin, &tmap_gin, &tail->full[s], 0, tile * kBwTile, slab, once);
          bulk_load_hint(st + offRec, tiles + (size_t)tile * kRec, (uint32_t)kRec, &tail->full[s], keep);
          ++iss;
          if (++s == stages) { s = 0; ph ^= 1u; }
        }
      }
      for (long long q = 0; q < (iss < stages ? iss : stages); ++q) {   // let issued copies land
        if (--s < 0) { s = stages - 1; ph ^= 1u; }
        mbar_drain(&tail->full[s], ph);
      }
      if (a_pending) mbar_drain(&tail->a_full, (uint32_t)(piece - 1) & 1u);
    }
  } else if (warp == kWarpMma) {
    // ===================================================== MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_mt = idesc_bf16_major(128, kMtCols, true, false);
      constexpr uint32_t idesc_d1 = idesc_bf16_major(128, kBwTile, true, true);
      constexpr uint32_t idesc_d1_ta = idesc_bf16_major(128, kBwTile, false, true);
      const uint32_t a_addr = smem_u32(sA);
      int s = 0;
      uint32_t ph = 0;
      long long k = 0;
      int piece = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const int chunk = u % nq;
        const int t0 = (int)((long long)chunk * ntiles / nq), t1 = (int)((long long)(chunk + 1) * ntiles / nq);
        for (int tile = t0; tile < t1; ++tile, ++k) {
          const bool first = tile == t0, last = tile == t1 - 1;
          const int b = (int)(k & 1);
          if (!wait_bar_sleep(&tail->full[s], ph, ctl, kErrWaitTimeout) ||
              (first && !wait_bar_sleep(&tail->a_full, (uint32_t)piece & 1u, ctl, kErrWaitTimeout)) ||
              (kTmA && first && !wait_bar_sleep(&tail->at_full, (uint32_t)piece & 1u, ctl, kErrWaitTimeout)) ||
              !wait_bar_sleep(&tail->d1_empty[b], ((uint32_t)(k >> 1) & 1u) ^ 1u, ctl, kErrWaitTimeout)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t x_addr = smem_u32(sStage + (size_t)s * kStageBytes);
          const uint32_t gt_addr = x_addr + (uint32_t)offRec;
          // G phi' first (the epilogue waits for it).  A = phi' planes 0 and
          // 1 from tensor memory in fp32 mode (filled once per unit), else
          // the shared slab MN-major (rows = gate rows = K); B = G planes
          // MN-major with N = 64 tokens, one 128-byte row (its atom stride is
          // unused)
#pragma unroll
          for (int g = 0; g < kGroups; ++g) {
#pragma unroll
            for (int q = 0; q < kNQ; ++q) {
              int gp, pp;
              product_planes(q, gp, pp);
#pragma unroll
              for (int ks = 0; ks < kBwRp / 16; ++ks) {
                const uint32_t dcol = tmem_base + (uint32_t)(b * kGroups * kBwTile + g * kBwTile);
                const uint64_t bdesc = sw128_desc_mn(gt_addr + (uint32_t)(gp * kBwPlaneBytes + ks * 2048), 1024);
                const uint32_t acc = (q == 0 && ks == 0) ? 0u : 1u;
                if (kTmA && pp < 2)
                  mma_bf16_ta(dcol, tmem_base + (uint32_t)(kAtCol0 + g * kAtCols + pp * (kBwRp / 2) + ks * 8),
                              bdesc, idesc_d1_ta, acc);
                else
                  mma_bf16(dcol, sw128_desc_mn(a_addr + (uint32_t)(g * 2 * kABlk + pp * kBwPlaneBytes + ks * 2048), kABlk),
                           bdesc, idesc_d1, acc);
              }
            }
          }
          mma_commit(&tail->d1_full[b]);
          // then x^T G, accumulated over the unit (the previous unit's sum
          // must have been read out first): A = x tile seen MN-major (rows =
          // tokens = K), B = G planes K-major
          if (first && piece > 0 &&
              !wait_bar_sleep(&tail->mt_empty, (uint32_t)(piece - 1) & 1u, ctl, kErrWaitTimeout)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int g = 0; g < kGroups; ++g) {
#pragma unroll
            for (int ks = 0; ks < kBwTile / 16; ++ks)
              mma_bf16(tmem_base + (uint32_t)(kMtCol0 + g * kMtCols),
                       sw128_desc_mn(x_addr + (uint32_t)(g * 2 * kBwTile * 128 + ks * 2048), kBwTile * 128),
                       sw128_desc(gt_addr + (uint32_t)(ks * 32)), idesc_mt, (first && ks == 0) ? 0u : 1u);
          }
          mma_commit(&tail->empty[s]);                // the slot's operands have been read
          if (last) {
            mma_commit(&tail->mt_full);
            mma_commit(&tail->a_free);
            ++piece;
          }
          if (++s == stages) { s = 0; ph ^= 1u; }
        }
      }
      mma_commit(&tail->mma_done);
      mbar_drain(&tail->mma_done, 0);
    }
  } else {
    // ===================================================== epilogue
    const int ew = warp - kWarpEpi0;          // 0..15
    const int grp = ew >> 3;                  // M-group: streams 2grp, 2grp+1
    const int half = (ew >> 2) & 1;           // tokens half*32 .. +32
    const int q = warp & 3;                   // TMEM lane quarter of this warp
    const int m = q * 32 + lane;              // row of the group (0..127)
    const int i = grp * 2 + (m >> 6);         // stream
    const int d = m & 63;                     // column of the slab
    // Per-lane byte offsets of the epilogue's shared-memory reads: x /
    // grad_h_in element pair (token half*32 + j + 4*odd, columns dp, dp+1)
    // in the swizzled tile, and the (hPre_i, RMS factor) pair of that token;
    // iteration e0 adds e0 rows (multiples of 8: the swizzle phase is
    // unchanged).  grad_x goes straight to global memory from registers.
    const int odd = lane & 1, dp = d & ~1;
    uint32_t xoff[4], soff[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int ej = j + 4 * odd;
      xoff[j] = (uint32_t)((half * kHalf + ej) * 128) + ((uint32_t)((dp >> 3) ^ ej) << 4) + ((uint32_t)(dp & 7) << 1);
      soff[j] = (uint32_t)((i * (2 * kBwTile) + 2 * (half * kHalf + ej)) * 4);
    }
    const uint32_t trow = (uint32_t)(kBwNS * D);   // elements from one token to the next
    int s = 0;
    uint32_t ph = 0;
    long long k = 0;
    int piece = 0;
    bool run = true;
    for (int u = blockIdx.x; u < nunits && run; u += gridDim.x) {
      const int slab = u / nq, chunk = u % nq;
      const int t0 = (int)((long long)chunk * ntiles / nq), t1 = (int)((long long)(chunk + 1) * ntiles / nq);
      if (kTmA && t0 < t1 && ew < 4) {
        // One warp per TMEM lane quarter copies phi' planes 0 and 1 of the
        // unit's slab into tensor memory as the A operand of G phi': lane m
        // = column m of group g, column c = gate rows 2c (low half) and
        // 2c + 1.  The slab is in shared memory once a_full completes, which
        // is after the previous unit's MMAs have all finished (a_free).
        if (!wait_bar_sleep(&tail->a_full, (uint32_t)piece & 1u, ctl, kErrWaitTimeout)) {
          run = false;
          break;
        }
#pragma unroll 1
        for (int g = 0; g < kGroups; ++g) {
          const int mm = q * 32 + lane;
          const uint8_t* src = sA + (g * 2 + (mm >> 6)) * kABlk;
          const int dc = mm & 63;
          uint32_t w[2 * (kBwRp / 2)];
#pragma unroll
          for (int c = 0; c < 2 * (kBwRp / 2); ++c) {
            const int pl = c / (kBwRp / 2), r = 2 * (c % (kBwRp / 2));
            const uint16_t lo = *reinterpret_cast<const uint16_t*>(src + pl * kBwPlaneBytes + swz(r, dc));
            const uint16_t hi = *reinterpret_cast<const uint16_t*>(src + pl * kBwPlaneBytes + swz(r + 1, dc));
            w[c] = (uint32_t)lo | ((uint32_t)hi << 16);
          }
          tmem_st32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(kAtCol0 + g * kAtCols), w);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tail->at_full);
      }
      for (int tile = t0; tile < t1; ++tile, ++k) {
        const bool last = tile == t1 - 1;
        const int b = (int)(k & 1);
        const int tok0 = tile * kBwTile + half * kHalf + 4 * odd;   // this lane's token at (e0, j) = (0, 0)
        const int lim = T - tok0;                                    // its tokens e0 + j < lim exist
        __nv_bfloat16* gout = gx + (size_t)tok0 * trow + (size_t)i * D + slab * 64 + dp;
        if (!wait_bar_sleep(&tail->full[s], ph, ctl, kErrWaitTimeout) ||
            !wait_bar_sleep(&tail->d1_full[b], (uint32_t)(k >> 1) & 1u, ctl, kErrWaitTimeout)) {
          run = false;
          break;
        }
        tc_fence_after();
        const uint8_t* st = sStage + (size_t)s * kStageBytes;
        const uint8_t* xs = st + i * (kBwTile * 128);
        const uint8_t* gxs = st + offGxp + i * (kBwTile * 128);
        const uint8_t* gin = st + offGin;
        const float* scal = reinterpret_cast<const float*>(st + offRec + P * kBwPlaneBytes);
        float acc[kHalf];
        {
          const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) +
                                 (uint32_t)(b * kGroups * kBwTile + grp * kBwTile + half * kHalf);
          float v0[16], v1[16];
          tmem_ld16(taddr, v0);
          tmem_ld16(taddr + 16, v1);
#pragma unroll
          for (int e = 0; e < 16; ++e) { acc[e] = v0[e]; acc[16 + e] = v1[e]; }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tail->d1_empty[b]);
        // Lanes 2p, 2p+1 hold columns d, d+1 (d even).  Each pair trades
        // one value so that the even lane forms both columns of token e and
        // the odd lane both columns of token e + 4 (rows 4 apart sit in
        // different bank groups of the swizzle): 4-byte shared accesses at
        // per-lane offsets fixed for the kernel plus compile-time steps.
        const uint8_t* xg = xs;
        const uint8_t* gg = gin;
        const uint8_t* sg = reinterpret_cast<const uint8_t*>(scal);
#pragma unroll
        for (int e0 = 0; e0 < kHalf; e0 += 8) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float sendv = odd ? acc[e0 + j] : acc[e0 + j + 4];
            const float recv = __shfl_xor_sync(0xffffffffu, sendv, 1);
            const float lo = odd ? recv : acc[e0 + j];
            const float hi = odd ? acc[e0 + j + 4] : recv;
            const uint32_t off = xoff[j] + (uint32_t)(e0 * 128);
            const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(xg + off));
            const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(gg + off));
            const float2 hc = *reinterpret_cast<const float2*>(sg + soff[j] + (uint32_t)(e0 * 8));
            float vlo = fmaf(hc.x, gf.x, lo), vhi = fmaf(hc.x, gf.y, hi);
            vlo = fmaf(hc.y, xf.x, vlo);
            vhi = fmaf(hc.y, xf.y, vhi);
            if constexpr (kGxp) {
              const float2 pf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(gxs + off));
              vlo += pf.x;
              vhi += pf.y;
            }
            if (e0 + j < lim) {
              const __nv_bfloat162 o = __floats2bfloat162_rn(vlo, vhi);
              __stcs(reinterpret_cast<unsigned int*>(gout + (e0 + j) * trow), *reinterpret_cast<const unsigned int*>(&o));
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&tail->empty[s]);      // this warp has read the slot
        if (last && half == 0) {
          // x^T G of this unit, summed over the planes -> partial buffer [u][r][k]
          if (!wait_bar_sleep(&tail->mt_full, (uint32_t)piece & 1u, ctl, kErrWaitTimeout)) {
            run = false;
            break;
          }
          tc_fence_after();
          float* dst = pieces + (size_t)u * kBwRp * (kBwNS * 64) + grp * 128 + m;
          const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(kMtCol0 + grp * kMtCols);
#pragma unroll
          for (int c0 = 0; c0 < kBwR; c0 += 8) {
            float sum[8];
#pragma unroll
            for (int pl = 0; pl < P; ++pl) {
              float v[8];
              tmem_ld8(taddr + (uint32_t)(pl * kBwRp + c0), v);
#pragma unroll
              for (int e = 0; e < 8; ++e) sum[e] = pl == 0 ? v[e] : sum[e] + v[e];
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) dst[(size_t)(c0 + e) * (kBwNS * 64)] = sum[e];
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tail->mt_empty);
        }
        if (last) ++piece;
        if (++s == stages) { s = 0; ph ^= 1u; }
      }
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                 : "memory");
  }
}

// =============================================================== final sums
// Column blocks: kFinCols columns k, three groups of eight gate rows each
// (one thread per column and group: all of a thread's unit loads are
// independent, and three times the threads of one per column); the groups'
// grad_gamma terms are added in group order.  Reduction blocks: one of
// grad_bias / grad_alpha each.
constexpr int kFinCols = 128, kFinGroups = 3, kFinRows = kBwR / kFinGroups;
constexpr int kFinalThreads = kFinCols * kFinGroups;
static_assert(kFinRows * kFinGroups == kBwR, "gate rows split evenly");

__global__ void __launch_bounds__(kFinalThreads) bw_final_kernel(BwFinalParams p, int col_blocks) {
  pdl_wait();
  const int K = kBwNS * p.D;
  __shared__ float red[kFinalThreads];
  if ((int)blockIdx.x < col_blocks) {
    const int grp = threadIdx.x / kFinCols, kk = threadIdx.x % kFinCols;
    const int k = blockIdx.x * kFinCols + kk;
    float gg = 0.0f;
    if (k < K) {
      const int i = k / p.D, dd = k % p.D;
      const int slab = dd / 64;
      const int mloc = i * 64 + (dd & 63);
      const int r0 = grp * kFinRows;
      float acc[kFinRows];
#pragma unroll
      for (int r = 0; r < kFinRows; ++r) acc[r] = 0.0f;
#pragma unroll
      for (int c = 0; c < kBwMaxChunks; ++c) {        // the slab's units, in order
        if (c < p.nq) {
          const float* src = p.pieces + (size_t)(slab * p.nq + c) * kBwRp * (kBwNS * 64) + (size_t)r0 * (kBwNS * 64) + mloc;
#pragma unroll
          for (int r = 0; r < kFinRows; ++r) acc[r] += src[(size_t)r * (kBwNS * 64)];
        }
      }
      const float gm = p.gamma ? __ldg(p.gamma + k) : 1.0f;
#pragma unroll
      for (int r = 0; r < kFinRows; ++r) {
        p.grad_phi[(size_t)(r0 + r) * K + k] = gm * acc[r];
        gg = fmaf(__ldg(p.phi + (size_t)(r0 + r) * K + k), acc[r], gg);
      }
    }
    red[threadIdx.x] = gg;
    __syncthreads();
    if (grp == 0 && k < K && p.grad_gamma) {
      float t = red[kk];
#pragma unroll
      for (int q = 1; q < kFinGroups; ++q) t += red[q * kFinCols + kk];
      p.grad_gamma[k] = t;
    }
    return;
  }
  // grad_bias[v] (v < R) and grad_alpha[v - R]: fixed-order sums of the partials
  const int v = blockIdx.x - col_blocks;
  const int colp = v;                       // column of the partial records
  float sacc = 0.0f;
  for (int j = threadIdx.x; j < p.nparts; j += kFinalThreads) sacc += p.partials[(size_t)j * 32 + colp];
  red[threadIdx.x] = sacc;
  __syncthreads();
  if ((int)threadIdx.x < kFinCols) {
    float t = red[threadIdx.x];
#pragma unroll
    for (int q = 1; q < kFinGroups; ++q) t += red[q * kFinCols + threadIdx.x];
    red[threadIdx.x] = t;                   // reads only entries no thread writes in this step
  }
  __syncthreads();
  for (int o = kFinCols / 2; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    if (v < kBwR) p.grad_bias[v] = red[0];
    else p.grad_alpha[v - kBwR] = red[0];
  }
}

// A launch that may begin while the previous launch on the stream finishes
// (the kernel itself waits for it: pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace

cudaError_t launch_bw_planes(const BwPlaneParams& pp, cudaStream_t s) {
  const long long total = (long long)pp.nslab * kBwNS * pp.P * kBwRp * 8;   // 16-byte pieces
  int blocks = (int)((total + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  bw_planes_kernel<<<blocks, 256, 0, s>>>(pp);
  return cudaGetLastError();
}

void bw_rowdot_shape(int D, size_t max_smem, int* tps, int* stages, size_t* smem_bytes) {
  const size_t tok = (size_t)(kBwNS + 1) * D * 2;
  size_t t = 65536 / tok;
  if (t < 1) t = 1;
  if (t > 16) t = 16;
  const size_t avail = max_smem > sizeof(RdTail) + 128 ? max_smem - sizeof(RdTail) - 128 : 0;
  size_t st = avail / (t * tok);
  if (st > (size_t)kRdMaxStages) st = kRdMaxStages;
  *tps = (int)t;
  // one stage when two whole token rows do not fit (D above ~11.6 k): each
  // CTA then loads and reduces one token at a time, and the 152 SMs' rows in
  // flight still cover HBM latency
  *stages = st >= 1 ? (int)st : 0;
  *smem_bytes = (size_t)(*stages) * t * tok + sizeof(RdTail);
}

cudaError_t launch_bw_rowdot(const BwRowdotParams& p, int grid, size_t smem_bytes, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(bw_rowdot_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
  if (e != cudaSuccess) return e;
  return launch_dependent(bw_rowdot_kernel, dim3(grid), dim3(kRdThreads), smem_bytes, s, p);
}

cudaError_t bw_token_blocks(int* blocks) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bw_token_kernel, kBwTokenWarps * 32, 0)) !=
      cudaSuccess)
    return e;
  long long b = (long long)sms * (per_sm > 0 ? per_sm : 1);
  if (b > kBwMaxTokenBlocks) b = kBwMaxTokenBlocks;
  *blocks = (int)b;
  return cudaSuccess;
}

cudaError_t launch_bw_token(const BwTokenParams& p, int blocks, cudaStream_t s) {
  return launch_dependent(bw_token_kernel, dim3(blocks), dim3(kBwTokenWarps * 32), 0, s, p);
}

cudaError_t launch_bw_main(const BwMainLaunch& L, cudaStream_t s) {
  const void* k = nullptr;
  if (L.P == 3) k = L.has_gxp ? reinterpret_cast<const void*>(&bw_main_kernel<3, true>)
                              : reinterpret_cast<const void*>(&bw_main_kernel<3, false>);
  else k = L.has_gxp ? reinterpret_cast<const void*>(&bw_main_kernel<2, true>)
                     : reinterpret_cast<const void*>(&bw_main_kernel<2, false>);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem_bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.grid, 1, 1);
  cfg.blockDim = dim3(kMainThreads, 1, 1);
  cfg.dynamicSmemBytes = L.smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int T = L.T, D = L.D, ntiles = L.ntiles, nslab = L.nslab, nq = L.nq, stages = L.stages;
  WaitTest wt = L.wt;
  const __nv_bfloat16* planes = L.planes;
  const uint8_t* tiles = L.tiles;
  float* pieces = L.pieces;
  __nv_bfloat16* gx = L.grad_x;
  uint32_t* err = L.err;
  void* args[] = {const_cast<CUtensorMap*>(&L.tmap_x), const_cast<CUtensorMap*>(&L.tmap_gin),
                  const_cast<CUtensorMap*>(&L.tmap_gxp), &planes, &tiles, &pieces, &gx, &err,
                  &T, &D, &ntiles, &nslab, &nq, &stages, &wt};
  return cudaLaunchKernelExC(&cfg, k, args);
}

cudaError_t launch_bw_final(const BwFinalParams& p, cudaStream_t s) {
  const int K = kBwNS * p.D;
  const int col_blocks = (K + kFinCols - 1) / kFinCols;
  const int blocks = col_blocks + kBwR + 3;
  return launch_dependent(bw_final_kernel, dim3(blocks), dim3(kFinalThreads), 0, s, p, col_blocks);
}

}  // namespace mhc
