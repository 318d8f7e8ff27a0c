// mhc_pre_gw.cu -- the grid-wide sm_103a forward.
//
// What is computed follows "CANN ops-transformer 中 aclnnMhcPreV2 算子接口
// 全解析" §三 and "aclnnMhcPreSinkhorn 接口与 MhcPreSinkhorn 实现剖析" §3.2;
// how it is laid out on the GPU is this file's own design.
//
// The forward is bound by reading x, and y needs every byte of x a second
// time once the token's gates are known.  The gates need the whole token
// (a reduction over n*D), so the second read can only hit L2 if the bytes
// loaded between a token's first touch and its gates stay small.  Here every
// CTA (one per SM, all resident: cooperative launch) works on the SAME
// 128-token tile at about the same time, each on its own slice of d:
//
//  * CTA b owns a contiguous run of (64-wide d-chunk, stream) units.  Their
//    phi-plane blocks stay in shared memory for the whole kernel; each tile
//    brings one 16 KB x box per unit (TMA, 128-byte swizzle).
//  * One thread issues tcgen05.mma over the CTA's units, M = 128 tokens,
//    N = NP plane rows, fp32 accumulate in TMEM (two buffers).  Four warps
//    add x^2 for their token rows from the same shared-memory boxes, read
//    the accumulators (thread = token = TMEM lane), fold the precision planes
//    and store the CTA's partial sums to a global ring.
//  * Token t of tile k is gated by CTA (128k + t) mod grid: once every CTA
//    has published tile k (a counter per ring slot), its gate warp sums the
//    partials in CTA order, computes invRms and the gates, writes the y
//    weights to the ring and counts the token as ready; the Sinkhorn warp
//    then produces comb off the critical path.
//  * When all tokens of tile k are ready, eight warps form y for the CTA's
//    own d-range, re-reading x (loaded moments ago by the whole GPU: an L2
//    hit) with plain 16-byte loads.
//
// Every wait is bounded by a timer.  A wait that gives up sets the error
// word and a grid-wide abort flag, and every CTA winds down.
#include "mhc_ptx.cuh"

namespace mhc {
namespace {

constexpr int kGwThreads = 512;
// Warp roles.
constexpr int kGwWarpX = 0, kGwWarpMma = 1, kGwWarpGate = 2, kGwWarpSink = 3, kGwWarpPub0 = 4,
              kGwWarpY0 = 8;
constexpr int kGwPubThreads = 128;
constexpr int kGwYThreads = kGwThreads - kGwWarpY0 * 32;   // 256
// Named barriers: 1 = publish warps, 2 = y warps.
constexpr int kGwBarPub = 1, kGwBarY = 2;

template <int NS, int RR, int P>
struct GwCfg {
  static constexpr int kNP = gw_np(RR, P);                      // MMA N
  static_assert(kNP <= 256, "N of one MMA is at most 256");
  static constexpr int kAccCols = kNP <= 32 ? 32 : kNP <= 64 ? 64 : kNP <= 128 ? 128 : 256;
  static constexpr uint32_t kTmemCols = 2u * kAccCols;          // two accumulators
  static constexpr int kPlaneBytes = kNP * 128;                 // one unit's phi-plane block
  static constexpr int kStr = partial_stride(RR);               // floats per partial
  static constexpr int kG4 = kStr / 4;                          // float4 groups per partial
  static constexpr int kG4Pad = kG4 <= 4 ? 4 : kG4 <= 8 ? 8 : kG4 <= 16 ? 16 : 32;
  static_assert(kG4 <= 32, "one lane per float4 group");
  static constexpr int kLpg = 32 / kG4Pad;                      // lanes summing one group
  static constexpr bool kThree = (RR == NS * NS + 2 * NS);
  static constexpr int kYB = NS <= 4 ? 4 : 2;                   // y items in flight per thread
};

struct GwTail {
  uint64_t x_full[kMaxStages], x_empty[kMaxStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t phi_full;
  uint64_t sink_full[2], sink_free[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t abort;
};
static_assert(sizeof(GwTail) <= kTailBytes, "barrier block outgrew its reservation");

struct GwCtl {
  volatile uint32_t* abort;    // shared: this CTA is winding down
  volatile uint32_t* gabort;   // global: some CTA gave up
  uint32_t* err;               // global error word
};

__device__ __noinline__ void gw_fail(const GwCtl& c, uint32_t code) {
  atomicOr(c.err, code);
  *c.abort = 1u;
  atomicExch(const_cast<uint32_t*>(c.gabort), 1u);
}

// Wait for phase `parity` of a local mbarrier; gives up after kWaitNs or as
// soon as this CTA or any other has given up.
__device__ __noinline__ bool gw_wait(uint64_t* bar, uint32_t parity, const GwCtl& c) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*c.abort || *c.gabort) {
        *c.abort = 1u;
        return false;
      }
      if (now_ns() - t0 > kWaitNs) {
        gw_fail(c, kErrWaitTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Wait until a global counter written by other CTAs reaches `target`
// (acquire: what they wrote before counting is visible afterwards).
__device__ __noinline__ bool gw_wait_count(const uint32_t* ctr, uint32_t target, const GwCtl& c) {
  if (ld_acquire_gpu(ctr) >= target) return true;
  const uint64_t t0 = now_ns();
  for (uint32_t it = 1;; ++it) {
    if (ld_acquire_gpu(ctr) >= target) return true;
    if ((it & 15u) == 0) {
      if (*c.abort || *c.gabort) {
        *c.abort = 1u;
        return false;
      }
      if (now_ns() - t0 > kWaitNs) {
        gw_fail(c, kErrGridWait);
        return false;
      }
    }
  }
}

__device__ __forceinline__ float f4_get(const float4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <int NS, int RR, int P>
__global__ void __launch_bounds__(kGwThreads, 1)
    mhc_pre_gw_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_p,
                      const EpiParams ep, const __nv_bfloat16* __restrict__ xg, const GwGeom g, uint32_t* hdr,
                      float* partials, float* coefs) {
  using C = GwCfg<NS, RR, P>;
  constexpr int NN = NS * NS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const GwLayout Ly = gw_layout(NS, RR, P, g.umax, g.xstages, g.own_max);
  const int XS = g.xstages;
  uint8_t* sPhi = smem + Ly.phi;
  uint8_t* sX = smem + Ly.x;
  float* ycoef = reinterpret_cast<float*>(smem + Ly.ycoef);   // [128][NS]
  float* sink_buf = reinterpret_cast<float*>(smem + Ly.sink); // [2][own_max][NN]
  int* sink_cnt = reinterpret_cast<int*>(smem + Ly.scnt);     // [2]
  GwTail* tail = reinterpret_cast<GwTail*>(smem + Ly.tail);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const int b = blockIdx.x;
  const int units = g.nch * NS;
  const int u0 = (int)((long long)b * units / G);
  const int U = (int)((long long)(b + 1) * units / G) - u0;   // units this CTA owns (>= 1)
  const size_t slot_bytes = (size_t)g.umax * kGwUnitBytes;
  uint32_t* arrive = hdr + kHdrArrive;
  uint32_t* ready = hdr + kHdrReady;
  uint32_t* ydone = hdr + kHdrYdone;
  GwCtl ctl{&tail->abort, hdr + kHdrAbort, hdr};

  // ---- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < XS; ++s) {
      mbar_init(&tail->x_full[s], 1);
      mbar_init(&tail->x_empty[s], 1 + 4);      // MMA commit + the four sum-of-squares warps
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tail->acc_full[a], 1);
      mbar_init(&tail->acc_empty[a], 4);        // four publish warps
      mbar_init(&tail->sink_full[a], 1);
      mbar_init(&tail->sink_free[a], 1);
    }
    mbar_init(&tail->phi_full, 1);
    mbar_init(&tail->mma_done, 1);
    tail->abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_p);
  }
  if (warp == kGwWarpMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tail->tmem_base)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tail->tmem_base;

  if (warp == kGwWarpX) {
    // ================================================= TMA: phi planes once, then x
    // Lane q issues unit q's box, so the CTA's boxes of one tile go out
    // together.
    const uint64_t keep = policy_evict_last();
    if (lane == 0) mbar_expect_tx(&tail->phi_full, (uint32_t)(U * C::kPlaneBytes));
    __syncwarp();
    if (lane < U) {
      const int u = u0 + lane, i = u / g.nch, j = u - i * g.nch;
      tma_load_3d_hint(sPhi + (size_t)lane * C::kPlaneBytes, &tmap_p, &tail->phi_full, j * kChunkK, 0, i, keep);
    }
    int xs = 0;
    uint32_t xph = 0;
    int issued = 0;
    for (int k = 0; k < g.num_tiles; ++k) {
      bool ok = true;
      if (lane == 0) ok = gw_wait(&tail->x_empty[xs], xph ^ 1u, ctl);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      if (lane == 0) mbar_expect_tx(&tail->x_full[xs], (uint32_t)(U * kGwUnitBytes));
      __syncwarp();
      if (lane < U) {
        const int u = u0 + lane, i = u / g.nch, j = u - i * g.nch;
        tma_load_3d_hint(sX + (size_t)xs * slot_bytes + (size_t)lane * kGwUnitBytes, &tmap_x, &tail->x_full[xs],
                         j * kChunkK, k * kGwTile, i, keep);
      }
      ++issued;
      if (++xs == XS) { xs = 0; xph ^= 1u; }
    }
    if (lane == 0) {   // let the copies in flight land before the CTA can exit
      for (int q = 0; q < (issued < XS ? issued : XS); ++q) {
        if (--xs < 0) { xs = XS - 1; xph ^= 1u; }
        mbar_drain(&tail->x_full[xs], xph);
      }
      mbar_drain(&tail->phi_full, 0);
    }
  } else if (warp == kGwWarpMma) {
    // ================================================= MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kMmaM, C::kNP);
      const uint32_t phi0 = smem_u32(sPhi);
      bool ok = gw_wait(&tail->phi_full, 0, ctl);
      int xs = 0;
      uint32_t xph = 0;
      for (int k = 0; k < g.num_tiles && ok; ++k) {
        const int acc = k & 1;
        const uint32_t acc_phase = (uint32_t)(k >> 1) & 1u;
        if (!gw_wait(&tail->acc_empty[acc], acc_phase ^ 1u, ctl)) break;
        if (!gw_wait(&tail->x_full[xs], xph, ctl)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * C::kAccCols);
        const uint32_t xb = smem_u32(sX + (size_t)xs * slot_bytes);
        for (int q = 0; q < U; ++q) {
          const uint32_t a0 = xb + (uint32_t)(q * kGwUnitBytes);
          const uint32_t b0 = phi0 + (uint32_t)(q * C::kPlaneBytes);
#pragma unroll
          for (int kk = 0; kk < kChunkK / 16; ++kk)
            mma_bf16(d, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc, (q | kk) ? 1u : 0u);
        }
        mma_commit(&tail->x_empty[xs]);
        mma_commit(&tail->acc_full[acc]);
        if (++xs == XS) { xs = 0; xph ^= 1u; }
      }
      mma_commit(&tail->mma_done);
      mbar_drain(&tail->mma_done, 0);
    }
  } else if (warp >= kGwWarpPub0 && warp < kGwWarpY0) {
    // ================================================= sum of squares + partials
    // Thread = token row of the tile = TMEM lane.
    const int t = threadIdx.x - kGwWarpPub0 * 32;   // 0..127
    const int wq = warp & 3;                        // TMEM lane quarter
    int xs = 0;
    uint32_t xph = 0;
    for (int k = 0; k < g.num_tiles; ++k) {
      const int acc = k & 1;
      const uint32_t acc_phase = (uint32_t)(k >> 1) & 1u;
      // x^2 over this CTA's units, straight from the swizzled boxes (the
      // order of a row's 16-byte pieces does not matter for a sum).
      if (!role_all<kGwBarPub, kGwPubThreads>(gw_wait(&tail->x_full[xs], xph, ctl))) break;
      float ssq = 0.0f;
      const uint8_t* xrow = sX + (size_t)xs * slot_bytes + (size_t)t * 128;
      for (int q = 0; q < U; ++q) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(xrow + (size_t)q * kGwUnitBytes + c * 16);
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h[e]);
            ssq = fmaf(f.x, f.x, ssq);
            ssq = fmaf(f.y, f.y, ssq);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->x_empty[xs]);
      if (++xs == XS) { xs = 0; xph ^= 1u; }

      // projection partials from TMEM
      if (!role_all<kGwBarPub, kGwPubThreads>(gw_wait(&tail->acc_full[acc], acc_phase, ctl))) break;
      tc_fence_after();
      float mix[RR];
#pragma unroll
      for (int r = 0; r < RR; ++r) mix[r] = 0.0f;
      const uint32_t taddr = tmem_base + ((uint32_t)(wq * 32) << 16) + (uint32_t)(acc * C::kAccCols);
#pragma unroll
      for (int grp = 0; grp < C::kNP / 16; ++grp) {
        float v[16];
        tmem_ld16(taddr + grp * 16, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int col = grp * 16 + e;
          if (col < P * RR) mix[col % RR] += v[e];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->acc_empty[acc]);

      // the ring slot is free once every token of tile k - kGwSlots is gated
      const int gs = k % kGwSlots;
      const uint32_t use = (uint32_t)(k / kGwSlots);
      bool ok = true;
      if (use > 0 && t == 0) ok = gw_wait_count(&ready[gs], use * (uint32_t)kGwTile, ctl);
      if (!role_all<kGwBarPub, kGwPubThreads>(ok)) break;
      float* dst = partials + (((size_t)gs * kGwTile + t) * G + b) * C::kStr;
#pragma unroll
      for (int r = 0; r < C::kStr; r += 4) {
        float4 v;
        v.x = r < RR ? mix[r] : (r == RR ? ssq : 0.0f);
        v.y = r + 1 < RR ? mix[r + 1] : (r + 1 == RR ? ssq : 0.0f);
        v.z = r + 2 < RR ? mix[r + 2] : (r + 2 == RR ? ssq : 0.0f);
        v.w = r + 3 < RR ? mix[r + 3] : (r + 3 == RR ? ssq : 0.0f);
        __stcg(reinterpret_cast<float4*>(dst + r), v);
      }
      role_sync<kGwBarPub, kGwPubThreads>();
      if (t == 0) {
        __threadfence();
        red_release_gpu(&arrive[gs], 1u);
      }
    }
  } else if (warp == kGwWarpGate) {
    // ================================================= gates of the tokens this CTA owns
    const int grp4 = lane % C::kG4Pad;
    const int sub = lane / C::kG4Pad;
    for (int k = 0; k < g.num_tiles; ++k) {
      const int gs = k % kGwSlots;
      const uint32_t use = (uint32_t)(k / kGwSlots);
      const int tile0 = k * kGwTile;
      const int valid = min(kGwTile, g.T - tile0);
      const int first = (int)(((long long)b - (long long)tile0 % G + G) % G);
      const int sb = k & 1;
      bool ok = true;
      if (k >= 2 && lane == 0) ok = gw_wait(&tail->sink_free[sb], ((uint32_t)(k >> 1) - 1u) & 1u, ctl);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      int cnt = 0;
      if (first < valid) {
        if (lane == 0) {
          ok = gw_wait_count(&arrive[gs], (use + 1u) * (uint32_t)G, ctl);
          if (ok && use > 0) ok = gw_wait_count(&ydone[gs], use * (uint32_t)G, ctl);
        }
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
        for (int t = first; t < valid; t += G, ++cnt) {
          // sum the CTAs' partials of row t in a fixed order: lane (sub, grp4)
          // adds CTAs sub, sub + kLpg, ... of float4 group grp4, then a fixed
          // butterfly over the subs.
          const float* src = partials + ((size_t)gs * kGwTile + t) * G * C::kStr;
          float4 s4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          if (grp4 < C::kG4) {
#pragma unroll 4
            for (int c = sub; c < G; c += C::kLpg) {
              const float4 v = __ldcg(reinterpret_cast<const float4*>(src + (size_t)c * C::kStr + grp4 * 4));
              s4.x += v.x;
              s4.y += v.y;
              s4.z += v.z;
              s4.w += v.w;
            }
          }
#pragma unroll
          for (int off = C::kG4Pad; off < 32; off <<= 1) {
            s4.x += __shfl_xor_sync(0xffffffffu, s4.x, off);
            s4.y += __shfl_xor_sync(0xffffffffu, s4.y, off);
            s4.z += __shfl_xor_sync(0xffffffffu, s4.z, off);
            s4.w += __shfl_xor_sync(0xffffffffu, s4.w, off);
          }
          float mix[RR];
#pragma unroll
          for (int r = 0; r < RR; ++r) mix[r] = __shfl_sync(0xffffffffu, f4_get(s4, r & 3), r >> 2);
          const float ssq = __shfl_sync(0xffffffffu, f4_get(s4, RR & 3), RR >> 2);
          if (lane == 0) {
            const int tok = tile0 + t;
            float cf[NS];
            const float inv_rms = token_gates<NS, RR>(ep, tok, mix, ssq, true, cf);
            float* cdst = coefs + ((size_t)gs * kGwTile + t) * NS;
#pragma unroll
            for (int i = 0; i < NS; ++i) __stcg(cdst + i, cf[i]);
            __threadfence();
            red_release_gpu(&ready[gs], 1u);
            float H[NN];
            residual_logits<NS, RR>(ep, mix, inv_rms, H);
            float* e = sink_buf + ((size_t)sb * g.own_max + cnt) * NN;
#pragma unroll
            for (int r = 0; r < NN; ++r) e[r] = H[r];
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        sink_cnt[sb] = cnt;
        mbar_arrive(&tail->sink_full[sb]);
      }
    }
  } else if (warp == kGwWarpSink) {
    // ================================================= Sinkhorn for comb (off y's path)
    for (int k = 0; k < g.num_tiles; ++k) {
      const int sb = k & 1;
      bool ok = true;
      if (lane == 0) ok = gw_wait(&tail->sink_full[sb], (uint32_t)(k >> 1) & 1u, ctl);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      const int cnt = sink_cnt[sb];
      const int tile0 = k * kGwTile;
      const int first = (int)(((long long)b - (long long)tile0 % G + G) % G);
      for (int o = lane; o < cnt; o += 32) {
        const float* e = sink_buf + ((size_t)sb * g.own_max + o) * NN;
        token_sinkhorn<NS, C::kThree>(ep, tile0 + first + o * G, e, true);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->sink_free[sb]);
    }
  } else if (warp >= kGwWarpY0) {
    // ================================================= y for this CTA's d-range
    const int yt = threadIdx.x - kGwWarpY0 * 32;
    const int nvec = g.D >> 3;                      // 16-byte vectors per row
    const int v0 = (int)((long long)b * nvec / G);
    const int nv = (int)((long long)(b + 1) * nvec / G) - v0;
    const uint64_t read_policy = policy_evict_first();
    for (int k = 0; k < g.num_tiles; ++k) {
      const int gs = k % kGwSlots;
      const uint32_t use = (uint32_t)(k / kGwSlots);
      const int tile0 = k * kGwTile;
      const int valid = min(kGwTile, g.T - tile0);
      bool ok = true;
      if (yt == 0) ok = gw_wait_count(&ready[gs], use * (uint32_t)kGwTile + (uint32_t)valid, ctl);
      if (!role_all<kGwBarY, kGwYThreads>(ok)) break;
      const float* csrc = coefs + (size_t)gs * kGwTile * NS;
      for (int e = yt; e < valid * NS; e += kGwYThreads) ycoef[e] = __ldcg(csrc + e);
      role_sync<kGwBarY, kGwYThreads>();
      if (yt == 0) atomicAdd(&ydone[gs], 1u);       // this CTA is done reading slot gs
      const int items = valid * nv;
      const __nv_bfloat16* xt = xg + (size_t)tile0 * NS * g.D;
      __nv_bfloat16* yo = ep.y + (size_t)tile0 * g.D;
      for (int base = yt; base < items; base += kGwYThreads * C::kYB) {
        uint4 xv[C::kYB][NS];
        int rowv[C::kYB], dv[C::kYB];
#pragma unroll
        for (int q = 0; q < C::kYB; ++q) {
          const int it = base + q * kGwYThreads;
          const int row = it / max(nv, 1);
          rowv[q] = it < items ? row : -1;
          dv[q] = (v0 + (it - row * nv)) * 8;
          if (it < items) {
            const __nv_bfloat16* src = xt + (size_t)row * NS * g.D + dv[q];
#pragma unroll
            for (int i = 0; i < NS; ++i) xv[q][i] = ld_global_v4_hint(src + (size_t)i * g.D, read_policy);
          }
        }
#pragma unroll
        for (int q = 0; q < C::kYB; ++q) {
          if (rowv[q] < 0) continue;
          float acc8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc8[e] = 0.0f;
#pragma unroll
          for (int i = 0; i < NS; ++i) {
            const float m = ycoef[rowv[q] * NS + i];
            const __nv_bfloat162* hh = reinterpret_cast<const __nv_bfloat162*>(&xv[q][i]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(hh[e]);
              acc8[2 * e] = fmaf(m, f.x, acc8[2 * e]);
              acc8[2 * e + 1] = fmaf(m, f.y, acc8[2 * e + 1]);
            }
          }
          uint4 o;
          __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
          for (int e = 0; e < 4; ++e) ob[e] = __floats2bfloat162_rn(acc8[2 * e], acc8[2 * e + 1]);
          st_global_v4_hint(yo + (size_t)rowv[q] * g.D + dv[q], o, read_policy);
        }
      }
      role_sync<kGwBarY, kGwYThreads>();             // ycoef is rewritten for the next tile
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kGwWarpMma) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(C::kTmemCols)
                 : "memory");
  }
}

template <int NS, int RR, int P>
const void* gw_kernel_ptr() {
  return reinterpret_cast<const void*>(&mhc_pre_gw_kernel<NS, RR, P>);
}

const void* gw_select(int n, int R, int P) {
#define MHC_CASE(NS_, RR_, P_) \
  if (n == NS_ && R == RR_ && P == P_) return gw_kernel_ptr<NS_, RR_, P_>();
  MHC_CASE(4, 24, 3) MHC_CASE(4, 24, 2) MHC_CASE(4, 8, 3) MHC_CASE(4, 8, 2)
  MHC_CASE(6, 48, 3) MHC_CASE(6, 48, 2) MHC_CASE(6, 12, 3) MHC_CASE(6, 12, 2)
  MHC_CASE(8, 80, 3) MHC_CASE(8, 80, 2) MHC_CASE(8, 16, 3) MHC_CASE(8, 16, 2)
#undef MHC_CASE
  return nullptr;
}

}  // namespace

cudaError_t gw_forward_capacity(int n, int R, int P, size_t smem_bytes, int* max_ctas) {
  *max_ctas = 0;
  const void* k = gw_select(n, R, P);
  if (!k) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kGwThreads, smem_bytes);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  *max_ctas = per_sm * sms;
  return cudaSuccess;
}

cudaError_t launch_gw_forward(const GwLaunch& L, cudaStream_t s) {
  const void* k = gw_select(L.epi.n, L.epi.R, L.P);
  if (!k) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.grid, 1, 1);
  cfg.blockDim = dim3(kGwThreads, 1, 1);
  cfg.dynamicSmemBytes = L.smem_bytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const __nv_bfloat16* xg = static_cast<const __nv_bfloat16*>(L.x);
  void* args[] = {const_cast<CUtensorMap*>(&L.tmap_x), const_cast<CUtensorMap*>(&L.tmap_p),
                  const_cast<EpiParams*>(&L.epi), &xg, const_cast<GwGeom*>(&L.g),
                  const_cast<uint32_t**>(&L.hdr), const_cast<float**>(&L.partials),
                  const_cast<float**>(&L.coefs)};
  return cudaLaunchKernelExC(&cfg, k, args);
}

}  // namespace mhc
