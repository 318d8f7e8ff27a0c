// mhc_pre_gw.cu -- the grid-wide sm_103a forward.
//
// What is computed follows "CANN ops-transformer 中 aclnnMhcPreV2 算子接口
// 全解析" §三 and "aclnnMhcPreSinkhorn 接口与 MhcPreSinkhorn 实现剖析" §3.2;
// how it is laid out on the GPU is this file's own design.
//
// The forward is bound by reading x, and y needs every byte of x a second
// time once the token's gates are known.  The gates need the whole token (a
// reduction over n*D), so the second read only hits L2 if little is loaded
// between a token's first touch and its gates.  Here the CTAs (one per SM,
// all resident: cooperative launch) form ng groups of G; group g takes the
// 64-token tiles k with k % ng == g, and all CTAs of a group work on the
// same tile at about the same time, each on its own slice of d:
//
//  * CTA r of a group owns a contiguous run of 64-wide d-chunks of one
//    stream.  Their phi-plane blocks stay in shared memory for the whole
//    kernel; each tile brings the run as one TMA box (8 KB per chunk,
//    128-byte swizzle): one issue per tile, since a thread issues only a
//    couple of boxes per microsecond whatever their size.
//  * One thread issues tcgen05.mma over the units, M = 128 (tile rows 0..63),
//    N = NP plane rows, fp32 accumulate in TMEM (two buffers).  Two warps add
//    x^2 for their rows from the same boxes, read the accumulators (thread =
//    token = TMEM lane), fold the precision planes and store the CTA's
//    partial sums to a global ring; a signalling thread makes them visible
//    and counts the CTA in, so the publishing warps never wait on the fence.
//  * Local token t of the group's m-th tile is gated by CTA (64m + t) mod G.
//    Two gate warps take alternate tiles: once every CTA of the group has
//    counted in, a gate warp sums the partials in CTA order, computes invRms
//    and the gates, writes the y weights to the ring and counts the token
//    ready.  The Sinkhorn warp runs the tokens of several tiles at once, one
//    per lane, off y's critical path.
//  * One warp waits for each tile to be fully gated and stages its y
//    weights in shared memory; seven warps form y for the CTA's own d-range,
//    loading the tile's x (loaded moments ago by the group: an L2 hit)
//    before the weights are there.
//
// Every wait is bounded by a timer.  A wait that gives up sets the error
// word and a grid-wide abort flag, and every CTA winds down.
#include "mhc_ptx.cuh"

namespace mhc {
namespace {

constexpr int kGwThreads = 512;
// Warp roles.
constexpr int kGwWarpX = 0, kGwWarpMma = 1, kGwWarpSig = 2, kGwWarpSink = 3, kGwWarpPub0 = 4,
              kGwWarpGate0 = 6, kGwWarpY0 = 8;
constexpr int kGwPubThreads = 64;                          // one per tile row (TMEM lanes 0..63)
constexpr int kGwWarpYc0 = kGwWarpY0 + 1;                  // y warps after the weight stager
constexpr int kGwYcWarps = kGwThreads / 32 - kGwWarpYc0;   // 7
constexpr int kGwYcThreads = kGwYcWarps * 32;              // 224
constexpr int kGwGateWarps = 2;
constexpr int kGwPubRing = 4;                              // publish -> signaller hand-off depth
// Named barriers: 1 = the publish warps, 2 = the two gate warps.
constexpr int kGwBarPub = 1, kGwBarGate = 2;

template <int NS, int RR, int P>
struct GwCfg {
  static constexpr int kNP = gw_np(RR, P);                      // MMA N
  static_assert(kNP <= 256, "N of one MMA is at most 256");
  static constexpr int kAccCols = kNP <= 32 ? 32 : kNP <= 64 ? 64 : kNP <= 128 ? 128 : 256;
  static constexpr uint32_t kTmemCols = 2u * kAccCols;          // two accumulators
  static constexpr int kPlaneBytes = plane_box_rows(RR, P) * 128;   // one chunk's plane block
  static constexpr int kStr = partial_stride(RR);               // floats per partial
  static constexpr int kG4 = kStr / 4;                          // float4 groups per partial
  static constexpr int kRounds = kG4 <= 8 ? 3 : 1;              // rounds of CTAs loaded at once
  static constexpr bool kThree = (RR == NS * NS + 2 * NS);
  static constexpr int kYB = NS <= 4 ? 4 : 2;                   // y items in flight per thread
};

struct GwTail {
  uint64_t x_full[kMaxStages], x_empty[kMaxStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t phi_full;
  uint64_t pub_done[kGwPubRing], sig_free[kGwPubRing];
  uint64_t sink_full[2], sink_free[2];
  uint64_t y_prog[kGwSlots];          // a tile of that ring slot is fully gated (seen by the watcher)
  uint64_t ycoef_full[2], ycoef_free[2];   // y weights of a tile staged / consumed
  uint64_t y_done[16];                     // this CTA's y warps finished tile m (index m % 16)
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t abort;
  float gate_half[96];                // single-tile runs: the second gate warp's half sum of a row
};
static_assert(sizeof(GwTail) <= kTailBytes, "barrier block outgrew its reservation");

struct GwCtl {
  volatile uint32_t* abort;    // shared: this CTA is winding down
  volatile uint32_t* gabort;   // global: some CTA gave up
  uint32_t* err;               // global error word
  uint64_t wait_ns;            // how long one wait may take before it gives up
};

__device__ __noinline__ void gw_fail(const GwCtl& c, uint32_t code) {
  atomicOr(c.err, code);
  *c.abort = 1u;
  atomicExch(const_cast<uint32_t*>(c.gabort), 1u);
}

// Wait for phase `parity` of a local mbarrier; gives up after c.wait_ns or
// as soon as this CTA or any other has given up.  A waiting thread sleeps in
// the barrier (woken when the phase completes), so waiting warps leave the
// issue slots to the working ones.
__device__ __noinline__ bool gw_wait(uint64_t* bar, uint32_t parity, const GwCtl& c) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test_sleep(bar, parity, 1000u)) return true;
    if ((it & 7u) == 0) {
      if (*c.abort || *c.gabort) {
        *c.abort = 1u;
        return false;
      }
      if (now_ns() - t0 > c.wait_ns) {
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
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Release at GPU scope: writes this thread made, or saw through a CTA barrier,
// are visible before the count changes.
__device__ __forceinline__ void red_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Wait until a global counter written by other CTAs reaches `target`
// (acquire: what they wrote before counting is visible afterwards).  While
// it is short, poll with plain loads and back off, so a waiting thread does
// not load the SM's memory pipeline; the final read is the acquire.
__device__ __noinline__ bool gw_wait_count(const uint32_t* ctr, uint32_t target, const GwCtl& c) {
  if (ld_acquire_gpu(ctr) >= target) return true;
  const uint64_t t0 = now_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(128);
    if (ld_relaxed_gpu(ctr) >= target) return ld_acquire_gpu(ctr) >= target;
    if ((it & 15u) == 0) {
      if (*c.abort || *c.gabort) {
        *c.abort = 1u;
        return false;
      }
      if (now_ns() - t0 > c.wait_ns) {
        gw_fail(c, kErrGridWait);
        return false;
      }
    }
  }
}

// Lane 0 waits; the result reaches the whole warp, and the warp barrier
// orders the other lanes' later reads after lane 0's acquire (a shuffle
// alone would let the compiler hoist those reads above the wait).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const GwCtl& c) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = gw_wait(bar, parity, c);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  __syncwarp();
  return ok;
}

// First local row t of a tile that CTA r of the group gates: (64m + t) % G == r.
__device__ __forceinline__ int first_owned(int m, int r, int G) {
  return (int)(((long long)r - (long long)m * kGwTile % G + G) % G);
}

template <int NS, int RR, int P>
__global__ void __launch_bounds__(kGwThreads, 1)
    mhc_pre_gw_kernel(const __grid_constant__ CUtensorMap tmap_x, const __nv_bfloat16* __restrict__ planes,
                      const EpiParams ep, const __nv_bfloat16* __restrict__ xg, const GwGeom g, uint32_t* hdr,
                      float* partials, float* coefs) {
  using C = GwCfg<NS, RR, P>;
  constexpr int NN = NS * NS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const GwLayout Ly = gw_layout(NS, RR, P, g.umax, g.xstages);
  const int XS = g.xstages;
  uint8_t* sPhi = smem + Ly.phi;
  uint8_t* sX = smem + Ly.x;
  float* ycoef = reinterpret_cast<float*>(smem + Ly.ycoef);   // [2][64][NS]
  float* sink_buf = reinterpret_cast<float*>(smem + Ly.sink); // [2][kGwSinkMax][NN]
  int* sink_cnt = reinterpret_cast<int*>(smem + Ly.scnt);     // [2][kGwSinkMax]: tokens per tile
  GwTail* tail = reinterpret_cast<GwTail*>(smem + Ly.tail);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = g.G;
  const int grp = blockIdx.x / G;                 // group
  const int r = blockIdx.x - grp * G;             // rank in the group
  const int my_tiles = grp < g.num_tiles ? (g.num_tiles - grp + g.ng - 1) / g.ng : 0;
  const int stream = r / g.gs;                     // this CTA's stream
  const int rs = r - stream * g.gs;
  const int j0 = (int)((long long)rs * g.nch / g.gs);
  const int U = (int)((long long)(rs + 1) * g.nch / g.gs) - j0;   // chunks this CTA owns (>= 1)
  const size_t slot_bytes = (size_t)g.umax * kGwUnitBytes;
  const int SB = g.sink_batch;
  uint32_t* arrive = hdr + kHdrArrive + grp * kGwSlots;
  uint32_t* ready = hdr + kHdrReady + grp * kGwSlots;
  uint32_t* ydone = hdr + kHdrYdone + grp * kGwSlots;
  float* gpart = partials + (size_t)grp * kGwSlots * kGwTile * G * C::kStr;
  float* gcoef = coefs + (size_t)grp * kGwSlots * kGwTile * NS;
  GwCtl ctl{&tail->abort, hdr + kHdrAbort, hdr, g.wt.wait_ns};

  // ---- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < XS; ++s) {
      mbar_init(&tail->x_full[s], 1);
      mbar_init(&tail->x_empty[s], 1 + 2);      // MMA commit + the two sum-of-squares warps
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tail->acc_full[a], 1);
      mbar_init(&tail->acc_empty[a], 2);        // two publish warps
      mbar_init(&tail->sink_full[a], SB);       // one arrival per tile of a batch
      mbar_init(&tail->sink_free[a], 1);
    }
    for (int j = 0; j < kGwPubRing; ++j) {
      mbar_init(&tail->pub_done[j], 2);         // two publish warps
      mbar_init(&tail->sig_free[j], 1);
    }
    for (int j = 0; j < kGwSlots; ++j) mbar_init(&tail->y_prog[j], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tail->ycoef_full[b], 1);
      mbar_init(&tail->ycoef_free[b], kGwYcWarps);
    }
    for (int j = 0; j < 16; ++j) mbar_init(&tail->y_done[j], kGwYcWarps);
    mbar_init(&tail->phi_full, 1);
    mbar_init(&tail->mma_done, 1);
    tail->abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmap_x);
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
    // Lane q issues unit q's box, so the CTA's boxes of one tile go out together.
    // A 4-D x box carries all umax chunks at once (its tail past this CTA's
    // run is the next CTA's data or zero fill, and is not used).  The plane
    // blocks of the run come once, one bulk copy per chunk.
    const uint64_t keep = policy_evict_last();
    const int nbox = g.box4d ? 1 : U;
    const uint32_t xbytes = (uint32_t)((g.box4d ? g.umax : U) * kGwUnitBytes);
    if (lane == 0) mbar_expect_tx(&tail->phi_full, (uint32_t)(U * C::kPlaneBytes));
    __syncwarp();
    if (lane < U)
      bulk_load_hint(sPhi + (size_t)lane * C::kPlaneBytes,
                     planes + ((size_t)(j0 + lane) * NS + stream) * (C::kPlaneBytes / 2), (uint32_t)C::kPlaneBytes,
                     &tail->phi_full, keep);
    int xs = 0;
    uint32_t xph = 0;
    int issued = 0;
    for (int m = 0; m < my_tiles; ++m) {
      if (!warp_wait(&tail->x_empty[xs], xph ^ 1u, ctl)) break;
      // Load no further than xlead tiles ahead of this CTA's y warps, so the
      // bytes loaded between a tile's first read and its re-read for y stay
      // within what L2 keeps.
      if (m >= g.xlead && !warp_wait(&tail->y_done[(m - g.xlead) & 15], (uint32_t)((m - g.xlead) >> 4) & 1u, ctl))
        break;
      if (g.wt.withhold_x && blockIdx.x == 0 && m == my_tiles - 1) break;   // test hook (see WaitTest)
      if (lane == 0) mbar_expect_tx(&tail->x_full[xs], xbytes);
      __syncwarp();
      if (lane < nbox) {
        const int k = grp + m * g.ng;
        uint8_t* dst = sX + (size_t)xs * slot_bytes;
        if (g.box4d)
          tma_load_4d_hint(dst, &tmap_x, &tail->x_full[xs], 0, k * kGwTile, j0, stream, keep);
        else
          tma_load_3d_hint(dst + (size_t)lane * kGwUnitBytes, &tmap_x, &tail->x_full[xs], (j0 + lane) * kChunkK,
                           k * kGwTile, stream, keep);
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
      for (int m = 0; m < my_tiles && ok; ++m) {
        const int acc = m & 1;
        const uint32_t acc_phase = (uint32_t)(m >> 1) & 1u;
        if (!gw_wait(&tail->acc_empty[acc], acc_phase ^ 1u, ctl)) break;
        if (!gw_wait(&tail->x_full[xs], xph, ctl)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * C::kAccCols);
        const uint32_t xb = smem_u32(sX + (size_t)xs * slot_bytes);
        for (int q = 0; q < U; ++q) {
          // A: 128 rows from this unit's 64-row box (rows 64..127 run on into
          // the next box and feed TMEM lanes that are never read).
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
  } else if (warp == kGwWarpPub0 || warp == kGwWarpPub0 + 1) {
    // ================================================= sum of squares + partials
    // Thread = tile row = TMEM lane (warps 4 and 5: lane quarters 0 and 1).
    const int t = threadIdx.x - kGwWarpPub0 * 32;   // 0..63
    const int wq = warp & 3;
    int xs = 0;
    uint32_t xph = 0;
    for (int m = 0; m < my_tiles; ++m) {
      const int acc = m & 1;
      const uint32_t acc_phase = (uint32_t)(m >> 1) & 1u;
      // x^2 over this CTA's chunks, straight from the swizzled boxes.  Lane t
      // reads its row's 16-byte pieces in the order they sit in the 128-byte
      // swizzle (piece c at c ^ (t & 7)), so a warp's loads spread over all
      // banks; the order of a row's pieces does not matter for a sum.
      if (!role_all<kGwBarPub, kGwPubThreads>(gw_wait(&tail->x_full[xs], xph, ctl))) break;
      float s8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) s8[e] = 0.0f;
      const uint8_t* xrow = sX + (size_t)xs * slot_bytes + (size_t)t * 128;
      for (int q = 0; q < U; ++q) {
        uint4 v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)
          v[c] = *reinterpret_cast<const uint4*>(xrow + (size_t)q * kGwUnitBytes + ((c ^ (t & 7)) << 4));
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[c]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h[e]);
            s8[2 * e] = fmaf(f.x, f.x, s8[2 * e]);
            s8[2 * e + 1] = fmaf(f.y, f.y, s8[2 * e + 1]);
          }
        }
      }
      const float ssq = tree_sum<8>(s8);
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->x_empty[xs]);
      if (++xs == XS) { xs = 0; xph ^= 1u; }

      // projection partials from TMEM
      if (!role_all<kGwBarPub, kGwPubThreads>(gw_wait(&tail->acc_full[acc], acc_phase, ctl))) break;
      tc_fence_after();
      float mix[RR];
#pragma unroll
      for (int rr = 0; rr < RR; ++rr) mix[rr] = 0.0f;
      const uint32_t taddr = tmem_base + ((uint32_t)(wq * 32) << 16) + (uint32_t)(acc * C::kAccCols);
#pragma unroll
      for (int gq = 0; gq < C::kNP / 16; ++gq) {
        float v[16];
        tmem_ld16(taddr + gq * 16, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int col = gq * 16 + e;
          if (col < P * RR) mix[col % RR] += v[e];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->acc_empty[acc]);

      // The ring slot is free once every token of the slot's previous tile is
      // gated, as the ring watcher reports.
      const int slot = m % kGwSlots;
      const uint32_t use = (uint32_t)(m / kGwSlots);
      bool ok = true;
      if (t == 0) {
        if (use > 0) ok = gw_wait(&tail->y_prog[slot], (use - 1u) & 1u, ctl);
        if (ok && m >= kGwPubRing)
          ok = gw_wait(&tail->sig_free[m % kGwPubRing], ((uint32_t)(m / kGwPubRing) - 1u) & 1u, ctl);
      }
      if (!role_all<kGwBarPub, kGwPubThreads>(ok)) break;
      float* dst = gpart + (((size_t)slot * kGwTile + t) * G + r) * C::kStr;
#pragma unroll
      for (int e = 0; e < C::kStr; e += 4) {
        float4 v;
        v.x = e < RR ? mix[e] : (e == RR ? ssq : 0.0f);
        v.y = e + 1 < RR ? mix[e + 1] : (e + 1 == RR ? ssq : 0.0f);
        v.z = e + 2 < RR ? mix[e + 2] : (e + 2 == RR ? ssq : 0.0f);
        v.w = e + 3 < RR ? mix[e + 3] : (e + 3 == RR ? ssq : 0.0f);
        __stcg(reinterpret_cast<float4*>(dst + e), v);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->pub_done[m % kGwPubRing]);   // release: this warp's stores
    }
  } else if (warp == kGwWarpSig) {
    // ================================================= count this CTA in
    // One fence covers every tile whose partials are stored by then, so a
    // signaller that fell behind catches up a batch at a time.
    if (lane == 0) {
      for (int m = 0; m < my_tiles;) {
        if (!gw_wait(&tail->pub_done[m % kGwPubRing], (uint32_t)(m / kGwPubRing) & 1u, ctl)) break;
        int last = m;
        while (last + 1 < my_tiles && last + 1 < m + kGwPubRing &&
               mbar_poll(&tail->pub_done[(last + 1) % kGwPubRing], (uint32_t)((last + 1) / kGwPubRing) & 1u))
          ++last;
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        for (int j = m; j <= last; ++j) {
          asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(&arrive[j % kGwSlots]) : "memory");
          mbar_arrive(&tail->sig_free[j % kGwPubRing]);
        }
        m = last + 1;
      }
    } else if (lane == 16) {
      // Ring watcher: marks each tile fully gated as soon as the group has
      // gated it, which frees its ring slot for the tile kGwSlots later (an
      // owner counts a token only after it has read the token's partials).
      for (int m = 0; m < my_tiles; ++m) {
        const int k = grp + m * g.ng;
        const int valid = min(kGwTile, g.T - k * kGwTile);
        const uint32_t target = (uint32_t)(m / kGwSlots) * (uint32_t)kGwTile + (uint32_t)valid;
        if (!gw_wait_count(&ready[m % kGwSlots], target, ctl)) break;
        mbar_arrive(&tail->y_prog[m % kGwSlots]);
      }
    }
  } else if (warp == kGwWarpGate0 || warp == kGwWarpGate0 + 1) {
    // ================================================= gates of the tokens this CTA owns
    const int gidx = warp - kGwWarpGate0;
    // With one tile (decode sizes) the other gate warp has nothing to do:
    // both take tile 0, each adds half of a row's partials (one pass of
    // loads each) and the first adds the second's half, in that order.
    const bool split = my_tiles == 1;
    for (int m = split ? 0 : gidx; m < my_tiles; m += kGwGateWarps) {
      const int k = grp + m * g.ng;
      const int tile0 = k * kGwTile;
      const int valid = min(kGwTile, g.T - tile0);
      const int slot = m % kGwSlots;
      const uint32_t use = (uint32_t)(m / kGwSlots);
      const int first = first_owned(m, r, G);
      const int q = m / SB, sb = q & 1, e0 = (m - q * SB) * g.own_max;
      // the Sinkhorn batch buffer is free once batch q - 2 is done
      if (q >= 2 && (m - q * SB) < kGwGateWarps &&
          !warp_wait(&tail->sink_free[sb], ((uint32_t)(q >> 1) - 1u) & 1u, ctl))
        break;
      int cnt = 0;
      if (first < valid) {
        bool ok = true;
        if (lane == 0) {
          // The slot's previous weights must have been read by every CTA (a
          // plain count: those reads completed before it was taken); the
          // partials of this tile must all be in (acquire).
          const uint32_t yd = use > 0 ? ld_relaxed_gpu(&ydone[slot]) : 0u;
          ok = gw_wait_count(&arrive[slot], (use + 1u) * (uint32_t)G, ctl);
          if (ok && use > 0 && yd < use * (uint32_t)G) ok = gw_wait_count(&ydone[slot], use * (uint32_t)G, ctl);
        }
        // both warps of a split pair leave together if either gave up
        if (split ? !role_all<kGwBarGate, 64>(ok) : !__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
        __syncwarp();                              // the lanes' reads below follow lane 0's acquire
        const int c_lo = split ? gidx * ((G + 1) / 2) : 0;
        const int c_hi = split ? min(G, (gidx + 1) * ((G + 1) / 2)) : G;
        for (int t = first; t < valid; t += G, ++cnt) {
          // Sum the CTAs' partials of row t in a fixed order: lane l adds
          // CTAs c_lo + l, c_lo + l + 32, ... then a fixed butterfly adds the
          // lanes.
          const float* src = gpart + ((size_t)slot * kGwTile + t) * G * C::kStr;
          float acc[C::kStr];
#pragma unroll
          for (int e = 0; e < C::kStr; ++e) acc[e] = 0.0f;
          for (int rd0 = 0; c_lo + rd0 * 32 < c_hi; rd0 += C::kRounds) {
            // kRounds rounds of CTAs per pass: every load of the pass is
            // issued before the first add
            float4 v[C::kRounds][C::kG4];
#pragma unroll
            for (int h = 0; h < C::kRounds; ++h) {
              const int c = c_lo + lane + 32 * (rd0 + h);
              const float4* s4 = reinterpret_cast<const float4*>(src + (size_t)(c < c_hi ? c : 0) * C::kStr);
#pragma unroll
              for (int q4 = 0; q4 < C::kG4; ++q4)
                v[h][q4] = c < c_hi ? __ldcg(s4 + q4) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
#pragma unroll
            for (int h = 0; h < C::kRounds; ++h) {
#pragma unroll
              for (int q4 = 0; q4 < C::kG4; ++q4) {
                acc[4 * q4] += v[h][q4].x;
                acc[4 * q4 + 1] += v[h][q4].y;
                acc[4 * q4 + 2] += v[h][q4].z;
                acc[4 * q4 + 3] += v[h][q4].w;
              }
            }
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
            for (int e = 0; e <= RR; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
          }
          if (split) {
            if (gidx == 1 && lane == 0) {
#pragma unroll
              for (int e = 0; e <= RR; ++e) tail->gate_half[e] = acc[e];
            }
            role_sync<kGwBarGate, 64>();           // the second half is in
            if (gidx == 0 && lane == 0) {
#pragma unroll
              for (int e = 0; e <= RR; ++e) acc[e] += tail->gate_half[e];
            }
            role_sync<kGwBarGate, 64>();           // and read before the next row overwrites it
            if (gidx == 1) continue;
          }
          if (lane == 0) {
            // gates and logits first: the Sinkhorn warp may start as soon as
            // the tile's logits are in; the y weights are counted ready once
            // for the tile, after the loop
            float mix[RR];
#pragma unroll
            for (int e = 0; e < RR; ++e) mix[e] = acc[e];
            const int tok = tile0 + t;
            float cf[NS];
            const float inv_rms = token_gates<NS, RR>(ep, tok, mix, acc[RR], true, cf);
            float H[NN];
            residual_logits<NS, RR>(ep, mix, inv_rms, H);
            float* eb = sink_buf + ((size_t)sb * kGwSinkMax + e0 + cnt) * NN;
#pragma unroll
            for (int i = 0; i < NN; ++i) eb[i] = H[i];
            float* cdst = gcoef + ((size_t)slot * kGwTile + t) * NS;
#pragma unroll
            for (int i = 0; i < NS; ++i) __stcg(cdst + i, cf[i]);
          }
        }
      }
      if (split && gidx == 1) break;               // the helper warp is done
      __syncwarp();
      if (lane == 0) {
        sink_cnt[sb * kGwSinkMax + (m - q * SB)] = cnt;
        mbar_arrive(&tail->sink_full[sb]);
        if (m == my_tiles - 1) {             // a short last batch: complete its phase
          for (int extra = m - q * SB + 1; extra < SB; ++extra) mbar_arrive(&tail->sink_full[sb]);
        }
        // this tile's y weights, stored above, become visible with the count
        if (cnt > 0) red_release_gpu(&ready[slot], (uint32_t)cnt);
      }
    }
  } else if (warp == kGwWarpSink) {
    // ================================================= Sinkhorn for comb, a batch of tiles at once
    const int batches = (my_tiles + SB - 1) / SB;
    for (int q = 0; q < batches; ++q) {
      const int sb = q & 1;
      if (!warp_wait(&tail->sink_full[sb], (uint32_t)(q >> 1) & 1u, ctl)) break;
      int total = 0;                               // tokens this CTA owns in the batch
      for (int mt = 0; mt < SB && q * SB + mt < my_tiles; ++mt) total += sink_cnt[sb * kGwSinkMax + mt];
      if (total == 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&tail->sink_free[sb]);
        continue;
      }
      const int mt = lane / g.own_max, o = lane - mt * g.own_max;   // lane -> (tile of batch, token)
      const int m = q * SB + mt;
      if (mt < SB && m < my_tiles && o < sink_cnt[sb * kGwSinkMax + mt]) {
        const int k = grp + m * g.ng;
        const int t = first_owned(m, r, G) + o * G;
        token_sinkhorn<NS, C::kThree>(ep, k * kGwTile + t,
                                      sink_buf + ((size_t)sb * kGwSinkMax + mt * g.own_max + o) * NN, true);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->sink_free[sb]);
    }
  } else if (warp == kGwWarpY0) {
    // ================================================= y weights of each tile
    // Waits until every token of the tile is gated, copies the weights into
    // one of two shared buffers for the y warps and counts this CTA done with
    // the slot.  A thread without loads of its own in flight does the
    // acquiring poll, so the poll costs one round trip.
    for (int m = 0; m < my_tiles; ++m) {
      const int k = grp + m * g.ng;
      const int valid = min(kGwTile, g.T - k * kGwTile);
      const int slot = m % kGwSlots;
      const uint32_t use = (uint32_t)(m / kGwSlots);
      const int b = m & 1;
      if (m >= 2 && !warp_wait(&tail->ycoef_free[b], ((uint32_t)(m >> 1) - 1u) & 1u, ctl)) break;
      bool ok = true;
      if (lane == 0) ok = gw_wait_count(&ready[slot], use * (uint32_t)kGwTile + (uint32_t)valid, ctl);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      __syncwarp();                                // the lanes' reads below follow lane 0's acquire
      const float* csrc = gcoef + (size_t)slot * kGwTile * NS;
      float* cdst = ycoef + (size_t)b * kGwTile * NS;
      // every load in flight before the first store (one round trip)
      constexpr int kPer = (kGwTile * NS + 31) / 32;
      float cv[kPer];
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        const int e = lane + 32 * q;
        cv[q] = e < valid * NS ? __ldcg(csrc + e) : 0.0f;
      }
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        const int e = lane + 32 * q;
        if (e < valid * NS) cdst[e] = cv[q];
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&tail->ycoef_full[b]);
        atomicAdd(&ydone[slot], 1u);            // the slot's weights are no longer needed here
      }
    }
  } else if (warp >= kGwWarpYc0) {
    // ================================================= y for this CTA's d-range
    const int yt = threadIdx.x - kGwWarpYc0 * 32;
    const int nvec = g.D >> 3;                      // 16-byte vectors per row
    const int v0 = (int)((long long)r * nvec / G);
    const int nv = (int)((long long)(r + 1) * nvec / G) - v0;
    const int nvd = nv > 0 ? nv : 1;
    const uint64_t read_policy = policy_evict_first();
    for (int m = 0; m < my_tiles; ++m) {
      const int k = grp + m * g.ng;
      const int tile0 = k * kGwTile;
      const int valid = min(kGwTile, g.T - tile0);
      const int items = valid * nv;
      const int b = m & 1;
      const float* w = ycoef + (size_t)b * kGwTile * NS;
      const __nv_bfloat16* xt = xg + (size_t)tile0 * NS * g.D;
      __nv_bfloat16* yo = ep.y + (size_t)tile0 * g.D;
      // The first batch of x loads goes out before the weights are known.
      uint4 xv[C::kYB][NS];
      int rowv[C::kYB], dv[C::kYB];
      auto load_batch = [&](int base) {
#pragma unroll
        for (int q = 0; q < C::kYB; ++q) {
          const int it = base + q * kGwYcThreads;
          const int row = it / nvd;
          rowv[q] = it < items ? row : -1;
          dv[q] = (v0 + (it - row * nvd)) * 8;
          if (it < items) {
            const __nv_bfloat16* src = xt + (size_t)row * NS * g.D + dv[q];
#pragma unroll
            for (int i = 0; i < NS; ++i) xv[q][i] = ld_global_v4_hint(src + (size_t)i * g.D, read_policy);
          }
        }
      };
      auto apply_batch = [&]() {
#pragma unroll
        for (int q = 0; q < C::kYB; ++q) {
          if (rowv[q] < 0) continue;
          float acc8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc8[e] = 0.0f;
#pragma unroll
          for (int i = 0; i < NS; ++i) {
            const float wi = w[rowv[q] * NS + i];
            const __nv_bfloat162* hh = reinterpret_cast<const __nv_bfloat162*>(&xv[q][i]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(hh[e]);
              acc8[2 * e] = fmaf(wi, f.x, acc8[2 * e]);
              acc8[2 * e + 1] = fmaf(wi, f.y, acc8[2 * e + 1]);
            }
          }
          uint4 o;
          __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
          for (int e = 0; e < 4; ++e) ob[e] = __floats2bfloat162_rn(acc8[2 * e], acc8[2 * e + 1]);
          st_global_v4_hint(yo + (size_t)rowv[q] * g.D + dv[q], o, read_policy);
        }
      };
      load_batch(yt);
      if (m + 1 < my_tiles) {
        // bring the next tile's rows into L2 while this one waits for its weights
        const int k1 = k + g.ng;
        const int valid1 = min(kGwTile, g.T - k1 * kGwTile);
        const __nv_bfloat16* x1 = xg + (size_t)k1 * kGwTile * NS * g.D + (size_t)v0 * 8;
        for (int e = yt; e < valid1 * NS; e += kGwYcThreads)
          for (int v = 0; v < nv; v += 8)
            asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(x1 + (size_t)e * g.D + v * 8));
      }
      if (!warp_wait(&tail->ycoef_full[b], (uint32_t)(m >> 1) & 1u, ctl)) break;
      apply_batch();
      for (int base = yt + kGwYcThreads * C::kYB; base < items; base += kGwYcThreads * C::kYB) {
        load_batch(base);
        apply_batch();
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&tail->ycoef_free[b]);
        mbar_arrive(&tail->y_done[m & 15]);
      }
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
  cfg.gridDim = dim3(L.g.ng * L.g.G, 1, 1);
  cfg.blockDim = dim3(kGwThreads, 1, 1);
  cfg.dynamicSmemBytes = L.smem_bytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const __nv_bfloat16* xg = static_cast<const __nv_bfloat16*>(L.x);
  const __nv_bfloat16* planes = L.planes;
  void* args[] = {const_cast<CUtensorMap*>(&L.tmap_x), const_cast<__nv_bfloat16**>(&planes),
                  const_cast<EpiParams*>(&L.epi), &xg, const_cast<GwGeom*>(&L.g),
                  const_cast<uint32_t**>(&L.hdr), const_cast<float**>(&L.partials),
                  const_cast<float**>(&L.coefs)};
  return cudaLaunchKernelExC(&cfg, k, args);
}

}  // namespace mhc
