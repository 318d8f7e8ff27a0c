// mhc_pre_tc.cu -- the sm_103a forward: TMA x tiles, tcgen05 projection into
// TMEM, register epilogue (RMS, gates, Sinkhorn) and the weighted sum y.
//
// What is computed follows "CANN ops-transformer 中 aclnnMhcPreV2 算子接口
// 全解析" §三 and "aclnnMhcPreSinkhorn 接口与 MhcPreSinkhorn 实现剖析" §3.2;
// how it is laid out on the GPU is this file's own design:
//
//  * A token tile is 128 tokens (the MMA's M, one TMEM lane per token).  A
//    cluster of C CTAs shares one tile; CTA c owns a contiguous range of
//    64-wide d-chunks and streams those chunks of all n streams, so each
//    byte of x is read from HBM once per tile and the tile's footprint per
//    SM stays small enough for the later re-read to hit L2.
//  * Per chunk, TMA brings x[128 tokens][64] (bf16, 128-byte swizzle) and the
//    matching 64 columns of the stacked phi planes [NP][64]; one thread issues
//    four tcgen05.mma (K = 16 each), M = 128, N = NP, fp32 accumulate in TMEM.
//  * Two warps sum x^2 for their token rows from the same shared-memory tile.
//  * Four epilogue warps read the accumulators (thread = token), fold the
//    precision planes, exchange per-CTA partial sums through distributed
//    shared memory, run gates + Sinkhorn for the rows this CTA owns, publish
//    the y weights to every CTA of the cluster, then form y for the CTA's
//    d-range by re-reading x (now in L2).
//  * Every wait is bounded by a timer; a wait that gives up sets the error
//    word in the workspace and the kernel winds down instead of hanging.
#include "mhc_common.cuh"

namespace mhc {
namespace {

constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per wait before giving up

// ----------------------------------------------------------------- PTX glue
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Arrive on the barrier at the same offset in CTA `rank` of this cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint64_t* bar, uint32_t rank) {
  asm volatile(
      "{\n\t.reg .b32 ra;\n\t"
      "mapa.shared::cluster.u32 ra, %0, %1;\n\t"
      "mbarrier.arrive.release.cluster.shared::cluster.b64 _, [ra];\n\t}" ::"r"(smem_u32(bar)),
      "r"(rank)
      : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_test_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

struct Ctl {
  volatile uint32_t* abort;   // shared: set once any wait in this CTA gave up
  uint32_t* err;              // global error word
};

// Wait for phase `parity` of `bar`.  Returns false (and raises the abort flag
// and error word) after kWaitNs, or as soon as another role has aborted.
template <bool kCluster>
__device__ __noinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Ctl& c, uint32_t code) {
  if (kCluster ? mbar_test_cluster(bar, parity) : mbar_test(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  for (uint32_t it = 1;; ++it) {
    if (kCluster ? mbar_test_cluster(bar, parity) : mbar_test(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*c.abort) return false;
      if (now_ns() - t0 > kWaitNs) {
        atomicOr(c.err, code);
        *c.abort = 1u;
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// K-major operand tile with 128-byte swizzle: rows of 128 bytes, 8-row
// groups 1024 bytes apart (the layout TMA writes for a 64 x rows bf16 box).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
  d |= static_cast<uint64_t>(1) << 16;                    // leading offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride between 8-row groups
  d |= static_cast<uint64_t>(1) << 46;                    // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                    // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: bf16 x bf16 -> fp32, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes; the wait is part
// of the same statement so no use of the registers can be hoisted above it.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15},"
      " [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ float ld_dsmem_f32(const float* local, uint32_t rank) {
  float v;
  asm volatile(
      "{\n\t.reg .b32 ra;\n\t"
      "mapa.shared::cluster.u32 ra, %1, %2;\n\t"
      "ld.shared::cluster.f32 %0, [ra];\n\t}"
      : "=f"(v)
      : "r"(smem_u32(local)), "r"(rank)
      : "memory");
  return v;
}
__device__ __forceinline__ void st_dsmem_f32(float* local, uint32_t rank, float v) {
  asm volatile(
      "{\n\t.reg .b32 ra;\n\t"
      "mapa.shared::cluster.u32 ra, %0, %1;\n\t"
      "st.shared::cluster.f32 [ra], %2;\n\t}" ::"r"(smem_u32(local)),
      "r"(rank), "f"(v)
      : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ void epi_bar_sync() {   // the four epilogue warps only
  asm volatile("bar.sync 1, 128;" ::: "memory");
}
// Barrier among the four epilogue warps that also ANDs a flag across them, so
// a wait that gave up in one thread makes all 128 leave together.
__device__ __forceinline__ bool epi_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok)
      : "memory");
  return r != 0;
}

// ------------------------------------------------------------ kernel body
struct Geometry {
  int T, n, D, K;
  int num_tiles, nd;           // token tiles; 64-wide d-chunks per stream
  int cluster, stages, np;
};

template <int NS, int RR, int P>
struct Cfg {
  static constexpr int kNP = ((P * RR + 15) / 16) * 16;
  static_assert(kNP <= 256, "N of one MMA is at most 256");
  static constexpr int kAccCols = kNP <= 32 ? 32 : kNP <= 64 ? 64 : kNP <= 128 ? 128 : 256;
  static constexpr uint32_t kTmemCols = 2 * kAccCols;   // two accumulator buffers
  static constexpr int kABytes = kTileM * 128;           // 16 KB
  static constexpr int kBBytes = kNP * 128;
  static constexpr int kPartStride = RR + 1;             // odd: conflict-free rows
};

struct SmemTail {                 // after the stage buffers
  uint64_t full[8], empty[8];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t ssq_full[2], ssq_empty[2];
  uint64_t part_full, coef_full;
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t abort;
};

template <int NS, int RR, int P>
__global__ void __launch_bounds__(kThreads, 1)
    mhc_pre_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                      const EpiParams ep, const __nv_bfloat16* __restrict__ xg, Geometry g, uint32_t* err) {
  using C = Cfg<NS, RR, P>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // Align the dynamic window to 1024 bytes (swizzle atoms).
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = g.stages;
  uint8_t* sA = smem;
  uint8_t* sB = sA + (size_t)S * C::kABytes;
  float* part = reinterpret_cast<float*>(sB + (size_t)S * C::kBBytes);     // [128][RR+1]
  float* ssq_buf = part + kTileM * C::kPartStride;                         // [2][128]
  float* coef_buf = ssq_buf + 2 * kTileM;                                  // [2][128][NS]
  SmemTail* tail = reinterpret_cast<SmemTail*>(
      (reinterpret_cast<uintptr_t>(coef_buf + 2 * kTileM * NS) + 15) & ~uintptr_t(15));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int CL = g.cluster;
  const uint32_t rank = CL > 1 ? cluster_rank() : 0u;
  const int cluster_id = blockIdx.x / CL;
  const int num_clusters = gridDim.x / CL;
  const int c0 = (int)((long long)rank * g.nd / CL);
  const int c1 = (int)((long long)(rank + 1) * g.nd / CL);
  const int my_chunks_per_stream = c1 - c0;
  const int chunks_per_tile = NS * my_chunks_per_stream;
  Ctl ctl{&tail->abort, err};

  // ---- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&tail->full[s], 1);
      mbar_init(&tail->empty[s], 1 + 2);        // MMA commit + two sum-of-squares warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tail->acc_full[b], 1);
      mbar_init(&tail->acc_empty[b], 4);
      mbar_init(&tail->ssq_full[b], 2);
      mbar_init(&tail->ssq_empty[b], 4);
    }
    mbar_init(&tail->part_full, CL);
    mbar_init(&tail->coef_full, CL);
    mbar_init(&tail->mma_done, 1);
    tail->abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_w);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tail->tmem_base)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  if (CL > 1) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = tail->tmem_base;

  if (warp == 0) {
    // ================================================= TMA producer
    if (lane == 0) {
      const uint32_t tx = C::kABytes + C::kBBytes;
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = cluster_id; tile < g.num_tiles && ok; tile += num_clusters) {
        for (int q = 0; q < chunks_per_tile; ++q) {
          const int i = q / my_chunks_per_stream;
          const int j = c0 + (q - i * my_chunks_per_stream);
          if (!wait_bar<false>(&tail->empty[stage], phase ^ 1u, ctl, kErrWaitTimeout)) { ok = false; break; }
          mbar_expect_tx(&tail->full[stage], tx);
          tma_load_3d(sA + (size_t)stage * C::kABytes, &tmap_x, &tail->full[stage], j * kChunkK, i,
                      tile * kTileM);
          tma_load_3d(sB + (size_t)stage * C::kBBytes, &tmap_w, &tail->full[stage], j * kChunkK, i, 0);
          ++issued;
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      // Let every copy this thread started land before the CTA can exit.
      const long long pending = issued < S ? issued : S;
      for (long long k = 0; k < pending; ++k) {
        if (--stage < 0) { stage = S - 1; phase ^= 1u; }
        wait_bar<false>(&tail->full[stage], phase, ctl, kErrWaitTimeout);
      }
    }
  } else if (warp == 1) {
    // ================================================= MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kTileM, C::kNP);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = cluster_id; tile < g.num_tiles && ok; tile += num_clusters) {
        if (!wait_bar<false>(&tail->acc_empty[acc], acc_phase ^ 1u, ctl, kErrWaitTimeout)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * C::kAccCols);
        for (int q = 0; q < chunks_per_tile; ++q) {
          if (!wait_bar<false>(&tail->full[stage], phase, ctl, kErrWaitTimeout)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + (size_t)stage * C::kABytes);
          const uint32_t b0 = smem_u32(sB + (size_t)stage * C::kBBytes);
#pragma unroll
          for (int kk = 0; kk < kChunkK / 16; ++kk) {
            mma_bf16(d_tmem, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc,
                     (q > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&tail->empty[stage]);       // frees the stage when these MMAs finish
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&tail->acc_full[acc]);          // accumulator complete
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      mma_commit(&tail->mma_done);
      wait_bar<false>(&tail->mma_done, 0, ctl, kErrWaitTimeout);
    }
  } else if (warp < 4) {
    // ================================================= sum of squares
    const int q = threadIdx.x - 64;                // rows q and q + 64
    int stage = 0;
    uint32_t phase = 0;
    int b = 0;
    uint32_t bphase = 0;
    bool ok = true;
    for (int tile = cluster_id; tile < g.num_tiles && ok; tile += num_clusters) {
      if (!__all_sync(0xffffffffu, wait_bar<false>(&tail->ssq_empty[b], bphase ^ 1u, ctl, kErrWaitTimeout)))
        break;
      float s0 = 0.0f, s1 = 0.0f;
      for (int c = 0; c < chunks_per_tile; ++c) {
        if (!__all_sync(0xffffffffu, wait_bar<false>(&tail->full[stage], phase, ctl, kErrWaitTimeout))) {
          ok = false;
          break;
        }
        const uint8_t* tileA = sA + (size_t)stage * C::kABytes;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = q + 64 * h;
          float acc = 0.0f;
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            // Rotate the 16-byte column by row so a warp's loads hit distinct banks.
            const int col = (p + row) & 7;
            const uint4 v = *reinterpret_cast<const uint4*>(tileA + row * 128 + col * 16);
            const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(hv[e]);
              acc = fmaf(f.x, f.x, acc);
              acc = fmaf(f.y, f.y, acc);
            }
          }
          if (h == 0) s0 += acc; else s1 += acc;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&tail->empty[stage]);
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      ssq_buf[b * kTileM + q] = s0;
      ssq_buf[b * kTileM + q + 64] = s1;
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->ssq_full[b]);
      if (++b == 2) { b = 0; bphase ^= 1u; }
    }
  } else {
    // ================================================= epilogue + y
    const int et = threadIdx.x - 128;              // 0..127 = TMEM lane = tile row
    const int wq = warp & 3;                       // TMEM lane quarter of this warp
    const int r0 = (int)((long long)rank * kTileM / CL);
    const int r1 = (int)((long long)(rank + 1) * kTileM / CL);
    const int dlo = c0 * kChunkK;
    const int dhi = min(c1 * kChunkK, g.D);
    const int w8 = (dhi - dlo) >> 3;               // 16-byte vectors per row
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t k = 0;                                // tiles done by this cluster member
    for (int tile = cluster_id; tile < g.num_tiles; tile += num_clusters, ++k) {
      // --- accumulators and sum of squares for row et
      if (!epi_all(wait_bar<false>(&tail->acc_full[acc], acc_phase, ctl, kErrWaitTimeout))) break;
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
      const int b = (int)(k & 1u);
      if (!epi_all(wait_bar<false>(&tail->ssq_full[b], (k >> 1) & 1u, ctl, kErrWaitTimeout))) break;
      float ssq = ssq_buf[b * kTileM + et];
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->ssq_empty[b]);
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }

      const int tok = tile * kTileM + et;
      float* coef = coef_buf + (size_t)(k & 1u) * kTileM * NS;
      if (CL == 1) {
        float cf[NS];
        token_epilogue<NS, RR>(ep, tok, mix, ssq, tok < g.T, cf);
#pragma unroll
        for (int i = 0; i < NS; ++i) coef[et * NS + i] = cf[i];
        epi_bar_sync();
      } else {
        // --- publish this CTA's partial sums, then reduce the rows it owns
        float* my = part + et * C::kPartStride;
#pragma unroll
        for (int r = 0; r < RR; ++r) my[r] = mix[r];
        my[RR] = ssq;
        epi_bar_sync();
        if (et == 0) {
          asm volatile("fence.acq_rel.cluster;" ::: "memory");
          for (int cr = 0; cr < CL; ++cr) mbar_arrive_remote(&tail->part_full, (uint32_t)cr);
        }
        if (!epi_all(wait_bar<true>(&tail->part_full, k & 1u, ctl, kErrClusterWait))) break;
        if (et >= r0 && et < r1) {
          float tot[RR];
          float tssq = 0.0f;
#pragma unroll
          for (int r = 0; r < RR; ++r) tot[r] = 0.0f;
          for (int cr = 0; cr < CL; ++cr) {
#pragma unroll
            for (int r = 0; r < RR; ++r) tot[r] += ld_dsmem_f32(my + r, (uint32_t)cr);
            tssq += ld_dsmem_f32(my + RR, (uint32_t)cr);
          }
          float cf[NS];
          token_epilogue<NS, RR>(ep, tok, tot, tssq, tok < g.T, cf);
          for (int cr = 0; cr < CL; ++cr) {
#pragma unroll
            for (int i = 0; i < NS; ++i) st_dsmem_f32(coef + et * NS + i, (uint32_t)cr, cf[i]);
          }
        }
        epi_bar_sync();
        if (et == 0) {
          asm volatile("fence.acq_rel.cluster;" ::: "memory");
          for (int cr = 0; cr < CL; ++cr) mbar_arrive_remote(&tail->coef_full, (uint32_t)cr);
        }
        if (!epi_all(wait_bar<true>(&tail->coef_full, k & 1u, ctl, kErrClusterWait))) break;
      }

      // --- y for this CTA's d-range: re-read x (L2), weights from shared memory
      const int rows = min(kTileM, g.T - tile * kTileM);
      const int items = rows * w8;
      for (int it = et; it < items; it += 128) {
        const int row = it / w8;
        const int v = it - row * w8;
        const size_t t = (size_t)tile * kTileM + row;
        float cf[NS];
#pragma unroll
        for (int i = 0; i < NS; ++i) cf[i] = coef[row * NS + i];
        weighted_sum8<NS>(xg + t * (size_t)g.K, g.D, dlo + 8 * v, cf, ep.y + t * (size_t)g.D);
      }
      epi_bar_sync();
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(C::kTmemCols)
                 : "memory");
  }
  if (CL > 1) cluster_sync_all();
}

template <int NS, int RR, int P>
const void* kernel_ptr() {
  return reinterpret_cast<const void*>(&mhc_pre_tc_kernel<NS, RR, P>);
}

const void* select_kernel(int n, int R, int P) {
#define MHC_CASE(NS_, RR_, P_) \
  if (n == NS_ && R == RR_ && P == P_) return kernel_ptr<NS_, RR_, P_>();
  MHC_CASE(4, 24, 3) MHC_CASE(4, 24, 2) MHC_CASE(4, 8, 3) MHC_CASE(4, 8, 2)
  MHC_CASE(6, 48, 3) MHC_CASE(6, 48, 2) MHC_CASE(6, 12, 3) MHC_CASE(6, 12, 2)
  MHC_CASE(8, 80, 3) MHC_CASE(8, 80, 2) MHC_CASE(8, 16, 3) MHC_CASE(8, 16, 2)
#undef MHC_CASE
  return nullptr;
}

}  // namespace

int tc_np(int R, int P) { return ((P * R + 15) / 16) * 16; }

cudaError_t tc_forward_occupancy(int n, int R, int P, size_t smem_bytes, int cluster, int* max_clusters) {
  *max_clusters = 0;
  const void* k = select_kernel(n, R, P);
  if (!k) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
  if (e != cudaSuccess) return e;
  if (cluster > 8) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(cluster, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(max_clusters, k, &cfg);
}

cudaError_t launch_tc_forward(const TcLaunch& L, cudaStream_t s) {
  const int n = L.epi.n, R = L.epi.R;
  const void* k = select_kernel(n, R, L.P);
  if (!k) return cudaErrorInvalidValue;
  Geometry g;
  g.T = L.epi.T;
  g.n = n;
  g.D = L.epi.D;
  g.K = n * L.epi.D;
  g.num_tiles = (L.epi.T + kTileM - 1) / kTileM;
  g.nd = (L.epi.D + kChunkK - 1) / kChunkK;
  g.cluster = L.cluster;
  g.stages = L.stages;
  g.np = L.NP;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = L.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(L.grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = L.smem_bytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const __nv_bfloat16* xg = static_cast<const __nv_bfloat16*>(L.x);
  void* args[] = {const_cast<CUtensorMap*>(&L.tmap_x), const_cast<CUtensorMap*>(&L.tmap_w),
                  const_cast<EpiParams*>(&L.epi), &xg, &g, const_cast<uint32_t**>(&L.err_word)};
  return cudaLaunchKernelExC(&cfg, k, args);
}

}  // namespace mhc
