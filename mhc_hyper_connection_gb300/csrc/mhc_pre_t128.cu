// mhc_pre_t128.cu -- the sm_103a forward for n = 4 with 128-token tiles.
//
// What is computed follows "CANN ops-transformer 中 aclnnMhcPreV2 算子接口
// 全解析" §三 and "aclnnMhcPreSinkhorn 接口与 MhcPreSinkhorn 实现剖析" §3.2;
// how it is laid out on the GPU is this file's own design.
//
// Same structure as the 64-token cluster kernel (mhc_pre_tc.cu) -- clusters
// of C CTAs share a token tile, CTA c owns a range of 64-wide d-chunks of
// all streams, partial sums meet in distributed shared memory -- with a
// tile of 128 tokens, which fills the M = 128 rows of every tcgen05.mma:
//
//  * x boxes are (64 columns, 128 tokens, 2 streams) = 32 KB; per stream of
//    a chunk the projection is 4 MMAs (K = 16 each), N = NP.  Per token that
//    is a quarter of the MMA instructions of the 64-token kernel, whose
//    single issuing thread bounds how fast a chunk can pass.
//  * The sum of squares comes from CUDA cores: the four publish warps
//    (thread = token = TMEM lane) add x^2 of their row from every x box
//    before it is released, reading the row's 16-byte pieces in the order
//    the 128-byte swizzle put them, so a warp's loads spread over all banks.
//  * The phi planes arrive as pre-swizzled blocks by linear bulk copy.
//  * Gates and y are as in the 64-token kernel: the owner of a row sums the
//    members' partials in rank order (deterministic), gates it and sends the
//    y weights to every member, then runs the row's Sinkhorn (off y's path:
//    the weights are already out); eight warps form y for this CTA's d-range
//    by re-reading x.
//
// Every wait is bounded by a timer; a wait that gives up sets the error word
// in the workspace and the kernel winds down instead of hanging.
#include "mhc_ptx.cuh"

namespace mhc {
namespace {

constexpr int kT = kT128Tile;          // tokens per tile = MMA M = TMEM lanes
constexpr int kSGt = 2;                // streams per x box
constexpr int kXBoxBytes = kSGt * kT * 128;   // 32 KB
// Warp roles.
constexpr int kW_X = 0, kW_MMA = 1, kW_W = 2, kW_GATE = 3, kW_PUB0 = 4, kW_Y0 = 8;
constexpr int kPubThr = 128;
constexpr int kYThr = kThreads - kW_Y0 * 32;   // 256
// Named barriers: 1 = publish warps, 2 = y warps.
constexpr int kBarP = 1, kBarYt = 2;

template <int RR, int P>
struct T128Cfg {
  static constexpr int NS = 4;
  static constexpr int kNP = ((P * RR + 15) / 16) * 16;          // MMA N of the projection
  static_assert(kNP <= 256, "N of one MMA is at most 256");
  static constexpr int kAccCols = kNP <= 32 ? 32 : kNP <= 64 ? 64 : kNP <= 128 ? 128 : 256;
  static constexpr uint32_t kTmemCols = 2u * kAccCols;           // two accumulators
  static constexpr int kGroups = NS / kSGt;                      // x boxes per d-chunk
  static constexpr int kWRows = plane_box_rows(RR, P);
  static constexpr int kWG = w_group(NS, RR, P);                 // streams per phi block run
  static constexpr int kWBoxes = NS / kWG;                       // phi runs per d-chunk
  static constexpr int kWBytes = kWG * kWRows * 128;
  static constexpr int kStr = partial_stride(RR);                // floats per published partial
  static constexpr bool kThree = (RR == NS * NS + 2 * NS);
  static constexpr int kYBatch = 4;                              // y items in flight per thread
};

struct T128Tail {
  uint64_t x_full[kMaxStages], x_empty[kMaxStages];
  uint64_t w_full[kMaxStages], w_empty[kMaxStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t part_full, part_free;
  uint64_t coef_full[kCoefBufs], coef_free[kCoefBufs];
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t abort;
};
static_assert(sizeof(T128Tail) <= kTailBytes, "barrier block outgrew its reservation");

template <int RR, int P>
__global__ void __launch_bounds__(kThreads, 1)
    mhc_pre_t128_kernel(const __grid_constant__ CUtensorMap tmap_x, const __nv_bfloat16* __restrict__ planes,
                        const EpiParams ep, const __nv_bfloat16* __restrict__ xg, Geometry g, uint32_t* err) {
  using C = T128Cfg<RR, P>;
  constexpr int NS = C::NS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const SmemLayout Ly = t128_layout(RR, P, g.xstages, g.wstages);
  const int XS = g.xstages, WS = g.wstages;
  uint8_t* sX = smem + Ly.x;
  uint8_t* sW = smem + Ly.w;
  float* recv = reinterpret_cast<float*>(smem + Ly.part);     // [CL][128/CL][kStr]
  float* owned = recv + (size_t)kT * C::kStr;                 // [128/CL][kStr] summed partials
  float* coef_buf = reinterpret_cast<float*>(smem + Ly.coef); // [kCoefBufs][128][NS]
  T128Tail* tail = reinterpret_cast<T128Tail*>(smem + Ly.tail);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int CL = g.cluster;
  const uint32_t rank = cluster_rank();
  const int cluster_id = blockIdx.x / CL;
  const int num_clusters = gridDim.x / CL;
  const int c0 = (int)((long long)rank * g.nd / CL);
  const int c1 = (int)((long long)(rank + 1) * g.nd / CL);
  const int rpo = kT / CL;                        // tile rows each member reduces (owns)
  Ctl ctl{&tail->abort, err};

  // ---- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < XS; ++s) {
      mbar_init(&tail->x_full[s], 1);
      mbar_init(&tail->x_empty[s], 1 + 4);      // MMA commit + the four sum-of-squares warps
    }
    for (int s = 0; s < WS; ++s) {
      mbar_init(&tail->w_full[s], 1);
      mbar_init(&tail->w_empty[s], 1);          // MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tail->acc_full[b], 1);
      mbar_init(&tail->acc_empty[b], 4);        // four publish warps
    }
    for (int b = 0; b < kCoefBufs; ++b) {
      mbar_init(&tail->coef_full[b], CL);
      mbar_init(&tail->coef_free[b], CL);
    }
    mbar_init(&tail->part_full, CL);            // one arrival per cluster member
    mbar_init(&tail->part_free, CL);
    mbar_init(&tail->mma_done, 1);
    tail->abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmap_x);
  }
  if (warp == kW_MMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tail->tmem_base)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = tail->tmem_base;

  if (warp == kW_X) {
    // ================================================= x producer (HBM)
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();
      int xs = 0;
      uint32_t xph = 0;
      long long iss = 0;
      bool ok = true;
      for (int tile = cluster_id; tile < g.num_tiles && ok; tile += num_clusters) {
        for (int j = c0; j < c1 && ok; ++j) {
          for (int grp = 0; grp < C::kGroups; ++grp) {
            if (!wait_bar<false>(&tail->x_empty[xs], xph ^ 1u, ctl, kErrWaitTimeout)) { ok = false; break; }
            mbar_expect_tx(&tail->x_full[xs], (uint32_t)kXBoxBytes);
            tma_load_3d_hint(sX + (size_t)xs * kXBoxBytes, &tmap_x, &tail->x_full[xs], j * kChunkK, tile * kT,
                             grp * kSGt, keep);
            ++iss;
            if (++xs == XS) { xs = 0; xph ^= 1u; }
          }
        }
      }
      for (long long q = 0; q < (iss < XS ? iss : XS); ++q) {     // let issued copies land
        if (--xs < 0) { xs = XS - 1; xph ^= 1u; }
        mbar_drain(&tail->x_full[xs], xph);
      }
    }
  } else if (warp == kW_W) {
    // ================================================= phi-plane producer (L2)
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();
      int ws = 0;
      uint32_t wph = 0;
      long long iss = 0;
      bool ok = true;
      for (int tile = cluster_id; tile < g.num_tiles && ok; tile += num_clusters) {
        for (int j = c0; j < c1 && ok; ++j) {
          for (int wg = 0; wg < C::kWBoxes; ++wg) {
            if (!wait_bar<false>(&tail->w_empty[ws], wph ^ 1u, ctl, kErrWaitTimeout)) { ok = false; break; }
            mbar_expect_tx(&tail->w_full[ws], (uint32_t)C::kWBytes);
            bulk_load_hint(sW + (size_t)ws * C::kWBytes,
                           planes + ((size_t)j * NS + (size_t)wg * C::kWG) * C::kWRows * kChunkK,
                           (uint32_t)C::kWBytes, &tail->w_full[ws], keep);
            ++iss;
            if (++ws == WS) { ws = 0; wph ^= 1u; }
          }
        }
      }
      for (long long q = 0; q < (iss < WS ? iss : WS); ++q) {
        if (--ws < 0) { ws = WS - 1; wph ^= 1u; }
        mbar_drain(&tail->w_full[ws], wph);
      }
    }
  } else if (warp == kW_MMA) {
    // ================================================= MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kMmaM, C::kNP);
      int xs = 0, ws = 0, acc = 0;
      uint32_t xph = 0, wph = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = cluster_id; tile < g.num_tiles && ok; tile += num_clusters) {
        if (!wait_bar<false>(&tail->acc_empty[acc], acc_phase ^ 1u, ctl, kErrWaitTimeout)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * C::kAccCols);
        bool first = true;
        for (int j = c0; j < c1 && ok; ++j) {
          uint32_t xbase = 0, wbase = 0;
          for (int i = 0; i < NS; ++i) {
            if (i % C::kWG == 0) {
              if (!wait_bar<false>(&tail->w_full[ws], wph, ctl, kErrWaitTimeout)) { ok = false; break; }
              wbase = smem_u32(sW + (size_t)ws * C::kWBytes);
            }
            if (i % kSGt == 0) {
              if (!wait_bar<false>(&tail->x_full[xs], xph, ctl, kErrWaitTimeout)) { ok = false; break; }
              xbase = smem_u32(sX + (size_t)xs * kXBoxBytes);
            }
            tc_fence_after();
            const uint32_t a0 = xbase + (uint32_t)((i % kSGt) * kT * 128);
            const uint32_t b0 = wbase + (uint32_t)((i % C::kWG) * C::kWRows * 128);
#pragma unroll
            for (int kk = 0; kk < kChunkK / 16; ++kk) {
              mma_bf16(d, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc, first ? 0u : 1u);
              first = false;
            }
            if (i % kSGt == kSGt - 1) {              // the MMA side of the x slot's release
              mma_commit(&tail->x_empty[xs]);
              if (++xs == XS) { xs = 0; xph ^= 1u; }
            }
            if (i % C::kWG == C::kWG - 1) {
              mma_commit(&tail->w_empty[ws]);
              if (++ws == WS) { ws = 0; wph ^= 1u; }
            }
          }
        }
        if (!ok) break;
        mma_commit(&tail->acc_full[acc]);          // accumulator complete
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      mma_commit(&tail->mma_done);
      mbar_drain(&tail->mma_done, 0);
    }
  } else if (warp >= kW_PUB0 && warp < kW_PUB0 + 4) {
    // ================================================= sum of squares + partials
    // Thread = tile row = TMEM lane (warps 4..7: lane quarters 0..3).
    const int et = threadIdx.x - kW_PUB0 * 32;    // 0..127
    const int wq = warp & 3;
    const int owner = et / rpo;
    const int slot = et - owner * rpo;
    int xs = 0, acc = 0;
    uint32_t xph = 0, acc_phase = 0;
    uint32_t k = 0;
    bool ok = true;
    for (int tile = cluster_id; tile < g.num_tiles && ok; tile += num_clusters, ++k) {
      // x^2 of this row from every box of the tile, each released after.
      float s8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) s8[e] = 0.0f;
      for (int j = c0; j < c1 && ok; ++j) {
        for (int grp = 0; grp < C::kGroups; ++grp) {
          // each warp takes the box on its own and releases it after reading
          // every lane waits on the barrier itself: each lane's own acquire
          // orders its reads of the box after the copy landed
          if (!__all_sync(0xffffffffu, wait_bar<false>(&tail->x_full[xs], xph, ctl, kErrWaitTimeout))) {
            ok = false;
            break;
          }
          const uint8_t* rowp = sX + (size_t)xs * kXBoxBytes + (size_t)et * 128;
#pragma unroll
          for (int s = 0; s < kSGt; ++s) {
            uint4 v[8];
#pragma unroll
            for (int c = 0; c < 8; ++c)
              v[c] = *reinterpret_cast<const uint4*>(rowp + (size_t)s * kT * 128 + ((c ^ (et & 7)) << 4));
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
          __syncwarp();
          if (lane == 0) mbar_arrive(&tail->x_empty[xs]);
          if (++xs == XS) { xs = 0; xph ^= 1u; }
        }
      }
      if (!ok) break;
      const float ssq = tree_sum<8>(s8);

      if (!role_all<kBarP, kPubThr>(wait_bar<false>(&tail->acc_full[acc], acc_phase, ctl, kErrWaitTimeout))) break;
      tc_fence_after();
      float mix[RR];
#pragma unroll
      for (int r = 0; r < RR; ++r) mix[r] = 0.0f;
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
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }

      // every owner must have consumed the previous tile's partials
      if (k > 0 && !role_all<kBarP, kPubThr>(wait_bar<true>(&tail->part_free, (k - 1) & 1u, ctl, kErrClusterWait)))
        break;
      float* dst = recv + ((size_t)((int)rank * rpo + slot)) * C::kStr;
#pragma unroll
      for (int r = 0; r < C::kStr; r += 4) {
        float4 v;
        v.x = r < RR ? mix[r] : (r == RR ? ssq : 0.0f);
        v.y = r + 1 < RR ? mix[r + 1] : (r + 1 == RR ? ssq : 0.0f);
        v.z = r + 2 < RR ? mix[r + 2] : (r + 2 == RR ? ssq : 0.0f);
        v.w = r + 3 < RR ? mix[r + 3] : (r + 3 == RR ? ssq : 0.0f);
        st_dsmem_v4(dst + r, (uint32_t)owner, v);
      }
      role_sync<kBarP, kPubThr>();
      if (et < CL) mbar_arrive_remote(&tail->part_full, (uint32_t)et);
    }
  } else if (warp == kW_GATE) {
    // ================================================= gates (critical for y)
    // Owned rows (lane + 32 h): sum the members' partials in rank order,
    // compute invRms and the gates, send the y weights to every member, then
    // run the rows' Sinkhorn.
    uint32_t k = 0;
    for (int tile = cluster_id; tile < g.num_tiles; tile += num_clusters, ++k) {
      if (!__all_sync(0xffffffffu, wait_bar<true>(&tail->part_full, k & 1u, ctl, kErrClusterWait))) break;
      for (int h = 0; h * 32 < rpo; ++h) {
        const int ot = lane + 32 * h;
        if (ot < rpo) {
          float tot[C::kStr];
#pragma unroll
          for (int r = 0; r < C::kStr; ++r) tot[r] = 0.0f;
          for (int cr = 0; cr < CL; ++cr) {
            const float* src = recv + ((size_t)(cr * rpo + ot)) * C::kStr;
#pragma unroll
            for (int r = 0; r < C::kStr; r += 4) {
              const float4 v = *reinterpret_cast<const float4*>(src + r);
              tot[r] += v.x;
              tot[r + 1] += v.y;
              tot[r + 2] += v.z;
              tot[r + 3] += v.w;
            }
          }
          float* o = owned + (size_t)ot * C::kStr;
#pragma unroll
          for (int r = 0; r < C::kStr; r += 4)
            *reinterpret_cast<float4*>(o + r) = make_float4(tot[r], tot[r + 1], tot[r + 2], tot[r + 3]);
        }
      }
      __syncwarp();
      if (lane < CL) mbar_arrive_remote(&tail->part_free, (uint32_t)lane);   // partials consumed

      const int cb = (int)(k % kCoefBufs);
      const uint32_t cuse = k / kCoefBufs;
      if (cuse > 0 &&
          !__all_sync(0xffffffffu, wait_bar<true>(&tail->coef_free[cb], (cuse - 1) & 1u, ctl, kErrClusterWait)))
        break;
      for (int h = 0; h * 32 < rpo; ++h) {
        const int ot = lane + 32 * h;
        if (ot < rpo) {
          const float* o = owned + (size_t)ot * C::kStr;
          float mix[RR];
#pragma unroll
          for (int r = 0; r < RR; ++r) mix[r] = o[r];
          const int row = (int)rank * rpo + ot;
          const int tok = tile * kT + row;
          float cf[NS];
          const float inv_rms = token_gates<NS, RR>(ep, tok, mix, o[RR], tok < g.T, cf);
          float* dst = coef_buf + ((size_t)cb * kT + row) * NS;
          for (int cr = 0; cr < CL; ++cr)
            st_dsmem_v4(dst, (uint32_t)cr, make_float4(cf[0], cf[1], cf[2], cf[3]));
          // keep the residual logits in the row's own owned-sum slot for the
          // Sinkhorn below (the two-gate form has none)
          if constexpr (C::kThree) {
            static_assert(NS * NS <= C::kStr, "logits fit the owned-sum slot");
            float H[NS * NS];
            residual_logits<NS, RR>(ep, mix, inv_rms, H);
            float* ho = owned + (size_t)ot * C::kStr;
#pragma unroll
            for (int r = 0; r < NS * NS; ++r) ho[r] = H[r];
          }
        }
      }
      __syncwarp();
      if (lane < CL) mbar_arrive_remote(&tail->coef_full[cb], (uint32_t)lane);
      // Sinkhorn for comb: y no longer waits on this tile.
      for (int h = 0; h * 32 < rpo; ++h) {
        const int ot = lane + 32 * h;
        if (ot < rpo) {
          const int tok = tile * kT + (int)rank * rpo + ot;
          token_sinkhorn<NS, C::kThree>(ep, tok, owned + (size_t)ot * C::kStr, tok < g.T);
        }
      }
      __syncwarp();
    }
  } else if (warp >= kW_Y0) {
    // ================================================= y for this member's d-range
    // y[t, d] = sum_i m_i x[t, i, d] over the rows of the tile and this
    // member's d-range, re-reading x with plain 16-byte loads (newest d
    // first); kYBatch items per thread are in flight at once.
    const int yt = threadIdx.x - kW_Y0 * 32;
    const uint64_t read_policy = policy_evict_first();
    const uint64_t ystore_policy = policy_evict_first();
    const int dlo = c0 * kChunkK;
    const int dhi = min(c1 * kChunkK, g.D);
    const int w8 = (dhi - dlo) >> 3;              // 16-byte vectors per row
    uint32_t k = 0;
    for (int tile = cluster_id; tile < g.num_tiles; tile += num_clusters, ++k) {
      const int cb = (int)(k % kCoefBufs);
      if (!role_all<kBarYt, kYThr>(wait_bar<true>(&tail->coef_full[cb], (k / kCoefBufs) & 1u, ctl,
                                                  kErrClusterWait)))
        break;
      const float* coef = coef_buf + (size_t)cb * kT * NS;
      const int rows = min(kT, g.T - tile * kT);
      const int items = rows * w8;
      const __nv_bfloat16* xt = xg + (size_t)tile * kT * NS * g.D;
      __nv_bfloat16* yt_out = ep.y + (size_t)tile * kT * g.D;
      for (int base = yt; base < items; base += kYThr * C::kYBatch) {
        uint4 xv[C::kYBatch][NS];
        int rowv[C::kYBatch], dv[C::kYBatch];
#pragma unroll
        for (int b = 0; b < C::kYBatch; ++b) {
          const int it = base + b * kYThr;
          const int row = it / w8;
          const int v = w8 - 1 - (it - row * w8);  // newest columns first
          rowv[b] = it < items ? row : -1;
          dv[b] = dlo + 8 * v;
          if (it < items) {
            const __nv_bfloat16* src = xt + ((size_t)row * NS) * g.D + dv[b];
#pragma unroll
            for (int i = 0; i < NS; ++i) xv[b][i] = ld_global_v4_hint(src + (size_t)i * g.D, read_policy);
          }
        }
#pragma unroll
        for (int b = 0; b < C::kYBatch; ++b) {
          if (rowv[b] < 0) continue;
          float acc8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc8[e] = 0.0f;
#pragma unroll
          for (int i = 0; i < NS; ++i) {
            const float m = coef[rowv[b] * NS + i];
            const __nv_bfloat162* hh = reinterpret_cast<const __nv_bfloat162*>(&xv[b][i]);
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
              const float2 f = __bfloat1622float2(hh[q2]);
              acc8[2 * q2] = fmaf(m, f.x, acc8[2 * q2]);
              acc8[2 * q2 + 1] = fmaf(m, f.y, acc8[2 * q2 + 1]);
            }
          }
          uint4 o;
          __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
          for (int q2 = 0; q2 < 4; ++q2) ob[q2] = __floats2bfloat162_rn(acc8[2 * q2], acc8[2 * q2 + 1]);
          st_global_v4_hint(yt_out + (size_t)rowv[b] * g.D + dv[b], o, ystore_policy);
        }
      }
      role_sync<kBarYt, kYThr>();                  // every y thread is done with coef[cb]
      if (yt < CL) mbar_arrive_remote(&tail->coef_free[cb], (uint32_t)yt);
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kW_MMA) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(C::kTmemCols)
                 : "memory");
  }
  cluster_sync_all();
}

template <int RR, int P>
const void* t128_ptr() {
  return reinterpret_cast<const void*>(&mhc_pre_t128_kernel<RR, P>);
}

const void* t128_select(int n, int R, int P) {
  if (n != 4) return nullptr;
  if (R == 24 && P == 3) return t128_ptr<24, 3>();
  if (R == 24 && P == 2) return t128_ptr<24, 2>();
  if (R == 8 && P == 3) return t128_ptr<8, 3>();
  if (R == 8 && P == 2) return t128_ptr<8, 2>();
  return nullptr;
}

cudaLaunchConfig_t t128_config(int cluster, int grid, size_t smem, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

bool t128_supported(int n, int R, int P) { return t128_select(n, R, P) != nullptr; }

cudaError_t t128_forward_occupancy(int n, int R, int P, size_t smem_bytes, int cluster, int* max_clusters) {
  *max_clusters = 0;
  const void* k = t128_select(n, R, P);
  if (!k) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
  if (e != cudaSuccess) return e;
  if (cluster > 8) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = t128_config(cluster, cluster, smem_bytes, nullptr, attr);
  return cudaOccupancyMaxActiveClusters(max_clusters, k, &cfg);
}

cudaError_t launch_t128_forward(const TcLaunch& L, cudaStream_t s) {
  const int n = L.epi.n, R = L.epi.R;
  const void* k = t128_select(n, R, L.P);
  if (!k) return cudaErrorInvalidValue;
  Geometry g;
  g.T = L.epi.T;
  g.D = L.epi.D;
  g.n = n;
  g.num_tiles = (L.epi.T + kT - 1) / kT;
  g.nd = (L.epi.D + kChunkK - 1) / kChunkK;
  g.cluster = L.cluster;
  g.xstages = L.xstages;
  g.wstages = L.wstages;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = t128_config(L.cluster, L.grid, L.smem_bytes, s, attr);
  const __nv_bfloat16* xg = static_cast<const __nv_bfloat16*>(L.x);
  const __nv_bfloat16* planes = L.planes;
  void* args[] = {const_cast<CUtensorMap*>(&L.tmap_x), const_cast<__nv_bfloat16**>(&planes),
                  const_cast<EpiParams*>(&L.epi), &xg, &g, const_cast<uint32_t**>(&L.err_word)};
  return cudaLaunchKernelExC(&cfg, k, args);
}

}  // namespace mhc
