// mhc_pre_tc.cu -- the sm_103a forward: TMA x tiles, tcgen05 projection into
// TMEM, register epilogue (RMS, gates, Sinkhorn) and the weighted sum y.
//
// What is computed follows "CANN ops-transformer 中 aclnnMhcPreV2 算子接口
// 全解析" §三 and "aclnnMhcPreSinkhorn 接口与 MhcPreSinkhorn 实现剖析" §3.2;
// how it is laid out on the GPU is this file's own design:
//
//  * A token tile is 64 tokens.  A cluster of C CTAs shares one tile; CTA c
//    owns a contiguous range of 64-wide d-chunks and streams those chunks of
//    all n streams, so each byte of x is read from HBM once per tile.
//  * Per chunk, TMA brings x[64 tokens][64] of a group of streams (bf16,
//    128-byte swizzle) and the matching 64 columns of the stacked phi planes;
//    one thread issues tcgen05.mma (M = 128, K = 16 each) into TMEM, two
//    streams per MMA where their planes fit N <= 256 (A rows 0..63 and
//    64..127 are the two streams' tokens), else one stream per MMA with A
//    rows 64..127 unused.
//  * Four publish warps (thread = token, one warp per TMEM lane quarter) sum
//    each token's squares from every x box as it lands (CUDA cores: an
//    x.x^T block on the tensor core would double its operand reads from
//    shared memory, which bound the MMA), then read the accumulators, fold
//    the precision planes and push the CTA's partial sums to the member that
//    owns the row (distributed shared memory).  The owner's gate warp sums
//    them in (rank, half) order, computes invRms and the gates, sends the y
//    weights to every member, then runs the rows' Sinkhorn for comb, off
//    y's path.
//  * Eight warps form y for the CTA's d-range by re-reading x from global
//    memory, newest chunk first.
//  * This kernel serves shapes whose phi blocks are too large to stay
//    resident in the grid-wide kernel (mhc_pre_gw.cu).
//  * Every wait is bounded by a timer; a wait that gives up sets the error
//    word in the workspace and the kernel winds down instead of hanging.
#include "mhc_ptx.cuh"

namespace mhc {
namespace {

// ------------------------------------------------------------ kernel body
template <int NS, int RR, int P, bool kRes = false>
struct Cfg {
  static constexpr int kNP = ((P * RR + 15) / 16) * 16;          // MMA N of the projection
  static_assert(kNP <= 256, "N of one MMA is at most 256");
  static constexpr int kAccBufs = kRes ? 1 : 2;                  // accumulator buffers
  static constexpr int kSG = stream_group(NS);                   // streams per x box
  static constexpr int kGroups = NS / kSG;                       // x boxes per d-chunk
  static_assert(NS % kSG == 0, "stream groups tile the streams");
  static constexpr int kXBytes = kSG * kStreamTile;              // one x box
  static constexpr int kWRows = plane_box_rows(RR, P);
  static constexpr int kWG = w_group(NS, RR, P);                 // streams per w box
  static constexpr int kWBoxes = NS / kWG;                       // w boxes per d-chunk
  static constexpr int kWBytes = kWG * kWRows * 128;             // one w box
  // Stream pairs: one MMA (M = 128, N = 2 kWRows) takes streams i and i+1
  // at once -- A rows 0..63 are stream i's tokens, rows 64..127 stream
  // i+1's (the next 8 KB of the x box), B is both streams' plane rows back
  // to back in the w box; accumulator rows 0..63 x columns [0, kWRows) and
  // rows 64..127 x columns [kWRows, 2 kWRows) are the two streams' partial
  // projections (the off-diagonal blocks are never read).  Without pairs
  // the MMA runs N = NP per stream and rows 64..127 are never read.
  static constexpr bool kPair = stream_pairs(NS, RR, P);
  static constexpr int kHalves = kPair ? 2 : 1;                  // published partials per member and row
  static constexpr int kStep = kPair ? 2 : 1;                    // streams per MMA
  static constexpr int kMmaN = kPair ? 2 * kWRows : kNP;
  static constexpr int kAccCols = kMmaN <= 64 ? 64 : kMmaN <= 128 ? 128 : 256;
  // Resident mode: the last chunks of each tile stay in TMEM for y.  A block
  // of 128 columns holds two chunks (lanes 0..63: one chunk's 64 tokens,
  // lanes 64..127: the next chunk's), each lane a token's 4 streams x 64
  // columns of bf16 pairs; the single accumulator follows the blocks.
  static constexpr int kTmBlocks = kRes ? (512 - kMmaN) / 128 : 0;
  static constexpr int kTmChunks = 2 * kTmBlocks;
  static constexpr int kAccBase = 128 * kTmBlocks;               // first accumulator column
  static constexpr uint32_t kTmemCols = kRes ? 512u : (uint32_t)(kAccCols * kAccBufs);
  static_assert(!kRes || (NS == 4 && kPair && kSG == 4 && kGroups == 1 && kTmBlocks >= 1),
                "resident mode: n = 4, stream pairs, one 4-stream x box per chunk");
  static_assert(kMmaN % 16 == 0 && kMmaN <= 256, "M = 128 takes N = 16 .. 256 in steps of 16");
  static constexpr int kStr = partial_stride(RR);                // floats per published partial
  static constexpr bool kThree = (RR == NS * NS + 2 * NS);
  // y items in flight per thread (re-read loads: 3 x NS x 16 B).  Four
  // measured the same at cluster 4 and 2% slower in tf32 mode and at cluster
  // 8; six spill.
  static constexpr int kYBatch = NS <= 4 ? 3 : 2;
};

struct SmemTail {
  uint64_t x_full[kMaxStages], x_empty[kMaxStages];
  uint64_t w_full[kMaxStages], w_empty[kMaxStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t part_full, part_free;
  uint64_t coef_full[kCoefBufs], coef_free[kCoefBufs];
  uint64_t mma_done;
  uint64_t tm_full[2], tm_free[2];              // resident mode: a TMEM buffer's chunks written / read by y
  uint32_t tmem_base;
  uint32_t abort;
  float ssq_hand[kTileT];                       // unpaired shapes: half 1's sums of squares for half 0
};
static_assert(sizeof(SmemTail) <= kTailBytes, "barrier block outgrew its reservation");

// Warp roles: one TMA producer per ring, so each ring has its own issuing
// thread; warps 4..7 cover the four TMEM lane quarters.
constexpr int kWarpX = 0, kWarpMma = 1, kWarpW = 2, kWarpGate = 3, kWarpPub0 = 4, kWarpYc0 = 8;
constexpr int kPubThreads = 128;
constexpr int kYThreads = kThreads - kWarpYc0 * 32;   // 256
// Named barriers: 1 = publish pair (64 threads), 2 = y warps.
constexpr int kBarPub = 1, kBarY = 2;

// Adds accumulator columns [CB, CB + P RR) of this warp's TMEM lanes, read
// in 16-column groups from a 16-aligned start, into the R projection sums
// (column CB + p R + r is plane p of row r).
template <int RR, int P, int CB, bool F16>
__device__ __forceinline__ void fold_planes(uint32_t taddr, float (&mix)[RR]) {
  constexpr int CA = CB & ~15;
  constexpr int kGroups = (CB + P * RR - CA + 15) / 16;
#pragma unroll
  for (int grp = 0; grp < kGroups; ++grp) {
    float v[16];
    tmem_ld16(taddr + (uint32_t)(CA + grp * 16), v);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int col = CA + grp * 16 + e - CB;
      if (col >= 0 && col < P * RR) mix[col % RR] += F16 ? v[e] * plane_scale(true, col / RR) : v[e];
    }
  }
}

// One token's Sinkhorn, kept out of line: it runs once per tile or batch, and
// inlined it would lengthen the register lifetimes of the whole gate path.
template <int NS, bool kThree>
__device__ __noinline__ void sinkhorn_call(const EpiParams& ep, int tok, const float* H, bool write) {
  token_sinkhorn<NS, kThree>(ep, tok, H, write);
}

// The y weights of one owned row to the same place in every cluster member.
template <int NS>
__device__ __forceinline__ void push_coefs(float* dst, int CL, const float (&cf)[NS]) {
  for (int cr = 0; cr < CL; ++cr) {
    if constexpr (NS % 4 == 0) {
#pragma unroll
      for (int i = 0; i < NS; i += 4)
        st_dsmem_v4(dst + i, (uint32_t)cr, make_float4(cf[i], cf[i + 1], cf[i + 2], cf[i + 3]));
    } else {
#pragma unroll
      for (int i = 0; i < NS; ++i) st_dsmem_f32(dst + i, (uint32_t)cr, cf[i]);
    }
  }
}

template <int NS, int RR, int P, bool F16, bool kRes>
__global__ void __launch_bounds__(kThreads, 1)
    mhc_pre_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __nv_bfloat16* __restrict__ planes,
                      const EpiParams ep, const __nv_bfloat16* __restrict__ xg, Geometry g, uint32_t* err) {
  using C = Cfg<NS, RR, P, kRes>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const SmemLayout Ly = smem_layout(NS, RR, P, g.xstages, g.wstages);
  const int XS = g.xstages, WS = g.wstages;
  uint8_t* sX = smem + Ly.x;
  uint8_t* sW = smem + Ly.w;
  float* recv = reinterpret_cast<float*>(smem + Ly.part);     // [CL][kHalves][64/CL][kStr]
  float* coef_buf = reinterpret_cast<float*>(smem + Ly.coef); // [kCoefBufs][64][NS]
  float* sink_h = reinterpret_cast<float*>(smem + Ly.sink);   // [32][NS * NS]: a Sinkhorn batch's logits
  int* sink_tok = reinterpret_cast<int*>(sink_h + 32 * NS * NS);   // [32]: their tokens (-1: none)
  SmemTail* tail = reinterpret_cast<SmemTail*>(smem + Ly.tail);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int CL = g.cluster;
  const uint32_t rank = cluster_rank();
  const int cluster_id = blockIdx.x / CL;
  const int num_clusters = gridDim.x / CL;
  const int c0 = (int)((long long)rank * g.nd / CL);
  const int c1 = (int)((long long)(rank + 1) * g.nd / CL);
  const int rpo = kTileT / CL;                    // tile rows each member reduces (owns)
  // resident mode: this member's last CT chunks (from jT on) stay in TMEM
  // for y; y re-reads the chunks before jT (loaded moments earlier) from L2.
  // The TMEM chunk slots form nbuf buffers of cpb slots used by alternate
  // tiles (slot s: lanes 64 (s & 1) .. + 63 of columns 128 (s >> 1) ..).
  const int nbuf = kRes ? (g.tm_bufs == 2 ? 2 : 1) : 1;
  const int cpb = C::kTmChunks / nbuf;
  const int CT = kRes ? min(c1 - c0, cpb) : 0;
  const int jT = c1 - CT;
  Ctl ctl{&tail->abort, err, g.wt.wait_ns};

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
    mbar_init(&tail->part_full, C::kHalves * CL);   // one arrival per member and published half
    mbar_init(&tail->part_free, CL);
    mbar_init(&tail->mma_done, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tail->tm_full[b], 4);            // four publish warps
      mbar_init(&tail->tm_free[b], kYThreads / 32);  // eight y warps
    }
    tail->abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tmap_x);
  }
  if (warp == kWarpMma) {
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

  if (warp == kWarpX) {
    // ================================================= x producer (HBM)
    if (lane == 0) {
      const uint64_t keep = policy_evict_last();
      int xs = 0;
      uint32_t xph = 0;
      long long iss = 0;
      bool ok = true;
      // test hook: CTA 0 leaves out its last box (see WaitTest)
      const int last_tile = cluster_id + ((g.num_tiles - 1 - cluster_id) / num_clusters) * num_clusters;
      for (int tile = cluster_id; tile < g.num_tiles && ok; tile += num_clusters) {
        for (int j = c0; j < c1 && ok; ++j) {
          for (int grp = 0; grp < C::kGroups; ++grp) {
            if (!wait_bar<false>(&tail->x_empty[xs], xph ^ 1u, ctl, kErrWaitTimeout)) { ok = false; break; }
            if (g.wt.withhold_x && blockIdx.x == 0 && tile == last_tile && j == c1 - 1 && grp == C::kGroups - 1)
              break;
            mbar_expect_tx(&tail->x_full[xs], (uint32_t)C::kXBytes);
            tma_load_3d_hint(sX + (size_t)xs * C::kXBytes, &tmap_x, &tail->x_full[xs], j * kChunkK,
                             tile * kTileT, grp * C::kSG, keep);
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
  } else if (warp == kWarpW) {
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
            // the plane blocks of streams wg*kWG .. +kWG of chunk j: one run
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
  } else if (warp == kWarpMma) {
    // ================================================= MMA issuer
    // Per stream (or stream pair) of each d-chunk: the projection into TMEM.
    if (lane == 0) {
      constexpr uint32_t idesc_proj = F16 ? idesc_f16(kMmaM, C::kMmaN) : idesc_bf16(kMmaM, C::kMmaN);
      int xs = 0, ws = 0, acc = 0;
      uint32_t xph = 0, wph = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = cluster_id; tile < g.num_tiles && ok; tile += num_clusters) {
        if (!wait_bar<false>(&tail->acc_empty[acc], acc_phase ^ 1u, ctl, kErrWaitTimeout)) break;
        tc_fence_after();
        const uint32_t d_proj = tmem_base + (uint32_t)(C::kAccBase + acc * C::kAccCols);
        bool first = true;
        for (int j = c0; j < c1 && ok; ++j) {
          uint32_t xbase = 0, wbase = 0;
          for (int i = 0; i < NS; i += C::kStep) {
            if (i % C::kWG == 0) {
              if (!wait_bar<false>(&tail->w_full[ws], wph, ctl, kErrWaitTimeout)) { ok = false; break; }
              wbase = smem_u32(sW + (size_t)ws * C::kWBytes);
            }
            if (i % C::kSG == 0) {
              if (!wait_bar<false>(&tail->x_full[xs], xph, ctl, kErrWaitTimeout)) { ok = false; break; }
              xbase = smem_u32(sX + (size_t)xs * C::kXBytes);
            }
            tc_fence_after();
            // A: 128 rows from this stream's token tile (rows 64..127: the
            // pair's second stream, or rows that run on into the next tile
            // and feed lanes that are never read).
            const uint32_t a0 = xbase + (uint32_t)((i % C::kSG) * kStreamTile);
            const uint32_t b0 = wbase + (uint32_t)((i % C::kWG) * C::kWRows * 128);
#pragma unroll
            for (int kk = 0; kk < kChunkK / 16; ++kk) {
              const uint32_t acc_in = first ? 0u : 1u;
              mma_bf16(d_proj, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc_proj, acc_in);
              first = false;
            }
            if ((i + C::kStep) % C::kSG == 0) {      // frees the x slot when these MMAs finish
              mma_commit(&tail->x_empty[xs]);
              if (++xs == XS) { xs = 0; xph ^= 1u; }
            }
            if ((i + C::kStep) % C::kWG == 0) {
              mma_commit(&tail->w_empty[ws]);
              if (++ws == WS) { ws = 0; wph ^= 1u; }
            }
          }
        }
        if (!ok) break;
        mma_commit(&tail->acc_full[acc]);          // accumulator complete
        if (++acc == C::kAccBufs) { acc = 0; acc_phase ^= 1u; }
      }
      mma_commit(&tail->mma_done);
      mbar_drain(&tail->mma_done, 0);
    }
  } else if (warp >= kWarpPub0 && warp < kWarpYc0) {
    // ================================================= sums of squares + partials
    // Warp 4 + q reads TMEM lane quarter q.  Half h = q / 2 of the warps
    // takes tile rows et = 0..63 (lane 64 h + et): its share of each row's
    // sum of squares (streams [sg0, sg1) of every x box, read in swizzled
    // order as the box lands, the box released after) and of the partial
    // projection (half 0: the unpaired or first-of-pair streams, half 1: the
    // second-of-pair streams), pushed to the member that owns the row.
    const int q = warp - kWarpPub0;                // TMEM lane quarter 0..3
    const int half = q >> 1;
    const int et = (q & 1) * 32 + lane;            // tile row 0..63
    const int owner = et / rpo;
    const int slot = et - owner * rpo;
    constexpr int kSgHalf = (C::kSG + 1) / 2;
    const int sg0 = half * kSgHalf;
    const int sg1 = min(C::kSG, sg0 + kSgHalf);
    int acc = 0, xs = 0;
    uint32_t acc_phase = 0, xph = 0;
    uint32_t k = 0;
    bool ok = true;
    for (int tile = cluster_id; tile < g.num_tiles && ok; tile += num_clusters, ++k) {
      float s8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) s8[e] = 0.0f;
      for (int j = c0; j < c1 && ok; ++j) {
        // resident mode: y must have read the tile that last used this TMEM
        // buffer before the first of this tile's chunks goes in
        if (kRes && j == jT && k >= (uint32_t)nbuf &&
            !__all_sync(0xffffffffu, wait_bar<false>(&tail->tm_free[k % nbuf], (k / nbuf - 1) & 1u, ctl,
                                                     kErrWaitTimeout))) {
          ok = false;
          break;
        }
        if (kRes && j == jT) tc_fence_after();
        for (int grp = 0; grp < C::kGroups; ++grp) {
          // every lane waits on the barrier itself: each lane's own acquire
          // orders its reads of the box after the copy landed
          if (!__all_sync(0xffffffffu, wait_bar<false>(&tail->x_full[xs], xph, ctl, kErrWaitTimeout))) {
            ok = false;
            break;
          }
          const uint8_t* rowp = sX + (size_t)xs * C::kXBytes + (size_t)et * 128;
          if (kRes && j >= jT) {
            // a TMEM chunk in slot sl: the warp of lane quarter q takes it
            // when sl's parity is q / 2 -- its token's row of all four
            // streams goes into TMEM (lane 32 q + lane = token et + 64 (sl &
            // 1)) and into the sum of squares; the other two warps leave it
            const int sl = (int)(k % nbuf) * cpb + (j - jT);
            if ((sl & 1) == (q >> 1)) {
              const uint32_t tx = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)((sl >> 1) * 128);
#pragma unroll
              for (int sg = 0; sg < C::kSG; ++sg) {
                uint4 v[8];
#pragma unroll
                for (int c = 0; c < 8; ++c)
                  v[c] = *reinterpret_cast<const uint4*>(rowp + (size_t)sg * kStreamTile + ((c ^ (et & 7)) << 4));
                uint32_t words[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                  words[4 * c] = v[c].x;
                  words[4 * c + 1] = v[c].y;
                  words[4 * c + 2] = v[c].z;
                  words[4 * c + 3] = v[c].w;
                }
                tmem_st32(tx + (uint32_t)(sg * 32), words);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                  const typename XType<F16>::T2* h2 = reinterpret_cast<const typename XType<F16>::T2*>(&v[c]);
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const float2 f = XType<F16>::to_f2(h2[e]);
                    s8[2 * e] = fmaf(f.x, f.x, s8[2 * e]);
                    s8[2 * e + 1] = fmaf(f.y, f.y, s8[2 * e + 1]);
                  }
                }
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&tail->x_empty[xs]);
            if (++xs == XS) { xs = 0; xph ^= 1u; }
            continue;
          }
          for (int sg = sg0; sg < sg1; ++sg) {
            uint4 v[8];
#pragma unroll
            for (int c = 0; c < 8; ++c)
              v[c] = *reinterpret_cast<const uint4*>(rowp + (size_t)sg * kStreamTile + ((c ^ (et & 7)) << 4));
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const typename XType<F16>::T2* h2 = reinterpret_cast<const typename XType<F16>::T2*>(&v[c]);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f = XType<F16>::to_f2(h2[e]);
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
      // all four warps leave together if any gave up (the producer stops on
      // the abort flag, so the others' waits end too)
      if (!role_all<kBarPub, kPubThreads>(ok)) break;
      if (kRes && CT > 0) {                        // this tile's TMEM chunks are in
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tail->tm_full[k % nbuf]);
      }
      float ssq = tree_sum<8>(s8);
      // unpaired: half 1 has no projection sums, so half 0 publishes its
      // sums of squares too (read after the barrier below; half 1 writes the
      // next tile's only after the barrier that ends this tile's publish)
      if (!C::kPair && half == 1) tail->ssq_hand[et] = ssq;
      if (!role_all<kBarPub, kPubThreads>(wait_bar<false>(&tail->acc_full[acc], acc_phase, ctl, kErrWaitTimeout)))
        break;
      if (!C::kPair && half == 0) ssq += tail->ssq_hand[et];
      tc_fence_after();
      float mix[RR];
#pragma unroll
      for (int r = 0; r < RR; ++r) mix[r] = 0.0f;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(C::kAccBase + acc * C::kAccCols);
      if (half == 0) fold_planes<RR, P, 0, F16>(taddr, mix);
      else if (C::kPair) fold_planes<RR, P, C::kWRows, F16>(taddr, mix);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->acc_empty[acc]);
      if (++acc == C::kAccBufs) { acc = 0; acc_phase ^= 1u; }

      // every owner must have consumed the previous tile's partials
      if (k > 0 &&
          !role_all<kBarPub, kPubThreads>(wait_bar<true>(&tail->part_free, (k - 1) & 1u, ctl, kErrClusterWait)))
        break;
      if (C::kPair || half == 0) {
        float* dst = recv + ((size_t)(((int)rank * C::kHalves + half) * rpo + slot)) * C::kStr;
#pragma unroll
        for (int r = 0; r < C::kStr; r += 4) {
          float4 v;
          v.x = r < RR ? mix[r] : (r == RR ? ssq : 0.0f);
          v.y = r + 1 < RR ? mix[r + 1] : (r + 1 == RR ? ssq : 0.0f);
          v.z = r + 2 < RR ? mix[r + 2] : (r + 2 == RR ? ssq : 0.0f);
          v.w = r + 3 < RR ? mix[r + 3] : (r + 3 == RR ? ssq : 0.0f);
          st_dsmem_v4(dst + r, (uint32_t)owner, v);
        }
      }
      role_sync<kBarPub, kPubThreads>();
      // one arrival per published half at every owner
      if ((q & 1) == 0 && (C::kPair || half == 0) && lane < CL) mbar_arrive_remote(&tail->part_full, (uint32_t)lane);
    }
  } else if (warp == kWarpGate) {
    // ================================================= gates (critical for y), then Sinkhorn
    // Owned rows: sum the members' partials of each row in a fixed order,
    // compute invRms and the gates, publish the y weights to every member,
    // then run the rows' Sinkhorn for comb (off y's path).
    //  * 32 or more owned rows (clusters of 1 or 2): a lane per row sums its
    //    partials in (rank, half) order; the Sinkhorn follows at once, one
    //    token per lane.
    //  * fewer (clusters of 4 to 16): lpr = 32 / rpo lanes share a row --
    //    lane ot lpr + p adds the partials p, p + lpr, ..., then a butterfly
    //    in fixed order adds the lanes -- and the Sinkhorn runs once per
    //    batch of lpr tiles with one token per lane (each tile hands its
    //    rows' logits to their batch lanes), so that its latency is paid
    //    once per batch rather than once per tile.
    const int lpr = rpo >= 32 ? 1 : 32 / rpo;
    const int nparts = C::kHalves * CL;
    sink_tok[lane] = -1;
    __syncwarp();
    uint32_t k = 0;
    for (int tile = cluster_id; tile < g.num_tiles; tile += num_clusters, ++k) {
      if (!__all_sync(0xffffffffu, wait_bar<true>(&tail->part_full, k & 1u, ctl, kErrClusterWait))) break;
      const int cb = (int)(k % kCoefBufs);
      const uint32_t cuse = k / kCoefBufs;
      if (lpr == 1) {
        float mix[2][RR];
        float ssq[2] = {0.0f, 0.0f};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int ot = lane + 32 * h;
          if (ot < rpo) {
            float tot[C::kStr];
#pragma unroll
            for (int r = 0; r < C::kStr; ++r) tot[r] = 0.0f;
            for (int cr = 0; cr < nparts; ++cr) {
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
#pragma unroll
            for (int r = 0; r < RR; ++r) mix[h][r] = tot[r];
            ssq[h] = tot[RR];
          }
        }
        __syncwarp();
        if (lane < CL) mbar_arrive_remote(&tail->part_free, (uint32_t)lane);
        if (cuse > 0 &&
            !__all_sync(0xffffffffu, wait_bar<true>(&tail->coef_free[cb], (cuse - 1) & 1u, ctl, kErrClusterWait)))
          break;
        float H[2][NS * NS];                       // residual logits, kept for the Sinkhorn
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int ot = lane + 32 * h;
          if (ot < rpo) {
            const int row = (int)rank * rpo + ot;
            const int tok = tile * kTileT + row;
            float cf[NS];
            const float inv_rms = token_gates<NS, RR>(ep, tok, mix[h], ssq[h], tok < g.T, cf);
            residual_logits<NS, RR>(ep, mix[h], inv_rms, H[h]);
            push_coefs<NS>(coef_buf + ((size_t)cb * kTileT + row) * NS, CL, cf);
          }
        }
        __syncwarp();
        if (lane < CL) mbar_arrive_remote(&tail->coef_full[cb], (uint32_t)lane);
        // Sinkhorn for comb: y no longer waits on this tile
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int ot = lane + 32 * h;
          if (ot < rpo) {
            const int tok = tile * kTileT + (int)rank * rpo + ot;
            sinkhorn_call<NS, C::kThree>(ep, tok, H[h], tok < g.T);
          }
        }
        __syncwarp();
        continue;
      }
      const int ot = lane / lpr;                   // owned row of this lane
      const int part = lane - ot * lpr;            // its share of the row's partials
      float tot[C::kStr];
#pragma unroll
      for (int r = 0; r < C::kStr; ++r) tot[r] = 0.0f;
      for (int cr = part; cr < nparts; cr += lpr) {
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
      for (int off = lpr >> 1; off > 0; off >>= 1) {
#pragma unroll
        for (int r = 0; r <= RR; ++r) tot[r] += __shfl_xor_sync(0xffffffffu, tot[r], off);
      }
      __syncwarp();
      if (lane < CL) mbar_arrive_remote(&tail->part_free, (uint32_t)lane);
      if (cuse > 0 &&
          !__all_sync(0xffffffffu, wait_bar<true>(&tail->coef_free[cb], (cuse - 1) & 1u, ctl, kErrClusterWait)))
        break;
      const int row = (int)rank * rpo + ot;
      // this tile's rows take entries kk rpo .. kk rpo + rpo - 1 of the batch
      const int kk = (int)(k % (uint32_t)lpr);
      if (part == 0) {
        const int tok = tile * kTileT + row;
        float mix[RR];
#pragma unroll
        for (int r = 0; r < RR; ++r) mix[r] = tot[r];
        float cf[NS];
        const float inv_rms = token_gates<NS, RR>(ep, tok, mix, tot[RR], tok < g.T, cf);
        float H[NS * NS];
        residual_logits<NS, RR>(ep, mix, inv_rms, H);
        push_coefs<NS>(coef_buf + ((size_t)cb * kTileT + row) * NS, CL, cf);
        float* hb = sink_h + (size_t)(kk * rpo + ot) * NS * NS;
#pragma unroll
        for (int e = 0; e < NS * NS; ++e) hb[e] = H[e];
        sink_tok[kk * rpo + ot] = tok;
      }
      __syncwarp();
      if (lane < CL) mbar_arrive_remote(&tail->coef_full[cb], (uint32_t)lane);
      if (kk == lpr - 1 || tile + num_clusters >= g.num_tiles) {
        const int bt = sink_tok[lane];
        if (bt >= 0) sinkhorn_call<NS, C::kThree>(ep, bt, sink_h + (size_t)lane * NS * NS, bt < g.T);
        __syncwarp();
        sink_tok[lane] = -1;
        __syncwarp();
      }
    }
  } else if (warp >= kWarpYc0) {
    // ================================================= y for this member's d-range
    // y[t, d] = sum_i m_i x[t, i, d] over the rows of the tile and this
    // member's d-range, re-reading x with plain 16-byte loads (newest d
    // first); kYBatch items per thread are in flight at once, and the next
    // kYBatch items' lines are prefetched into L2.
    const int yt = threadIdx.x - kWarpYc0 * 32;
    const uint64_t read_policy = policy_evict_first();
    const uint64_t ystore_policy = policy_evict_first();
    const int dlo = c0 * kChunkK;
    const int dhi = min(jT * kChunkK, g.D);       // resident mode: the chunks before jT only
    const int w8 = (dhi - dlo) >> 3;              // 16-byte vectors per row
    uint32_t k = 0;
    for (int tile = cluster_id; tile < g.num_tiles; tile += num_clusters, ++k) {
      const int cb = (int)(k % kCoefBufs);
      if (!role_all<kBarY, kYThreads>(wait_bar<true>(&tail->coef_full[cb], (k / kCoefBufs) & 1u, ctl,
                                                     kErrClusterWait)))
        break;
      const float* coef = coef_buf + (size_t)cb * kTileT * NS;
      const int rows = min(kTileT, g.T - tile * kTileT);
      if constexpr (kRes) {
        // y from the TMEM chunks: the warp of lane quarter q = warp % 4 has
        // token et = 32 (q & 1) + lane of the slots sl with sl % 2 == q / 2;
        // the two warps of a quarter split each chunk's eight 16-byte pieces
        const int tb = (int)(k % nbuf);
        if (!role_all<kBarY, kYThreads>(wait_bar<false>(&tail->tm_full[tb], (k / nbuf) & 1u, ctl, kErrWaitTimeout)))
          break;
        tc_fence_after();
        const int qy = warp & 3;
        const int sub = (warp - kWarpYc0) >> 2;
        const int et = (qy & 1) * 32 + lane;
        const int tok = tile * kTileT + et;
        float cf[NS];
#pragma unroll
        for (int i = 0; i < NS; ++i) cf[i] = coef[et * NS + i];
        __nv_bfloat16* yrow = ep.y + (size_t)tok * g.D;
        for (int m = 0; m < CT; ++m) {
          const int sl = tb * cpb + m;
          if ((sl & 1) != (qy >> 1)) continue;
          const uint32_t tx = tmem_base + ((uint32_t)(qy * 32) << 16) + (uint32_t)((sl >> 1) * 128);
#pragma unroll
          for (int pp = 0; pp < 2; ++pp) {          // two pieces of 8 columns at a time
            const int pc = sub * 4 + pp * 2;        // first piece
            uint32_t w[NS][8];
            static_assert(NS == 4, "the resident y reads four streams at once");
            tmem_ld8x4_u32(tx + (uint32_t)(pc * 4), w);
            const int d0 = (jT + m) * kChunkK + pc * 8;
            if (et < rows) {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                if (d0 + h * 8 >= g.D) continue;
                float acc8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc8[e] = 0.0f;
#pragma unroll
                for (int i = 0; i < NS; ++i) {
#pragma unroll
                  for (int q2 = 0; q2 < 4; ++q2) {
                    typename XType<F16>::T2 hv;
                    const uint32_t wv = w[i][h * 4 + q2];
                    memcpy(&hv, &wv, 4);
                    const float2 f = XType<F16>::to_f2(hv);
                    acc8[2 * q2] = fmaf(cf[i], f.x, acc8[2 * q2]);
                    acc8[2 * q2 + 1] = fmaf(cf[i], f.y, acc8[2 * q2 + 1]);
                  }
                }
                uint4 o;
                typename XType<F16>::T2* ob = reinterpret_cast<typename XType<F16>::T2*>(&o);
#pragma unroll
                for (int q2 = 0; q2 < 4; ++q2) ob[q2] = XType<F16>::from_f2(acc8[2 * q2], acc8[2 * q2 + 1]);
                st_global_v4_hint(yrow + d0 + h * 8, o, ystore_policy);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tail->tm_free[tb]);   // a later tile may refill the buffer
      }
      const int items = rows * w8;
      const __nv_bfloat16* xt = xg + (size_t)tile * kTileT * g.n * g.D;
      __nv_bfloat16* yt_out = ep.y + (size_t)tile * kTileT * g.D;
      for (int base = yt; base < items; base += kYThreads * C::kYBatch) {
        if ((lane & 7) == 0) {
          // pull the lines of the next iteration's items into L2 (one lane
          // per 128-byte line): more of the re-read in flight at no register
          // cost (2% at prefill; two or four iterations ahead were no better)
#pragma unroll
          for (int b = 0; b < C::kYBatch; ++b) {
            const int it = base + (C::kYBatch + b) * kYThreads;
            if (it < items) {
              const int row = it / w8;
              const int v = w8 - 1 - (it - row * w8);
              const __nv_bfloat16* src = xt + ((size_t)row * NS) * g.D + dlo + 8 * v;
#pragma unroll
              for (int i = 0; i < NS; ++i) asm volatile("prefetch.global.L2 [%0];" ::"l"(src + (size_t)i * g.D));
            }
          }
        }
        uint4 xv[C::kYBatch][NS];
        int rowv[C::kYBatch], dv[C::kYBatch];
#pragma unroll
        for (int b = 0; b < C::kYBatch; ++b) {
          const int it = base + b * kYThreads;
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
            const typename XType<F16>::T2* hh = reinterpret_cast<const typename XType<F16>::T2*>(&xv[b][i]);
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
              const float2 f = XType<F16>::to_f2(hh[q2]);
              acc8[2 * q2] = fmaf(m, f.x, acc8[2 * q2]);
              acc8[2 * q2 + 1] = fmaf(m, f.y, acc8[2 * q2 + 1]);
            }
          }
          uint4 o;
          typename XType<F16>::T2* ob = reinterpret_cast<typename XType<F16>::T2*>(&o);
#pragma unroll
          for (int q2 = 0; q2 < 4; ++q2) ob[q2] = XType<F16>::from_f2(acc8[2 * q2], acc8[2 * q2 + 1]);
          st_global_v4_hint(yt_out + (size_t)rowv[b] * g.D + dv[b], o, ystore_policy);
        }
      }
      role_sync<kBarY, kYThreads>();               // every y thread is done with coef[cb]
      if (yt < CL) mbar_arrive_remote(&tail->coef_free[cb], (uint32_t)yt);
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(C::kTmemCols)
                 : "memory");
  }
  cluster_sync_all();
}

template <int NS, int RR, int P, bool F16, bool kRes>
const void* kernel_ptr() {
  return reinterpret_cast<const void*>(&mhc_pre_tc_kernel<NS, RR, P, F16, kRes>);
}

// bf16 x: every n; fp16 x: n = 4.  Resident mode: n = 4.
const void* select_kernel(int n, int R, int P, bool fp16, bool res) {
#define MHC_CASE(NS_, RR_, P_) \
  if (!fp16 && !res && n == NS_ && R == RR_ && P == P_) return kernel_ptr<NS_, RR_, P_, false, false>();
#define MHC_CASE16(NS_, RR_, P_) \
  if (fp16 && n == NS_ && R == RR_ && P == P_)                                   \
    return res ? kernel_ptr<NS_, RR_, P_, true, true>() : kernel_ptr<NS_, RR_, P_, true, false>();
#define MHC_CASER(NS_, RR_, P_) \
  if (!fp16 && res && n == NS_ && R == RR_ && P == P_) return kernel_ptr<NS_, RR_, P_, false, true>();
  MHC_CASE(4, 24, 3) MHC_CASE(4, 24, 2) MHC_CASE(4, 8, 3) MHC_CASE(4, 8, 2)
  MHC_CASE(6, 48, 3) MHC_CASE(6, 48, 2) MHC_CASE(6, 12, 3) MHC_CASE(6, 12, 2)
  MHC_CASE(8, 80, 3) MHC_CASE(8, 80, 2) MHC_CASE(8, 16, 3) MHC_CASE(8, 16, 2)
  MHC_CASE16(4, 24, 3) MHC_CASE16(4, 24, 2) MHC_CASE16(4, 8, 3) MHC_CASE16(4, 8, 2)
  MHC_CASER(4, 24, 3) MHC_CASER(4, 24, 2) MHC_CASER(4, 8, 3) MHC_CASER(4, 8, 2)
#undef MHC_CASE
#undef MHC_CASE16
#undef MHC_CASER
  return nullptr;
}

cudaLaunchConfig_t cluster_config(int cluster, int grid, size_t smem, cudaStream_t s,
                                  cudaLaunchAttribute* attr) {
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

int tc_np(int R, int P) { return ((P * R + 15) / 16) * 16; }

bool tc_resident_supported(int n, int R, int P) { return n == 4 && stream_pairs(n, R, P); }

cudaError_t tc_forward_occupancy(int n, int R, int P, bool fp16, bool resident, size_t smem_bytes, int cluster,
                                 int* max_clusters) {
  *max_clusters = 0;
  const void* k = select_kernel(n, R, P, fp16, resident);
  if (!k) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
  if (e != cudaSuccess) return e;
  if (cluster > 8) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config(cluster, cluster, smem_bytes, nullptr, attr);
  return cudaOccupancyMaxActiveClusters(max_clusters, k, &cfg);
}

cudaError_t launch_tc_forward(const TcLaunch& L, cudaStream_t s) {
  const int n = L.epi.n, R = L.epi.R;
  const void* k = select_kernel(n, R, L.P, L.fp16 != 0, L.resident != 0);
  if (!k) return cudaErrorInvalidValue;
  Geometry g;
  g.T = L.epi.T;
  g.D = L.epi.D;
  g.num_tiles = (L.epi.T + kTileT - 1) / kTileT;
  g.nd = (L.epi.D + kChunkK - 1) / kChunkK;
  g.cluster = L.cluster;
  g.n = n;
  g.xstages = L.xstages;
  g.wstages = L.wstages;
  g.wt = L.wt;
  g.tm_bufs = L.tm_bufs;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config(L.cluster, L.grid, L.smem_bytes, s, attr);
  const __nv_bfloat16* xg = static_cast<const __nv_bfloat16*>(L.x);
  const __nv_bfloat16* planes = L.planes;
  void* args[] = {const_cast<CUtensorMap*>(&L.tmap_x), const_cast<__nv_bfloat16**>(&planes),
                  const_cast<EpiParams*>(&L.epi), &xg, &g, const_cast<uint32_t**>(&L.err_word)};
  return cudaLaunchKernelExC(&cfg, k, args);
}

}  // namespace mhc
