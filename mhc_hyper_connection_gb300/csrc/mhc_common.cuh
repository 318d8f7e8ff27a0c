// mhc_common.cuh -- shared device code and launch plumbing of the sm_103a
// mHC pre-mapping forward library.
//
// The per-token epilogue below follows "CANN ops-transformer 中 aclnnMhcPreV2
// 算子接口全解析" §三 (scale by invRms, split pre/post/res, sigmoid gates,
// affine residual logits) and "CANN ops-transformer 算子详解：aclnnMhcPreSinkhorn
// 接口与 MhcPreSinkhorn 实现剖析" §3.2 (Sinkhorn: row softmax + eps, a column
// step, then (row, column) x (numIters - 1), each dividing by sum + eps).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mhc {

// Device error word bits (written into the first 4 bytes of the workspace).
enum : uint32_t {
  kErrWaitTimeout = 1u << 0,   // an mbarrier wait gave up
  kErrClusterWait = 1u << 1,   // a cluster exchange wait gave up
  kErrGridWait = 1u << 2,      // a wait on another CTA's global counter gave up
  kErrPlaneRange = 1u << 3,    // fp16 x: a phi . gamma entry lies outside the fp16 range
};

// Element type of x and y: the conversions the kernels need.
template <bool kF16>
struct XType;
template <>
struct XType<false> {
  using T2 = __nv_bfloat162;
  static __device__ __forceinline__ float2 to_f2(T2 v) { return __bfloat1622float2(v); }
  static __device__ __forceinline__ T2 from_f2(float a, float b) { return __floats2bfloat162_rn(a, b); }
};
template <>
struct XType<true> {
  using T2 = __half2;
  static __device__ __forceinline__ float2 to_f2(T2 v) { return __half22float2(v); }
  static __device__ __forceinline__ T2 from_f2(float a, float b) { return __floats2half2_rn(a, b); }
};
// fp16 planes hold phi . gamma as h0 + h1 2^-11 + h2 2^-22 (each plane
// scaled into fp16's range); bf16 planes need no scale.
__host__ __device__ constexpr float plane_scale(bool f16, int plane) {
  return !f16 ? 1.0f : plane == 0 ? 1.0f : plane == 1 ? 1.0f / 2048.0f : 1.0f / 4194304.0f;
}

// Workspace layout: [0, 256) header, then the phi planes, then the exchange
// rings of the grid-wide forward.  Header words (uint32): 0 error word,
// 1 grid-wide abort flag, [16, 32) partial-arrival counters, [32, 48)
// gated-token counters, [48, 64) y-done counters, one per (group, ring
// slot).  The plane preparation kernel zeroes the whole header before every
// forward.
constexpr size_t kWsHeader = 256;
constexpr int kHdrWords = 64;
constexpr int kHdrAbort = 1, kHdrArrive = 16, kHdrReady = 32, kHdrYdone = 48;

struct EpiParams {
  int T;
  int n, D, R, alpha_len, num_iters;
  float norm_eps, hc_eps;
  const float* bias;           // [R]
  const float* pre_mix;        // [T, n] or null
  __nv_bfloat16* y;            // [T, D]
  float* h_post;               // [T, n]
  float* h_res;                // [T, n, n] or null
  float* h_pre;                // [T, n] or null
  float* inv_rms;              // [T] or null
  float* h_mix;                // [T, R] or null
  float* sum_out;              // [2I, T, n] or null
  float* norm_out;             // [2I, T, n, n] or null
  const float* alpha;          // device alpha (read by kernels)
};

__device__ __forceinline__ float sigmoidf_(float z) { return __fdividef(1.0f, 1.0f + expf(-z)); }

// Sum of v[0..N) as a balanced tree (shorter dependency chain than a scan).
template <int N>
__device__ __forceinline__ float tree_sum(const float* v) {
  if constexpr (N == 1) {
    return v[0];
  } else {
    return tree_sum<N / 2>(v) + tree_sum<N - N / 2>(v + N / 2);
  }
}

// One Sinkhorn column step: every column divided by (its sum + eps).
template <int NS>
__device__ __forceinline__ void sinkhorn_col(float* P, float eps, bool wb, float* sums) {
#pragma unroll
  for (int j = 0; j < NS; ++j) {
    float c[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) c[i] = P[i * NS + j];
    const float s = tree_sum<NS>(c) + eps;
    const float rs = __fdividef(1.0f, s);
#pragma unroll
    for (int i = 0; i < NS; ++i) P[i * NS + j] *= rs;
    if (wb) sums[j] = s;
  }
}
// One Sinkhorn row step: every row divided by (its sum + eps).
template <int NS>
__device__ __forceinline__ void sinkhorn_row(float* P, float eps, bool wb, float* sums) {
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    const float s = tree_sum<NS>(P + i * NS) + eps;
    const float rs = __fdividef(1.0f, s);
#pragma unroll
    for (int j = 0; j < NS; ++j) P[i * NS + j] *= rs;
    if (wb) sums[i] = s;
  }
}

// Per-token gates ("aclnnMhcPreV2 算子接口全解析" §三): scales the projection
// by the RMS reciprocal, writes invRms / hMix / hPre / hPost when `write`,
// returns the weights of y in coef (pre_mix row when given, else hPre) and
// the RMS reciprocal.  RR = NS*NS + 2*NS is the three-gate form, RR = 2*NS
// the two-gate form (hPost + hcEps, no residual path).
template <int NS, int RR>
__device__ __forceinline__ float token_gates_r(const EpiParams& p, int t, const float (&mix)[RR], float inv_rms,
                                               bool write, float (&coef)[NS]);

template <int NS, int RR>
__device__ __forceinline__ float token_gates(const EpiParams& p, int t, const float (&mix)[RR], float ssq,
                                             bool write, float (&coef)[NS]) {
  const float K = (float)(NS * p.D);
  return token_gates_r<NS, RR>(p, t, mix, __frsqrt_rn(ssq / K + p.norm_eps), write, coef);
}

// The same gates from a given RMS reciprocal (the composite route's
// Sinkhorn stage receives it from its own stage).
template <int NS, int RR>
__device__ __forceinline__ float token_gates_r(const EpiParams& p, int t, const float (&mix)[RR], float inv_rms,
                                               bool write, float (&coef)[NS]) {
  constexpr bool kThree = (RR == NS * NS + 2 * NS);
  static_assert(kThree || RR == 2 * NS, "R must be n*n+2n or 2n");
  const float hc_eps = p.hc_eps;
  const float a0 = __ldg(p.alpha), a1 = __ldg(p.alpha + 1);
  if (write) {
    if (p.inv_rms) p.inv_rms[t] = inv_rms;
    if (p.h_mix) {
#pragma unroll
      for (int r = 0; r < RR; ++r) p.h_mix[(size_t)t * RR + r] = mix[r];
    }
  }
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    const float pre = sigmoidf_(a0 * (mix[i] * inv_rms) + __ldg(p.bias + i)) + hc_eps;
    float post = 2.0f * sigmoidf_(a1 * (mix[NS + i] * inv_rms) + __ldg(p.bias + NS + i));
    if (!kThree) post += hc_eps;
    coef[i] = pre;
    if (write) {
      p.h_post[(size_t)t * NS + i] = post;
      if (p.h_pre) p.h_pre[(size_t)t * NS + i] = pre;
    }
  }
  if (p.pre_mix) {
#pragma unroll
    for (int i = 0; i < NS; ++i) coef[i] = __ldg(p.pre_mix + (size_t)t * NS + i);
  }
  return inv_rms;
}

// Residual logits of one token: H = alpha2 * pRes + bias2, pRes the res
// segment of the projection scaled by invRms, reshaped row-major to n x n.
template <int NS, int RR>
__device__ __forceinline__ void residual_logits(const EpiParams& p, const float (&mix)[RR], float inv_rms,
                                                float (&H)[NS * NS]) {
  constexpr int NN = NS * NS;
  if constexpr (RR == NN + 2 * NS) {
    const float a2 = __ldg(p.alpha + 2);
#pragma unroll
    for (int e = 0; e < NN; ++e) H[e] = a2 * (mix[2 * NS + e] * inv_rms) + __ldg(p.bias + 2 * NS + e);
  } else {
#pragma unroll
    for (int e = 0; e < NN; ++e) H[e] = 0.0f;
  }
}

// Residual mix of one token ("aclnnMhcPreSinkhorn 接口与 MhcPreSinkhorn 实现
// 剖析" §3.2) from its logits H: softmax over each row + eps, a column step,
// then (row, column) x (numIters - 1); each step divides by (sum + eps).
// Writes comb and, when sum_out is set, every step's sums and matrices.
// Two-gate form (no residual path): comb is zero.
template <int NS, bool kThree>
__device__ __forceinline__ void token_sinkhorn(const EpiParams& p, int t, const float* H, bool write) {
  constexpr int NN = NS * NS;
  if constexpr (!kThree) {
    if (write && p.h_res) {
#pragma unroll
      for (int e = 0; e < NN; ++e) p.h_res[(size_t)t * NN + e] = 0.0f;
    }
  } else {
    const float hc_eps = p.hc_eps;
    float P[NN];
#pragma unroll
    for (int e = 0; e < NN; ++e) P[e] = H[e];
    const size_t Tn = (size_t)p.T * NS, Tnn = (size_t)p.T * NN;
    const bool wb = write && (p.sum_out != nullptr);
    float* sums = wb ? p.sum_out : nullptr;
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      float m = P[i * NS];
#pragma unroll
      for (int j = 1; j < NS; ++j) m = fmaxf(m, P[i * NS + j]);
      float e[NS];
#pragma unroll
      for (int j = 0; j < NS; ++j) e[j] = expf(P[i * NS + j] - m);
      const float s = tree_sum<NS>(e);
      const float rs = __fdividef(1.0f, s);
#pragma unroll
      for (int j = 0; j < NS; ++j) P[i * NS + j] = fmaf(e[j], rs, hc_eps);
      if (wb) sums[(size_t)t * NS + i] = s;
    }
    if (wb) {
#pragma unroll
      for (int e = 0; e < NN; ++e) p.norm_out[(size_t)t * NN + e] = P[e];
    }
    sinkhorn_col<NS>(P, hc_eps, wb, wb ? sums + Tn + (size_t)t * NS : nullptr);
    if (wb) {
#pragma unroll
      for (int e = 0; e < NN; ++e) p.norm_out[Tnn + (size_t)t * NN + e] = P[e];
    }
    // without the backward's outputs the steps run with no stores between
    // them (the same arithmetic, a tighter loop)
    if (!wb) {
      for (int it = 1; it < p.num_iters; ++it) {
        sinkhorn_row<NS>(P, hc_eps, false, nullptr);
        sinkhorn_col<NS>(P, hc_eps, false, nullptr);
      }
    } else
    for (int it = 1; it < p.num_iters; ++it) {
      const int k = 2 * it;
      sinkhorn_row<NS>(P, hc_eps, wb, wb ? sums + k * Tn + (size_t)t * NS : nullptr);
      if (wb) {
#pragma unroll
        for (int e = 0; e < NN; ++e) p.norm_out[k * Tnn + (size_t)t * NN + e] = P[e];
      }
      sinkhorn_col<NS>(P, hc_eps, wb, wb ? sums + (k + 1) * Tn + (size_t)t * NS : nullptr);
      if (wb) {
#pragma unroll
        for (int e = 0; e < NN; ++e) p.norm_out[(k + 1) * Tnn + (size_t)t * NN + e] = P[e];
      }
    }
    if (write && p.h_res) {
#pragma unroll
      for (int e = 0; e < NN; ++e) p.h_res[(size_t)t * NN + e] = P[e];
    }
  }
}

// ---------------------------------------------------------------------------
// Host-side launch descriptions shared by the API translation unit and the
// kernel translation units.
// ---------------------------------------------------------------------------
// The phi planes are stored as the shared-memory image the MMA reads: for
// each 64-wide d-chunk j and stream i a block of RB = P*R (rounded up to 8)
// rows of 128 bytes (row p*R + r = plane p of phi row r; rows past P*R and
// columns past D are zero), with the 128-byte swizzle already applied (the
// 16-byte piece c of row r sits at c ^ (r & 7)).  Blocks are ordered
// [chunk][stream], so the blocks of consecutive streams of one chunk are one
// contiguous run that a single bulk copy brings in.
struct PlaneParams {
  const float* phi;        // [R, n*D]
  const float* gamma;      // [n*D] or null
  __nv_bfloat16* planes;   // [nch][n][RB][64], swizzled
  int R, P, n, D, nch, RB; // P = 3 (fp32) or 2 (tf32)
  int tf32;
  int fp16;                // planes in fp16 (scaled, see plane_scale) for fp16 x
  int vec16;               // phi (and gamma) 16-byte aligned: vector loads
  uint32_t* err_word;      // workspace header: all kHdrWords words are zeroed
};

cudaError_t launch_prepare_planes(const PlaneParams& pp, cudaStream_t s);

constexpr int kMmaM = 128;         // rows of one tcgen05.mma (TMEM lanes)
constexpr int kTileT = 64;         // tokens per tile: MMA rows 0..63 (rows 64..127: a stream pair's second stream)
constexpr int kChunkK = 64;        // bf16 elements per 128-byte swizzle row
constexpr int kStreamTile = kTileT * 128;   // one stream of one d-chunk of a tile (8 KB)
constexpr int kThreads = 512;      // 16 warps: 2 TMA producers, MMA, 2 publish, gates, Sinkhorn, 8 y
constexpr int kMaxStages = 8;      // ring depth limit (barrier arrays)
constexpr int kCoefBufs = 3;       // y-weight buffers between the gate warps and the y warps
constexpr size_t kTailBytes = 1024; // barriers and flags

// Streams per x box: the box is (64 columns, 64 tokens, this many
// streams): 32 KB for n = 4 and n = 8 (two boxes per d-chunk), 24 KB for
// n = 6.  Big boxes matter: one issuing thread completes only about two
// boxes per microsecond, whatever their size.
__host__ __device__ constexpr int stream_group(int n) { return n == 6 ? 3 : 4; }
// Rows of one stream's phi planes in a w box: P*R rounded up to 8.  The
// MMA's N = P*R rounded up to 16 reads the rest from the next stream (or
// slot); those accumulator columns are never read.
__host__ __device__ constexpr int plane_box_rows(int R, int P) { return ((P * R + 7) / 8) * 8; }
// Streams per w box: the largest divisor of n whose planes stay within 36 KB.
__host__ __device__ constexpr int w_group(int n, int R, int P) {
  return (n % 4 == 0 && 4 * plane_box_rows(R, P) * 128 <= 36864)   ? 4
         : (n % 3 == 0 && 3 * plane_box_rows(R, P) * 128 <= 36864) ? 3
         : (n % 2 == 0 && 2 * plane_box_rows(R, P) * 128 <= 36864) ? 2
                                                                    : 1;
}
// Whether the 64-token kernel runs two streams per MMA: the box holds an
// even number of streams, and two streams' plane rows fit N <= 256.
__host__ __device__ constexpr bool stream_pairs(int n, int R, int P) {
  return stream_group(n) % 2 == 0 && w_group(n, R, P) % 2 == 0 && 2 * plane_box_rows(R, P) <= 256;
}
// Floats per published partial (R sums + the sum of squares), padded to 16 bytes.
__host__ __device__ constexpr int partial_stride(int R) { return ((R + 1 + 3) / 4) * 4; }
// Floats per Sinkhorn hand-off entry: the n*n residual logits of one token.
__host__ __device__ constexpr int sink_stride(int n) { return n * n; }

// Byte offsets of the forward kernel's shared-memory regions (after the
// base is rounded up to 1024); `total` includes that rounding slack.  The x
// and w rings are back to back, so an operand read that runs past a slot
// stays inside the window.
struct SmemLayout {
  size_t x, w, part, coef, sink, tail, total;
};
__host__ __device__ inline SmemLayout smem_layout(int n, int R, int P, int xs, int ws) {
  SmemLayout L;
  size_t o = 0;
  L.x = o;    o += (size_t)xs * stream_group(n) * kStreamTile;
  L.w = o;    o += (size_t)ws * w_group(n, R, P) * plane_box_rows(R, P) * 128;
  o += 1024;  // the B operand of N = NP rows reads up to 8 rows past the last w box
  // two partials per member and row with stream pairs (each half of the
  // publish warps has projection sums), else one
  L.part = o; o += (stream_pairs(n, R, P) ? 2 : 1) * (size_t)kTileT * partial_stride(R) * 4;
  L.coef = o; o += (size_t)kCoefBufs * kTileT * n * 4;
  L.sink = o; o += (size_t)32 * n * n * 4 + 32 * 4;   // a Sinkhorn batch: 32 tokens' logits and indices
  o = (o + 15) & ~size_t(15);
  L.tail = o; o += kTailBytes;
  L.total = o + 1024;
  return L;
}

// Wait limit and test hook shared by the forward kernels: wait_ns bounds
// every wait; withhold_x = 1 makes CTA 0's x producer leave out its last
// copy (it issues nothing for it), so the waits on it give up and the run
// ends through the abort path with the error word set -- a host-requested
// test of that path that faults nothing.
struct WaitTest {
  uint64_t wait_ns;
  int withhold_x;
};

struct Geometry {
  int T, D, n;
  int num_tiles, nd;           // token tiles; 64-wide d-chunks per stream
  int cluster, xstages, wstages;
  int tm_bufs;                 // resident mode: TMEM chunk buffers (1 or 2)
  WaitTest wt;
};

struct TcLaunch {
  EpiParams epi;
  const void* x;           // bf16 [T, n, D] (re-read for y)
  CUtensorMap tmap_x;      // x as (D, T, n): box (64, 64 tokens, stream group), 128B swizzle
  const __nv_bfloat16* planes;   // swizzled plane blocks (see PlaneParams)
  int NP, P;
  int fp16;                // x and y fp16 (planes fp16)
  int resident;            // 1: the last chunks of each CTA's range stay in TMEM for y
  int tm_bufs;             // resident mode: TMEM chunk buffers used by alternate tiles (1 or 2)
  int cluster;             // CTAs per token tile (split over d-chunks)
  int grid;                // CTAs (multiple of cluster)
  int xstages, wstages;
  size_t smem_bytes;
  uint32_t* err_word;
  WaitTest wt;
};

// ---------------------------------------------------------------------------
// Post-mapping (hc_post): out[t][j] = post[t][j] x[t] + sum_i comb[t][i][j] residual[t][i].
// ---------------------------------------------------------------------------
struct PostLaunch {
  int64_t T, n, D;
  const void* x;           // bf16 [T, D]
  const void* residual;    // bf16 [T, n, D]
  const float* post;       // [T, n]
  const float* comb;       // [T, n, n]
  void* out;               // bf16 [T, n, D]
};
cudaError_t launch_post(const PostLaunch& L, cudaStream_t s);

// ---------------------------------------------------------------------------
// Composite route (the pages' two-operator path, a debug aid): invRms, the
// projection ("mixes"), then gates + Sinkhorn + y from them.
struct StageLaunch {
  int T, n, D, R, fp16;
  float norm_eps;
  const void* x;               // [T, n, D] bf16 or fp16
  const float* phi;            // [R, nD]
  const float* gamma;          // [nD] or null
  float* inv_rms;              // [T]
  float* mixes;                // [T, R]
};
cudaError_t launch_stage_inv_rms(const StageLaunch& L, cudaStream_t s);
cudaError_t launch_stage_mixes(const StageLaunch& L, cudaStream_t s);
// ep holds the outputs (y, h_post, h_res, h_pre, sum_out, norm_out and, when
// set, copies of inv_rms / h_mix); mixes and inv_rms are the stage inputs.
cudaError_t launch_stage_sinkhorn(const EpiParams& ep, const void* x, const float* mixes, const float* inv_rms,
                                  int fp16, cudaStream_t s);

// Resolved by the kernel translation unit for the given (n, R, P).
cudaError_t launch_tc_forward(const TcLaunch& L, cudaStream_t s);
// Clusters of the given size that fit on the device at once (0: unsupported).
cudaError_t tc_forward_occupancy(int n, int R, int P, bool fp16, bool resident, size_t smem_bytes, int cluster,
                                 int* max_clusters);
// Shapes the resident mode of the cluster kernel takes (n = 4, stream pairs).
bool tc_resident_supported(int n, int R, int P);
int tc_np(int R, int P);

// ---------------------------------------------------------------------------
// Grid-wide forward: one CTA per SM, all resident (cooperative launch), split
// into ng groups of G CTAs that take alternate 64-token tiles.  Every CTA of a
// group owns a fixed run of 64-wide d-chunks of one stream and works on every
// tile of its group; per-CTA partial sums meet in a global ring, one CTA per
// token gates it, and each CTA forms y for its own d-range.
// ---------------------------------------------------------------------------
constexpr int kGwTile = 64;                   // tokens per tile (rows 0..63 of an M = 128 MMA)
constexpr int kGwUnitBytes = kGwTile * 128;   // one (d-chunk, stream) x box: 8 KB
constexpr int kGwSlots = 8;                   // exchange-ring depth per group, in tiles
constexpr int kGwMaxGroups = 2;               // kGwMaxGroups * kGwSlots <= 16 header words
constexpr int kGwSinkMax = 32;                // Sinkhorn tokens per batch (one per lane)

__host__ __device__ constexpr int gw_np(int R, int P) { return ((P * R + 15) / 16) * 16; }

struct GwLayout {
  size_t phi, x, ycoef, sink, scnt, tail, total;
};
// Shared memory of the grid-wide kernel: the CTA's resident phi-plane blocks
// (RB rows each, back to back, plus 1 KB that the N = NP operand reads run into),
// the x ring (xs slots of umax units, plus one unit of slack that the M = 128
// operand reads run into), the y weights of two tiles, two Sinkhorn batches
// and the barrier block.
__host__ __device__ inline GwLayout gw_layout(int n, int R, int P, int umax, int xs) {
  GwLayout L;
  size_t o = 0;
  L.phi = o;   o += (size_t)umax * plane_box_rows(R, P) * 128 + 1024;   // + the N = NP over-read
  L.x = o;     o += ((size_t)xs * umax + 1) * kGwUnitBytes;
  L.ycoef = o; o += 2 * (size_t)kGwTile * n * 4;
  L.sink = o;  o += 2 * (size_t)kGwSinkMax * n * n * 4;
  L.scnt = o;  o += 2 * (size_t)kGwSinkMax * 4;
  o = (o + 15) & ~size_t(15);
  L.tail = o;  o += kTailBytes;
  L.total = o + 1024;
  return L;
}
// Bytes of the exchange rings after the planes for up to `ctas` CTAs in all:
// partials [groups][slots][64][G][stride] and y weights [groups][slots][64][n].
inline size_t gw_ring_bytes(int n, int R, int ctas) {
  return (size_t)kGwSlots * kGwTile * ctas * partial_stride(R) * 4 +
         (size_t)kGwMaxGroups * kGwSlots * kGwTile * n * 4;
}

struct GwGeom {
  int T, D, n;
  int num_tiles;   // 64-token tiles
  int nch;         // 64-wide d-chunks per stream
  int ng;          // groups (tiles k with k % ng == g go to group g)
  int G;           // CTAs per group: n streams x gs CTAs per stream
  int gs;          // CTAs per stream; CTA r takes stream r / gs, a run of its chunks
  int box4d;       // 1: a CTA's chunks of a tile come as one 4-D box (D % 64 == 0)
  int umax;        // most chunks any CTA owns
  int xstages;     // x ring depth
  int own_max;     // most tokens of one tile any CTA gates
  int sink_batch;  // tiles per Sinkhorn batch (sink_batch * own_max <= kGwSinkMax)
  int xlead;       // most tiles the x loads run ahead of this CTA's y (1..15)
  WaitTest wt;
};

struct GwLaunch {
  EpiParams epi;
  const void* x;           // bf16 [T, n, D] (re-read for y)
  CUtensorMap tmap_x;      // x as (64, T, chunks, n), box (64, 64 tokens, umax, 1), or as
                           // (D, T, n), box (64, 64, 1) when D % 64 != 0; 128B swizzle
  const __nv_bfloat16* planes;   // swizzled plane blocks (see PlaneParams)
  int P;
  GwGeom g;
  size_t smem_bytes;
  uint32_t* hdr;           // workspace header
  float* partials;         // exchange ring of partial sums
  float* coefs;            // exchange ring of y weights
};

// Largest number of CTAs of the grid-wide kernel resident at once for this
// shared-memory size (0: it does not fit).
cudaError_t gw_forward_capacity(int n, int R, int P, size_t smem_bytes, int* max_ctas);
cudaError_t launch_gw_forward(const GwLaunch& L, cudaStream_t s);

// ---------------------------------------------------------------------------
// Backward of the pre-mapping (n = 4, three gates).  Five launches:
//  1. planes: phi . gamma per 64-column slab as P bf16 planes, row-padded to
//     kBwRp rows, swizzled for the tensor core; zeroes the header;
//  2. row dot: H_pre_grad[t][i] = grad_h_in[t] . x[t][i] (whole rows streamed
//     through a bulk-copy ring);
//  2b. token stage: per token the gate and Sinkhorn backward -> G = H_mix_grad
//     (as P bf16 planes in a per-64-token tile record) and the RMS factor;
//     per-warp partial sums of grad_alpha / grad_bias;
//  3. main: per (slab, token tile) grad_x = gx3 + G phi' + c x (+ grad_x_post)
//     and x^T G accumulated over the tiles of a unit (slab, token chunk);
//  4. final: grad_phi / grad_gamma from the run partials, grad_alpha /
//     grad_bias from the warp partials, all in fixed order.
constexpr int kBwNS = 4, kBwR = 24, kBwRp = 32;   // streams, gate rows, rows padded to the MMA K step
constexpr int kBwTile = 64;                        // tokens per tile
constexpr int kBwPlaneBytes = kBwRp * 128;         // one plane: kBwRp rows of 64 bf16
constexpr int kBwScalarBytes = kBwTile * 32;       // [stream][token] (hPre_i, RMS factor) pairs
constexpr int kBwMaxMainGrid = 160;                // main-kernel CTAs the workspace is sized for
constexpr int kBwMaxTokenBlocks = 1024;            // token-stage blocks (8 warps each)
constexpr int kBwTokenWarps = 8;

__host__ __device__ constexpr int bw_slab_bytes(int P) { return kBwNS * P * kBwPlaneBytes; }
__host__ __device__ constexpr int bw_tile_rec_bytes(int P) { return P * kBwPlaneBytes + kBwScalarBytes; }
__host__ __device__ constexpr int bw_mt_cols(int P) { return P * kBwRp; }
__host__ __device__ constexpr int bw_stage_bytes(int P, bool gxp) {
  return kBwNS * kBwTile * 128 * (gxp ? 2 : 1) + kBwTile * 128 + bw_tile_rec_bytes(P);
}
constexpr int kBwTailBytes = 1024;

constexpr int kBwMaxChunks = 8;                    // token chunks per slab (units = slabs x chunks)
__host__ __device__ constexpr size_t bw_piece_bytes() { return (size_t)kBwRp * kBwNS * 64 * 4; }

struct BwPlaneParams {
  const float* phi;        // [R, nD]
  const float* gamma;      // [nD] or null
  __nv_bfloat16* planes;   // [nslab][NS][P][kBwRp][64], swizzled
  uint32_t* hdr;           // workspace header (zeroed)
  int D, nslab, P, tf32;
  int vec16;               // phi (and gamma) 16-byte aligned: vector loads
};

struct BwRowdotParams {
  int T, D, tps, stages;       // tokens per ring stage, ring depth
  const __nv_bfloat16* x;      // [T, n, D]
  const __nv_bfloat16* g_in;   // [T, D]
  float* hg;                   // [T, n]: H_pre_grad
  uint32_t* err;
};

struct BwTokenParams {
  int T, D, ntiles, num_iters, P, tf32;
  float hc_eps;
  const float* hg;             // [T, n]: H_pre_grad from the row-dot kernel
  const float* g_post;         // [T, n]
  const float* g_res;          // [T, n, n]
  const float* inv_rms;        // [T]
  const float* h_mix;          // [T, R]
  const float* h_pre;          // [T, n]
  const float* h_post;         // [T, n]
  const float* sum_out;        // [2I, T, n] or null
  const float* norm_out;       // [2I, T, n, n] or null
  const float* alpha;          // [3]
  uint8_t* tiles;              // [ntiles] tile records
  float* partials;             // [blocks * 8][32]
  int saved16;                 // sum_out and norm_out 16-byte aligned: asynchronous 16-byte copies
};

struct BwMainLaunch {
  CUtensorMap tmap_x, tmap_gin, tmap_gxp;
  const __nv_bfloat16* planes;
  __nv_bfloat16* grad_x;       // [T][n][D], written by the epilogue warps
  const uint8_t* tiles;
  float* pieces;               // [nslab * nq][kBwRp][NS * 64]: x^T G per unit, planes summed
  uint32_t* err;
  int T, D, ntiles, nslab, nq, P, stages, has_gxp, grid;
  size_t smem_bytes;
  WaitTest wt;                 // wait limit; withhold_x: CTA 0 leaves out its last tile's copies
};

struct BwFinalParams {
  int D, nslab, nq;
  const float* pieces;
  const float* phi;                // [R, nD]
  const float* gamma;              // [nD] or null
  float* grad_phi;                 // [R, nD]
  float* grad_gamma;               // [nD] or null
  const float* partials;           // [nparts][32]
  int nparts;
  float* grad_alpha;               // [3]
  float* grad_bias;                // [R]
};

cudaError_t launch_bw_planes(const BwPlaneParams& p, cudaStream_t s);
// Row-dot ring: tokens per stage and stage count for this shape (0 stages:
// does not fit), and its launch.
void bw_rowdot_shape(int D, size_t max_smem, int* tps, int* stages, size_t* smem_bytes);
cudaError_t launch_bw_rowdot(const BwRowdotParams& p, int grid, size_t smem_bytes, cudaStream_t s);
cudaError_t bw_token_blocks(int* blocks);      // token-stage grid for this device
cudaError_t launch_bw_token(const BwTokenParams& p, int blocks, cudaStream_t s);
cudaError_t launch_bw_main(const BwMainLaunch& L, cudaStream_t s);
cudaError_t launch_bw_final(const BwFinalParams& p, cudaStream_t s);

}  // namespace mhc
