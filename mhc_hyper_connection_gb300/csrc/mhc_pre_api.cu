// mhc_pre_api.cu -- host side of the C ABI declared in include/mhc_pre.h:
// argument checks, workspace sizing, tensor maps, launch configuration.
//
// The two-phase shape of the API (size the workspace, then run on a stream)
// and the status codes follow "aclnnMhcPreSinkhorn 接口与 MhcPreSinkhorn 实现
// 剖析" §4, §6 and "aclnnMhcPreV2 算子接口全解析" §四, §5.4; the optional
// output group (all or none) follows the same page's §7.3.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "mhc_common.cuh"
#include "../../include/mhc_pre.h"
#include "../../include/mhc_post.h"
#include "../../include/mhc_pre_backward.h"
#include "../../include/mhc_pre_stages.h"

struct mhc_pre_s {
  mhc_pre_config cfg;
  int R;        // projection rows
  int P;        // precision planes (3: fp32, 2: tf32)
  int NP;       // MMA N = P*R rounded up to 16
  cudaEvent_t ev_before = nullptr, ev_after = nullptr;   // optional timing hooks
  int last_cluster = 0, last_grid = 0, last_stages = 0, last_ystages = 0;   // last launch shape
  const char* last_kernel = "";                                              // and its kernel
  void* last_noalloc_word = nullptr;   // error word of the last run when it was mhc_pre_run_noalloc
  mhc::WaitTest wait_test{2000000000ull, 0};   // device wait limit and test hook (mhc_pre_set_wait_test)
};

namespace {

thread_local char g_last_error[512] = "";

mhc_status_t fail(mhc_status_t code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry-point lookup (the
// library does not link the driver library directly).
CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D bf16 map: dims[0] contiguous, byte strides of dims 1 and 2 given
// explicitly (they need not increase), 128-byte swizzle, zero fill outside.
bool encode_3d(CUtensorMap* map, const void* base, const uint64_t dims[3], const uint64_t strides[2],
               const uint32_t box[3]) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {strides[0], strides[1]};
  cuuint32_t b[3] = {box[0], box[1], box[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), d, st, b, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D bf16 map, same conventions (byte strides of dims 1..3 explicit).
bool encode_4d(CUtensorMap* map, const void* base, const uint64_t dims[4], const uint64_t strides[3],
               const uint32_t box[4]) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t st[3] = {strides[0], strides[1], strides[2]};
  cuuint32_t b[4] = {box[0], box[1], box[2], box[3]};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), d, st, b, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct DeviceInfo {
  bool ok = false;
  int sms = 0;
  size_t max_smem = 0;
  size_t l2_bytes = 0;
};

DeviceInfo device_info(int dev) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool known[64] = {};
  std::lock_guard<std::mutex> lk(mu);
  if (dev < 0 || dev >= 64) return DeviceInfo{};
  if (!known[dev]) {
    DeviceInfo d;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) == cudaSuccess) {
      d.ok = (prop.major == 10 && prop.minor == 3);
      d.sms = prop.multiProcessorCount;
      d.max_smem = prop.sharedMemPerBlockOptin;
      d.l2_bytes = (size_t)prop.l2CacheSize;
    }
    cache[dev] = d;
    known[dev] = true;
  }
  return cache[dev];
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Swizzled plane blocks: [chunk][stream][RB rows][128 bytes].
size_t planes_bytes(const mhc_pre_s* h) {
  const size_t nch = (size_t)((h->cfg.D + mhc::kChunkK - 1) / mhc::kChunkK);
  const size_t RB = (size_t)mhc::plane_box_rows(h->R, h->P);
  return (nch * (size_t)h->cfg.n * RB * 128 + 255) & ~size_t(255);
}

// Exchange rings of the grid-wide forward, sized for its largest grid so the
// workspace does not depend on the device.
constexpr int kGwMaxGrid = 160;
size_t gw_rings_bytes(const mhc_pre_s* h) {
  return mhc::gw_ring_bytes((int)h->cfg.n, h->R, kGwMaxGrid);
}

// Returned by run_grid_wide when the shape or device does not suit it.
constexpr mhc_status_t MHC_ERR_NOT_SUITABLE = -1;

mhc::EpiParams epi_params(const mhc_pre_s* h, const mhc_pre_args* a) {
  const mhc_pre_config& c = h->cfg;
  mhc::EpiParams e;
  memset(&e, 0, sizeof e);
  e.T = (int)a->T;
  e.n = (int)c.n;
  e.D = (int)c.D;
  e.R = h->R;
  e.alpha_len = c.alpha_len;
  e.num_iters = c.num_iters;
  e.norm_eps = (float)c.norm_eps;
  e.hc_eps = (float)c.hc_eps;
  e.alpha = a->alpha;
  e.bias = a->bias;
  e.pre_mix = a->pre_mix;
  e.y = static_cast<__nv_bfloat16*>(a->y);
  e.h_post = a->h_post;
  e.h_res = a->h_res;
  e.h_pre = a->h_pre;
  e.inv_rms = a->inv_rms;
  e.h_mix = a->h_mix;
  e.sum_out = a->sum_out;
  e.norm_out = a->norm_out;
  return e;
}

// The grid-wide forward: one CTA per SM in ng groups of G = n * gs, CTA r of
// a group owning a run of the d-chunks of stream r / gs; MHC_ERR_NOT_SUITABLE
// when its resident phi blocks and a two-slot x ring do not fit, or the grid
// cannot be resident at once.  Two groups when there are enough tiles to keep
// both busy (the handle's gw_groups overrides).
mhc_status_t run_grid_wide(mhc_pre_s* h, const mhc_pre_args* a, const DeviceInfo& di,
                           __nv_bfloat16* planes, cudaStream_t s) {
  const int n = (int)h->cfg.n, D = (int)h->cfg.D, R = h->R;
  const int nch = (D + mhc::kChunkK - 1) / mhc::kChunkK;
  const int num_tiles = (int)((a->T + mhc::kGwTile - 1) / mhc::kGwTile);
  const int sms = di.sms < kGwMaxGrid ? di.sms : kGwMaxGrid;
  int ng = h->cfg.gw_groups ? h->cfg.gw_groups : (num_tiles >= 8 ? 2 : 1);
  ng = ng < 1 ? 1 : (ng > mhc::kGwMaxGroups ? mhc::kGwMaxGroups : ng);
  int gs = sms / ng / n;
  if (gs > nch) gs = nch;
  if (gs < 1) return MHC_ERR_NOT_SUITABLE;
  const int G = n * gs;
  const int umax = (nch + gs - 1) / gs;
  const bool box4d = (D % mhc::kChunkK) == 0;
  const int own_max = (mhc::kGwTile + G - 1) / G;
  if (umax > 32 || own_max > mhc::kGwSinkMax) return MHC_ERR_NOT_SUITABLE;
  int sink_batch = mhc::kGwSinkMax / own_max;
  if (sink_batch > 8) sink_batch = 8;
  int xmax = h->cfg.gw_x_stages ? h->cfg.gw_x_stages : mhc::kMaxStages;
  xmax = xmax < 2 ? 2 : (xmax > mhc::kMaxStages ? mhc::kMaxStages : xmax);
  int xs = 0;
  for (int c = xmax; c >= 2 && !xs; --c)
    if (mhc::gw_layout(n, R, h->P, umax, c).total <= di.max_smem) xs = c;
  if (!xs) return MHC_ERR_NOT_SUITABLE;
  const size_t smem = mhc::gw_layout(n, R, h->P, umax, xs).total;
  int cap = 0;
  if (mhc::gw_forward_capacity(n, R, h->P, smem, &cap) != cudaSuccess) {
    cudaGetLastError();
    return MHC_ERR_NOT_SUITABLE;
  }
  if (cap < ng * G) return MHC_ERR_NOT_SUITABLE;

  mhc::GwLaunch L;
  memset(&L, 0, sizeof L);
  L.epi = epi_params(h, a);
  L.x = a->x;
  L.P = h->P;
  L.g.T = (int)a->T;
  L.g.D = D;
  L.g.n = n;
  L.g.num_tiles = num_tiles;
  L.g.nch = nch;
  L.g.ng = ng;
  L.g.G = G;
  L.g.gs = gs;
  L.g.box4d = box4d ? 1 : 0;
  L.g.umax = umax;
  L.g.xstages = xs;
  L.g.own_max = own_max;
  L.g.sink_batch = sink_batch;
  int xlead = h->cfg.gw_x_lead ? h->cfg.gw_x_lead : 6;
  L.g.xlead = xlead < 1 ? 1 : (xlead > 15 ? 15 : xlead);
  L.g.wt = h->wait_test;
  L.smem_bytes = smem;
  uint8_t* ws = static_cast<uint8_t*>(a->workspace);
  L.hdr = reinterpret_cast<uint32_t*>(ws);
  L.partials = reinterpret_cast<float*>(ws + mhc::kWsHeader + planes_bytes(h));
  L.coefs = L.partials + (size_t)mhc::kGwSlots * mhc::kGwTile * (ng * G) * mhc::partial_stride(R);
  L.planes = planes;
  {
    const uint64_t K2 = (uint64_t)n * D * 2;
    bool enc;
    if (box4d) {
      // x [T][n][D] seen as (64, T, chunk, n), box (64, 64 tokens, umax chunks, 1
      // stream): shared memory then holds one 64-row block per chunk.
      const uint64_t xd[4] = {(uint64_t)mhc::kChunkK, (uint64_t)a->T, (uint64_t)nch, (uint64_t)n};
      const uint64_t xst[3] = {K2, (uint64_t)mhc::kChunkK * 2, (uint64_t)D * 2};
      const uint32_t xb[4] = {(uint32_t)mhc::kChunkK, (uint32_t)mhc::kGwTile, (uint32_t)umax, 1u};
      enc = encode_4d(&L.tmap_x, a->x, xd, xst, xb);
    } else {
      // x as (D, T, n), box (64, 64 tokens, 1 stream), one box per chunk.
      const uint64_t xd[3] = {(uint64_t)D, (uint64_t)a->T, (uint64_t)n};
      const uint64_t st[2] = {K2, (uint64_t)D * 2};
      const uint32_t xb[3] = {(uint32_t)mhc::kChunkK, (uint32_t)mhc::kGwTile, 1u};
      enc = encode_3d(&L.tmap_x, a->x, xd, st, xb);
    }
    if (!enc) return fail(MHC_ERR_RUNTIME, "tensor map encoding failed");
  }
  h->last_cluster = 0;
  h->last_kernel = "mhc_pre_gw_kernel";
  h->last_grid = ng * G;
  h->last_stages = xs;
  h->last_ystages = ng;
  if (h->ev_before && cudaEventRecord(h->ev_before, s) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "recording the timing event failed");
  if (mhc::launch_gw_forward(L, s) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "forward launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  if (h->ev_after && cudaEventRecord(h->ev_after, s) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "recording the timing event failed");
  return MHC_OK;
}

}  // namespace

extern "C" {

void mhc_pre_config_default(mhc_pre_config* c) {
  if (!c) return;
  c->n = 4;
  c->D = 0;
  c->alpha_len = 3;
  c->num_iters = 20;
  c->norm_eps = 1e-6;
  c->hc_eps = 1e-6;
  c->impl_mode = MHC_IMPL_FP32;
  c->need_backward = 0;
  c->batch_consistent = 0;
  c->x_dtype = MHC_DTYPE_BF16;
  c->kernel = MHC_KERNEL_AUTO;
  c->cluster = 0;
  c->x_stages = 0;
  c->w_stages = 0;
  c->gw_groups = 0;
  c->gw_x_stages = 0;
  c->gw_x_lead = 0;
  c->tm_buffers = 0;
}

const char* mhc_pre_last_error(void) { return g_last_error; }

const char* mhc_pre_status_string(mhc_status_t s) {
  switch (s) {
    case MHC_OK: return "success";
    case MHC_ERR_NULLPTR: return "a required pointer is NULL";
    case MHC_ERR_PARAM_INVALID: return "invalid parameter (shape, mode, alignment or output group)";
    case MHC_ERR_RUNTIME: return "CUDA runtime or device-side failure";
    default: return "unknown status";
  }
}

mhc_status_t mhc_pre_create(mhc_pre_t* out, const mhc_pre_config* cfg) {
  g_last_error[0] = 0;
  if (!out || !cfg) return fail(MHC_ERR_NULLPTR, "out and cfg must be non-NULL");
  *out = nullptr;
  const mhc_pre_config& c = *cfg;
  if (c.n != 4 && c.n != 6 && c.n != 8) return fail(MHC_ERR_PARAM_INVALID, "n must be 4, 6 or 8 (got %lld)", (long long)c.n);
  if (c.D < 16 || c.D > 16384 || (c.D % 16) != 0)
    return fail(MHC_ERR_PARAM_INVALID, "D must be a multiple of 16 in [16, 16384] (got %lld)", (long long)c.D);
  if (c.alpha_len != 2 && c.alpha_len != 3) return fail(MHC_ERR_PARAM_INVALID, "alpha_len must be 2 or 3");
  if (c.num_iters < 1 || c.num_iters > 100) return fail(MHC_ERR_PARAM_INVALID, "num_iters must be in [1, 100]");
  if (c.impl_mode != MHC_IMPL_FP32 && c.impl_mode != MHC_IMPL_TF32)
    return fail(MHC_ERR_PARAM_INVALID, "impl_mode must be 0 (fp32) or 1 (tf32)");
  if (c.need_backward != 0 && c.need_backward != 1) return fail(MHC_ERR_PARAM_INVALID, "need_backward must be 0 or 1");
  if (c.batch_consistent != 0 && c.batch_consistent != 1)
    return fail(MHC_ERR_PARAM_INVALID, "batch_consistent must be 0 or 1");
  if (c.x_dtype != MHC_DTYPE_BF16 && c.x_dtype != MHC_DTYPE_FP16)
    return fail(MHC_ERR_PARAM_INVALID, "x_dtype must be MHC_DTYPE_BF16 or MHC_DTYPE_FP16");
  if (c.x_dtype == MHC_DTYPE_FP16 && c.n != 4)
    return fail(MHC_ERR_PARAM_INVALID, "fp16 x is supported for n = 4");
  if (!(c.norm_eps >= 0.0) || !(c.hc_eps >= 0.0)) return fail(MHC_ERR_PARAM_INVALID, "eps values must be >= 0");
  if (c.kernel != MHC_KERNEL_AUTO && c.kernel != MHC_KERNEL_CLUSTER && c.kernel != MHC_KERNEL_GRID &&
      c.kernel != MHC_KERNEL_RESIDENT)
    return fail(MHC_ERR_PARAM_INVALID, "kernel must be MHC_KERNEL_AUTO, _CLUSTER, _GRID or _RESIDENT");
  if (c.cluster != 0 && c.cluster != 1 && c.cluster != 2 && c.cluster != 4 && c.cluster != 8 && c.cluster != 16)
    return fail(MHC_ERR_PARAM_INVALID, "cluster must be 0 (automatic), 1, 2, 4, 8 or 16");
  if ((c.x_stages != 0 && (c.x_stages < 2 || c.x_stages > mhc::kMaxStages)) ||
      (c.w_stages != 0 && (c.w_stages < 2 || c.w_stages > mhc::kMaxStages)) ||
      (c.gw_x_stages != 0 && (c.gw_x_stages < 2 || c.gw_x_stages > mhc::kMaxStages)))
    return fail(MHC_ERR_PARAM_INVALID, "ring depths must be 0 (automatic) or 2..%d", mhc::kMaxStages);
  if (c.gw_groups < 0 || c.gw_groups > mhc::kGwMaxGroups)
    return fail(MHC_ERR_PARAM_INVALID, "gw_groups must be 0 (automatic), 1 or %d", mhc::kGwMaxGroups);
  if (c.gw_x_lead < 0 || c.gw_x_lead > 15) return fail(MHC_ERR_PARAM_INVALID, "gw_x_lead must be 0..15");
  if (c.tm_buffers < 0 || c.tm_buffers > 2) return fail(MHC_ERR_PARAM_INVALID, "tm_buffers must be 0, 1 or 2");
  if (c.batch_consistent && c.cluster != 0)
    return fail(MHC_ERR_PARAM_INVALID, "batch_consistent fixes the cluster size; leave cluster 0");
  mhc_pre_s* h = new (std::nothrow) mhc_pre_s;
  if (!h) return fail(MHC_ERR_RUNTIME, "out of host memory");
  h->cfg = c;
  h->R = (int)(c.alpha_len == 3 ? c.n * c.n + 2 * c.n : 2 * c.n);
  h->P = (c.impl_mode == MHC_IMPL_FP32) ? 3 : 2;
  h->NP = mhc::tc_np(h->R, h->P);
  *out = h;
  return MHC_OK;
}

mhc_status_t mhc_pre_workspace_size(mhc_pre_t h, int64_t T, size_t* bytes) {
  g_last_error[0] = 0;
  if (!h || !bytes) return fail(MHC_ERR_NULLPTR, "handle and bytes must be non-NULL");
  if (T < 0) return fail(MHC_ERR_PARAM_INVALID, "T must be >= 0");
  *bytes = (T == 0) ? 0 : mhc::kWsHeader + planes_bytes(h) + gw_rings_bytes(h);
  return MHC_OK;
}

mhc_status_t mhc_pre_run(mhc_pre_t h, const mhc_pre_args* a, void* stream) {
  g_last_error[0] = 0;
  if (!h || !a) return fail(MHC_ERR_NULLPTR, "handle and args must be non-NULL");
  h->last_noalloc_word = nullptr;
  const mhc_pre_config& c = h->cfg;
  const int64_t T = a->T;
  if (T < 0 || T > (int64_t(1) << 30)) return fail(MHC_ERR_PARAM_INVALID, "T must be in [0, 2^30]");
  if (T == 0) return MHC_OK;   // empty input: nothing to check or launch (pointers may be NULL)
  if (!a->x || (!a->phi && !a->weights) || !a->alpha || !a->bias || !a->y || !a->h_post)
    return fail(MHC_ERR_NULLPTR, "x, phi (or weights), alpha, bias, y and h_post are required");
  if (a->weights && !aligned(a->weights, 256))
    return fail(MHC_ERR_PARAM_INVALID, "weights must be 256-byte aligned");
  if (c.alpha_len == 3 && !a->h_res) return fail(MHC_ERR_NULLPTR, "h_res is required with alpha of length 3");
  if (a->pre_mix && !a->h_pre) return fail(MHC_ERR_NULLPTR, "h_pre is required when pre_mix is given");
  if (c.need_backward) {
    if (!a->h_pre || !a->inv_rms || !a->h_mix)
      return fail(MHC_ERR_NULLPTR, "need_backward: h_pre, inv_rms and h_mix are required");
    if (c.alpha_len == 3 && (!a->sum_out || !a->norm_out))
      return fail(MHC_ERR_NULLPTR, "need_backward: sum_out and norm_out are required");
    if (c.alpha_len == 2 && (a->sum_out || a->norm_out))
      return fail(MHC_ERR_PARAM_INVALID, "sum_out / norm_out do not exist without the residual path");
  } else if (a->inv_rms || a->h_mix || a->sum_out || a->norm_out) {
    return fail(MHC_ERR_PARAM_INVALID, "inv_rms, h_mix, sum_out, norm_out must be NULL unless need_backward");
  }
  if (!aligned(a->x, 16) || !aligned(a->y, 16))
    return fail(MHC_ERR_PARAM_INVALID, "x and y must be 16-byte aligned");
  const void* f32[] = {a->phi, a->alpha, a->bias, a->gamma, a->pre_mix, a->h_post, a->h_res,
                       a->h_pre, a->inv_rms, a->h_mix, a->sum_out, a->norm_out};
  for (const void* p : f32)
    if (p && !aligned(p, 4)) return fail(MHC_ERR_PARAM_INVALID, "fp32 tensors must be 4-byte aligned");
  size_t need = 0;
  mhc_pre_workspace_size(h, T, &need);
  if (!a->workspace) return fail(MHC_ERR_NULLPTR, "workspace is required (%zu bytes)", need);
  if (!aligned(a->workspace, 256)) return fail(MHC_ERR_PARAM_INVALID, "workspace must be 256-byte aligned");
  if (a->workspace_bytes < need)
    return fail(MHC_ERR_PARAM_INVALID, "workspace too small: %zu < %zu bytes", a->workspace_bytes, need);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(MHC_ERR_RUNTIME, "no CUDA device");
  const DeviceInfo di = device_info(dev);
  if (!di.ok) return fail(MHC_ERR_RUNTIME, "device %d is not an sm_103 GPU", dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  const int n = (int)c.n, D = (int)c.D, R = h->R, NP = h->NP;
  uint8_t* ws = static_cast<uint8_t*>(a->workspace);
  uint32_t* err = reinterpret_cast<uint32_t*>(ws);
  __nv_bfloat16* planes = reinterpret_cast<__nv_bfloat16*>(ws + mhc::kWsHeader);

  // 1. phi (x gamma) -> stacked bf16 precision planes; clears the error word.
  //    With prepared weights: their header (zeroed, or the fp16 range bit)
  //    becomes the workspace header and their planes are used as they are.
  if (a->weights) {
    planes = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(const_cast<void*>(a->weights)) + mhc::kWsHeader);
    const cudaError_t ce = cudaMemcpyAsync(ws, a->weights, mhc::kWsHeader, cudaMemcpyDeviceToDevice, s);
    if (ce != cudaSuccess) return fail(MHC_ERR_RUNTIME, "copying the weights header failed: %s", cudaGetErrorString(ce));
  }
  mhc::PlaneParams pp;
  pp.phi = a->phi;
  pp.gamma = a->gamma;
  pp.planes = planes;
  pp.R = R;
  pp.P = h->P;
  pp.n = n;
  pp.D = D;
  pp.nch = (D + mhc::kChunkK - 1) / mhc::kChunkK;
  pp.RB = mhc::plane_box_rows(R, h->P);
  pp.tf32 = (c.impl_mode == MHC_IMPL_TF32);
  pp.fp16 = (c.x_dtype == MHC_DTYPE_FP16);
  pp.vec16 = aligned(a->phi, 16) && (!a->gamma || aligned(a->gamma, 16));
  pp.err_word = err;
  if (!a->weights && mhc::launch_prepare_planes(pp, s) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "plane preparation launch failed: %s", cudaGetErrorString(cudaGetLastError()));

  // 2. the fused forward.  The grid-wide kernel spreads a few token tiles
  //    over every SM; up to kGwAutoMaxT tokens it runs when the cluster kernel
  //    would have a single tile or need more than one round of clusters, the
  //    cases where it is faster (D = 7168, kernel time: T = 64 22.8 against
  //    26.7 us, T = 512 36.2 against 39.9 us; but T = 256 35.0 against 26.7,
  //    and T = 768 43.3 against 40.3).  The handle's `kernel` field forces
  //    one (tests and tuning runs).  fp16 x and batch-consistent mode always
  //    run the cluster kernel.
  const bool fp16 = c.x_dtype == MHC_DTYPE_FP16;
  const bool consistent = c.batch_consistent != 0;
  const bool force_grid = c.kernel == MHC_KERNEL_GRID;
  const bool force_cluster = c.kernel == MHC_KERNEL_CLUSTER;
  constexpr int64_t kGwAutoMaxT = 512;
  const bool gw_ok = !consistent && !fp16;
  if (force_grid) {
    if (!gw_ok) return fail(MHC_ERR_PARAM_INVALID, "the grid-wide forward takes bf16 x outside batch-consistent mode");
    mhc_status_t st = run_grid_wide(h, a, di, planes, s);
    if (st != MHC_ERR_NOT_SUITABLE) return st;
    return fail(MHC_ERR_PARAM_INVALID, "the grid-wide forward does not fit this shape");
  }
  // Resident mode of the cluster kernel: the last chunks of each CTA's
  // range stay in TMEM for y, so y re-reads only the others.  Chosen
  // automatically for n = 4 from 4096 tokens (measured at D = 7168: T = 4096
  // 105 against 107 us, 8192 190 against 199, 32768 645 against 666 us, at
  // cluster 4; at D = 4096 it ties with the plain kernel at cluster 2).
  constexpr int64_t kResAutoMinT = 4096;
  const bool res_ok = !consistent && mhc::tc_resident_supported(n, R, h->P);
  const bool resident = c.kernel == MHC_KERNEL_RESIDENT || (c.kernel == MHC_KERNEL_AUTO && res_ok && T >= kResAutoMinT);
  if (resident && !res_ok)
    return fail(MHC_ERR_PARAM_INVALID, "the resident forward takes n = 4 outside batch-consistent mode");
  const int tile_t = mhc::kTileT;
  auto layout = [&](int xsn, int wsn) { return mhc::smem_layout(n, R, h->P, xsn, wsn); };
  mhc::TcLaunch L;
  memset(&L, 0, sizeof L);
  L.epi = epi_params(h, a);
  L.NP = NP;
  L.P = h->P;
  L.fp16 = fp16 ? 1 : 0;
  L.err_word = err;
  L.planes = planes;
  L.wt = h->wait_test;
  {
    // x [T][n][D] seen as (D, T, n), box (64, tile tokens, stream group); the
    // plane blocks are read with bulk copies.
    const uint64_t K2 = (uint64_t)n * D * 2;
    const uint64_t xd[3] = {(uint64_t)D, (uint64_t)T, (uint64_t)n};
    const uint64_t xs[2] = {K2, (uint64_t)D * 2};
    const uint32_t xb[3] = {(uint32_t)mhc::kChunkK, (uint32_t)tile_t, (uint32_t)mhc::stream_group(n)};
    if (!encode_3d(&L.tmap_x, a->x, xd, xs, xb))
      return fail(MHC_ERR_RUNTIME, "tensor map encoding failed");
  }

  // Ring depths: x boxes come from HBM and want bytes in flight, phi-plane
  // boxes come from L2 and want enough depth to hide its latency.  At
  // prefill three of each beat four x with two phi (0.688 vs 0.697 ms), so:
  // the deepest phi ring (up to wmax) that leaves at least three x stages,
  // then the deepest x ring; failing that, the deepest x ring first.
  const int nd = (D + mhc::kChunkK - 1) / mhc::kChunkK;
  const int num_tiles = (int)((T + tile_t - 1) / tile_t);
  const size_t budget = di.max_smem;
  int xmax = c.x_stages ? c.x_stages : 6, wmax = c.w_stages ? c.w_stages : 3;
  xmax = xmax < 2 ? 2 : (xmax > mhc::kMaxStages ? mhc::kMaxStages : xmax);
  wmax = wmax < 2 ? 2 : (wmax > mhc::kMaxStages ? mhc::kMaxStages : wmax);
  int xst = 0, wst = 0;
  for (int wsn = wmax; wsn >= 2 && !xst; --wsn)
    for (int xsn = xmax; xsn >= 3; --xsn)
      if (layout(xsn, wsn).total <= budget) {
        xst = xsn;
        wst = wsn;
        break;
      }
  for (int xsn = xmax; xsn >= 2 && !xst; --xsn)
    for (int wsn = wmax; wsn >= 2; --wsn)
      if (layout(xsn, wsn).total <= budget) {
        xst = xsn;
        wst = wsn;
        break;
      }
  if (!xst) return fail(MHC_ERR_RUNTIME, "shape does not fit in shared memory");
  const size_t smem = layout(xst, wst).total;

  // Cluster size: the one that keeps the most SMs busy on this many tiles.
  // Ties go to the larger cluster: each member then reduces and gates fewer
  // rows of a tile, which shortens the per-tile critical path.
  // The handle's `cluster` field forces a size (for tuning runs).
  // Batch-consistent mode pins cluster 2 (1 when there is a single d-chunk):
  // a token's reduction is then split the same way whatever T is.
  // Resident mode without a forced size: 4 CTAs per cluster from D = 6144
  // (144 SMs busy; the re-read chunks are read again sooner than at 2),
  // else 2.
  int res_cluster = D >= 6144 ? 4 : 2;
  while (res_cluster > nd) res_cluster >>= 1;
  const int forced = consistent ? (nd >= 2 ? 2 : 1)
                                : (c.cluster ? (int)c.cluster : (resident && c.kernel == MHC_KERNEL_AUTO ? res_cluster : 0));
  if (forced > nd) return fail(MHC_ERR_PARAM_INVALID, "cluster %d exceeds the %d d-chunks of a stream", forced, nd);
  int cluster = 0;
  int max_clusters = 0;
  long long best_sms = -1;
  for (int cand : {1, 2, 4, 8, 16}) {
    if ((forced && cand != forced) || cand > nd) continue;
    int mc = 0;
    const cudaError_t oe = mhc::tc_forward_occupancy(n, R, h->P, fp16, resident, smem, cand, &mc);
    if (oe != cudaSuccess || mc <= 0) {
      cudaGetLastError();
      continue;
    }
    const long long sms = (long long)(num_tiles < mc ? num_tiles : mc) * cand;
    if (sms >= best_sms) {
      best_sms = sms;
      cluster = cand;
      max_clusters = mc;
    }
  }
  if (max_clusters <= 0)
    return fail(forced ? MHC_ERR_PARAM_INVALID : MHC_ERR_RUNTIME, "no cluster configuration fits this device");
  if (gw_ok && !force_cluster && !resident && !c.cluster && T <= kGwAutoMaxT) {
    const int rounds = (num_tiles + max_clusters - 1) / max_clusters;
    if (num_tiles == 1 || rounds > 1) {
      mhc_status_t st = run_grid_wide(h, a, di, planes, s);
      if (st != MHC_ERR_NOT_SUITABLE) return st;
    }
  }
  // Each cluster keeps its tile slice of x (64 tokens of all n streams) in
  // flight from its first read to y's re-read, so fewer clusters in flight
  // keep more of the re-read in L2.  (1) As few clusters as take the same
  // number of rounds of tiles (T = 16384: 64 instead of 76 clusters of 2 at
  // D = 4096, 32 instead of 36 clusters of 4 at D = 7168; 1-5% faster for
  // the resident and the plain kernel, n = 4 and 8).  (2) When the slices
  // overflow L2 by a little, two fewer clusters than fit -- if that trims at
  // most a tenth of the clusters and adds at most a last round of a tenth of
  // them to ten or more full rounds: at prefill (D = 7168, T = 32768, 35 slices fit) 34 clusters of 4
  // measured 1.7% faster than 35 and 36 in both precision modes.  Not in
  // batch-consistent mode, whose launch shape stays fixed.
  if (!c.cluster && !consistent) {
    const long long tiles = num_tiles;
    const long long rounds = (tiles + max_clusters - 1) / max_clusters;
    long long cl = (tiles + rounds - 1) / rounds;
    if (di.l2_bytes > 0) {
      const double slice = (double)mhc::kTileT * n * D * 2.0;
      const long long fit = (long long)((double)di.l2_bytes / slice) - 2;
      if (fit > 0 && fit < cl && 10 * fit >= 9LL * max_clusters) {
        const long long r2 = (tiles + fit - 1) / fit;
        if (r2 == rounds || (r2 == rounds + 1 && rounds >= 10 && 10 * (tiles - rounds * fit) <= fit)) cl = fit;
      }
    }
    if (cl < max_clusters) max_clusters = (int)cl;
  }
  L.resident = resident ? 1 : 0;
  L.tm_bufs = c.tm_buffers ? c.tm_buffers : 1;
  L.cluster = cluster;
  L.grid = (num_tiles < max_clusters ? num_tiles : max_clusters) * cluster;
  L.x = a->x;
  L.xstages = xst;
  L.wstages = wst;
  L.smem_bytes = smem;
  h->last_cluster = cluster;
  h->last_grid = L.grid;
  h->last_stages = xst;
  h->last_ystages = wst;
  h->last_kernel = resident ? "mhc_pre_tc_kernel_resident" : "mhc_pre_tc_kernel";
  if (h->ev_before && cudaEventRecord(h->ev_before, s) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "recording the timing event failed");
  if (mhc::launch_tc_forward(L, s) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "forward launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  if (h->ev_after && cudaEventRecord(h->ev_after, s) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "recording the timing event failed");
  return MHC_OK;
}

mhc_status_t mhc_pre_status(mhc_pre_t h, const void* workspace, void* stream) {
  g_last_error[0] = 0;
  if (!h) return fail(MHC_ERR_NULLPTR, "handle must be non-NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(MHC_ERR_RUNTIME, "stream error: %s", cudaGetErrorString(e));
  // the error word: in the caller's workspace, or, after a no-alloc run, in
  // the library's fixed scratch array
  const void* word_at = workspace ? workspace : h->last_noalloc_word;
  if (word_at) {
    uint32_t word = 0;
    e = cudaMemcpy(&word, word_at, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(MHC_ERR_RUNTIME, "reading the error word: %s", cudaGetErrorString(e));
    if (word & mhc::kErrPlaneRange)
      return fail(MHC_ERR_RUNTIME, "phi . gamma has an entry outside the fp16 range (error word 0x%x)", word);
    if (word != 0) return fail(MHC_ERR_RUNTIME, "device-side wait gave up (error word 0x%x)", word);
  }
  return MHC_OK;
}

}  // extern "C"

// Fixed scratch for mhc_pre_run_noalloc: one array per device, reused by every
// call (the error word at its start is cleared by each run; the phi planes
// after it are rewritten by each run).
static __device__ __align__(256) unsigned char g_noalloc_scratch[MHC_PRE_STATIC_SCRATCH_BYTES];

namespace {
// Device address of g_noalloc_scratch, looked up with the device current
// (host code cannot use the symbol itself as a pointer) and cached per device
// together with the context it belongs to: a new context on that device (a
// cudaDeviceReset in between) makes the next call look it up again.
void* noalloc_scratch(int dev, cudaError_t* err) {
  static std::mutex mu;
  static void* addr[64] = {};
  static CUcontext ctx_of[64] = {};
  std::lock_guard<std::mutex> lk(mu);
  *err = cudaSuccess;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  const CtxGetCurrentFn ctx_current = ctx_get_current_fn();
  CUcontext ctx = nullptr;
  if (addr[dev] && ctx_current && ctx_current(&ctx) == CUDA_SUCCESS && ctx && ctx == ctx_of[dev]) return addr[dev];
  // first call on this device, or a different context: the lookup binds the
  // device's primary context, which is then the current one
  void* p = nullptr;
  *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (*err != cudaSuccess) return nullptr;
  ctx = nullptr;
  if (!ctx_current || ctx_current(&ctx) != CUDA_SUCCESS || !ctx) {
    *err = cudaErrorDeviceUninitialized;
    return nullptr;
  }
  addr[dev] = p;
  ctx_of[dev] = ctx;
  return p;
}
}  // namespace

extern "C" {

mhc_status_t mhc_pre_run_noalloc(mhc_pre_t h, const mhc_pre_args* a, void* stream) {
  g_last_error[0] = 0;
  if (!h || !a) return fail(MHC_ERR_NULLPTR, "handle and args must be non-NULL");
  if (a->workspace || a->workspace_bytes)
    return fail(MHC_ERR_PARAM_INVALID, "mhc_pre_run_noalloc takes no workspace (pass NULL, 0)");
  if (a->T == 0) return MHC_OK;
  size_t need = 0;
  const mhc_status_t st = mhc_pre_workspace_size(h, a->T, &need);
  if (st != MHC_OK) return st;
  if (need > MHC_PRE_STATIC_SCRATCH_BYTES)
    return fail(MHC_ERR_PARAM_INVALID,
                "this shape needs %zu bytes of scratch, over the fixed %zu-byte array of "
                "mhc_pre_run_noalloc; use mhc_pre_run with a workspace",
                need, (size_t)MHC_PRE_STATIC_SCRATCH_BYTES);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(MHC_ERR_RUNTIME, "no CUDA device");
  cudaError_t e;
  void* scratch = noalloc_scratch(dev, &e);
  if (!scratch) return fail(MHC_ERR_RUNTIME, "looking up the scratch array failed: %s", cudaGetErrorString(e));
  mhc_pre_args b = *a;
  b.workspace = scratch;
  b.workspace_bytes = MHC_PRE_STATIC_SCRATCH_BYTES;
  const mhc_status_t rs = mhc_pre_run(h, &b, stream);
  if (rs == MHC_OK) h->last_noalloc_word = scratch;   // mhc_pre_status(h, NULL, s) reads it there
  return rs;
}

mhc_status_t mhc_pre_weights_size(mhc_pre_t h, size_t* bytes) {
  g_last_error[0] = 0;
  if (!h || !bytes) return fail(MHC_ERR_NULLPTR, "handle and bytes must be non-NULL");
  *bytes = mhc::kWsHeader + planes_bytes(h);
  return MHC_OK;
}

mhc_status_t mhc_pre_prepare_weights(mhc_pre_t h, const float* phi, const float* gamma, void* weights,
                                     size_t weights_bytes, void* stream) {
  g_last_error[0] = 0;
  if (!h || !phi || !weights) return fail(MHC_ERR_NULLPTR, "handle, phi and weights must be non-NULL");
  if (!aligned(weights, 256)) return fail(MHC_ERR_PARAM_INVALID, "weights must be 256-byte aligned");
  if (!aligned(phi, 4) || (gamma && !aligned(gamma, 4)))
    return fail(MHC_ERR_PARAM_INVALID, "phi and gamma must be 4-byte aligned");
  size_t need = 0;
  mhc_pre_weights_size(h, &need);
  if (weights_bytes < need)
    return fail(MHC_ERR_PARAM_INVALID, "weights buffer too small: %zu < %zu bytes", weights_bytes, need);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(MHC_ERR_RUNTIME, "no CUDA device");
  if (!device_info(dev).ok) return fail(MHC_ERR_RUNTIME, "device %d is not an sm_103 GPU", dev);
  const mhc_pre_config& c = h->cfg;
  uint8_t* wb = static_cast<uint8_t*>(weights);
  mhc::PlaneParams pp;
  pp.phi = phi;
  pp.gamma = gamma;
  pp.planes = reinterpret_cast<__nv_bfloat16*>(wb + mhc::kWsHeader);
  pp.R = h->R;
  pp.P = h->P;
  pp.n = (int)c.n;
  pp.D = (int)c.D;
  pp.nch = (int)((c.D + mhc::kChunkK - 1) / mhc::kChunkK);
  pp.RB = mhc::plane_box_rows(h->R, h->P);
  pp.tf32 = (c.impl_mode == MHC_IMPL_TF32);
  pp.fp16 = (c.x_dtype == MHC_DTYPE_FP16);
  pp.vec16 = aligned(phi, 16) && (!gamma || aligned(gamma, 16));
  pp.err_word = reinterpret_cast<uint32_t*>(wb);   // the header: zeroed, or the fp16 range bit
  if (mhc::launch_prepare_planes(pp, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "plane preparation launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  return MHC_OK;
}

mhc_status_t mhc_pre_set_wait_test(mhc_pre_t h, uint32_t wait_limit_us, int32_t withhold_last_x_copy) {
  g_last_error[0] = 0;
  if (!h) return fail(MHC_ERR_NULLPTR, "handle must be non-NULL");
  if (withhold_last_x_copy != 0 && withhold_last_x_copy != 1)
    return fail(MHC_ERR_PARAM_INVALID, "withhold_last_x_copy must be 0 or 1");
  if (wait_limit_us > 10000000u) return fail(MHC_ERR_PARAM_INVALID, "wait_limit_us must be at most 10 s");
  h->wait_test.wait_ns = wait_limit_us ? (uint64_t)wait_limit_us * 1000ull : 2000000000ull;
  h->wait_test.withhold_x = withhold_last_x_copy;
  return MHC_OK;
}

mhc_status_t mhc_pre_set_profile_events(mhc_pre_t h, void* before, void* after) {
  g_last_error[0] = 0;
  if (!h) return fail(MHC_ERR_NULLPTR, "handle must be non-NULL");
  h->ev_before = static_cast<cudaEvent_t>(before);
  h->ev_after = static_cast<cudaEvent_t>(after);
  return MHC_OK;
}

mhc_status_t mhc_pre_last_launch(mhc_pre_t h, int32_t* cluster, int32_t* grid, int32_t* stages,
                                 int32_t* ystages) {
  g_last_error[0] = 0;
  if (!h) return fail(MHC_ERR_NULLPTR, "handle must be non-NULL");
  if (cluster) *cluster = h->last_cluster;
  if (grid) *grid = h->last_grid;
  if (stages) *stages = h->last_stages;
  if (ystages) *ystages = h->last_ystages;
  return MHC_OK;
}

const char* mhc_pre_last_kernel(mhc_pre_t h) { return h ? h->last_kernel : ""; }

mhc_status_t mhc_post_run(int64_t T, int64_t n, int64_t D, const void* x, const void* residual, const float* post,
                          const float* comb, void* out, void* stream) {
  g_last_error[0] = 0;
  if (T < 0 || T > (int64_t(1) << 30)) return fail(MHC_ERR_PARAM_INVALID, "T must be in [0, 2^30]");
  if (n < 1 || n > 8) return fail(MHC_ERR_PARAM_INVALID, "n must be in [1, 8] (got %lld)", (long long)n);
  if (D < 8 || D > (int64_t(1) << 20) || (D % 8) != 0)
    return fail(MHC_ERR_PARAM_INVALID, "D must be a positive multiple of 8 (got %lld)", (long long)D);
  if (T == 0) return MHC_OK;
  if (!x || !residual || !post || !comb || !out) return fail(MHC_ERR_NULLPTR, "x, residual, post, comb, out are required");
  if (!aligned(x, 16) || !aligned(residual, 16) || !aligned(out, 16))
    return fail(MHC_ERR_PARAM_INVALID, "x, residual and out must be 16-byte aligned");
  if (!aligned(post, 4) || !aligned(comb, 4)) return fail(MHC_ERR_PARAM_INVALID, "post and comb must be 4-byte aligned");
  mhc::PostLaunch L;
  L.T = T;
  L.n = n;
  L.D = D;
  L.x = x;
  L.residual = residual;
  L.post = post;
  L.comb = comb;
  L.out = out;
  if (mhc::launch_post(L, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "post-mapping launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  return MHC_OK;
}

void mhc_pre_destroy(mhc_pre_t h) { delete h; }

}  // extern "C"

// ---------------------------------------------------------------- backward
namespace {

// Backward workspace: [0, 256) header | phi . gamma planes per slab | tile
// records (G planes + hPre + RMS factor) | x^T G partial sums of the work
// units (slab, token chunk) | token-stage partial sums | H_pre_grad [T][n].
struct BwLayout {
  size_t planes, tiles, pieces, partials, hg, total;
};

BwLayout bw_layout(const mhc_pre_s* h, int64_t T) {
  const int P = h->P;
  const size_t nslab = (size_t)(h->cfg.D / 64);
  const size_t ntiles = (size_t)((T + mhc::kBwTile - 1) / mhc::kBwTile);
  auto up = [](size_t v) { return (v + 255) & ~size_t(255); };
  BwLayout L;
  L.planes = mhc::kWsHeader;
  L.tiles = L.planes + up(nslab * (size_t)mhc::bw_slab_bytes(P));
  L.pieces = L.tiles + up(ntiles * (size_t)mhc::bw_tile_rec_bytes(P));
  L.partials = L.pieces + up(nslab * mhc::kBwMaxChunks * mhc::bw_piece_bytes());
  L.hg = L.partials + up((size_t)mhc::kBwMaxTokenBlocks * mhc::kBwTokenWarps * 32 * sizeof(float));
  L.total = L.hg + up((size_t)T * mhc::kBwNS * sizeof(float));
  return L;
}

mhc_status_t bw_scope(const mhc_pre_s* h) {
  if (h->cfg.alpha_len != 3) return fail(MHC_ERR_PARAM_INVALID, "the backward needs a three-gate handle (alpha_len 3)");
  if (h->cfg.n != 4) return fail(MHC_ERR_PARAM_INVALID, "the backward supports n = 4 (got %lld)", (long long)h->cfg.n);
  if (h->cfg.D % 64 != 0)
    return fail(MHC_ERR_PARAM_INVALID, "the backward needs D a multiple of 64 (got %lld)", (long long)h->cfg.D);
  if (h->cfg.x_dtype != MHC_DTYPE_BF16) return fail(MHC_ERR_PARAM_INVALID, "the backward takes bf16 x");
  return MHC_OK;
}

}  // namespace

extern "C" {

mhc_status_t mhc_pre_backward_workspace_size(mhc_pre_t h, int64_t T, size_t* bytes) {
  g_last_error[0] = 0;
  if (!h || !bytes) return fail(MHC_ERR_NULLPTR, "handle and bytes must be non-NULL");
  if (T < 0 || T > (int64_t(1) << 30)) return fail(MHC_ERR_PARAM_INVALID, "T must be in [0, 2^30]");
  const mhc_status_t sc = bw_scope(h);
  if (sc != MHC_OK) return sc;
  *bytes = (T == 0) ? 0 : bw_layout(h, T).total;
  return MHC_OK;
}

mhc_status_t mhc_pre_backward_run(mhc_pre_t h, const mhc_pre_bwd_args* a, void* stream) {
  g_last_error[0] = 0;
  if (!h || !a) return fail(MHC_ERR_NULLPTR, "handle and args must be non-NULL");
  const mhc_status_t sc = bw_scope(h);
  if (sc != MHC_OK) return sc;
  const int64_t T = a->T;
  if (T < 0 || T > (int64_t(1) << 30)) return fail(MHC_ERR_PARAM_INVALID, "T must be in [0, 2^30]");
  if (T == 0) return MHC_OK;
  if (!a->x || !a->phi || !a->alpha || !a->grad_h_in || !a->grad_h_post || !a->grad_h_res || !a->inv_rms ||
      !a->h_mix || !a->h_pre || !a->h_post || !a->grad_x || !a->grad_phi || !a->grad_alpha || !a->grad_bias ||
      !a->workspace)
    return fail(MHC_ERR_NULLPTR, "a required tensor or the workspace is NULL");
  if ((a->sum_out == nullptr) != (a->norm_out == nullptr))
    return fail(MHC_ERR_PARAM_INVALID, "sum_out and norm_out go together (both or neither)");
  if ((a->gamma == nullptr) != (a->grad_gamma == nullptr))
    return fail(MHC_ERR_PARAM_INVALID, "grad_gamma is required exactly when gamma is given");
  const void* v16[] = {a->x, a->grad_h_in, a->grad_x, a->grad_x_post, a->workspace};
  for (const void* p : v16)
    if (p && !aligned(p, 16)) return fail(MHC_ERR_PARAM_INVALID, "bf16 tensors and the workspace must be 16-byte aligned");
  const void* v4[] = {a->phi, a->alpha, a->gamma, a->grad_h_post, a->grad_h_res, a->inv_rms, a->h_mix, a->h_pre,
                      a->h_post, a->sum_out, a->norm_out, a->grad_phi, a->grad_alpha, a->grad_bias, a->grad_gamma};
  for (const void* p : v4)
    if (p && !aligned(p, 4)) return fail(MHC_ERR_PARAM_INVALID, "fp32 tensors must be 4-byte aligned");
  const BwLayout L = bw_layout(h, T);
  if (a->workspace_bytes < L.total)
    return fail(MHC_ERR_PARAM_INVALID, "workspace too small: %zu bytes given, %zu needed", a->workspace_bytes, L.total);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(MHC_ERR_RUNTIME, "no CUDA device");
  const DeviceInfo di = device_info(dev);
  if (!di.ok) return fail(MHC_ERR_RUNTIME, "device %d is not an sm_103 GPU", dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int n = (int)h->cfg.n, D = (int)h->cfg.D, P = h->P;
  const int nslab = D / 64;
  const int ntiles = (int)((T + mhc::kBwTile - 1) / mhc::kBwTile);
  uint8_t* ws = static_cast<uint8_t*>(a->workspace);
  uint32_t* err = reinterpret_cast<uint32_t*>(ws);
  __nv_bfloat16* planes = reinterpret_cast<__nv_bfloat16*>(ws + L.planes);
  uint8_t* tiles = ws + L.tiles;
  float* pieces = reinterpret_cast<float*>(ws + L.pieces);
  float* partials = reinterpret_cast<float*>(ws + L.partials);

  // main-kernel geometry
  const bool gxp = a->grad_x_post != nullptr;
  const size_t fixed = (size_t)mhc::bw_slab_bytes(P) + mhc::kBwTailBytes + 1024;
  const size_t stage = (size_t)mhc::bw_stage_bytes(P, gxp);
  int stages = (int)((di.max_smem - fixed) / stage);
  if (stages > 4) stages = 4;
  if (stages < 2) return fail(MHC_ERR_RUNTIME, "not enough shared memory for the backward pipeline");
  // Token chunks per slab: the count (at most kBwMaxChunks and the tile
  // count) whose units fill whole waves of the grid best; ties go to fewer
  // chunks (fewer partial sums).
  long long grid = di.sms < mhc::kBwMaxMainGrid ? di.sms : mhc::kBwMaxMainGrid;
  int nq = 1;
  double best = -1.0;
  for (int q = 1; q <= mhc::kBwMaxChunks && q <= ntiles; ++q) {
    const long long units = (long long)nslab * q;
    const long long waves = (units + grid - 1) / grid;
    const double eff = (double)units / (double)(waves * grid);
    if (eff > best + 1e-9) {
      best = eff;
      nq = q;
    }
  }
  if (grid > (long long)nslab * nq) grid = (long long)nslab * nq;

  mhc::BwMainLaunch M;
  {
    const uint64_t dims[4] = {64, (uint64_t)T, (uint64_t)nslab, (uint64_t)n};
    const uint64_t strides[3] = {(uint64_t)n * D * 2, 128, (uint64_t)D * 2};
    const uint32_t box[4] = {64, (uint32_t)mhc::kBwTile, 1, (uint32_t)n};
    if (!encode_4d(&M.tmap_x, a->x, dims, strides, box) ||
        !encode_4d(&M.tmap_gxp, gxp ? a->grad_x_post : a->x, dims, strides, box))
      return fail(MHC_ERR_RUNTIME, "encoding the x / grad_x_post tensor maps failed");
    const uint64_t gd[3] = {64, (uint64_t)T, (uint64_t)nslab};
    const uint64_t gs[2] = {(uint64_t)D * 2, 128};
    const uint32_t gb[3] = {64, (uint32_t)mhc::kBwTile, 1};
    if (!encode_3d(&M.tmap_gin, a->grad_h_in, gd, gs, gb))
      return fail(MHC_ERR_RUNTIME, "encoding the grad_h_in tensor map failed");
  }
  M.planes = planes;
  M.grad_x = static_cast<__nv_bfloat16*>(a->grad_x);
  M.tiles = tiles;
  M.pieces = pieces;
  M.err = err;
  M.T = (int)T;
  M.D = D;
  M.ntiles = ntiles;
  M.nslab = nslab;
  M.P = P;
  M.stages = stages;
  M.has_gxp = gxp ? 1 : 0;
  M.grid = (int)grid;
  M.nq = nq;
  M.smem_bytes = fixed + (size_t)stages * stage;
  M.wt = h->wait_test;

  mhc::BwPlaneParams pp;
  pp.phi = a->phi;
  pp.gamma = a->gamma;
  pp.planes = planes;
  pp.hdr = err;
  pp.D = D;
  pp.nslab = nslab;
  pp.P = P;
  pp.tf32 = (h->cfg.impl_mode == MHC_IMPL_TF32) ? 1 : 0;
  pp.vec16 = aligned(a->phi, 16) && (!a->gamma || aligned(a->gamma, 16));

  mhc::BwRowdotParams rp;
  rp.T = (int)T;
  rp.D = D;
  rp.x = static_cast<const __nv_bfloat16*>(a->x);
  rp.g_in = static_cast<const __nv_bfloat16*>(a->grad_h_in);
  rp.hg = reinterpret_cast<float*>(ws + L.hg);
  rp.err = err;
  size_t rd_smem = 0;
  mhc::bw_rowdot_shape(D, di.max_smem, &rp.tps, &rp.stages, &rd_smem);
  if (rp.stages < 1) return fail(MHC_ERR_RUNTIME, "not enough shared memory for the row-dot ring");
  const long long rd_groups = (T + rp.tps - 1) / rp.tps;
  const int rd_grid = (int)(rd_groups < di.sms ? rd_groups : di.sms);

  mhc::BwTokenParams tp;
  tp.hg = rp.hg;
  tp.T = (int)T;
  tp.D = D;
  tp.ntiles = ntiles;
  tp.num_iters = (int)h->cfg.num_iters;
  tp.P = P;
  tp.tf32 = pp.tf32;
  tp.hc_eps = (float)h->cfg.hc_eps;
  tp.g_post = a->grad_h_post;
  tp.g_res = a->grad_h_res;
  tp.inv_rms = a->inv_rms;
  tp.h_mix = a->h_mix;
  tp.h_pre = a->h_pre;
  tp.h_post = a->h_post;
  tp.sum_out = a->sum_out;
  tp.norm_out = a->norm_out;
  tp.saved16 = aligned(a->sum_out, 16) && aligned(a->norm_out, 16) ? 1 : 0;
  tp.alpha = a->alpha;
  tp.tiles = tiles;
  tp.partials = partials;
  int tblocks = 0;
  if (mhc::bw_token_blocks(&tblocks) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "token-stage occupancy query failed: %s", cudaGetErrorString(cudaGetLastError()));
  // two tokens per warp
  const long long tmax = ((long long)ntiles * mhc::kBwTile + 2 * mhc::kBwTokenWarps - 1) / (2 * mhc::kBwTokenWarps);
  if (tblocks > tmax) tblocks = (int)tmax;

  mhc::BwFinalParams fp;
  fp.D = D;
  fp.nslab = nslab;
  fp.nq = nq;
  fp.pieces = pieces;
  fp.phi = a->phi;
  fp.gamma = a->gamma;
  fp.grad_phi = a->grad_phi;
  fp.grad_gamma = a->grad_gamma;
  fp.partials = partials;
  fp.nparts = tblocks * mhc::kBwTokenWarps;
  fp.grad_alpha = a->grad_alpha;
  fp.grad_bias = a->grad_bias;

  cudaError_t e;
  if ((e = mhc::launch_bw_planes(pp, s)) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "backward plane launch failed: %s", cudaGetErrorString(e));
  if ((e = mhc::launch_bw_rowdot(rp, rd_grid, rd_smem, s)) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "backward row-dot launch failed: %s", cudaGetErrorString(e));
  if ((e = mhc::launch_bw_token(tp, tblocks, s)) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "backward token-stage launch failed: %s", cudaGetErrorString(e));
  if (h->ev_before) cudaEventRecord(h->ev_before, s);
  if ((e = mhc::launch_bw_main(M, s)) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "backward main launch failed: %s", cudaGetErrorString(e));
  if (h->ev_after) cudaEventRecord(h->ev_after, s);
  if ((e = mhc::launch_bw_final(fp, s)) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "backward final launch failed: %s", cudaGetErrorString(e));
  h->last_cluster = 1;
  h->last_grid = (int)grid;
  h->last_stages = stages;
  h->last_ystages = tblocks;
  h->last_kernel = "bw_main_kernel";
  return MHC_OK;
}

}  // extern "C"

// ---------------------------------------------------------- composite route
namespace {

mhc_status_t stage_device(cudaStream_t* s, void* stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(MHC_ERR_RUNTIME, "no CUDA device");
  if (!device_info(dev).ok) return fail(MHC_ERR_RUNTIME, "device %d is not an sm_103 GPU", dev);
  *s = static_cast<cudaStream_t>(stream);
  return MHC_OK;
}

mhc::StageLaunch stage_launch(const mhc_pre_s* h, int64_t T, const void* x) {
  mhc::StageLaunch L;
  memset(&L, 0, sizeof L);
  L.T = (int)T;
  L.n = (int)h->cfg.n;
  L.D = (int)h->cfg.D;
  L.R = h->R;
  L.fp16 = h->cfg.x_dtype == MHC_DTYPE_FP16 ? 1 : 0;
  L.norm_eps = (float)h->cfg.norm_eps;
  L.x = x;
  return L;
}

}  // namespace

extern "C" {

mhc_status_t mhc_pre_inv_rms_run(mhc_pre_t h, int64_t T, const void* x, float* inv_rms, void* stream) {
  g_last_error[0] = 0;
  if (!h) return fail(MHC_ERR_NULLPTR, "handle must be non-NULL");
  if (T < 0 || T > (int64_t(1) << 30)) return fail(MHC_ERR_PARAM_INVALID, "T must be in [0, 2^30]");
  if (T == 0) return MHC_OK;
  if (!x || !inv_rms) return fail(MHC_ERR_NULLPTR, "x and inv_rms are required");
  if (!aligned(x, 16) || !aligned(inv_rms, 4)) return fail(MHC_ERR_PARAM_INVALID, "x must be 16-byte aligned");
  cudaStream_t s = nullptr;
  const mhc_status_t st = stage_device(&s, stream);
  if (st != MHC_OK) return st;
  mhc::StageLaunch L = stage_launch(h, T, x);
  L.inv_rms = inv_rms;
  if (mhc::launch_stage_inv_rms(L, s) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "inv_rms launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  return MHC_OK;
}

mhc_status_t mhc_pre_mixes_run(mhc_pre_t h, int64_t T, const void* x, const float* phi, const float* gamma,
                               float* mixes, void* stream) {
  g_last_error[0] = 0;
  if (!h) return fail(MHC_ERR_NULLPTR, "handle must be non-NULL");
  if (T < 0 || T > (int64_t(1) << 30)) return fail(MHC_ERR_PARAM_INVALID, "T must be in [0, 2^30]");
  if (T == 0) return MHC_OK;
  if (!x || !phi || !mixes) return fail(MHC_ERR_NULLPTR, "x, phi and mixes are required");
  if (!aligned(x, 16)) return fail(MHC_ERR_PARAM_INVALID, "x must be 16-byte aligned");
  if (!aligned(phi, 4) || !aligned(mixes, 4) || (gamma && !aligned(gamma, 4)))
    return fail(MHC_ERR_PARAM_INVALID, "fp32 tensors must be 4-byte aligned");
  cudaStream_t s = nullptr;
  const mhc_status_t st = stage_device(&s, stream);
  if (st != MHC_OK) return st;
  mhc::StageLaunch L = stage_launch(h, T, x);
  L.phi = phi;
  L.gamma = gamma;
  L.mixes = mixes;
  if (mhc::launch_stage_mixes(L, s) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "mixes launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  return MHC_OK;
}

mhc_status_t mhc_pre_sinkhorn_run(mhc_pre_t h, const mhc_pre_args* a, const float* mixes, const float* inv_rms,
                                  void* stream) {
  g_last_error[0] = 0;
  if (!h || !a) return fail(MHC_ERR_NULLPTR, "handle and args must be non-NULL");
  const mhc_pre_config& c = h->cfg;
  const int64_t T = a->T;
  if (T < 0 || T > (int64_t(1) << 30)) return fail(MHC_ERR_PARAM_INVALID, "T must be in [0, 2^30]");
  if (T == 0) return MHC_OK;
  if (!a->x || !a->alpha || !a->bias || !a->y || !a->h_post || !mixes || !inv_rms)
    return fail(MHC_ERR_NULLPTR, "x, alpha, bias, y, h_post, mixes and inv_rms are required");
  if (c.alpha_len == 3 && !a->h_res) return fail(MHC_ERR_NULLPTR, "h_res is required with alpha of length 3");
  if (a->pre_mix && !a->h_pre) return fail(MHC_ERR_NULLPTR, "h_pre is required when pre_mix is given");
  if (c.need_backward) {
    if (!a->h_pre || !a->inv_rms || !a->h_mix)
      return fail(MHC_ERR_NULLPTR, "need_backward: h_pre, inv_rms and h_mix are required");
    if (c.alpha_len == 3 && (!a->sum_out || !a->norm_out))
      return fail(MHC_ERR_NULLPTR, "need_backward: sum_out and norm_out are required");
    if (c.alpha_len == 2 && (a->sum_out || a->norm_out))
      return fail(MHC_ERR_PARAM_INVALID, "sum_out / norm_out do not exist without the residual path");
  } else if (a->inv_rms || a->h_mix || a->sum_out || a->norm_out) {
    return fail(MHC_ERR_PARAM_INVALID, "inv_rms, h_mix, sum_out, norm_out must be NULL unless need_backward");
  }
  if (!aligned(a->x, 16) || !aligned(a->y, 16)) return fail(MHC_ERR_PARAM_INVALID, "x and y must be 16-byte aligned");
  const void* f32[] = {a->alpha, a->bias, a->pre_mix, a->h_post, a->h_res, a->h_pre, a->inv_rms,
                       a->h_mix, a->sum_out, a->norm_out, mixes, inv_rms};
  for (const void* p : f32)
    if (p && !aligned(p, 4)) return fail(MHC_ERR_PARAM_INVALID, "fp32 tensors must be 4-byte aligned");
  cudaStream_t s = nullptr;
  const mhc_status_t st = stage_device(&s, stream);
  if (st != MHC_OK) return st;
  const mhc::EpiParams ep = epi_params(h, a);
  if (mhc::launch_stage_sinkhorn(ep, a->x, mixes, inv_rms, c.x_dtype == MHC_DTYPE_FP16 ? 1 : 0, s) != cudaSuccess)
    return fail(MHC_ERR_RUNTIME, "sinkhorn-stage launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  return MHC_OK;
}

}  // extern "C"
