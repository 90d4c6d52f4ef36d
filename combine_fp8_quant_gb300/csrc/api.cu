// api.cu -- the C ABI of libmoeperm (include/moeperm.h): host-side argument
// validation, workspace carving and kernel launches. No allocation, no
// synchronisation (except moe_status_sync), no host <-> device traffic.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/moeperm.h"
#include "common.cuh"
#include "kernels.h"

// Host-side caches of launch queries. An occupancy query or a device
// attribute read costs the host about as much as a launch, and a
// shared-memory opt-in more; each is asked once per key. Occupancy and device
// attributes are properties of the device; the shared-memory opt-in is a
// function attribute of the CUDA context, so it is cached per context (a
// context created again after cudaDeviceReset has a new id and opts in
// afresh). The tables are small and fixed: once one is full, new keys are
// simply asked every time.
namespace moeperm {
namespace {
std::mutex g_cache_mu;
struct OccEntry { const void* kernel; int threads; size_t smem; int dev; int value; };
OccEntry g_occ[256];
int g_nocc = 0;
struct SmemEntry { const void* kernel; unsigned long long ctx; size_t dyn; };
SmemEntry g_smem[128];
int g_nsmem = 0;
struct AttrEntry { int attr; int dev; int value; };
AttrEntry g_attr[64];
int g_nattr = 0;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
std::once_flag g_ctx_once;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// Driver entry points for the current context and its id, looked up once
// through the runtime (the library does not link the driver library).
void find_context_entry_points() {
  void* f1 = nullptr;
  void* f2 = nullptr;
  cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound;
  cudaDriverEntryPointQueryResult q2 = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) !=
          cudaSuccess ||
      cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) !=
          cudaSuccess ||
      q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess) {
    (void)cudaGetLastError();
    return;
  }
  g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
  g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f2);
}
}  // namespace

cudaError_t current_context_id(unsigned long long* id) {
  *id = 0;
  std::call_once(g_ctx_once, find_context_entry_points);
  if (g_ctx_get_current == nullptr || g_ctx_get_id == nullptr) return cudaErrorSymbolNotFound;
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return cudaErrorUnknown;
  if (ctx == nullptr) return cudaSuccess;
  return g_ctx_get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

cudaError_t occupancy_cached(const void* kernel, int threads, size_t smem, int* per_sm) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  {
    std::lock_guard<std::mutex> g(g_cache_mu);
    for (int i = 0; i < g_nocc; ++i) {
      const OccEntry& e = g_occ[i];
      if (e.kernel == kernel && e.threads == threads && e.smem == smem && e.dev == dev) {
        *per_sm = e.value;
        return cudaSuccess;
      }
    }
  }
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, kernel, threads, smem);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> g(g_cache_mu);
  if (g_nocc < 256) g_occ[g_nocc++] = OccEntry{kernel, threads, smem, dev, *per_sm};
  return cudaSuccess;
}

cudaError_t opt_in_smem_cached(const void* kernel, size_t dyn) {
  unsigned long long ctx = 0;
  // no context id (none current yet, or no driver entry point): set the
  // attribute every time rather than trust a cache entry
  const bool cacheable = current_context_id(&ctx) == cudaSuccess && ctx != 0;
  if (cacheable) {
    std::lock_guard<std::mutex> g(g_cache_mu);
    for (int i = 0; i < g_nsmem; ++i)
      if (g_smem[i].kernel == kernel && g_smem[i].ctx == ctx && g_smem[i].dyn >= dyn) return cudaSuccess;
  }
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (err != cudaSuccess) return err;
  if (!cacheable) return cudaSuccess;
  err = current_context_id(&ctx);  // the call above may have created the context
  if (err != cudaSuccess || ctx == 0) return cudaSuccess;
  std::lock_guard<std::mutex> g(g_cache_mu);
  for (int i = 0; i < g_nsmem; ++i)
    if (g_smem[i].kernel == kernel && g_smem[i].ctx == ctx) {
      if (g_smem[i].dyn < dyn) g_smem[i].dyn = dyn;
      return cudaSuccess;
    }
  if (g_nsmem < 128) g_smem[g_nsmem++] = SmemEntry{kernel, ctx, dyn};
  return cudaSuccess;
}

cudaError_t device_attr_cached(cudaDeviceAttr attr, int* value) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  {
    std::lock_guard<std::mutex> g(g_cache_mu);
    for (int i = 0; i < g_nattr; ++i)
      if (g_attr[i].attr == (int)attr && g_attr[i].dev == dev) {
        *value = g_attr[i].value;
        return cudaSuccess;
      }
  }
  err = cudaDeviceGetAttribute(value, attr, dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> g(g_cache_mu);
  if (g_nattr < 64) g_attr[g_nattr++] = AttrEntry{(int)attr, dev, *value};
  return cudaSuccess;
}

}  // namespace moeperm

using namespace moeperm;

namespace {

constexpr int kMaxK = 32;
constexpr int kMaxL = 1024;
constexpr int64_t kMaxAssignments = int64_t(1) << 20;
constexpr int kMaxHidden = 32768;   // one pass of 2 chunks x 1024 threads per row
constexpr size_t kWsHeader = 256;  // reserved header before the chunk table

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int num_sms_cached() {
  int n = 0;
  return device_attr_cached(cudaDevAttrMultiProcessorCount, &n) == cudaSuccess ? n : 0;
}

bool fmt_ok(int fmt, int g) {
  if (g == 128) return fmt == MOE_SCALE_UE8M0_U8 || fmt == MOE_SCALE_UE8M0_PACKED ||
                       fmt == MOE_SCALE_F32_POW2 || fmt == MOE_SCALE_F32;
  if (g == 32) return fmt == MOE_SCALE_UE8M0_U8 || fmt == MOE_SCALE_MX_E8M0;
  return false;
}

// Leading-dimension rule of a scale buffer whose blocks hold `rows_per_block` rows.
bool ld_ok(int fmt, int64_t ld, int64_t rows_per_block, int G) {
  if (fmt == MOE_SCALE_UE8M0_PACKED) return ld >= rows_per_block && ld % 4 == 0 && ld > 0;
  return ld >= G;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

struct DispatchCommon {
  const void* x; int64_t ldx; int32_t T; const int32_t* d_num_tokens; int32_t H;
  const int32_t* ids; const float* w; int32_t K, E, L, g; int fmt;
  void* xq; void* scales; int64_t ld_s; int32_t* src2dst; float* row_weights;
  void* ws; size_t ws_bytes;
};

moe_status_t check_common(const DispatchCommon& c) {
  if (c.T < 0 || c.H <= 0 || c.H % 16 || (c.g != 32 && c.g != 128) || c.H % c.g) return MOE_ERR_INVALID_ARG;
  if (!fmt_ok(c.fmt, c.g)) return MOE_ERR_INVALID_ARG;
  if (c.K < 1 || c.K > kMaxK || c.L < 1 || c.L > kMaxL || c.E < c.L) return MOE_ERR_INVALID_ARG;
  if ((int64_t)c.T * c.K > kMaxAssignments || c.H > kMaxHidden) return MOE_ERR_INVALID_ARG;
  if (route_geometry((int64_t)c.T * c.K, c.L, route_table_pref(c.H, c.L)).S == 0) return MOE_ERR_INVALID_ARG;
  if (c.T > 0) {
    if (!c.x || !aligned16(c.x) || c.ldx < c.H || c.ldx % 8) return MOE_ERR_INVALID_ARG;
    if (!c.ids || !c.src2dst) return MOE_ERR_INVALID_ARG;
  }
  if (c.row_weights && !c.w) return MOE_ERR_INVALID_ARG;
  if (!c.ws || !aligned16(c.ws) || c.ws_bytes < moe_workspace_bytes(c.T, c.K, c.L))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status_t run_dispatch(const DispatchCommon& c, int mode, int32_t block_e, int32_t cap,
                          int32_t* m_indices, int64_t bound, int32_t* counts, int32_t* starts,
                          int32_t* psum, int32_t* total, int32_t* masked_m, int32_t* d_status,
                          cudaStream_t stream) {
  const int sms = num_sms_cached();
  if (sms <= 0) return MOE_ERR_CUDA;
  const int64_t A = (int64_t)c.T * c.K;
  if (A <= kSmallSlots) {  // latency-bound: one launch, no workspace traffic
    ScatterArgs sa{};
    sa.x = static_cast<const uint16_t*>(c.x); sa.ldx = c.ldx; sa.T = c.T;
    sa.d_num_tokens = c.d_num_tokens; sa.H = c.H; sa.ids = c.ids; sa.w = c.w;
    sa.K = c.K; sa.L = c.L; sa.E = c.E; sa.mode = mode; sa.block_e = block_e; sa.cap = cap;
    sa.xq = static_cast<uint8_t*>(c.xq); sa.scales = c.scales; sa.ld_s = c.ld_s;
    sa.src2dst = c.src2dst; sa.row_weights = c.row_weights;
    sa.m_indices = m_indices; sa.bound = bound;
    sa.counts = counts; sa.starts = starts; sa.psum = psum; sa.total = total;
    sa.masked_m = masked_m; sa.status = d_status;
    return cuda_status(launch_dispatch_small(sa, c.g, c.fmt, sms, stream));
  }
  const RouteGeom geom = route_geometry(A, c.L, route_table_pref(c.H, c.L));
  int32_t* table = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(c.ws) + kWsHeader);

  RoutePlanArgs rp{};
  rp.ids = c.ids; rp.d_num_tokens = c.d_num_tokens;
  rp.T = c.T; rp.K = c.K; rp.L = c.L;
  rp.chunk = geom.chunk; rp.nchunks = (int32_t)geom.nchunks;
  rp.lrank = c.src2dst; rp.table = table; rp.status = d_status;
  rp.queue = reinterpret_cast<int32_t*>(c.ws);  // first word of the reserved header
  if (launch_route_plan(rp, geom, stream) != cudaSuccess) return MOE_ERR_CUDA;

  ScatterArgs sa{};
  sa.x = static_cast<const uint16_t*>(c.x); sa.ldx = c.ldx; sa.T = c.T;
  sa.d_num_tokens = c.d_num_tokens; sa.H = c.H; sa.ids = c.ids; sa.w = c.w;
  sa.K = c.K; sa.L = c.L; sa.E = c.E; sa.mode = mode; sa.block_e = block_e; sa.cap = cap;
  sa.chunk = rp.chunk; sa.nchunks = rp.nchunks; sa.table = table; sa.queue = rp.queue;
  sa.xq = static_cast<uint8_t*>(c.xq); sa.scales = c.scales; sa.ld_s = c.ld_s;
  sa.src2dst = c.src2dst; sa.row_weights = c.row_weights;
  sa.m_indices = m_indices; sa.bound = bound;
  sa.counts = counts; sa.starts = starts; sa.psum = psum; sa.total = total;
  sa.masked_m = masked_m; sa.status = d_status;
  return cuda_status(launch_quant_scatter(sa, c.g, c.fmt, sms, /*after_route_plan=*/true, stream));
}

}  // namespace

extern "C" {

int64_t moe_compact_bound(int64_t A, int32_t L, int32_t block_e) {
  if (A < 0 || L < 1 || block_e < 1) return 0;
  const int64_t n = A < L ? A : L;
  return (int64_t)block_e * (n + (A - n) / block_e);
}

int32_t moe_should_use_masked(int32_t E, int32_t L) { return (E > L && L <= 32) ? 1 : 0; }

size_t moe_scale_bytes(moe_scale_fmt_t fmt, int64_t rows, int32_t H, int32_t g) {
  if (rows < 0 || H <= 0 || (g != 32 && g != 128) || H % g || !fmt_ok(fmt, g)) return 0;
  const int64_t G = H / g;
  if (fmt == MOE_SCALE_UE8M0_U8 || fmt == MOE_SCALE_MX_E8M0) return (size_t)(rows * G);
  if (fmt == MOE_SCALE_F32_POW2 || fmt == MOE_SCALE_F32) return (size_t)(rows * G * 4);
  return (size_t)(((G + 3) / 4) * 4 * ((rows + 3) / 4 * 4));
}

size_t moe_workspace_bytes(int32_t T, int32_t K, int32_t L) {
  if (T < 0 || K < 1 || L < 1) return 0;
  const int64_t A = (int64_t)T * K;
  // the larger table of the two preferences, so one workspace fits every H
  // (a preference that no chain meets falls back to the shortest chain under
  // the hard limit, which can be the larger table)
  int64_t nc = 0;
  for (int64_t pref : {kRouteTablePrefSmall, kRouteTablePref}) {
    const RouteGeom geom = route_geometry(A, L, pref);
    if (geom.S == 0) return 0;
    if (geom.nchunks > nc) nc = geom.nchunks;
  }
  return kWsHeader + (size_t)nc * (size_t)L * sizeof(int32_t);
}

moe_status_t moe_dispatch_compact(
    const void* x, int64_t ldx, int32_t T, const int32_t* d_num_tokens, int32_t H,
    const int32_t* topk_ids, const float* topk_weights, int32_t K, int32_t E, int32_t L,
    int32_t block_e, int32_t g, moe_scale_fmt_t fmt,
    void* xq, void* scales, int64_t ld_s, int32_t* m_indices, int64_t bound,
    int32_t* src2dst, int32_t* counts, int32_t* starts, int32_t* psum, int32_t* total,
    float* row_weights, void* workspace, size_t workspace_bytes, int32_t* d_status,
    moe_stream_t stream) {
  DispatchCommon c{x, ldx, T, d_num_tokens, H, topk_ids, topk_weights, K, E, L, g, (int)fmt,
                   xq, scales, ld_s, src2dst, row_weights, workspace, workspace_bytes};
  moe_status_t st = check_common(c);
  if (st != MOE_OK) return st;
  if (block_e < 1) return MOE_ERR_INVALID_ARG;
  const int64_t need = moe_compact_bound((int64_t)T * K, L, block_e);
  if (bound < need || bound >= (int64_t(1) << 31)) return MOE_ERR_INVALID_ARG;
  if (!counts || !starts || !psum || !total) return MOE_ERR_INVALID_ARG;
  if (bound > 0 && (!m_indices || !xq || !aligned16(xq) || !scales || !aligned16(scales)))
    return MOE_ERR_INVALID_ARG;
  if (bound > 0 && !ld_ok(fmt, ld_s, bound, H / g)) return MOE_ERR_INVALID_ARG;
  return run_dispatch(c, kModeCompact, block_e, 0, m_indices, bound, counts, starts, psum,
                      total, nullptr, d_status, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_dispatch_masked(
    const void* x, int64_t ldx, int32_t T, const int32_t* d_num_tokens, int32_t H,
    const int32_t* topk_ids, const float* topk_weights, int32_t K, int32_t E, int32_t L,
    int32_t cap, int32_t g, moe_scale_fmt_t fmt,
    void* xq, void* scales, int64_t ld_s, int32_t* masked_m, int32_t* src2dst,
    float* row_weights, int32_t* psum, int32_t psum_align, void* workspace,
    size_t workspace_bytes, int32_t* d_status, moe_stream_t stream) {
  DispatchCommon c{x, ldx, T, d_num_tokens, H, topk_ids, topk_weights, K, E, L, g, (int)fmt,
                   xq, scales, ld_s, src2dst, row_weights, workspace, workspace_bytes};
  moe_status_t st = check_common(c);
  if (st != MOE_OK) return st;
  if (cap < 1 || (int64_t)L * cap >= (int64_t(1) << 31)) return MOE_ERR_INVALID_ARG;
  if (!masked_m || !xq || !aligned16(xq) || !scales || !aligned16(scales)) return MOE_ERR_INVALID_ARG;
  if (!ld_ok(fmt, ld_s, cap, H / g)) return MOE_ERR_INVALID_ARG;
  // the expanded layout of the slab rows ends below align * L + L * cap
  if (psum && (psum_align < 1 || (int64_t)L * (psum_align + (int64_t)cap) >= (int64_t(1) << 31)))
    return MOE_ERR_INVALID_ARG;
  return run_dispatch(c, kModeMasked, psum ? psum_align : 1, cap, nullptr, 0, nullptr, nullptr,
                      psum, nullptr, masked_m, d_status, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_quant_group(const void* x, int64_t ldx, int32_t T_cap, const int32_t* d_num_live,
                             int32_t H, int32_t g, moe_scale_fmt_t fmt, void* xq, void* scales,
                             int64_t ld_s, int32_t* d_status, moe_stream_t stream) {
  if (T_cap < 0 || H <= 0 || H % 16 || H > kMaxHidden || (g != 32 && g != 128) || H % g ||
      !fmt_ok(fmt, g))
    return MOE_ERR_INVALID_ARG;
  if (T_cap == 0) return MOE_OK;
  if (!x || !aligned16(x) || ldx < H || ldx % 8) return MOE_ERR_INVALID_ARG;
  if (!xq || !aligned16(xq) || !scales || !aligned16(scales)) return MOE_ERR_INVALID_ARG;
  if (!ld_ok(fmt, ld_s, T_cap, H / g)) return MOE_ERR_INVALID_ARG;
  const int sms = num_sms_cached();
  if (sms <= 0) return MOE_ERR_CUDA;
  ScatterArgs sa{};
  sa.x = static_cast<const uint16_t*>(x); sa.ldx = ldx; sa.T = T_cap; sa.d_num_tokens = d_num_live;
  sa.H = H; sa.K = 1; sa.L = 1; sa.mode = kModeIdentity; sa.cap = 0; sa.chunk = 1;
  sa.xq = static_cast<uint8_t*>(xq); sa.scales = scales; sa.ld_s = ld_s; sa.status = d_status;
  return cuda_status(launch_quant_scatter(sa, g, (int)fmt, sms, /*after_route_plan=*/false,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_combine(const void* y, int64_t ldy, int64_t R, const int32_t* src2dst,
                         const float* w, int32_t T, const int32_t* d_num_tokens, int32_t K,
                         int32_t H, void* out, int32_t* d_status, moe_stream_t stream) {
  if (T < 0 || K < 1 || K > kMaxK || H <= 0 || H % 8 || R < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!src2dst || !out || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if (R > 0 && (!y || !aligned16(y) || ldy < H || ldy % 8)) return MOE_ERR_INVALID_ARG;
  const int sms = num_sms_cached();
  if (sms <= 0) return MOE_ERR_CUDA;
  CombineArgs ca{};
  ca.y = static_cast<const uint16_t*>(y); ca.ldy = ldy; ca.R = R; ca.src2dst = src2dst; ca.w = w;
  ca.T = T; ca.d_num_tokens = d_num_tokens; ca.K = K; ca.H = H;
  ca.out = static_cast<uint16_t*>(out); ca.status = d_status;
  return cuda_status(launch_combine(ca, sms, reinterpret_cast<cudaStream_t>(stream)));
}

static moe_status_t repack_common(int to_slab, const void* src, void* dst, int32_t elem_bytes,
                                  int32_t H, int64_t R, const void* src_scales, int64_t ld_src,
                                  void* dst_scales, int64_t ld_dst, const int32_t* psum, int32_t L,
                                  int32_t align, int32_t cap, moe_scale_fmt_t fmt, int32_t g,
                                  const float* row_weights, int32_t* masked_m, int32_t* m_indices,
                                  int32_t* d_status, cudaStream_t stream) {
  if ((elem_bytes != 1 && elem_bytes != 2) || H <= 0 || H % 16 || R < 0) return MOE_ERR_INVALID_ARG;
  if (L < 1 || L > kMaxL || align < 1 || cap < 1 || (int64_t)L * cap >= (int64_t(1) << 31))
    return MOE_ERR_INVALID_ARG;
  if (R >= (int64_t(1) << 31) || !psum) return MOE_ERR_INVALID_ARG;
  if (!src || !dst || !aligned16(src) || !aligned16(dst)) return MOE_ERR_INVALID_ARG;
  if ((src_scales == nullptr) != (dst_scales == nullptr)) return MOE_ERR_INVALID_ARG;
  int G = 0;
  if (src_scales) {
    if (elem_bytes != 1 || (g != 32 && g != 128) || H % g || !fmt_ok(fmt, g)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(src_scales) || !aligned16(dst_scales)) return MOE_ERR_INVALID_ARG;
    G = H / g;
    const int64_t ld_exp = to_slab ? ld_src : ld_dst;
    const int64_t ld_slab = to_slab ? ld_dst : ld_src;
    if (!ld_ok(fmt, ld_exp, R, G) || !ld_ok(fmt, ld_slab, cap, G)) return MOE_ERR_INVALID_ARG;
  }
  if (row_weights && elem_bytes != 2) return MOE_ERR_INVALID_ARG;
  const int sms = num_sms_cached();
  if (sms <= 0) return MOE_ERR_CUDA;
  RepackArgs ra{};
  ra.to_slab = to_slab; ra.src = static_cast<const uint8_t*>(src); ra.dst = static_cast<uint8_t*>(dst);
  ra.elem_bytes = elem_bytes; ra.H = H; ra.R = R;
  ra.src_scales = src_scales; ra.ld_src_s = ld_src; ra.dst_scales = dst_scales; ra.ld_dst_s = ld_dst;
  ra.psum = psum; ra.L = L; ra.align = align; ra.cap = cap; ra.fmt = (int)fmt; ra.G = G;
  ra.row_weights = row_weights; ra.masked_m = masked_m; ra.m_indices = m_indices; ra.status = d_status;
  return cuda_status(launch_repack(ra, sms, stream));
}

moe_status_t moe_expand_to_slab(const void* exp, int32_t elem_bytes, int32_t H, int64_t R,
                                const void* exp_scales, int64_t ld_es, const int32_t* psum,
                                int32_t L, int32_t align, int32_t cap, moe_scale_fmt_t fmt,
                                int32_t g, void* slab, void* slab_scales, int64_t ld_ss,
                                int32_t* masked_m, int32_t* d_status, moe_stream_t stream) {
  if (!masked_m) return MOE_ERR_INVALID_ARG;
  return repack_common(1, exp, slab, elem_bytes, H, R, exp_scales, ld_es, slab_scales, ld_ss,
                       psum, L, align, cap, fmt, g, nullptr, masked_m, nullptr, d_status,
                       reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_expand_from_slab(const void* slab, int32_t elem_bytes, int32_t H,
                                  const void* slab_scales, int64_t ld_ss, const int32_t* psum,
                                  int32_t L, int32_t align, int32_t cap, moe_scale_fmt_t fmt,
                                  int32_t g, const float* row_weights, void* exp, int64_t R,
                                  void* exp_scales, int64_t ld_es, int32_t* m_indices,
                                  int32_t* d_status, moe_stream_t stream) {
  return repack_common(0, slab, exp, elem_bytes, H, R, slab_scales, ld_ss, exp_scales, ld_es,
                       psum, L, align, cap, fmt, g, row_weights, nullptr, m_indices, d_status,
                       reinterpret_cast<cudaStream_t>(stream));
}

static moe_status_t requant_common(const void* q, int64_t ldq, const void* s_tok, int s_fmt,
                                   int32_t T, int32_t H, int mode, void* q_out, float* d_scale_out,
                                   void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (T < 0 || H <= 0 || H % 16 || !d_scale_out) return MOE_ERR_INVALID_ARG;
  if (s_fmt != MOE_TOKSCALE_F32 && s_fmt != MOE_TOKSCALE_UE8M0) return MOE_ERR_INVALID_ARG;
  if (mode != MOE_REQUANT_MAX_SCALE && mode != MOE_REQUANT_AMAX) return MOE_ERR_INVALID_ARG;
  if (T > 0) {
    if (!q || !aligned16(q) || ldq < H || ldq % 16 || !s_tok) return MOE_ERR_INVALID_ARG;
    if (!q_out || !aligned16(q_out)) return MOE_ERR_INVALID_ARG;
    if (mode == MOE_REQUANT_AMAX &&
        (!workspace || !aligned16(workspace) || workspace_bytes < (size_t)T * sizeof(float)))
      return MOE_ERR_INVALID_ARG;
  }
  const int sms = num_sms_cached();
  if (sms <= 0) return MOE_ERR_CUDA;
  RequantArgs ra{};
  ra.q = static_cast<const uint8_t*>(q); ra.ldq = ldq; ra.s_tok = s_tok;
  ra.s_fmt = s_fmt; ra.mode = mode; ra.T = T; ra.H = H;
  ra.q_out = static_cast<uint8_t*>(q_out); ra.scale_out = d_scale_out;
  ra.ws = static_cast<float*>(workspace);
  return cuda_status(launch_requant(ra, sms, stream));
}

moe_status_t fp8_requant_per_tensor(const void* q, int64_t ldq, const float* s_tok, int32_t T,
                                    int32_t H, void* q_out, float* d_scale_out,
                                    moe_stream_t stream) {
  return requant_common(q, ldq, s_tok, MOE_TOKSCALE_F32, T, H, MOE_REQUANT_MAX_SCALE, q_out,
                        d_scale_out, nullptr, 0, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t fp8_requant_per_tensor_ex(const void* q, int64_t ldq, const void* s_tok,
                                       moe_tokscale_fmt_t s_fmt, int32_t T, int32_t H,
                                       moe_requant_mode_t mode, void* q_out, float* d_scale_out,
                                       void* workspace, size_t workspace_bytes,
                                       moe_stream_t stream) {
  return requant_common(q, ldq, s_tok, (int)s_fmt, T, H, (int)mode, q_out, d_scale_out,
                        workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_status_sync(const int32_t* d_status, moe_stream_t stream) {
  if (!d_status) return MOE_ERR_INVALID_ARG;
  int32_t v = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, d_status, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (v & MOE_STATUS_BAD_LAYOUT) return MOE_ERR_BAD_LAYOUT;
  if (v & MOE_STATUS_LIVE_OVERFLOW) return MOE_ERR_LIVE_OVERFLOW;
  if (v & MOE_STATUS_OVERFLOW) return MOE_ERR_OVERFLOW;
  return MOE_OK;
}

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (rejected before launch)";
    case MOE_ERR_OVERFLOW: return "an expert received more rows than its slab capacity";
    case MOE_ERR_LIVE_OVERFLOW: return "live-row count larger than the buffer";
    case MOE_ERR_BAD_LAYOUT: return "prefix sums or row indices inconsistent with the buffers";
    case MOE_ERR_CUDA: return "CUDA runtime error";
  }
  return "unknown status";
}

const char* moe_version(void) { return "moeperm 0.1 sm_103a"; }

}  // extern "C"
