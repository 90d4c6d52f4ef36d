// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernel translation units. Not installed; the public interface is
// include/moeperm.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moeperm {

// Largest chunk table (chunks x local experts, int32) a dispatch may use: the
// scatter launch holds it in shared memory (64 KiB).
constexpr int kMaxTableInts = 16384;

// ---------------------------------------------------------------------------
// Route plan: per-chunk expert histograms and stable in-chunk ranks.
// ---------------------------------------------------------------------------
struct RoutePlanArgs {
  const int32_t* ids;          // [T, K]
  const int32_t* d_num_tokens; // optional live tokens
  int32_t T, K, L;
  int32_t chunk;               // assignments per chunk (= 32 * warps * S)
  int32_t nchunks;
  int32_t* lrank;              // [T*K] out: stable rank inside the chunk, -1 dropped
  int32_t* table;              // [nchunks, L] out: chunk histogram
  int32_t* status;
  int32_t* queue;              // optional: set to 0 (the scatter's token counter)
};
// Launch geometry of the route plan: S slots per lane (the length of each
// warp's dependent chain), warps per CTA, chunk = 32 * warps * S slots per CTA.
struct RouteGeom {
  int S;                       // 0: the chunk table cannot fit kMaxTableInts
  int warps;
  int32_t chunk;
  int64_t nchunks;
};
// The shortest chain S whose table (chunks x L) fits table_pref ints, else
// the shortest whose table fits kMaxTableInts. A smaller table costs a longer
// chain but less shared memory and fewer table loads in every scatter CTA.
// Measured on GB300 across T, H, L, E and top-k: a token with few kept slots
// (L <= 128 local experts) or a narrow row gives each scatter CTA little work
// per token, so its loop is latency-bound and the residency that a small
// table leaves (4 rather than 3 CTAs per SM at H = 7168) decides; with more
// experts the loop is bandwidth-bound and the shorter chain wins.
constexpr int64_t kRouteTablePref = 8192;
constexpr int64_t kRouteTablePrefSmall = 2048;
constexpr int kNarrowRow = 4096;   // H below this: the small-table preference
constexpr int kFewExperts = 128;   // L up to this: the small-table preference
inline int64_t route_table_pref(int H, int L) {
  return (H < kNarrowRow || L <= kFewExperts) ? kRouteTablePrefSmall : kRouteTablePref;
}
RouteGeom route_geometry(int64_t A, int L, int64_t table_pref);
cudaError_t launch_route_plan(const RoutePlanArgs& a, const RouteGeom& g, cudaStream_t s);

// ---------------------------------------------------------------------------
// Quantise + scatter (dispatch) / quantise live rows (identity mode).
// ---------------------------------------------------------------------------
struct ScatterArgs {
  const uint16_t* x;
  int64_t ldx;
  int32_t T;
  const int32_t* d_num_tokens;
  int32_t H;
  const int32_t* ids;
  const float* w;
  int32_t K, L;
  int32_t E;                   // all experts (the ids range over [0, E); local ones are [0, L))
  int32_t mode;
  int32_t block_e, cap;
  int32_t chunk, nchunks;
  const int32_t* table;        // route-plan chunk histograms [nchunks, L]
  uint8_t* xq;
  void* scales;
  int64_t ld_s;
  int32_t* src2dst;            // in: chunk rank, out: final row (-1 dropped)
  float* row_weights;
  int32_t* m_indices;          // compact: [bound]
  int64_t bound;
  int32_t* counts;             // compact outputs [L] (CTA 0 writes them)
  int32_t* starts;
  int32_t* psum;
  int32_t* total;              // [1]
  int32_t* masked_m;           // masked output [L]
  int32_t* status;
  int32_t stages, pre;         // scatter: staging ring size, tokens staged before the wait
  int32_t direct;              // scatter: 1 = direct stores, no staging (few kept slots per token)
  int32_t* queue;              // direct mode: token counter, reset to 0 by the route plan
  int32_t dyn;                 // direct mode: tokens taken from the counter (set at launch)
  int32_t nstat;               // staged mode: static tokens per CTA, the rest from the counter
                               // (0: every token static; set at launch)
};
cudaError_t launch_quant_scatter(const ScatterArgs& a, int g, int fmt, int num_sms,
                                 bool after_route_plan, cudaStream_t s);

// Single-launch dispatch for small problems (T*K <= kSmallSlots): every CTA
// ranks all slots itself; no chunk table, no route-plan launch. Measured on
// GB300 (H = 7168, top-8): faster than the two-launch plan up to 2048 slots,
// equal at 2048, slower at 4096 (the redundant ranking grows with T*K).
constexpr int64_t kSmallSlots = 2048;
// The one-launch kernel ranks at most 8 warps x 32 lanes x 16 steps slots.
constexpr int64_t kSmallSlotsMax = 4096;
static_assert(kSmallSlots <= kSmallSlotsMax, "the one-launch dispatch ranks at most 4096 slots");
cudaError_t launch_dispatch_small(const ScatterArgs& a, int g, int fmt, int num_sms,
                                  cudaStream_t s);

// ---------------------------------------------------------------------------
// Combine
// ---------------------------------------------------------------------------
struct CombineArgs {
  const uint16_t* y;
  int64_t ldy;
  int64_t R;
  const int32_t* src2dst;
  const float* w;
  int32_t T;
  const int32_t* d_num_tokens;
  int32_t K, H;
  uint16_t* out;
  int32_t* status;
};
cudaError_t launch_combine(const CombineArgs& a, int num_sms, cudaStream_t s);

// ---------------------------------------------------------------------------
// Expanded <-> slab repack
// ---------------------------------------------------------------------------
struct RepackArgs {
  int32_t to_slab;             // 1: expanded -> slab, 0: slab -> expanded
  const uint8_t* src;
  uint8_t* dst;
  int32_t elem_bytes, H;
  int64_t R;                   // expanded rows
  const void* src_scales;
  int64_t ld_src_s;
  void* dst_scales;
  int64_t ld_dst_s;
  const int32_t* psum;
  int32_t L, align, cap, fmt, G;
  const float* row_weights;    // slab -> expanded, bf16 only
  int32_t* masked_m;           // expanded -> slab
  int32_t* m_indices;          // slab -> expanded, optional [R]
  int32_t* status;
};
cudaError_t launch_repack(const RepackArgs& a, int num_sms, cudaStream_t s);

// ---------------------------------------------------------------------------
// Per-token -> per-tensor requant
// ---------------------------------------------------------------------------
constexpr int kTokScaleF32 = 0;    // per-token scales: fp32
constexpr int kTokScaleE8M0 = 1;   // per-token scales: e8m0 bytes, 2^(b - 127)
constexpr int kRequantMaxScale = 0;
constexpr int kRequantAmax = 1;
struct RequantArgs {
  const uint8_t* q;
  int64_t ldq;
  const void* s_tok;
  int32_t s_fmt, mode;
  int32_t T, H;
  uint8_t* q_out;
  float* scale_out;
  float* ws;                   // amax mode: [T] per-row s * amax
};
cudaError_t launch_requant(const RequantArgs& a, int num_sms, cudaStream_t s);

}  // namespace moeperm
