// combine.cu -- gather expert outputs back to token order, weighted by the
// top-k weights (PR #33128 风险与影响 item 2: post_permute via src2dst).
//
//   out[t, :] = bf16_RNE( sum_{k : src2dst[t,k] >= 0} w[t,k] * y[src2dst[t,k], :] )
//   fp32 accumulator from +0, one fused multiply-add per slot in ascending k.
//
// Design: warp-centric and barrier-free. The work is split into units
// (token t, slice of 256 columns); warp i of the persistent grid takes units
// i, i + nwarps, ..., so neighbouring warps read neighbouring slices of the
// same source rows. Lane k < K holds slot k's row and weight and broadcasts
// them with shuffles; the slots of the warp's NEXT unit are loaded while the
// current unit is processed, so their latency never sits in front of the row
// loads. Each lane issues the 16-byte loads of a batch of source rows before
// the batch's FMAs: at most 4 rows (4 rows in flight with 32 warps per SM
// measured faster than 8 rows with 24 warps on the 8192-token prefill
// workload), in ceil(K/4) batches of equal size (top-6 as 3 + 3 rather than
// 4 + 2: 96% of the copy bandwidth instead of 93%). y is read once per kept
// slot and out written once: the kernel is bound by HBM reads.
#include "common.cuh"
#include "kernels.h"

namespace moeperm {

namespace {

// Largest batch of source rows in flight per lane (4 rows at 32 warps per SM
// beat 8 rows at 24 warps on the prefill workload: 163.8 against 182.3 us).
constexpr int kMaxBatch = 4;
// CTAs per SM the kernel is compiled for (8 warps each: 32 warps per SM).
constexpr int kMinBlocks = 4;
constexpr int kThreads = 256;

struct Slot {
  int row;
  float w;
};

// Slot `lane` of token t (row -1 beyond K or for a dropped / bad slot).
__device__ __forceinline__ Slot load_slot(const CombineArgs& p, int t, int n_live, int lane) {
  Slot s{-1, 0.0f};
  if (t < n_live && lane < p.K) {
    const int64_t a = (int64_t)t * p.K + lane;
    int row = __ldg(p.src2dst + a);
    if (row >= 0 && (int64_t)row >= p.R) {
      set_status(p.status, kStBadLayout);
      row = -1;
    }
    s.row = row;
    s.w = (p.w != nullptr) ? __ldg(p.w + a) : 1.0f;
  }
  return s;
}

template <int kBatch>  // source rows in flight per lane
__global__ void __launch_bounds__(kThreads, kMinBlocks) combine_kernel(CombineArgs p) {
  const int lane = threadIdx.x & 31;
  const int gwarp = (int)((blockIdx.x * kThreads + threadIdx.x) >> 5);
  const int nwarps = (int)((gridDim.x * kThreads) >> 5);
  const int nch = p.H / 8;                  // 8-element chunks per row
  const int spt = (nch + 31) / 32;          // slices per token
  const int n_live = live_count(p.d_num_tokens, p.T, p.status, blockIdx.x == 0 && threadIdx.x == 0);
  // unit (t, s) advances by nwarps units per step: (dt, ds) with a carry, no division in the loop
  const int dt = nwarps / spt, ds = nwarps % spt;
  int t = gwarp / spt, s = gwarp % spt;
  Slot cur = load_slot(p, t, n_live, lane);
  while (t < n_live) {
    int tn = t + dt, sn = s + ds;
    if (sn >= spt) {
      sn -= spt;
      ++tn;
    }
    const Slot nxt = load_slot(p, tn, n_live, lane);
    const int c = s * 32 + lane;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (int k0 = 0; k0 < p.K; k0 += kBatch) {
      uint4 v[kBatch];
      unsigned kept = 0;  // bit j: slot k0 + j contributes
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        int row = __shfl_sync(0xffffffffu, cur.row, (k0 + j) & 31);
        if (k0 + j >= p.K) row = -1;
        kept |= (row >= 0 ? 1u : 0u) << j;
        v[j] = (row >= 0 && c < nch) ? ld_nc_v4(p.y + (int64_t)row * p.ldy + c * 8)
                                     : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const float wk = __shfl_sync(0xffffffffu, cur.w, (k0 + j) & 31);
        if ((kept >> j) & 1u) {
          acc[0] = __fmaf_rn(wk, bf16_lo(v[j].x), acc[0]);
          acc[1] = __fmaf_rn(wk, bf16_hi(v[j].x), acc[1]);
          acc[2] = __fmaf_rn(wk, bf16_lo(v[j].y), acc[2]);
          acc[3] = __fmaf_rn(wk, bf16_hi(v[j].y), acc[3]);
          acc[4] = __fmaf_rn(wk, bf16_lo(v[j].z), acc[4]);
          acc[5] = __fmaf_rn(wk, bf16_hi(v[j].z), acc[5]);
          acc[6] = __fmaf_rn(wk, bf16_lo(v[j].w), acc[6]);
          acc[7] = __fmaf_rn(wk, bf16_hi(v[j].w), acc[7]);
        }
      }
    }
    if (c < nch) {
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      st_v4(p.out + (int64_t)t * p.H + c * 8, o);
    }
    cur = nxt;
    t = tn;
    s = sn;
  }
}

template <int kBatch>
cudaError_t launch_batch(const CombineArgs& a, int num_sms, cudaStream_t s) {
  int per_sm = 0;
  cudaError_t err = occupancy(combine_kernel<kBatch>, kThreads, 0, &per_sm);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  const int64_t spt = (a.H / 8 + 31) / 32;
  const int64_t units = (int64_t)a.T * spt;
  int64_t grid = (int64_t)num_sms * per_sm;
  const int64_t need = (units + (kThreads / 32) - 1) / (kThreads / 32);
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  combine_kernel<kBatch><<<(unsigned)grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, int num_sms, cudaStream_t s) {
  // the fewest batches of at most kMaxBatch rows, of equal size
  static_assert(kMaxBatch == 4, "one case per batch size below");
  const int nb = (a.K + kMaxBatch - 1) / kMaxBatch;
  const int batch = (a.K + nb - 1) / nb;
  switch (batch) {
    case 1: return launch_batch<1>(a, num_sms, s);
    case 2: return launch_batch<2>(a, num_sms, s);
    case 3: return launch_batch<3>(a, num_sms, s);
    default: return launch_batch<4>(a, num_sms, s);
  }
}

}  // namespace moeperm
