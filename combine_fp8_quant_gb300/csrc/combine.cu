// combine.cu -- gather expert outputs back to token order, weighted by the
// top-k weights (PR #33128 风险与影响 item 2: post_permute via src2dst).
//
//   out[t, :] = bf16_RNE( sum_{k : src2dst[t,k] >= 0} w[t,k] * y[src2dst[t,k], :] )
//   fp32 accumulator from +0, one fused multiply-add per slot in ascending k.
//
// Design: persistent grid; a CTA owns one token at a time and each thread owns
// 8-element (16-byte) chunks of it. There is no barrier: every thread reads
// the token's K row indices and weights itself (the warp's loads of the same
// words are one broadcast transaction), and the indices of the CTA's NEXT
// token are prefetched into registers while the current token is processed,
// so their latency never sits in front of the row loads. A thread issues the
// loads of up to 8 source rows for each of its CPT chunks before the first
// FMA. y is read once per kept slot and out written once: the kernel is bound
// by HBM reads.
#include "common.cuh"
#include "kernels.h"

namespace moeperm {

namespace {

constexpr int kBatch = 8;   // source rows loaded before accumulating
constexpr int kCPT = 2;     // 8-element chunks per thread per pass

struct Slots {
  int row[kBatch];
  float w[kBatch];
};

__device__ __forceinline__ void load_slots(const CombineArgs& p, int t, int n_live, int k0,
                                           Slots& s) {
#pragma unroll
  for (int j = 0; j < kBatch; ++j) {
    const int k = k0 + j;
    int row = -1;
    float w = 0.0f;
    if (t < n_live && k < p.K) {
      const int64_t a = (int64_t)t * p.K + k;
      row = __ldg(p.src2dst + a);
      if (row >= 0 && (int64_t)row >= p.R) {
        set_status(p.status, kStBadLayout);
        row = -1;
      }
      w = (p.w != nullptr) ? __ldg(p.w + a) : 1.0f;
    }
    s.row[j] = row;
    s.w[j] = w;
  }
}

__global__ void __launch_bounds__(256) combine_kernel(CombineArgs p) {
  const int tid = threadIdx.x, bd = blockDim.x;
  const int nch = p.H / 8;
  const int n_live = live_count(p.d_num_tokens, p.T, p.status, blockIdx.x == 0 && tid == 0);
  Slots next;
  load_slots(p, blockIdx.x, n_live, 0, next);
  for (int t = blockIdx.x; t < n_live; t += gridDim.x) {
    const Slots first = next;
    load_slots(p, t + gridDim.x, n_live, 0, next);  // prefetch the next token's slots
    uint16_t* orow = p.out + (int64_t)t * p.H;
    for (int c0 = 0; c0 < nch; c0 += kCPT * bd) {
      float acc[kCPT][8];
#pragma unroll
      for (int i = 0; i < kCPT; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
      for (int k0 = 0; k0 < p.K; k0 += kBatch) {
        Slots s;
        if (k0 == 0) s = first; else load_slots(p, t, n_live, k0, s);
        uint4 v[kCPT][kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
#pragma unroll
          for (int i = 0; i < kCPT; ++i) {
            const int c = c0 + i * bd + tid;
            if (s.row[j] >= 0 && c < nch)
              v[i][j] = ld_nc_v4(p.y + (int64_t)s.row[j] * p.ldy + c * 8);
            else
              v[i][j] = make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          if (s.row[j] >= 0) {
            const float wk = s.w[j];
#pragma unroll
            for (int i = 0; i < kCPT; ++i) {
              acc[i][0] = __fmaf_rn(wk, bf16_lo(v[i][j].x), acc[i][0]);
              acc[i][1] = __fmaf_rn(wk, bf16_hi(v[i][j].x), acc[i][1]);
              acc[i][2] = __fmaf_rn(wk, bf16_lo(v[i][j].y), acc[i][2]);
              acc[i][3] = __fmaf_rn(wk, bf16_hi(v[i][j].y), acc[i][3]);
              acc[i][4] = __fmaf_rn(wk, bf16_lo(v[i][j].z), acc[i][4]);
              acc[i][5] = __fmaf_rn(wk, bf16_hi(v[i][j].z), acc[i][5]);
              acc[i][6] = __fmaf_rn(wk, bf16_lo(v[i][j].w), acc[i][6]);
              acc[i][7] = __fmaf_rn(wk, bf16_hi(v[i][j].w), acc[i][7]);
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kCPT; ++i) {
        const int c = c0 + i * bd + tid;
        if (c < nch) {
          uint4 o;
          o.x = pack_bf16x2(acc[i][0], acc[i][1]);
          o.y = pack_bf16x2(acc[i][2], acc[i][3]);
          o.z = pack_bf16x2(acc[i][4], acc[i][5]);
          o.w = pack_bf16x2(acc[i][6], acc[i][7]);
          st_v4(orow + c * 8, o);
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, int num_sms, cudaStream_t s) {
  // Threads per CTA: enough chunks per thread that a thread covers its share of
  // the row in about two passes of kCPT chunks; at most 256.
  const int nch = a.H / 8;
  int bd = (nch + 2 * kCPT - 1) / (2 * kCPT);
  bd = (bd + 31) / 32 * 32;
  if (bd > 256) bd = 256;
  if (bd < 32) bd = 32;
  int per_sm = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_kernel, bd, 0);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  int64_t grid = (int64_t)num_sms * per_sm;
  if (grid > a.T) grid = a.T;
  if (grid < 1) grid = 1;
  combine_kernel<<<(unsigned)grid, bd, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moeperm
