// dispatch_small.cu -- the whole dispatch in ONE launch for small problems
// (T*K <= 2048 slots: decode batches), where launch latency, not bandwidth,
// sets the time.
//
// Computes exactly what route_plan.cu + quant_scatter.cu compute (same
// layout, same stable row order, same quantisation; PR #33128 实现拆解 items
// 2-4 and code excerpts _get_compact_all_tokens / _fwd_kernel_ep_scatter_1;
// PR #29525 masked slab, masked_m, overflow), but every CTA ranks ALL slots
// itself in shared memory instead of reading a chunk table written by a first
// launch. The slots are few, so the redundant ranking costs each CTA a few
// microseconds of on-chip work and no inter-CTA communication at all.
//
// Per CTA (256 threads = 8 warps):
//   1. issue the loads of its first token's row;
//   2. warp w ranks the slots [w*32*S, (w+1)*32*S) in order: peer masks from
//      one ballot per bit of the expert id, a per-warp counter per expert in
//      shared memory advanced step by step (stable ranks);
//   3. per expert, an exclusive scan over the 8 warps and the count; compact:
//      a block scan of the block_e-aligned counts gives the segment starts;
//   4. every slot's row goes to shared memory; CTA 0 writes counts / starts /
//      psum / total (or masked_m and the overflow flag); the CTAs share the
//      m_indices fill and write src2dst / row weights of their own tokens;
//   5. quantise its tokens (a 16-element chunk pair per thread per pass,
//      xor-shuffle group max, exponent from the float's bits, hardware e4m3
//      converts) and store each 16-byte vector to every destination row.
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "scales.cuh"

namespace moeperm {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kCPT = 2;


template <int GSZ, int FMT, int S>
__global__ void __launch_bounds__(kThreads) dispatch_small_kernel(ScatterArgs p) {
  extern __shared__ int32_t sm[];
  __shared__ int32_t s_wsum[33];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = p.L, K = p.K, H = p.H;
  const int nch = H / 16, G = H / GSZ, G4 = (G + 3) / 4;
  int32_t* hw = sm;                   // [kWarps][L] per-warp counters -> warp bases
  int32_t* st = hw + kWarps * L;      // [L] expert row base (compact start, masked 0)
  int32_t* ps = st + L;               // [L] count, then compact psum
  int32_t* rows_all = ps + L;         // [T*K] row of every slot
  int32_t* exps_all = rows_all + (int64_t)p.T * K;  // [T*K] expert of every slot

  const int n_live = live_count(p.d_num_tokens, p.T, p.status, blockIdx.x == 0 && tid == 0);
  const int64_t A = (int64_t)p.T * K, A_live = (int64_t)n_live * K;

  // 1. first token's loads
  const int t0 = blockIdx.x;
  uint4 v[kCPT][2];
#pragma unroll
  for (int i = 0; i < kCPT; ++i) {
    const int c = i * kThreads + tid;
    if (t0 < n_live && c < nch) {
      const uint16_t* xr = p.x + (int64_t)t0 * p.ldx + c * 16;
      v[i][0] = ld_nc_v4(xr);
      v[i][1] = ld_nc_v4(xr + 8);
    } else {
      v[i][0] = v[i][1] = make_uint4(0, 0, 0, 0);
    }
  }

  // 2. stable ranks of all slots
  for (int i = tid; i < kWarps * L; i += kThreads) hw[i] = 0;
  const int base = warp * 32 * S;
  int32_t r[S];
#pragma unroll
  for (int i = 0; i < S; ++i) {
    const int64_t a = base + i * 32 + lane;
    const int e = (a < A_live) ? __ldg(p.ids + a) : -1;
    r[i] = (e >= 0 && e < L) ? e : -1;
  }
  __syncthreads();
  int32_t* myhw = hw + warp * L;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int nbits = (L > 1) ? 32 - __clz(L - 1) : 0;
#pragma unroll
  for (int i = 0; i < S; ++i) {
    const int e = r[i];
    unsigned m = __ballot_sync(0xffffffffu, e >= 0);
    for (int b = 0; b < nbits; ++b) {
      const unsigned bit = (unsigned)(e >> b) & 1u;
      const unsigned bal = __ballot_sync(0xffffffffu, bit);
      m &= bit ? bal : ~bal;
    }
    const unsigned peers = (e >= 0) ? m : 0u;
    const int lower = __popc(peers & lt_mask);
    int rank = 0;
    if (e >= 0) rank = myhw[e] + lower;
    __syncwarp();
    if (e >= 0 && lower == 0) myhw[e] += __popc(peers);
    __syncwarp();
    r[i] = (e >= 0) ? ((rank << 11) | (e + 1)) : 0;
  }
  __syncthreads();

  // 3. warp bases and counts per expert; segment starts
  for (int e = tid; e < L; e += kThreads) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int c = hw[w * L + e];
      hw[w * L + e] = run;
      run += c;
    }
    ps[e] = run;
  }
  __syncthreads();
  if (p.mode == kModeCompact) {
    const int total = aligned_starts(ps, st, L, p.block_e, INT_MAX, s_wsum);
    for (int e = tid; e < L; e += kThreads) ps[e] += st[e];  // count -> psum
    if (blockIdx.x == 0 && tid == 0) *p.total = total;
    __syncthreads();
    if (blockIdx.x == 0)
      for (int e = tid; e < L; e += kThreads) {
        p.counts[e] = ps[e] - st[e];
        p.starts[e] = st[e];
        p.psum[e] = ps[e];
      }
    if (p.m_indices != nullptr)
      for (int64_t rr = (int64_t)blockIdx.x * kThreads + tid; rr < p.bound;
           rr += (int64_t)gridDim.x * kThreads) {
        int lo2 = 0, hi2 = L - 1;  // largest e with start[e] <= rr (start[0] = 0)
        while (lo2 < hi2) {
          const int mid = (lo2 + hi2 + 1) >> 1;
          if (st[mid] <= rr) lo2 = mid; else hi2 = mid - 1;
        }
        p.m_indices[rr] = (rr < ps[lo2]) ? lo2 : -1;
      }
  } else {
    // masked: slab rows need no start, so st takes the expanded-layout starts
    // of the slab's real rows when psum is asked for (PR #29525 _build_layout)
    bool overflow = false;
    for (int e = tid; e < L; e += kThreads) {
      if (blockIdx.x == 0) p.masked_m[e] = min(ps[e], p.cap);
      if (ps[e] > p.cap) overflow = true;
    }
    if (overflow && blockIdx.x == 0) set_status(p.status, kStOverflow);
    if (p.psum != nullptr && blockIdx.x == 0) {  // uniform over the CTA
      aligned_starts(ps, st, L, p.block_e, p.cap, s_wsum);
      for (int e = tid; e < L; e += kThreads) p.psum[e] = st[e] + min(ps[e], p.cap);
    }
    __syncthreads();
  }

  // 4. rows of all slots (each lane resolves its own slots)
#pragma unroll
  for (int i = 0; i < S; ++i) {
    const int64_t a = base + i * 32 + lane;
    if (a >= A) continue;
    const int pk = r[i];
    int row = -1;
    if (pk) {
      const int e = (pk & 0x7FF) - 1;
      const int j = hw[warp * L + e] + (pk >> 11);  // rank among all slots of e
      if (p.mode == kModeCompact) row = st[e] + j;
      else if (j < p.cap) row = e * p.cap + j;
    }
    rows_all[a] = row;
    exps_all[a] = pk ? (pk & 0x7FF) - 1 : -1;
  }
  __syncthreads();

  // src2dst and row weights of this CTA's tokens (each slot written once)
  for (int t = blockIdx.x; t < p.T; t += gridDim.x)
    for (int k = tid; k < K; k += kThreads) {
      const int64_t a = (int64_t)t * K + k;
      const int row = rows_all[a];
      p.src2dst[a] = row;
      if (row >= 0 && p.row_weights != nullptr) p.row_weights[row] = __ldg(p.w + a);
    }

  // 5. quantise + scatter this CTA's tokens
  for (int t = t0; t < n_live; t += gridDim.x) {
    const int* rows = rows_all + (int64_t)t * K;
    const int* exps = exps_all + (int64_t)t * K;
    for (int c0 = 0; c0 < nch; c0 += kCPT * kThreads) {
      if (t != t0 || c0 > 0) {
#pragma unroll
        for (int i = 0; i < kCPT; ++i) {
          const int c = c0 + i * kThreads + tid;
          if (c < nch) {
            const uint16_t* xr = p.x + (int64_t)t * p.ldx + c * 16;
            v[i][0] = ld_nc_v4(xr);
            v[i][1] = ld_nc_v4(xr + 8);
          } else {
            v[i][0] = v[i][1] = make_uint4(0, 0, 0, 0);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kCPT; ++i) {
        const int c = c0 + i * kThreads + tid;
        const bool active = c < nch;
        uint32_t m = amax16_bf16(v[i][0], v[i][1]);
#pragma unroll
        for (int off = 1; off < GSZ / 16; off <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
        const float amax = __uint_as_float(m << 16);
        int e = 0;
        float sval = 0.0f;
        uint2 q0, q1;
        if constexpr (FMT == kFmtF32) {
          sval = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
          q0 = quant8_div(v[i][0], sval);
          q1 = quant8_div(v[i][1], sval);
        } else {
          e = (FMT == kFmtMX) ? mx_exponent(amax) : group_exponent(amax);
          const float inv = exp2_neg(e);
          q0 = quant8(v[i][0], inv);
          q1 = quant8(v[i][1], inv);
        }
        const uint4 q = make_uint4(q0.x, q0.y, q1.x, q1.y);
        if (active)
          for (int k = 0; k < K; ++k) {
            const int row = rows[k];
            if (row >= 0) st_v4(p.xq + (int64_t)row * H + c * 16, q);
          }
        const int cw = c0 + i * kThreads + (tid & ~31);
        if (cw < nch)
          store_scales<GSZ, FMT>(p, K, rows, exps, lane, active, e, sval, cw * 16 / GSZ, G, G4);
      }
    }
  }
}

template <int GSZ, int FMT, int S>
cudaError_t launch_s(const ScatterArgs& a, int num_sms, cudaStream_t s) {
  const size_t smem = ((size_t)kWarps * a.L + 2 * (size_t)a.L + 2 * (size_t)a.T * a.K) * sizeof(int32_t);
  cudaError_t err = opt_in_smem(dispatch_small_kernel<GSZ, FMT, S>, smem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = occupancy(dispatch_small_kernel<GSZ, FMT, S>, kThreads, smem, &per_sm);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  int64_t grid = (int64_t)num_sms * per_sm;
  if (grid > a.T) grid = a.T;
  if (grid < 1) grid = 1;
  dispatch_small_kernel<GSZ, FMT, S><<<(unsigned)grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <int GSZ, int FMT>
cudaError_t launch_f(const ScatterArgs& a, int num_sms, cudaStream_t s) {
  const int64_t A = (int64_t)a.T * a.K;
  static_assert(kWarps * 32 * 16 == kSmallSlotsMax, "ranking capacity of one CTA");
  if (A > kSmallSlotsMax) return cudaErrorInvalidValue;  // slots past the capacity would stay unranked
  if (A <= 256) return launch_s<GSZ, FMT, 1>(a, num_sms, s);
  if (A <= 1024) return launch_s<GSZ, FMT, 4>(a, num_sms, s);
  if (A <= 2048) return launch_s<GSZ, FMT, 8>(a, num_sms, s);
  return launch_s<GSZ, FMT, 16>(a, num_sms, s);
}

}  // namespace

cudaError_t launch_dispatch_small(const ScatterArgs& a, int g, int fmt, int num_sms,
                                  cudaStream_t s) {
  if (g == 128) {
    if (fmt == kFmtPacked) return launch_f<128, kFmtPacked>(a, num_sms, s);
    if (fmt == kFmtU8) return launch_f<128, kFmtU8>(a, num_sms, s);
    if (fmt == kFmtF32) return launch_f<128, kFmtF32>(a, num_sms, s);
    return launch_f<128, kFmtF32Pow2>(a, num_sms, s);
  }
  if (fmt == kFmtMX) return launch_f<32, kFmtMX>(a, num_sms, s);
  return launch_f<32, kFmtU8>(a, num_sms, s);
}

}  // namespace moeperm
