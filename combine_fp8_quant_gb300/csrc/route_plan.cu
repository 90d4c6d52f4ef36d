// route_plan.cu -- expert histogram and stable ranks for the compact and
// masked dispatch layouts (first of the two dispatch launches).
//
// What it computes (PR #33128 实现拆解 items 2-3 and code excerpts
// _get_compact_all_tokens / _fwd_kernel_ep_scatter_1; PR #29525 _build_layout):
//   kept slot   a = t*K + k of a live token with 0 <= id < L (others dropped)
//   table[c][e] = kept slots of chunk c routed to expert e
//   lrank[a]    = kept slots a' < a of the same chunk with the same expert
// The prefix sums over chunks and experts (segment starts, psum, total,
// masked_m) are formed from this table by every CTA of the scatter launch.
//
// Design (fixed grid of `nchunks` CTAs of kRouteWarps warps): CTA c owns slots
// [c*chunk, (c+1)*chunk); warp w owns a contiguous sub-range of 32*S of them,
// walked in order in steps of 32. In a step, ballots over the bits of the
// expert id group the lanes with the same expert; a lane's rank among them is
// the popcount of its lower peers, and the lowest peer adds the group size to
// the warp's per-expert counter in shared memory. A per-expert scan over the
// warps turns the warp-local ranks into chunk-local ones. Deterministic and stable, with no
// global atomics. The CTA signals the dependent scatter launch at its start,
// so that launch is scheduled while this one runs (it waits for this grid's
// results before reading them).
#include "common.cuh"
#include "kernels.h"

namespace moeperm {

namespace {

constexpr int kWarps = kRouteWarps;
constexpr int kThreads = kRouteThreads;
constexpr int kGroup = 8;  // steps whose peer masks are formed together
#ifndef MOEPERM_ROUTE_MAX_CHUNKS
#define MOEPERM_ROUTE_MAX_CHUNKS 16
#endif

template <int S>
__global__ void __launch_bounds__(kThreads) route_plan_kernel(RoutePlanArgs p) {
  extern __shared__ int32_t smem[];  // [kWarps][L] per-warp histograms
  pdl_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = p.L;

  for (int i = tid; i < kWarps * L; i += kThreads) smem[i] = 0;
  const int n_live = live_count(p.d_num_tokens, p.T, p.status, blockIdx.x == 0 && tid == 0);
  const int64_t A = (int64_t)p.T * p.K;
  const int64_t A_live = (int64_t)n_live * p.K;
  const int64_t base = (int64_t)blockIdx.x * p.chunk + (int64_t)warp * (32 * S);
  int32_t v[S];  // the slot's expert id, then (rank << 11) | (expert + 1); 0 = dropped
#pragma unroll
  for (int i = 0; i < S; ++i) {
    const int64_t a = base + i * 32 + lane;
    v[i] = (a < A_live) ? __ldg(p.ids + a) : -1;
  }
  __syncthreads();

  // Lanes with the same expert ("peers") are found with one ballot per bit of
  // the expert id: a lane keeps the lanes that agree with it on every bit.
  // The masks of 8 steps are formed first (independent), then the per-warp
  // counters are advanced step by step in order, which fixes a stable rank.
  int32_t* myhw = smem + warp * L;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int nbits = (L > 1) ? 32 - __clz(L - 1) : 0;
#pragma unroll
  for (int i0 = 0; i0 < S; i0 += kGroup) {
    unsigned peers[kGroup];
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      if (i0 + j >= S) break;
      int e = v[i0 + j];
      if (e < 0 || e >= L) e = -1;
      v[i0 + j] = e;
      unsigned m = __ballot_sync(0xffffffffu, e >= 0);
      for (int b = 0; b < nbits; ++b) {
        const unsigned bit = (unsigned)(e >> b) & 1u;
        const unsigned bal = __ballot_sync(0xffffffffu, bit);
        m &= bit ? bal : ~bal;
      }
      peers[j] = (e >= 0) ? m : 0u;
    }
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      if (i0 + j >= S) break;
      const int e = v[i0 + j];
      const int lower = __popc(peers[j] & lt_mask);
      int rank = 0;
      if (e >= 0) rank = myhw[e] + lower;
      __syncwarp();
      if (e >= 0 && lower == 0) myhw[e] += __popc(peers[j]);
      __syncwarp();
      v[i0 + j] = (e >= 0) ? ((rank << 11) | (e + 1)) : 0;
    }
  }
  __syncthreads();

  // per-expert exclusive scan over the warps; chunk histogram to the table
  for (int e = tid; e < L; e += kThreads) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int c = smem[w * L + e];
      smem[w * L + e] = run;
      run += c;
    }
    p.table[(int64_t)blockIdx.x * L + e] = run;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < S; ++i) {
    const int64_t a = base + i * 32 + lane;
    if (a < A) {
      const int pk = v[i];
      p.lrank[a] = pk ? (myhw[(pk & 0x7FF) - 1] + (pk >> 11)) : -1;
    }
  }
}

}  // namespace

int route_plan_S(int64_t A, int L) {
  // Smallest S whose chunk table fits kMaxTableInts (the scatter launch holds
  // it in shared memory), preferring at most 16 chunks (a smaller table for
  // every scatter CTA to scan).
  const int cand[] = {1, 4, 16, 64};
  for (int S : cand) {
    const int64_t nc = (A + (int64_t)kThreads * S - 1) / ((int64_t)kThreads * S);
    if (nc <= MOEPERM_ROUTE_MAX_CHUNKS && nc * L <= kMaxTableInts) return S;
  }
  for (int S : cand) {
    const int64_t nc = (A + (int64_t)kThreads * S - 1) / ((int64_t)kThreads * S);
    if (nc * L <= kMaxTableInts) return S;
  }
  return 0;  // too large for one call
}

cudaError_t launch_route_plan(const RoutePlanArgs& a, int S, cudaStream_t s) {
  const size_t smem = (size_t)kWarps * a.L * sizeof(int32_t);
  dim3 grid(a.nchunks), block(kThreads);
  switch (S) {
    case 1: route_plan_kernel<1><<<grid, block, smem, s>>>(a); break;
    case 4: route_plan_kernel<4><<<grid, block, smem, s>>>(a); break;
    case 16: route_plan_kernel<16><<<grid, block, smem, s>>>(a); break;
    default: route_plan_kernel<64><<<grid, block, smem, s>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace moeperm
