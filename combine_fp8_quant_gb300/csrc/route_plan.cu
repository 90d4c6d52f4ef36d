// route_plan.cu -- expert histogram, stable ranks and prefix sums for the
// compact and masked dispatch layouts.
//
// What it computes (PR #33128 实现拆解 items 2-3 and code excerpts
// _get_compact_all_tokens / _fwd_kernel_ep_scatter_1; PR #29525 _build_layout):
//   count[e]  = kept slots routed to local expert e (ids outside [0, L) dropped)
//   rank(a)   = kept slots a' < a with the same expert (rows follow t*K + k)
//   compact:  start[e] = sum_{e'<e} align(count[e'], block_e),
//             psum[e] = start[e] + count[e], total = sum align(count)
//   masked:   masked_m[e] = min(count[e], cap), overflow when count[e] > cap
//
// Design (one launch, fixed grid of `nchunks` CTAs of 8 warps):
//   * CTA c owns assignments [c*chunk, (c+1)*chunk); warp w owns a contiguous
//     sub-range of 32*S of them, walked in steps of 32 in order. In a step,
//     __match_any_sync groups the lanes with the same expert; a lane's rank
//     among them is the popcount of the lower peers, and the lowest peer adds
//     the group size to the warp's per-expert counter in shared memory. This
//     gives a deterministic, stable rank without global atomics.
//   * The 8 per-warp histograms are scanned per expert into warp bases, the
//     CTA's total histogram goes to the workspace table, and each slot's rank
//     inside the chunk is written to `lrank` (the caller's src2dst buffer,
//     rewritten with final rows by the scatter kernel).
//   * The last CTA to finish (a ticket taken with atomicInc after a
//     __threadfence, so no CTA ever waits for another) scans the table: per
//     expert an exclusive sum over chunks (the chunk's row base), the expert
//     totals, and a block-wide exclusive scan of the aligned counts. The
//     ticket wraps back to zero, so the workspace is ready for the next call.
#include "common.cuh"
#include "kernels.h"

namespace moeperm {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

template <int S>
__global__ void __launch_bounds__(kThreads) route_plan_kernel(RoutePlanArgs p) {
  extern __shared__ int32_t smem[];  // [kWarps][L] per-warp histograms
  __shared__ int s_last;
  __shared__ int32_t s_wsum[kWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = p.L;

  for (int i = tid; i < kWarps * L; i += kThreads) smem[i] = 0;
  const int n_live = live_count(p.d_num_tokens, p.T, p.status, blockIdx.x == 0 && tid == 0);
  const int64_t A = (int64_t)p.T * p.K;
  const int64_t A_live = (int64_t)n_live * p.K;
  __syncthreads();

  // --- stable ranks inside the warp's sub-range ---------------------------
  int32_t* myhw = smem + warp * L;
  const int64_t base = (int64_t)blockIdx.x * p.chunk + (int64_t)warp * (32 * S);
  int32_t v[S];  // the slot's expert id, then (rank << 11) | (expert + 1); 0 = dropped
#pragma unroll
  for (int i = 0; i < S; ++i) {
    const int64_t a = base + i * 32 + lane;
    v[i] = (a < A_live) ? __ldg(p.ids + a) : -1;
  }
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < S; ++i) {
    int e = v[i];
    if (e < 0 || e >= L) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int lower = __popc(peers & lt_mask);
    int rank = 0;
    if (e >= 0) rank = myhw[e] + lower;
    __syncwarp();
    if (e >= 0 && lower == 0) myhw[e] += __popc(peers);
    __syncwarp();
    v[i] = (e >= 0) ? ((rank << 11) | (e + 1)) : 0;
  }
  __syncthreads();

  // --- per-expert scan over the warps; chunk histogram to the table -------
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

  // --- last CTA: prefix sums over chunks and experts ----------------------
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned t = atomicInc(p.ticket, (unsigned)(p.nchunks - 1));
    s_last = (t == (unsigned)(p.nchunks - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  int32_t* s_cnt = smem;        // [L] counts
  int32_t* s_start = smem + L;  // [L] row base of each expert
  const int NC = p.nchunks;
  for (int e = tid; e < L; e += kThreads) {
    int sum = 0;
#pragma unroll 16
    for (int c = 0; c < NC; ++c) sum += __ldcg(p.table + (int64_t)c * L + e);
    s_cnt[e] = sum;
  }
  __syncthreads();

  if (p.mode == kModeCompact) {
    // exclusive scan of align(count) over experts; thread i owns a contiguous run
    const int per = (L + kThreads - 1) / kThreads;
    const int lo = min(tid * per, L), hi = min(lo + per, L);
    const int b = p.block_e;
    int local = 0;
    for (int e = lo; e < hi; ++e) local += (s_cnt[e] + b - 1) / b * b;
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int nb = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += nb;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    int wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += s_wsum[w];
    int run = wbase + incl - local;
    for (int e = lo; e < hi; ++e) {
      s_start[e] = run;
      run += (s_cnt[e] + b - 1) / b * b;
    }
    if (tid == kThreads - 1) *p.total = run;
    __syncthreads();
  } else {
    for (int e = tid; e < L; e += kThreads) s_start[e] = 0;
    __syncthreads();
  }

  bool overflow = false;
  for (int e = tid; e < L; e += kThreads) {
    const int cnt = s_cnt[e];
    const int st = s_start[e];
    int run = st;
#pragma unroll 16
    for (int c = 0; c < NC; ++c) {
      int32_t* cell = p.table + (int64_t)c * L + e;
      const int h = __ldcg(cell);
      *cell = run;
      run += h;
    }
    if (p.mode == kModeCompact) {
      p.counts[e] = cnt;
      p.starts[e] = st;
      p.psum[e] = st + cnt;
    } else {
      p.masked_m[e] = min(cnt, p.cap);
      if (cnt > p.cap) overflow = true;
    }
  }
  if (overflow) set_status(p.status, kStOverflow);
}

}  // namespace

int route_plan_S(int64_t A) {
  // Smallest S with at most 16 chunks; S = 64 allows up to 64 chunks (A <= 2^20).
  const int cand[] = {1, 4, 16};
  for (int S : cand)
    if ((A + (int64_t)kThreads * S - 1) / ((int64_t)kThreads * S) <= 16) return S;
  return 64;
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
