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
// Design (grid of `nchunks` CTAs of W warps each, both chosen per launch by
// route_geometry): CTA c owns slots [c*chunk, (c+1)*chunk); warp w owns a
// contiguous sub-range of 32*S of them, walked in order in steps of 32. In a
// step, the lanes with the same expert are grouped (one match instruction, or
// one ballot per bit of the expert id); a lane's rank among them is the
// popcount of its lower peers, and the lowest peer adds the group size to the
// warp's per-expert counter in shared memory. A per-expert scan over the
// warps turns the warp-local ranks into chunk-local ones. Deterministic and
// stable, with no global atomics. The steps of one warp form a dependent
// chain, so the launch keeps S (the chain length) short and puts up to 32
// warps in a CTA instead: the chunk size, and so the table the scatter launch
// scans, stays small without a long chain. The CTA signals the dependent
// scatter launch at its start, so that launch is scheduled while this one
// runs (it waits for this grid's results before reading them).
#include "common.cuh"
#include "kernels.h"

namespace moeperm {

namespace {

constexpr int kGroup = 8;  // steps whose peer masks are formed together
// Per-warp histograms (warps x local experts, int32) a CTA may hold: 48 KiB.
constexpr int kHistInts = 12288;
// Warps a CTA may have for chain length S: the S = 64 kernel keeps its 64
// expert ids in registers and is built for 256 threads.
constexpr int max_warps_for(int S) { return S > 16 ? 8 : 32; }

template <int S>
__global__ void __launch_bounds__(32 * max_warps_for(S)) route_plan_kernel(RoutePlanArgs p) {
  extern __shared__ int32_t smem[];  // [warps][L] per-warp histograms
  pdl_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, bd = blockDim.x;
  const int nw = bd >> 5;
  const int L = p.L;

  for (int i = tid; i < nw * L; i += bd) smem[i] = 0;
  if (p.queue != nullptr && blockIdx.x == 0 && tid == 0) *p.queue = 0;  // read only after this grid ends
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

  // Lanes with the same expert ("peers"): one match over the warp (one
  // ballot per bit of the expert id measured the same). The masks of 8 steps are formed first (independent), then
  // the per-warp counters are advanced step by step in order, which fixes a
  // stable rank.
  int32_t* myhw = smem + warp * L;
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int i0 = 0; i0 < S; i0 += kGroup) {
    unsigned peers[kGroup];
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      if (i0 + j >= S) break;
      int e = v[i0 + j];
      if (e < 0 || e >= L) e = -1;
      v[i0 + j] = e;
      const unsigned m = __match_any_sync(0xffffffffu, e);
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

  // per-expert exclusive scan over the warps (8 loads in flight, then 8
  // stores); chunk histogram to the table
  for (int e = tid; e < L; e += bd) {
    int run = 0, w = 0;
    for (; w + 8 <= nw; w += 8) {
      int h[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) h[j] = smem[(w + j) * L + e];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        smem[(w + j) * L + e] = run;
        run += h[j];
      }
    }
    for (; w < nw; ++w) {
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

RouteGeom route_geometry(int64_t A, int L, int64_t table_pref) {
  RouteGeom g{};
  if (L < 1) return g;
  const int wmax = L >= kHistInts ? 1 : (kHistInts / L < 32 ? kHistInts / L : 32);
  const int cand[] = {1, 2, 4, 8, 16, 64};
  for (int64_t limit : {table_pref, (int64_t)kMaxTableInts}) {
    for (int S : cand) {
      const int W = wmax < max_warps_for(S) ? wmax : max_warps_for(S);
      const int64_t chunk = (int64_t)32 * W * S;
      int64_t nc = (A + chunk - 1) / chunk;
      if (nc < 1) nc = 1;
      if (nc * L <= limit) {
        g.S = S;
        g.warps = W;
        g.chunk = (int32_t)chunk;
        g.nchunks = nc;
        return g;
      }
    }
  }
  return g;  // S == 0: too large for one call
}

cudaError_t launch_route_plan(const RoutePlanArgs& a, const RouteGeom& g, cudaStream_t s) {
  const size_t smem = (size_t)g.warps * a.L * sizeof(int32_t);
  dim3 grid((unsigned)a.nchunks), block(32 * g.warps);
  cudaError_t err = cudaSuccess;
  switch (g.S) {
    case 1: err = opt_in_smem(route_plan_kernel<1>, smem); if (!err) route_plan_kernel<1><<<grid, block, smem, s>>>(a); break;
    case 2: err = opt_in_smem(route_plan_kernel<2>, smem); if (!err) route_plan_kernel<2><<<grid, block, smem, s>>>(a); break;
    case 4: err = opt_in_smem(route_plan_kernel<4>, smem); if (!err) route_plan_kernel<4><<<grid, block, smem, s>>>(a); break;
    case 8: err = opt_in_smem(route_plan_kernel<8>, smem); if (!err) route_plan_kernel<8><<<grid, block, smem, s>>>(a); break;
    case 16: err = opt_in_smem(route_plan_kernel<16>, smem); if (!err) route_plan_kernel<16><<<grid, block, smem, s>>>(a); break;
    case 64: err = opt_in_smem(route_plan_kernel<64>, smem); if (!err) route_plan_kernel<64><<<grid, block, smem, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace moeperm
