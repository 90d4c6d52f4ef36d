// quant_scatter.cu -- FP8 group quantisation fused with the dispatch scatter.
//
// What it computes:
//   * [PR #33128 实现拆解 item 3; PR #36119 实现拆解 item 1] each token row is
//     quantised ONCE: per group of g elements e = ceil(log2(max(amax,1e-10)/448)),
//     scale byte e + 127, q = RNE_e4m3(x * 2^-e) -- the power-of-two scale is
//     chosen directly, never an fp32 scale rounded afterwards;
//   * the packed row and its scales are then written to the destination row of
//     every kept (token, slot): compact row = chunk row base + chunk rank,
//     masked row = e * cap + rank (dropped past cap);
//   * src2dst is rewritten from chunk ranks to final rows, row weights copied;
//   * compact only: m_indices over the whole static bound -- expert id on valid
//     rows, -1 on padding rows and on the tail [PR #33128 _fwd_kernel_ep_scatter_1].
//   The identity mode (row t -> row t, K = 1) is the live-row quantiser of
//   PR #36119: rows >= the device live count are never touched.
//
// Design: a persistent grid (a multiple of the SM count, independent of the
// routing) walks the live tokens; each CTA owns a token at a time. A thread
// owns 16-element chunks (two 16-byte loads, one 16-byte e4m3 store per
// destination); the g/16 lanes of a group reduce the group max with xor
// shuffles on sign-cleared bf16 bit patterns. All loads of a pass are issued
// before any math, and every payload store is a full 16-byte vector, so each
// warp writes 512 contiguous bytes per destination row. Scales: for the packed
// UE8M0 layout a warp covers exactly one 32-bit word (4 groups of 128), built
// with shuffles and written once per destination.
#include "common.cuh"
#include "kernels.h"

namespace moeperm {

namespace {

constexpr int kCPT = 2;        // 16-element chunks per thread per pass
constexpr int kMaxK = 32;

template <int GSZ, int FMT>
__device__ __forceinline__ void store_scales(const ScatterArgs& p, int nslots,
                                             const int* s_dst, const int64_t* s_pk,
                                             int lane, bool active, int e,
                                             int group_base, int G) {
  constexpr int GL = GSZ / 16;     // lanes per group
  constexpr int GPW = 32 / GL;     // groups per warp
  const uint32_t byte = active ? (uint32_t)(e + 127) : 0u;
  const int gidx = group_base + lane / GL;
  const bool leader = active && (lane % GL) == 0;
  if constexpr (FMT == kFmtPacked) {
    static_assert(GSZ == 128, "packed layout is defined for groups of 128");
    const uint32_t word = __shfl_sync(0xffffffffu, byte, 0) |
                          (__shfl_sync(0xffffffffu, byte, 8) << 8) |
                          (__shfl_sync(0xffffffffu, byte, 16) << 16) |
                          (__shfl_sync(0xffffffffu, byte, 24) << 24);
    if (lane == 0 && active) {
      const int64_t wofs = (int64_t)(group_base / 4) * p.ld_s;
      uint32_t* sc = reinterpret_cast<uint32_t*>(p.scales);
      for (int k = 0; k < nslots; ++k)
        if (s_dst[k] >= 0) sc[s_pk[k] + wofs] = word;
    }
  } else if constexpr (FMT == kFmtU8) {
    constexpr int WPW = GPW / 4;   // whole 4-group words per warp
    const int q = lane % WPW;
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) word |= __shfl_sync(0xffffffffu, byte, (4 * q + j) * GL) << (8 * j);
    const bool word_ok = (p.ld_s % 4) == 0;
    uint8_t* sc = reinterpret_cast<uint8_t*>(p.scales);
    if (word_ok && lane < WPW && group_base + 4 * q + 3 < G) {
      for (int k = 0; k < nslots; ++k)
        if (s_dst[k] >= 0)
          *reinterpret_cast<uint32_t*>(sc + (int64_t)s_dst[k] * p.ld_s + group_base + 4 * q) = word;
    }
    const bool by_word = word_ok && ((gidx / 4) * 4 + 3 < G);
    if (leader && !by_word) {
      for (int k = 0; k < nslots; ++k)
        if (s_dst[k] >= 0) sc[(int64_t)s_dst[k] * p.ld_s + gidx] = (uint8_t)byte;
    }
  } else {
    if (leader) {
      float* sc = reinterpret_cast<float*>(p.scales);
      const float v = __uint_as_float((uint32_t)(e + 127) << 23);
      for (int k = 0; k < nslots; ++k)
        if (s_dst[k] >= 0) sc[(int64_t)s_dst[k] * p.ld_s + gidx] = v;
    }
  }
}

template <int GSZ, int FMT>
__global__ void __launch_bounds__(1024) quant_scatter_kernel(ScatterArgs p) {
  extern __shared__ int32_t s_geo[];  // compact: [2*L] starts, psum
  __shared__ int s_dst[2][kMaxK];
  __shared__ int64_t s_pk[2][kMaxK];
  const int tid = threadIdx.x, lane = tid & 31;
  const int bd = blockDim.x;
  const int H = p.H;
  const int nch = H / 16;
  const int G = H / GSZ;
  const int G4 = (G + 3) / 4;
  const int nslots = (p.mode == kModeIdentity) ? 1 : p.K;
  const int n_live = live_count(p.d_num_tokens, p.T, p.status,
                                p.mode == kModeIdentity && blockIdx.x == 0 && tid == 0);

  // ---- compact: m_indices over [0, bound) --------------------------------
  if (p.mode == kModeCompact && p.m_indices != nullptr) {
    const int L = p.L;
    for (int i = tid; i < L; i += bd) {
      s_geo[i] = p.starts[i];
      s_geo[L + i] = p.psum[i];
    }
    __syncthreads();
    for (int64_t r = (int64_t)blockIdx.x * bd + tid; r < p.bound; r += (int64_t)gridDim.x * bd) {
      int lo = 0, hi = L - 1;  // largest e with starts[e] <= r (starts[0] = 0)
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_geo[mid] <= r) lo = mid; else hi = mid - 1;
      }
      p.m_indices[r] = (r < s_geo[L + lo]) ? lo : -1;
    }
  }

  // ---- tokens -------------------------------------------------------------
  // The first pass of a token's x loads is issued before the barrier, so it
  // overlaps the dependent lookups (id -> rank -> chunk base) of its rows.
  int it = 0;
  for (int t = blockIdx.x; t < n_live; t += gridDim.x, ++it) {
    const int buf = it & 1;
    const uint16_t* xrow = p.x + (int64_t)t * p.ldx;
    uint4 v[kCPT][2];
    auto load_pass = [&](int c0) {
#pragma unroll
      for (int i = 0; i < kCPT; ++i) {
        const int c = c0 + i * bd + tid;
        if (c < nch) {
          v[i][0] = ld_nc_v4(xrow + c * 16);
          v[i][1] = ld_nc_v4(xrow + c * 16 + 8);
        } else {
          v[i][0] = v[i][1] = make_uint4(0, 0, 0, 0);
        }
      }
    };
    load_pass(0);
    if (tid < nslots) {
      const int k = tid;
      int row = -1;
      int64_t pk = 0;
      if (p.mode == kModeIdentity) {
        row = t;
        pk = t;
      } else {
        const int64_t a = (int64_t)t * p.K + k;
        const int e = __ldg(p.ids + a);
        if (e >= 0 && e < p.L) {
          const int lr = p.src2dst[a];
          const int b = __ldcg(p.table + (a / p.chunk) * p.L + e);
          if (p.mode == kModeCompact) {
            row = b + lr;
            if (lr < 0 || row < 0 || (int64_t)row >= p.bound) {  // never write outside the buffer
              set_status(p.status, kStBadLayout);
              row = -1;
            }
            pk = row;
          } else {
            const int j = b + lr;
            if (lr < 0 || j < 0) {
              set_status(p.status, kStBadLayout);
            } else if (j < p.cap) {
              row = e * p.cap + j;
              pk = (int64_t)e * G4 * p.ld_s + j;
            }
          }
        }
        p.src2dst[a] = row;
        if (row >= 0 && p.row_weights != nullptr) p.row_weights[row] = __ldg(p.w + a);
      }
      s_dst[buf][k] = row;
      s_pk[buf][k] = pk;
    }
    __syncthreads();

    for (int c0 = 0; c0 < nch; c0 += kCPT * bd) {
      if (c0 > 0) load_pass(c0);
#pragma unroll
      for (int i = 0; i < kCPT; ++i) {
        const int c = c0 + i * bd + tid;
        const bool active = c < nch;
        uint32_t m = amax16_bf16(v[i][0], v[i][1]);
#pragma unroll
        for (int off = 1; off < GSZ / 16; off <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
        const int e = group_exponent(__uint_as_float(m << 16));
        const float inv = exp2_neg(e);
        const uint2 q0 = quant8(v[i][0], inv), q1 = quant8(v[i][1], inv);
        const uint4 q = make_uint4(q0.x, q0.y, q1.x, q1.y);
        if (active) {
          for (int k = 0; k < nslots; ++k) {
            const int row = s_dst[buf][k];
            if (row >= 0) st_v4(p.xq + (int64_t)row * H + c * 16, q);
          }
        }
        const int cw = c0 + i * bd + (tid & ~31);  // first chunk of this warp
        if (cw < nch)
          store_scales<GSZ, FMT>(p, nslots, s_dst[buf], s_pk[buf], lane, active, e,
                                 cw * 16 / GSZ, G);
      }
    }
  }
}

template <int GSZ, int FMT>
cudaError_t launch_one(const ScatterArgs& a, int num_sms, cudaStream_t s) {
  const int nch = a.H / 16;
  int bd = (nch + kCPT - 1) / kCPT;
  bd = (bd + 31) / 32 * 32;
  if (bd > 1024) bd = 1024;
  const size_t smem = (a.mode == kModeCompact) ? (size_t)2 * a.L * sizeof(int32_t) : 0;
  int per_sm = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, quant_scatter_kernel<GSZ, FMT>, bd, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  int64_t grid = (int64_t)num_sms * per_sm;
  if (grid > a.T) grid = a.T;
  if (grid < 1) grid = 1;
  quant_scatter_kernel<GSZ, FMT><<<(unsigned)grid, bd, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_scatter(const ScatterArgs& a, int g, int fmt, int num_sms,
                                 cudaStream_t s) {
  if (g == 128) {
    if (fmt == kFmtPacked) return launch_one<128, kFmtPacked>(a, num_sms, s);
    if (fmt == kFmtU8) return launch_one<128, kFmtU8>(a, num_sms, s);
    return launch_one<128, kFmtF32>(a, num_sms, s);
  }
  return launch_one<32, kFmtU8>(a, num_sms, s);
}

}  // namespace moeperm
