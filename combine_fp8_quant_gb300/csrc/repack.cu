// repack.cu -- expanded (128-aligned psum) layout <-> masked per-expert slab
// (PR #29525 实现拆解 item 3: expand_to_masked_slab / masked_slab_to_expand /
// ep_expand_init_m_indices_from_psum; 关键源码片段 _build_layout).
//
//   expert e owns expanded rows [align(psum[e-1]), psum[e]), psum[-1] = 0
//   to_slab:   slab[e, j] = exp[start_e + j], masked_m[e] = min(count_e, cap)
//   from_slab: exp[start_e + j] = slab[e, j]   (optionally bf16_RNE(w_r * v))
//              m_indices[r] = e on real rows, -1 elsewhere
//   count_e > cap -> MOE_STATUS_OVERFLOW, rows past cap untouched (fail fast);
//   psum inconsistent with the R expanded rows -> MOE_STATUS_BAD_LAYOUT.
//
// Design: a fixed worker pool (grid = SMs x resident CTAs, capped by R) walks
// the R expanded rows, one row per warp, so the launch never depends on the
// routing; a warp finds its row's expert by binary search over the segment
// starts held in shared memory and copies the row with 16-byte vectors, 8 per
// lane issued before the first store of each pass (a 7 KB e4m3 row in two
// passes), at 64 registers so that 3+ CTAs fit per SM. Scales follow each side's own layout (stride
// aware): row-major bytes / floats, or column-major packed UE8M0 words with
// one block per expert on the slab side; pad bytes of the last packed word are
// cleared.
#include "common.cuh"
#include "kernels.h"

namespace moeperm {

namespace {

constexpr int kThreads = 256;
constexpr int kPass = 8;       // 16-byte chunks per lane in flight (8 with 3 CTAs/SM measured fastest)
constexpr int kMinBlocks = 3;  // CTAs per SM the kernel is compiled for (64 registers)

__global__ void __launch_bounds__(kThreads, kMinBlocks) repack_kernel(RepackArgs p) {
  extern __shared__ int32_t sm[];
  int32_t* s_start = sm;
  int32_t* s_psum = sm + p.L;
  const int tid = threadIdx.x, lane = tid & 31;
  const int gwarp = (int)((blockIdx.x * kThreads + threadIdx.x) >> 5);
  const int nwarps = (int)((gridDim.x * kThreads) >> 5);
  const int L = p.L;
  for (int e = tid; e < L; e += kThreads) {
    const int pe = __ldg(p.psum + e);
    s_psum[e] = pe;
    s_start[e] = (e == 0) ? 0 : (int)align_up64(__ldg(p.psum + e - 1), p.align);
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    int bits = 0;
    for (int e = tid; e < L; e += kThreads) {
      const int cnt = s_psum[e] - s_start[e];
      if (cnt < 0 || (int64_t)s_psum[e] > p.R) bits |= kStBadLayout;
      if (cnt > p.cap) bits |= kStOverflow;
      if (p.to_slab && p.masked_m != nullptr) p.masked_m[e] = min(max(cnt, 0), p.cap);
    }
    if (bits) set_status(p.status, bits);
  }

  const int64_t rowbytes = (int64_t)p.H * p.elem_bytes;
  const int nch = (int)(rowbytes / 16);
  const int G = p.G, G4 = (G + 3) / 4;
  const bool scales = p.src_scales != nullptr && p.dst_scales != nullptr && G > 0;
  const bool weighted = !p.to_slab && p.row_weights != nullptr && p.elem_bytes == 2;
  for (int64_t r = gwarp; r < p.R; r += nwarps) {
    int lo = 0, hi = L - 1;  // largest e with start[e] <= r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_start[mid] <= r) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const bool real = r < s_psum[e] && r >= s_start[e];
    if (!p.to_slab && p.m_indices != nullptr && lane == 0) p.m_indices[r] = real ? e : -1;
    const int64_t j = r - s_start[e];
    if (!real || j >= p.cap) continue;
    const int64_t srow = (int64_t)e * p.cap + j;  // slab row
    const uint8_t* src = p.src + (p.to_slab ? r : srow) * rowbytes;
    uint8_t* dst = p.dst + (p.to_slab ? srow : r) * rowbytes;
    const float wr = weighted ? __ldg(p.row_weights + r) : 1.0f;
    for (int c0 = 0; c0 < nch; c0 += 32 * kPass) {
      uint4 v[kPass];
#pragma unroll
      for (int i = 0; i < kPass; ++i) {
        const int c = c0 + i * 32 + lane;
        v[i] = (c < nch) ? ld_nc_v4(src + (int64_t)c * 16) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < kPass; ++i) {
        const int c = c0 + i * 32 + lane;
        if (c < nch) {
          uint4 o = v[i];
          if (weighted) {
            o.x = pack_bf16x2(__fmul_rn(wr, bf16_lo(v[i].x)), __fmul_rn(wr, bf16_hi(v[i].x)));
            o.y = pack_bf16x2(__fmul_rn(wr, bf16_lo(v[i].y)), __fmul_rn(wr, bf16_hi(v[i].y)));
            o.z = pack_bf16x2(__fmul_rn(wr, bf16_lo(v[i].z)), __fmul_rn(wr, bf16_hi(v[i].z)));
            o.w = pack_bf16x2(__fmul_rn(wr, bf16_lo(v[i].w)), __fmul_rn(wr, bf16_hi(v[i].w)));
          }
          st_v4(dst + (int64_t)c * 16, o);
        }
      }
    }
    if (scales) {
      if (p.fmt == kFmtPacked) {
        const uint32_t* s32 = reinterpret_cast<const uint32_t*>(p.src_scales);
        uint32_t* d32 = reinterpret_cast<uint32_t*>(p.dst_scales);
        for (int w = lane; w < G4; w += 32) {
          const int64_t xw = (int64_t)w * (p.to_slab ? p.ld_src_s : p.ld_dst_s) + r;
          const int64_t sw = (int64_t)e * G4 * (p.to_slab ? p.ld_dst_s : p.ld_src_s) +
                             (int64_t)w * (p.to_slab ? p.ld_dst_s : p.ld_src_s) + j;
          uint32_t word = __ldg(s32 + (p.to_slab ? xw : sw));
          if (w == G4 - 1 && (G & 3)) word &= (1u << (8 * (G & 3))) - 1u;
          d32[p.to_slab ? sw : xw] = word;
        }
      } else if (p.fmt == kFmtU8 || p.fmt == kFmtMX) {
        const uint8_t* s8 = reinterpret_cast<const uint8_t*>(p.src_scales);
        uint8_t* d8 = reinterpret_cast<uint8_t*>(p.dst_scales);
        const int64_t so = (p.to_slab ? r : srow) * p.ld_src_s;
        const int64_t dof = (p.to_slab ? srow : r) * p.ld_dst_s;
        for (int gi = lane; gi < G; gi += 32) d8[dof + gi] = __ldg(s8 + so + gi);
      } else {
        const float* sf = reinterpret_cast<const float*>(p.src_scales);
        float* df = reinterpret_cast<float*>(p.dst_scales);
        const int64_t so = (p.to_slab ? r : srow) * p.ld_src_s;
        const int64_t dof = (p.to_slab ? srow : r) * p.ld_dst_s;
        for (int gi = lane; gi < G; gi += 32) df[dof + gi] = __ldg(sf + so + gi);
      }
    }
  }
}

}  // namespace

cudaError_t launch_repack(const RepackArgs& a, int num_sms, cudaStream_t s) {
  const size_t smem = (size_t)2 * a.L * sizeof(int32_t);
  int per_sm = 0;
  cudaError_t err = occupancy(repack_kernel, kThreads, smem, &per_sm);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  int64_t grid = (int64_t)num_sms * per_sm;
  const int64_t need = (a.R + kThreads / 32 - 1) / (kThreads / 32);  // one warp per expanded row
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  repack_kernel<<<(unsigned)grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moeperm
