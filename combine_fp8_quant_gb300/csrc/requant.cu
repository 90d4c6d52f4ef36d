// requant.cu -- per-token -> per-tensor FP8 requantisation
// (PR #14162 实现拆解 items 1-2, fp8_per_token_to_per_tensor_quant; 风险与影响
// item 3: the original kernel assumes plain fp32 per-token scales and does not
// handle e8m0 ones).
//
//   s[t]  = the token's scale: fp32, or 2^(b - 127) for an e8m0 byte b
//   S     = max_t s[t]                                   (max-scale mode)
//         = fl32(max_t fl32(s[t] * amax_t) / 448)        (amax mode, amax_t =
//           max_h |decode(q[t,h])|: the largest dequantised value maps to 448)
//   S = 1 if T = 0 or the maximum is 0 (then r = 0)
//   q_out[t, h] = RNE_e4m3( fl32( decode(q[t, h]) * fl32(s[t] / S) ) )
//
// Design: the max-scale mode is one launch. Rows go one per warp; each warp
// first issues the loads of the first pass of its first row (8 x 16 bytes per
// lane), then its CTA reduces the T scales (float4 / byte loads, L2-resident) while
// they are in flight, and the warp converts and stores: 16 e4m3 bytes per lane
// per vector, widened exactly with cvt.rn.f16x2.e4m3x2, scaled in fp32,
// narrowed with cvt.rn.satfinite.e4m3x2.f32. The amax mode adds a first launch
// that writes fl32(s[t] * amax_t) per row to the workspace (the row maximum is
// a byte-wise __vmaxu4 of sign-cleared codes: for finite e4m3 the code order is
// the magnitude order); the second launch reduces that array instead of the
// scales. q (tens of MB) is still in L2 for the second read. The sources
// hard-code a 1024-wide hidden block; here a CTA covers the whole row.
#include "common.cuh"
#include "kernels.h"

namespace moeperm {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t requant4(uint32_t w, float r) {
  const float2 a = e4m3x2_to_float2(w & 0xFFFFu);
  const float2 b = e4m3x2_to_float2(w >> 16);
  return cvt_e4m3x2(__fmul_rn(a.x, r), __fmul_rn(a.y, r)) |
         (cvt_e4m3x2(__fmul_rn(b.x, r), __fmul_rn(b.y, r)) << 16);
}

// 2^(b - 127) for an e8m0 byte (b = 0 is the fp32 subnormal 2^-127).
__device__ __forceinline__ float e8m0_value(uint32_t b) {
  return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

template <int SFMT>
__device__ __forceinline__ float token_scale(const RequantArgs& p, int t) {
  if constexpr (SFMT == kTokScaleF32) return __ldg(reinterpret_cast<const float*>(p.s_tok) + t);
  else return e8m0_value(__ldg(reinterpret_cast<const uint8_t*>(p.s_tok) + t));
}

__device__ __forceinline__ float block_max(float m, float* s_red) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) s_red[warp] = m;
  __syncthreads();
  float r = 0.0f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) r = fmaxf(r, s_red[w]);
  return r;
}

// max over n non-negative floats (float4 loads when aligned)
__device__ __forceinline__ float reduce_floats(const float* a, int n, float* s_red) {
  const int tid = threadIdx.x;
  float m = 0.0f;
  if ((reinterpret_cast<uintptr_t>(a) & 15u) == 0) {
    const float4* a4 = reinterpret_cast<const float4*>(a);
    for (int i = tid; i < n / 4; i += kThreads) {
      const float4 v = __ldcg(a4 + i);
      m = fmaxf(fmaxf(m, fmaxf(v.x, v.y)), fmaxf(v.z, v.w));
    }
    for (int t = 4 * (n / 4) + tid; t < n; t += kThreads) m = fmaxf(m, __ldcg(a + t));
  } else {
    for (int t = tid; t < n; t += kThreads) m = fmaxf(m, __ldcg(a + t));
  }
  return block_max(m, s_red);
}

// max over n e8m0 bytes, as the scale value
__device__ __forceinline__ float reduce_e8m0(const uint8_t* b, int n, float* s_red) {
  uint32_t m = 0;
  for (int t = threadIdx.x; t < n; t += kThreads) m = max(m, (uint32_t)__ldg(b + t));
  return block_max(m ? e8m0_value(m) : 0.0f, s_red);
}

// Rows are processed one per warp: a lane issues kPass 16-byte loads of its
// row before the first conversion of each pass (8: a 7 KB row in two passes,
// within 80 registers so that 3 CTAs fit per SM).
constexpr int kPass = 8;
constexpr int kMinBlocks = 3;  // CTAs per SM the rescale kernel is compiled for (80 registers)

// amax mode, launch 1: ws[t] = fl32(s[t] * max_h |decode(q[t, h])|)
template <int SFMT>
__global__ void __launch_bounds__(kThreads) requant_rowmax_kernel(RequantArgs p) {
  const int lane = threadIdx.x & 31;
  const int gwarp = (int)((blockIdx.x * kThreads + threadIdx.x) >> 5);
  const int nwarps = (int)((gridDim.x * kThreads) >> 5);
  const int nch = p.H / 16;
  for (int t = gwarp; t < p.T; t += nwarps) {
    const uint8_t* src = p.q + (int64_t)t * p.ldq;
    uint32_t m = 0;
    for (int c0 = 0; c0 < nch; c0 += 32 * kPass) {
      uint4 v[kPass];
#pragma unroll
      for (int j = 0; j < kPass; ++j) {
        const int c = c0 + j * 32 + lane;
        v[j] = (c < nch) ? ld_nc_v4(src + (int64_t)c * 16) : make_uint4(0, 0, 0, 0);
      }
      const uint32_t k = 0x7F7F7F7Fu;
#pragma unroll
      for (int j = 0; j < kPass; ++j)
        m = __vmaxu4(m, __vmaxu4(__vmaxu4(v[j].x & k, v[j].y & k), __vmaxu4(v[j].z & k, v[j].w & k)));
    }
    m = max(max(m & 0xFFu, (m >> 8) & 0xFFu), max((m >> 16) & 0xFFu, m >> 24));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) p.ws[t] = __fmul_rn(token_scale<SFMT>(p, t), e4m3x2_to_float2(m).x);
  }
}

template <int SFMT, int MODE>
__global__ void __launch_bounds__(kThreads, kMinBlocks) requant_kernel(RequantArgs p) {
  __shared__ float s_red[kThreads / 32];
  const int lane = threadIdx.x & 31, tid = threadIdx.x;
  const int gwarp = (int)((blockIdx.x * kThreads + threadIdx.x) >> 5);
  const int nwarps = (int)((gridDim.x * kThreads) >> 5);
  const int nch = p.H / 16;
  // Each warp's first row is loaded before the scale reduction so the two
  // latencies overlap.
  int t = gwarp;
  uint4 v[kPass];
#pragma unroll
  for (int j = 0; j < kPass; ++j) {
    const int c = j * 32 + lane;
    v[j] = (t < p.T && c < nch) ? ld_nc_v4(p.q + (int64_t)t * p.ldq + (int64_t)c * 16)
                                : make_uint4(0, 0, 0, 0);
  }
  float S;
  if constexpr (MODE == kRequantAmax) {
    S = __fdiv_rn(reduce_floats(p.ws, p.T, s_red), 448.0f);
  } else if constexpr (SFMT == kTokScaleF32) {
    S = reduce_floats(reinterpret_cast<const float*>(p.s_tok), p.T, s_red);
  } else {
    S = reduce_e8m0(reinterpret_cast<const uint8_t*>(p.s_tok), p.T, s_red);
  }
  if (blockIdx.x == 0 && tid == 0) *p.scale_out = (S > 0.0f) ? S : 1.0f;

  bool preloaded = true;
  for (; t < p.T; t += nwarps) {
    const float r = (S > 0.0f) ? __fdiv_rn(token_scale<SFMT>(p, t), S) : 0.0f;
    const uint8_t* src = p.q + (int64_t)t * p.ldq;
    uint8_t* dst = p.q_out + (int64_t)t * p.H;
    for (int c0 = 0; c0 < nch; c0 += 32 * kPass) {
      if (!preloaded) {
#pragma unroll
        for (int j = 0; j < kPass; ++j) {
          const int c = c0 + j * 32 + lane;
          v[j] = (c < nch) ? ld_nc_v4(src + (int64_t)c * 16) : make_uint4(0, 0, 0, 0);
        }
      }
      preloaded = false;
#pragma unroll
      for (int j = 0; j < kPass; ++j) {
        const int c = c0 + j * 32 + lane;
        if (c < nch)
          st_v4(dst + (int64_t)c * 16, make_uint4(requant4(v[j].x, r), requant4(v[j].y, r),
                                                  requant4(v[j].z, r), requant4(v[j].w, r)));
      }
    }
  }
}

template <typename Kern>
cudaError_t launch_rows(Kern k, const RequantArgs& a, int num_sms, cudaStream_t s) {
  int per_sm = 0;
  cudaError_t err = occupancy(k, kThreads, 0, &per_sm);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  int64_t grid = (int64_t)num_sms * per_sm;
  const int64_t need = ((int64_t)a.T + kThreads / 32 - 1) / (kThreads / 32);  // one warp per row
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  k<<<(unsigned)grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <int SFMT>
cudaError_t launch_fmt(const RequantArgs& a, int num_sms, cudaStream_t s) {
  if (a.mode == kRequantAmax) {
    cudaError_t err = launch_rows(requant_rowmax_kernel<SFMT>, a, num_sms, s);
    if (err != cudaSuccess) return err;
    return launch_rows(requant_kernel<SFMT, kRequantAmax>, a, num_sms, s);
  }
  return launch_rows(requant_kernel<SFMT, kRequantMaxScale>, a, num_sms, s);
}

}  // namespace

cudaError_t launch_requant(const RequantArgs& a, int num_sms, cudaStream_t s) {
  return a.s_fmt == kTokScaleF32 ? launch_fmt<kTokScaleF32>(a, num_sms, s)
                                 : launch_fmt<kTokScaleE8M0>(a, num_sms, s);
}

}  // namespace moeperm
