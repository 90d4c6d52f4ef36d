// common.cuh -- device helpers shared by the sm_103a kernels of libmoeperm.
//
// Number formats:
//   bf16 values travel as raw 16-bit words, two per 32-bit register (element 0
//   in the low half), so the absolute maximum of a group is an unsigned 16-bit
//   max of sign-cleared words (for finite values the bit order is the value
//   order) -- no float compare is needed.
//   e4m3 (OCP E4M3) conversions use the hardware pair converts
//   cvt.rn.satfinite.e4m3x2.f32 (round to nearest even, saturating to +-448)
//   and cvt.rn.f16x2.e4m3x2 (exact widening).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moeperm {

// Device status bits (same values as MOE_STATUS_* in the public header).
constexpr int kStOverflow = 0x1;
constexpr int kStLiveOverflow = 0x2;
constexpr int kStBadLayout = 0x4;

// Scale layouts (same values as moe_scale_fmt_t).
constexpr int kFmtU8 = 0;
constexpr int kFmtPacked = 1;
constexpr int kFmtF32Pow2 = 2;
constexpr int kFmtF32 = 3;   // plain fp32 group scale amax / 448
constexpr int kFmtMX = 4;    // OCP MX E8M0 (floor exponent, saturating elements)

// Route-plan modes.
constexpr int kModeCompact = 0;
constexpr int kModeMasked = 1;
constexpr int kModeIdentity = 2;  // row t -> row t (live-row quantisation)

__device__ __forceinline__ void set_status(int32_t* status, int bits) {
  if (status != nullptr) atomicOr(status, bits);
}

// Live-row count read on the device: min(*d_n, cap) (and >= 0); flags n > cap.
__device__ __forceinline__ int live_count(const int32_t* d_n, int cap, int32_t* status,
                                          bool report) {
  if (d_n == nullptr) return cap;
  int n = __ldg(d_n);
  if (n > cap) {
    if (report) set_status(status, kStLiveOverflow);
    n = cap;
  }
  return n < 0 ? 0 : n;
}

// ---------------------------------------------------------------------------
// bf16 helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// max |x| over the 16 bf16 values of two 16-byte vectors, as a bf16 bit pattern
// in the low half of the result.
__device__ __forceinline__ uint32_t amax16_bf16(const uint4& a, const uint4& b) {
  const uint32_t m = 0x7FFF7FFFu;
  uint32_t r = __vmaxu2(__vmaxu2(a.x & m, a.y & m), __vmaxu2(a.z & m, a.w & m));
  r = __vmaxu2(r, __vmaxu2(__vmaxu2(b.x & m, b.y & m), __vmaxu2(b.z & m, b.w & m)));
  return max(r & 0xFFFFu, r >> 16);
}

// fp32 -> bf16 (round to nearest even) pair pack, element `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------------------
// e4m3 helpers
// ---------------------------------------------------------------------------

// Two floats -> two e4m3 bytes (RNE, satfinite); `lo` lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

// Two e4m3 bytes (low byte first) -> two floats, exactly (e4m3 -> f16 -> f32).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_bytes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two_bytes));
  float2 f;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(f.x), "=f"(f.y)
      : "r"(h2));
  return f;
}

// Power-of-two group exponent: the smallest integer e with 448 * 2^e >= a,
// a = max(amax, 1e-10). With a = 1.m * 2^E (a normal float): 448 = 1.75 * 2^8,
// so e = E - 8 when 1.m <= 1.75 and E - 7 otherwise. Exact, no division.
__device__ __forceinline__ int group_exponent(float amax) {
  const float a = fmaxf(amax, 1e-10f);
  const uint32_t bits = __float_as_uint(a);
  const int E = (int)(bits >> 23) - 127;
  const uint32_t mant = bits & 0x7FFFFFu;
  int e = E - 8 + (mant > 0x600000u ? 1 : 0);
  return min(max(e, -127), 127);
}

// OCP MX shared exponent for E4M3 elements: floor(log2(amax)) - 8, at least
// -127 (zero and tiny amax give -127). For a normal float the floor of log2 is
// its unbiased exponent field.
__device__ __forceinline__ int mx_exponent(float amax) {
  const int Eb = (int)(__float_as_uint(amax) >> 23) & 0xFF;
  return max(Eb - 135, -127);
}

// 2^-e as a float (e in [-127, 126]).
__device__ __forceinline__ float exp2_neg(int e) {
  return __uint_as_float((uint32_t)(127 - e) << 23);  // e = -127 gives 2^127
}

// Quantise 8 bf16 values by an fp32 scale s: RNE_e4m3(fl32(x / s)), one IEEE
// fp32 division per element.
__device__ __forceinline__ uint2 quant8_div(const uint4& v, float s) {
  uint2 r;
  r.x = cvt_e4m3x2(__fdiv_rn(bf16_lo(v.x), s), __fdiv_rn(bf16_hi(v.x), s)) |
        (cvt_e4m3x2(__fdiv_rn(bf16_lo(v.y), s), __fdiv_rn(bf16_hi(v.y), s)) << 16);
  r.y = cvt_e4m3x2(__fdiv_rn(bf16_lo(v.z), s), __fdiv_rn(bf16_hi(v.z), s)) |
        (cvt_e4m3x2(__fdiv_rn(bf16_lo(v.w), s), __fdiv_rn(bf16_hi(v.w), s)) << 16);
  return r;
}

// Quantise 8 bf16 values (one 16-byte vector) by 2^-e into 8 e4m3 bytes.
__device__ __forceinline__ uint2 quant8(const uint4& v, float inv) {
  uint2 r;
  r.x = cvt_e4m3x2(__fmul_rn(bf16_lo(v.x), inv), __fmul_rn(bf16_hi(v.x), inv)) |
        (cvt_e4m3x2(__fmul_rn(bf16_lo(v.y), inv), __fmul_rn(bf16_hi(v.y), inv)) << 16);
  r.y = cvt_e4m3x2(__fmul_rn(bf16_lo(v.z), inv), __fmul_rn(bf16_hi(v.z), inv)) |
        (cvt_e4m3x2(__fmul_rn(bf16_lo(v.w), inv), __fmul_rn(bf16_hi(v.w), inv)) << 16);
  return r;
}

// ---------------------------------------------------------------------------
// Memory helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_v4(void* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Programmatic dependent launch: a primary grid lets its dependent be
// scheduled early; the dependent waits for the primary's completion (and the
// visibility of its memory) before touching its results. Both are no-ops for
// launches without the programmatic attribute.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Bulk (TMA) copy of `bytes` from shared memory to global memory, tracked in
// the issuing thread's bulk groups, with an L2 cache policy (from
// createpolicy) on the written lines. Both addresses 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_store_s2g_hint(void* gdst, uint32_t ssrc, uint32_t bytes,
                                                    uint64_t policy) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
               ::"l"(gdst), "r"(ssrc), "r"(bytes), "l"(policy)
               : "memory");
}
// Bulk (TMA) prefetch of `bytes` of global memory into L2 with an L2 cache
// policy (16-byte aligned address, bytes a multiple of 16); nothing waits for it.
__device__ __forceinline__ void bulk_prefetch_l2_hint(const void* g, uint32_t bytes, uint64_t policy) {
  asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;"
               ::"l"(g), "r"(bytes), "l"(policy)
               : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Asynchronous 16-byte copy global -> shared (both addresses 16-byte
// aligned), completed by cp_async_wait_all() in the issuing thread.
__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
               ::"r"((uint32_t)__cvta_generic_to_shared(sdst)), "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to bulk copies.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Host-side launch queries, cached per device (they cost more host time than
// a launch; api.cu): resident CTAs per SM for (kernel, threads, dynamic shared
// memory), and the opt-in that lets a kernel take `dyn` bytes of dynamic shared
// memory. Without the opt-in a CTA is limited to 48 KiB of dynamic plus static
// shared memory; the static arrays of these kernels stay under 1 KiB.
cudaError_t occupancy_cached(const void* kernel, int threads, size_t smem, int* per_sm);
// Unique id of the CUDA context current on this thread (0 when none is).
cudaError_t current_context_id(unsigned long long* id);
cudaError_t opt_in_smem_cached(const void* kernel, size_t dyn);
cudaError_t device_attr_cached(cudaDeviceAttr attr, int* value);
template <typename Kern>
inline cudaError_t opt_in_smem(Kern kernel, size_t dyn) {
  if (dyn + 1024 <= 48 * 1024) return cudaSuccess;
  return opt_in_smem_cached(reinterpret_cast<const void*>(kernel), dyn);
}
template <typename Kern>
inline cudaError_t occupancy(Kern kernel, int threads, size_t smem, int* per_sm) {
  return occupancy_cached(reinterpret_cast<const void*>(kernel), threads, smem, per_sm);
}

__device__ __forceinline__ int64_t align_up64(int64_t c, int64_t b) { return (c + b - 1) / b * b; }

// Segment starts of a layout whose segments are padded to multiples of b, in
// expert order: st[e] = sum over e' < e of align(min(cnt[e'], clamp), b), for
// e < L (PR #33128 compact starts; PR #29525 _build_layout starts). One CTA:
// thread i owns a contiguous run of experts; a warp scan joins the runs of a
// warp and warp 0 scans the warp totals. Returns the total in every thread.
// Every thread of the CTA must call it (blockDim.x a multiple of 32); it
// begins reading cnt and ends with a barrier. s_wsum: at least 33 ints of
// shared memory.
__device__ __forceinline__ int aligned_starts(const int32_t* cnt, int32_t* st, int L, int b,
                                              int clamp, int32_t* s_wsum) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, bd = blockDim.x;
  const int nwarps = bd >> 5;
  const int per = (L + bd - 1) / bd;
  const int lo = min(tid * per, L), hi = min(lo + per, L);
  int local = 0;
  for (int e = lo; e < hi; ++e) local += (min(cnt[e], clamp) + b - 1) / b * b;
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int nb = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += nb;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the warp totals; the grand total in s_wsum[32]
    const int v = lane < nwarps ? s_wsum[lane] : 0;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int nb = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += nb;
    }
    __syncwarp();
    if (lane < nwarps) s_wsum[lane] = x - v;
    if (lane == 31) s_wsum[32] = x;
  }
  __syncthreads();
  int run = s_wsum[warp] + incl - local;
  for (int e = lo; e < hi; ++e) {
    st[e] = run;
    run += (min(cnt[e], clamp) + b - 1) / b * b;
  }
  const int total = s_wsum[32];
  __syncthreads();
  return total;
}

}  // namespace moeperm
