// quant_scatter.cu -- FP8 group quantisation fused with the dispatch scatter
// (second dispatch launch), and the live-row quantiser.
//
// What it computes:
//   * [PR #33128 实现拆解 item 3; PR #36119 实现拆解 item 1] each token row is
//     quantised ONCE: per group of g elements e = ceil(log2(max(amax,1e-10)/448)),
//     scale byte e + 127, q = RNE_e4m3(x * 2^-e) -- the power-of-two scale is
//     chosen directly, never an fp32 scale rounded afterwards;
//   * the layout from the route plan's chunk histograms: per expert the count,
//     compact start[e] = sum_{e'<e} align(count[e'], block_e), psum, total,
//     masked_m = min(count, cap) and the overflow flag;
//   * the row of every kept (token, slot): compact start[e] + (slots of e in
//     earlier chunks) + chunk rank; masked e*cap + rank, dropped past cap;
//   * the quantised row and its scales written to each of the token's rows;
//     src2dst rewritten from chunk ranks to rows; row weights copied;
//   * compact only: m_indices over the whole static bound -- expert id on valid
//     rows, -1 on padding rows and on the tail [PR #33128 _fwd_kernel_ep_scatter_1].
//   The identity mode (row t -> row t, one slot) is the live-row quantiser of
//   PR #36119: rows >= the device live count are never touched. With a single
//   destination per row it runs barrier-free with direct 16-byte stores, and
//   so does a dispatch whose tokens keep few slots (K * L / E <= 3, decided on
//   the host from scalars alone): there the per-token barrier of the staged
//   path costs more than the bulk copies save. For rows of two chunks per
//   thread that direct mode takes its tokens from a counter instead of a
//   fixed strided set, so that CTAs end together (see the loop below).
//
// Design: a persistent grid (SMs x resident CTAs, independent of the routing)
// walks the live tokens, t = blockIdx.x + i * gridDim.x -- in the staged mode
// with enough tokens per CTA only the first part of them, the rest coming from
// a token counter once a CTA's own tokens are done (SMs differ in how fast
// they drain their stores, so a fixed split leaves the slowest SMs working
// alone at the end; the tail loop below). One thread owns two
// 16-element chunks of a row (two 16-byte loads each), so a single pass
// covers H <= 32768; rows up to 5120 elements take one chunk per thread
// instead, so that their CTAs keep enough threads (and loads) in flight.
//   Prologue: this grid is already resident while the route plan runs
//   (programmatic dependent launch), so before waiting for it a CTA reads and
//   quantises its first few tokens into their staging buffers (inputs only:
//   their rows are not known yet) and loads the expert ids of its first slots
//   (one per thread). After the wait it bulk-prefetches the rows of its next
//   few tokens into L2 and loads the chunk table (<= 64 KiB)
//   into shared memory, scans it, and resolves the rows of all of its own
//   slots at once. The route plan therefore needs no serial "last block" and
//   no fence. Tokens with no kept slot (all their experts remote) are dropped
//   from the walk. The m_indices fill runs after the token loop, while the
//   last bulk copies drain.
//   Token loop: the next token's loads are issued before the current token is
//   processed; the g/16 lanes of a group reduce the group max with xor
//   shuffles on sign-cleared bf16 bit patterns; the exponent comes from the
//   float's bit fields; conversion is cvt.rn.satfinite.e4m3x2.f32. The e4m3
//   row is staged in shared memory and thread 0 writes it to each of the
//   token's destination rows with one bulk (TMA) copy per row, so the payload
//   -- 80% of the kernel's traffic -- leaves the SM as large asynchronous
//   transfers (with an evict_first L2 policy: nothing reads them back here)
//   instead of per-thread stores. Scales are small direct stores:
//   for the packed UE8M0 layout exactly one 32-bit word per warp (4 groups of
//   128) per destination, the K destinations written from K lanes at once
//   (scales.cuh).
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "scales.cuh"

namespace moeperm {

namespace {

// Largest staging ring (rows in flight to the bulk-copy engine) and number of
// tokens quantised before the wait on the route plan; the launch lowers both
// when shared memory is short (large H with a large chunk table). Measured on
// the prefill workload: 4 buffers / 2 early tokens 102.7-103.0 us, 3 / 2
// 105.6, 5 / 2 106.7 (5 buffers drop to 3 CTAs per SM), 6 / 4 104.2; with the
// post-wait prefetch 4 / 2 105.1-105.6, 4 / 1, 4 / 3 and 5 / 2 within 0.4 us,
// 3 / 2 109.6-110.3; with the counter tail 4 / 1 102.4-102.6 against
// 100.8-101.1.
constexpr int kStages = 4;
constexpr int kPre = 2;
// Rows up to this width take one 16-element chunk per thread (twice the
// threads per CTA); wider rows take two (H = 2048: 59 against 67 us; H = 7168:
// 105 against 109 us the other way round).
constexpr int kCpt1MaxH = 5120;
static_assert(kCpt1MaxH <= 16384, "one chunk per thread covers at most 1024 x 16 elements");
// Tokens after the early-staged ones whose x rows are bulk-prefetched into L2
// (evict_last) right after the wait on the route plan, so that the reads run
// while the CTA builds the layout instead of delaying the wait (staged path;
// measured against 2 tokens before the wait: dispatch 105.1-105.8 -> 104.0-104.4 us,
// step 266.9-267.7 -> 265.6-266.1 us; 2 / 4 / 8 / 10 / 14 after the wait:
// 104.7 / 104.6 / 105.1 / 104.8 / 108.1 us). With the counter tail, 3 / 6 / 9 /
// 12: prefill 103.5-104.2 / 100.6-101.3 / 99.9-100.7 / 100.6; the other
// shape-sweep shapes 0.4-1.7 us faster with 9 than with 6, 12 within 0.4 of 9.
constexpr int kPrefetchAfterWait = 9;
// Staged mode, tail from the token counter: with at least kTailMinTokens
// tokens per CTA, a CTA's last tokens' worth are not assigned statically but
// taken from a counter once its static tokens are done, so that CTAs on
// faster SMs take more of them (per-CTA loop ends on the prefill spread from
// 83 to 99 us, SM by SM). How many (tail_tokens below) depends on the work
// per token, f = K * L / E kept slots expected per row: every slot kept
// (f >= 7.5, wide rows) takes kTailPct% of the CTA's tokens; fewer kept slots
// take one token per kTailDiv (one fewer below f = 5.5); narrow rows one.
// Dispatch us, H = 7168, tail tokens per CTA none / 1 / 2 / 4 / 45%:
//   T = 8192 (17 per CTA): f = 8 105.3 / 103.0 / 102.5 / 102.1 / 101.3;
//     f = 7 98.3 / 93.1 / 92.8 / 92.5 / 94.3; f = 6 86.9 / 85.3 / 85.2 /
//     87.2 / 89.6; f = 5 77.7 / 79.3 / 78.5 / 79.6 / 79.0; f = 4 67.8 /
//     70.2 / 71.6 / 73.2 / 73.6;
//   T = 16384, f = 4: 128.8 / 126.1 / 125.9 / 126.7 / 131.4;
//   T = 32768 (71 per CTA): f = 4 247.7 / 243.0 / 240.1 / 239.5 / 249.2;
//     f = 6 331.2 / 325.5 / 322.0 / 314.8 / 322.1; f = 8 391.5 / 389.0 /
//     387.1 / 382.4 (5) / 373.2 (32);
//   T = 4096 (8 per CTA), f = 8: 57.8 / 58.2 / 59.9. Tokens per CTA 12 / 13 /
//   16, f = 8, no tail against the 45% tail: 72.3-72.6 / 80.9-81.0 / 94.3-94.6
//   against 73.2-73.6 / 78.7-79.4 / 90.0-90.1.
//   Narrow rows (one chunk per thread), none / 1 / 3: H = 4096 66.3 / 62.4 /
//   64.0, H = 5120 64.9 / 64.5 / 65.6, H = 2048 55.6 / 53.8 / 55.7.
constexpr int kTailMinTokens = 13;
constexpr int kTailPct = 45;
constexpr int kTailDiv = 17;
// Direct stores instead of staging when the expected kept slots per token,
// K * L / E (uniform routing), are at most this many (staged -> direct at
// T = 8192, H = 7168: f = 1 47.1 -> 43.0 us, f = 3 62.9 -> 61.5, f = 4
// 69.1 -> 72.0).
constexpr int kDirectFanout = 3;
static_assert(kStages >= 2 && kStages <= 6, "staging ring of 2 to 6 rows");

// Dynamic shared memory: [table nchunks*L | starts L | psum L | rows ntok*K |
// experts ntok*K | token list ntok] (dispatch modes only), then, at a 128-byte boundary,
// p.stages staged rows of H bytes and the scales of the tokens staged early
// (p.pre x CPT x threads words, CPT = 16-element chunks per thread).
__host__ __device__ inline size_t layout_bytes(const ScatterArgs& p, int64_t ntok) {
  if (p.mode == kModeIdentity) return 0;
  return ((size_t)p.nchunks * p.L + 2 * (size_t)p.L + 2 * (size_t)ntok * p.K + (size_t)ntok) *
         sizeof(int32_t);
}
__host__ __device__ inline size_t stage_offset(const ScatterArgs& p, int64_t ntok) {
  return (layout_bytes(p, ntok) + 127) / 128 * 128;
}
__host__ __device__ inline size_t smem_bytes(const ScatterArgs& p, int64_t ntok, int bd, int cpt) {
  if (p.mode == kModeIdentity) return 0;  // direct stores, nothing staged
  if (p.direct) return stage_offset(p, ntok);
  return stage_offset(p, ntok) + (size_t)p.stages * p.H + (size_t)p.pre * cpt * bd * sizeof(int32_t);
}

// Wait until at most n - 2 bulk groups of this thread still read shared
// memory (n = staging ring size, 2..6; the wait takes an immediate).
__device__ __forceinline__ void wait_ring(int n) {
  switch (n) {
    case 2: bulk_wait_read<0>(); break;
    case 3: bulk_wait_read<1>(); break;
    case 4: bulk_wait_read<2>(); break;
    case 5: bulk_wait_read<3>(); break;
    default: bulk_wait_read<4>(); break;
  }
}
// Tokens per CTA the row buffer is sized for (ceil(T / grid)).
__device__ inline int64_t ntok_smem(const ScatterArgs& p) {
  return ((int64_t)p.T + gridDim.x - 1) / gridDim.x;
}


template <int CPT>
__device__ __forceinline__ void load_row(uint4 (&v)[CPT][2], const uint16_t* xrow, int nch,
                                         int bd, int tid) {
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    const int c = i * bd + tid;
    if (xrow != nullptr && c < nch) {
      v[i][0] = ld_nc_v4(xrow + c * 16);
      v[i][1] = ld_nc_v4(xrow + c * 16 + 8);
    } else {
      v[i][0] = v[i][1] = make_uint4(0, 0, 0, 0);
    }
  }
}

// Layout prologue of a dispatch CTA (see the file comment). Leaves in shared
// memory: the exclusive per-expert prefix over chunks (tbl), the expert row
// base (st: compact start, masked 0) and, for compact, psum (ps).
__device__ void layout_prologue(const ScatterArgs& p, int32_t* tbl, int32_t* st, int32_t* ps,
                                int32_t* s_wsum) {
  const int tid = threadIdx.x, bd = blockDim.x;
  const int L = p.L, NC = p.nchunks;
  // the whole table in flight at once: 16-byte asynchronous copies (the
  // table starts 16-byte aligned in the workspace), the odd tail by loads
  const int n = NC * L, n4 = n / 4;
  for (int i = tid; i < n4; i += bd) cp_async16(tbl + 4 * i, p.table + 4 * i);
  for (int i = 4 * n4 + tid; i < n; i += bd) tbl[i] = __ldcg(p.table + i);
  cp_async_wait_all();
  __syncthreads();
  for (int e = tid; e < L; e += bd) {
    int run = 0, c = 0;
    for (; c + 8 <= NC; c += 8) {  // 8 loads in flight, then 8 stores
      int h[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) h[j] = tbl[(c + j) * L + e];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        tbl[(c + j) * L + e] = run;
        run += h[j];
      }
    }
    for (; c < NC; ++c) {
      const int h = tbl[c * L + e];
      tbl[c * L + e] = run;
      run += h;
    }
    ps[e] = run;  // count, for now
  }
  __syncthreads();
  if (p.mode == kModeCompact) {
    // segment starts: exclusive scan of align(count) over experts
    const int total = aligned_starts(ps, st, L, p.block_e, INT_MAX, s_wsum);
    for (int e = tid; e < L; e += bd) ps[e] += st[e];  // count -> psum
    if (blockIdx.x == 0 && tid == 0) *p.total = total;
    __syncthreads();
    if (blockIdx.x == 0) {
      for (int e = tid; e < L; e += bd) {
        p.counts[e] = ps[e] - st[e];
        p.starts[e] = st[e];
        p.psum[e] = ps[e];
      }
    }
  } else {
    // masked: masked_m = min(count, cap) and the overflow flag; st is free
    // here (slab rows need no start) and takes the expanded-layout starts of
    // the slab's real rows when psum is asked for (PR #29525 _build_layout)
    bool overflow = false;
    for (int e = tid; e < L; e += bd) {
      const int cnt = ps[e];
      if (blockIdx.x == 0) p.masked_m[e] = min(cnt, p.cap);
      if (cnt > p.cap) overflow = true;
    }
    if (overflow && blockIdx.x == 0) set_status(p.status, kStOverflow);
    if (p.psum != nullptr && blockIdx.x == 0) {  // uniform over the CTA
      aligned_starts(ps, st, L, p.block_e, p.cap, s_wsum);
      for (int e = tid; e < L; e += bd) p.psum[e] = st[e] + min(ps[e], p.cap);
    }
    __syncthreads();
  }
}

// Quantises one thread's 16-element chunk (a, b) of a row: the group maximum
// over the GSZ/16 lanes of the group (xor shuffles over sign-cleared bf16
// bits), the group's exponent e (or plain fp32 scale sval) and the 16 e4m3
// codes. Every lane of the warp must call it.
template <int GSZ, int FMT>
__device__ __forceinline__ uint4 quant_chunk(const uint4& a, const uint4& b, int& e, float& sval) {
  uint32_t m = amax16_bf16(a, b);
#pragma unroll
  for (int off = 1; off < GSZ / 16; off <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
  const float amax = __uint_as_float(m << 16);
  uint2 q0, q1;
  e = 0;
  sval = 0.0f;
  if constexpr (FMT == kFmtF32) {
    sval = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
    q0 = quant8_div(a, sval);
    q1 = quant8_div(b, sval);
  } else {
    e = (FMT == kFmtMX) ? mx_exponent(amax) : group_exponent(amax);
    const float inv = exp2_neg(e);
    q0 = quant8(a, inv);
    q1 = quant8(b, inv);
  }
  return make_uint4(q0.x, q0.y, q1.x, q1.y);
}

// Row of slot a (expert e, chunk-local rank lr) from the prologue's tables;
// -1 if dropped. A rank that does not fit the layout (only possible if the
// workspace was altered between the launches) flags BAD_LAYOUT and drops the
// slot, so no write ever leaves the buffers.
__device__ __forceinline__ int slot_row(const ScatterArgs& p, const int32_t* tbl, const int32_t* st,
                                        int64_t a, int e, int lr) {
  if (e < 0 || e >= p.L) return -1;
  const int base = tbl[(int)(a / p.chunk) * p.L + e];
  if (p.mode == kModeCompact) {
    const int row = st[e] + base + lr;
    if (lr < 0 || row < 0 || (int64_t)row >= p.bound) {
      set_status(p.status, kStBadLayout);
      return -1;
    }
    return row;
  }
  const int j = base + lr;
  if (lr < 0 || j < 0) {
    set_status(p.status, kStBadLayout);
    return -1;
  }
  return j < p.cap ? e * p.cap + j : -1;
}

template <int GSZ, int FMT, int CPT>
__global__ void __launch_bounds__(1024, 1) quant_scatter_kernel(ScatterArgs p) {
  extern __shared__ int32_t sm[];
  __shared__ int32_t s_wsum[33];
  __shared__ int32_t s_nlist;
  // tokens taken from the counter (direct mode with the counter, or the
  // staged mode's tail; never both in one launch): a ring of entries, each a
  // token and the rows and experts of its slots (K <= 32)
  __shared__ int32_t s_q[3];
  __shared__ int32_t s_qrows[3][32];
  __shared__ int32_t s_qexps[3][32];
  const int tid = threadIdx.x, lane = tid & 31, bd = blockDim.x;
  const int H = p.H;
  const int nch = H / 16;
  const int G = H / GSZ;
  const int G4 = (G + 3) / 4;
  const bool identity = p.mode == kModeIdentity;
  const int nslots = identity ? 1 : p.K;
  const int n_live = live_count(p.d_num_tokens, p.T, p.status,
                                identity && blockIdx.x == 0 && tid == 0);
  const int ntok_all =
      n_live > (int)blockIdx.x ? (n_live - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const bool tail = p.nstat > 0;  // staged mode only (set at launch)
  const int ntok = tail && ntok_all > p.nstat ? p.nstat : ntok_all;  // static tokens of this CTA
  const bool dyn = p.dyn != 0;  // direct mode with the token counter (one extra warp, see below)
  const int nsl = identity || dyn ? 0 : ntok * p.K;  // slots of this CTA: i -> token i / K, slot i % K
  auto slot_of = [&](int i) -> int64_t {
    return (int64_t)(blockIdx.x + (i / p.K) * gridDim.x) * p.K + (i % p.K);
  };

  // Inputs only, before anything waits: the first token's row and the expert
  // id of this thread's first slot.
  uint4 v[CPT][2];
  load_row(v, ntok > 0 && !dyn ? p.x + (int64_t)blockIdx.x * p.ldx : nullptr, nch, bd, tid);
  const int64_t a0 = tid < nsl ? slot_of(tid) : -1;
  const int e0 = a0 >= 0 ? __ldg(p.ids + a0) : -1;

  uint8_t* stage = reinterpret_cast<uint8_t*>(sm) + stage_offset(p, ntok_smem(p));
  int32_t* pre_s = reinterpret_cast<int32_t*>(stage + (size_t)p.stages * H);  // [pre][CPT][bd]
  int32_t* rows_s = sm;  // identity mode: unused
  int32_t* exps_s = sm;  // expert of each slot (masked scale blocks)
  int32_t* list_s = sm;  // iteration -> token index of this CTA (dispatch modes)
  int nlist = ntok;
  int32_t* st = sm;
  int32_t* ps = sm;
  int npre = 0;
  if (!identity) {
    // The first p.pre tokens are quantised into their staging buffers while the
    // route plan still runs (their rows are not known yet); their scales wait
    // in shared memory.
    npre = p.direct ? 0 : (ntok < p.pre ? ntok : p.pre);
    for (int j = 0; j < npre; ++j) {
      uint4 vn[CPT][2];
      load_row(vn, j + 1 < npre ? p.x + (int64_t)(blockIdx.x + (j + 1) * gridDim.x) * p.ldx : nullptr,
               nch, bd, tid);
      uint8_t* sb = stage + (size_t)j * H;
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const int c = i * bd + tid;
        int e;
        float sval;
        const uint4 qv = quant_chunk<GSZ, FMT>(v[i][0], v[i][1], e, sval);
        if (c < nch) *reinterpret_cast<uint4*>(sb + c * 16) = qv;
        pre_s[(j * CPT + i) * bd + tid] = (FMT == kFmtF32) ? __float_as_int(sval) : e;
      }
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        v[i][0] = vn[i][0];
        v[i][1] = vn[i][1];
      }
    }

    pdl_wait_primary();
    if (!p.direct && tid == 0) {  // the rows of the next tokens into L2 while the layout is built
      const uint64_t pol = l2_policy_evict_last();
      for (int j = npre; j < ntok && j < npre + kPrefetchAfterWait; ++j)
        bulk_prefetch_l2_hint(p.x + (int64_t)(blockIdx.x + j * gridDim.x) * p.ldx, (uint32_t)(2 * H), pol);
    }
    const int lr0 = a0 >= 0 ? __ldcg(p.src2dst + a0) : -1;  // in flight with the table loads
    const int L = p.L;
    int32_t* tbl = sm;
    st = tbl + p.nchunks * L;
    ps = st + L;
    rows_s = ps + L;
    exps_s = rows_s + (size_t)ntok_smem(p) * p.K;
    list_s = exps_s + (size_t)ntok_smem(p) * p.K;
    layout_prologue(p, tbl, st, ps, s_wsum);

    // rows of every slot this CTA will scatter
    for (int i = tid; i < nsl; i += bd) {
      int64_t a;
      int e, lr;
      if (i == tid) {
        a = a0;
        e = e0;
        lr = lr0;
      } else {
        a = slot_of(i);
        e = __ldg(p.ids + a);
        lr = __ldcg(p.src2dst + a);
      }
      const int row = slot_row(p, tbl, st, a, e, lr);
      p.src2dst[a] = row;
      if (row >= 0 && p.row_weights != nullptr) p.row_weights[row] = __ldg(p.w + a);
      rows_s[i] = row;
      exps_s[i] = e;
    }
    __syncthreads();

    // The tokens to walk: the staged ones, then, in order, every later token
    // with at least one kept slot. A token whose experts are all remote is
    // neither read nor quantised.
    if (tid < 32 && !dyn) {
      int base = npre;
      for (int t0 = npre; t0 < ntok; t0 += 32) {
        const int it = t0 + lane;
        bool kept = false;
        if (it < ntok)
          for (int k = 0; k < p.K; ++k) kept |= rows_s[it * p.K + k] >= 0;
        const unsigned m = __ballot_sync(0xffffffffu, kept);
        if (kept) list_s[base + __popc(m & ((1u << lane) - 1u))] = it;
        base += __popc(m);
      }
      if (lane == 0) s_nlist = base;
    }
    for (int j = tid; j < npre; j += bd) list_s[j] = j;
    __syncthreads();
    nlist = dyn ? 0 : s_nlist;
    if (!dyn && npre == 0 && nlist > 0 && list_s[0] != 0)  // no early tokens: v holds token 0 already
      load_row(v, p.x + (int64_t)(blockIdx.x + list_s[0] * gridDim.x) * p.ldx, nch, bd, tid);
  }

  // ---- identity mode (live-row quantiser): one destination per row, so no
  // staging and no barrier. Every warp runs on its own: the next row's loads
  // go out first, then the warp quantises its chunks and stores each 16-byte
  // vector straight to the row (a warp writes 512 contiguous bytes).
  if (identity) {
    for (int it = 0; it < ntok; ++it) {
      const int t = blockIdx.x + it * gridDim.x;
      const int tn = t + gridDim.x;
      uint4 vn[CPT][2];
      load_row(vn, tn < n_live ? p.x + (int64_t)tn * p.ldx : nullptr, nch, bd, tid);
      const int rows[1] = {t};
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const int c = i * bd + tid;
        const bool active = c < nch;
        int e;
        float sval;
        const uint4 qv = quant_chunk<GSZ, FMT>(v[i][0], v[i][1], e, sval);
        if (active) st_v4(p.xq + (int64_t)t * H + c * 16, qv);
        const int cw = i * bd + (tid & ~31);  // first chunk of this warp
        if (cw < nch) store_scales<GSZ, FMT>(p, 1, rows, rows, lane, active, e, sval, cw * 16 / GSZ, G, G4);
      }
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        v[i][0] = vn[i][0];
        v[i][1] = vn[i][1];
      }
    }
    return;
  }

  // ---- direct mode with the token counter. The static strided assignment
  // gives each CTA a fixed set of tokens, but how many of them have a kept
  // slot varies (2 to 14 of 13 at 32 of 256 experts local), and so does when
  // each CTA finishes. Here each CTA starts with token blockIdx.x and then
  // takes tokens gridDim.x, gridDim.x + 1, ... from a counter that the route
  // plan set to 0; every token below the live count is taken exactly once,
  // and the CTA that takes it resolves its rows and rewrites its src2dst
  // entries. The block's last warp is the producer: it finds the next token
  // with a kept slot (resolving rows as it goes) two tokens ahead, while the
  // other warps quantise and store the current one and load the next one; a
  // barrier per token publishes the producer's slot.
  if (dyn) {
    const int bdc = bd - 32;
    const bool producer = tid >= bdc;
    const int K = p.K;
    auto take = [&](int start, int slot) -> int {  // producer warp only
      int t = start;
      if (t < 0) {
        int nt = 0;
        if (lane == 0) nt = (int)gridDim.x + atomicAdd(p.queue, 1);
        t = __shfl_sync(0xffffffffu, nt, 0);
      }
      for (;;) {
        if (t >= n_live) return n_live;
        bool kept = false;
        if (lane < K) {
          const int64_t a = (int64_t)t * K + lane;
          const int e = __ldg(p.ids + a);
          const int row = slot_row(p, sm, st, a, e, __ldcg(p.src2dst + a));
          p.src2dst[a] = row;
          if (row >= 0 && p.row_weights != nullptr) p.row_weights[row] = __ldg(p.w + a);
          s_qrows[slot][lane] = row;
          s_qexps[slot][lane] = e;
          kept = row >= 0;
        }
        if (__any_sync(0xffffffffu, kept)) return t;
        int nt = 0;
        if (lane == 0) nt = (int)gridDim.x + atomicAdd(p.queue, 1);
        t = __shfl_sync(0xffffffffu, nt, 0);
      }
    };
    if (producer) {
      const int t0 = take(ntok > 0 ? (int)blockIdx.x : -1, 0);
      const int t1 = t0 < n_live ? take(-1, 1) : n_live;
      if (lane == 0) {
        s_q[0] = t0;
        s_q[1] = t1;
      }
    }
    __syncthreads();
    int t = s_q[0];
    if (!producer) load_row(v, t < n_live ? p.x + (int64_t)t * p.ldx : nullptr, nch, bdc, tid);
    for (int n = 0; t < n_live; ++n) {
      const int tn = s_q[(n + 1) % 3];
      if (producer) {
        const int t2 = tn < n_live ? take(-1, (n + 2) % 3) : n_live;
        if (lane == 0) s_q[(n + 2) % 3] = t2;
      } else {
        uint4 vn[CPT][2];
        load_row(vn, tn < n_live ? p.x + (int64_t)tn * p.ldx : nullptr, nch, bdc, tid);
        const int* rows = s_qrows[n % 3];
        const int* exps = s_qexps[n % 3];
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
          const int c = i * bdc + tid;
          const bool active = c < nch;
          int e;
          float sval;
          const uint4 qv = quant_chunk<GSZ, FMT>(v[i][0], v[i][1], e, sval);
          if (active)
            for (int k = 0; k < K; ++k)
              if (rows[k] >= 0) st_v4(p.xq + (int64_t)rows[k] * H + c * 16, qv);
          const int cw = i * bdc + (tid & ~31);  // first chunk of this warp
          if (cw < nch)
            store_scales<GSZ, FMT>(p, K, rows, exps, lane, active, e, sval, cw * 16 / GSZ, G, G4);
        }
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
          v[i][0] = vn[i][0];
          v[i][1] = vn[i][1];
        }
      }
      __syncthreads();
      t = tn;
    }
  }

  // ---- direct mode: few kept slots per token, so no staging and no barrier;
  // each warp stores its 16-byte vectors straight to every destination row.
  if (p.direct) {
    for (int n = 0; n < nlist; ++n) {
      const int it = list_s[n];
      const int itn = n + 1 < nlist ? list_s[n + 1] : -1;
      uint4 vn[CPT][2];
      load_row(vn, itn >= 0 ? p.x + (int64_t)(blockIdx.x + itn * gridDim.x) * p.ldx : nullptr,
               nch, bd, tid);
      const int* rows = rows_s + it * p.K;
      const int* exps = exps_s + it * p.K;
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const int c = i * bd + tid;
        const bool active = c < nch;
        int e;
        float sval;
        const uint4 qv = quant_chunk<GSZ, FMT>(v[i][0], v[i][1], e, sval);
        if (active)
          for (int k = 0; k < p.K; ++k)
            if (rows[k] >= 0) st_v4(p.xq + (int64_t)rows[k] * H + c * 16, qv);
        const int cw = i * bd + (tid & ~31);  // first chunk of this warp
        if (cw < nch)
          store_scales<GSZ, FMT>(p, p.K, rows, exps, lane, active, e, sval, cw * 16 / GSZ, G, G4);
      }
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        v[i][0] = vn[i][0];
        v[i][1] = vn[i][1];
      }
    }
    nlist = 0;  // nothing left for the staged loop below
  }

  // ---- token loop (dispatch modes; the identity mode returned above) --------
  // The quantised row is staged in shared memory (p.stages rotating buffers)
  // and thread 0 writes it to every destination row with bulk copies, so the
  // payload stores leave the SM as a few large TMA transfers. One barrier per
  // token publishes the staged row; before it, thread 0 waits until the bulk
  // copies that last read the NEXT buffer are done, so after it every thread
  // may overwrite that buffer. Tokens staged before the wait only have their
  // scales stored here.
  const uint32_t stage_s = (uint32_t)__cvta_generic_to_shared(stage);
  int ident_row[1];
  // evict_first on the payload rows: nothing here reads them back (prefill
  // 103.1-103.4 -> 103.1-103.3 us, 32 of 256 experts local 47.1 -> 45.1 us)
  const uint64_t st_policy = l2_policy_evict_first();
  int n = 0;
  for (; n < nlist; ++n) {
    const int it = identity ? n : list_s[n];
    const int t = blockIdx.x + it * gridDim.x;
    const bool staged = n < npre;  // the staged tokens are list entries 0 .. npre-1
    const bool fetch = n + 1 >= npre;
    uint4 vn[CPT][2];
    if (fetch) {
      const int itn = n + 1 < nlist ? (identity ? n + 1 : list_s[n + 1]) : -1;
      load_row(vn, itn >= 0 ? p.x + (int64_t)(blockIdx.x + itn * gridDim.x) * p.ldx : nullptr,
               nch, bd, tid);
    }
    const int* rows;
    const int* exps = exps_s + it * p.K;
    if (identity) {
      ident_row[0] = t;
      rows = ident_row;
    } else {
      rows = rows_s + it * p.K;
    }
    const int buf = n % p.stages;
    uint8_t* sb = stage + (size_t)buf * H;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      const int c = i * bd + tid;
      const bool active = c < nch;
      int e;
      float sval;
      if (staged) {
        const int w = pre_s[(it * CPT + i) * bd + tid];
        e = w;
        sval = __int_as_float(w);
      } else {
        const uint4 qv = quant_chunk<GSZ, FMT>(v[i][0], v[i][1], e, sval);
        if (active) *reinterpret_cast<uint4*>(sb + c * 16) = qv;
      }
      const int cw = i * bd + (tid & ~31);  // first chunk of this warp
      if (cw < nch)
        store_scales<GSZ, FMT>(p, nslots, rows, exps, lane, active, e, sval, cw * 16 / GSZ, G, G4);
    }
    fence_proxy_async_smem();
    if (tid == 0) wait_ring(p.stages);
    __syncthreads();
    if (tid == 0) {
      for (int k = 0; k < nslots; ++k) {
        const int row = rows[k];
        if (row < 0) continue;
        bulk_store_s2g_hint(p.xq + (int64_t)row * H, stage_s + (uint32_t)(buf * H), (uint32_t)H, st_policy);
      }
      bulk_commit();
    }
    if (fetch) {
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        v[i][0] = vn[i][0];
        v[i][1] = vn[i][1];
      }
    }
  }

  // ---- tail: tokens [nstat * grid, n_live) from the counter the route plan
  // reset, each taken exactly once (which CTA takes a token changes no
  // output: its rows follow from the layout alone). Warp 0 claims the next token with a kept
  // slot and resolves its rows (rewriting its src2dst entries) into the other
  // of two ring entries while the current token is quantised; the staging
  // ring and its barrier continue from the static loop. Claiming only one
  // token ahead keeps the counter's tokens free for the CTAs that finish
  // first (claiming two ahead, with the next row loaded one token ahead as in
  // the static loop, measured 106.1-106.6 against 103.6-104.1 us).
  if (tail) {
    const int K = p.K;
    const int64_t pool0 = (int64_t)p.nstat * gridDim.x;
    int32_t* s_dt = s_q;
    auto claim = [&](int slot) {  // warp 0 only
      for (;;) {
        int tc = 0;
        if (lane == 0) tc = (int)(pool0 + atomicAdd(p.queue, 1));
        tc = __shfl_sync(0xffffffffu, tc, 0);
        if (tc >= n_live) {
          if (lane == 0) s_dt[slot] = n_live;
          return;
        }
        if (lane == 0)
          bulk_prefetch_l2_hint(p.x + (int64_t)tc * p.ldx, (uint32_t)(2 * H), l2_policy_evict_last());
        bool kept = false;
        for (int k = lane; k < K; k += 32) {
          const int64_t a = (int64_t)tc * K + k;
          const int e = __ldg(p.ids + a);
          const int row = slot_row(p, sm, st, a, e, __ldcg(p.src2dst + a));
          p.src2dst[a] = row;
          if (row >= 0 && p.row_weights != nullptr) p.row_weights[row] = __ldg(p.w + a);
          s_qrows[slot][k] = row;
          s_qexps[slot][k] = e;
          kept |= row >= 0;
        }
        if (__any_sync(0xffffffffu, kept)) {
          if (lane == 0) s_dt[slot] = tc;
          return;
        }
      }
    };
    if (tid < 32) claim(0);
    __syncthreads();
    int t = s_dt[0];
    load_row(v, t < n_live ? p.x + (int64_t)t * p.ldx : nullptr, nch, bd, tid);
    for (int k = 0; t < n_live; ++k, ++n) {
      const int cur = k & 1;
      if (tid < 32) claim(cur ^ 1);  // the next token, while this one's row arrives
      const int* rows = s_qrows[cur];
      const int* exps = s_qexps[cur];
      const int buf = n % p.stages;
      uint8_t* sb = stage + (size_t)buf * H;
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const int c = i * bd + tid;
        const bool active = c < nch;
        int e;
        float sval;
        const uint4 qv = quant_chunk<GSZ, FMT>(v[i][0], v[i][1], e, sval);
        if (active) *reinterpret_cast<uint4*>(sb + c * 16) = qv;
        const int cw = i * bd + (tid & ~31);
        if (cw < nch) store_scales<GSZ, FMT>(p, K, rows, exps, lane, active, e, sval, cw * 16 / GSZ, G, G4);
      }
      fence_proxy_async_smem();
      if (tid == 0) wait_ring(p.stages);
      __syncthreads();
      if (tid == 0) {
        for (int j = 0; j < K; ++j) {
          const int row = rows[j];
          if (row < 0) continue;
          bulk_store_s2g_hint(p.xq + (int64_t)row * H, stage_s + (uint32_t)(buf * H), (uint32_t)H, st_policy);
        }
        bulk_commit();
      }
      t = s_dt[cur ^ 1];
      load_row(v, t < n_live ? p.x + (int64_t)t * p.ldx : nullptr, nch, bd, tid);
    }
  }

  // compact: m_indices over the whole static bound, while the last bulk
  // copies drain
  if (p.mode == kModeCompact && p.m_indices != nullptr) {
    const int L = p.L;
    for (int64_t r = (int64_t)blockIdx.x * bd + tid; r < p.bound; r += (int64_t)gridDim.x * bd) {
      int lo = 0, hi = L - 1;  // largest e with start[e] <= r (start[0] = 0)
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (st[mid] <= r) lo = mid; else hi = mid - 1;
      }
      p.m_indices[r] = (r < ps[lo]) ? lo : -1;
    }
  }
  if (tid == 0) bulk_wait_all();
}

template <int GSZ, int FMT, int CPT>
cudaError_t launch_one(const ScatterArgs& a0, int num_sms, bool pdl, cudaStream_t s) {
  const int nch = a0.H / 16;
  int bd = (nch + CPT - 1) / CPT;
  bd = (bd + 31) / 32 * 32;
  if (bd > 1024) return cudaErrorInvalidValue;  // H > 32768 is rejected on the host
  int optin = 0;
  cudaError_t err = device_attr_cached(cudaDevAttrMaxSharedMemoryPerBlockOptin, &optin);
  if (err != cudaSuccess) return err;
  const size_t budget = (size_t)optin - 1024;  // room for the static arrays
  // Resident CTAs per SM with a provisional row buffer of 16 tokens per CTA;
  // the grid is then fixed and the row buffer sized for ceil(T / grid) tokens.
  // The staging ring and the early tokens shrink (down to two buffers and
  // none) until one CTA fits the shared-memory budget.
  ScatterArgs a = a0;
  a.direct = 0;
  if (a.mode != kModeIdentity) {
    a.direct = (int64_t)a.K * a.L <= (int64_t)kDirectFanout * a.E ? 1 : 0;
  }
  auto fit = [&](int64_t ntok) {
    a.stages = a.direct ? 0 : kStages;
    a.pre = (a.mode == kModeIdentity || a.direct) ? 0 : kPre;
    while (smem_bytes(a, ntok, bd, CPT) > budget && (a.pre > 0 || a.stages > 2)) {
      if (a.pre > 0) --a.pre; else --a.stages;
    }
    if (a.pre > a.stages) a.pre = a.stages;
  };
  // direct mode with the token counter: one extra warp (the producer)
  // (wide rows only: at two chunks per thread a token is enough work to hide
  // the per-token barrier; with narrow rows the static assignment is faster,
  // T = 16384, H = 2048: 31.2 against 36.1 us)
  a.dyn = (CPT == 2 && a.direct && a.queue != nullptr && a.K <= 32 && bd + 32 <= 1024) ? 1 : 0;
  const int block = bd + (a.dyn ? 32 : 0);
  fit(16);
  int per_sm = 0;
  err = opt_in_smem(quant_scatter_kernel<GSZ, FMT, CPT>, smem_bytes(a, 16, bd, CPT));
  if (err != cudaSuccess) return err;
  err = occupancy(quant_scatter_kernel<GSZ, FMT, CPT>, block, smem_bytes(a, 16, bd, CPT), &per_sm);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  int64_t grid = (int64_t)num_sms * per_sm;
  if (grid > a.T) grid = a.T;
  if (grid < 1) grid = 1;
  const int64_t ntok_max = (a.T + grid - 1) / grid;
  fit(ntok_max);
  // staged mode with enough tokens per CTA: the tail comes from the counter
  a.nstat = 0;
  const int64_t per = a.T / grid;
  if (a.mode != kModeIdentity && !a.direct && a.queue != nullptr && a.K <= 32 &&
      per >= kTailMinTokens) {
    const int64_t kl2 = 2 * (int64_t)a.K * a.L;  // 2 f E
    int64_t tail_tokens = 1;
    if (CPT == 2) {
      if (kl2 >= 15 * (int64_t)a.E) tail_tokens = (per * kTailPct + 99) / 100;
      else if (kl2 >= 11 * (int64_t)a.E) tail_tokens = per / kTailDiv > 1 ? per / kTailDiv : 1;
      else tail_tokens = per / kTailDiv - 1;
    }
    if (tail_tokens > 0) a.nstat = (int32_t)(per - tail_tokens);
  }
  const size_t smem = smem_bytes(a, ntok_max, bd, CPT);
  err = opt_in_smem(quant_scatter_kernel<GSZ, FMT, CPT>, smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, quant_scatter_kernel<GSZ, FMT, CPT>, a);
}

template <int CPT>
cudaError_t launch_cpt(const ScatterArgs& a, int g, int fmt, int num_sms, bool pdl, cudaStream_t s) {
  if (g == 128) {
    if (fmt == kFmtPacked) return launch_one<128, kFmtPacked, CPT>(a, num_sms, pdl, s);
    if (fmt == kFmtU8) return launch_one<128, kFmtU8, CPT>(a, num_sms, pdl, s);
    if (fmt == kFmtF32) return launch_one<128, kFmtF32, CPT>(a, num_sms, pdl, s);
    return launch_one<128, kFmtF32Pow2, CPT>(a, num_sms, pdl, s);
  }
  if (fmt == kFmtMX) return launch_one<32, kFmtMX, CPT>(a, num_sms, pdl, s);
  return launch_one<32, kFmtU8, CPT>(a, num_sms, pdl, s);
}

}  // namespace

cudaError_t launch_quant_scatter(const ScatterArgs& a, int g, int fmt, int num_sms,
                                 bool after_route_plan, cudaStream_t s) {
  // Narrow rows: one chunk per thread, so a CTA still has enough threads to
  // keep loads in flight (measured on GB300: H = 2048 dispatch 67 -> 59 us;
  // at H = 7168 two chunks per thread are faster, 105 against 109 us).
  if (a.H <= kCpt1MaxH) return launch_cpt<1>(a, g, fmt, num_sms, after_route_plan, s);
  return launch_cpt<2>(a, g, fmt, num_sms, after_route_plan, s);
}

}  // namespace moeperm
