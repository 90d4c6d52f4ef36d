/*
 * moeperm.h -- C ABI of libmoeperm.so: the single-GPU MoE token permute,
 * FP8 group quantisation, combine and requantisation path, written for
 * GB300 (sm_103a).
 *
 * Sources (SGLang pull-request digests, cited by page title and section):
 *   [P1] "PR #33128 DeepGEMM standard MoE dispatch: compact layout and UE8M0
 *        requant" -- 实现拆解 (implementation) items 2-4; 关键源码片段 (code
 *        excerpts) _should_use_masked_standard_layout, _get_compact_all_tokens,
 *        _fwd_kernel_ep_scatter_1; 风险与影响 item 2 (src2dst, post-permute).
 *   [P2] "PR #14162 W4AFP8 DeepEP low-latency FP8 dispatch" -- 实现拆解 items
 *        1-2 (fp8_per_token_to_per_tensor_quant); 评论区精华 (review).
 *   [P3] "PR #29525 DeepEPv2 ElasticBuffer MoE A2A backend" -- 实现拆解 items
 *        3-4 (expand_to_masked_slab, masked_slab_to_expand, 128-aligned psum,
 *        fixed worker pool, stride-aware packed UE8M0 scales); 关键源码片段
 *        _build_layout / _check_expand_roundtrip; 评论区精华 item 1 (masked
 *        tail), 风险与影响 item 1 (overflow must fail fast).
 *   [P4] "PR #36119 MXFP8 MoRI dispatch" -- 功能与动机 (quantise live rows
 *        only), 实现拆解 items 1 and 4 (group 32, e8m0, 224 scales at 7168,
 *        empty batch).
 *
 * General contract (every data call):
 *   - All tensor arguments are DEVICE pointers owned by the caller. The library
 *     never allocates, frees or synchronises (except moe_status_sync).
 *   - Every data call enqueues its kernels on `stream` and returns without
 *     waiting. The grid of every launch depends only on scalar arguments and
 *     the device's SM count, never on routing contents or device-side counts,
 *     so every call that takes its buffers from the caller (all but
 *     moe_dispatch_compact_noalloc, described on its own below) can be
 *     captured in a CUDA graph and replayed with new contents of the same
 *     shapes.
 *   - Argument errors (null required pointer, misalignment, unsupported
 *     sizes / format / group pairs, a workspace that is too small) return
 *     MOE_ERR_INVALID_ARG before anything is launched.
 *   - Data-dependent errors (an expert above its slab capacity, a live-row
 *     count above the buffer, inconsistent prefix sums, an out-of-range row
 *     index) never cause an out-of-bounds access: the kernel writes only
 *     in-bounds rows and ORs a MOE_STATUS_* bit into the caller's device word
 *     `d_status`. The caller clears that word; bits accumulate across calls
 *     until then. moe_status_sync() turns the word into a moe_status_t.
 *   - Output rows the definition does not name (padding rows, slab rows past
 *     an expert's count, rows of non-live tokens) are NOT written, as with an
 *     uninitialised buffer [P1 实现拆解 item 4]. The only exception is
 *     m_indices, which is written over its whole length.
 *   - A launch failure returns MOE_ERR_CUDA (cudaGetLastError is consumed).
 *   - bf16 tensors are raw 16-bit bfloat16 values, e4m3 tensors raw OCP E4M3
 *     bytes. Row offsets are computed in 64-bit.
 *   - Quantisation [P1 实现拆解 item 3, P4]: for each group of g consecutive
 *     elements, e = ceil(log2(max(amax, 1e-10) / 448)) (the smallest e with
 *     448 * 2^e >= max(amax, 1e-10)), the stored scale byte is e + 127 and each
 *     element is RNE_e4m3(x * 2^-e). Inputs are finite.
 */
#ifndef MOEPERM_H
#define MOEPERM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* rejected on the host, nothing launched */
  MOE_ERR_OVERFLOW = 2,      /* an expert received more rows than its slab capacity */
  MOE_ERR_LIVE_OVERFLOW = 3, /* device live-row count larger than the buffer's rows */
  MOE_ERR_BAD_LAYOUT = 4,    /* prefix sums / row indices inconsistent with the buffers */
  MOE_ERR_CUDA = 5           /* a CUDA runtime call or launch failed */
} moe_status_t;

/* Bits ORed into the caller's device status word. */
#define MOE_STATUS_OVERFLOW 0x1
#define MOE_STATUS_LIVE_OVERFLOW 0x2
#define MOE_STATUS_BAD_LAYOUT 0x4

/*
 * Scale layouts ([P3 实现拆解 items 3-4: Blackwell column-major packed UE8M0 vs
 * Hopper row-major fp32]; [P4 实现拆解 item 1: one e8m0 byte per group]).
 * G = H / g groups per row, G4 = ceil(G / 4).
 *
 *  MOE_SCALE_UE8M0_U8     uint8 [rows, ld_s], ld_s >= G; byte (r, j) at r*ld_s + j
 *                         holds e + 127. Bytes j >= G of a row are not written.
 *  MOE_SCALE_UE8M0_PACKED int32 words, column-major per block: rows are split
 *                         into blocks (the whole buffer for a compact or expanded
 *                         layout; one block of `cap` rows per expert for a slab).
 *                         Word (r, w) of block b is at b*G4*ld_s + w*ld_s + r, with
 *                         ld_s >= rows-per-block and ld_s % 4 == 0 (16-byte
 *                         columns). Word w holds groups 4w..4w+3, group 4w in the
 *                         least significant byte; bytes past group G-1 are 0.
 *  MOE_SCALE_F32_POW2     float [rows, ld_s], ld_s >= G; element (r, j) = 2^e.
 *  MOE_SCALE_F32          float [rows, ld_s], ld_s >= G; a plain fp32 group scale
 *                         s = fl32(max(amax, 1e-10) / 448) and q = RNE_e4m3(fl32(x / s))
 *                         (the fp32-scale form that direct UE8M0 replaces
 *                         [P1 实现拆解 item 3]; [P4 功能与动机: group-128 fp32 scales]).
 *  MOE_SCALE_MX_E8M0      uint8 [rows, ld_s] like MOE_SCALE_UE8M0_U8, but with the
 *                         OCP MX exponent rule: X = floor(log2 amax) - 8 (at least
 *                         -127), byte X + 127, q = RNE_e4m3(x * 2^-X) saturated to
 *                         +-448 (the block maximum lands in [256, 512)).
 *
 * Supported (format, group) pairs: g = 128 with U8, PACKED, F32_POW2 or F32;
 * g = 32 with U8 (the MXFP8 layout of [P4]) or MX_E8M0.
 */
typedef enum {
  MOE_SCALE_UE8M0_U8 = 0,
  MOE_SCALE_UE8M0_PACKED = 1,
  MOE_SCALE_F32_POW2 = 2,
  MOE_SCALE_F32 = 3,
  MOE_SCALE_MX_E8M0 = 4
} moe_scale_fmt_t;

/* ------------------------------------------------------------------ */
/* Host helpers (no GPU work)                                          */
/* ------------------------------------------------------------------ */

/* [P1 code excerpt _get_compact_all_tokens] Static row count of the compact
 * layout for A = T*K assignments over L local experts with segments padded to
 * block_e rows: block_e * (n + (A - n) / block_e), n = min(A, L). Every
 * routing fits. Returns 0 for A < 0, L < 1 or block_e < 1. */
int64_t moe_compact_bound(int64_t A, int32_t L, int32_t block_e);

/* [P1 code excerpt _should_use_masked_standard_layout] 1 iff E > L and L <= 32
 * (masked slab layout), else 0 (compact layout). */
int32_t moe_should_use_masked(int32_t E, int32_t L);

/* Bytes of a scale buffer of `fmt` for `rows` rows of H elements in groups of g,
 * with the tightest leading dimension (U8: G, F32: G floats, PACKED: rows
 * rounded up to 4, G4 words per row). 0 on an invalid combination. */
size_t moe_scale_bytes(moe_scale_fmt_t fmt, int64_t rows, int32_t H, int32_t g);

/* Bytes of device workspace the dispatch calls need for T tokens, K slots and L
 * local experts: a 256-byte reserved header and the [chunks, L] int32 table of
 * per-chunk expert histograms (at most 64 KiB; larger T*K x L combinations are
 * rejected, and this returns 0 for them). The workspace needs no
 * initialisation. One workspace must not be used by two calls that can run at
 * once. */
size_t moe_workspace_bytes(int32_t T, int32_t K, int32_t L);

/* ------------------------------------------------------------------ */
/* Dispatch: route + quantise + scatter                                */
/* ------------------------------------------------------------------ */

/*
 * moe_dispatch_compact -- [P1 实现拆解 items 2-4, code excerpts
 * _get_compact_all_tokens and _fwd_kernel_ep_scatter_1; P3 实现拆解 item 4 and
 * _build_layout (the same 128-aligned psum layout)].
 *
 * Inputs
 *   x [T, ldx] bf16              activations, rows 16-byte aligned (ldx % 8 == 0)
 *   T                            token rows of x / topk_ids / topk_weights
 *   d_num_tokens (optional)      device int32: live tokens n <= T; tokens >= n are
 *                                not routed and their x / ids / weights rows are
 *                                never read. NULL means n = T. n > T is clamped
 *                                and sets MOE_STATUS_LIVE_OVERFLOW.
 *   H                            hidden size, H % 16 == 0 and H % g == 0
 *   topk_ids [T, K] int32        expert id per slot; ids outside [0, L) are not
 *                                local and are dropped (src2dst = -1)
 *   topk_weights [T, K] f32      (optional) copied to row_weights
 *   K (1..32), E (>= L), L (1..1024) experts in the model / local experts
 *   block_e                      segment alignment (>= 1), 128 in the sources
 *   g, fmt                       group size and scale layout (pairs above)
 * Outputs (rows of the compact layout, bound = moe_compact_bound(T*K, L, block_e);
 * the caller's buffers must hold at least `bound` rows; when bound is 0, i.e.
 * T = 0, xq / scales / m_indices may be NULL)
 *   xq [bound, H] e4m3           row r = quantised token of the slot that owns r
 *   scales (fmt, ld_s)           scales of the same rows
 *   m_indices [bound] int32      expert id on valid rows, -1 on padding rows and on
 *                                the tail [total, bound) -- written in full
 *   src2dst [T, K] int32         row of each slot, -1 if dropped (all T rows written)
 *   counts, starts, psum [L]     rows per expert, segment start (a multiple of
 *                                block_e), start + count
 *   total [1]                    sum over experts of count rounded up to block_e
 *   row_weights [bound] f32      (optional) topk weight of the slot owning each row
 * Rows of an expert follow ascending t*K + k (a deterministic, stable order).
 * The segment of expert e is [starts[e], starts[e] + align(counts[e])); starts
 * are the exclusive prefix sums of the aligned counts.
 * Limits: T*K <= 2^20, H <= 32768, and the chunk table within 64 KiB.
 * Workspace: moe_workspace_bytes(T, K, L) bytes (no initialisation needed).
 * Launches (fixed grids, the same results either way): for T*K <= 2048
 * slots, one launch in which every CTA ranks all slots in shared memory;
 * otherwise two -- the route plan (chunk histograms and stable ranks), then
 * the layout + quantise + scatter + m_indices launch. The second is started
 * early with programmatic dependent launch: its CTAs quantise their first
 * tokens while the route plan runs and wait for its results on the device.
 * With enough tokens per CTA its last tokens are handed out through a counter
 * in the workspace (reset by the route plan), so that which CTA handles a
 * token varies between calls; no output depends on it.
 */
moe_status_t moe_dispatch_compact(
    const void* x, int64_t ldx, int32_t T, const int32_t* d_num_tokens, int32_t H,
    const int32_t* topk_ids, const float* topk_weights, int32_t K, int32_t E, int32_t L,
    int32_t block_e, int32_t g, moe_scale_fmt_t fmt,
    void* xq, void* scales, int64_t ld_s, int32_t* m_indices, int64_t bound,
    int32_t* src2dst, int32_t* counts, int32_t* starts, int32_t* psum, int32_t* total,
    float* row_weights, void* workspace, size_t workspace_bytes, int32_t* d_status,
    moe_stream_t stream);

/*
 * moe_dispatch_compact_noalloc -- moe_dispatch_compact without a caller-provided
 * workspace. The SGLang pages have no counterpart of this call: it exists for
 * callers of this library, not for the method.
 *
 * Who it is for: callers that cannot allocate device memory -- a plugin whose
 * host engine owns every device allocation and passes in only inputs and
 * outputs, a serving loop that forbids allocation after start-up so that its
 * memory footprint stays fixed, a runtime held to a fixed device-memory
 * budget. It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Arguments, outputs, results and errors are those of moe_dispatch_compact
 * without `workspace` / `workspace_bytes`; the caller still passes every input
 * and output buffer. The scratch lives in one static device array of 65,792
 * bytes (64 KiB + 256, the largest moe_workspace_bytes of any accepted size)
 * that every GPU loading the library holds until the process exits; a call
 * whose moe_workspace_bytes(T, K, L) is 0 or exceeds it returns
 * MOE_ERR_INVALID_ARG before any CUDA work is enqueued.
 *
 * - Set-up: the first call in each CUDA context (normally once per device)
 *   looks up the array's device address with cudaGetSymbolAddress, with that
 *   device current, and caches it under the context's id (a context created
 *   again after cudaDeviceReset is looked up afresh). Make that first call on
 *   each device before any stream capture begins.
 * - Each call enqueues only the dispatch kernels on `stream`. Nothing in the
 *   array needs to start at zero (every word a kernel reads was written
 *   earlier in the same call), so a call clears nothing.
 * - All calls share the one array and it keeps the last call's contents:
 *   calls that can overlap on the GPU (calls on different streams, or from
 *   different host threads) race on it and must be serialised by the caller,
 *   e.g. by issuing them all on one stream.
 */
moe_status_t moe_dispatch_compact_noalloc(
    const void* x, int64_t ldx, int32_t T, const int32_t* d_num_tokens, int32_t H,
    const int32_t* topk_ids, const float* topk_weights, int32_t K, int32_t E, int32_t L,
    int32_t block_e, int32_t g, moe_scale_fmt_t fmt,
    void* xq, void* scales, int64_t ld_s, int32_t* m_indices, int64_t bound,
    int32_t* src2dst, int32_t* counts, int32_t* starts, int32_t* psum, int32_t* total,
    float* row_weights, int32_t* d_status, moe_stream_t stream);

/*
 * moe_dispatch_masked -- [P1 实现拆解 item 2-3 (masked path,
 * moe_ep_deepgemm_preprocess), P3 关键源码片段 (masked slab [E_local, max_m,
 * hidden], masked_m = real counts)].
 *
 * Same inputs as moe_dispatch_compact, plus
 *   cap                          slab rows per local expert (max_m), >= 1
 *   psum_align                   segment alignment of the psum output (>= 1;
 *                                128 in [P3]); ignored when psum is NULL
 * Outputs
 *   xq [L, cap, H] e4m3          slab row (e, j) = j-th slot routed to e
 *   scales (fmt, ld_s)           for PACKED one block of `cap` rows per expert
 *   masked_m [L] int32           min(count, cap)
 *   src2dst [T, K] int32         e*cap + j, or -1 if dropped or past capacity
 *   row_weights [L*cap] f32      (optional)
 *   psum [L] int32               (optional) the expanded (psum) layout of the
 *                                slab's real rows [P3 实现拆解 item 3, 关键源码片段
 *                                _build_layout]: psum[e] = align(psum[e-1],
 *                                psum_align) + masked_m[e], psum[-1] = 0. It is
 *                                the psum moe_expand_from_slab / moe_expand_to_slab
 *                                take with align = psum_align, so a decode step
 *                                can repack the slab without reading counts on
 *                                the host; its rows fit moe_compact_bound(T*K, L,
 *                                psum_align) expanded rows.
 * An expert with more than cap slots sets MOE_STATUS_OVERFLOW; its slots past
 * cap are not written (fail fast, never truncate silently: [P3 风险与影响 1]).
 * Workspace and launches as moe_dispatch_compact.
 */
moe_status_t moe_dispatch_masked(
    const void* x, int64_t ldx, int32_t T, const int32_t* d_num_tokens, int32_t H,
    const int32_t* topk_ids, const float* topk_weights, int32_t K, int32_t E, int32_t L,
    int32_t cap, int32_t g, moe_scale_fmt_t fmt,
    void* xq, void* scales, int64_t ld_s, int32_t* masked_m, int32_t* src2dst,
    float* row_weights, int32_t* psum, int32_t psum_align, void* workspace,
    size_t workspace_bytes, int32_t* d_status, moe_stream_t stream);

/*
 * moe_quant_group -- [P4 功能与动机 and 实现拆解 item 1: quantise on the send side
 * over the live rows only]. Quantises rows [0, n) of x, n = *d_num_live (or
 * T_cap when NULL; n > T_cap is clamped and sets MOE_STATUS_LIVE_OVERFLOW).
 * Rows >= n of x are never read and rows >= n of xq / scales never written; the
 * launch does not depend on n.
 *   x [T_cap, ldx] bf16, xq [T_cap, H] e4m3, scales (fmt, ld_s) over T_cap rows.
 * Launches: 1.
 */
moe_status_t moe_quant_group(
    const void* x, int64_t ldx, int32_t T_cap, const int32_t* d_num_live, int32_t H,
    int32_t g, moe_scale_fmt_t fmt, void* xq, void* scales, int64_t ld_s,
    int32_t* d_status, moe_stream_t stream);

/* ------------------------------------------------------------------ */
/* Combine                                                             */
/* ------------------------------------------------------------------ */

/*
 * moe_combine -- [P1 风险与影响 item 2, post_permute_deep_gemm_to_standard via
 * src2dst]. out[t, :] = bf16_RNE( sum over k with src2dst[t,k] >= 0 of
 * w[t,k] * y[src2dst[t,k], :] ), accumulated in fp32 with one fused
 * multiply-add per slot in ascending k, starting from +0. A token with every
 * slot dropped gets zeros.
 *   y [R, ldy] bf16               expert outputs in any row layout (compact rows,
 *                                 slab rows e*cap + j, expanded rows); ldy % 8 == 0
 *   src2dst [T, K] int32          rows of y; an index >= R sets MOE_STATUS_BAD_LAYOUT
 *                                 and that slot is skipped
 *   w [T, K] f32                  (optional; NULL means every weight is 1)
 *   d_num_tokens (optional)       live tokens n; rows t >= n of out are not written
 *   out [T, H] bf16               H % 8 == 0
 * Launches: 1.
 */
moe_status_t moe_combine(
    const void* y, int64_t ldy, int64_t R, const int32_t* src2dst, const float* w,
    int32_t T, const int32_t* d_num_tokens, int32_t K, int32_t H, void* out,
    int32_t* d_status, moe_stream_t stream);

/* ------------------------------------------------------------------ */
/* Expanded (psum) layout <-> masked slab repack                        */
/* ------------------------------------------------------------------ */

/*
 * moe_expand_to_slab -- [P3 实现拆解 item 3 expand_to_masked_slab; 关键源码片段
 * _build_layout]. In the expanded layout expert e owns rows
 * [align(psum[e-1]), psum[e]) of exp (psum[-1] = 0, `align` >= 1). Copies row j
 * of expert e to slab row (e, j) for j < min(count_e, cap), with its scales when
 * exp_scales / slab_scales are given (e4m3 payload only), and writes
 * masked_m[e] = min(count_e, cap). count_e > cap sets MOE_STATUS_OVERFLOW;
 * psum inconsistent with R sets MOE_STATUS_BAD_LAYOUT (nothing is read past R).
 *   exp [R, H] elements of elem_bytes (1 = e4m3, 2 = bf16); exp_scales (fmt, ld_es)
 *   slab [L, cap, H]; slab_scales (fmt, ld_ss; PACKED: one block of cap rows per
 *   expert)
 * Launches: 1 (fixed grid over the R expanded rows).
 */
moe_status_t moe_expand_to_slab(
    const void* exp, int32_t elem_bytes, int32_t H, int64_t R, const void* exp_scales,
    int64_t ld_es, const int32_t* psum, int32_t L, int32_t align, int32_t cap,
    moe_scale_fmt_t fmt, int32_t g, void* slab, void* slab_scales, int64_t ld_ss,
    int32_t* masked_m, int32_t* d_status, moe_stream_t stream);

/*
 * moe_expand_from_slab -- [P3 实现拆解 item 3 masked_slab_to_expand: top-k
 * weights fused on real rows only; ep_expand_init_m_indices_from_psum]. The
 * inverse of moe_expand_to_slab: expanded row align(psum[e-1]) + j = slab row
 * (e, j) for j < min(count_e, cap). With row_weights (bf16 payload only, indexed
 * by expanded row) the stored row is bf16_RNE(fp32(w_r * v)). Scales are copied
 * when both scale pointers are given. m_indices (optional) [R]: e on real rows,
 * -1 on every other row. Expanded rows that are not real rows are not written.
 * count_e > cap sets MOE_STATUS_OVERFLOW and rows past cap are not written.
 * Launches: 1.
 */
moe_status_t moe_expand_from_slab(
    const void* slab, int32_t elem_bytes, int32_t H, const void* slab_scales, int64_t ld_ss,
    const int32_t* psum, int32_t L, int32_t align, int32_t cap, moe_scale_fmt_t fmt,
    int32_t g, const float* row_weights, void* exp, int64_t R, void* exp_scales,
    int64_t ld_es, int32_t* m_indices, int32_t* d_status, moe_stream_t stream);

/* ------------------------------------------------------------------ */
/* Per-token -> per-tensor requant                                      */
/* ------------------------------------------------------------------ */

/*
 * fp8_requant_per_tensor -- [P2 实现拆解 items 1-2:
 * fp8_per_token_to_per_tensor_quant; 风险与影响 item 3: plain fp32 per-token
 * scales]. S = max_t s_tok[t] (S = 1 when T = 0 or every scale is 0);
 * q_out[t, h] = RNE_e4m3( fp32( decode(q[t, h]) * fp32(s_tok[t] / S) ) ).
 * Scales are finite and >= 0.
 *   q [T, ldq] e4m3 (ldq % 16 == 0), s_tok [T] f32, q_out [T, H] e4m3 (H % 16 == 0),
 *   d_scale_out [1] f32 receives S.
 * Launches: 1.
 */
moe_status_t fp8_requant_per_tensor(
    const void* q, int64_t ldq, const float* s_tok, int32_t T, int32_t H, void* q_out,
    float* d_scale_out, moe_stream_t stream);

/* Per-token input scale format and per-tensor scale rule of the extended requant. */
typedef enum {
  MOE_TOKSCALE_F32 = 0,    /* float [T] */
  MOE_TOKSCALE_UE8M0 = 1   /* uint8 [T] e8m0 bytes: scale 2^(b - 127) (b = 255 is out of contract) */
} moe_tokscale_fmt_t;
typedef enum {
  MOE_REQUANT_MAX_SCALE = 0, /* S = max_t s[t] */
  MOE_REQUANT_AMAX = 1       /* S = fl32(max_t fl32(s[t] * amax_t) / 448), amax_t = max_h |decode(q[t,h])| */
} moe_requant_mode_t;

/*
 * fp8_requant_per_tensor_ex -- fp8_requant_per_tensor for e8m0 per-token scales
 * ([P2 风险与影响 item 3]: the original kernel assumes plain fp32 scales and
 * does not handle Blackwell e8m0 ones) and with an amax-based per-tensor scale
 * that maps the largest dequantised value to 448. With MOE_TOKSCALE_F32 and
 * MOE_REQUANT_MAX_SCALE it computes exactly what fp8_requant_per_tensor does.
 *   s_tok [T] in s_fmt; workspace: >= 4*T bytes, 16-byte aligned, for
 *   MOE_REQUANT_AMAX (may be NULL otherwise; needs no initialisation).
 *   q' = RNE_e4m3(fl32(decode(q) * fl32(s[t] / S))); S = 1 when T = 0 or the
 *   maximum is 0.
 * Launches: 1 (max-scale) or 2 (amax: per-row maxima, then the rescale).
 */
moe_status_t fp8_requant_per_tensor_ex(
    const void* q, int64_t ldq, const void* s_tok, moe_tokscale_fmt_t s_fmt, int32_t T,
    int32_t H, moe_requant_mode_t mode, void* q_out, float* d_scale_out, void* workspace,
    size_t workspace_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------ */
/* Status                                                              */
/* ------------------------------------------------------------------ */

/* Waits for `stream`, reads the device status word and returns MOE_OK or the
 * most severe error it holds: MOE_ERR_BAD_LAYOUT, then MOE_ERR_LIVE_OVERFLOW,
 * then MOE_ERR_OVERFLOW (MOE_ERR_CUDA if the wait or copy fails). The non-graph
 * "fail fast" check of [P3 风险与影响 item 1]. */
moe_status_t moe_status_sync(const int32_t* d_status, moe_stream_t stream);

/* Static description of a status code. */
const char* moe_status_string(moe_status_t s);

/* Version string of the library build. */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOEPERM_H */
