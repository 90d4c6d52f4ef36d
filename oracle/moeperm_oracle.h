/*
 * moeperm_oracle.h -- plain, slow, single-threaded CPU oracle for the MoE
 * permute / FP8-quantise / combine / requantise path.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's
 * CPU-baseline leg use this library. It shares no code, header, table or
 * constant with the CUDA library; the two are compared element by element.
 *
 * Sources (SGLang pull-request digests, cited by page title and section):
 *   [P1] "PR #33128: DeepGEMM standard MoE dispatch, compact layout, UE8M0"
 *        sections "实现拆解" (implementation) and "关键源码片段" (code excerpts):
 *        _should_use_masked_standard_layout, _get_compact_all_tokens,
 *        _fwd_kernel_ep_scatter_1 (m_indices = expert id / -1), direct UE8M0
 *        activation quantisation, post-permute via src2dst.
 *   [P2] "PR #14162: W4AFP8 DeepEP low-latency FP8 dispatch", sections
 *        "实现拆解" and "评论区精华": per-token -> per-tensor FP8 requant.
 *   [P3] "PR #29525: DeepEPv2 (ElasticBuffer) MoE A2A backend", sections
 *        "实现拆解" item 3 and the _build_layout / _check_expand_roundtrip
 *        excerpt: 128-aligned psum layout, expand <-> masked slab repack,
 *        masked_m = counts, overflow fail-fast, stride-aware packed UE8M0.
 *   [P4] "PR #36119: MXFP8 MoRI dispatch", section "实现拆解" items 1 and 4:
 *        group-32 e8m0 scales, scale_dim = hidden/32, live rows only.
 *   [OCP] OCP 8-bit Floating Point Specification (OFP8), E4M3 encoding.
 *
 * Conventions: bf16 tensors are uint16 bit patterns, e4m3 tensors are uint8
 * bit patterns. Every function writes only the elements its definition
 * names; everything else in the caller's buffers is left untouched.
 */
#ifndef MOEPERM_ORACLE_H
#define MOEPERM_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Scale layouts (the oracle's own numbering). */
#define REF_FMT_UE8M0_U8 0     /* uint8 [rows, ld] row-major, byte = e + 127 */
#define REF_FMT_UE8M0_PACKED 1 /* int32 words, column-major per block, 4 groups/word, LSB first */
#define REF_FMT_F32_POW2 2     /* float [rows, ld] row-major, value 2^e */
#define REF_FMT_F32 3          /* float [rows, ld]: s = fl32(max(amax,1e-10)/448), q = RNE(fl32(x/s)) */
#define REF_FMT_MX_E8M0 4      /* uint8 [rows, ld]: OCP MX rule X = floor(log2 amax) - 8, byte X+127,
                                  q = RNE_e4m3(x * 2^-X) saturated to +-448 */

/* Data-dependent status bits returned by the layout functions. */
#define REF_ST_OVERFLOW 1      /* an expert received more rows than its slab capacity */
#define REF_ST_LIVE_OVERFLOW 2 /* live-row count above the buffer capacity */
#define REF_ST_BAD_LAYOUT 4    /* prefix sums inconsistent with the buffer */

/* e4m3 (OCP E4M3, bias 7, no infinities, max 448). */
uint8_t ref_e4m3_encode(double v);
double ref_e4m3_decode(uint8_t c);
void ref_e4m3_encode_array(const double* v, int64_t n, uint8_t* out);
void ref_e4m3_decode_array(const uint8_t* c, int64_t n, double* out);

/* Power-of-two group exponent e = ceil(log2(max(amax, 1e-10f) / 448)). */
int32_t ref_group_exponent(float amax);
void ref_group_exponent_array(const float* amax, int64_t n, int32_t* out);

/* OCP MX shared exponent for E4M3 elements: floor(log2(amax)) - 8, clamped to
 * [-127, 127]; amax = 0 gives -127. */
int32_t ref_mx_exponent(float amax);
void ref_mx_exponent_array(const float* amax, int64_t n, int32_t* out);

/* fp32 -> bf16, round to nearest even. */
uint16_t ref_bf16_rne(float f);

/* [P1] compact row bound and layout heuristic. */
int64_t ref_compact_bound(int64_t A, int64_t L, int64_t block_e);
int32_t ref_should_use_masked(int64_t E, int64_t L);

/* Quantise one bf16 row of H elements in groups of g: q[H] bytes, ebytes[H/g]. */
void ref_quant_row(const uint16_t* x, int32_t H, int32_t g, uint8_t* q, uint8_t* ebytes);
/* The same for any format: per group the stored scale as a float (2^e for the
 * power-of-two formats, amax/448 for REF_FMT_F32) and its byte (e + 127, or 0
 * for REF_FMT_F32). */
void ref_quant_row_fmt(const uint16_t* x, int32_t H, int32_t g, int32_t fmt, uint8_t* q,
                       uint8_t* ebytes, float* svals);

/* Scale bytes required for `rows` rows (packed: rows rounded up to 4). */
int64_t ref_scale_bytes(int32_t fmt, int64_t rows, int32_t H, int32_t g);

/* [P4] quantise live rows [0, n_live) of x[T_cap, ldx]. Returns status bits. */
int32_t ref_quant_group(const uint16_t* x, int64_t ldx, int32_t T_cap, int32_t n_live,
                        int32_t H, int32_t g, int32_t fmt, uint8_t* xq, void* scales,
                        int64_t ld_s);

/* [P1][P3] compact dispatch: route plan + quantise + scatter + m_indices. */
int32_t ref_dispatch_compact(const uint16_t* x, int64_t ldx, int32_t T, int32_t n_live,
                             int32_t H, const int32_t* topk_ids, const float* topk_weights,
                             int32_t K, int32_t L, int32_t block_e, int32_t g, int32_t fmt,
                             uint8_t* xq, void* scales, int64_t ld_s, int32_t* m_indices,
                             int64_t bound, int32_t* src2dst, int32_t* counts,
                             int32_t* starts, int32_t* psum, int32_t* total,
                             float* row_weights);

/* [P1][P3] masked dispatch into per-expert slabs [L, cap, H]. psum (optional,
 * [L]) receives the expanded layout of the slab's real rows [P3 _build_layout]:
 * psum[e] = align(psum[e-1], psum_align) + masked_m[e], psum[-1] = 0. */
int32_t ref_dispatch_masked(const uint16_t* x, int64_t ldx, int32_t T, int32_t n_live,
                            int32_t H, const int32_t* topk_ids, const float* topk_weights,
                            int32_t K, int32_t L, int32_t cap, int32_t g, int32_t fmt,
                            uint8_t* xq, void* scales, int64_t ld_s, int32_t* masked_m,
                            int32_t* src2dst, float* row_weights, int32_t* psum,
                            int32_t psum_align);

/* [P1] combine: fp64 reference out[t,h] = sum_k w*y, plus sum_k |w*y|. */
void ref_combine_f64(const uint16_t* y, int64_t ldy, const int32_t* src2dst,
                     const float* w, int32_t T, int32_t K, int32_t H, double* out,
                     double* absmass);
/* [P1] combine, fp32 fused multiply-add in slot order, stored as bf16. */
void ref_combine_f32(const uint16_t* y, int64_t ldy, const int32_t* src2dst,
                     const float* w, int32_t T, int32_t K, int32_t H, uint16_t* out);

/* [P2] per-token -> per-tensor e4m3 requant. Returns nothing; writes S. */
void ref_requant(const uint8_t* q, int64_t ldq, const float* s_tok, int32_t T, int32_t H,
                 uint8_t* q_out, float* S_out);

/* [P2] requant variants. s_fmt: 0 = fp32 per-token scales, 1 = e8m0 bytes
 * (scale 2^(b - 127)). mode: 0 = S = max_t s[t]; 1 = S = fl32(max_t fl32(s[t] *
 * amax_t) / 448) with amax_t = max_h |decode(q[t, h])| (the per-tensor scale
 * that maps the largest dequantised value to 448). Then, as ref_requant,
 * q' = RNE_e4m3(fl32(decode(q) * fl32(s[t] / S))); S = 1 and r = 0 when S is 0. */
void ref_requant_ex(const uint8_t* q, int64_t ldq, const void* s_tok, int32_t s_fmt, int32_t T,
                    int32_t H, int32_t mode, uint8_t* q_out, float* S_out);

/* [P3] expanded psum layout -> masked slab. Returns status bits. */
int32_t ref_expand_to_slab(const uint8_t* exp, int32_t elem_bytes, int32_t H, int64_t R,
                           const void* exp_scales, int64_t ld_es, const int32_t* psum,
                           int32_t L, int32_t align, int32_t cap, int32_t fmt, int32_t g,
                           uint8_t* slab, void* slab_scales, int64_t ld_ss,
                           int32_t* masked_m);

/* [P3] masked slab -> expanded psum layout (optional bf16 row weights). */
int32_t ref_expand_from_slab(const uint8_t* slab, int32_t elem_bytes, int32_t H,
                             const void* slab_scales, int64_t ld_ss, const int32_t* psum,
                             int32_t L, int32_t align, int32_t cap, int32_t fmt, int32_t g,
                             const float* row_weights, uint8_t* exp, int64_t R,
                             void* exp_scales, int64_t ld_es, int32_t* m_indices);

#ifdef __cplusplus
}
#endif
#endif /* MOEPERM_ORACLE_H */
