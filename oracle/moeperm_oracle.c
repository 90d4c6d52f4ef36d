/*
 * moeperm_oracle.c -- plain CPU oracle for the MoE permute / FP8-quantise /
 * combine / requantise path. TEST INFRASTRUCTURE ONLY (see the header).
 *
 * Written for a reader checking it against the sources by eye: scalar loops,
 * no blocking, no fusion, no reordering. Floating point is exact (double) where
 * the definition is exact; where a floating-point rounding decides a stored
 * byte and the sources do not fix the precision, the oracle takes the same
 * precision as the GPU kernel and says so at the function.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared (no -ffast-math).
 */
#include "moeperm_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* [OCP] E4M3: sign bit, 4 exponent bits (bias 7), 3 mantissa bits.    */
/* No infinities; S.1111.111 is NaN; the largest finite value is 448.  */
/* ------------------------------------------------------------------ */

/* Value of the non-negative code c in [0, 126], straight from the spec. */
static double e4m3_code_value(int c) {
  int E = (c >> 3) & 0xF;
  int M = c & 0x7;
  if (E == 0) return ldexp((double)M, -9);        /* subnormal: M * 2^-3 * 2^(1-7) */
  return ldexp(1.0 + (double)M / 8.0, E - 7);     /* normal */
}

double ref_e4m3_decode(uint8_t c) {
  int mag = c & 0x7F;
  if (mag == 0x7F) return NAN;
  double v = e4m3_code_value(mag);
  return (c & 0x80) ? -v : v;
}

/* Nearest of the 127 non-negative finite codes; ties go to the code whose
 * mantissa LSB is 0 (round to nearest even); magnitudes above 448 saturate to
 * 448 (satfinite); the sign is kept, so -0 encodes as 0x80. */
uint8_t ref_e4m3_encode(double v) {
  if (isnan(v)) return 0x7F;
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs(v);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  /* largest code c with value(c) <= a (codes are increasing in value) */
  int lo = 0, hi = 126;
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (e4m3_code_value(mid) <= a) lo = mid; else hi = mid - 1;
  }
  int c = lo;
  double vc = e4m3_code_value(c);
  if (vc == a) return (uint8_t)(sign | c);
  double vn = e4m3_code_value(c + 1);  /* c + 1 <= 126 because a < 448 */
  double dl = a - vc, du = vn - a;     /* both exact (Sterbenz / vc = 0) */
  int pick;
  if (dl < du) pick = c;
  else if (du < dl) pick = c + 1;
  else pick = (c & 1) ? c + 1 : c;
  return (uint8_t)(sign | pick);
}

void ref_e4m3_encode_array(const double* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ref_e4m3_encode(v[i]);
}

void ref_e4m3_decode_array(const uint8_t* c, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ref_e4m3_decode(c[i]);
}

/* ------------------------------------------------------------------ */
/* [P1] direct UE8M0 activation quantisation: the group scale is a power */
/* of two chosen directly from the group's absolute maximum (no fp32    */
/* scale that is rounded afterwards).                                   */
/*   e = ceil(log2(a / 448)),  a = max(amax, 1e-10f)                     */
/* i.e. the smallest integer e with 448 * 2^e >= a, so a / 2^e lies in   */
/* (224, 448] and nothing saturates. All comparisons are exact.         */
/* ------------------------------------------------------------------ */
int32_t ref_group_exponent(float amax) {
  const float eps = 1e-10f;
  double a = (double)(amax > eps ? amax : eps);
  int k = (int)ceil(log2(a / 448.0));               /* first guess */
  while (ldexp(448.0, k) < a) ++k;                   /* exact fix-ups */
  while (ldexp(448.0, k - 1) >= a) --k;
  if (k < -127) k = -127;
  if (k > 127) k = 127;
  return k;
}

void ref_group_exponent_array(const float* amax, int64_t n, int32_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ref_group_exponent(amax[i]);
}

/* [OCP MX] E8M0 shared scale of a block of E4M3 elements: the largest power of
 * two not above amax, divided by 2^8 (448 = 1.75 * 2^8 is the largest E4M3
 * value, so emax = 8). Elements that then exceed 448 saturate. */
int32_t ref_mx_exponent(float amax) {
  double a = (double)amax;
  if (!(a > 0.0)) return -127;
  int k = (int)floor(log2(a));                       /* first guess */
  while (ldexp(1.0, k) > a) --k;                     /* exact fix-ups */
  while (ldexp(1.0, k + 1) <= a) ++k;
  int X = k - 8;
  if (X < -127) X = -127;
  if (X > 127) X = 127;
  return X;
}

void ref_mx_exponent_array(const float* amax, int64_t n, int32_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ref_mx_exponent(amax[i]);
}

static double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

uint16_t ref_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* Quantise one row in any format.
 *  power-of-two formats (U8, PACKED, F32_POW2): e = ref_group_exponent(amax),
 *    q = RNE_e4m3(x * 2^-e) (exact product), byte e + 127, value 2^e;
 *  MX_E8M0: X = ref_mx_exponent(amax), q = RNE_e4m3(x * 2^-X) saturated,
 *    byte X + 127, value 2^X;
 *  F32: s = fl32(max(amax, 1e-10f) / 448) (one IEEE fp32 division), q =
 *    RNE_e4m3(fl32(x / s)) -- the sources do not fix the precision of the
 *    quotient, so the kernel's (an IEEE fp32 division) is taken; byte 0. */
void ref_quant_row_fmt(const uint16_t* x, int32_t H, int32_t g, int32_t fmt, uint8_t* q,
                       uint8_t* ebytes, float* svals) {
  int32_t G = H / g;
  for (int32_t gi = 0; gi < G; ++gi) {
    double amax = 0.0;
    for (int32_t h = gi * g; h < (gi + 1) * g; ++h) {
      double a = fabs(bf16_value(x[h]));
      if (a > amax) amax = a;
    }
    if (fmt == REF_FMT_F32) {
      const float eps = 1e-10f;
      float a = (float)amax > eps ? (float)amax : eps;
      float sc = a / 448.0f;                                   /* fp32 division */
      ebytes[gi] = 0;
      if (svals) svals[gi] = sc;
      for (int32_t h = gi * g; h < (gi + 1) * g; ++h) {
        float v = (float)bf16_value(x[h]) / sc;                /* fp32 division */
        q[h] = ref_e4m3_encode((double)v);
      }
      continue;
    }
    int32_t e = (fmt == REF_FMT_MX_E8M0) ? ref_mx_exponent((float)amax)
                                         : ref_group_exponent((float)amax);
    ebytes[gi] = (uint8_t)(e + 127);
    if (svals) svals[gi] = (float)ldexp(1.0, e);
    for (int32_t h = gi * g; h < (gi + 1) * g; ++h)
      q[h] = ref_e4m3_encode(ldexp(bf16_value(x[h]), -e));  /* saturates above 448 */
  }
}

void ref_quant_row(const uint16_t* x, int32_t H, int32_t g, uint8_t* q, uint8_t* ebytes) {
  ref_quant_row_fmt(x, H, g, REF_FMT_UE8M0_U8, q, ebytes, NULL);
}

/* ------------------------------------------------------------------ */
/* Scale layouts.                                                      */
/*  U8:     byte (row, gi) at row * ld + gi                             */
/*  F32:    float (row, gi) = 2^(byte-127) at row * ld + gi             */
/*  PACKED: rows are grouped in blocks of `rpb` rows (one block for a   */
/*          compact / expanded buffer, one per expert for a slab). In   */
/*          block b, int32 word (r, w) sits at b*G4*ld + w*ld + r and   */
/*          holds groups 4w..4w+3 with group 4w in the least            */
/*          significant byte; bytes past the last group are 0.          */
/* ------------------------------------------------------------------ */
static int32_t g4_of(int32_t G) { return (G + 3) / 4; }

static void put_scale(int32_t fmt, void* s, int64_t ld, int64_t rpb, int32_t G, int64_t row,
                      int32_t gi, uint8_t byte) {
  if (fmt == REF_FMT_UE8M0_U8 || fmt == REF_FMT_MX_E8M0) {
    ((uint8_t*)s)[row * ld + gi] = byte;
  } else if (fmt == REF_FMT_F32_POW2) {
    ((float*)s)[row * ld + gi] = (float)ldexp(1.0, (int)byte - 127);
  } else {
    int64_t b = row / rpb, r = row % rpb;
    int64_t word = b * (int64_t)g4_of(G) * ld + (int64_t)(gi / 4) * ld + r;
    ((uint8_t*)s)[word * 4 + (gi % 4)] = byte;
  }
}

/* Write the zero pad bytes of a packed row's last word (no-op otherwise). */
static void put_scale_pads(int32_t fmt, void* s, int64_t ld, int64_t rpb, int32_t G, int64_t row) {
  if (fmt != REF_FMT_UE8M0_PACKED) return;
  for (int32_t gi = G; gi < g4_of(G) * 4; ++gi) put_scale(fmt, s, ld, rpb, G, row, gi, 0);
}

/* Copy one scale element (U8: 1 byte, F32: 4 bytes, PACKED: 1 byte of a word). */
static void copy_scale(int32_t fmt, const void* src, int64_t lds, int64_t rpbs, int64_t srow,
                       void* dst, int64_t ldd, int64_t rpbd, int64_t drow, int32_t G, int32_t gi) {
  if (fmt == REF_FMT_UE8M0_U8 || fmt == REF_FMT_MX_E8M0) {
    ((uint8_t*)dst)[drow * ldd + gi] = ((const uint8_t*)src)[srow * lds + gi];
  } else if (fmt == REF_FMT_F32_POW2 || fmt == REF_FMT_F32) {
    ((float*)dst)[drow * ldd + gi] = ((const float*)src)[srow * lds + gi];
  } else {
    int64_t bs = srow / rpbs, rs = srow % rpbs;
    int64_t ws = bs * (int64_t)g4_of(G) * lds + (int64_t)(gi / 4) * lds + rs;
    uint8_t byte = ((const uint8_t*)src)[ws * 4 + (gi % 4)];
    put_scale(fmt, dst, ldd, rpbd, G, drow, gi, byte);
  }
}

/* Store group gi's scale of a row: the float value for REF_FMT_F32, else the byte. */
static void put_group_scale(int32_t fmt, void* s, int64_t ld, int64_t rpb, int32_t G,
                            int64_t row, int32_t gi, uint8_t byte, float val) {
  if (fmt == REF_FMT_F32) ((float*)s)[row * ld + gi] = val;
  else put_scale(fmt, s, ld, rpb, G, row, gi, byte);
}

int64_t ref_scale_bytes(int32_t fmt, int64_t rows, int32_t H, int32_t g) {
  int32_t G = H / g;
  if (fmt == REF_FMT_UE8M0_U8 || fmt == REF_FMT_MX_E8M0) return rows * G;
  if (fmt == REF_FMT_F32_POW2 || fmt == REF_FMT_F32) return rows * G * 4;
  return (int64_t)g4_of(G) * 4 * ((rows + 3) / 4 * 4);
}

/* ------------------------------------------------------------------ */
/* [P1] layout choice and static compact bound                         */
/* ------------------------------------------------------------------ */
int32_t ref_should_use_masked(int64_t E, int64_t L) { return (E > L && L <= 32) ? 1 : 0; }

/* Each non-empty expert takes at least one block of block_e rows; the
 * remaining assignments fill whole blocks: block_e * (n + (A - n) / block_e),
 * n = min(A, L). */
int64_t ref_compact_bound(int64_t A, int64_t L, int64_t block_e) {
  int64_t n = A < L ? A : L;
  return block_e * (n + (A - n) / block_e);
}

static int64_t align_up(int64_t c, int64_t b) { return (c + b - 1) / b * b; }

/* ------------------------------------------------------------------ */
/* Route plan shared by both dispatch layouts (plain definition):       */
/*   slot a = t*K + k of a live token is kept iff 0 <= id < L;          */
/*   count[e] = number of kept slots with id e;                         */
/*   rank(a)  = number of kept slots a' < a with the same id            */
/*   (rows of an expert follow ascending t*K + k).                      */
/* ------------------------------------------------------------------ */
static void route_ranks(const int32_t* ids, int32_t T, int32_t n_live, int32_t K, int32_t L,
                        int32_t* counts, int32_t* rank) {
  for (int32_t e = 0; e < L; ++e) counts[e] = 0;
  for (int64_t a = 0; a < (int64_t)T * K; ++a) {
    int32_t t = (int32_t)(a / K);
    int32_t e = (t < n_live) ? ids[a] : -1;
    if (e >= 0 && e < L) {
      rank[a] = counts[e];
      counts[e] += 1;
    } else {
      rank[a] = -1;
    }
  }
}

int32_t ref_quant_group(const uint16_t* x, int64_t ldx, int32_t T_cap, int32_t n_live,
                        int32_t H, int32_t g, int32_t fmt, uint8_t* xq, void* scales,
                        int64_t ld_s) {
  int32_t st = 0;
  if (n_live > T_cap) { st |= REF_ST_LIVE_OVERFLOW; n_live = T_cap; }
  if (n_live < 0) n_live = 0;
  int32_t G = H / g;
  uint8_t eb[4096];
  float sv[4096];
  for (int32_t t = 0; t < n_live; ++t) {
    ref_quant_row_fmt(x + (int64_t)t * ldx, H, g, fmt, xq + (int64_t)t * H, eb, sv);
    for (int32_t gi = 0; gi < G; ++gi)
      put_group_scale(fmt, scales, ld_s, INT64_MAX, G, t, gi, eb[gi], sv[gi]);
    put_scale_pads(fmt, scales, ld_s, INT64_MAX, G, t);
  }
  return st;
}

int32_t ref_dispatch_compact(const uint16_t* x, int64_t ldx, int32_t T, int32_t n_live,
                             int32_t H, const int32_t* topk_ids, const float* topk_weights,
                             int32_t K, int32_t L, int32_t block_e, int32_t g, int32_t fmt,
                             uint8_t* xq, void* scales, int64_t ld_s, int32_t* m_indices,
                             int64_t bound, int32_t* src2dst, int32_t* counts,
                             int32_t* starts, int32_t* psum, int32_t* total,
                             float* row_weights) {
  int32_t st = 0;
  if (n_live > T) { st |= REF_ST_LIVE_OVERFLOW; n_live = T; }
  if (n_live < 0) n_live = 0;
  int64_t A = (int64_t)T * K;
  int32_t* rank = (int32_t*)malloc(sizeof(int32_t) * (size_t)(A > 0 ? A : 1));
  route_ranks(topk_ids, T, n_live, K, L, counts, rank);

  /* [P1][P3] segments in expert order, each padded to a multiple of block_e:
   * start[e] = sum_{e' < e} align(count[e']), psum[e] = start[e] + count[e]. */
  int64_t acc = 0;
  for (int32_t e = 0; e < L; ++e) {
    starts[e] = (int32_t)acc;
    psum[e] = (int32_t)(acc + counts[e]);
    acc += align_up(counts[e], block_e);
  }
  *total = (int32_t)acc;

  /* [P1] m_indices: the expert id on valid rows, -1 on padding rows and on
   * the unused tail [total, bound). */
  for (int64_t r = 0; r < bound; ++r) m_indices[r] = -1;
  for (int32_t e = 0; e < L; ++e)
    for (int64_t r = starts[e]; r < psum[e]; ++r) m_indices[r] = e;

  int32_t G = H / g;
  uint8_t* qrow = (uint8_t*)malloc((size_t)H);
  uint8_t eb[4096];
  float sv[4096];
  for (int32_t t = 0; t < T; ++t) {
    int quantised = 0;
    for (int32_t k = 0; k < K; ++k) {
      int64_t a = (int64_t)t * K + k;
      if (rank[a] < 0) { src2dst[a] = -1; continue; }
      int32_t e = topk_ids[a];
      int64_t row = starts[e] + rank[a];
      src2dst[a] = (int32_t)row;
      if (row_weights) row_weights[row] = topk_weights[a];
      if (!quantised) { ref_quant_row_fmt(x + (int64_t)t * ldx, H, g, fmt, qrow, eb, sv); quantised = 1; }
      memcpy(xq + row * H, qrow, (size_t)H);
      for (int32_t gi = 0; gi < G; ++gi)
        put_group_scale(fmt, scales, ld_s, INT64_MAX, G, row, gi, eb[gi], sv[gi]);
      put_scale_pads(fmt, scales, ld_s, INT64_MAX, G, row);
    }
  }
  free(qrow);
  free(rank);
  return st;
}

int32_t ref_dispatch_masked(const uint16_t* x, int64_t ldx, int32_t T, int32_t n_live,
                            int32_t H, const int32_t* topk_ids, const float* topk_weights,
                            int32_t K, int32_t L, int32_t cap, int32_t g, int32_t fmt,
                            uint8_t* xq, void* scales, int64_t ld_s, int32_t* masked_m,
                            int32_t* src2dst, float* row_weights, int32_t* psum,
                            int32_t psum_align) {
  int32_t st = 0;
  if (n_live > T) { st |= REF_ST_LIVE_OVERFLOW; n_live = T; }
  if (n_live < 0) n_live = 0;
  int64_t A = (int64_t)T * K;
  int32_t* rank = (int32_t*)malloc(sizeof(int32_t) * (size_t)(A > 0 ? A : 1));
  int32_t* counts = (int32_t*)malloc(sizeof(int32_t) * (size_t)L);
  route_ranks(topk_ids, T, n_live, K, L, counts, rank);

  /* [P3] masked_m = rows actually held by the slab; an expert with more than
   * cap rows is an overflow: flagged, never written past its slab. */
  for (int32_t e = 0; e < L; ++e) {
    masked_m[e] = counts[e] < cap ? counts[e] : cap;
    if (counts[e] > cap) st |= REF_ST_OVERFLOW;
  }
  /* [P3 _build_layout] the expanded layout of the slab's real rows: expert e
   * starts at the previous segment end rounded up to psum_align and ends
   * masked_m[e] rows later (psum[-1] = 0). */
  if (psum) {
    int64_t prev_end = 0;
    for (int32_t e = 0; e < L; ++e) {
      int64_t seg_start = align_up(prev_end, psum_align);
      psum[e] = (int32_t)(seg_start + masked_m[e]);
      prev_end = psum[e];
    }
  }
  int32_t G = H / g;
  uint8_t* qrow = (uint8_t*)malloc((size_t)H);
  uint8_t eb[4096];
  float sv[4096];
  for (int32_t t = 0; t < T; ++t) {
    int quantised = 0;
    for (int32_t k = 0; k < K; ++k) {
      int64_t a = (int64_t)t * K + k;
      if (rank[a] < 0 || rank[a] >= cap) { src2dst[a] = -1; continue; }
      int32_t e = topk_ids[a];
      int64_t row = (int64_t)e * cap + rank[a];
      src2dst[a] = (int32_t)row;
      if (row_weights) row_weights[row] = topk_weights[a];
      if (!quantised) { ref_quant_row_fmt(x + (int64_t)t * ldx, H, g, fmt, qrow, eb, sv); quantised = 1; }
      memcpy(xq + row * H, qrow, (size_t)H);
      for (int32_t gi = 0; gi < G; ++gi)
        put_group_scale(fmt, scales, ld_s, cap, G, row, gi, eb[gi], sv[gi]);
      put_scale_pads(fmt, scales, ld_s, cap, G, row);
    }
  }
  free(qrow);
  free(counts);
  free(rank);
  return st;
}

/* ------------------------------------------------------------------ */
/* [P1] post-permute combine: out[t] = sum over kept slots of w * y[row] */
/* ------------------------------------------------------------------ */
void ref_combine_f64(const uint16_t* y, int64_t ldy, const int32_t* src2dst,
                     const float* w, int32_t T, int32_t K, int32_t H, double* out,
                     double* absmass) {
  for (int32_t t = 0; t < T; ++t) {
    for (int32_t h = 0; h < H; ++h) {
      double s = 0.0, m = 0.0;
      for (int32_t k = 0; k < K; ++k) {
        int32_t row = src2dst[(int64_t)t * K + k];
        if (row < 0) continue;
        double wk = w ? (double)w[(int64_t)t * K + k] : 1.0;
        double p = wk * bf16_value(y[(int64_t)row * ldy + h]);
        s += p;
        m += fabs(p);
      }
      out[(int64_t)t * H + h] = s;
      if (absmass) absmass[(int64_t)t * H + h] = m;
    }
  }
}

/* Same sum in the kernel's precision: fp32 accumulator starting at +0,
 * one fused multiply-add per kept slot in ascending k, then bf16 RNE. */
void ref_combine_f32(const uint16_t* y, int64_t ldy, const int32_t* src2dst,
                     const float* w, int32_t T, int32_t K, int32_t H, uint16_t* out) {
  for (int32_t t = 0; t < T; ++t) {
    for (int32_t h = 0; h < H; ++h) {
      float acc = 0.0f;
      for (int32_t k = 0; k < K; ++k) {
        int32_t row = src2dst[(int64_t)t * K + k];
        if (row < 0) continue;
        float wk = w ? w[(int64_t)t * K + k] : 1.0f;
        acc = fmaf(wk, (float)bf16_value(y[(int64_t)row * ldy + h]), acc);
      }
      out[(int64_t)t * H + h] = ref_bf16_rne(acc);
    }
  }
}

/* ------------------------------------------------------------------ */
/* [P2] per-token -> per-tensor requant.                               */
/*   S = max_t s[t];  q'[t,h] = RNE_e4m3( decode(q[t,h]) * (s[t] / S) ) */
/* The sources do not fix the precision of the rescale; the oracle takes */
/* the kernel's: r = s[t] / S as one fp32 division, the product rounded  */
/* to fp32, then encoded. S = 0 (or T = 0) gives S = 1 and r = 0.        */
/* ------------------------------------------------------------------ */
void ref_requant(const uint8_t* q, int64_t ldq, const float* s_tok, int32_t T, int32_t H,
                 uint8_t* q_out, float* S_out) {
  float S = 0.0f;
  for (int32_t t = 0; t < T; ++t)
    if (s_tok[t] > S) S = s_tok[t];
  *S_out = (S > 0.0f) ? S : 1.0f;
  for (int32_t t = 0; t < T; ++t) {
    float r = (S > 0.0f) ? s_tok[t] / S : 0.0f;
    for (int32_t h = 0; h < H; ++h) {
      float v = (float)ref_e4m3_decode(q[(int64_t)t * ldq + h]);  /* exact */
      float p = v * r;                                             /* fp32 RN */
      q_out[(int64_t)t * H + h] = ref_e4m3_encode((double)p);
    }
  }
}

void ref_requant_ex(const uint8_t* q, int64_t ldq, const void* s_tok, int32_t s_fmt, int32_t T,
                    int32_t H, int32_t mode, uint8_t* q_out, float* S_out) {
  float* s = (float*)malloc(sizeof(float) * (size_t)(T > 0 ? T : 1));
  for (int32_t t = 0; t < T; ++t)
    s[t] = (s_fmt == 0) ? ((const float*)s_tok)[t]
                        : (float)ldexp(1.0, (int)((const uint8_t*)s_tok)[t] - 127);
  float S = 0.0f;
  for (int32_t t = 0; t < T; ++t) {
    float v = s[t];
    if (mode == 1) {
      double amax = 0.0;
      for (int32_t h = 0; h < H; ++h) {
        double a = fabs(ref_e4m3_decode(q[(int64_t)t * ldq + h]));
        if (a > amax) amax = a;
      }
      v = s[t] * (float)amax;                                 /* fp32 product */
    }
    if (v > S) S = v;
  }
  if (mode == 1) S = S / 448.0f;                              /* fp32 division */
  *S_out = (S > 0.0f) ? S : 1.0f;
  for (int32_t t = 0; t < T; ++t) {
    float r = (S > 0.0f) ? s[t] / S : 0.0f;
    for (int32_t h = 0; h < H; ++h) {
      float v = (float)ref_e4m3_decode(q[(int64_t)t * ldq + h]);
      float p = v * r;
      q_out[(int64_t)t * H + h] = ref_e4m3_encode((double)p);
    }
  }
  free(s);
}

/* ------------------------------------------------------------------ */
/* [P3] expanded psum layout <-> masked slab.                           */
/* Expert e owns rows [align(psum[e-1]), psum[e]) with psum[-1] = 0.    */
/* ------------------------------------------------------------------ */
static int32_t psum_geometry(const int32_t* psum, int32_t L, int32_t align, int64_t R,
                             int64_t* start, int64_t* count) {
  int32_t st = 0;
  int64_t prev = 0;
  for (int32_t e = 0; e < L; ++e) {
    start[e] = align_up(prev, align);
    count[e] = (int64_t)psum[e] - start[e];
    if (count[e] < 0 || psum[e] > R) st |= REF_ST_BAD_LAYOUT;
    prev = psum[e];
  }
  return st;
}

int32_t ref_expand_to_slab(const uint8_t* exp, int32_t elem_bytes, int32_t H, int64_t R,
                           const void* exp_scales, int64_t ld_es, const int32_t* psum,
                           int32_t L, int32_t align, int32_t cap, int32_t fmt, int32_t g,
                           uint8_t* slab, void* slab_scales, int64_t ld_ss,
                           int32_t* masked_m) {
  int64_t* start = (int64_t*)malloc(sizeof(int64_t) * (size_t)L);
  int64_t* count = (int64_t*)malloc(sizeof(int64_t) * (size_t)L);
  int32_t st = psum_geometry(psum, L, align, R, start, count);
  if (st) { free(start); free(count); return st; }
  int64_t rowbytes = (int64_t)H * elem_bytes;
  int32_t G = (exp_scales && slab_scales) ? H / g : 0;
  for (int32_t e = 0; e < L; ++e) {
    masked_m[e] = (int32_t)(count[e] < cap ? count[e] : cap);
    if (count[e] > cap) st |= REF_ST_OVERFLOW;
    for (int64_t j = 0; j < count[e] && j < cap; ++j) {
      int64_t src = start[e] + j, dst = (int64_t)e * cap + j;
      memcpy(slab + dst * rowbytes, exp + src * rowbytes, (size_t)rowbytes);
      for (int32_t gi = 0; gi < G; ++gi)
        copy_scale(fmt, exp_scales, ld_es, INT64_MAX, src, slab_scales, ld_ss, cap, dst, G, gi);
      if (G) put_scale_pads(fmt, slab_scales, ld_ss, cap, G, dst);
    }
  }
  free(start);
  free(count);
  return st;
}

int32_t ref_expand_from_slab(const uint8_t* slab, int32_t elem_bytes, int32_t H,
                             const void* slab_scales, int64_t ld_ss, const int32_t* psum,
                             int32_t L, int32_t align, int32_t cap, int32_t fmt, int32_t g,
                             const float* row_weights, uint8_t* exp, int64_t R,
                             void* exp_scales, int64_t ld_es, int32_t* m_indices) {
  int64_t* start = (int64_t*)malloc(sizeof(int64_t) * (size_t)L);
  int64_t* count = (int64_t*)malloc(sizeof(int64_t) * (size_t)L);
  int32_t st = psum_geometry(psum, L, align, R, start, count);
  if (st) { free(start); free(count); return st; }
  int64_t rowbytes = (int64_t)H * elem_bytes;
  int32_t G = (exp_scales && slab_scales) ? H / g : 0;
  /* [P3] m_indices of the expanded layout: expert id on real rows, -1 else. */
  if (m_indices) {
    for (int64_t r = 0; r < R; ++r) m_indices[r] = -1;
    for (int32_t e = 0; e < L; ++e)
      for (int64_t j = 0; j < count[e]; ++j) m_indices[start[e] + j] = e;
  }
  for (int32_t e = 0; e < L; ++e) {
    if (count[e] > cap) st |= REF_ST_OVERFLOW;
    for (int64_t j = 0; j < count[e] && j < cap; ++j) {
      int64_t dst = start[e] + j, src = (int64_t)e * cap + j;
      if (row_weights && elem_bytes == 2) {
        /* [P3] top-k weight applied on real rows only: bf16_RNE(w * v). */
        const uint16_t* s16 = (const uint16_t*)(slab + src * rowbytes);
        uint16_t* d16 = (uint16_t*)(exp + dst * rowbytes);
        float wr = row_weights[dst];
        for (int32_t h = 0; h < H; ++h) d16[h] = ref_bf16_rne(wr * (float)bf16_value(s16[h]));
      } else {
        memcpy(exp + dst * rowbytes, slab + src * rowbytes, (size_t)rowbytes);
      }
      for (int32_t gi = 0; gi < G; ++gi)
        copy_scale(fmt, slab_scales, ld_ss, cap, src, exp_scales, ld_es, INT64_MAX, dst, G, gi);
      if (G) put_scale_pads(fmt, exp_scales, ld_es, INT64_MAX, G, dst);
    }
  }
  free(start);
  free(count);
  return st;
}
