/*
 * CPU oracle for MXFP8 grouped-matmul-finalize-routing.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg; never by the product path.  It shares no code
 * with the CUDA library.
 *
 * What it computes (write-up "grouped_matmul_finalize_routing 的 MXFP8 实现与精度验证",
 * section 2.1 formula and section 2.2 stages 1-4; aclnnGroupedMatmulFinalizeRoutingV3,
 * "计算公式" items 1-4):
 *
 *   for each expert e with token range [s_e, t_e) (section 4.3 group_list formats),
 *   for each token t in it and each output column n:
 *     acc(t,n) = sum_{k<K} A(t,k) * B(e,k,n)
 *       A(t,k)   = fp8(x1[t,k])    * 2^(pertoken_scale[t, k/64, (k/32)%2] - 127)
 *       B(e,k,n) = fp8(x2[e,k,n])  * 2^(scale[k/64, n, (k/32)%2] - 127)
 *     out[row_index[t], n] += logit[t] * acc(t,n)          (stages 2 and 3)
 *   then out[offset + i, n] += shared_weight * shared_input[i, n]   (stage 4)
 *
 * Readings taken where the pages are loose:
 *   - one E8M0 scale per 32 consecutive K elements, stored as the (ceil(K/64), 2)
 *     pair: element k uses pair k/64, half (k/32)%2 (the golden expands the
 *     scales by 32 along K, section 6.3, although section 2.1 says 64);
 *   - the scale may carry a leading expert dimension (aclnn's 4-D form); without
 *     it every expert shares one scale tensor (the write-up's kernel passes the
 *     whole scale to every expert, section 5.3);
 *   - a scale pair whose second half lies entirely at k >= K is padding and is
 *     never read;
 *   - token ranges are made contiguous and clamped to [0, M]: start_0 = 0,
 *     start_e = end_{e-1}, end_e = clamp(g[e] (type 0) or start_e + g[e] (type 1),
 *     start_e, M); an input that needs clamping raises ORACLE_BAD_GROUP_LIST;
 *   - a token whose row_index is outside [0, batch) contributes nothing and
 *     raises ORACLE_BAD_ROW_INDEX;
 *   - bias (aclnn V3 biasOptional, BF16 on the MX path; the pages give no formula)
 *     is read as a per-expert, per-column term added to acc(t,n) before the logit
 *     weighting: out[row_index[t], n] += logit[t] * (acc(t,n) + bias[e,n]);
 *   - logit == NULL means weight 1 (has_logit=False, section 5.3);
 *     shared_input == NULL skips stage 4;
 *   - MXFP4 (aclnn V3, Atlas 350 MX scenarios): x1 and x2 hold E2M1 codes two per
 *     byte along the contiguous dimension, the even element in the low nibble
 *     (reading); scales are the same E8M0 per 32 elements;
 *   - contributions are added in ascending token order, the shared term last
 *     (the golden's per-expert index_add_ followed by the shared add, section 6.3).
 *
 * Products of two decoded FP8 values times two powers of two are exact in
 * double, so each acc(t,n) carries only the rounding of K double additions.
 */
#include "gmmfr_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* OCP 8-bit floating point, E4M3 ("FN" variant): sign, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent 0 is subnormal (m * 2^-9); no infinities;
 * S.1111.111 is NaN; largest finite 448. */
static double decode_e4m3fn(uint32_t b) {
  const int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
  return s ? -v : v;
}

/* OCP 8-bit floating point, E5M2: sign, 5 exponent bits with bias 15, 2 mantissa
 * bits; exponent 0 is subnormal (m * 2^-16); exponent 31 is Inf (m = 0) or NaN. */
static double decode_e5m2(uint32_t b) {
  const int s = (b >> 7) & 1, e = (b >> 2) & 31, m = b & 3;
  double v;
  if (e == 31) {
    if (m) return NAN;
    return s ? -INFINITY : INFINITY;
  }
  if (e == 0)
    v = ldexp((double)m, -16);
  else
    v = ldexp((double)(4 + m), e - 17); /* (1 + m/4) * 2^(e-15) */
  return s ? -v : v;
}

/* OCP FP4 E2M1: sign, 2 exponent bits with bias 1, 1 mantissa bit; exponent 0 is
 * subnormal (m * 0.5); no Inf or NaN; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
static double decode_e2m1(uint32_t b) {
  const int s = (b >> 3) & 1, e = (b >> 1) & 3, m = b & 1;
  const double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -v : v;
}

double oracle_decode_fp8(int fmt, uint32_t code) {
  if (fmt == ORACLE_E2M1) return decode_e2m1(code & 15);
  return fmt == ORACLE_E5M2 ? decode_e5m2(code & 255) : decode_e4m3fn(code & 255);
}

/* element i of a row stored with `fmt` (two E2M1 codes per byte, even element low) */
static uint32_t element_code(const uint8_t* row, int64_t i, int fmt) {
  if (fmt != ORACLE_E2M1) return row[i];
  const uint8_t b = row[i / 2];
  return (i & 1) ? (b >> 4) : (b & 15);
}

/* OCP MX scale E8M0: 2^(b - 127); 0xFF is NaN. */
double oracle_decode_e8m0(uint32_t code) {
  code &= 255;
  if (code == 255) return NAN;
  return ldexp(1.0, (int)code - 127);
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double oracle_decode_bf16(uint32_t bits) {
  union {
    uint32_t u;
    float f;
  } c;
  c.u = (bits & 0xFFFFu) << 16;
  return (double)c.f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

int oracle_expert_ranges(const oracle_args* a, int64_t* start, int64_t* end) {
  int flags = 0;
  int64_t prev_end = 0;
  for (int64_t e = 0; e < a->E; ++e) {
    const int64_t g = a->group_list[e];
    const int64_t s = prev_end;
    int64_t t;
    if (a->group_list_type == 0) {
      /* prefix sums: expert e owns [g[e-1], g[e]) with g[-1] = 0 */
      if (g < s || g > a->M) flags |= ORACLE_BAD_GROUP_LIST;
      t = g < s ? s : (g > a->M ? a->M : g);
    } else {
      /* counts: expert e owns [sum g[:e], sum g[:e] + g[e]) */
      if (g < 0 || g > a->M - s) flags |= ORACLE_BAD_GROUP_LIST;
      t = g < 0 ? s : (g > a->M - s ? a->M : s + g);
    }
    start[e] = s;
    end[e] = t;
    prev_end = t;
  }
  return flags;
}

static int64_t scale_index(const oracle_args* a, int64_t e, int64_t k, int64_t n) {
  const int64_t Ks = (a->K + 63) / 64;
  const int64_t base = a->scale_per_expert ? e * Ks * a->N * 2 : 0;
  if (a->transpose_x2) return base + (n * Ks + k / 64) * 2 + (k / 32) % 2;
  return base + ((k / 64) * a->N + n) * 2 + (k / 32) % 2;
}

static uint32_t x2_code(const oracle_args* a, int64_t e, int64_t k, int64_t n) {
  const int p = a->x2_fmt == ORACLE_E2M1 ? 2 : 1;  /* elements per byte */
  if (a->transpose_x2) return element_code(a->x2 + (e * a->N + n) * (a->K / p), k, a->x2_fmt);
  return element_code(a->x2 + (e * a->K + k) * (a->N / p), n, a->x2_fmt);
}

/* A(t,k): token value times its block scale */
static double token_value(const oracle_args* a, int64_t t, int64_t k) {
  const int64_t Ks = (a->K + 63) / 64;
  const int p = a->x1_fmt == ORACLE_E2M1 ? 2 : 1;
  const double v = oracle_decode_fp8(a->x1_fmt, element_code(a->x1 + t * (a->K / p), k, a->x1_fmt));
  const double s = oracle_decode_e8m0(a->pertoken_scale[(t * Ks + k / 64) * 2 + (k / 32) % 2]);
  return v * s;
}

/* B(e,k,n): weight value times its block scale */
static double weight_value(const oracle_args* a, int64_t e, int64_t k, int64_t n) {
  const double v = oracle_decode_fp8(a->x2_fmt, x2_code(a, e, k, n));
  const double s = oracle_decode_e8m0(a->scale[scale_index(a, e, k, n)]);
  return v * s;
}

static int row_flags(const oracle_args* a, const int64_t* start, const int64_t* end) {
  int flags = 0;
  for (int64_t e = 0; e < a->E; ++e)
    for (int64_t t = start[e]; t < end[e]; ++t)
      if (a->row_index[t] < 0 || a->row_index[t] >= a->batch) flags |= ORACLE_BAD_ROW_INDEX;
  return flags;
}

enum { NBLK = 64 };

int oracle_gmmfr(const oracle_args* a, double* out64, double* absb) {
  const int64_t M = a->M, K = a->K, N = a->N, E = a->E;
  int64_t* start = (int64_t*)malloc(sizeof(int64_t) * (size_t)(E > 0 ? E : 1));
  int64_t* end = (int64_t*)malloc(sizeof(int64_t) * (size_t)(E > 0 ? E : 1));
  int flags = oracle_expert_ranges(a, start, end);
  flags |= row_flags(a, start, end);
  (void)M;

  for (int64_t i = 0; i < a->batch * N; ++i) {
    out64[i] = (double)a->out_init[i];
    absb[i] = 0.0;
  }

  const int64_t nblocks = (N + NBLK - 1) / NBLK;
  for (int64_t e = 0; e < E; ++e) {
    if (start[e] >= end[e]) continue;
    /* Each thread owns a block of output columns and walks the expert's tokens
     * in ascending order, so every out64 element sees its additions in
     * ascending token order. */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t nb = 0; nb < nblocks; ++nb) {
      const int64_t n0 = nb * NBLK;
      const int64_t nn = (N - n0) < NBLK ? (N - n0) : NBLK;
      double* w = (double*)malloc(sizeof(double) * (size_t)(K * NBLK + 1));
      double* arow = (double*)malloc(sizeof(double) * (size_t)(K + 1));
      double acc[NBLK], ab[NBLK];
      /* dequantised weights of this expert for columns [n0, n0+nn) */
      for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < nn; ++j) w[k * NBLK + j] = weight_value(a, e, k, n0 + j);
      for (int64_t t = start[e]; t < end[e]; ++t) {
        const int64_t r = a->row_index[t];
        if (r < 0 || r >= a->batch) continue;
        const double lg = a->logit ? (double)a->logit[t] : 1.0;
        for (int64_t k = 0; k < K; ++k) arow[k] = token_value(a, t, k);
        for (int64_t j = 0; j < nn; ++j) acc[j] = ab[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
          const double av = arow[k];
          for (int64_t j = 0; j < nn; ++j) {
            const double p = av * w[k * NBLK + j];
            acc[j] += p;
            ab[j] += fabs(p);
          }
        }
        for (int64_t j = 0; j < nn; ++j) {
          const double b = a->bias ? oracle_decode_bf16(a->bias[e * N + n0 + j]) : 0.0;
          out64[r * N + n0 + j] += lg * (acc[j] + b);
          absb[r * N + n0 + j] += fabs(lg) * (ab[j] + fabs(b));
        }
      }
      free(w);
      free(arow);
    }
  }

  if (a->shared_input) {
    for (int64_t i = 0; i < a->shared_rows; ++i) {
      const int64_t r = a->shared_offset + i;
      if (r < 0 || r >= a->batch) continue;
      for (int64_t n = 0; n < N; ++n)
        out64[r * N + n] += a->shared_weight * oracle_decode_bf16(a->shared_input[i * N + n]);
    }
  }
  free(start);
  free(end);
  return flags;
}

int oracle_gmmfr_sampled(const oracle_args* a, int64_t n_samples, const int64_t* rows,
                         const int64_t* cols, double* out_vals, double* absb_vals) {
  const int64_t K = a->K, N = a->N, E = a->E;
  int64_t* start = (int64_t*)malloc(sizeof(int64_t) * (size_t)(E > 0 ? E : 1));
  int64_t* end = (int64_t*)malloc(sizeof(int64_t) * (size_t)(E > 0 ? E : 1));
  int flags = oracle_expert_ranges(a, start, end);
  flags |= row_flags(a, start, end);

#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t i = 0; i < n_samples; ++i) {
    const int64_t r = rows[i], n = cols[i];
    double v = (double)a->out_init[r * N + n];
    double bnd = 0.0;
    for (int64_t e = 0; e < E; ++e) {
      for (int64_t t = start[e]; t < end[e]; ++t) {
        if (a->row_index[t] != r) continue;
        const double lg = a->logit ? (double)a->logit[t] : 1.0;
        double acc = 0.0, ab = 0.0;
        for (int64_t k = 0; k < K; ++k) {
          const double p = token_value(a, t, k) * weight_value(a, e, k, n);
          acc += p;
          ab += fabs(p);
        }
        const double b = a->bias ? oracle_decode_bf16(a->bias[e * N + n]) : 0.0;
        v += lg * (acc + b);
        bnd += fabs(lg) * (ab + fabs(b));
      }
    }
    if (a->shared_input && r >= a->shared_offset && r < a->shared_offset + a->shared_rows)
      v += a->shared_weight * oracle_decode_bf16(a->shared_input[(r - a->shared_offset) * N + n]);
    out_vals[i] = v;
    absb_vals[i] = bnd;
  }
  free(start);
  free(end);
  return flags;
}
