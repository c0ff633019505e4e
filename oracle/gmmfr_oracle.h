/*
 * CPU oracle for MXFP8 grouped-matmul-finalize-routing.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  It shares nothing with
 * the CUDA path.
 *
 * Every value is decoded exactly and accumulated in IEEE double.
 * Layouts are those of the operator's input table ("grouped_matmul_finalize_routing
 * 的 MXFP8 实现与精度验证", section 3.1), all row-major and contiguous.
 */
#ifndef GMMFR_ORACLE_H
#define GMMFR_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element formats; E2M1 (OCP FP4) is stored two per byte, the even element in
 * the low nibble, along the row's contiguous dimension (K for x1 and a
 * transposed x2, N for a non-transposed x2) */
enum { ORACLE_E4M3 = 0, ORACLE_E5M2 = 1, ORACLE_E2M1 = 2 };

/* error flags returned by the oracle (the readings of invalid input) */
enum {
  ORACLE_BAD_GROUP_LIST = 1, /* negative count, decreasing prefix sum, or total > M */
  ORACLE_BAD_ROW_INDEX = 2   /* a routed token's row_index outside [0, batch) */
};

typedef struct {
  int64_t M, K, N, E, batch;
  int32_t x1_fmt, x2_fmt;
  int32_t transpose_x2;      /* x2 is [E,N,K] and scale [N,ceil(K/64),2] */
  int32_t scale_per_expert;  /* scale has a leading [E] dimension */
  int32_t group_list_type;   /* 0: prefix sums, 1: counts */
  int32_t _pad;
  const uint8_t* x1;             /* [M,K] */
  const uint8_t* x2;             /* [E,K,N] or [E,N,K] */
  const uint8_t* scale;          /* [(E,)ceil(K/64),N,2] or [(E,)N,ceil(K/64),2] */
  const uint8_t* pertoken_scale; /* [M,ceil(K/64),2] */
  const int64_t* group_list;     /* [E] */
  const float* logit;            /* [M] or NULL (weight 1) */
  const int64_t* row_index;      /* [M] */
  const uint16_t* shared_input;  /* [shared_rows,N] bf16 bits, or NULL */
  int64_t shared_rows;
  int64_t shared_offset;
  double shared_weight;
  const float* out_init;         /* [batch,N] */
  const uint16_t* bias;          /* [E,N] bf16 bits, or NULL */
} oracle_args;

/* Decoders of single codes, exposed so the tests can pin them. */
double oracle_decode_fp8(int fmt, uint32_t code);
double oracle_decode_e8m0(uint32_t code);
double oracle_decode_bf16(uint32_t bits);

/* Expert token ranges [start[e], end[e]) from group_list; returns error flags. */
int oracle_expert_ranges(const oracle_args* a, int64_t* start, int64_t* end);

/* Full result: out64[batch,N] and absb[batch,N] = sum over contributions of
 * |logit|*sum_k|a_k*b_k|.  Returns error flags. */
int oracle_gmmfr(const oracle_args* a, double* out64, double* absb);

/* Selected elements only: out_vals[i] and absb_vals[i] for (rows[i], cols[i]).
 * Same arithmetic, same order, as oracle_gmmfr.  Returns error flags. */
int oracle_gmmfr_sampled(const oracle_args* a, int64_t n_samples, const int64_t* rows,
                         const int64_t* cols, double* out_vals, double* absb_vals);

int oracle_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
