/* CPU oracle for the batched constrained logits sampler.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline / reference arm may load this library.  It shares no code, header,
 * table or constant with the CUDA library; the two meet only through the seeded
 * input arrays the tests pass to both.
 *
 * Every pointer is a HOST pointer.  Optional inputs may be NULL (see oracle.c for
 * the defaults).  The oracle never fails on data: a row whose parameters or ids are
 * out of range gets status 2 (INVALID), token -1 and logprob -inf.
 */
#ifndef CLS_ORACLE_H
#define CLS_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t B, V;
  int32_t logits_is_bf16;          /* 0: float32 logits, 1: uint16 bfloat16 bit patterns */
  const void* logits;              /* [B, row_stride] */
  int64_t row_stride;              /* elements */
  const float* temperatures;       /* [B] or NULL (1.0) */
  const int32_t* top_ks;           /* [B] or NULL (-1 = whole vocabulary) */
  const float* top_ps;             /* [B] or NULL (1.0) */
  const float* min_ps;             /* [B] or NULL (0.0) */
  const float* rep;                /* [B] or NULL (1.0) */
  const float* freq;               /* [B] or NULL (0.0) */
  const float* pres;               /* [B] or NULL (0.0) */
  const int32_t* hist_offs;        /* [B+1] or NULL */
  const int32_t* hist_ids;
  const int32_t* bias_offs;        /* [B+1] or NULL */
  const int32_t* bias_ids;
  const float* bias_vals;
  const int32_t* bitmask;          /* [B, bitmask_row_stride] or NULL */
  int64_t bitmask_row_stride;      /* words */
  const uint64_t* seeds;           /* [B] or NULL (0) */
  const int64_t* positions;        /* [B] or NULL (step) */
  int64_t step;
  /* outputs */
  int32_t* tokens;                 /* [B] */
  double* logprobs;                /* [B] or NULL */
  int32_t* status;                 /* [B] or NULL */
  float* transformed;              /* [B, V] or NULL: z' */
  int32_t* kept_count;             /* [B] or NULL */
  float* cut;                      /* [B] or NULL: smallest y in the kept set */
  float* race_gap;                 /* [B] or NULL: best - second race score (+inf if one) */
  float* race_best;                /* [B] or NULL: best race score (-inf if none) */
  int32_t nthreads;                /* 0 = all online cores */
  double* logprobs_orig;           /* [B] or NULL: ln p(token) under softmax(z'), T = 1 */
  double* logprobs_kept;           /* [B] or NULL: ln p(token) renormalised over the kept set
                                      (0 for greedy rows: the kept set is the token alone) */
  int32_t mode;                    /* bit flags: CLS_ORACLE_JOINT, CLS_ORACLE_SCORE_ONLY */
  const int32_t* tid_offs;         /* [B+1] or NULL: per-row lists of requested token ids */
  const int32_t* tid_ids;
  double* tid_logprobs;            /* [tid_offs[B]] or NULL: ln p(id) at T, pre-truncation */
  const int32_t* top_ns;           /* [B] or NULL: how many most probable tokens to report */
  int32_t top_n_stride;            /* row stride of top_ids / top_logprobs */
  int32_t* top_ids;                /* [B, top_n_stride]: by z' descending, then id ascending */
  double* top_logprobs;            /* [B, top_n_stride]: ln p at T, pre-truncation */
} cls_oracle_args;

/* Largest N the top-N outputs accept per row (more, or more than the stride: INVALID). */
#define CLS_ORACLE_TOP_N_MAX 32

/* mode bits.  JOINT: top-p is taken over the whole distribution and intersected with the
 * top-k set (instead of top-p over the renormalised top-k set).  SCORE_ONLY: no draw;
 * every row takes the greedy route (argmax, its logprob) and only the logprobs of the
 * requested ids are of interest. */
#define CLS_ORACLE_JOINT 1
#define CLS_ORACLE_SCORE_ONLY 2

/* Runs the whole batch.  Returns the number of threads used (>= 1). */
int cls_oracle_sample(const cls_oracle_args* a);

/* Building blocks exposed for the oracle's own pins. */
void cls_oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
float cls_oracle_uniform(uint64_t seed, int64_t position, int64_t token);
float cls_oracle_exp32(float y);
uint64_t cls_oracle_weight_fx(float y);
uint64_t cls_oracle_ceil_scaled(uint64_t W, float p);

#ifdef __cplusplus
}
#endif
#endif
