/* Plain CPU oracle of the batched constrained logits sampler.
 *
 * TEST INFRASTRUCTURE ONLY: only the tests, the smoke check and the benchmark's
 * CPU-baseline / reference arm load this file's library.  It shares no code, header,
 * table or constant with the CUDA library.
 *
 * One row at a time, with dense V-sized arrays and a full sort wherever a rank or a
 * cumulative mass is needed.  The steps follow the pages in their own order:
 *
 *   1. sanitise non-finite logits            SGLang source teardown (10), "_preprocess_logits"
 *   2. additive penalties, then scaling       same page, "Order semantics of the penalties"
 *   3. logit_bias, duplicate ids: last wins   same page, "Why logit_bias is built from triples"
 *   4. grammar bitmask: bit 0 -> -inf         same page, "Bitmask: one int32 covers 32 tokens"
 *   5. greedy iff T < 1e-5 or top_k <= 1      same page, "Field groups" (is_all_greedy: top_k <= 1);
 *                                             GLM-5.3 output side, "Sampling" (temperature < 1e-5)
 *   6. temperature, softmax statistics        SGLang teardown (10), "The maths of the three cuts"
 *   7. top-k -> top-p -> min-p, sequentially  same section (S_k, S_p, S_m and the FlashInfer min-p order)
 *   8. a draw keyed by (seed, position)       same page, "Call site" (position drives the seed);
 *                                             GLM-5.3 output side (one generator per request)
 *   9. logprob of the sampled token           same page, "Numerical consistency of logprobs"
 *
 * Precision.  Steps 1-6 use IEEE single precision exactly as written (build with
 * -ffp-contract=off so no multiply-add is fused).  The softmax normaliser and the
 * logprob are double.  Two decisions that floating point turns into integers are taken
 * in single precision, the precision the pages give the sampler (logits are cast to
 * FP32 before the softmax, GLM-5.3 output side): the top-p weights (exp32 below, summed
 * exactly in 2^-40 fixed point) and the race scores.
 */
#define _GNU_SOURCE
#include "oracle.h"

#include <float.h>
#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORACLE_OK = 0, ORACLE_OVERFLOW = 1, ORACLE_INVALID = 2 };

/* ------------------------------------------------------------------ random numbers */

/* Philox4x32 with 10 rounds, as published by Salmon, Moraes, Dror and Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3" (SC'11): each round multiplies
 * counter words 0 and 2 by two fixed odd constants, swaps the halves of the products
 * and xors in the other counter words and the key; the key is bumped by two Weyl
 * constants between rounds. */
void cls_oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
    uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    uint32_t n1 = (uint32_t)p1;
    uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    uint32_t n3 = (uint32_t)p0;
    c0 = n0;
    c1 = n1;
    c2 = n2;
    c3 = n3;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

/* The per-token uniform of a request.  The pages only ask that a request's random
 * stream be keyed by the request (seed) and the position of the token being sampled,
 * independent of the batch it is in.  This build fixes the layout: key = seed,
 * counter = (token / 4, position low, position high, 0), output word token % 4, and
 * U = (top 23 bits + 1/2) / 2^23, which is exact in float and lies in (0, 1). */
float cls_oracle_uniform(uint64_t seed, int64_t position, int64_t token) {
  uint64_t pos = (uint64_t)position;
  uint32_t ctr[4] = {(uint32_t)((uint64_t)token >> 2), (uint32_t)pos, (uint32_t)(pos >> 32), 0u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  cls_oracle_philox4x32_10(ctr, key, out);
  uint32_t x = out[token & 3];
  float u = (float)(x >> 9) + 0.5f;
  return u * 0x1p-23f;
}

/* ------------------------------------------------------------------ top-p weights */

/* exp32(y) for y <= 0: the single-precision exponential that the top-p weights use.
 * Cody-Waite reduction y = n*ln2 + r with |r| <= ln2/2 (ln2 split into a 15-bit head and
 * a tail), then the degree-7 Taylor polynomial of e^r evaluated by Horner's rule with
 * fused multiply-adds, then scaling by 2^n.  Every step is one correctly rounded IEEE
 * operation, so any IEEE machine gets the same bits.  Below y = -32 the weight is 0:
 * e^-32 is under the 2^-40 resolution of the fixed-point sums. */
float cls_oracle_exp32(float y) {
  if (!(y >= -32.0f)) return 0.0f;
  float n = rintf(y * 0x1.715476p+0f); /* y * log2(e) */
  float r = fmaf(-n, 0x1.62e4p-1f, y);
  r = fmaf(-n, 0x1.7f7d1cp-20f, r);
  float q = 1.0f / 5040.0f;
  q = fmaf(q, r, 1.0f / 720.0f);
  q = fmaf(q, r, 1.0f / 120.0f);
  q = fmaf(q, r, 1.0f / 24.0f);
  q = fmaf(q, r, 1.0f / 6.0f);
  q = fmaf(q, r, 0.5f);
  q = fmaf(q, r, 1.0f);
  q = fmaf(q, r, 1.0f);
  return ldexpf(q, (int)n);
}

/* The weight of a token in 2^-40 fixed point, rounded down. */
uint64_t cls_oracle_weight_fx(float y) {
  float w = cls_oracle_exp32(y);
  return (uint64_t)(w * 0x1p40f);
}

/* ceil(p * W) exactly, for p in (0, 1]: p = pm / 2^s with pm a 24-bit integer. */
uint64_t cls_oracle_ceil_scaled(uint64_t W, float p) {
  int e;
  float f = frexpf(p, &e);
  uint32_t pm = (uint32_t)ldexpf(f, 24);
  int s = 24 - e;
  unsigned __int128 prod = (unsigned __int128)W * pm;
  if (s >= 128) return prod != 0 ? 1u : 0u;
  unsigned __int128 one = 1;
  return (uint64_t)((prod + ((one << s) - 1)) >> s);
}

/* ------------------------------------------------------------------ one row */

typedef struct {
  float* z;
  float* y;
  int32_t* count;
  float* bias;
  unsigned char* has_bias;
  unsigned char* keep;
  float* sorted;
  struct yid {
    float y;
    int32_t id;
  } * order;
} row_scratch;

static int cmp_float_desc(const void* a, const void* b) {
  float x = *(const float*)a, y = *(const float*)b;
  return (x < y) - (x > y);
}

static int cmp_yid_desc(const void* a, const void* b) {
  const struct yid* p = (const struct yid*)a;
  const struct yid* q = (const struct yid*)b;
  if (p->y != q->y) return (p->y < q->y) - (p->y > q->y);
  return (p->id > q->id) - (p->id < q->id);
}

static float load_logit(const cls_oracle_args* a, int r, int i) {
  if (a->logits_is_bf16) {
    const uint16_t* row = (const uint16_t*)a->logits + (int64_t)r * a->row_stride;
    uint32_t bits = (uint32_t)row[i] << 16;
    float v;
    memcpy(&v, &bits, sizeof v);
    return v;
  }
  return ((const float*)a->logits)[(int64_t)r * a->row_stride + i];
}

/* Step 1.  The pages replace non-finite logits by a small finite number so that the
 * row stays samplable.  Reading taken here: NaN becomes -inf (never sampled), +inf
 * becomes the largest float and -inf the most negative float. */
static float sanitize(float v) {
  if (isnan(v)) return -INFINITY;
  if (v == INFINITY) return FLT_MAX;
  if (v == -INFINITY) return -FLT_MAX;
  return v;
}

static void write_row(const cls_oracle_args* a, int r, int status, int token, double lp, int kept,
                      float cut, float gap, float best, double lp_orig, double lp_kept) {
  a->tokens[r] = token;
  if (a->logprobs) a->logprobs[r] = lp;
  if (a->logprobs_orig) a->logprobs_orig[r] = lp_orig;
  if (a->logprobs_kept) a->logprobs_kept[r] = lp_kept;
  if (a->status) a->status[r] = status;
  if (a->kept_count) a->kept_count[r] = kept;
  if (a->cut) a->cut[r] = cut;
  if (a->race_gap) a->race_gap[r] = gap;
  if (a->race_best) a->race_best[r] = best;
}

static void sample_row(const cls_oracle_args* a, int r, row_scratch* s) {
  const int V = a->V;
  int status = ORACLE_OK;
  float T = a->temperatures ? a->temperatures[r] : 1.0f;
  int k = a->top_ks ? a->top_ks[r] : -1;
  float p = a->top_ps ? a->top_ps[r] : 1.0f;
  float mp = a->min_ps ? a->min_ps[r] : 0.0f;
  float rep = a->rep ? a->rep[r] : 1.0f;
  float freq = a->freq ? a->freq[r] : 0.0f;
  float pres = a->pres ? a->pres[r] : 0.0f;
  uint64_t seed = a->seeds ? a->seeds[r] : 0u;
  int64_t pos = a->positions ? a->positions[r] : a->step;

  if (isnan(T) || T == INFINITY) status = ORACLE_INVALID;
  if (k < -1) status = ORACLE_INVALID;
  if (!(p > 0.0f && p <= 1.0f)) status = ORACLE_INVALID;
  if (!(mp >= 0.0f && mp <= 1.0f)) status = ORACLE_INVALID;
  if (!(rep > 0.0f) || isinf(rep) || !isfinite(freq) || !isfinite(pres)) status = ORACLE_INVALID;

  /* 1. sanitise */
  for (int i = 0; i < V; ++i) s->z[i] = sanitize(load_logit(a, r, i));

  /* 2. penalties: c_i = occurrences of i in the row's history.  Additive first
   *    (z - freq*c - pres), then the repetition scaling (divide a positive logit,
   *    multiply a non-positive one). */
  memset(s->count, 0, sizeof(int32_t) * (size_t)V);
  if (a->hist_offs) {
    int32_t lo = a->hist_offs[r], hi = a->hist_offs[r + 1];
    if (lo < 0 || hi < lo) {
      status = ORACLE_INVALID;
    } else {
      for (int32_t j = lo; j < hi; ++j) {
        int32_t id = a->hist_ids[j];
        if (id < 0 || id >= V)
          status = ORACLE_INVALID;
        else
          s->count[id] += 1;
      }
    }
  }
  for (int i = 0; i < V; ++i) {
    int32_t c = s->count[i];
    if (c > 0) {
      float z = s->z[i];
      z = z - freq * (float)c;
      z = z - pres;
      z = (z > 0.0f) ? z / rep : z * rep;
      s->z[i] = z;
    }
  }

  /* 3. logit_bias: for a repeated id the last entry of the row wins */
  memset(s->has_bias, 0, (size_t)V);
  if (a->bias_offs) {
    int32_t lo = a->bias_offs[r], hi = a->bias_offs[r + 1];
    if (lo < 0 || hi < lo) {
      status = ORACLE_INVALID;
    } else {
      for (int32_t j = lo; j < hi; ++j) {
        int32_t id = a->bias_ids[j];
        float b = a->bias_vals[j];
        if (id < 0 || id >= V || isnan(b)) {
          status = ORACLE_INVALID;
        } else {
          s->bias[id] = b;
          s->has_bias[id] = 1;
        }
      }
    }
  }
  for (int i = 0; i < V; ++i)
    if (s->has_bias[i]) s->z[i] = s->z[i] + s->bias[i];

  /* requested token ids (logprobs of given tokens): an id outside the vocabulary makes
   * the row INVALID, like the other id lists */
  int32_t tlo = 0, thi = 0;
  if (a->tid_offs) {
    tlo = a->tid_offs[r];
    thi = a->tid_offs[r + 1];
    if (tlo < 0 || thi < tlo) {
      status = ORACLE_INVALID;
      thi = tlo = 0;
    } else {
      for (int32_t j = tlo; j < thi; ++j)
        if (a->tid_ids[j] < 0 || a->tid_ids[j] >= V) status = ORACLE_INVALID;
    }
  }
  if (a->tid_logprobs)
    for (int32_t j = tlo; j < thi; ++j) a->tid_logprobs[j] = -INFINITY;

  /* top-N most probable tokens: N in [0, min(32, stride)], else INVALID */
  int topn = 0;
  if (a->top_ns) {
    int32_t n = a->top_ns[r];
    if (n < 0 || n > CLS_ORACLE_TOP_N_MAX || n > a->top_n_stride) {
      status = ORACLE_INVALID;
    } else {
      topn = n;
      for (int j = 0; j < n; ++j) {
        a->top_ids[(int64_t)r * a->top_n_stride + j] = -1;
        a->top_logprobs[(int64_t)r * a->top_n_stride + j] = -INFINITY;
      }
    }
  }

  /* An overflow in steps 2-3 is folded back the same way as step 1 treats its
   * input, except that -inf stays -inf (the token is out). */
  for (int i = 0; i < V; ++i) {
    if (isnan(s->z[i])) s->z[i] = -INFINITY;
    else if (s->z[i] == INFINITY) s->z[i] = FLT_MAX;
  }

  /* 4. grammar bitmask: a 0 bit sets the logit to -inf */
  if (a->bitmask) {
    const int32_t* words = a->bitmask + (int64_t)r * a->bitmask_row_stride;
    for (int i = 0; i < V; ++i) {
      uint32_t w = (uint32_t)words[i >> 5];
      if (((w >> (i & 31)) & 1u) == 0u) s->z[i] = -INFINITY;
    }
  }
  if (a->transformed) memcpy(a->transformed + (int64_t)r * V, s->z, sizeof(float) * (size_t)V);

  if (status != ORACLE_OK) {
    write_row(a, r, status, -1, -INFINITY, 0, -INFINITY, INFINITY, -INFINITY, -INFINITY, -INFINITY);
    return;
  }

  /* candidates: tokens whose transformed logit is above -inf */
  int n_cand = 0;
  float m = -INFINITY;
  int arg = -1;
  for (int i = 0; i < V; ++i) {
    if (s->z[i] > -INFINITY) {
      ++n_cand;
      if (s->z[i] > m) { /* strict: ties keep the lowest id */
        m = s->z[i];
        arg = i;
      }
    }
  }
  if (n_cand == 0) {
    write_row(a, r, ORACLE_INVALID, -1, -INFINITY, 0, -INFINITY, INFINITY, -INFINITY, -INFINITY, -INFINITY);
    return;
  }

  /* 5./6. greedy decision, temperature and the softmax normaliser */
  int greedy = (T < 1e-5f) || k == 0 || k == 1 || (a->mode & CLS_ORACLE_SCORE_ONLY);
  float Teff = (T >= 1e-5f) ? T : 1.0f;
  float invT = 1.0f / Teff;
  double S = 0.0;
  for (int i = 0; i < V; ++i) {
    if (s->z[i] > -INFINITY) {
      s->y[i] = (s->z[i] - m) * invT;
      S += exp((double)s->y[i]);
    } else {
      s->y[i] = -INFINITY;
    }
  }
  double logS = log(S);
  /* the N most probable tokens (SGLang page, the output container's top logprobs):
   * candidates ordered by z' descending -- the same order as y, which is monotone in z'
   * -- with equal z' by id ascending; fewer than N candidates leave -1 / -inf */
  if (topn > 0) {
    int n = 0;
    for (int i = 0; i < V; ++i)
      if (s->z[i] > -INFINITY) {
        s->order[n].y = s->z[i];
        s->order[n].id = i;
        ++n;
      }
    qsort(s->order, (size_t)n, sizeof(s->order[0]), cmp_yid_desc);
    for (int j = 0; j < topn && j < n; ++j) {
      int id = s->order[j].id;
      a->top_ids[(int64_t)r * a->top_n_stride + j] = id;
      a->top_logprobs[(int64_t)r * a->top_n_stride + j] = (double)s->y[id] - logS;
    }
  }
  /* logprobs of the requested ids, under the same distribution as the drawn token's:
   * y_id - ln S (-inf for a masked id) */
  if (a->tid_logprobs)
    for (int32_t j = tlo; j < thi; ++j) {
      int id = a->tid_ids[j];
      a->tid_logprobs[j] = s->z[id] > -INFINITY ? (double)s->y[id] - logS : -INFINITY;
    }
  /* the original (pre-temperature) distribution: log_softmax of z' at T = 1
   * (SGLang page, "Numerical consistency of logprobs": logprobs before temperature) */
  double S1 = 0.0;
  for (int i = 0; i < V; ++i)
    if (s->z[i] > -INFINITY) {
      float d = s->z[i] - m;
      S1 += exp((double)d);
    }
  float d_arg = s->z[arg] - m;
  if (greedy) {
    /* the kept set of a greedy row is the token alone: its renormalised logprob is 0 */
    write_row(a, r, ORACLE_OK, arg, (double)s->y[arg] - logS, 1, s->y[arg], INFINITY, -INFINITY,
              (double)d_arg - log(S1), 0.0);
    return;
  }

  /* 7a. top-k: keep the tokens whose probability is at least the k-th largest one
   *     (counting repeats); every token tied with the k-th value stays. */
  for (int i = 0; i < V; ++i) s->keep[i] = (s->z[i] > -INFINITY);
  if (k >= 2 && k < n_cand) {
    int n = 0;
    for (int i = 0; i < V; ++i)
      if (s->keep[i]) s->sorted[n++] = s->y[i];
    qsort(s->sorted, (size_t)n, sizeof(float), cmp_float_desc);
    float tk = s->sorted[k - 1];
    for (int i = 0; i < V; ++i)
      if (s->keep[i] && s->y[i] < tk) s->keep[i] = 0;
  }

  /* 7b'. joint mode: top-p over the whole candidate set, intersected with the top-k
   *      set.  Token i passes iff the mass of the candidates strictly more probable than
   *      i is below p times the mass of all candidates. */
  int joint = (a->mode & CLS_ORACLE_JOINT) != 0;
  if (joint && p < 1.0f) {
    int n = 0;
    uint64_t W = 0;
    for (int i = 0; i < V; ++i) {
      if (s->z[i] > -INFINITY) {
        s->order[n].y = s->y[i];
        s->order[n].id = i;
        ++n;
        W += cls_oracle_weight_fx(s->y[i]);
      }
    }
    qsort(s->order, (size_t)n, sizeof(s->order[0]), cmp_yid_desc);
    uint64_t C = cls_oracle_ceil_scaled(W, p);
    uint64_t above = 0; /* mass of the candidates strictly above the current level */
    int j = 0;
    while (j < n) {
      int j2 = j;
      uint64_t level_mass = 0;
      while (j2 < n && s->order[j2].y == s->order[j].y) {
        level_mass += cls_oracle_weight_fx(s->order[j2].y);
        ++j2;
      }
      if (!(above < C))
        for (int t = j; t < j2; ++t) s->keep[s->order[t].id] = 0;
      above += level_mass;
      j = j2;
    }
  }

  /* 7b. top-p on the renormalised top-k set: token i stays iff the mass of the
   *     strictly more probable tokens is below p times the set's mass, so tokens of
   *     equal probability are all in or all out.  Weights are exp32(y) in 2^-40 fixed
   *     point, so the sums are exact and the comparison with ceil(p * W) is exact. */
  if (!joint && p < 1.0f) {
    int n = 0;
    uint64_t W = 0;
    for (int i = 0; i < V; ++i) {
      if (s->keep[i]) {
        s->order[n].y = s->y[i];
        s->order[n].id = i;
        ++n;
        W += cls_oracle_weight_fx(s->y[i]);
      }
    }
    qsort(s->order, (size_t)n, sizeof(s->order[0]), cmp_yid_desc);
    uint64_t C = cls_oracle_ceil_scaled(W, p);
    uint64_t above = 0;
    int j = 0;
    while (j < n) {
      int j2 = j;
      uint64_t level_mass = 0;
      while (j2 < n && s->order[j2].y == s->order[j].y) {
        level_mass += cls_oracle_weight_fx(s->order[j2].y);
        ++j2;
      }
      if (!(above < C)) {
        for (int t = j; t < n; ++t) s->keep[s->order[t].id] = 0;
        break;
      }
      above += level_mass;
      j = j2;
    }
  }

  /* 7c. min-p: p_i >= p_max * min_p, i.e. y_i >= ln(min_p) since y_max = 0 */
  if (mp > 0.0f) {
    float L = (float)log((double)mp);
    for (int i = 0; i < V; ++i)
      if (s->keep[i] && !(s->y[i] >= L)) s->keep[i] = 0;
  }

  /* 8. exponential race over the kept set: token = argmax_i w_i / E_i with
   *    E_i = -ln U_i, i.e. argmax of y_i - ln E_i; ties go to the lowest id. */
  int kept = 0, tok = -1;
  float best = -INFINITY, second = -INFINITY, cut = INFINITY;
  double SK = 0.0; /* mass of the kept set, for the renormalised logprob */
  for (int i = 0; i < V; ++i) {
    if (!s->keep[i]) continue;
    ++kept;
    SK += exp((double)s->y[i]);
    if (s->y[i] < cut) cut = s->y[i];
    float u = cls_oracle_uniform(seed, pos, i);
    float e = -logf(u);
    float score = s->y[i] - logf(e);
    if (score > best) {
      second = best;
      best = score;
      tok = i;
    } else if (score > second) {
      second = score;
    }
  }
  /* 9. logprob of the drawn token under the full (pre-truncation) distribution at T */
  /* the distribution the token was drawn from: softmax(y) renormalised over the kept
   * set (GLM page, "Sampling": the top-k/top-p sampler's processed logprobs) */
  float d_tok = s->z[tok] - m;
  write_row(a, r, ORACLE_OK, tok, (double)s->y[tok] - logS, kept, cut,
            kept > 1 ? best - second : INFINITY, best, (double)d_tok - log(S1), (double)s->y[tok] - log(SK));
}

/* ------------------------------------------------------------------ batch driver */

typedef struct {
  const cls_oracle_args* a;
  int tid, nthreads;
} worker_arg;

static void* worker(void* p) {
  worker_arg* w = (worker_arg*)p;
  const cls_oracle_args* a = w->a;
  size_t V = (size_t)(a->V > 0 ? a->V : 1);
  row_scratch s;
  s.z = (float*)malloc(V * sizeof(float));
  s.y = (float*)malloc(V * sizeof(float));
  s.count = (int32_t*)malloc(V * sizeof(int32_t));
  s.bias = (float*)malloc(V * sizeof(float));
  s.has_bias = (unsigned char*)malloc(V);
  s.keep = (unsigned char*)malloc(V);
  s.sorted = (float*)malloc(V * sizeof(float));
  s.order = (struct yid*)malloc(V * sizeof(struct yid));
  for (int r = w->tid; r < a->B; r += w->nthreads) sample_row(a, r, &s);
  free(s.z);
  free(s.y);
  free(s.count);
  free(s.bias);
  free(s.has_bias);
  free(s.keep);
  free(s.sorted);
  free(s.order);
  return NULL;
}

int cls_oracle_sample(const cls_oracle_args* a) {
  int nt = a->nthreads;
  if (nt <= 0) {
    cpu_set_t set;
    nt = 1;
    if (sched_getaffinity(0, sizeof set, &set) == 0) nt = CPU_COUNT(&set);
    if (nt <= 0) nt = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nt <= 0) nt = 1;
  }
  if (a->B > 0 && nt > a->B) nt = a->B;
  if (nt < 1) nt = 1;
  if (a->B <= 0) return nt;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
  worker_arg* wa = (worker_arg*)malloc(sizeof(worker_arg) * (size_t)nt);
  for (int t = 0; t < nt; ++t) {
    wa[t].a = a;
    wa[t].tid = t;
    wa[t].nthreads = nt;
  }
  for (int t = 1; t < nt; ++t) pthread_create(&th[t], NULL, worker, &wa[t]);
  worker(&wa[0]);
  for (int t = 1; t < nt; ++t) pthread_join(th[t], NULL);
  free(th);
  free(wa);
  return nt;
}
