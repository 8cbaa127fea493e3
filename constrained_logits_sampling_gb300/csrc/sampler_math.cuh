// Exact per-token arithmetic of the sampler (device side).
//
// Every function here is either exact IEEE single-precision arithmetic (one correctly
// rounded operation per step, no contraction) or integer arithmetic, so the decisions
// that turn floats into integers (kept set, sampled id) do not depend on the order in
// which the GPU visits tokens.  Page references: "SGLang source teardown (10):
// Sampling, Grammar and structured output" (SGLang page), "GLM-5.3 inference (7):
// output side" (GLM page).
#pragma once

#include <cfloat>
#include <cmath>
#include <cstdint>

namespace clsample {

constexpr float kGreedyEps = 1e-5f;  // temperature below this is greedy (GLM page, "Sampling")

// Non-finite logits: NaN -> -inf (never drawn), +inf -> FLT_MAX, -inf -> -FLT_MAX, so the
// row stays samplable (SGLang page, "_preprocess_logits").
__device__ __forceinline__ float sanitize(float v) {
  if (v != v) return -INFINITY;
  return fminf(fmaxf(v, -FLT_MAX), FLT_MAX);
}

// An overflow of the penalty / bias arithmetic folds back like sanitising, except that
// -inf stays -inf (the token is out).
__device__ __forceinline__ float guard(float v) {
  if (v != v) return -INFINITY;
  return v == INFINITY ? FLT_MAX : v;
}

// Frequency / presence penalties (additive) then the repetition penalty (divide a
// positive logit, multiply a non-positive one), for a token seen `cnt` > 0 times
// (SGLang page, "Order semantics of the penalties").
__device__ __forceinline__ float apply_penalties(float z, uint32_t cnt, float freq, float pres, float rep) {
  z = __fsub_rn(z, __fmul_rn(freq, (float)cnt));
  z = __fsub_rn(z, pres);
  return (z > 0.0f) ? __fdiv_rn(z, rep) : __fmul_rn(z, rep);
}

// Order-preserving key of a float (larger value -> larger key); -0 folds onto +0.
__device__ __forceinline__ uint32_t fkey(float x) {
  uint32_t b = __float_as_uint(x == 0.0f ? 0.0f : x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t k) {
  uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(b);
}

// Tempered logit y = fl32(fl32(z - m) * fl32(1/T)) of a candidate (z > -inf).
__device__ __forceinline__ float y_of(float z, float m, float invT) {
  float y = __fmul_rn(__fsub_rn(z, m), invT);
  return y == 0.0f ? 0.0f : y;
}

// exp32: single-precision e^y for y <= 0, the weight the top-p cut sums.  Cody-Waite
// reduction y = n*ln2 + r (ln2 split into a 15-bit head and a tail), degree-7 Taylor
// polynomial of e^r by Horner's rule with fused multiply-adds, scaling by 2^n.  Each
// step is one correctly rounded IEEE operation.  e^-32 lies below the 2^-40 resolution
// of the fixed-point weights, so y < -32 gives 0.
__device__ __forceinline__ float exp32(float y) {
  if (!(y >= -32.0f)) return 0.0f;
  const float n = rintf(__fmul_rn(y, 0x1.715476p+0f));
  float r = __fmaf_rn(-n, 0x1.62e4p-1f, y);
  r = __fmaf_rn(-n, 0x1.7f7d1cp-20f, r);
  float q = 1.0f / 5040.0f;
  q = __fmaf_rn(q, r, 1.0f / 720.0f);
  q = __fmaf_rn(q, r, 1.0f / 120.0f);
  q = __fmaf_rn(q, r, 1.0f / 24.0f);
  q = __fmaf_rn(q, r, 1.0f / 6.0f);
  q = __fmaf_rn(q, r, 0.5f);
  q = __fmaf_rn(q, r, 1.0f);
  q = __fmaf_rn(q, r, 1.0f);
  // q * 2^n is exact: n >= -47, so 2^n is a normal float and the product stays normal
  return __fmul_rn(q, __int_as_float(((int)n + 127) << 23));
}

// Top-p weight of a token in 2^-40 fixed point, rounded down.  Sums of these are exact
// and independent of the summation order.
__device__ __forceinline__ unsigned long long weight_fx(float y) {
  return __float2ull_rz(__fmul_rn(exp32(y), 0x1p40f));
}

// ceil(p * W) exactly for p in (0, 1]: p = pm * 2^-s with a 24-bit integer pm, and the
// 88-bit product W * pm is kept in two 64-bit halves.  A token is kept by top-p iff the
// mass of the strictly more probable tokens is below this bound (SGLang page, "The maths
// of the three cuts": S_p).
__device__ inline unsigned long long ceil_scaled(unsigned long long W, float p) {
  int e;
  const float f = frexpf(p, &e);
  const unsigned long long pm = (unsigned long long)ldexpf(f, 24);
  const int s = 24 - e;
  const unsigned long long lo = W * pm;
  const unsigned long long hi = __umul64hi(W, pm);
  if (s >= 128) return (lo | hi) ? 1ull : 0ull;
  unsigned long long add_lo, add_hi;
  if (s >= 64) {
    add_lo = ~0ull;
    add_hi = (s == 64) ? 0ull : ((1ull << (s - 64)) - 1ull);
  } else {
    add_lo = (1ull << s) - 1ull;
    add_hi = 0ull;
  }
  const unsigned long long sum_lo = lo + add_lo;
  const unsigned long long carry = sum_lo < lo ? 1ull : 0ull;
  const unsigned long long sum_hi = hi + add_hi + carry;
  if (s >= 64) return s == 64 ? sum_hi : (sum_hi >> (s - 64));
  if (s == 0) return sum_lo;
  return (sum_lo >> s) | (sum_hi << (64 - s));
}

// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11).
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    if (i) {
      k.x += 0x9E3779B9u;
      k.y += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
  }
  return c;
}

// The four race uniforms of tokens 4q .. 4q+3 of a request: Philox at counter
// (q, position low, position high, 0) under the request's seed.
__device__ __forceinline__ uint4 race_words(uint32_t q, unsigned long long seed, unsigned long long pos) {
  return philox4x32_10(make_uint4(q, (uint32_t)pos, (uint32_t)(pos >> 32), 0u),
                       make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
}

__device__ __forceinline__ uint32_t pick_word(uint4 x, int j) {
  return j == 0 ? x.x : j == 1 ? x.y : j == 2 ? x.z : x.w;
}

// U in (0, 1) from one Philox output word: (top 23 bits + 1/2) / 2^23, exact in fp32.
__device__ __forceinline__ float word_to_uniform(uint32_t x) {
  return __fmul_rn(__fadd_rn(__uint2float_rn(x >> 9), 0.5f), 0x1p-23f);
}

// Race score of a kept token: y - ln E with E = -ln U, the Gumbel form of
// argmax p_i / E_i (exponential race).
__device__ __forceinline__ float race_score(float y, uint32_t x) {
  const float e = -logf(word_to_uniform(x));
  return __fsub_rn(y, logf(e));
}

// (value, id) order used for every argmax: larger value, then lower id.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Fast race score: y - ln(-ln U) with hardware logarithms, -ln U by its series where U is
// close to 1 (1 - U is exact there).  Within about 1e-4 of race_score for every U the
// Philox layout produces; a token pays for the exact score only if its fast score is
// within kFastTol of the best exact score so far.
constexpr float kFastTol = 1e-3f;
// Largest race bonus -ln(-ln U) over the uniforms Philox words give: U <= 1 - 2^-24,
// so -ln U >= 5.96e-8 and the bonus is at most 16.636.
constexpr float kGumbelMax = 16.7f;
__device__ __forceinline__ float fast_race(float y, uint32_t x) {
  const float u = word_to_uniform(x);
  const float d = 1.0f - u;
  const float e = d < 0.125f ? d * (1.0f + d * (0.5f + d * (0.33333334f + d * (0.25f + d * 0.2f)))) : -__logf(u);
  return y - __logf(e);
}

__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

}  // namespace clsample
