// Batched constrained logits sampler for GB300 (sm_103a).
//
// One thread-block cluster samples one row.  The row's V logits are split into C
// contiguous slices ("chunks", a multiple of 32 tokens so that every CTA owns whole
// bitmask words); CTA `rank` of the cluster keeps its slice resident in shared memory
// for the whole call, so HBM sees every logit exactly once.  Row-wide quantities
// (max, argmax, softmax normaliser, radix-select histograms, race winners) are
// exchanged through distributed shared memory (DSMEM) between hardware cluster
// barriers.  Nothing is written to global memory except the per-row outputs.
//
// The arithmetic that decides integers (kept set, sampled id) is exact and identical on
// any IEEE machine: y = fl32(fl32(z' - m) * fl32(1/T)); top-k compares y; top-p sums the
// fixed-point weights floor(exp32(y) * 2^40) exactly and compares with ceil(p * W);
// min-p compares y with fl32(ln min_p).  The race score y - ln(-ln U) is fp32.
//
// Page references: "SGLang source teardown (10): Sampling, Grammar and structured
// output" (SGLang page) and "GLM-5.3 inference (7): output side" (GLM page).

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "clsample.h"

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kHashCap = 1024;  // distinct penalised/biased ids per CTA slice
constexpr uint32_t kEmpty = 0xFFFFFFFFu;
constexpr int kMaxCluster = 16;
constexpr float kGreedyEps = 1e-5f;

enum : int { kRowOk = 0, kRowOverflow = 1, kRowInvalid = 2 };
enum : int { kFlagInvalid = 1, kFlagOverflow = 2 };

struct Geometry {
  int C;      // CTAs per row (cluster size)
  int chunk;  // tokens per CTA, multiple of 32
  int smem;   // dynamic shared memory bytes per CTA
};

struct LaunchParams {
  clsample_args_t a;
  int C;
  int chunk;
  int vec_ok;  // logits rows are 16-byte (f32) / 8-byte (bf16) aligned for vector loads
};

// ---------------------------------------------------------------- shared memory layout

// Dynamic shared memory of one CTA (offsets in bytes from the base):
//   zs      f32[chunk]          transformed logits z' of the slice (padding = -inf)
//   modbits u32[chunk/32]       1 = token is penalised or biased (handled separately)
//   hkey    u32[kHashCap]       hash of the slice's penalised/biased local ids
//   hcnt    u32[kHashCap]       occurrences in the history
//   hbias   i32[kHashCap]       index of the last logit_bias entry for the id, or -1
//   hist_c  u32[2][256]         radix histogram, counts (double-buffered across passes)
//   hist_w  u64[2][256]         radix histogram, fixed-point weights
//   merged  u64[2][256]         cluster-merged counts and weights
struct Smem {
  float* zs;
  uint32_t* modbits;
  uint32_t* hkey;
  uint32_t* hcnt;
  int32_t* hbias;
  uint32_t* hist_c;
  unsigned long long* hist_w;
  unsigned long long* merged_c;
  unsigned long long* merged_w;
};

__host__ __device__ inline size_t smem_bytes_for(int chunk) {
  size_t b = 0;
  b += sizeof(float) * (size_t)chunk;
  b += sizeof(uint32_t) * (size_t)(chunk / 32);
  b += sizeof(uint32_t) * kHashCap * 3;
  b = (b + 15) & ~size_t(15);
  b += sizeof(uint32_t) * 2 * 256;
  b += sizeof(unsigned long long) * 2 * 256;
  b += sizeof(unsigned long long) * 2 * 256;
  return b;
}

__device__ inline Smem carve(unsigned char* base, int chunk) {
  Smem s;
  size_t off = 0;
  s.zs = reinterpret_cast<float*>(base + off);
  off += sizeof(float) * (size_t)chunk;
  s.modbits = reinterpret_cast<uint32_t*>(base + off);
  off += sizeof(uint32_t) * (size_t)(chunk / 32);
  s.hkey = reinterpret_cast<uint32_t*>(base + off);
  off += sizeof(uint32_t) * kHashCap;
  s.hcnt = reinterpret_cast<uint32_t*>(base + off);
  off += sizeof(uint32_t) * kHashCap;
  s.hbias = reinterpret_cast<int32_t*>(base + off);
  off += sizeof(int32_t) * kHashCap;
  off = (off + 15) & ~size_t(15);
  s.hist_c = reinterpret_cast<uint32_t*>(base + off);
  off += sizeof(uint32_t) * 2 * 256;
  s.hist_w = reinterpret_cast<unsigned long long*>(base + off);
  off += sizeof(unsigned long long) * 2 * 256;
  s.merged_c = reinterpret_cast<unsigned long long*>(base + off);
  off += sizeof(unsigned long long) * 256;
  s.merged_w = reinterpret_cast<unsigned long long*>(base + off);
  return s;
}

// Per-CTA values published to the other CTAs of the cluster.  Each exchange round has
// its own fields, so a fast CTA never overwrites a value a slow CTA is still reading.
struct Exchange {
  float m;          // slice max of z' (-inf if none)
  int arg;          // lowest global id reaching m (INT_MAX if none)
  float S;          // sum of 2^((z' - m) * c) over the slice's candidates
  int ncand;        // candidates (z' > -inf)
  int flags;        // kFlagInvalid | kFlagOverflow
  unsigned long long W;  // top-p: fixed-point mass of the slice's part of S_k
  float race_s;     // best race score of the slice
  int race_tok;     // its id (lowest id on ties)
  int kept;         // kept tokens in the slice
  float ymin;       // smallest y of a kept token in the slice
};

struct RowParams {
  float T, p, mp, rep, freq, pres;
  int k;
  unsigned long long seed;
  long long pos;
  int invalid;
};

// ---------------------------------------------------------------- scalar helpers

// Non-finite logits: NaN -> -inf (never drawn), +inf -> FLT_MAX, -inf -> -FLT_MAX
// (SGLang page, "_preprocess_logits": keep the row samplable).
__device__ __forceinline__ float sanitize(float v) {
  if (v != v) return -INFINITY;
  return fminf(fmaxf(v, -FLT_MAX), FLT_MAX);
}

// An overflow of the penalty/bias arithmetic folds back like sanitising, except that
// -inf stays -inf.
__device__ __forceinline__ float guard(float v) {
  if (v != v) return -INFINITY;
  return v == INFINITY ? FLT_MAX : v;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Order-preserving key of y (larger y -> larger key); -0 is folded onto +0.
__device__ __forceinline__ uint32_t ykey(float y) {
  uint32_t b = __float_as_uint(y == 0.0f ? 0.0f : y);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_to_y(uint32_t k) {
  uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(b);
}

// y = fl32(fl32(z - m) * invT), -inf for non-candidates.
__device__ __forceinline__ float y_of(float z, float m, float invT) {
  if (!(z > -INFINITY)) return -INFINITY;
  float y = __fmul_rn(__fsub_rn(z, m), invT);
  return y == 0.0f ? 0.0f : y;
}

// exp32: single-precision e^y for y <= 0 used by the top-p weights.  Cody-Waite
// reduction y = n*ln2 + r (ln2 split into a 15-bit head and a tail), degree-7 Taylor
// polynomial of e^r by Horner's rule with fused multiply-adds, scaling by 2^n.  Each
// step is one correctly rounded IEEE operation.  e^-32 is below the 2^-40 resolution
// of the weights, so y < -32 gives 0.
__device__ __forceinline__ float exp32(float y) {
  if (!(y >= -32.0f)) return 0.0f;
  float n = rintf(__fmul_rn(y, 0x1.715476p+0f));
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
  return ldexpf(q, (int)n);
}

__device__ __forceinline__ unsigned long long weight_fx(float y) {
  return __float2ull_rz(__fmul_rn(exp32(y), 0x1p40f));
}

// ceil(p * W) for p in (0, 1]: p = pm * 2^-s with a 24-bit integer pm.
__device__ inline unsigned long long ceil_scaled(unsigned long long W, float p) {
  int e;
  float f = frexpf(p, &e);
  unsigned long long pm = (unsigned long long)ldexpf(f, 24);
  int s = 24 - e;
  // prod = W * pm as a 128-bit value (hi:lo)
  unsigned long long lo = W * pm;
  unsigned long long hi = __umul64hi(W, pm);
  if (s >= 128) return (lo | hi) ? 1ull : 0ull;
  // add 2^s - 1 then shift right by s
  unsigned long long add_lo, add_hi;
  if (s >= 64) {
    add_lo = ~0ull;
    add_hi = (s == 64) ? 0ull : ((1ull << (s - 64)) - 1ull);
  } else {
    add_lo = (1ull << s) - 1ull;
    add_hi = 0ull;
  }
  unsigned long long sum_lo = lo + add_lo;
  unsigned long long carry = sum_lo < lo ? 1ull : 0ull;
  unsigned long long sum_hi = hi + add_hi + carry;
  if (s >= 64) return s == 64 ? sum_hi : (sum_hi >> (s - 64));
  if (s == 0) return sum_lo;
  return (sum_lo >> s) | (sum_hi << (64 - s));
}

// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, SC'11).
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

// U in (0,1) from one Philox output word: (top 23 bits + 1/2) / 2^23, exact in fp32.
__device__ __forceinline__ float word_to_uniform(uint32_t x) {
  return __fmul_rn(__fadd_rn(__uint2float_rn(x >> 9), 0.5f), 0x1p-23f);
}

// Race score of a kept token: y - ln E with E = -ln U (Gumbel form of argmax w / E).
__device__ __forceinline__ float race_score(float y, uint32_t x) {
  const float u = word_to_uniform(x);
  const float e = -logf(u);
  return __fsub_rn(y, logf(e));
}

// (value, id) "better": larger value, then lower id.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Merge two (max, sum 2^((z-max)c)) pairs.
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2, float c) {
  const float mm = fmaxf(m, m2);
  if (mm == -INFINITY) {
    m = mm;
    s = 0.0f;
    return;
  }
  s = s * ex2_approx(__fmul_rn(m - mm, c)) + s2 * ex2_approx(__fmul_rn(m2 - mm, c));
  m = mm;
}

// ---------------------------------------------------------------- block reductions

template <typename T>
__device__ __forceinline__ T shfl_down(T v, int d) {
  return __shfl_down_sync(0xffffffffu, v, d);
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, unsigned long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += shfl_down(v, d);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int w = 0; w < kWarps; ++w) t += red[w];
  return t;
}

// ---------------------------------------------------------------- logits loaders

struct LoadF32 {
  const float* row;
  int len;
  bool vec;
  __device__ __forceinline__ float4 load4(int e) const {
    if (vec && e + 3 < len) return __ldcs(reinterpret_cast<const float4*>(row + e));
    float4 v;
    v.x = e + 0 < len ? __ldcs(row + e + 0) : 0.0f;
    v.y = e + 1 < len ? __ldcs(row + e + 1) : 0.0f;
    v.z = e + 2 < len ? __ldcs(row + e + 2) : 0.0f;
    v.w = e + 3 < len ? __ldcs(row + e + 3) : 0.0f;
    return v;
  }
};

__device__ __forceinline__ float bf16_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

struct LoadBF16 {
  const uint16_t* row;
  int len;
  bool vec;
  __device__ __forceinline__ float4 load4(int e) const {
    float4 v;
    if (vec && e + 3 < len) {
      const uint2 w = __ldcs(reinterpret_cast<const uint2*>(row + e));
      v.x = bf16_to_f32(w.x & 0xFFFFu);
      v.y = bf16_to_f32(w.x >> 16);
      v.z = bf16_to_f32(w.y & 0xFFFFu);
      v.w = bf16_to_f32(w.y >> 16);
      return v;
    }
    v.x = e + 0 < len ? bf16_to_f32(__ldcs(row + e + 0)) : 0.0f;
    v.y = e + 1 < len ? bf16_to_f32(__ldcs(row + e + 1)) : 0.0f;
    v.z = e + 2 < len ? bf16_to_f32(__ldcs(row + e + 2)) : 0.0f;
    v.w = e + 3 < len ? bf16_to_f32(__ldcs(row + e + 3)) : 0.0f;
    return v;
  }
};

// ---------------------------------------------------------------- hash of penalised ids

// Inserts local id l; returns the slot or -1 when the table is full (bounded probing).
__device__ __forceinline__ int hash_insert(uint32_t* hkey, uint32_t l) {
  uint32_t h = (l * 2654435761u) & (kHashCap - 1);
  for (int probe = 0; probe < kHashCap; ++probe) {
    const uint32_t slot = (h + probe) & (kHashCap - 1);
    const uint32_t prev = atomicCAS(&hkey[slot], kEmpty, l);
    if (prev == kEmpty || prev == l) return (int)slot;
  }
  return -1;
}

// ---------------------------------------------------------------- cluster radix select

// Finds, among this row's candidates with y >= ylo, the key K* such that
//   unweighted: K* is the `target`-th largest key (1-based, repeats counted);
//   weighted:   the running fixed-point weight, summed from the largest key down,
//               first reaches `target` at key K*.
// Four passes of 8-bit digits, most significant first; each pass histograms the
// elements that match the digits chosen so far, merges the C histograms through DSMEM
// and picks the digit.  Returns K*, or sets *err if the histograms run dry (which the
// callers' targets make impossible).
template <bool kWeighted>
__device__ uint32_t cluster_select(const cg::cluster_group& cluster, const Smem& S, int C, int chunk,
                                   float m, float invT, float ylo, unsigned long long target,
                                   int* sel_digit, unsigned long long* sel_above, int* err) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0, pmask = 0;
  const int nvec = chunk / 4;
  const float4* z4p = reinterpret_cast<const float4*>(S.zs);
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const int buf = pass & 1;
    uint32_t* hc = S.hist_c + buf * 256;
    unsigned long long* hw = S.hist_w + buf * 256;
    if (tid < 256) {
      hc[tid] = 0u;
      hw[tid] = 0ull;
    }
    __syncthreads();
    for (int base = 0; base < nvec; base += kThreads) {
      const int f = base + tid;
      float4 z4 = f < nvec ? z4p[f] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      const float zz[4] = {z4.x, z4.y, z4.z, z4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float y = y_of(zz[j], m, invT);
        const uint32_t key = ykey(y);
        const bool pred = (zz[j] > -INFINITY) && (y >= ylo) && ((key & pmask) == prefix);
        const uint32_t digit = pred ? ((key >> shift) & 0xFFu) : 0xFFFFFFFFu;
        if (!kWeighted) {
          const uint32_t peers = __match_any_sync(0xffffffffu, digit);
          if (pred && lane == __ffs(peers) - 1) atomicAdd(&hc[digit], (uint32_t)__popc(peers));
        } else {
          if (pred) atomicAdd(&hw[digit], weight_fx(y));
        }
      }
    }
    __syncthreads();
    cluster.sync();  // every CTA's histogram of this pass is complete
    if (tid < 256) {
      unsigned long long sc = 0, sw = 0;
      for (int r = 0; r < C; ++r) {
        if (!kWeighted) {
          const uint32_t* rc = cluster.map_shared_rank(hc, r);
          sc += rc[tid];
        } else {
          const unsigned long long* rw = cluster.map_shared_rank(hw, r);
          sw += rw[tid];
        }
      }
      S.merged_c[tid] = kWeighted ? sw : sc;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l covers bins 255-8l .. 248-8l, scanned from the top down
      unsigned long long v[8];
      unsigned long long lsum = 0;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        v[t] = S.merged_c[255 - 8 * lane - t];
        lsum += v[t];
      }
      unsigned long long incl = lsum;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const unsigned long long o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
      }
      const uint32_t hit = __ballot_sync(0xffffffffu, incl >= target);
      const int first = hit ? __ffs(hit) - 1 : -1;
      if (lane == (first < 0 ? 0 : first)) {
        if (first < 0) {
          *err = 1;
          *sel_digit = 0;
          *sel_above = 0;
        } else {
          unsigned long long cum = incl - lsum;
          int d = 255 - 8 * lane - 7;
          for (int t = 0; t < 8; ++t) {
            if (cum + v[t] >= target) {
              d = 255 - 8 * lane - t;
              break;
            }
            cum += v[t];
          }
          *sel_digit = d;
          *sel_above = cum;
        }
      }
    }
    __syncthreads();
    prefix |= (uint32_t)(*sel_digit) << shift;
    pmask |= 0xFFu << shift;
    target -= *sel_above;
    __syncthreads();
  }
  return prefix;
}

// ---------------------------------------------------------------- the kernel

template <typename Loader, typename Elem>
__global__ void __launch_bounds__(kThreads, 2) sampler_kernel(const LaunchParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ Exchange xchg;
  __shared__ RowParams rp;
  __shared__ unsigned long long red_u64[kWarps];
  __shared__ float red_f[kWarps * 4];
  __shared__ int red_i[kWarps * 4];
  __shared__ int sh_flags;
  __shared__ int sh_sel_digit;
  __shared__ unsigned long long sh_sel_above;
  __shared__ int sh_sel_err;

  const cg::cluster_group cluster = cg::this_cluster();
  const clsample_args_t& a = P.a;
  const int C = P.C;
  const int chunk = P.chunk;
  const int rank = (int)cluster.block_rank();
  const int row = (int)(blockIdx.x / (unsigned)C);
  const int V = a.V;
  const int c0 = rank * chunk;
  const int c1 = min(V, c0 + chunk);
  const int len = max(0, c1 - c0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const Smem S = carve(smem_raw, chunk);

  // ---- row parameters (validated identically by every CTA of the cluster)
  if (tid == 0) {
    RowParams q;
    q.T = a.temperatures ? a.temperatures[row] : 1.0f;
    q.k = a.top_ks ? a.top_ks[row] : -1;
    q.p = a.top_ps ? a.top_ps[row] : 1.0f;
    q.mp = a.min_ps ? a.min_ps[row] : 0.0f;
    q.rep = a.rep ? a.rep[row] : 1.0f;
    q.freq = a.freq ? a.freq[row] : 0.0f;
    q.pres = a.pres ? a.pres[row] : 0.0f;
    q.seed = a.seeds ? a.seeds[row] : 0ull;
    q.pos = a.positions ? a.positions[row] : a.step;
    int bad = 0;
    bad |= (q.T != q.T) || (q.T == INFINITY);
    bad |= (q.k < -1);
    bad |= !(q.p > 0.0f && q.p <= 1.0f);
    bad |= !(q.mp >= 0.0f && q.mp <= 1.0f);
    bad |= !(q.rep > 0.0f) || (q.rep == INFINITY) || !isfinite(q.freq) || !isfinite(q.pres);
    q.invalid = bad;
    rp = q;
    sh_flags = 0;
    sh_sel_err = 0;
  }
  const bool has_hist = a.hist_offs != nullptr;
  const bool has_bias = a.bias_offs != nullptr;
  const bool has_mod = has_hist || has_bias;
  for (int i = tid; i < chunk / 32; i += kThreads) S.modbits[i] = 0u;
  if (has_mod) {
    for (int i = tid; i < kHashCap; i += kThreads) {
      S.hkey[i] = kEmpty;
      S.hcnt[i] = 0u;
      S.hbias[i] = -1;
    }
  }
  __syncthreads();

  // ---- penalised / biased ids of this slice: count history occurrences and keep the
  //      last bias entry per id (SGLang page, "Why logit_bias is built from triples")
  if (has_mod) {
    int flags = 0;
    if (has_hist) {
      const int lo = a.hist_offs[row], hi = a.hist_offs[row + 1];
      if (lo < 0 || hi < lo) {
        flags |= kFlagInvalid;
      } else {
        for (int j = lo + tid; j < hi; j += kThreads) {
          const int id = __ldg(a.hist_ids + j);
          if (id < 0 || id >= V) {
            flags |= kFlagInvalid;
          } else if (id >= c0 && id < c1) {
            const int slot = hash_insert(S.hkey, (uint32_t)(id - c0));
            if (slot < 0) flags |= kFlagOverflow;
            else atomicAdd(&S.hcnt[slot], 1u);
          }
        }
      }
    }
    if (has_bias) {
      const int lo = a.bias_offs[row], hi = a.bias_offs[row + 1];
      if (lo < 0 || hi < lo) {
        flags |= kFlagInvalid;
      } else {
        for (int j = lo + tid; j < hi; j += kThreads) {
          const int id = __ldg(a.bias_ids + j);
          const float b = __ldg(a.bias_vals + j);
          if (id < 0 || id >= V || b != b) {
            flags |= kFlagInvalid;
          } else if (id >= c0 && id < c1) {
            const int slot = hash_insert(S.hkey, (uint32_t)(id - c0));
            if (slot < 0) flags |= kFlagOverflow;
            else atomicMax(&S.hbias[slot], j);
          }
        }
      }
    }
    if (flags) atomicOr(&sh_flags, flags);
    __syncthreads();
    for (int i = tid; i < kHashCap; i += kThreads) {
      const uint32_t l = S.hkey[i];
      if (l != kEmpty) atomicOr(&S.modbits[l >> 5], 1u << (l & 31));
    }
    __syncthreads();
  }

  // ---- pass 1: load the slice once from HBM, sanitise, mask, keep it in shared
  //      memory; per-thread max / argmax / online sum of 2^((z'-max)c) / count over
  //      the tokens that are not penalised or biased
  const RowParams q = rp;
  const bool greedy_rule = (q.T < kGreedyEps) || q.k == 0 || q.k == 1;
  const float Teff = (q.T >= kGreedyEps) ? q.T : 1.0f;
  const float c_log2 = 1.4426950408889634f / Teff;  // log2(e) / T for the normaliser
  float tm = -INFINITY, ts = 0.0f;
  int targ = INT_MAX, tcnt = 0;
  {
    Loader ld;
    ld.row = reinterpret_cast<const Elem*>(a.logits) + (long long)row * a.logits_row_stride + c0;
    ld.len = len;
    ld.vec = P.vec_ok != 0;
    const int32_t* bmrow = a.bitmask ? a.bitmask + (long long)row * a.bitmask_row_stride : nullptr;
    const int nvec = chunk / 4;
    constexpr int U = 4;
    float4* z4p = reinterpret_cast<float4*>(S.zs);
    for (int base = 0; base < nvec; base += kThreads * U) {
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int f = base + u * kThreads + tid;
        v[u] = (f < nvec && 4 * f < len) ? ld.load4(4 * f) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int f = base + u * kThreads + tid;
        if (f >= nvec) continue;
        const int e = 4 * f;
        uint32_t allow = 0xFu;
        if (e + 4 > len) allow = (e >= len) ? 0u : ((1u << (len - e)) - 1u);
        if (bmrow && e < len) allow &= ((uint32_t)__ldg(bmrow + ((c0 + e) >> 5)) >> (e & 31)) & 0xFu;
        const uint32_t mod = has_mod ? ((S.modbits[e >> 5] >> (e & 31)) & 0xFu) : 0u;
        float zz[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        float bm = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          zz[j] = ((allow >> j) & 1u) ? sanitize(zz[j]) : -INFINITY;
          if (!((mod >> j) & 1u) && zz[j] > -INFINITY) {
            ++tcnt;
            if (zz[j] > bm) {
              bm = zz[j];
              bi = c0 + e + j;
            }
          }
        }
        z4p[f] = make_float4(zz[0], zz[1], zz[2], zz[3]);
        if (bm > -INFINITY) {
          if (better(bm, bi, tm, targ)) {
            if (bm > tm) {
              ts = ts * ex2_approx(__fmul_rn(tm - bm, c_log2));
              tm = bm;
            }
            targ = bi;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (!((mod >> j) & 1u)) ts += ex2_approx(__fmul_rn(zz[j] - tm, c_log2));
        }
      }
    }
  }
  __syncthreads();

  // ---- penalties, then bias, on the slice's listed ids (SGLang page, "Order semantics
  //      of the penalties"); the mask was already applied and -inf stays -inf
  if (has_mod) {
    for (int i = tid; i < kHashCap; i += kThreads) {
      const uint32_t l = S.hkey[i];
      if (l == kEmpty) continue;
      float z = S.zs[l];
      const uint32_t cnt = S.hcnt[i];
      if (cnt > 0u) {
        z = __fsub_rn(z, __fmul_rn(q.freq, (float)cnt));
        z = __fsub_rn(z, q.pres);
        z = (z > 0.0f) ? __fdiv_rn(z, q.rep) : __fmul_rn(z, q.rep);
      }
      const int bj = S.hbias[i];
      if (bj >= 0) z = __fadd_rn(z, __ldg(a.bias_vals + bj));
      z = guard(z);
      S.zs[l] = z;
      if (z > -INFINITY) {
        ++tcnt;
        const int gid = c0 + (int)l;
        if (better(z, gid, tm, targ)) {
          if (z > tm) {
            ts = ts * ex2_approx(__fmul_rn(tm - z, c_log2));
            tm = z;
          }
          targ = gid;
        }
        ts += ex2_approx(__fmul_rn(z - tm, c_log2));
      }
    }
    __syncthreads();
  }

  if (a.dbg_transformed) {
    float* out = a.dbg_transformed + (long long)row * V + c0;
    for (int i = tid; i < len; i += kThreads) out[i] = S.zs[i];
  }

  // ---- block reduction of (max, argmax, sum, count)
  {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      const float om = shfl_down(tm, d);
      const float os = shfl_down(ts, d);
      const int oa = shfl_down(targ, d);
      const int oc = shfl_down(tcnt, d);
      float m2 = tm, s2 = ts;
      merge_ms(m2, s2, om, os, c_log2);
      if (better(om, oa, tm, targ)) targ = oa;
      tm = m2;
      ts = s2;
      tcnt += oc;
    }
    if (lane == 0) {
      red_f[warp * 4 + 0] = tm;
      red_f[warp * 4 + 1] = ts;
      red_i[warp * 4 + 0] = targ;
      red_i[warp * 4 + 1] = tcnt;
    }
    __syncthreads();
    if (tid == 0) {
      float m = -INFINITY, s = 0.0f;
      int arg = INT_MAX, cnt = 0;
      for (int w = 0; w < kWarps; ++w) {
        const float wm = red_f[w * 4 + 0];
        const int wa = red_i[w * 4 + 0];
        if (better(wm, wa, m, arg)) arg = wa;
        merge_ms(m, s, wm, red_f[w * 4 + 1], c_log2);
        cnt += red_i[w * 4 + 1];
      }
      xchg.m = m;
      xchg.arg = arg;
      xchg.S = s;
      xchg.ncand = cnt;
      xchg.flags = sh_flags;
    }
  }
  cluster.sync();  // exchange 1: slice statistics

  // ---- row statistics, combined in rank order by every CTA (identical results)
  float m = -INFINITY, Ssum = 0.0f;
  int arg = INT_MAX, ncand = 0, flags = 0;
  for (int r = 0; r < C; ++r) {
    const Exchange* x = cluster.map_shared_rank(&xchg, r);
    const float xm = x->m;
    const int xa = x->arg;
    if (better(xm, xa, m, arg)) arg = xa;
    merge_ms(m, Ssum, xm, x->S, c_log2);
    ncand += x->ncand;
    flags |= x->flags;
  }
  int status = kRowOk;
  if (q.invalid || (flags & kFlagInvalid) || ncand == 0) status = kRowInvalid;
  else if (flags & kFlagOverflow) status = kRowOverflow;
  const float lnS = logf(Ssum);

  if (status != kRowOk || greedy_rule) {
    if (rank == 0 && tid == 0) {
      const bool ok = status == kRowOk;
      a.tokens[row] = ok ? arg : -1;
      if (a.logprobs) a.logprobs[row] = ok ? -lnS : -INFINITY;  // y of the argmax is 0
      if (a.row_status) a.row_status[row] = status;
      if (a.dbg_kept_count) a.dbg_kept_count[row] = ok ? 1 : 0;
      if (a.dbg_cut) a.dbg_cut[row] = ok ? 0.0f : -INFINITY;
    }
    cluster.sync();  // no CTA leaves while another may still read its shared memory
    return;
  }

  // ---- truncation thresholds on y = (z' - m) * (1/T)
  const float invT = __frcp_rn(q.T);
  float tk = -INFINITY;
  if (q.k >= 2 && q.k < ncand) {
    const uint32_t key = cluster_select<false>(cluster, S, C, chunk, m, invT, -INFINITY,
                                               (unsigned long long)q.k, &sh_sel_digit, &sh_sel_above,
                                               &sh_sel_err);
    tk = key_to_y(key);
  }
  float tp = -INFINITY;
  if (q.p < 1.0f) {
    // W_k: exact fixed-point mass of S_k (the candidates with y >= tk)
    unsigned long long w = 0;
    const float4* z4p = reinterpret_cast<const float4*>(S.zs);
    for (int f = tid; f < chunk / 4; f += kThreads) {
      const float4 z4 = z4p[f];
      const float zz[4] = {z4.x, z4.y, z4.z, z4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float y = y_of(zz[j], m, invT);
        if (zz[j] > -INFINITY && y >= tk) w += weight_fx(y);
      }
    }
    w = block_sum_u64(w, red_u64);
    if (tid == 0) xchg.W = w;
    cluster.sync();  // exchange 2: top-k mass
    unsigned long long W = 0;
    for (int r = 0; r < C; ++r) W += cluster.map_shared_rank(&xchg, r)->W;
    const unsigned long long Cth = ceil_scaled(W, q.p);
    const uint32_t key = cluster_select<true>(cluster, S, C, chunk, m, invT, tk, Cth, &sh_sel_digit,
                                              &sh_sel_above, &sh_sel_err);
    tp = key_to_y(key);
  }
  float tm_cut = -INFINITY;
  if (q.mp > 0.0f) tm_cut = (float)log((double)q.mp);
  const float cut = fmaxf(tk, fmaxf(tp, tm_cut));

  // ---- exponential race over K = {candidates : y >= cut}
  float bs = -INFINITY, ymin = INFINITY;
  int btok = INT_MAX, kept = 0;
  {
    const uint2 key = make_uint2((uint32_t)q.seed, (uint32_t)(q.seed >> 32));
    const uint32_t plo = (uint32_t)(unsigned long long)q.pos, phi = (uint32_t)((unsigned long long)q.pos >> 32);
    const float4* z4p = reinterpret_cast<const float4*>(S.zs);
    for (int f = tid; f < chunk / 4; f += kThreads) {
      const float4 z4 = z4p[f];
      const float zz[4] = {z4.x, z4.y, z4.z, z4.w};
      float yy[4];
      uint32_t keep = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        yy[j] = y_of(zz[j], m, invT);
        if (zz[j] > -INFINITY && yy[j] >= cut) keep |= 1u << j;
      }
      if (!keep) continue;
      const int gid0 = c0 + 4 * f;
      const uint4 x = philox4x32_10(make_uint4((uint32_t)(gid0 >> 2), plo, phi, 0u), key);
      const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (!((keep >> j) & 1u)) continue;
        ++kept;
        ymin = fminf(ymin, yy[j]);
        const float s = race_score(yy[j], xw[j]);
        if (better(s, gid0 + j, bs, btok)) {
          bs = s;
          btok = gid0 + j;
        }
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      const float os = shfl_down(bs, d);
      const int ot = shfl_down(btok, d);
      const int ok = shfl_down(kept, d);
      const float oy = shfl_down(ymin, d);
      if (better(os, ot, bs, btok)) {
        bs = os;
        btok = ot;
      }
      kept += ok;
      ymin = fminf(ymin, oy);
    }
    if (lane == 0) {
      red_f[warp * 4 + 2] = bs;
      red_f[warp * 4 + 3] = ymin;
      red_i[warp * 4 + 2] = btok;
      red_i[warp * 4 + 3] = kept;
    }
    __syncthreads();
    if (tid == 0) {
      float s = -INFINITY, yl = INFINITY;
      int t = INT_MAX, kc = 0;
      for (int w = 0; w < kWarps; ++w) {
        if (better(red_f[w * 4 + 2], red_i[w * 4 + 2], s, t)) {
          s = red_f[w * 4 + 2];
          t = red_i[w * 4 + 2];
        }
        yl = fminf(yl, red_f[w * 4 + 3]);
        kc += red_i[w * 4 + 3];
      }
      xchg.race_s = s;
      xchg.race_tok = t;
      xchg.kept = kc;
      xchg.ymin = yl;
    }
  }
  cluster.sync();  // exchange 3: race winners
  if (rank == 0 && tid == 0) {
    float s = -INFINITY, yl = INFINITY;
    int t = INT_MAX, kc = 0;
    for (int r = 0; r < C; ++r) {
      const Exchange* x = cluster.map_shared_rank(&xchg, r);
      if (better(x->race_s, x->race_tok, s, t)) {
        s = x->race_s;
        t = x->race_tok;
      }
      yl = fminf(yl, x->ymin);
      kc += x->kept;
    }
    const bool ok = (t != INT_MAX) && !sh_sel_err;
    a.tokens[row] = ok ? t : -1;
    if (a.logprobs) {
      // y of the drawn token, recomputed from its transformed logit
      float lp = -INFINITY;
      if (ok) {
        const int owner = t / chunk;
        const float* zsr = cluster.map_shared_rank(S.zs, owner);
        lp = y_of(zsr[t - owner * chunk], m, invT) - lnS;
      }
      a.logprobs[row] = lp;
    }
    if (a.row_status) a.row_status[row] = ok ? kRowOk : kRowOverflow;
    if (a.dbg_kept_count) a.dbg_kept_count[row] = kc;
    if (a.dbg_cut) a.dbg_cut[row] = yl;
  }
  cluster.sync();  // keep every CTA's shared memory alive until rank 0 is done
}

// ---------------------------------------------------------------- diagnostics kernels

__global__ void debug_weights_kernel(const float* y, unsigned long long* w, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) w[i] = weight_fx(y[i]);
}

__global__ void debug_uniforms_kernel(const uint64_t* seeds, const int64_t* pos, const int64_t* tok, float* u,
                                      int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const unsigned long long s = seeds[i], p = (unsigned long long)pos[i];
  const long long t = tok[i];
  const uint4 x = philox4x32_10(make_uint4((uint32_t)((unsigned long long)t >> 2), (uint32_t)p, (uint32_t)(p >> 32), 0u),
                                make_uint2((uint32_t)s, (uint32_t)(s >> 32)));
  const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
  u[i] = word_to_uniform(xw[t & 3]);
}

// ---------------------------------------------------------------- host side

Geometry geometry_for(int vocab) {
  Geometry g{0, 0, 0};
  if (vocab <= 0) return g;
  int C = (vocab + 2047) / 2048;
  if (C > 8) C = 8;
  if (C < 1) C = 1;
  int chunk = ((vocab + C - 1) / C + 31) / 32 * 32;
  if (smem_bytes_for(chunk) > 112 * 1024 && C == 8) {  // two CTAs per SM no longer fit
    C = kMaxCluster;
    chunk = ((vocab + C - 1) / C + 31) / 32 * 32;
  }
  g.C = C;
  g.chunk = chunk;
  g.smem = (int)smem_bytes_for(chunk);
  if (g.smem > 227 * 1024) g.C = 0;
  return g;
}

}  // namespace

struct clsample_handle {
  int max_batch;
  int vocab;
  int device;
  Geometry g;
};

extern "C" {

const char* clsample_strerror(int code) {
  switch (code) {
    case CLSAMPLE_SUCCESS: return "success";
    case CLSAMPLE_ERR_NULL: return "a required pointer is NULL";
    case CLSAMPLE_ERR_BATCH: return "batch size out of range";
    case CLSAMPLE_ERR_VOCAB: return "vocabulary size invalid, different from the handle's, or too large";
    case CLSAMPLE_ERR_STRIDE: return "row stride smaller than the row";
    case CLSAMPLE_ERR_DTYPE: return "unknown logits dtype";
    case CLSAMPLE_ERR_CUDA: return "CUDA runtime error";
    case CLSAMPLE_ERR_DEVICE: return "wrong or unsupported CUDA device";
    default: return "unknown error";
  }
}

int clsample_geometry(int32_t vocab, int32_t* cluster, int32_t* chunk, int32_t* smem_bytes) {
  const Geometry g = geometry_for(vocab);
  if (g.C == 0) return CLSAMPLE_ERR_VOCAB;
  if (cluster) *cluster = g.C;
  if (chunk) *chunk = g.chunk;
  if (smem_bytes) *smem_bytes = g.smem;
  return CLSAMPLE_SUCCESS;
}

int clsample_create(int32_t max_batch, int32_t vocab, clsample_t** out) {
  if (!out) return CLSAMPLE_ERR_NULL;
  *out = nullptr;
  if (max_batch < 0) return CLSAMPLE_ERR_BATCH;
  const Geometry g = geometry_for(vocab);
  if (g.C == 0) return CLSAMPLE_ERR_VOCAB;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CLSAMPLE_ERR_CUDA;
  int major = 0, minor = 0, optin = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return CLSAMPLE_ERR_CUDA;
  if (major != 10 || minor != 3) return CLSAMPLE_ERR_DEVICE;
  if (g.smem > optin) return CLSAMPLE_ERR_VOCAB;
  const void* kernels[2] = {reinterpret_cast<const void*>(&sampler_kernel<LoadF32, float>),
                            reinterpret_cast<const void*>(&sampler_kernel<LoadBF16, uint16_t>)};
  for (const void* k : kernels) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem) != cudaSuccess)
      return CLSAMPLE_ERR_CUDA;
    if (g.C > 8 && cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      return CLSAMPLE_ERR_CUDA;
  }
  clsample_t* h = new clsample_t;
  h->max_batch = max_batch;
  h->vocab = vocab;
  h->device = dev;
  h->g = g;
  *out = h;
  return CLSAMPLE_SUCCESS;
}

void clsample_destroy(clsample_t* h) { delete h; }

int clsample_apply(clsample_t* h, const clsample_args_t* a, clsample_stream_t stream) {
  if (!h || !a) return CLSAMPLE_ERR_NULL;
  if (a->B < 0 || a->B > h->max_batch) return CLSAMPLE_ERR_BATCH;
  if (a->V != h->vocab) return CLSAMPLE_ERR_VOCAB;
  if (a->logits_dtype != CLSAMPLE_LOGITS_F32 && a->logits_dtype != CLSAMPLE_LOGITS_BF16) return CLSAMPLE_ERR_DTYPE;
  if (a->B == 0) return CLSAMPLE_SUCCESS;
  if (!a->logits || !a->tokens) return CLSAMPLE_ERR_NULL;
  if (a->hist_offs && !a->hist_ids) return CLSAMPLE_ERR_NULL;
  if (a->bias_offs && (!a->bias_ids || !a->bias_vals)) return CLSAMPLE_ERR_NULL;
  if (a->logits_row_stride < a->V) return CLSAMPLE_ERR_STRIDE;
  if (a->bitmask && a->bitmask_row_stride < (a->V + 31) / 32) return CLSAMPLE_ERR_STRIDE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CLSAMPLE_ERR_CUDA;
  if (dev != h->device) return CLSAMPLE_ERR_DEVICE;

  LaunchParams P;
  P.a = *a;
  P.C = h->g.C;
  P.chunk = h->g.chunk;
  const uintptr_t base = reinterpret_cast<uintptr_t>(a->logits);
  if (a->logits_dtype == CLSAMPLE_LOGITS_F32)
    P.vec_ok = (base % 16 == 0) && (a->logits_row_stride % 4 == 0);
  else
    P.vec_ok = (base % 8 == 0) && (a->logits_row_stride % 4 == 0);

  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)a->B * (unsigned)P.C, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)h->g.smem;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)P.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t err;
  if (a->logits_dtype == CLSAMPLE_LOGITS_F32)
    err = cudaLaunchKernelEx(&cfg, sampler_kernel<LoadF32, float>, P);
  else
    err = cudaLaunchKernelEx(&cfg, sampler_kernel<LoadBF16, uint16_t>, P);
  return err == cudaSuccess ? CLSAMPLE_SUCCESS : CLSAMPLE_ERR_CUDA;
}

int clsample_debug_weights(const float* y, uint64_t* w, int32_t n, clsample_stream_t stream) {
  if (n < 0) return CLSAMPLE_ERR_BATCH;
  if (n == 0) return CLSAMPLE_SUCCESS;
  if (!y || !w) return CLSAMPLE_ERR_NULL;
  debug_weights_kernel<<<(n + 255) / 256, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      y, reinterpret_cast<unsigned long long*>(w), n);
  return cudaGetLastError() == cudaSuccess ? CLSAMPLE_SUCCESS : CLSAMPLE_ERR_CUDA;
}

int clsample_debug_uniforms(const uint64_t* seeds, const int64_t* positions, const int64_t* tokens, float* u,
                            int32_t n, clsample_stream_t stream) {
  if (n < 0) return CLSAMPLE_ERR_BATCH;
  if (n == 0) return CLSAMPLE_SUCCESS;
  if (!seeds || !positions || !tokens || !u) return CLSAMPLE_ERR_NULL;
  debug_uniforms_kernel<<<(n + 255) / 256, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(seeds, positions,
                                                                                                tokens, u, n);
  return cudaGetLastError() == cudaSuccess ? CLSAMPLE_SUCCESS : CLSAMPLE_ERR_CUDA;
}

}  // extern "C"
