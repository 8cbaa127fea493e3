// Batched constrained logits sampler for GB300 (sm_103a).
//
// One thread-block cluster samples one row.  The row's V logits are split into C
// contiguous slices (a multiple of 32 tokens, so that every CTA owns whole bitmask
// words).  Each CTA pulls its slice into shared memory with a single TMA bulk copy
// issued at entry, so the whole slice is in flight while the CTA reads the row's token
// history and logit_bias lists; HBM sees every logit exactly once and nothing but the
// per-row outputs is written back.
//
//   pass A    sanitise + mask + penalties/bias (the few penalised tokens live in a small
//             hash with their final value), slice max, lowest argmax and an online sum of
//             exp((z' - max)/T); per-thread maxima give a lower bound of the top-k cut.
//   exchange  every CTA pushes its slice statistics into every CTA's shared memory
//             (DSMEM) and one cluster barrier publishes them.  Greedy rows end here.
//   pass B    the tokens that can survive truncation (y >= a provable bound) are
//             compacted; a leader CTA gathers them (DSMEM stores + a remote mbarrier
//             arrive) and finishes top-k -> top-p -> min-p and the exponential race alone.
//   slow path rows without a usable bound (top-p alone, very large k, compaction
//             overflow) run cluster-wide radix selects over the resident slices.
//
// The arithmetic that decides integers (kept set, drawn id) is exact and identical on
// any IEEE machine (sampler_math.cuh).  Page references: "SGLang source teardown (10):
// Sampling, Grammar and structured output" (SGLang page) and "GLM-5.3 inference (7):
// output side" (GLM page).

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "clsample.h"
#include "cluster_sync.cuh"
#include "sampler_math.cuh"

namespace cg = cooperative_groups;

namespace {

using namespace clsample;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kHashCap = 1024;   // distinct penalised / biased ids per slice
constexpr int kCandCap = 512;    // compacted candidates per slice
constexpr int kMaxCluster = 16;
constexpr uint32_t kEmpty = 0xFFFFFFFFu;
// The slice's bulk copy is issued as this many TMA copies (all on one mbarrier).
#ifndef CLSAMPLE_BULK_PIECES
#define CLSAMPLE_BULK_PIECES 1
#endif
constexpr int kBulkPieces = CLSAMPLE_BULK_PIECES;
// Longest slice: pass A keeps a bit per token of the slice in the histogram area.
constexpr int kMaxChunk = 32 * 1024;

enum : int { kRowOk = 0, kRowOverflow = 1, kRowInvalid = 2 };
enum : int { kFlagInvalid = 1, kFlagOverflow = 2, kFlagTimeout = 4 };

struct Geometry {
  int C;      // CTAs per row (cluster size)
  int chunk;  // tokens per CTA, multiple of 32
  int smem;   // dynamic shared memory per CTA for this element size
  int cap;    // compacted candidates per CTA the leader can gather
};

struct LaunchParams {
  clsample_args_t a;
  int C;
  int chunk;
  int cap;
  int bulk_ok;  // every row start is 16-byte aligned: the slice can be bulk-copied
};

struct Cand {
  float y;
  int id;
};

// Slice statistics pushed to every CTA after pass A.
struct X1 {
  float m;      // slice max of z' (-inf if no candidate)
  int arg;      // lowest id reaching m (INT_MAX if none)
  float s;      // sum over the slice's candidates of 2^((z' - m) * log2(e) / T)
  int flags;    // kFlag*
  float lk;     // max over warps of the warp's k-th largest thread max of z' (-inf: unknown)
  float lkc;    // min over warps of the ceil(k / (16 C))-th largest thread max (-inf: unknown)
};

// Slice results pushed to every CTA after pass B (and by the slow path).
struct X2 {
  int count;                // compacted candidates (may exceed the capacity)
  int flags;
  unsigned long long w;     // fixed-point weight partial (top-p mass)
  float race_s;             // best race score of the slice
  int race_tok;             // its id
  int kept;                 // kept tokens of the slice
  float ymin;               // smallest y of a kept token
  float ytok;               // y of the slice's winner
};

struct RowParams {
  float T, p, mp, rep, freq, pres;
  int k;
  unsigned long long seed;
  unsigned long long pos;
  int invalid;
};

struct RowState {
  float m;
  int arg;
  float S;
  int flags;
  float bound;  // lower bound of the k-th largest z' (-inf if none)
};

// ---------------------------------------------------------------- shared memory layout

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Dynamic shared memory of one CTA:
//   raw       chunk * esize       the slice as loaded (f32 or bf16 bits); the leader
//                                  reuses it to gather the cluster's candidates
//   live      u32[chunk/32]       allowed by the bitmask, inside the row, not penalised
//   hkey/hcnt/hbias/hval          hash of the slice's penalised / biased tokens: local id,
//                                  history count, last bias entry, its value then final z'
//   cand      Cand[kCandCap]      compacted candidates of the slice
//   hist_c    u32[256]            local radix histogram (counts); also the sort buffer
//   hist_w    u64[256]            local radix histogram (fixed-point weights)
//   mrg_c     u32[2][256]         cluster-merged histograms (DSMEM atomics from every
//   mrg_w     u64[2][256]         CTA), double-buffered across passes
struct Smem {
  unsigned char* raw;
  uint32_t* live;
  uint32_t* hkey;
  uint32_t* hcnt;
  int32_t* hbias;
  float* hval;
  Cand* cand;
  uint32_t* hist_c;
  unsigned long long* hist_w;
  uint32_t* mrg_c;
  unsigned long long* mrg_w;
};

// The top-p histogram (kWarps x 64 bins of u64) reuses cand + hist_c + hist_w, which
// are contiguous; pass A's per-token `modbits` (kMaxChunk bits) reuses hist_c + hist_w.
static_assert(sizeof(uint32_t) * kThreads + sizeof(unsigned long long) * 256 >= kMaxChunk / 8,
              "pass A modbits do not fit the histogram area");
static_assert(sizeof(Cand) * kCandCap + sizeof(uint32_t) * kThreads + sizeof(unsigned long long) * 256 >=
                  sizeof(unsigned long long) * kWarps * 64,
              "top-p histogram does not fit the candidate area");

__host__ __device__ inline size_t smem_bytes_for(int chunk, int esize) {
  size_t b = align_up((size_t)chunk * esize, 128);
  b += sizeof(uint32_t) * (size_t)(chunk / 32);
  b = align_up(b, 16);
  b += (sizeof(uint32_t) * 3 + sizeof(float)) * kHashCap;
  b += sizeof(Cand) * kCandCap;
  b = align_up(b, 16);
  b += sizeof(uint32_t) * kThreads;  // >= 256 counts; sized for the 512-entry sort
  b += sizeof(unsigned long long) * 256;
  b += sizeof(uint32_t) * 2 * 256;
  b += sizeof(unsigned long long) * 2 * 256;
  return b;
}

__device__ inline Smem carve(unsigned char* base, int chunk, int esize) {
  Smem s;
  size_t off = 0;
  s.raw = base;
  off = align_up((size_t)chunk * esize, 128);
  s.live = reinterpret_cast<uint32_t*>(base + off);
  off += sizeof(uint32_t) * (size_t)(chunk / 32);
  off = align_up(off, 16);
  s.hkey = reinterpret_cast<uint32_t*>(base + off);
  off += sizeof(uint32_t) * kHashCap;
  s.hcnt = reinterpret_cast<uint32_t*>(base + off);
  off += sizeof(uint32_t) * kHashCap;
  s.hbias = reinterpret_cast<int32_t*>(base + off);
  off += sizeof(int32_t) * kHashCap;
  s.hval = reinterpret_cast<float*>(base + off);
  off += sizeof(float) * kHashCap;
  s.cand = reinterpret_cast<Cand*>(base + off);
  off += sizeof(Cand) * kCandCap;
  off = align_up(off, 16);
  s.hist_c = reinterpret_cast<uint32_t*>(base + off);
  off += sizeof(uint32_t) * kThreads;
  s.hist_w = reinterpret_cast<unsigned long long*>(base + off);
  off += sizeof(unsigned long long) * 256;
  s.mrg_c = reinterpret_cast<uint32_t*>(base + off);
  off += sizeof(uint32_t) * 2 * 256;
  s.mrg_w = reinterpret_cast<unsigned long long*>(base + off);
  return s;
}

// ---------------------------------------------------------------- slice access

template <bool kBF16>
struct Slice {
  const unsigned char* raw;
  // four raw logits of tokens 4f .. 4f+3 of the slice, widened to f32
  __device__ __forceinline__ float4 load4(int f) const {
    if (kBF16) {
      const uint2 w = reinterpret_cast<const uint2*>(raw)[f];
      return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                         __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
    } else {
      return reinterpret_cast<const float4*>(raw)[f];
    }
  }
  __device__ __forceinline__ float load1(int i) const {
    if (kBF16) return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(raw)[i] << 16);
    return reinterpret_cast<const float*>(raw)[i];
  }
};

__device__ __forceinline__ float comp(const float4& v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// live bits of tokens 4f .. 4f+3
__device__ __forceinline__ uint32_t live4(const uint32_t* live, int f) {
  return (live[f >> 3] >> ((f & 7) * 4)) & 0xFu;
}

// ---------------------------------------------------------------- hash of penalised ids

// Inserts local id l; returns its slot, or -1 when the table is full (bounded probing).
__device__ __forceinline__ int hash_insert(uint32_t* hkey, uint32_t l) {
  const uint32_t h = (l * 2654435761u) & (kHashCap - 1);
  for (int probe = 0; probe < kHashCap; ++probe) {
    const uint32_t slot = (h + probe) & (kHashCap - 1);
    const uint32_t prev = atomicCAS(&hkey[slot], kEmpty, l);
    if (prev == kEmpty || prev == l) return (int)slot;
  }
  return -1;
}

// Slot of local id l (which must be present); -1 if absent (bounded probing).
__device__ __forceinline__ int hash_find(const uint32_t* hkey, uint32_t l) {
  const uint32_t h = (l * 2654435761u) & (kHashCap - 1);
  for (int probe = 0; probe < kHashCap; ++probe) {
    const uint32_t slot = (h + probe) & (kHashCap - 1);
    const uint32_t k = hkey[slot];
    if (k == l) return (int)slot;
    if (k == kEmpty) return -1;
  }
  return -1;
}

// ---------------------------------------------------------------- warp / block helpers

__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2, float c) {
  const float mm = fmaxf(m, m2);
  if (mm == -INFINITY) {
    m = mm;
    s = 0.0f;
    return;
  }
  s = s * ex2_approx((m - mm) * c) + s2 * ex2_approx((m2 - mm) * c);
  m = mm;
}

__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// Block-wide sum of a u64 (all threads receive it).  `red` holds kWarps entries.
__device__ unsigned long long block_sum_u64(unsigned long long v, unsigned long long* red) {
  v = warp_sum_u64(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long t = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t += red[w];
  return t;
}

__device__ int block_min_i(int v, int* red) {
  v = warp_min_i(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  int t = INT_MAX;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t = min(t, red[w]);
  return t;
}

// Race partials of one thread, reduced over the block into `out` (thread 0 writes).
struct Race {
  float s;      // best score
  int tok;      // its id
  float ybest;  // its y
  int kept;
  float ymin;
  __device__ void init() {
    s = -INFINITY;
    tok = INT_MAX;
    ybest = -INFINITY;
    kept = 0;
    ymin = INFINITY;
  }
  __device__ __forceinline__ void add(float y, int id, uint32_t word) {
    ++kept;
    ymin = fminf(ymin, y);
    const float sc = race_score(y, word);
    if (better(sc, id, s, tok)) {
      s = sc;
      tok = id;
      ybest = y;
    }
  }
  __device__ void merge(float s2, int t2, float yb2, int k2, float y2) {
    if (better(s2, t2, s, tok)) {
      s = s2;
      tok = t2;
      ybest = yb2;
    }
    kept += k2;
    ymin = fminf(ymin, y2);
  }
  __device__ void merge(const X2& x) { merge(x.race_s, x.race_tok, x.ytok, x.kept, x.ymin); }
  // a kept token that provably cannot win the race
  __device__ __forceinline__ void count_only(float y) {
    ++kept;
    ymin = fminf(ymin, y);
  }
  __device__ void warp_reduce() {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      const float s2 = __shfl_xor_sync(0xffffffffu, s, d);
      const int t2 = __shfl_xor_sync(0xffffffffu, tok, d);
      const float b2 = __shfl_xor_sync(0xffffffffu, ybest, d);
      const int k2 = __shfl_xor_sync(0xffffffffu, kept, d);
      const float y2 = __shfl_xor_sync(0xffffffffu, ymin, d);
      merge(s2, t2, b2, k2, y2);
    }
  }
  __device__ void to(X2& x) const {
    x.race_s = s;
    x.race_tok = tok;
    x.ytok = ybest;
    x.kept = kept;
    x.ymin = ymin;
  }
};

// Block reduction of the race; thread 0 receives the result.  `buf` holds kWarps X2.
__device__ void block_reduce_race(Race& r, X2* buf) {
  r.warp_reduce();
  __syncthreads();
  if ((threadIdx.x & 31) == 0) r.to(buf[threadIdx.x >> 5]);
  __syncthreads();
  if (threadIdx.x == 0) {
    Race t;
    t.init();
    for (int w = 0; w < kWarps; ++w) t.merge(buf[w]);
    r = t;
  }
}

// Writes a sampled row's outputs.
__device__ void write_sampled(const clsample_args_t& a, int row, const Race& r, float lnS, bool ok) {
  ok = ok && r.tok != INT_MAX;
  a.tokens[row] = ok ? r.tok : -1;
  if (a.logprobs) a.logprobs[row] = ok ? r.ybest - lnS : -INFINITY;
  if (a.row_status) a.row_status[row] = ok ? kRowOk : kRowOverflow;
  if (a.dbg_kept_count) a.dbg_kept_count[row] = ok ? r.kept : 0;
  if (a.dbg_cut) a.dbg_cut[row] = ok ? r.ymin : -INFINITY;
}

// Pushes the calling CTA's record `*mine` into slot `rank` of `dst` in every CTA of the
// cluster (threads 0 .. C-1 each write one copy).  A cluster barrier must follow.
template <typename T>
__device__ __forceinline__ void push_all(const cg::cluster_group& cluster, T* dst, const T* mine, int rank,
                                         int C) {
  if ((int)threadIdx.x < C) *cluster.map_shared_rank(dst + rank, (unsigned)threadIdx.x) = *mine;
}

// ---------------------------------------------------------------- radix digit choice

// Given a 256-bin histogram (top bin = largest keys), finds the bin where the running
// total from the top first reaches `target`; writes the bin and the total above it.
// Run by one full warp.  Sets *none when the histogram holds less than `target`.
template <typename H>
__device__ void pick_digit(const H* hist, unsigned long long target, int* digit, unsigned long long* above,
                           int* none) {
  const int lane = threadIdx.x & 31;
  unsigned long long v[8];
  unsigned long long lsum = 0;
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    v[t] = hist[255 - 8 * lane - t];
    lsum += v[t];
  }
  unsigned long long incl = lsum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const unsigned long long o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  const uint32_t hit = __ballot_sync(0xffffffffu, incl >= target);
  if (hit == 0) {
    if (lane == 0) {
      *none = 1;
      *digit = 0;
      *above = 0;
    }
    return;
  }
  const int first = __ffs(hit) - 1;
  if (lane == first) {
    unsigned long long cum = incl - lsum;
    int d = 255 - 8 * lane - 7;
    for (int t = 0; t < 8; ++t) {
      if (cum + v[t] >= target) {
        d = 255 - 8 * lane - t;
        break;
      }
      cum += v[t];
    }
    *none = 0;
    *digit = d;
    *above = cum;
  }
}

// Adds one element to a local radix histogram with warp aggregation.  Every lane of the
// warp must call it (pred false for lanes without an element).
template <bool kWeighted>
__device__ __forceinline__ void hist_add(uint32_t* hc, unsigned long long* hw, bool pred, uint32_t digit,
                                         unsigned long long w) {
  const uint32_t d = pred ? digit : 0xFFFFFFFFu;
  const uint32_t peers = __match_any_sync(0xffffffffu, d);
  const int lane = threadIdx.x & 31;
  const bool leader = pred && lane == __ffs(peers) - 1;
  if (!kWeighted) {
    if (leader) atomicAdd(&hc[digit], (uint32_t)__popc(peers));
  } else {
    // weights < 2^41: sum the low 21 bits and the high part separately (each < 2^26)
    const uint32_t lo = pred ? (uint32_t)(w & 0x1FFFFFu) : 0u;
    const uint32_t hi = pred ? (uint32_t)(w >> 21) : 0u;
    const uint32_t slo = __reduce_add_sync(peers, lo);
    const uint32_t shi = __reduce_add_sync(peers, hi);
    if (leader) atomicAdd(&hw[digit], ((unsigned long long)shi << 21) + slo);
  }
}

// ---------------------------------------------------------------- per-token helpers

// max of |a|, |b| that propagates NaN: a float4 is finite iff the max of its four
// magnitudes is below +inf.
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ bool finite4(const float4& v) {
  return max_nan(max_nan(fabsf(v.x), fabsf(v.y)), max_nan(fabsf(v.z), fabsf(v.w))) < INFINITY;
}

// Smallest float z with y_of(z, m, invT) >= theta (theta <= 0).  y_of is monotone in z,
// so {candidates : y >= theta} = {candidates : z >= result} exactly.
__device__ float z_threshold(float theta, float m, float invT) {
  if (!(theta > -INFINITY)) return -INFINITY;
  if (y_of(-FLT_MAX, m, invT) >= theta) return -FLT_MAX;
  uint32_t lo = fkey(-FLT_MAX), hi = fkey(m);  // y(lo) < theta <= y(hi) = 0
  while (hi - lo > 1u) {
    const uint32_t mid = lo + (hi - lo) / 2u;
    if (y_of(key_to_float(mid), m, invT) >= theta) hi = mid;
    else lo = mid;
  }
  return key_to_float(hi);
}

// Warp-cooperative version of z_threshold: a 32-ary search over float keys (about
// seven steps); every lane returns the result.  The whole warp must call it.
__device__ float z_threshold_warp(float theta, float m, float invT) {
  if (!(theta > -INFINITY)) return -INFINITY;
  if (y_of(-FLT_MAX, m, invT) >= theta) return -FLT_MAX;
  const int lane = threadIdx.x & 31;
  uint32_t lo = fkey(-FLT_MAX), hi = fkey(m);  // y(lo) < theta <= y(hi)
  while (hi - lo > 1u) {
    const uint32_t s1 = hi - lo - 1u;  // probes lie in [lo + 1, hi - 1]
    const uint32_t probe = lo + 1u + (uint32_t)(((unsigned long long)lane * s1) / 32ull);
    const bool ok = y_of(key_to_float(probe), m, invT) >= theta;
    const uint32_t bal = __ballot_sync(0xffffffffu, ok);
    if (bal) {
      const int first = __ffs(bal) - 1;
      const uint32_t pf = __shfl_sync(0xffffffffu, probe, first);
      const uint32_t pb = __shfl_sync(0xffffffffu, probe, first > 0 ? first - 1 : 0);
      hi = pf;
      if (first > 0) lo = pb;
    } else {
      lo = __shfl_sync(0xffffffffu, probe, 31);
    }
  }
  return key_to_float(hi);
}

// -ln(-ln U) over the 23-bit uniform grid stays below 16.64, so a token with
// y + kGumbelMax < best cannot win (or tie) the race.
constexpr float kGumbelMax = 16.75f;

// y-bins of the top-p histogram: bin b holds -(b+1)/4 < y <= -b/4; the last bin also
// holds everything below.
constexpr int kPBins = 64;
__device__ __forceinline__ int pbin(float y) {
  const int b = __float2int_rz(__fmul_rn(-y, 4.0f));
  return b < kPBins - 1 ? b : kPBins - 1;
}

// ---------------------------------------------------------------- the kernel

template <bool kBF16>
__global__ void __launch_bounds__(kThreads, 2) sampler_kernel(const LaunchParams P) {
  extern __shared__ __align__(128) unsigned char smem_base[];
  __shared__ X1 x1[kMaxCluster];
  __shared__ X2 x2[kMaxCluster];
  __shared__ X1 x1_mine;
  __shared__ X2 x2_mine;
  __shared__ __align__(8) unsigned long long mbar_load;
  __shared__ __align__(8) unsigned long long mbar_gather;
  __shared__ RowParams rp;
  __shared__ RowState rs;
  __shared__ float red_f[kWarps * 2];
  __shared__ int red_i[kWarps * 2];
  __shared__ unsigned long long red_u[kWarps];
  __shared__ X2 red_x[kWarps];
  __shared__ float red_wb[kWarps * 2];
  __shared__ int sh_csr[4];
  __shared__ float sh_zth, sh_res;
  __shared__ int sh_bstar, sh_nl;
  __shared__ int sh_flags, sh_count, sh_digit, sh_none;
  __shared__ unsigned long long sh_above;

  const cg::cluster_group cluster = cg::this_cluster();
  const clsample_args_t& a = P.a;
  const int C = P.C;
  const int chunk = P.chunk;
  const int cap = P.cap;
  const int rank = (int)cluster.block_rank();
  const int row = (int)(blockIdx.x / (unsigned)C);
  const int V = a.V;
  const int c0 = rank * chunk;
  const int len = max(0, min(V, c0 + chunk) - c0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nvec = chunk / 4;
  constexpr int kEsize = kBF16 ? 2 : 4;
  const Smem S = carve(smem_base, chunk, kEsize);
  const Slice<kBF16> sl{S.raw};
  const unsigned char* gsrc =
      reinterpret_cast<const unsigned char*>(a.logits) + ((long long)row * a.logits_row_stride + c0) * kEsize;
  const int32_t* bmrow = a.bitmask ? a.bitmask + (long long)row * a.bitmask_row_stride : nullptr;
  const bool has_hist = a.hist_offs != nullptr;
  const bool has_bias = a.bias_offs != nullptr;
  const bool has_mod = has_hist || has_bias;
  const uint32_t bulk_bytes = P.bulk_ok ? (uint32_t)(((size_t)len * kEsize) & ~(size_t)15) : 0u;

  // DSMEM may only be touched once every CTA of the cluster runs: arrive now, wait just
  // before the first push.
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  // ---- 0. the slice's bulk copy starts first; the row's small inputs are fetched in
  //         parallel by different warps (one memory round trip)
  if (tid == 0) {
    sh_flags = 0;
    sh_count = 0;
    mbar_init(&mbar_load, 1);
    mbar_init(&mbar_gather, (uint32_t)C);
    fence_mbar_init();
    if (bulk_bytes) {
      mbar_arrive_expect_tx(&mbar_load, bulk_bytes);
      const uint32_t piece = ((bulk_bytes + kBulkPieces - 1) / kBulkPieces + 15u) & ~15u;
      for (uint32_t off = 0; off < bulk_bytes; off += piece) {
        const uint32_t sz = bulk_bytes - off < piece ? bulk_bytes - off : piece;
        bulk_copy_g2s(S.raw + off, gsrc + off, sz, &mbar_load);
      }
    } else {
      mbar_arrive_local(&mbar_load);
    }
  } else if (tid == 32) {
    RowParams q;
    q.T = a.temperatures ? a.temperatures[row] : 1.0f;
    q.k = a.top_ks ? a.top_ks[row] : -1;
    q.p = a.top_ps ? a.top_ps[row] : 1.0f;
    q.mp = a.min_ps ? a.min_ps[row] : 0.0f;
    q.rep = a.rep ? a.rep[row] : 1.0f;
    q.freq = a.freq ? a.freq[row] : 0.0f;
    q.pres = a.pres ? a.pres[row] : 0.0f;
    q.seed = a.seeds ? (unsigned long long)a.seeds[row] : 0ull;
    q.pos = (unsigned long long)(a.positions ? a.positions[row] : a.step);
    int bad = 0;
    bad |= (q.T != q.T) || (q.T == INFINITY);
    bad |= (q.k < -1);
    bad |= !(q.p > 0.0f && q.p <= 1.0f);
    bad |= !(q.mp >= 0.0f && q.mp <= 1.0f);
    bad |= !(q.rep > 0.0f) || (q.rep == INFINITY) || !isfinite(q.freq) || !isfinite(q.pres);
    q.invalid = bad;
    rp = q;
  } else if (tid == 64) {
    sh_csr[0] = has_hist ? a.hist_offs[row] : 0;
    sh_csr[1] = has_hist ? a.hist_offs[row + 1] : 0;
    sh_csr[2] = has_bias ? a.bias_offs[row] : 0;
    sh_csr[3] = has_bias ? a.bias_offs[row + 1] : 0;
  }
  // live words: allowed by the bitmask and inside the row
  for (int w = tid; w < chunk / 32; w += kThreads) {
    const int e = 32 * w;
    uint32_t word = 0u;
    if (e < len) {
      word = bmrow ? (uint32_t)__ldg(bmrow + (c0 >> 5) + w) : 0xFFFFFFFFu;
      const int rem = len - e;
      if (rem < 32) word &= (1u << rem) - 1u;
    }
    S.live[w] = word;
  }
  if (has_mod) {
    for (int i = tid; i < kHashCap; i += kThreads) {
      S.hkey[i] = kEmpty;
      S.hcnt[i] = 0u;
      S.hbias[i] = -1;
    }
  }
  for (int i = tid; i < 2 * 256; i += kThreads) {
    S.mrg_c[i] = 0u;
    S.mrg_w[i] = 0ull;
  }
  __syncthreads();

  // ---- penalised / biased tokens of this slice (SGLang page, "Order semantics of the
  //      penalties" and "Why logit_bias is built from triples": last duplicate wins)
  if (has_mod) {
    int flags = 0;
    const int c1 = c0 + len;
    const int hlo = sh_csr[0], hhi = sh_csr[1], blo = sh_csr[2], bhi = sh_csr[3];
    if (hlo < 0 || hhi < hlo || blo < 0 || bhi < blo) flags |= kFlagInvalid;
    const bool hok = has_hist && hlo >= 0 && hhi >= hlo;
    const bool bok = has_bias && blo >= 0 && bhi >= blo;
    // this thread's first bias entry is fetched together with the history ids
    const int bj0 = blo + tid;
    int bid0 = INT_MIN;
    float bval0 = 0.0f;
    if (bok && bj0 < bhi) {
      bid0 = __ldg(a.bias_ids + bj0);
      bval0 = __ldg(a.bias_vals + bj0);
    }
    if (hok) {
      for (int base = hlo; base < hhi; base += 8 * kThreads) {
        int ids[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = base + u * kThreads + tid;
          ids[u] = j < hhi ? __ldg(a.hist_ids + j) : INT_MIN;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int id = ids[u];
          if (id == INT_MIN) continue;
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
    // bias: the largest entry index per id wins; its owner then stores the value
    int myslot = -1;
    if (bok) {
      for (int j = bj0; j < bhi; j += kThreads) {
        const int id = j == bj0 ? bid0 : __ldg(a.bias_ids + j);
        const float b = j == bj0 ? bval0 : __ldg(a.bias_vals + j);
        if (id < 0 || id >= V || b != b) {
          flags |= kFlagInvalid;
        } else if (id >= c0 && id < c1) {
          const int slot = hash_insert(S.hkey, (uint32_t)(id - c0));
          if (slot < 0) flags |= kFlagOverflow;
          else atomicMax(&S.hbias[slot], j);
          if (j == bj0) myslot = slot;
        }
      }
    }
    if (flags) atomicOr(&sh_flags, flags);
    __syncthreads();
    if (bok) {
      for (int j = bj0; j < bhi; j += kThreads) {
        const int slot = j == bj0 ? myslot : -2;
        if (j == bj0) {
          if (slot >= 0 && S.hbias[slot] == j) S.hval[slot] = bval0;
        } else {
          const int id = __ldg(a.bias_ids + j);
          if (id >= c0 && id < c1) {
            for (int i = 0; i < kHashCap; ++i)
              if (S.hkey[i] == (uint32_t)(id - c0) && S.hbias[i] == j) S.hval[i] = __ldg(a.bias_vals + j);
          }
        }
      }
    }
  }

  // ---- 1. the slice has landed (bounded wait); rows that are not 16-byte aligned and
  //         the ragged tail come in with plain loads
  // one thread polls; the others sleep in the block barrier below
  if (tid == 0 && !mbar_wait(&mbar_load, 0)) atomicOr(&sh_flags, kFlagTimeout);
  {
    const int done = (int)(bulk_bytes / kEsize);
    for (int i = done + tid; i < len; i += kThreads) {
      if (kBF16)
        reinterpret_cast<uint16_t*>(S.raw)[i] = __ldg(reinterpret_cast<const unsigned short*>(gsrc) + i);
      else
        reinterpret_cast<float*>(S.raw)[i] = __ldg(reinterpret_cast<const float*>(gsrc) + i);
    }
  }
  __syncthreads();
  // the phase is complete: one poll gives every thread its own acquire of the copy
  (void)mbar_try_wait(&mbar_load, 0);
  const RowParams q = rp;

  // ---- 2. final z' of the penalised / biased tokens (the mask applies to them too);
  //         then they leave the live set and are marked in `modbits` (the histogram
  //         area is free until pass A ends), so pass A can fold them in token order
  uint32_t* modbits = S.hist_c;
  if (has_mod) {
    for (int i = tid; i < chunk / 32; i += kThreads) modbits[i] = 0u;
    for (int i = tid; i < kHashCap; i += kThreads) {
      const uint32_t l = S.hkey[i];
      if (l == kEmpty) continue;
      float z = sanitize(sl.load1((int)l));
      if (!((S.live[l >> 5] >> (l & 31)) & 1u)) z = -INFINITY;
      const uint32_t cnt = S.hcnt[i];
      if (cnt) z = apply_penalties(z, cnt, q.freq, q.pres, q.rep);
      if (S.hbias[i] >= 0) z = __fadd_rn(z, S.hval[i]);
      S.hval[i] = guard(z);
    }
    __syncthreads();
    for (int i = tid; i < kHashCap; i += kThreads) {
      const uint32_t l = S.hkey[i];
      if (l == kEmpty) continue;
      atomicAnd(&S.live[l >> 5], ~(1u << (l & 31)));
      atomicOr(&modbits[l >> 5], 1u << (l & 31));
    }
  }
  if (a.dbg_transformed) {
    float* out = a.dbg_transformed + (long long)row * V + c0;
    for (int i = tid; i < len; i += kThreads) {
      const int g = c0 + i;
      const bool allowed = !bmrow || (((uint32_t)__ldg(bmrow + (g >> 5)) >> (g & 31)) & 1u);
      out[i] = allowed ? sanitize(sl.load1(i)) : -INFINITY;
    }
    __syncthreads();
    if (has_mod)
      for (int i = tid; i < kHashCap; i += kThreads)
        if (S.hkey[i] != kEmpty) out[S.hkey[i]] = S.hval[i];
  }
  __syncthreads();

  // ---- 3. pass A: max, lazy argmax and online sum of exp((z' - max) / T_eff)
  const bool greedy = (q.T < kGreedyEps) || q.k == 0 || q.k == 1;
  const float Teff = (q.T >= kGreedyEps) ? q.T : 1.0f;
  const float cS = 1.4426950408889634f / Teff;
  // values of tokens 4f..4f+3 for pass A: live -> sanitised raw, penalised / biased ->
  // their final z' from the hash, otherwise -inf
  auto pass_a_values = [&](int f, uint32_t wd, const float4& v, float* z) {
    const uint32_t md = has_mod ? live4(modbits, f) : 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if ((wd >> j) & 1u) {
        z[j] = sanitize(comp(v, j));
      } else if ((md >> j) & 1u) {
        const int slot = hash_find(S.hkey, (uint32_t)(4 * f + j));
        z[j] = slot >= 0 ? S.hval[slot] : -INFINITY;
      } else {
        z[j] = -INFINITY;
      }
    }
  };
  // one online state: running max, sum of 2^((z - max) cS), first float4 reaching max
  struct OnlineState {
    float m, s;
    int f;
  };
  auto pass_a_step = [&](OnlineState& st, int f) {
    const uint32_t wd = live4(S.live, f);
    if (!wd && !(has_mod && live4(modbits, f))) return;
    const float4 v = sl.load4(f);
    float z[4];
    if (wd == 0xFu && finite4(v)) {
      z[0] = v.x;
      z[1] = v.y;
      z[2] = v.z;
      z[3] = v.w;
    } else {
      pass_a_values(f, wd, v, z);
    }
    const float fm = fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3]));
    if (!(fm > -INFINITY)) return;
    if (fm > st.m) {
      st.s *= ex2_approx((st.m - fm) * cS);
      st.m = fm;
      st.f = f;
    }
    const float e0 = ex2_approx((z[0] - st.m) * cS), e1 = ex2_approx((z[1] - st.m) * cS);
    const float e2 = ex2_approx((z[2] - st.m) * cS), e3 = ex2_approx((z[3] - st.m) * cS);
    st.s += (e0 + e1) + (e2 + e3);
  };
  OnlineState st0{-INFINITY, 0.0f, -1}, st1{-INFINITY, 0.0f, -1};
  for (int f = tid; f < nvec; f += 2 * kThreads) {
    pass_a_step(st0, f);
    if (f + kThreads < nvec) pass_a_step(st1, f + kThreads);
  }
  float sm = fmaxf(st0.m, st1.m), ss = 0.0f;
  if (sm > -INFINITY) ss = st0.s * ex2_approx((st0.m - sm) * cS) + st1.s * ex2_approx((st1.m - sm) * cS);
  // this thread's lowest id reaching its max: rescan the first float4 of each state
  int targ = INT_MAX;
  for (int t = 0; t < 2; ++t) {
    const OnlineState& st = t == 0 ? st0 : st1;
    if (st.f < 0 || st.m != sm) continue;
    float z[4];
    pass_a_values(st.f, live4(S.live, st.f), sl.load4(st.f), z);
    for (int j = 0; j < 4; ++j)
      if (z[j] == sm) {
        targ = min(targ, c0 + 4 * st.f + j);
        break;
      }
  }
  // warp-level lower bounds of the top-k cut from the per-thread maxima (disjoint
  // groups): a warp's j-th largest group max guarantees j tokens at or above it
  const bool topk_row = !greedy && !q.invalid && q.k >= 2;
  float wlk = -INFINITY, wlkc = INFINITY;
  if (topk_row) {
    uint32_t key = fkey(sm);
#pragma unroll
    for (int kk = 2; kk <= 32; kk <<= 1) {
#pragma unroll
      for (int j = kk >> 1; j > 0; j >>= 1) {
        const uint32_t other = __shfl_xor_sync(0xffffffffu, key, j);
        const bool up = (lane & kk) == 0;
        const bool lower = (lane & j) == 0;
        key = (lower == up) ? min(key, other) : max(key, other);
      }
    }
    // ascending across lanes: the j-th largest sits in lane 32 - j
    const int k1 = q.k, k2 = (q.k + kWarps * C - 1) / (kWarps * C);
    const uint32_t v1 = __shfl_sync(0xffffffffu, key, k1 <= 32 ? 32 - k1 : 0);
    const uint32_t v2 = __shfl_sync(0xffffffffu, key, k2 <= 32 ? 32 - k2 : 0);
    wlk = k1 <= 32 ? key_to_float(v1) : -INFINITY;
    wlkc = k2 <= 32 ? key_to_float(v2) : -INFINITY;
  }
  // block reduction of (max, sum, argmax) and of the bounds
  {
    float m2 = sm, s2 = ss;
    int a2 = targ;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, m2, d);
      const float os = __shfl_xor_sync(0xffffffffu, s2, d);
      const int oa = __shfl_xor_sync(0xffffffffu, a2, d);
      if (better(om, oa, m2, a2)) a2 = oa;
      merge_ms(m2, s2, om, os, cS);
    }
    if (lane == 0) {
      red_f[warp * 2] = m2;
      red_f[warp * 2 + 1] = s2;
      red_i[warp * 2] = a2;
      red_wb[warp * 2] = wlk;
      red_wb[warp * 2 + 1] = wlkc;
    }
    __syncthreads();
    if (warp == 0) {
      const bool in = lane < kWarps;
      float m = in ? red_f[lane * 2] : -INFINITY, s = in ? red_f[lane * 2 + 1] : 0.0f;
      int arg = in ? red_i[lane * 2] : INT_MAX;
      float lk = in ? red_wb[lane * 2] : -INFINITY, lkc = in ? red_wb[lane * 2 + 1] : INFINITY;
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, d);
        const float os = __shfl_xor_sync(0xffffffffu, s, d);
        const int oa = __shfl_xor_sync(0xffffffffu, arg, d);
        if (better(om, oa, m, arg)) arg = oa;
        merge_ms(m, s, om, os, cS);
        lk = fmaxf(lk, __shfl_xor_sync(0xffffffffu, lk, d));
        lkc = fminf(lkc, __shfl_xor_sync(0xffffffffu, lkc, d));
      }
      if (lane == 0) {
        x1_mine.m = m;
        x1_mine.s = s;
        x1_mine.arg = arg;
        x1_mine.lk = lk;
        x1_mine.lkc = topk_row ? lkc : -INFINITY;
        x1_mine.flags = sh_flags;
      }
    }
  }
  __syncthreads();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  push_all(cluster, x1, &x1_mine, rank, C);
  cluster.sync();  // exchange 1

  // ---- 4. row statistics, combined identically by every CTA
  if (warp == 0) {
    const bool in = lane < C;
    const float lm = in ? x1[lane].m : -INFINITY;
    const int la = in ? x1[lane].arg : INT_MAX;
    float m = lm;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
    int arg = (in && lm == m) ? la : INT_MAX;
    arg = warp_min_i(arg);
    const float term = (in && lm > -INFINITY) ? x1[lane].s * ex2_approx((lm - m) * cS) : 0.0f;
    float tot = 0.0f;  // fixed order (lanes 0..31): every CTA gets the same bits
    for (int r = 0; r < 32; ++r) tot += __shfl_sync(0xffffffffu, term, r);
    int fl = in ? x1[lane].flags : 0;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) fl |= __shfl_xor_sync(0xffffffffu, fl, d);
    float lk = in ? x1[lane].lk : -INFINITY;
    float lkc = in ? x1[lane].lkc : INFINITY;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      lk = fmaxf(lk, __shfl_xor_sync(0xffffffffu, lk, d));
      lkc = fminf(lkc, __shfl_xor_sync(0xffffffffu, lkc, d));
    }
    if (lane == 0) {
      rs.m = m;
      rs.arg = arg;
      rs.S = tot;
      rs.flags = fl;
      rs.bound = fmaxf(lk, lkc);
    }
  }
  __syncthreads();
  const float m = rs.m;
  int status = kRowOk;
  if (q.invalid || (rs.flags & kFlagInvalid) || !(m > -INFINITY)) status = kRowInvalid;
  else if (rs.flags & (kFlagOverflow | kFlagTimeout)) status = kRowOverflow;
  const float lnS = logf(rs.S);

  if (status != kRowOk || greedy) {
    if (rank == 0 && tid == 0) {
      const bool ok = status == kRowOk;
      a.tokens[row] = ok ? rs.arg : -1;
      if (a.logprobs) a.logprobs[row] = ok ? -lnS : -INFINITY;  // y of the argmax is 0
      if (a.row_status) a.row_status[row] = status;
      if (a.dbg_kept_count) a.dbg_kept_count[row] = ok ? 1 : 0;
      if (a.dbg_cut) a.dbg_cut[row] = ok ? 0.0f : -INFINITY;
    }
    if ((rs.flags & kFlagTimeout) && tid == 0) mbar_wait(&mbar_load, 0);
    return;  // every remote access of this row happened before the barrier
  }

  // ---- 5. truncation plan.  y = (z' - m) * (1/T); K = {y >= cut} is an upper set.
  const float invT = __frcp_rn(q.T);
  const float L = q.mp > 0.0f ? (float)log((double)q.mp) : -INFINITY;  // min-p: y >= ln(min_p)
  const bool kfin = q.k >= 2;
  enum { kFast, kTopP, kUntrunc, kSlow };
  int plan = kSlow;
  bool needW = false;
  float theta = -INFINITY;
  if (kfin && rs.bound > -INFINITY) {
    plan = kFast;  // every token of S_k has y >= y(bound)
    theta = y_of(rs.bound, m, invT);
    if (q.p >= 1.0f) theta = fmaxf(theta, L);
  } else if (q.mp > 0.0f && (q.p >= 1.0f || !kfin)) {
    plan = kFast;  // K lies in {y >= ln min_p}
    theta = L;
    needW = q.p < 1.0f;  // top-p renormalises over the whole row
  } else if (!kfin && q.p >= 1.0f) {
    plan = kUntrunc;  // K = every allowed token
  } else if (!kfin) {
    plan = kTopP;  // top-p alone
  }
  const unsigned long long seed = q.seed, pos = q.pos;
  Cand* cand = S.cand;

  // ---- the leader's part after a gather: top-k -> top-p -> min-p and the race over
  //      the candidates every CTA stored into its slot of the leader's raw slice
  const Cand* G = reinterpret_cast<const Cand*>(S.raw);
  const int span = C * cap;
  const int lgcap = __ffs(cap) - 1;  // cap is a power of two
  auto gvalid = [&](int i) -> bool { return i < span && (i & (cap - 1)) < x2[i >> lgcap].count; };
  // radix select over the gathered set (entries with y >= ylo); see pick_digit
  auto local_select = [&](bool weighted, float ylo, unsigned long long target, bool* found) -> float {
    uint32_t prefix = 0u, pmask = 0u;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      if (tid < 256) {
        S.hist_c[tid] = 0u;
        S.hist_w[tid] = 0ull;
      }
      __syncthreads();
      for (int base = 0; base < span; base += kThreads) {
        const int i = base + tid;
        const bool ok = gvalid(i);
        const float y = ok ? G[i].y : -INFINITY;
        const uint32_t key = fkey(y);
        const bool pred = ok && y >= ylo && (key & pmask) == prefix;
        if (weighted)
          hist_add<true>(S.hist_c, S.hist_w, pred, (key >> shift) & 0xFFu, pred ? weight_fx(y) : 0ull);
        else
          hist_add<false>(S.hist_c, S.hist_w, pred, (key >> shift) & 0xFFu, 0ull);
      }
      __syncthreads();
      if (warp == 0) {
        if (weighted) pick_digit(S.hist_w, target, &sh_digit, &sh_above, &sh_none);
        else pick_digit(S.hist_c, target, &sh_digit, &sh_above, &sh_none);
      }
      __syncthreads();
      if (sh_none) {
        *found = false;
        __syncthreads();
        return -INFINITY;
      }
      prefix |= (uint32_t)sh_digit << shift;
      pmask |= 0xFFu << shift;
      target -= sh_above;
      __syncthreads();
    }
    *found = true;
    return key_to_float(prefix);
  };
  // Exact select over the gathered set, entries with y >= ylo, all within [lo, hi]:
  // one 1024-bucket histogram (bucket order follows y), then the crossing bucket's
  // entries are resolved by counting.  Sets *resolved = false when that bucket holds
  // more than 1024 entries (heavy ties); the caller then uses local_select.
  auto bucket_select = [&](bool weighted, float lo, float hi, float ylo, unsigned long long target,
                           bool* found, bool* resolved) -> float {
    unsigned long long* bk = reinterpret_cast<unsigned long long*>(S.hist_c);  // hist + mrg: 10 KB
    const float scale = hi > lo ? 1024.0f / (hi - lo) : 0.0f;
    auto bucket = [&](float y) -> int {
      const int b = __float2int_rz(__fmul_rn(hi - y, scale));
      return b < 0 ? 0 : (b > 1023 ? 1023 : b);
    };
    bk[2 * tid] = 0ull;
    bk[2 * tid + 1] = 0ull;
    if (tid == 0) {
      sh_nl = 0;
      sh_bstar = -1;
    }
    __syncthreads();
    for (int i = tid; i < span; i += kThreads) {
      if (!gvalid(i)) continue;
      const float y = G[i].y;
      if (!(y >= ylo)) continue;
      atomicAdd(&bk[bucket(y)], weighted ? weight_fx(y) : 1ull);
    }
    __syncthreads();
    {
      const unsigned long long v0 = bk[2 * tid], v1 = bk[2 * tid + 1], loc = v0 + v1;
      unsigned long long x = loc;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const unsigned long long o = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += o;
      }
      if (lane == 31) red_u[warp] = x;
      __syncthreads();
      unsigned long long before = 0;
      for (int w = 0; w < warp; ++w) before += red_u[w];
      const unsigned long long excl = before + x - loc, incl = before + x;
      if (excl < target && target <= incl) {
        if (excl + v0 >= target) {
          sh_bstar = 2 * tid;
          sh_above = excl;
        } else {
          sh_bstar = 2 * tid + 1;
          sh_above = excl + v0;
        }
      }
    }
    __syncthreads();
    const int bstar = sh_bstar;
    if (bstar < 0) {
      *found = false;
      *resolved = true;
      return -INFINITY;
    }
    const unsigned long long t2 = target - sh_above;
    // the crossing bucket's entries, gathered into the (now free) histogram area
    Cand* Lb = reinterpret_cast<Cand*>(S.hist_c);
    for (int i = tid; i < span; i += kThreads) {
      if (!gvalid(i)) continue;
      const Cand cd = G[i];
      if (!(cd.y >= ylo) || bucket(cd.y) != bstar) continue;
      const int p = atomicAdd(&sh_nl, 1);
      if (p < 1024) Lb[p] = cd;
    }
    __syncthreads();
    const int nl = sh_nl;
    if (nl > 1024) {
      *resolved = false;
      *found = false;
      __syncthreads();
      return -INFINITY;
    }
    for (int i = tid; i < nl; i += kThreads) {
      const float yi = Lb[i].y;
      unsigned long long gt = 0, ge = 0;
      for (int j = 0; j < nl; ++j) {
        const float yj = Lb[j].y;
        const unsigned long long wj = weighted ? weight_fx(yj) : 1ull;
        if (yj > yi) gt += wj;
        if (yj >= yi) ge += wj;
      }
      if (gt < t2 && t2 <= ge) sh_res = yi;
    }
    __syncthreads();
    *found = true;
    *resolved = true;
    return sh_res;
  };
  // selects with the bucket method, falling back to the radix select
  auto leader_select = [&](bool weighted, float lo, float hi, float ylo, unsigned long long target,
                           bool* found) -> float {
    bool resolved;
    const float v = bucket_select(weighted, lo, hi, ylo, target, found, &resolved);
    if (resolved) return v;
    return local_select(weighted, ylo, target, found);
  };
  // every CTA stores its `count` candidates into slot `rank` of the leader's raw slice
  // and arrives on the leader's gather barrier; only the leader continues
  auto gather = [&](int count) -> bool {
    Cand* dst = cluster.map_shared_rank(reinterpret_cast<Cand*>(S.raw), 0u) + rank * cap;
    for (int i = tid; i < count; i += kThreads) dst[i] = cand[i];
    __syncthreads();
    if (tid == 0) mbar_arrive_remote(&mbar_gather, 0u);
    if (rank != 0) return false;
    if (tid == 0) sh_none = mbar_wait_cluster(&mbar_gather, 0) ? 0 : 1;
    __syncthreads();
    (void)mbar_try_wait_cluster(&mbar_gather, 0);  // every thread acquires the peers' stores
    return true;
  };
  // appends (y, id) to the slice's candidate list; the whole warp calls it
  auto append = [&](bool keep, float y, int id) {
    const uint32_t bal = __ballot_sync(0xffffffffu, keep);
    if (!bal) return;
    const int leader = __ffs(bal) - 1;
    int basepos = 0;
    if (lane == leader) basepos = atomicAdd(&sh_count, __popc(bal));
    basepos = __shfl_sync(0xffffffffu, basepos, leader);
    if (keep) {
      const int p = basepos + __popc(bal & ((1u << lane) - 1u));
      if (p < cap) cand[p] = Cand{y, id};
    }
  };
  auto finish_mine = [&](unsigned long long w, const Race& race) {
    __syncthreads();
    if (tid == 0) {
      x2_mine.count = sh_count;
      x2_mine.flags = sh_count > cap ? kFlagOverflow : 0;
      x2_mine.w = w;
      race.to(x2_mine);
    }
    __syncthreads();
    push_all(cluster, x2, &x2_mine, rank, C);
    cluster.sync();
  };

  if (plan == kFast || plan == kUntrunc) {
    // ---- pass B: compaction at z >= zth (exact), or the whole race
    if (warp == 0) {
      const float zt = z_threshold_warp(theta, m, invT);
      if (lane == 0) sh_zth = zt;
    }
    __syncthreads();
    const float zth = sh_zth;
    unsigned long long w = 0;
    Race race;
    race.init();
    for (int base = 0; base < nvec; base += kThreads) {
      const int f = base + tid;
      const uint32_t wd = f < nvec ? live4(S.live, f) : 0u;
      float z[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (wd) {
        const float4 v = sl.load4(f);
        if (wd == 0xFu && finite4(v)) {
          z[0] = v.x;
          z[1] = v.y;
          z[2] = v.z;
          z[3] = v.w;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) z[j] = ((wd >> j) & 1u) ? sanitize(comp(v, j)) : -INFINITY;
        }
        if (needW) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (z[j] > -INFINITY) w += weight_fx(y_of(z[j], m, invT));
        }
        if (plan == kUntrunc) {
          float y[4];
          bool live_any = false, worth = false;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            y[j] = z[j] > -INFINITY ? y_of(z[j], m, invT) : -INFINITY;
            if (z[j] > -INFINITY) {
              live_any = true;
              worth |= y[j] + kGumbelMax >= race.s;
            }
          }
          if (worth) {
            const uint4 x = race_words((uint32_t)((c0 >> 2) + f), seed, pos);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (z[j] > -INFINITY) race.add(y[j], c0 + 4 * f + j, pick_word(x, j));
          } else if (live_any) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (z[j] > -INFINITY) race.count_only(y[j]);
          }
        }
      }
      if (plan == kFast) {
        const bool any = __any_sync(0xffffffffu, z[0] >= zth || z[1] >= zth || z[2] >= zth || z[3] >= zth);
        if (any) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const bool keep = z[j] > -INFINITY && z[j] >= zth;
            append(keep, keep ? y_of(z[j], m, invT) : 0.0f, c0 + 4 * f + j);
          }
        }
      }
    }
    if (has_mod) {
      for (int base = 0; base < kHashCap; base += kThreads) {
        const int i = base + tid;
        float z = -INFINITY;
        if (S.hkey[i] != kEmpty) z = S.hval[i];
        const int g = c0 + (int)S.hkey[i];
        const float y = z > -INFINITY ? y_of(z, m, invT) : -INFINITY;
        if (z > -INFINITY) {
          if (needW) w += weight_fx(y);
          if (plan == kUntrunc) race.add(y, g, pick_word(race_words((uint32_t)(g >> 2), seed, pos), g & 3));
        }
        if (plan == kFast) append(z > -INFINITY && z >= zth, y, g);
      }
    }
    if (needW) w = block_sum_u64(w, red_u);
    if (plan == kUntrunc) block_reduce_race(race, red_x);
    finish_mine(w, race);  // exchange 2

    if (plan == kUntrunc) {
      // the winner is the same in every CTA; its owner writes the outputs
      if (tid == 0) {
        Race r;
        r.init();
        for (int c = 0; c < C; ++c) r.merge(x2[c]);
        const int owner = r.tok == INT_MAX ? 0 : r.tok / chunk;
        if (rank == owner) write_sampled(a, row, r, lnS, true);
      }
      if ((rs.flags & kFlagTimeout) && tid == 0) mbar_wait(&mbar_load, 0);
      return;
    }

    bool overflow = false;
    for (int c = 0; c < C; ++c) overflow |= (x2[c].flags & kFlagOverflow) != 0;
    if (!overflow) {
      if (!gather(x2[rank].count)) {
        if ((rs.flags & kFlagTimeout) && tid == 0) mbar_wait(&mbar_load, 0);
        return;
      }
      const bool gathered = sh_none == 0;
      int ntot = 0;
      for (int c = 0; c < C; ++c) ntot += x2[c].count;
      float tk = -INFINITY;
      if (kfin && ntot >= q.k) {
        bool found;
        const float v = leader_select(false, theta, 0.0f, -INFINITY, (unsigned long long)q.k, &found);
        if (found) tk = v;
      }
      float tp = -INFINITY;
      if (q.p < 1.0f) {
        unsigned long long mset = 0;
        for (int i = tid; i < span; i += kThreads)
          if (gvalid(i) && G[i].y >= tk) mset += weight_fx(G[i].y);
        mset = block_sum_u64(mset, red_u);
        unsigned long long Wk = mset;
        if (!kfin) {
          Wk = 0;
          for (int c = 0; c < C; ++c) Wk += x2[c].w;
        }
        const unsigned long long cth = ceil_scaled(Wk, q.p);
        if (mset >= cth) {
          bool found;
          const float v = leader_select(true, theta, 0.0f, tk, cth, &found);
          if (found) tp = v;
        }
      }
      const float cut = fmaxf(tk, fmaxf(tp, L));
      Race race2;
      race2.init();
      for (int i = tid; i < span; i += kThreads) {
        if (!gvalid(i)) continue;
        const Cand cd = G[i];
        if (!(cd.y >= cut)) continue;
        race2.add(cd.y, cd.id, pick_word(race_words((uint32_t)(cd.id >> 2), seed, pos), cd.id & 3));
      }
      block_reduce_race(race2, red_x);
      if (tid == 0) write_sampled(a, row, race2, lnS, gathered);
      if ((rs.flags & kFlagTimeout) && tid == 0) mbar_wait(&mbar_load, 0);
      return;
    }
  } else if (plan == kTopP) {
    // ---- pass B': exact top-p mass of the row and its histogram over quarter-unit y
    //      bins (warp-private, in the candidate area)
    unsigned long long* whist = reinterpret_cast<unsigned long long*>(S.cand);
    for (int i = tid; i < kWarps * kPBins; i += kThreads) whist[i] = 0ull;
    __syncthreads();
    unsigned long long w = 0;
    unsigned long long* mine = whist + warp * kPBins;
    for (int f = tid; f < nvec; f += kThreads) {
      const uint32_t wd = live4(S.live, f);
      if (!wd) continue;
      const float4 v = sl.load4(f);
      const bool fastv = wd == 0xFu && finite4(v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float z = fastv ? comp(v, j) : (((wd >> j) & 1u) ? sanitize(comp(v, j)) : -INFINITY);
        if (!(z > -INFINITY)) continue;
        const float y = y_of(z, m, invT);
        const unsigned long long qw = weight_fx(y);
        if (!qw) continue;
        w += qw;
        atomicAdd(mine + pbin(y), qw);
      }
    }
    if (has_mod) {
      for (int i = tid; i < kHashCap; i += kThreads) {
        if (S.hkey[i] == kEmpty) continue;
        const float z = S.hval[i];
        if (!(z > -INFINITY)) continue;
        const float y = y_of(z, m, invT);
        const unsigned long long qw = weight_fx(y);
        if (!qw) continue;
        w += qw;
        atomicAdd(mine + pbin(y), qw);
      }
    }
    w = block_sum_u64(w, red_u);
    // merge the warp histograms and push them into every CTA's merged copy
    if (tid < kPBins) {
      unsigned long long t = 0;
      for (int wp = 0; wp < kWarps; ++wp) t += whist[wp * kPBins + tid];
      if (t)
        for (int r = 0; r < C; ++r) atomicAdd(cluster.map_shared_rank(S.mrg_w + tid, (unsigned)r), t);
    }
    Race none_race;
    none_race.init();
    finish_mine(w, none_race);  // exchange 2
    unsigned long long W = 0;
    for (int c = 0; c < C; ++c) W += x2[c].w;
    const unsigned long long cth = ceil_scaled(W, q.p);
    // crossing bin: the running mass from the top first reaches cth in bin bstar
    int bstar = kPBins - 1;
    unsigned long long above = 0;
    {
      unsigned long long cum = 0;
      for (int b = 0; b < kPBins; ++b) {
        const unsigned long long nb = cum + S.mrg_w[b];
        if (nb >= cth) {
          bstar = b;
          above = cum;
          break;
        }
        cum = nb;
      }
    }
    if (bstar < kPBins - 1) {
      // ---- pass C: tokens above the crossing bin are certainly kept: race them here;
      //      tokens of the crossing bin go to the leader
      const float yhi = -(float)bstar * 0.25f, ylo = -(float)(bstar + 1) * 0.25f;
      __syncthreads();
      if (tid == 0) sh_count = 0;
      __syncthreads();
      Race race;
      race.init();
      for (int base = 0; base < nvec; base += kThreads) {
        const int f = base + tid;
        const uint32_t wd = f < nvec ? live4(S.live, f) : 0u;
        float y[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (wd) {
          const float4 v = sl.load4(f);
          const bool fastv = wd == 0xFu && finite4(v);
          bool worth = false;
          uint32_t sure = 0u;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float z = fastv ? comp(v, j) : (((wd >> j) & 1u) ? sanitize(comp(v, j)) : -INFINITY);
            if (!(z > -INFINITY)) continue;
            y[j] = y_of(z, m, invT);
            if (y[j] > yhi) {
              sure |= 1u << j;
              worth |= y[j] + kGumbelMax >= race.s;
            }
          }
          if (sure) {
            if (worth) {
              const uint4 x = race_words((uint32_t)((c0 >> 2) + f), seed, pos);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if ((sure >> j) & 1u) race.add(y[j], c0 + 4 * f + j, pick_word(x, j));
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if ((sure >> j) & 1u) race.count_only(y[j]);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) append(y[j] > ylo && y[j] <= yhi, y[j], c0 + 4 * f + j);
      }
      if (has_mod) {
        for (int base = 0; base < kHashCap; base += kThreads) {
          const int i = base + tid;
          float y = -INFINITY;
          int g = 0;
          if (S.hkey[i] != kEmpty && S.hval[i] > -INFINITY) {
            y = y_of(S.hval[i], m, invT);
            g = c0 + (int)S.hkey[i];
            if (y > yhi) race.add(y, g, pick_word(race_words((uint32_t)(g >> 2), seed, pos), g & 3));
          }
          append(y > ylo && y <= yhi, y, g);
        }
      }
      block_reduce_race(race, red_x);
      finish_mine(0ull, race);  // exchange 3
      bool overflow = false;
      for (int c = 0; c < C; ++c) overflow |= (x2[c].flags & kFlagOverflow) != 0;
      if (!overflow) {
        if (!gather(x2[rank].count)) {
          if ((rs.flags & kFlagTimeout) && tid == 0) mbar_wait(&mbar_load, 0);
          return;
        }
        const bool gathered = sh_none == 0;
        // the cut lies in the crossing bin: a weighted select over its tokens
        bool found;
        const float vstar = leader_select(true, ylo, yhi, -INFINITY, cth - above, &found);
        Race race2;
        race2.init();
        for (int i = tid; i < span; i += kThreads) {
          if (!gvalid(i)) continue;
          const Cand cd = G[i];
          if (!(cd.y >= vstar)) continue;
          race2.add(cd.y, cd.id, pick_word(race_words((uint32_t)(cd.id >> 2), seed, pos), cd.id & 3));
        }
        block_reduce_race(race2, red_x);
        if (tid == 0) {
          for (int c = 0; c < C; ++c) race2.merge(x2[c]);
          write_sampled(a, row, race2, lnS, gathered && found);
        }
        if ((rs.flags & kFlagTimeout) && tid == 0) mbar_wait(&mbar_load, 0);
        return;
      }
    }
    // the crossing bin is the open-ended last one, or the band overflowed: slow path
  }

  // ---- slow path: cluster-wide radix selects over the resident slices.  Histograms
  //      are pushed into every CTA's merged copy with DSMEM atomics, one barrier per
  //      digit; the merged copies are double-buffered and cleared after use.
  for (int i = tid; i < 2 * 256; i += kThreads) {
    S.mrg_c[i] = 0u;
    S.mrg_w[i] = 0ull;
  }
  cluster.sync();  // every merged copy is clear before the first push
  int gpass = 0;
  auto cluster_select = [&](bool weighted, float ylo, unsigned long long target, bool* found) -> float {
    uint32_t prefix = 0u, pmask = 0u;
    bool ok_all = true;
    for (int pass = 0; pass < 4; ++pass, ++gpass) {
      const int shift = 24 - 8 * pass;
      const int buf = gpass & 1;
      if (tid < 256) {
        S.hist_c[tid] = 0u;
        S.hist_w[tid] = 0ull;
      }
      __syncthreads();
      for (int base = 0; base < nvec; base += kThreads) {
        const int f = base + tid;
        const uint32_t wd = f < nvec ? live4(S.live, f) : 0u;
        const float4 v = wd ? sl.load4(f) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          bool pred = false;
          float y = -INFINITY;
          if ((wd >> j) & 1u) {
            const float z = sanitize(comp(v, j));
            if (z > -INFINITY) {
              y = y_of(z, m, invT);
              pred = y >= ylo && (fkey(y) & pmask) == prefix;
            }
          }
          const uint32_t digit = (fkey(y) >> shift) & 0xFFu;
          if (weighted)
            hist_add<true>(S.hist_c, S.hist_w, pred, digit, pred ? weight_fx(y) : 0ull);
          else
            hist_add<false>(S.hist_c, S.hist_w, pred, digit, 0ull);
        }
      }
      if (has_mod) {
        for (int base = 0; base < kHashCap; base += kThreads) {
          const int i = base + tid;
          bool pred = false;
          float y = -INFINITY;
          if (S.hkey[i] != kEmpty) {
            const float z = S.hval[i];
            if (z > -INFINITY) {
              y = y_of(z, m, invT);
              pred = y >= ylo && (fkey(y) & pmask) == prefix;
            }
          }
          const uint32_t digit = (fkey(y) >> shift) & 0xFFu;
          if (weighted)
            hist_add<true>(S.hist_c, S.hist_w, pred, digit, pred ? weight_fx(y) : 0ull);
          else
            hist_add<false>(S.hist_c, S.hist_w, pred, digit, 0ull);
        }
      }
      __syncthreads();
      for (int i = tid; i < 256 * C; i += kThreads) {
        const int bin = i & 255, r = i >> 8;
        if (weighted) {
          const unsigned long long hv = S.hist_w[bin];
          if (hv) atomicAdd(cluster.map_shared_rank(S.mrg_w + buf * 256 + bin, (unsigned)r), hv);
        } else {
          const uint32_t hv = S.hist_c[bin];
          if (hv) atomicAdd(cluster.map_shared_rank(S.mrg_c + buf * 256 + bin, (unsigned)r), hv);
        }
      }
      cluster.sync();
      if (warp == 0) {
        if (weighted) pick_digit(S.mrg_w + buf * 256, target, &sh_digit, &sh_above, &sh_none);
        else pick_digit(S.mrg_c + buf * 256, target, &sh_digit, &sh_above, &sh_none);
      }
      __syncthreads();
      const bool none = sh_none != 0;
      const int dg = sh_digit;
      const unsigned long long ab = sh_above;
      // clear this buffer for its next use (two passes later, after another barrier)
      if (tid < 256) {
        S.mrg_c[buf * 256 + tid] = 0u;
        S.mrg_w[buf * 256 + tid] = 0ull;
      }
      __syncthreads();
      if (none) ok_all = false;
      if (ok_all) {
        prefix |= (uint32_t)dg << shift;
        pmask |= 0xFFu << shift;
        target -= ab;
      }
    }
    *found = ok_all;
    return ok_all ? key_to_float(prefix) : -INFINITY;
  };

  float tk = -INFINITY;
  if (kfin) {
    bool found;
    const float v = cluster_select(false, -INFINITY, (unsigned long long)q.k, &found);
    if (found) tk = v;  // fewer than k candidates: top-k keeps them all
  }
  float tp = -INFINITY;
  if (q.p < 1.0f) {
    unsigned long long w = 0;
    for (int f = tid; f < nvec; f += kThreads) {
      const uint32_t wd = live4(S.live, f);
      if (!wd) continue;
      const float4 v = sl.load4(f);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (!((wd >> j) & 1u)) continue;
        const float z = sanitize(comp(v, j));
        if (!(z > -INFINITY)) continue;
        const float y = y_of(z, m, invT);
        if (y >= tk) w += weight_fx(y);
      }
    }
    if (has_mod)
      for (int i = tid; i < kHashCap; i += kThreads) {
        if (S.hkey[i] == kEmpty) continue;
        const float z = S.hval[i];
        if (!(z > -INFINITY)) continue;
        const float y = y_of(z, m, invT);
        if (y >= tk) w += weight_fx(y);
      }
    w = block_sum_u64(w, red_u);
    if (tid == 0) x2_mine.w = w;
    __syncthreads();
    push_all(cluster, x2, &x2_mine, rank, C);
    cluster.sync();
    unsigned long long W = 0;
    for (int c = 0; c < C; ++c) W += x2[c].w;
    bool found;
    const float v = cluster_select(true, tk, ceil_scaled(W, q.p), &found);
    if (found) tp = v;
  }
  const float cut = fmaxf(tk, fmaxf(tp, L));
  Race race;
  race.init();
  for (int f = tid; f < nvec; f += kThreads) {
    const uint32_t wd = live4(S.live, f);
    if (!wd) continue;
    const float4 v = sl.load4(f);
    float y[4];
    uint32_t keep = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      y[j] = -INFINITY;
      if (!((wd >> j) & 1u)) continue;
      const float z = sanitize(comp(v, j));
      if (!(z > -INFINITY)) continue;
      y[j] = y_of(z, m, invT);
      if (y[j] >= cut) keep |= 1u << j;
    }
    if (!keep) continue;
    const uint4 x = race_words((uint32_t)((c0 >> 2) + f), seed, pos);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if ((keep >> j) & 1u) race.add(y[j], c0 + 4 * f + j, pick_word(x, j));
  }
  if (has_mod)
    for (int i = tid; i < kHashCap; i += kThreads) {
      if (S.hkey[i] == kEmpty) continue;
      const float z = S.hval[i];
      if (!(z > -INFINITY)) continue;
      const float y = y_of(z, m, invT);
      if (!(y >= cut)) continue;
      const int g = c0 + (int)S.hkey[i];
      race.add(y, g, pick_word(race_words((uint32_t)(g >> 2), seed, pos), g & 3));
    }
  block_reduce_race(race, red_x);
  __syncthreads();
  if (tid == 0) race.to(x2_mine);
  __syncthreads();
  push_all(cluster, x2, &x2_mine, rank, C);
  cluster.sync();
  // the winner is the same in every CTA; its owner writes the outputs
  if (tid == 0) {
    Race r;
    r.init();
    for (int c = 0; c < C; ++c) r.merge(x2[c]);
    const int owner = r.tok == INT_MAX ? 0 : r.tok / chunk;
    if (rank == owner) write_sampled(a, row, r, lnS, true);
  }
  if ((rs.flags & kFlagTimeout) && tid == 0) mbar_wait(&mbar_load, 0);
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
  const long long t = tok[i];
  const uint4 x = race_words((uint32_t)((unsigned long long)t >> 2), seeds[i], (unsigned long long)pos[i]);
  u[i] = word_to_uniform(pick_word(x, (int)(t & 3)));
}

// ---------------------------------------------------------------- host side

Geometry geometry_for(int vocab, int esize) {
  Geometry g{0, 0, 0, 0};
  if (vocab <= 0) return g;
  int C = (vocab + 2047) / 2048;
  if (C > 8) C = 8;
  if (C < 1) C = 1;
  int chunk = ((vocab + C - 1) / C + 31) / 32 * 32;
  if (smem_bytes_for(chunk, 4) > 112 * 1024 && C == 8) {  // two CTAs per SM no longer fit
    C = kMaxCluster;
    chunk = ((vocab + C - 1) / C + 31) / 32 * 32;
  }
  if (chunk > kMaxChunk) return g;  // C = 0: vocabulary too large
  g.C = C;
  g.chunk = chunk;
  g.smem = (int)smem_bytes_for(chunk, esize);
  const int by_raw = (int)((size_t)chunk * esize / (sizeof(Cand) * C));
  int cap = 1;  // largest power of two within both limits
  while (cap * 2 <= by_raw && cap * 2 <= kCandCap) cap *= 2;
  g.cap = cap;
  if ((int)smem_bytes_for(chunk, 4) > 227 * 1024) g.C = 0;
  return g;
}

}  // namespace

struct clsample_handle {
  int max_batch;
  int vocab;
  int device;
  Geometry g32, g16;
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
  const Geometry g = geometry_for(vocab, 4);
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
  const Geometry g32 = geometry_for(vocab, 4), g16 = geometry_for(vocab, 2);
  if (g32.C == 0) return CLSAMPLE_ERR_VOCAB;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CLSAMPLE_ERR_CUDA;
  int major = 0, minor = 0, optin = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return CLSAMPLE_ERR_CUDA;
  if (major != 10 || minor != 3) return CLSAMPLE_ERR_DEVICE;
  if (g32.smem > optin) return CLSAMPLE_ERR_VOCAB;
  const void* k32 = reinterpret_cast<const void*>(&sampler_kernel<false>);
  const void* k16 = reinterpret_cast<const void*>(&sampler_kernel<true>);
  if (cudaFuncSetAttribute(k32, cudaFuncAttributeMaxDynamicSharedMemorySize, g32.smem) != cudaSuccess ||
      cudaFuncSetAttribute(k16, cudaFuncAttributeMaxDynamicSharedMemorySize, g16.smem) != cudaSuccess)
    return CLSAMPLE_ERR_CUDA;
  if (g32.C > 8) {
    if (cudaFuncSetAttribute(k32, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
        cudaFuncSetAttribute(k16, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      return CLSAMPLE_ERR_CUDA;
  }
  clsample_t* h = new clsample_t;
  h->max_batch = max_batch;
  h->vocab = vocab;
  h->device = dev;
  h->g32 = g32;
  h->g16 = g16;
  *out = h;
  return CLSAMPLE_SUCCESS;
}

void clsample_destroy(clsample_t* h) { delete h; }

static void fill_launch(const Geometry& g, unsigned nclusters, cudaStream_t stream, cudaLaunchConfig_t* cfg,
                        cudaLaunchAttribute* attr) {
  std::memset(cfg, 0, sizeof *cfg);
  cfg->gridDim = dim3(nclusters * (unsigned)g.C, 1, 1);
  cfg->blockDim = dim3(kThreads, 1, 1);
  cfg->dynamicSmemBytes = (size_t)g.smem;
  cfg->stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)g.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg->attrs = attr;
  cfg->numAttrs = 1;
}

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

  const bool bf16 = a->logits_dtype == CLSAMPLE_LOGITS_BF16;
  const Geometry& g = bf16 ? h->g16 : h->g32;
  const int esize = bf16 ? 2 : 4;
  LaunchParams P;
  P.a = *a;
  P.C = g.C;
  P.chunk = g.chunk;
  P.cap = g.cap;
  const uintptr_t base = reinterpret_cast<uintptr_t>(a->logits);
  P.bulk_ok = (base % 16 == 0) && (((long long)a->logits_row_stride * esize) % 16 == 0);

  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  fill_launch(g, (unsigned)a->B, reinterpret_cast<cudaStream_t>(stream), &cfg, attr);
  const cudaError_t err = bf16 ? cudaLaunchKernelEx(&cfg, sampler_kernel<true>, P)
                               : cudaLaunchKernelEx(&cfg, sampler_kernel<false>, P);
  return err == cudaSuccess ? CLSAMPLE_SUCCESS : CLSAMPLE_ERR_CUDA;
}

int clsample_occupancy(clsample_t* h, int32_t logits_dtype, int32_t* max_active_clusters) {
  if (!h || !max_active_clusters) return CLSAMPLE_ERR_NULL;
  if (logits_dtype != CLSAMPLE_LOGITS_F32 && logits_dtype != CLSAMPLE_LOGITS_BF16) return CLSAMPLE_ERR_DTYPE;
  const bool bf16 = logits_dtype == CLSAMPLE_LOGITS_BF16;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  fill_launch(bf16 ? h->g16 : h->g32, 1u, nullptr, &cfg, attr);
  int n = 0;
  const cudaError_t err = bf16 ? cudaOccupancyMaxActiveClusters(&n, sampler_kernel<true>, &cfg)
                               : cudaOccupancyMaxActiveClusters(&n, sampler_kernel<false>, &cfg);
  if (err != cudaSuccess) return CLSAMPLE_ERR_CUDA;
  *max_active_clusters = n;
  return CLSAMPLE_SUCCESS;
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
