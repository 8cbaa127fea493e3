// Batched constrained logits sampler for GB300 (sm_103a).
//
// One thread-block cluster samples one row.  The row's V logits are split into C
// contiguous slices (a multiple of 32 tokens, so that every CTA owns whole bitmask
// words), one per CTA.  A CTA keeps only small tables in shared memory (about 51 KB), so
// four CTAs share an SM and about 76 rows are in flight at once.  Logits move only
// through the TMA unit: every pass over the slice streams it through a 4-stage ring of
// 4 KB shared-memory buffers filled by bulk copies (cp.async.bulk) that complete on
// mbarriers, so the SM's load/store queues stay free for shared-memory work, shuffles and
// DSMEM.  The first pass reads HBM; later passes find the slice in L2.  Nothing but the
// per-row outputs is written back.
//
//   pass A    sanitise + mask + penalties/bias (the few penalised tokens live in a small
//             hash and get their final value on the way), slice max, lowest argmax and an
//             online sum of exp((z' - max)/T); per-thread maxima bound the top-k cut.
//   exchange  every CTA pushes its slice statistics into every CTA's shared memory
//             (DSMEM) and one cluster barrier publishes them.  Greedy rows end here.
//   pass B    the tokens that can survive truncation (y >= a provable bound) are
//             compacted; a leader CTA gathers them (DSMEM stores + a remote mbarrier
//             arrive) and finishes top-k -> top-p -> min-p and the exponential race alone.
//   slow path rows without a usable bound (very large k, compaction overflow) run
//             cluster-wide radix selects, one pass over the slice per digit.
//
// Cold, bulky steps are out-of-line functions so that the instruction stream of the hot
// path stays small.  The arithmetic that decides integers (kept set, drawn id) is exact
// and identical on any IEEE machine (sampler_math.cuh).  Page references: "SGLang source
// teardown (10): Sampling, Grammar and structured output" (SGLang page) and "GLM-5.3
// inference (7): output side" (GLM page).

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "clsample.h"
#include "cluster_sync.cuh"
#include "sampler_math.cuh"

namespace cg = cooperative_groups;

namespace {

using namespace clsample;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMinBlocks = 4;      // CTAs per SM the register budget is sized for
constexpr int kHashCap = 1024;     // hash slots of the penalty kernel
constexpr int kPenCap = 512;       // distinct penalised / biased ids per slice
constexpr int kCandCap = 4096;     // compacted candidates per slice (global scratch)
constexpr int kWhistBytes = 4096;  // top-p warp histograms (kWarps x 64 split counters)
constexpr int kMaxCluster = 8;     // portable cluster size
constexpr int kGatherCap = 4096;   // candidates the leader keeps in shared memory
constexpr int kMaxChunk = 32 * 1024;  // longest slice
constexpr int kStageBytes = 8192;     // one ring stage: two 16-byte vectors per thread
constexpr int kStages = 4;            // ring depth
constexpr int kReload = 4;            // 16-byte loads in flight per thread when re-reading
constexpr uint32_t kEmpty = 0xFFFFFFFFu;
// penalised-token table: count | kBiasBit (a logit_bias entry applies) | kAllowedBit
constexpr uint32_t kAllowedBit = 0x80000000u;
constexpr uint32_t kBiasBit = 0x40000000u;
constexpr uint32_t kCountMask = 0x3FFFFFFFu;
constexpr uint32_t kPenBias = 0x80000000u;  // in PenEntry::id

enum : int { kRowOk = 0, kRowOverflow = 1, kRowInvalid = 2 };
enum : int { kFlagInvalid = 1, kFlagOverflow = 2, kFlagRing = 4 };  // kFlagRing: a ring stage never landed
enum : int { kPlanFast = 0, kPlanTopP = 1, kPlanUntrunc = 2, kPlanSlow = 3 };

struct Geometry {
  int C;      // CTAs per row (cluster size)
  int chunk;  // tokens per CTA, multiple of 32
  int smem;   // dynamic shared memory per CTA
  int cap;    // compacted candidates per CTA the leader can gather
};

struct Cand {
  float y;
  int id;
};

// One penalised / biased token of a slice, as the penalty kernel lists it.
struct __align__(16) PenEntry {
  uint32_t id;     // local id | kPenBias when a logit_bias entry applies
  uint32_t count;  // occurrences in the row's history (saturates at kCountMask)
  float bias;      // the last bias entry's value
  uint32_t pad;
};

struct LaunchParams {
  clsample_args_t a;
  int C;
  int chunk;
  int cap;
  int vec_ok;         // every row start is 16-byte aligned: slices stream through the TMA ring
  PenEntry* pen;      // [B * C][kPenCap] penalised-token lists (scratch)
  int2* pen_n;        // [B * C] list length, flags
  Cand* cand;         // [B * C][kCandCap] compacted candidates (scratch)
  int* row_class;     // [B] cost class of each row (scratch)
  int* row_order;     // [B] the row each cluster samples, heaviest class first (scratch)
  unsigned* ticket;   // CTAs of the preparation kernel that have finished (scratch)
};

// The row sampled by the calling CTA's cluster (clusters take rows heaviest first).
__device__ __forceinline__ int cluster_row(const LaunchParams& P) {
  return __ldg(P.row_order + blockIdx.x / (unsigned)P.C);
}

// Slice statistics pushed to every CTA after pass A.
// Lower bounds of the k-th largest z' come from maxima of disjoint token groups: each
// thread keeps one maximum per stage slot (kGroups groups), and the 32 maxima of one slot
// across a warp form a "group set".  A set whose j-th largest maximum is L guarantees j
// tokens at or above L.  For j = 2^i (i < kNJ) every CTA reports the minimum of L over
// its sets that reach j maxima above -inf, and how many sets do; n such sets guarantee
// n*j tokens.
constexpr int kNJ = 6;  // j = 1, 2, 4, ..., 32

struct X1 {
  float m;         // slice max of z' (-inf if no candidate)
  int arg;         // lowest id reaching m (INT_MAX if none)
  float s;         // sum over the slice's candidates of 2^((z' - m) * log2(e) / T)
  int flags;       // kFlag*
  float lk;        // max over warps of the warp's k-th largest thread max (k <= 32; else -inf)
  float lj[kNJ];   // min over the CTA's groups reaching 2^i maxima of the 2^i-th largest
  unsigned char nj[8];  // how many groups reach 2^i (i < kNJ)
  int nallowed;    // allowed tokens of the slice (at least its candidates)
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

// Row statistics and the truncation plan, identical in every CTA after exchange 1.
struct RowState {
  float m;      // max z'
  int arg;      // lowest id reaching it
  float S;      // sum of 2^((z' - m) cS)
  int flags;
  float bound;  // lower bound of the k-th largest z' (-inf if none)
  int nallowed_max;  // the largest per-slice allowed-token count
  float lnS;
  float invT;
  float L;      // min-p cut in y: ln(min_p), or -inf
  float theta;  // lower bound of the kept set in y (kPlanFast)
  int plan;
  int needW;    // kPlanFast: the top-p mass is taken over the whole row
  int all;      // kPlanFast: every candidate of the row is compacted (theta = -inf)
  float s0;     // race score of the argmax token, which every kept set contains: a lower
                // bound of the winning score that seeds every race
};

// ---------------------------------------------------------------- shared memory

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr size_t kOffHistC = kWhistBytes;                                   // 4 KB
constexpr size_t kOffHistW = kOffHistC + sizeof(uint32_t) * 256;            // 5 KB
constexpr size_t kOffMrgC = kOffHistW + sizeof(unsigned long long) * 256;  // 7 KB
constexpr size_t kR2Bytes = 9 * 1024;

// Dynamic shared memory of one CTA (byte offsets):
//   ring      kStages x kStageBytes   the slice's stream (TMA destination); in the
//                                     leader, once every CTA has finished reading its
//                                     slice: the cluster's gathered candidates
//   live      u32[chunk/32]           allowed by the bitmask, inside the row, not penalised
//   mod       u32[chunk/32]           penalised / biased tokens
//   prank     u16[chunk/32]           rank of each mod word's first penalised token
//   pid/pcnt/pbias/pz [kPenCap]       the penalised tokens in token order: local id;
//                                     count | kBiasBit | kAllowedBit; bias; raw logit in
//                                     pass A, then the final z'
//   r2 (9 KB) cand Cand[512] | hist_c u32[256] | hist_w u64[256] | mrg_c u32[2][256];
//             mrg_w u64[2][256] overlays cand (slow path); the top-p warp histograms
//             (kWarps x 64 u64) overlay cand and their merged copy is the start of
//             mrg_c; the leader's bucket select overlays [0, 8 KB)
struct Layout {
  uint32_t live, mod, prank, pid, pcnt, pbias, pz, r2, total;
};

__host__ __device__ inline Layout layout_for(int chunk) {
  Layout L;
  const size_t words = (size_t)(chunk / 32);
  size_t off = (size_t)kStages * kStageBytes;
  L.live = (uint32_t)off;
  off = align_up(off + sizeof(uint32_t) * words, 16);
  L.mod = (uint32_t)off;
  off = align_up(off + sizeof(uint32_t) * words, 16);
  L.prank = (uint32_t)off;
  off = align_up(off + sizeof(uint16_t) * words, 16);
  L.pid = (uint32_t)off;
  off = align_up(off + sizeof(uint16_t) * kPenCap, 16);
  L.pcnt = (uint32_t)off;
  off += sizeof(uint32_t) * kPenCap;
  L.pbias = (uint32_t)off;
  off += sizeof(float) * kPenCap;
  L.pz = (uint32_t)off;
  off += sizeof(float) * kPenCap;
  L.r2 = (uint32_t)align_up(off, 128);
  L.total = L.r2 + kR2Bytes;
  return L;
}
static_assert(sizeof(Cand) * kGatherCap <= (size_t)kStages * kStageBytes, "gather area overflows the ring");
static_assert(kR2Bytes >= kOffMrgC + sizeof(uint32_t) * 2 * 256, "r2 tables overflow");
static_assert(sizeof(unsigned long long) * 2 * 256 <= kOffHistC, "mrg_w overlaps the histograms");
static_assert(sizeof(unsigned long long) * 1024 <= kR2Bytes && sizeof(Cand) * 1024 <= kR2Bytes,
              "bucket select does not fit r2");  // in the leader every r2 table is dead
static_assert(2 * sizeof(uint32_t) * kWarps * 64 <= kWhistBytes, "top-p histogram does not fit r2");
static_assert(sizeof(float) * kWarps * 4 * kNJ <= kOffMrgC, "pass A group-set bounds overlap the merged bins");
static_assert(1024 % kThreads == 0, "bucket scan assumes whole buckets per thread");
static_assert(kStageBytes % (16 * kThreads) == 0, "a stage holds whole vectors per thread");
static_assert(kPenCap % kThreads == 0 && kPenCap <= 65536 && kMaxChunk <= 65536, "16-bit ids and ranks");

extern __shared__ __align__(128) unsigned char smem_dyn[];

struct Smem {
  unsigned char* ring;
  uint32_t* live;
  uint32_t* mod;
  uint16_t* prank;
  uint16_t* pid;
  uint32_t* pcnt;
  float* pbias;
  float* pz;
  uint32_t* mrg_c;
  unsigned long long* mrg_w;
  Cand* gather;
  uint32_t* hist_c;
  unsigned long long* hist_w;
  unsigned char* r2;
};

__device__ __forceinline__ Smem carve(int chunk) {
  const Layout L = layout_for(chunk);
  unsigned char* b = smem_dyn;
  Smem s;
  s.ring = b;
  s.live = reinterpret_cast<uint32_t*>(b + L.live);
  s.mod = reinterpret_cast<uint32_t*>(b + L.mod);
  s.prank = reinterpret_cast<uint16_t*>(b + L.prank);
  s.pid = reinterpret_cast<uint16_t*>(b + L.pid);
  s.pcnt = reinterpret_cast<uint32_t*>(b + L.pcnt);
  s.pbias = reinterpret_cast<float*>(b + L.pbias);
  s.pz = reinterpret_cast<float*>(b + L.pz);
  s.r2 = b + L.r2;
  s.hist_c = reinterpret_cast<uint32_t*>(s.r2 + kOffHistC);
  s.hist_w = reinterpret_cast<unsigned long long*>(s.r2 + kOffHistW);
  s.mrg_c = reinterpret_cast<uint32_t*>(s.r2 + kOffMrgC);
  s.mrg_w = reinterpret_cast<unsigned long long*>(s.r2);
  s.gather = reinterpret_cast<Cand*>(b);
  return s;
}

// Static per-CTA state shared by the kernel's functions.
struct Shared {
  X1 x1[kMaxCluster];
  X2 x2[kMaxCluster];
  X1 x1_mine;
  X2 x2_mine;
  unsigned long long full[kStages];  // ring stage barriers (one arrival + the copy's bytes)
  RowParams rp;
  RowState rs;
  float red_f[kWarps * 2];
  int red_i[kWarps * 2];
  unsigned long long red_u[kWarps];
  X2 red_x[kWarps];
  float red_wb[kWarps * 2];
  int csr[4];
  float zth, res;
  int bstar, nl, flags, count, digit, none, npen;
  int nallowed;
  unsigned long long above;
};
__shared__ Shared sh;

// The calling CTA's place in the launch.
struct Geo {
  int C, chunk, cap, rank, row, c0, len, nvec;
  int bulk_tokens;  // tokens of the slice that stream through the ring (0: none)
  int nst;          // ring stages per pass
  const unsigned char* g;  // the slice's first logit
};

template <bool kBF16>
__device__ __forceinline__ Geo geo(const LaunchParams& P) {
  constexpr int kEsize = kBF16 ? 2 : 4;
  Geo g;
  g.C = P.C;
  g.chunk = P.chunk;
  g.cap = P.cap;
  g.rank = (int)cg::this_cluster().block_rank();
  g.row = cluster_row(P);
  g.c0 = g.rank * g.chunk;
  g.len = max(0, min(P.a.V, g.c0 + g.chunk) - g.c0);
  g.nvec = g.chunk / 4;
  const int bulk = P.vec_ok ? (int)(((size_t)g.len * kEsize) & ~(size_t)15) : 0;
  g.bulk_tokens = bulk / kEsize;
  g.nst = (bulk + kStageBytes - 1) / kStageBytes;
  g.g = reinterpret_cast<const unsigned char*>(P.a.logits) +
        ((long long)g.row * P.a.logits_row_stride + g.c0) * kEsize;
  return g;
}

// ---------------------------------------------------------------- slice access

// Raw logit i of the slice from global memory, widened to f32.
template <bool kBF16>
__device__ __forceinline__ float gload1(const unsigned char* g, int i) {
  if (kBF16) return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(g) + i) << 16);
  return __ldg(reinterpret_cast<const float*>(g) + i);
}

// Tokens 4f .. 4f+3 from global memory (plain loads; tokens past the row read as 0).
template <bool kBF16>
__device__ __forceinline__ float4 gload4(const Geo& g, int f) {
  const int i = 4 * f;
  return make_float4(i < g.len ? gload1<kBF16>(g.g, i) : 0.0f, i + 1 < g.len ? gload1<kBF16>(g.g, i + 1) : 0.0f,
                     i + 2 < g.len ? gload1<kBF16>(g.g, i + 2) : 0.0f,
                     i + 3 < g.len ? gload1<kBF16>(g.g, i + 3) : 0.0f);
}

// Tokens 4f .. 4f+3 by one aligned load (the slice start is 16-byte aligned and the
// vector lies inside the row), widened to f32.
template <bool kBF16>
__device__ __forceinline__ float4 vload4(const Geo& g, int f) {
  if (kBF16) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(g.g) + f);
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                       __uint_as_float(w.y & 0xFFFF0000u));
  }
  return __ldg(reinterpret_cast<const float4*>(g.g) + f);
}

// Vector v (4 tokens) of a ring stage buffer, widened to f32.
template <bool kBF16>
__device__ __forceinline__ float4 sload4(const unsigned char* buf, int v) {
  if (kBF16) {
    const uint2 w = reinterpret_cast<const uint2*>(buf)[v];
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                       __uint_as_float(w.y & 0xFFFF0000u));
  }
  return reinterpret_cast<const float4*>(buf)[v];
}

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

// ---------------------------------------------------------------- out-of-line math

// The exact race score and the Philox words are long instruction sequences; the cold
// call sites share one out-of-line copy of each (the per-vector race loops inline Philox,
// and the exact score is rare behind the fast screen in Race::add).
__device__ __noinline__ float race_score_call(float y, uint32_t word) { return race_score(y, word); }
__device__ __noinline__ uint4 race_words_call(uint32_t q, unsigned long long seed, unsigned long long pos) {
  return race_words(q, seed, pos);
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

// Race partials of one thread, reduced over the block into `out` (thread 0 writes).
constexpr float kScoreMargin = 1e-3f;

struct Race {
  float s;      // best score
  int tok;      // its id
  float ybest;  // its y
  int kept;
  float ymin;
  __device__ void init(float s0 = -INFINITY) {
    s = s0;
    tok = INT_MAX;
    ybest = -INFINITY;
    kept = 0;
    ymin = INFINITY;
  }
  __device__ __forceinline__ void add(float y, int id, uint32_t word) {
    ++kept;
    ymin = fminf(ymin, y);
    // screen with a fast score (within 1e-4 of the exact one): a token whose fast score
    // stays kScoreMargin below the best cannot win, so only near-winners pay for the
    // exact score.  E = -ln U: the fast logarithm for U <= 7/8; above, with t = 1 - U
    // (exact), the series t (1 + t/2 + t^2/3 + t^3/4), relative error below 1e-4.
    const float u = word_to_uniform(word);
    const float t = 1.0f - u;
    const float e = u <= 0.875f ? -__logf(u) : t * (1.0f + t * (0.5f + t * (0.33333334f + t * 0.25f)));
    if (y - __logf(e) + kScoreMargin < s) return;
    const float sc = race_score_call(y, word);
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
__device__ __noinline__ void write_sampled(const clsample_args_t& a, int row, const Race& r, float lnS, bool ok) {
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

// Adds a weight (<= 2^40) to a split 64-bit shared counter {c[0]: units of 1, c[1]: units
// of 2^21} with native 32-bit atomics; a wrap of c[0] (the adder sees it) carries 2^11
// into c[1].  Exact for up to 8191 additions; read it back with split_get.
__device__ __forceinline__ void split_add(uint32_t* c, unsigned long long w) {
  const uint32_t lo = (uint32_t)(w & 0x1FFFFFu);
  const uint32_t old = atomicAdd(c, lo);
  atomicAdd(c + 1, (uint32_t)(w >> 21) + (old + lo < old ? (1u << 11) : 0u));
}
__device__ __forceinline__ unsigned long long split_get(const uint32_t* c) {
  return ((unsigned long long)c[1] << 21) + c[0];
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
// so {candidates : y >= theta} = {candidates : z >= result} exactly.  Warp-cooperative:
// a 32-ary search over float keys (about seven steps); every lane returns the result.
// The whole warp must call it.
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

// ---------------------------------------------------------------- the TMA ring

// Issues stage k of a pass (stage sequence number s picks the buffer) on its barrier.
// Thread 0 only.
template <bool kBF16>
__device__ __forceinline__ void ring_issue(const Geo& g, const Smem& S, int k, uint32_t s) {
  constexpr int kEsize = kBF16 ? 2 : 4;
  const int off = k * kStageBytes;
  const uint32_t bytes = (uint32_t)min(kStageBytes, g.bulk_tokens * kEsize - off);
  const uint32_t slot = s % kStages;
  mbar_arrive_expect_tx(&sh.full[slot], bytes);
  bulk_copy_g2s(S.ring + slot * kStageBytes, g.g + off, bytes, &sh.full[slot]);
}

// Issues the first stages of pass `pass` (thread 0 only).
template <bool kBF16>
__device__ __forceinline__ void ring_start(const Geo& g, const Smem& S, int pass) {
  const uint32_t seq0 = (uint32_t)pass * (uint32_t)g.nst;
  for (int k = 0; k < min(kStages, g.nst); ++k) ring_issue<kBF16>(g, S, k, seq0 + k);
}

// Waits (bounded, suspending) for ring stage s.  Thread 0 only; a stage that never lands
// marks the row OVERFLOW.
__device__ __forceinline__ void ring_wait(uint32_t s) {
  if (!mbar_wait_sleep(&sh.full[s % kStages], (s / kStages) & 1u)) atomicOr(&sh.flags, kFlagRing);
}

// One pass over the slice: body(f, wd, v) for every 4-token vector f, with its live bits
// wd and raw values v widened to f32 (valid for every vector that starts inside the row;
// lanes without a vector get f = nvec, past the row, and wd = 0).
// Stage sequence numbers continue across the CTA's passes (pass p uses p*nst ..
// p*nst + nst - 1), which fixes each ring buffer's barrier parity.  Aligned rows stream
// through the ring; the ragged tail and unaligned rows come in by plain loads.  Every
// thread calls it; every lane of a warp makes the same number of body calls (wd = 0 where
// it has no vector), so bodies may use warp collectives.  `started`: thread 0 already
// issued the pass's first stages.
template <bool kBF16, bool kSlot = false, class Body>
__device__ __forceinline__ void stream(const Geo& g, const Smem& S, int& pass, bool started, Body&& body) {
  constexpr int kEsize = kBF16 ? 2 : 4;
  constexpr int kVecPerStage = kStageBytes / (4 * kEsize);
  constexpr int kVPT = kVecPerStage / kThreads;
  const int tid = threadIdx.x;
  if (pass == 0 && g.nst > 0) {
    const uint32_t seq0 = 0u;
    if (tid == 0 && !started) ring_start<kBF16>(g, S, pass);
#pragma unroll 1
    for (int k = 0; k < g.nst; ++k) {
      const uint32_t s = seq0 + (uint32_t)k;
      // thread 0 sleeps on the stage's barrier; the block barrier then also says that
      // every thread is done with stage k - 1, whose buffer is refilled at once
      if (tid == 0) ring_wait(s);
      __syncthreads();
      if (tid == 0 && k >= 1 && k - 1 + kStages < g.nst)
        ring_issue<kBF16>(g, S, k - 1 + kStages, s - 1 + kStages);
      (void)mbar_try_wait(&sh.full[s % kStages], (s / kStages) & 1u);  // this thread's acquire
      const unsigned char* buf = S.ring + (s % kStages) * kStageBytes;
#pragma unroll
      for (int t = 0; t < kVPT; ++t) {
        const int fl = t * kThreads + tid;
        const int f = k * kVecPerStage + fl;
        const bool in = 4 * f < g.bulk_tokens;
        const uint32_t wd = in ? live4(S.live, f) : 0u;
        const float4 v = in ? sload4<kBF16>(buf, fl) : make_float4(0.f, 0.f, 0.f, 0.f);
        // vectors past the ring part: f = nvec (past the row).  With kSlot the body also
        // gets the vector's slot t in the stage (a compile-time constant after unrolling)
        if constexpr (kSlot) body(in ? f : g.nvec, wd, v, t);
        else body(in ? f : g.nvec, wd, v);
      }
    }
  }
  if (pass > 0 && g.bulk_tokens > 0) {
    // later passes find the slice in L2: plain 16-byte loads, kReload per thread in
    // flight (bulk copies would queue behind the HBM copies of other CTAs' first passes)
    const int nv = g.bulk_tokens / 4;
#pragma unroll 1
    for (int base = 0; base < nv; base += kReload * kThreads) {
      float4 v[kReload];
      uint32_t wd[kReload];
#pragma unroll
      for (int u = 0; u < kReload; ++u) {
        const int f = base + u * kThreads + tid;
        const bool in = f < nv;
        wd[u] = in ? live4(S.live, f) : 0u;  // later passes read only live tokens
        v[u] = wd[u] ? vload4<kBF16>(g, f) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kReload; ++u) {
        const int f = base + u * kThreads + tid;
        if constexpr (kSlot) body(f < nv ? f : g.nvec, wd[u], v[u], 0);
        else body(f < nv ? f : g.nvec, wd[u], v[u]);
      }
    }
  }
  // the ragged tail, and whole unaligned slices: plain loads
  const int f_end = (g.len + 3) / 4;
#pragma unroll 1
  for (int base = g.bulk_tokens / 4; base < f_end; base += kThreads) {
    const int f = base + tid;
    const bool in = f < f_end;
    const uint32_t wd = in ? live4(S.live, f) : 0u;
    const float4 v = in ? gload4<kBF16>(g, f) : make_float4(0.f, 0.f, 0.f, 0.f);
    if constexpr (kSlot) body(in ? f : g.nvec, wd, v, 0);
    else body(in ? f : g.nvec, wd, v);
  }
  __syncthreads();  // the ring is free for the next pass; the bodies' shared writes are visible
  ++pass;
}

// Adds n occurrences of local id l to the history counts; kFlagOverflow if the hash is
// full.
__device__ __forceinline__ int count_id(uint32_t* hkey, uint32_t* hcnt, uint32_t l, uint32_t n) {
  const int slot = hash_insert(hkey, l);
  if (slot < 0) return kFlagOverflow;
  atomicAdd(&hcnt[slot], n);
  return 0;
}

// ---------------------------------------------------------------- row preparation

constexpr int kPrepThreads = 128;
constexpr int kPrepWarps = kPrepThreads / 32;
constexpr int kClasses = 5;

// Expected cost class of a row from its parameters alone (0 = heaviest): top-p alone,
// then untruncated or very large k, then large k or top-p over a min-p set, then the
// other sampling rows, then greedy or invalid rows.  Only the launch order uses it.
__device__ __forceinline__ int row_class(const clsample_args_t& a, int row) {
  const float T = a.temperatures ? a.temperatures[row] : 1.0f;
  const int k = a.top_ks ? a.top_ks[row] : -1;
  const float p = a.top_ps ? a.top_ps[row] : 1.0f;
  const float mp = a.min_ps ? a.min_ps[row] : 0.0f;
  if (!(T >= kGreedyEps) || k == 0 || k == 1 || k < -1) return 4;
  const bool kfin = k >= 2;
  if (!kfin && p < 1.0f && !(mp > 0.0f)) return 0;
  if ((!kfin && !(mp > 0.0f)) || k >= 512) return 1;
  if (k >= 64 || (!kfin && p < 1.0f)) return 2;
  return 3;
}

// One CTA per (row, slice), ahead of the sampler.
//  * The slice's distinct penalised or biased token ids with their history count and the
//    last bias entry (SGLang page, "Order semantics of the penalties" and "Why
//    logit_bias is built from triples": the last duplicate wins), sorted by id, into the
//    slice's scratch list.  Duplicate history ids are counted once per warp (Zipf-like
//    histories repeat their frequent ids many times).  A slice with more than kPenCap
//    distinct ids is flagged OVERFLOW.
//  * The launch order of the sampler's rows, heaviest first: every slice-0 CTA writes
//    its row's class; the last CTA to finish (a ticket counter) sorts the rows by class,
//    stably, and resets the ticket.
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const __grid_constant__ LaunchParams P) {
  __shared__ uint32_t hkey[kHashCap];
  __shared__ uint32_t hcnt[kHashCap];
  __shared__ int32_t hbias[kHashCap];
  __shared__ uint32_t mod[kMaxChunk / 32];
  __shared__ uint16_t wbase[kMaxChunk / 32];
  __shared__ int red[kPrepWarps * kClasses];
  __shared__ int csr[4];
  __shared__ int flags_sh, last_sh;
  const clsample_args_t& a = P.a;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rc = (int)blockIdx.x;  // row * C + slice
  const int row = rc / P.C, slice = rc % P.C, c0 = slice * P.chunk;
  const int len = max(0, min(a.V, c0 + P.chunk) - c0);
  const int c1 = c0 + len;
  const bool has_hist = a.hist_offs != nullptr;
  const bool has_bias = a.bias_offs != nullptr;
  if (tid == 0) {
    csr[0] = has_hist ? a.hist_offs[row] : 0;
    csr[1] = has_hist ? a.hist_offs[row + 1] : 0;
    csr[2] = has_bias ? a.bias_offs[row] : 0;
    csr[3] = has_bias ? a.bias_offs[row + 1] : 0;
    flags_sh = 0;
    if (slice == 0) P.row_class[row] = row_class(a, row);
  }
  if (has_hist || has_bias) {
    for (int i = tid; i < kHashCap; i += kPrepThreads) {
      hkey[i] = kEmpty;
      hcnt[i] = 0u;
      hbias[i] = -1;
    }
    for (int w = tid; w < P.chunk / 32; w += kPrepThreads) mod[w] = 0u;
  }
  __syncthreads();

  if (has_hist || has_bias) {
    int flags = 0;
    const int hlo = csr[0], hhi = csr[1], blo = csr[2], bhi = csr[3];
    if (hlo < 0 || hhi < hlo || blo < 0 || bhi < blo) flags |= kFlagInvalid;
    const bool hok = has_hist && hlo >= 0 && hhi >= hlo;
    const bool bok = has_bias && blo >= 0 && bhi >= blo;
    if (hok) {
      for (int base = hlo; base < hhi; base += 16 * kPrepThreads) {
        int ids[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int j = base + u * kPrepThreads + tid;
          ids[u] = j < hhi ? __ldg(a.hist_ids + j) : INT_MIN;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int id = ids[u];
          if (id != INT_MIN && (id < 0 || id >= a.V)) flags |= kFlagInvalid;
          const bool mine = id >= c0 && id < c1;
          const uint32_t peers = __match_any_sync(0xffffffffu, mine ? id : -1);
          if (mine && lane == __ffs(peers) - 1)
            flags |= count_id(hkey, hcnt, (uint32_t)(id - c0), (uint32_t)__popc(peers));
        }
      }
    }
    // bias: the largest entry index per id wins (its value is read back at the end)
    if (bok) {
      for (int j = blo + tid; j < bhi; j += kPrepThreads) {
        const int id = __ldg(a.bias_ids + j);
        const float b = __ldg(a.bias_vals + j);
        if (id < 0 || id >= a.V || b != b) {
          flags |= kFlagInvalid;
        } else if (id >= c0 && id < c1) {
          const int slot = hash_insert(hkey, (uint32_t)(id - c0));
          if (slot < 0) flags |= kFlagOverflow;
          else atomicMax(&hbias[slot], j);
        }
      }
    }
    if (flags) atomicOr(&flags_sh, flags);
    __syncthreads();
    for (int i = tid; i < kHashCap; i += kPrepThreads) {
      const uint32_t l = hkey[i];
      if (l != kEmpty) atomicOr(&mod[l >> 5], 1u << (l & 31));
    }
    __syncthreads();
    // rank of every id = ids below it: an exclusive scan of the words' popcounts
    constexpr int kPer = (kMaxChunk / 32) / kPrepThreads;
    const int nw = P.chunk / 32;
    int cnt[kPer], loc = 0;
#pragma unroll
    for (int t = 0; t < kPer; ++t) {
      const int w = tid * kPer + t;
      cnt[t] = w < nw ? __popc(mod[w]) : 0;
      loc += cnt[t];
    }
    int x = loc;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += o;
    }
    if (lane == 31) red[warp] = x;
    __syncthreads();
    int total = 0, before = 0;
    for (int w = 0; w < kPrepWarps; ++w) {
      total += red[w];
      if (w < warp) before += red[w];
    }
    int e = before + x - loc;
#pragma unroll
    for (int t = 0; t < kPer; ++t) {
      const int w = tid * kPer + t;
      if (w < nw) wbase[w] = (uint16_t)e;
      e += cnt[t];
    }
    __syncthreads();
    PenEntry* out = P.pen + (size_t)rc * kPenCap;
    for (int i = tid; i < kHashCap; i += kPrepThreads) {
      const uint32_t l = hkey[i];
      if (l == kEmpty) continue;
      const int r = wbase[l >> 5] + __popc(mod[l >> 5] & ((1u << (l & 31)) - 1u));
      if (r >= kPenCap) continue;
      PenEntry en;
      const int bj = hbias[i];
      en.id = l | (bj >= 0 ? kPenBias : 0u);
      en.count = min(hcnt[i], kCountMask);
      en.bias = bj >= 0 ? __ldg(a.bias_vals + bj) : 0.0f;
      en.pad = 0u;
      out[r] = en;
    }
    if (tid == 0) {
      int f = flags_sh;
      if (total > kPenCap) f |= kFlagOverflow;
      P.pen_n[rc] = make_int2(min(total, kPenCap), f);
    }
  }

  // the launch order, by the CTA that finishes last
  __threadfence();
  __syncthreads();
  if (tid == 0) last_sh = atomicAdd(P.ticket, 1u) == gridDim.x - 1 ? 1 : 0;
  __syncthreads();
  if (!last_sh) return;
  __threadfence();
  const int B = a.B;
  const int per = (B + kPrepThreads - 1) / kPrepThreads;  // consecutive rows per thread
  const int r0 = min(B, tid * per), r1 = min(B, r0 + per);
  int cnt[kClasses] = {0, 0, 0, 0, 0};
  for (int r = r0; r < r1; ++r) ++cnt[__ldcg(P.row_class + r)];
  // exclusive scan over threads, per class; then class offsets
  int base[kClasses];
  int cls_total[kClasses];
#pragma unroll
  for (int c = 0; c < kClasses; ++c) {
    int x = cnt[c];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += o;
    }
    if (lane == 31) red[warp * kClasses + c] = x;
    base[c] = x - cnt[c];
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < kClasses; ++c) {
    int tot = 0;
    for (int w = 0; w < kPrepWarps; ++w) {
      if (w < warp) base[c] += red[w * kClasses + c];
      tot += red[w * kClasses + c];
    }
    cls_total[c] = tot;
  }
  int start = 0;
#pragma unroll
  for (int c = 0; c < kClasses; ++c) {
    base[c] += start;
    start += cls_total[c];
  }
  for (int r = r0; r < r1; ++r) P.row_order[base[__ldcg(P.row_class + r)]++] = r;
  if (tid == 0) *P.ticket = 0u;  // ready for the next call on this stream
}

// ---------------------------------------------------------------- prologue

// Row parameters, the slice's live bits (bitmask words clipped to the row) and its
// penalised / biased tokens from the penalty kernel's list (sorted by id, so an entry's
// index is the token's rank); the bitmask's verdict on each moves into its entry.  The
// first ring stages of pass A are issued before anything else, so the slice is on its
// way while the small inputs arrive.
template <bool kBF16>
__device__ __noinline__ void prologue(const LaunchParams& P) {
  const Geo g = geo<kBF16>(P);
  const Smem S = carve(g.chunk);
  const clsample_args_t& a = P.a;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = g.row, c0 = g.c0, len = g.len;
  const int32_t* bmrow = a.bitmask ? a.bitmask + (long long)row * a.bitmask_row_stride : nullptr;
  const bool has_mod = a.hist_offs != nullptr || a.bias_offs != nullptr;
  const int rc = row * g.C + g.rank;

  if (tid == 0) {
    sh.flags = 0;
    sh.count = 0;
    sh.nallowed = 0;
    for (int i = 0; i < kStages; ++i) mbar_init(&sh.full[i], 1);
    fence_mbar_init();
    ring_start<kBF16>(g, S, 0);
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
    sh.rp = q;
  } else if (tid == 64) {
    const int2 nf = has_mod ? P.pen_n[rc] : make_int2(0, 0);
    sh.npen = nf.x;
    sh.csr[0] = nf.y;  // the penalty kernel's flags
  }
  // the list is loaded whole (its length arrives with it): two entries per thread
  PenEntry en[kPenCap / kThreads];
  if (has_mod) {
#pragma unroll
    for (int t = 0; t < kPenCap / kThreads; ++t) en[t] = P.pen[(size_t)rc * kPenCap + t * kThreads + tid];
  }
  for (int w = tid; w < g.chunk / 32; w += kThreads) {
    const int e = 32 * w;
    uint32_t word = 0u;
    if (e < len) {
      word = bmrow ? (uint32_t)__ldg(bmrow + (c0 >> 5) + w) : 0xFFFFFFFFu;
      const int rem = len - e;
      if (rem < 32) word &= (1u << rem) - 1u;
    }
    S.live[w] = word;
    S.mod[w] = 0u;
  }
  S.mrg_c[tid] = 0u;  // merged histograms peers add into (top-p bins, top-k refinement)
  __syncthreads();
  if (!has_mod) {
    int na = 0;
    for (int w = tid; w < g.chunk / 32; w += kThreads) na += __popc(S.live[w]);
    na = __reduce_add_sync(0xffffffffu, na);
    if (lane == 0 && na) atomicAdd(&sh.nallowed, na);
    return;
  }
  const int npen = sh.npen;
  if (tid == 0 && sh.csr[0]) sh.flags |= sh.csr[0];
  // the bitmask's verdict on each penalised token moves into its entry; the token
  // leaves the live set (pass A gives it its final value)
#pragma unroll
  for (int t = 0; t < kPenCap / kThreads; ++t) {
    const int r = t * kThreads + tid;
    if (r >= npen) continue;
    const uint32_t l = en[t].id & ~kPenBias;
    const uint32_t bit = 1u << (l & 31);
    uint32_t c = en[t].count & kCountMask;
    if (en[t].id & kPenBias) c |= kBiasBit;
    if (S.live[l >> 5] & bit) c |= kAllowedBit;
    S.pid[r] = (uint16_t)l;
    S.pcnt[r] = c;
    S.pbias[r] = en[t].bias;
    atomicAnd(&S.live[l >> 5], ~bit);
    atomicOr(&S.mod[l >> 5], bit);
  }
  __syncthreads();
  // token-order rank of each mod word's first token: an exclusive scan of the popcounts
  {
    constexpr int kPer = (kMaxChunk / 32) / kThreads;
    const int nw = g.chunk / 32;
    int cnt[kPer], loc = 0;
#pragma unroll
    for (int t = 0; t < kPer; ++t) {
      const int w = tid * kPer + t;
      cnt[t] = w < nw ? __popc(S.mod[w]) : 0;
      loc += cnt[t];
    }
    int x = loc;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += o;
    }
    if (lane == 31) sh.red_i[warp] = x;
    __syncthreads();
    int excl = x - loc;
    for (int w = 0; w < warp; ++w) excl += sh.red_i[w];
#pragma unroll
    for (int t = 0; t < kPer; ++t) {
      const int w = tid * kPer + t;
      if (w < nw) S.prank[w] = (uint16_t)excl;
      excl += cnt[t];
    }
  }
  // allowed tokens of the slice: plain live ones plus allowed penalised ones
  {
    int na = 0;
    for (int w = tid; w < g.chunk / 32; w += kThreads) na += __popc(S.live[w]);
    for (int r = tid; r < npen; r += kThreads) na += (S.pcnt[r] & kAllowedBit) ? 1 : 0;
    na = __reduce_add_sync(0xffffffffu, na);
    if (lane == 0 && na) atomicAdd(&sh.nallowed, na);
  }
  __syncthreads();
}

// ---------------------------------------------------------------- pass A

// Pass A: slice max, lowest argmax and online sum of 2^((z' - max) cS), cS = log2(e)/T_eff;
// per-warp lower bounds of the top-k cut from the per-thread maxima.  Leaves the slice
// record in sh.x1_mine.
template <bool kBF16>
__device__ __noinline__ void pass_a(const LaunchParams& P) {
  const Geo g = geo<kBF16>(P);
  const Smem S = carve(g.chunk);
  const clsample_args_t& a = P.a;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RowParams q = sh.rp;
  const bool has_mod = a.hist_offs != nullptr || a.bias_offs != nullptr;
  const bool greedy = (q.T < kGreedyEps) || q.k == 0 || q.k == 1;
  const float Teff = (q.T >= kGreedyEps) ? q.T : 1.0f;
  const float cS = 1.4426950408889634f / Teff;
  const int c0 = g.c0;
  constexpr int kGroups = kStageBytes / (4 * (kBF16 ? 2 : 4)) / kThreads;  // vectors per thread per stage
  static_assert(kGroups <= 4, "red_j holds four group sets per warp");

  // the thread's online state; a thread visits its tokens in increasing order, so the
  // first token reaching the running max is the lowest
  float sm = -INFINITY, ss = 0.0f;
  int targ = INT_MAX;
  // the maxima of the thread's vectors in each stage slot: kGroups disjoint token groups
  // per thread for the top-k bounds
  float gm[kGroups];
#pragma unroll
  for (int t = 0; t < kGroups; ++t) gm[t] = -INFINITY;
  int pass = 0;
  stream<kBF16, true>(g, S, pass, true, [&](int f, uint32_t wd, const float4& v, int t) {
    if (has_mod && 4 * f < g.len) {
      // penalised / biased tokens: keep the raw logit (rank order) for the fold below
      const uint32_t mw = S.mod[f >> 3];
      const int sh4 = (f & 7) * 4;
      const uint32_t md = (mw >> sh4) & 0xFu;
      if (md) {
        int r = S.prank[f >> 3] + __popc(mw & ((1u << sh4) - 1u));
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if ((md >> j) & 1u) S.pz[r++] = comp(v, j);
      }
    }
    if (!wd) return;
    float4 z = v;
    if (!(wd == 0xFu && finite4(v)))
      z = make_float4((wd & 1u) ? sanitize(v.x) : -INFINITY, (wd & 2u) ? sanitize(v.y) : -INFINITY,
                      (wd & 4u) ? sanitize(v.z) : -INFINITY, (wd & 8u) ? sanitize(v.w) : -INFINITY);
    const float fm = fmaxf(fmaxf(z.x, z.y), fmaxf(z.z, z.w));
    if (!(fm > -INFINITY)) return;
    gm[t] = fmaxf(gm[t], fm);
    if (fm > sm) {
      ss *= ex2_approx((sm - fm) * cS);
      sm = fm;
      targ = c0 + 4 * f + (z.x == fm ? 0 : z.y == fm ? 1 : z.z == fm ? 2 : 3);
    }
    const float e0 = ex2_approx((z.x - sm) * cS), e1 = ex2_approx((z.y - sm) * cS);
    const float e2 = ex2_approx((z.z - sm) * cS), e3 = ex2_approx((z.w - sm) * cS);
    ss += (e0 + e1) + (e2 + e3);
  });
  // the penalised / biased tokens in token order: penalties, then bias, on the sanitised
  // raw logit (the mask applies to them too); the final z' goes into the hash and into
  // the thread's online state
  if (has_mod) {
    const int npen = sh.npen;
    for (int r = tid; r < npen; r += kThreads) {
      const uint32_t c = S.pcnt[r];
      float zz = (c & kAllowedBit) ? sanitize(S.pz[r]) : -INFINITY;
      const uint32_t cnt = c & kCountMask;
      if (cnt) zz = apply_penalties(zz, cnt, q.freq, q.pres, q.rep);
      if (c & kBiasBit) zz = __fadd_rn(zz, S.pbias[r]);
      zz = guard(zz);
      S.pz[r] = zz;
      if (!(zz > -INFINITY)) continue;
      const int id = c0 + (int)S.pid[r];
      gm[0] = fmaxf(gm[0], zz);  // a disjoint token set joins the thread's first group
      if (zz > sm) {
        ss = ss * ex2_approx((sm - zz) * cS) + 1.0f;
        sm = zz;
        targ = id;
      } else {
        ss += ex2_approx((zz - sm) * cS);
        if (zz == sm && id < targ) targ = id;
      }
    }
  }

  // group-set lower bounds of the top-k cut (see X1); lane i < kNJ of set t holds its
  // 2^i-th largest maximum
  const bool topk_row = !greedy && !q.invalid && q.k >= 2;
  float wlk = -INFINITY;
  float wlj[kGroups];
#pragma unroll
  for (int t = 0; t < kGroups; ++t) wlj[t] = -INFINITY;
  if (topk_row) {
#pragma unroll
    for (int t = 0; t < kGroups; ++t) {
      uint32_t key = fkey(gm[t]);
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
      const int k1 = q.k;
      const uint32_t v1 = __shfl_sync(0xffffffffu, key, k1 <= 32 ? 32 - k1 : 0);
      if (k1 <= 32) wlk = fmaxf(wlk, key_to_float(v1));
      const uint32_t vj = __shfl_sync(0xffffffffu, key, 32 - (1 << min(lane, kNJ - 1)));
      wlj[t] = lane < kNJ ? key_to_float(vj) : -INFINITY;
    }
  }
  // block reduction of (max, sum, argmax) and of the bounds
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
    sh.red_f[warp * 2] = m2;
    sh.red_f[warp * 2 + 1] = s2;
    sh.red_i[warp * 2] = a2;
    sh.red_wb[warp * 2] = wlk;
  }
  // per group set, in r2 (free until exchange 1; the top-p merged bins are not touched)
  float(*red_j)[kNJ] = reinterpret_cast<float(*)[kNJ]>(S.r2);
#pragma unroll
  for (int t = 0; t < kGroups; ++t)
    if (lane < kNJ) red_j[warp * kGroups + t][lane] = wlj[t];
  __syncthreads();
  if (warp == 0) {
    const bool in = lane < kWarps;
    float m = in ? sh.red_f[lane * 2] : -INFINITY, s = in ? sh.red_f[lane * 2 + 1] : 0.0f;
    int arg = in ? sh.red_i[lane * 2] : INT_MAX;
    float lk = in ? sh.red_wb[lane * 2] : -INFINITY;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, m, d);
      const float os = __shfl_xor_sync(0xffffffffu, s, d);
      const int oa = __shfl_xor_sync(0xffffffffu, arg, d);
      if (better(om, oa, m, arg)) arg = oa;
      merge_ms(m, s, om, os, cS);
      lk = fmaxf(lk, __shfl_xor_sync(0xffffffffu, lk, d));
    }
    // lane i < kNJ: the 2^i bounds over the group sets that reach 2^i maxima
    float lj = INFINITY;
    uint32_t nj = 0;
    if (lane < kNJ)
      for (int w = 0; w < kWarps * kGroups; ++w) {
        const float v = red_j[w][lane];
        if (v > -INFINITY) {
          lj = fminf(lj, v);
          ++nj;
        }
      }
    if (lane < kNJ) {
      sh.x1_mine.lj[lane] = topk_row ? lj : INFINITY;
      sh.x1_mine.nj[lane] = topk_row ? (unsigned char)nj : 0;
    }
    if (lane == 0) {
      sh.x1_mine.m = m;
      sh.x1_mine.s = s;
      sh.x1_mine.arg = arg;
      sh.x1_mine.lk = lk;
      sh.x1_mine.flags = sh.flags;
      sh.x1_mine.nallowed = sh.nallowed;
    }
  }
  // the transformed logits, on request (debugging aid): plain values first, then the
  // penalised / biased tokens' final z' from the hash
  if (a.dbg_transformed) {
    float* out = a.dbg_transformed + (long long)g.row * a.V + c0;
    const int32_t* bmrow = a.bitmask ? a.bitmask + (long long)g.row * a.bitmask_row_stride : nullptr;
    for (int i = tid; i < g.len; i += kThreads) {
      const int gi = c0 + i;
      const bool allowed = !bmrow || (((uint32_t)__ldg(bmrow + (gi >> 5)) >> (gi & 31)) & 1u);
      out[i] = allowed ? sanitize(gload1<kBF16>(g.g, i)) : -INFINITY;
    }
    __syncthreads();
    if (has_mod)
      for (int r = tid; r < sh.npen; r += kThreads) out[S.pid[r]] = S.pz[r];
  }
  __syncthreads();
}

// ---------------------------------------------------------------- exchange 1

// Every CTA pushes its slice record into every CTA (DSMEM) and one cluster barrier
// publishes them; every CTA then combines them in the same order into sh.rs.
__device__ __noinline__ void exchange1(const LaunchParams& P) {
  const cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = P.C;
  const int rank = (int)cluster.block_rank();
  const RowParams q = sh.rp;
  const float Teff = (q.T >= kGreedyEps) ? q.T : 1.0f;
  const float cS = 1.4426950408889634f / Teff;
  // DSMEM may only be touched once every CTA of the cluster runs (the kernel arrived on
  // the cluster barrier at entry)
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  push_all(cluster, sh.x1, &sh.x1_mine, rank, C);
  cluster.sync();
  if (warp == 0) {
    const bool in = lane < C;
    const float lm = in ? sh.x1[lane].m : -INFINITY;
    const int la = in ? sh.x1[lane].arg : INT_MAX;
    const float ls = in ? sh.x1[lane].s : 0.0f;
    int fl = in ? sh.x1[lane].flags : 0;
    float lk = in ? sh.x1[lane].lk : -INFINITY;
    int nal = in ? sh.x1[lane].nallowed : 0;
    float m = lm;
#pragma unroll
    for (int d = 4; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
    m = __shfl_sync(0xffffffffu, m, 0);  // lanes >= C may hold their own partial maxima
    int arg = (in && lm == m) ? la : INT_MAX;
    const float term = (in && lm > -INFINITY) ? ls * ex2_approx((lm - m) * cS) : 0.0f;
#pragma unroll
    for (int d = 4; d > 0; d >>= 1) {
      arg = min(arg, __shfl_xor_sync(0xffffffffu, arg, d));
      fl |= __shfl_xor_sync(0xffffffffu, fl, d);
      lk = fmaxf(lk, __shfl_xor_sync(0xffffffffu, lk, d));
      nal = max(nal, __shfl_xor_sync(0xffffffffu, nal, d));
    }
    // the 2^i bounds: lane i combines the CTAs; usable when its warps guarantee k tokens
    float bj = -INFINITY;
    if (lane < kNJ) {
      float lj = INFINITY;
      uint32_t n = 0;
      for (int c = 0; c < C; ++c) {
        lj = fminf(lj, sh.x1[c].lj[lane]);
        n += sh.x1[c].nj[lane];
      }
      if (n > 0 && (unsigned long long)n << lane >= (unsigned long long)max(sh.rp.k, 0)) bj = lj;
    }
    for (int d = 4; d > 0; d >>= 1) bj = fmaxf(bj, __shfl_xor_sync(0xffffffffu, bj, d));
    // the sum in a fixed order (ranks 0 .. C-1): every CTA gets the same bits
    float tot = 0.0f;
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) tot += __shfl_sync(0xffffffffu, term, r);
    if (lane == 0) {
      sh.rs.m = m;
      sh.rs.arg = arg;
      sh.rs.S = tot;
      sh.rs.flags = fl;
      sh.rs.bound = fmaxf(lk, bj);
      sh.rs.nallowed_max = nal;
      sh.rs.lnS = logf(tot);
    }
  }
  __syncthreads();
}
// ---------------------------------------------------------------- row end and plan

// Greedy, INVALID and OVERFLOW rows end after exchange 1; rank 0 writes the argmax (its
// y is 0, so its logprob is -ln S).  Returns true (in every thread) if the row ended.
__device__ __noinline__ bool finish_early(const LaunchParams& P) {
  const RowParams q = sh.rp;
  const float m = sh.rs.m;
  const int fl = sh.rs.flags;
  int status = kRowOk;
  if (q.invalid || (fl & kFlagInvalid) || !(m > -INFINITY)) status = kRowInvalid;
  else if (fl & (kFlagOverflow | kFlagRing)) status = kRowOverflow;
  const bool greedy = (q.T < kGreedyEps) || q.k == 0 || q.k == 1;
  if (status == kRowOk && !greedy) return false;
  if (threadIdx.x == 0 && cg::this_cluster().block_rank() == 0) {
    const clsample_args_t& a = P.a;
    const int row = cluster_row(P);
    const bool ok = status == kRowOk;
    a.tokens[row] = ok ? sh.rs.arg : -1;
    if (a.logprobs) a.logprobs[row] = ok ? -sh.rs.lnS : -INFINITY;
    if (a.row_status) a.row_status[row] = status;
    if (a.dbg_kept_count) a.dbg_kept_count[row] = ok ? 1 : 0;
    if (a.dbg_cut) a.dbg_cut[row] = ok ? 0.0f : -INFINITY;
  }
  return true;
}

// Truncation plan.  y = (z' - m) * (1/T); the kept set K = {y >= cut} is an upper set.
__device__ __noinline__ void plan_row(const LaunchParams& P) {
  if (threadIdx.x == 0) {
    const RowParams q = sh.rp;
    RowState& rs = sh.rs;
    rs.invT = __frcp_rn(q.T);
    rs.L = q.mp > 0.0f ? (float)log((double)q.mp) : -INFINITY;  // min-p: y >= ln(min_p)
    const bool kfin = q.k >= 2;
    int plan = kPlanSlow, needW = 0, all = 0;
    float theta = -INFINITY;
    if (kfin && rs.bound > -INFINITY) {
      plan = kPlanFast;  // every token of S_k has y >= y(bound)
      theta = y_of(rs.bound, rs.m, rs.invT);
      if (q.p >= 1.0f) theta = fmaxf(theta, rs.L);
    } else if (rs.nallowed_max <= kCandCap) {
      plan = kPlanFast;  // few candidates: the leader sees all of them
      all = 1;
    } else if (q.mp > 0.0f && (q.p >= 1.0f || !kfin)) {
      plan = kPlanFast;  // K lies in {y >= ln min_p}
      theta = rs.L;
      needW = q.p < 1.0f;  // top-p renormalises over the whole row
    } else if (!kfin && q.p >= 1.0f) {
      plan = kPlanUntrunc;  // K = every allowed token
    } else if (!kfin) {
      plan = kPlanTopP;  // top-p alone
    }
    rs.plan = plan;
    rs.needW = needW;
    rs.all = all;
    rs.theta = theta;
    const int arg = rs.arg;  // its y is 0
    rs.s0 = race_score(0.0f, pick_word(race_words_call((uint32_t)(arg >> 2), q.seed, q.pos), arg & 3));
  }
  __syncthreads();
}

// ---------------------------------------------------------------- candidates and the leader

// Appends (y, id) to the slice's candidate list; the whole warp calls it.
__device__ __forceinline__ void append(Cand* cand, int cap, bool keep, float y, int id) {
  const int lane = threadIdx.x & 31;
  const uint32_t bal = __ballot_sync(0xffffffffu, keep);
  if (!bal) return;
  const int leader = __ffs(bal) - 1;
  int basepos = 0;
  if (lane == leader) basepos = atomicAdd(&sh.count, __popc(bal));
  basepos = __shfl_sync(0xffffffffu, basepos, leader);
  if (keep) {
    const int p = basepos + __popc(bal & ((1u << lane) - 1u));
    if (p < cap) cand[p] = Cand{y, id};
  }
}

// Publishes the slice's pass-B record (candidate count, top-p mass partial, race) to
// every CTA: exchange 2 (or 3).
__device__ void finish_mine(int cap, unsigned long long w, const Race& race) {
  const cg::cluster_group cluster = cg::this_cluster();
  __threadfence();  // the compacted candidates (global) before the cluster barrier
  __syncthreads();
  if (threadIdx.x == 0) {
    sh.x2_mine.count = sh.count;
    sh.x2_mine.flags = (sh.count > cap ? kFlagOverflow : 0) | (sh.flags & kFlagRing);
    sh.x2_mine.w = w;
    race.to(sh.x2_mine);
  }
  __syncthreads();
  push_all(cluster, sh.x2, &sh.x2_mine, (int)cluster.block_rank(), (int)cluster.num_blocks());
  cluster.sync();
}

__device__ __forceinline__ int x2_flags(int C) {
  int f = 0;
  for (int c = 0; c < C; ++c) f |= sh.x2[c].flags;
  return f;
}

// After the last exchange every CTA's candidates sit in its global segment (the counts
// are known to every CTA).  Only the leader (rank 0) continues: it packs them, in rank
// order, into its shared gather area (the ring is free: every CTA has finished reading
// its slice), or, when there are more than kGatherCap, into its own global segments.
// Returns the packed array (nullptr in the other CTAs) and their number in *n.
__device__ const Cand* collect_at_leader(const LaunchParams& P, const Smem& S, int* n) {
  const cg::cluster_group cluster = cg::this_cluster();
  if (cluster.block_rank() != 0) return nullptr;
  const int tid = threadIdx.x;
  const int C = P.C;
  const int row = cluster_row(P);
  Cand* seg = P.cand + (size_t)row * C * kCandCap;
  int ntot = 0;
  for (int c = 0; c < C; ++c) ntot += sh.x2[c].count;
  *n = ntot;
  if (ntot <= kGatherCap) {
    int off = 0;
    for (int c = 0; c < C; ++c) {
      const int cnt = sh.x2[c].count;
      for (int i = tid; i < cnt; i += kThreads) S.gather[off + i] = seg[(size_t)c * kCandCap + i];
      off += cnt;
    }
    __syncthreads();
    return S.gather;
  }
  // in place, segment by segment: each moves towards lower addresses, read whole first
  int off = sh.x2[0].count;
  for (int c = 1; c < C; ++c) {
    const int cnt = sh.x2[c].count;
    Cand tmp[kCandCap / kThreads];
#pragma unroll
    for (int t = 0; t < kCandCap / kThreads; ++t) {
      const int i = t * kThreads + tid;
      if (i < cnt) tmp[t] = seg[(size_t)c * kCandCap + i];
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < kCandCap / kThreads; ++t) {
      const int i = t * kThreads + tid;
      if (i < cnt) seg[off + i] = tmp[t];
    }
    __syncthreads();
    off += cnt;
  }
  return seg;
}

// Radix select over the gathered set (entries with y >= ylo): the largest value v such
// that the count (or fixed-point weight) of entries >= v reaches `target`.
__device__ __noinline__ float local_select(int chunk, const Cand* G, int n, bool weighted, float ylo,
                                           unsigned long long target, bool* found) {
  const Smem S = carve(chunk);
  const int tid = threadIdx.x, warp = tid >> 5;
  uint32_t prefix = 0u, pmask = 0u;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    if (tid < 256) {
      S.hist_c[tid] = 0u;
      S.hist_w[tid] = 0ull;
    }
    __syncthreads();
    for (int base = 0; base < n; base += kThreads) {
      const int i = base + tid;
      const bool ok = i < n;
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
      if (weighted) pick_digit(S.hist_w, target, &sh.digit, &sh.above, &sh.none);
      else pick_digit(S.hist_c, target, &sh.digit, &sh.above, &sh.none);
    }
    __syncthreads();
    if (sh.none) {
      *found = false;
      __syncthreads();
      return -INFINITY;
    }
    prefix |= (uint32_t)sh.digit << shift;
    pmask |= 0xFFu << shift;
    target -= sh.above;
    __syncthreads();
  }
  *found = true;
  return key_to_float(prefix);
}

// Exact select over the gathered set, entries with y >= ylo, all within [lo, hi]: one
// 1024-bucket histogram (bucket order follows y), then the crossing bucket's entries are
// resolved by counting.  Falls back to local_select when that bucket holds more than
// 1024 entries (heavy ties).
__device__ __noinline__ float leader_select(int chunk, const Cand* G, int n, bool weighted, float lo, float hi,
                                            float ylo, unsigned long long target, bool* found) {
  const Smem S = carve(chunk);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* bk = reinterpret_cast<uint32_t*>(S.r2);  // split counters, two u32 per bucket
  constexpr int kPer = 1024 / kThreads;  // consecutive buckets per thread
  const float scale = hi > lo ? 1024.0f / (hi - lo) : 0.0f;
  auto bucket = [&](float y) -> int {
    const int b = __float2int_rz(__fmul_rn(hi - y, scale));
    return b < 0 ? 0 : (b > 1023 ? 1023 : b);
  };
#pragma unroll
  for (int t = 0; t < 2 * kPer; ++t) bk[2 * kPer * tid + t] = 0u;
  if (tid == 0) {
    sh.nl = 0;
    sh.bstar = -1;
  }
  __syncthreads();
  for (int i = tid; i < n; i += kThreads) {
    const float y = G[i].y;
    if (!(y >= ylo)) continue;
    split_add(bk + 2 * bucket(y), weighted ? weight_fx(y) : 1ull);
  }
  __syncthreads();
  {
    unsigned long long vb[kPer], loc = 0;
#pragma unroll
    for (int t = 0; t < kPer; ++t) {
      vb[t] = split_get(bk + 2 * (kPer * tid + t));
      loc += vb[t];
    }
    unsigned long long x = loc;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const unsigned long long o = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += o;
    }
    if (lane == 31) sh.red_u[warp] = x;
    __syncthreads();
    unsigned long long before = 0;
    for (int w = 0; w < warp; ++w) before += sh.red_u[w];
    const unsigned long long excl = before + x - loc, incl = before + x;
    if (excl < target && target <= incl) {
      unsigned long long cum = excl;
      for (int t = 0; t < kPer; ++t) {
        if (cum + vb[t] >= target) {
          sh.bstar = kPer * tid + t;
          sh.above = cum;
          break;
        }
        cum += vb[t];
      }
    }
  }
  __syncthreads();
  const int bstar = sh.bstar;
  if (bstar < 0) {
    *found = false;
    return -INFINITY;
  }
  const unsigned long long t2 = target - sh.above;
  // the crossing bucket's entries, gathered into the (now free) bucket area
  Cand* Lb = reinterpret_cast<Cand*>(S.r2);
  __syncthreads();
  for (int i = tid; i < n; i += kThreads) {
    const Cand cd = G[i];
    if (!(cd.y >= ylo) || bucket(cd.y) != bstar) continue;
    const int p = atomicAdd(&sh.nl, 1);
    if (p < 1024) Lb[p] = cd;
  }
  __syncthreads();
  const int nl = sh.nl;
  if (nl > 1024) {
    __syncthreads();
    return local_select(chunk, G, n, weighted, ylo, target, found);
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
    if (gt < t2 && t2 <= ge) sh.res = yi;
  }
  __syncthreads();
  *found = true;
  return sh.res;
}

// The race over the gathered entries with y >= cut (block-reduced into thread 0).
__device__ __noinline__ Race leader_race(const Cand* G, int n, float cut, unsigned long long seed,
                                         unsigned long long pos) {
  Race r;
  r.init(sh.rs.s0);
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const Cand cd = G[i];
    if (!(cd.y >= cut)) continue;
    r.add(cd.y, cd.id, pick_word(race_words_call((uint32_t)(cd.id >> 2), seed, pos), cd.id & 3));
  }
  block_reduce_race(r, sh.red_x);
  return r;
}

// ---------------------------------------------------------------- routes

// A top-k row whose candidates exceed the leader's shared area: a cluster-wide histogram
// of the candidates' y over 256 equal buckets of [lo, 0] (pushed with DSMEM atomics into
// every CTA's merged copy, zeroed by the prologue) fixes the bucket where the count from
// the top first reaches k; every CTA then keeps, in place, only its candidates in that
// bucket or above (an upper set that still holds the top-k set) and the counts are
// exchanged again.
__device__ __noinline__ void refine_topk(const LaunchParams& P, const Smem& S, Cand* mycand, float lo, int k) {
  const cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = P.C, rank = (int)cluster.block_rank();
  const int cnt = min(sh.x2[rank].count, kCandCap);
  const float scale = 256.0f / -lo;
  auto bucket = [&](float y) -> int {
    const int b = __float2int_rz(__fmul_rn(-y, scale));
    return b < 0 ? 0 : (b > 255 ? 255 : b);
  };
  S.hist_c[tid] = 0u;
  __syncthreads();
  Cand mine[kCandCap / kThreads];
#pragma unroll
  for (int t = 0; t < kCandCap / kThreads; ++t) {
    const int i = t * kThreads + tid;
    if (i < cnt) {
      mine[t] = mycand[i];
      atomicAdd(&S.hist_c[bucket(mine[t].y)], 1u);
    }
  }
  __syncthreads();
  {
    const uint32_t v = S.hist_c[tid];
    if (v)
      for (int r = 0; r < C; ++r) atomicAdd(cluster.map_shared_rank(S.mrg_c + tid, (unsigned)r), v);
  }
  cluster.sync();
  // the bucket where the running count from the top (bucket 0) first reaches k
  {
    const uint32_t v = S.mrg_c[tid];
    uint32_t x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += o;
    }
    if (lane == 31) sh.red_i[warp] = (int)x;
    if (tid == 0) sh.bstar = 255;
    __syncthreads();
    uint32_t before = 0;
    for (int w = 0; w < warp; ++w) before += (uint32_t)sh.red_i[w];
    if (before + x >= (uint32_t)k && before + x - v < (uint32_t)k) sh.bstar = tid;
  }
  __syncthreads();
  const int bstar = sh.bstar;
  if (tid == 0) sh.count = 0;
  __syncthreads();
#pragma unroll
  for (int t = 0; t < kCandCap / kThreads; ++t) {
    const int i = t * kThreads + tid;
    if (i < cnt && bucket(mine[t].y) <= bstar) mycand[atomicAdd(&sh.count, 1)] = mine[t];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) sh.x2_mine.count = sh.count;
  __syncthreads();
  push_all(cluster, sh.x2, &sh.x2_mine, rank, C);
  cluster.sync();
}

// Rows with a provable bound (top-k, min-p) and untruncated rows.  Pass B compacts the
// tokens at z >= zth (the exact z-space image of the y bound) and/or races every token;
// the leader finishes top-k -> top-p -> min-p and the race over the gathered candidates.
// Returns false when a compaction overflowed (the slow path takes over).
template <bool kBF16>
__device__ __noinline__ bool route_fast(const LaunchParams& P, int& pass) {
  const Geo g = geo<kBF16>(P);
  const Smem S = carve(g.chunk);
  const clsample_args_t& a = P.a;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RowParams q = sh.rp;
  const float m = sh.rs.m, invT = sh.rs.invT, lnS = sh.rs.lnS, L = sh.rs.L, theta = sh.rs.theta;
  const int plan = sh.rs.plan;
  const bool needW = sh.rs.needW != 0;
  const bool has_mod = a.hist_offs != nullptr || a.bias_offs != nullptr;
  const bool kfin = q.k >= 2;
  const unsigned long long seed = q.seed, pos = q.pos;
  const int c0 = g.c0, cap = kCandCap, C = g.C;
  Cand* mycand = P.cand + ((size_t)g.row * C + g.rank) * kCandCap;  // this slice's segment
  if (warp == 0) {
    const float zt = z_threshold_warp(theta, m, invT);
    if (lane == 0) sh.zth = zt;
  }
  __syncthreads();
  const float zth = sh.zth;
  unsigned long long w = 0;
  Race race;
  race.init(sh.rs.s0);
  stream<kBF16>(g, S, pass, false, [&](int f, uint32_t wd, const float4& v) {
    float z[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    if (wd) {
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
#pragma unroll 1
        for (int j = 0; j < 4; ++j)
          if (z[j] > -INFINITY) w += weight_fx(y_of(z[j], m, invT));
      }
      if (plan == kPlanUntrunc) {
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
#pragma unroll 1
          for (int j = 0; j < 4; ++j)
            if (z[j] > -INFINITY) race.add(y[j], c0 + 4 * f + j, pick_word(x, j));
        } else if (live_any) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (z[j] > -INFINITY) race.count_only(y[j]);
        }
      }
    }
    if (plan == kPlanFast) {
      const bool any = __any_sync(0xffffffffu, z[0] >= zth || z[1] >= zth || z[2] >= zth || z[3] >= zth);
      if (any) {
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          const bool keep = z[j] > -INFINITY && z[j] >= zth;
          append(mycand, cap, keep, keep ? y_of(z[j], m, invT) : 0.0f, c0 + 4 * f + j);
        }
      }
    }
  });
  if (has_mod) {
    const int npen = sh.npen;
    for (int base = 0; base < npen; base += kThreads) {
      const int i = base + tid;
      const float z = i < npen ? S.pz[i] : -INFINITY;
      const int gi = c0 + (i < npen ? (int)S.pid[i] : 0);
      const float y = z > -INFINITY ? y_of(z, m, invT) : -INFINITY;
      if (z > -INFINITY) {
        if (needW) w += weight_fx(y);
        if (plan == kPlanUntrunc) race.add(y, gi, pick_word(race_words_call((uint32_t)(gi >> 2), seed, pos), gi & 3));
      }
      if (plan == kPlanFast) append(mycand, cap, z > -INFINITY && z >= zth, y, gi);
    }
  }
  if (needW) w = block_sum_u64(w, sh.red_u);
  if (plan == kPlanUntrunc) block_reduce_race(race, sh.red_x);
  finish_mine(cap, w, race);  // exchange 2
  const int fl = x2_flags(C);

  if (plan == kPlanUntrunc) {
    // the winner is the same in every CTA; its owner writes the outputs
    if (tid == 0) {
      Race r;
      r.init();
      for (int c = 0; c < C; ++c) r.merge(sh.x2[c]);
      const int owner = r.tok == INT_MAX ? 0 : r.tok / g.chunk;
      if (g.rank == owner) write_sampled(a, g.row, r, lnS, !(fl & kFlagRing));
    }
    return true;
  }
  if (fl & kFlagOverflow) return false;
  {
    int n = 0;
    for (int c = 0; c < C; ++c) n += sh.x2[c].count;
    if (kfin && n > kGatherCap && theta > -INFINITY && theta < 0.0f) refine_topk(P, S, mycand, theta, q.k);
  }
  int ntot = 0;
  const Cand* G = collect_at_leader(P, S, &ntot);
  if (!G) return true;
  const bool gathered = !(fl & kFlagRing);
  // the bucket range: [theta, 0], or the gathered candidates' finite range
  float lo = theta;
  if (!(lo > -INFINITY)) {
    float ymin = INFINITY;
    for (int i = tid; i < ntot; i += kThreads) {
      const float y = G[i].y;
      if (y > -INFINITY) ymin = fminf(ymin, y);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) ymin = fminf(ymin, __shfl_xor_sync(0xffffffffu, ymin, d));
    if (lane == 0) sh.red_f[warp] = ymin;
    __syncthreads();
    lo = INFINITY;
    for (int w = 0; w < kWarps; ++w) lo = fminf(lo, sh.red_f[w]);
    if (!(lo < 0.0f)) lo = -1.0f;
    __syncthreads();
  }
  float tk = -INFINITY;
  if (kfin && ntot >= q.k) {
    bool found;
    const float v = leader_select(g.chunk, G, ntot, false, lo, 0.0f, -INFINITY, (unsigned long long)q.k, &found);
    if (found) tk = v;
  }
  float tp = -INFINITY;
  if (q.p < 1.0f) {
    unsigned long long mset = 0;
    for (int i = tid; i < ntot; i += kThreads)
      if (G[i].y >= tk) mset += weight_fx(G[i].y);
    mset = block_sum_u64(mset, sh.red_u);
    unsigned long long Wk = mset;  // top-k set (or every candidate) gathered: its mass
    if (!kfin && !sh.rs.all) {
      Wk = 0;
      for (int c = 0; c < C; ++c) Wk += sh.x2[c].w;
    }
    const unsigned long long cth = ceil_scaled(Wk, q.p);
    if (mset >= cth) {
      bool found;
      const float v = leader_select(g.chunk, G, ntot, true, lo, 0.0f, tk, cth, &found);
      if (found) tp = v;
    }
  }
  const float cut = fmaxf(tk, fmaxf(tp, L));
  const Race r = leader_race(G, ntot, cut, seed, pos);
  if (tid == 0) write_sampled(a, g.row, r, lnS, gathered);
  return true;
}

// Top-p alone: the exact top-p mass of the row and its histogram over quarter-unit y bins
// (warp-private, in the candidate area) fix the crossing bin (exchange 2); pass C races
// the tokens above it in place and sends the crossing bin's tokens to the leader, which
// resolves the cut inside the bin.  Returns false (slow path) when the crossing bin is
// the open-ended last one or the band overflowed.
template <bool kBF16>
__device__ __noinline__ bool route_topp(const LaunchParams& P, int& pass) {
  const Geo g = geo<kBF16>(P);
  const Smem S = carve(g.chunk);
  const clsample_args_t& a = P.a;
  const int tid = threadIdx.x, warp = tid >> 5;
  const RowParams q = sh.rp;
  const float m = sh.rs.m, invT = sh.rs.invT, lnS = sh.rs.lnS;
  const bool has_mod = a.hist_offs != nullptr || a.bias_offs != nullptr;
  const unsigned long long seed = q.seed, pos = q.pos;
  const int c0 = g.c0, cap = kCandCap, C = g.C;
  Cand* mycand = P.cand + ((size_t)g.row * C + g.rank) * kCandCap;  // this slice's segment
  const cg::cluster_group cluster = cg::this_cluster();

  // warp-private split counters (two u32 per bin): a warp adds at most 4160 weights
  uint32_t* whist = reinterpret_cast<uint32_t*>(S.r2);
  for (int i = tid; i < 2 * kWarps * kPBins; i += kThreads) whist[i] = 0u;
  __syncthreads();
  unsigned long long w = 0, wlast = 0;
  uint32_t* mine = whist + 2 * warp * kPBins;
  stream<kBF16>(g, S, pass, false, [&](int f, uint32_t wd, const float4& v) {
    if (!wd) return;
    const bool fastv = wd == 0xFu && finite4(v);
#pragma unroll 1
    for (int j = 0; j < 4; ++j) {
      const float z = fastv ? comp(v, j) : (((wd >> j) & 1u) ? sanitize(comp(v, j)) : -INFINITY);
      if (!(z > -INFINITY)) continue;
      const float y = y_of(z, m, invT);
      const unsigned long long qw = weight_fx(y);
      if (!qw) continue;
      w += qw;
      const int b = pbin(y);
      if (b == kPBins - 1) wlast += qw;  // the open-ended last bin: one add per thread below
      else split_add(mine + 2 * b, qw);
    }
  });
  if (has_mod) {
    for (int i = tid; i < sh.npen; i += kThreads) {
      const float z = S.pz[i];
      if (!(z > -INFINITY)) continue;
      const float y = y_of(z, m, invT);
      const unsigned long long qw = weight_fx(y);
      if (!qw) continue;
      w += qw;
      split_add(mine + 2 * pbin(y), qw);
    }
  }
  {
    const unsigned long long wl = warp_sum_u64(wlast);  // < 2^53: split_add holds it
    if ((tid & 31) == 0 && wl) split_add(mine + 2 * (kPBins - 1), wl);
  }
  w = block_sum_u64(w, sh.red_u);
  // merge the warp histograms and push them into every CTA's merged copy
  unsigned long long* pmrg = reinterpret_cast<unsigned long long*>(S.mrg_c);  // zeroed by the prologue
  if (tid < kPBins) {
    unsigned long long t = 0;
    for (int wp = 0; wp < kWarps; ++wp) t += split_get(whist + 2 * (wp * kPBins + tid));
    if (t)
      for (int r = 0; r < C; ++r) atomicAdd(cluster.map_shared_rank(pmrg + tid, (unsigned)r), t);
  }
  Race none_race;
  none_race.init();
  finish_mine(cap, w, none_race);  // exchange 2
  unsigned long long W = 0;
  for (int c = 0; c < C; ++c) W += sh.x2[c].w;
  const unsigned long long cth = ceil_scaled(W, q.p);
  // crossing bin: the running mass from the top first reaches cth in bin bstar
  int bstar = kPBins - 1;
  unsigned long long above = 0;
  {
    unsigned long long cum = 0;
    for (int b = 0; b < kPBins; ++b) {
      const unsigned long long nb = cum + pmrg[b];
      if (nb >= cth) {
        bstar = b;
        above = cum;
        break;
      }
      cum = nb;
    }
  }
  if (bstar >= kPBins - 1) return false;
  // pass C: tokens above the crossing bin are certainly kept: race them here; tokens of
  // the crossing bin go to the leader
  const float yhi = -(float)bstar * 0.25f, ylo = -(float)(bstar + 1) * 0.25f;
  __syncthreads();
  if (tid == 0) sh.count = 0;
  __syncthreads();
  Race race;
  race.init(sh.rs.s0);
  stream<kBF16>(g, S, pass, false, [&](int f, uint32_t wd, const float4& v) {
    float y[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    if (wd) {
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
          const uint4 x = race_words_call((uint32_t)((c0 >> 2) + f), seed, pos);
#pragma unroll 1
          for (int j = 0; j < 4; ++j)
            if ((sure >> j) & 1u) race.add(y[j], c0 + 4 * f + j, pick_word(x, j));
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if ((sure >> j) & 1u) race.count_only(y[j]);
        }
      }
    }
    const bool any = __any_sync(0xffffffffu, (y[0] > ylo && y[0] <= yhi) || (y[1] > ylo && y[1] <= yhi) ||
                                                 (y[2] > ylo && y[2] <= yhi) || (y[3] > ylo && y[3] <= yhi));
    if (any) {
#pragma unroll 1
      for (int j = 0; j < 4; ++j) append(mycand, cap, y[j] > ylo && y[j] <= yhi, y[j], c0 + 4 * f + j);
    }
  });
  if (has_mod) {
    const int npen = sh.npen;
    for (int base = 0; base < npen; base += kThreads) {
      const int i = base + tid;
      float y = -INFINITY;
      int gi = 0;
      if (i < npen && S.pz[i] > -INFINITY) {
        y = y_of(S.pz[i], m, invT);
        gi = c0 + (int)S.pid[i];
        if (y > yhi) race.add(y, gi, pick_word(race_words_call((uint32_t)(gi >> 2), seed, pos), gi & 3));
      }
      append(mycand, cap, y > ylo && y <= yhi, y, gi);
    }
  }
  block_reduce_race(race, sh.red_x);
  finish_mine(cap, 0ull, race);  // exchange 3
  const int fl = x2_flags(C);
  if (fl & kFlagOverflow) return false;
  int ntot = 0;
  const Cand* G = collect_at_leader(P, S, &ntot);
  if (!G) return true;
  const bool gathered = !(fl & kFlagRing);
  // the cut lies in the crossing bin: a weighted select over its tokens
  bool found;
  const float vstar = leader_select(g.chunk, G, ntot, true, ylo, yhi, -INFINITY, cth - above, &found);
  Race r = leader_race(G, ntot, vstar, seed, pos);
  if (tid == 0) {
    for (int c = 0; c < C; ++c) r.merge(sh.x2[c]);
    write_sampled(a, g.row, r, lnS, gathered && found);
  }
  return true;
}

// Cluster-wide radix select over the slices (one pass over the slice per 8-bit digit):
// the largest value v such that the count (or fixed-point weight) of kept-side tokens
// with y >= v reaches `target`, among tokens with y >= ylo.  Histograms are pushed into
// every CTA's merged copy with DSMEM atomics, one cluster barrier per digit; the merged
// copies are double-buffered and cleared after use.
template <bool kBF16>
__device__ __noinline__ float cluster_select(const LaunchParams& P, int& pass, int& gpass, bool weighted, float ylo,
                                             unsigned long long target, bool* found) {
  const Geo g = geo<kBF16>(P);
  const Smem S = carve(g.chunk);
  const clsample_args_t& a = P.a;
  const cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x, warp = tid >> 5;
  const float m = sh.rs.m, invT = sh.rs.invT;
  const bool has_mod = a.hist_offs != nullptr || a.bias_offs != nullptr;
  uint32_t prefix = 0u, pmask = 0u;
  bool ok_all = true;
  for (int dpass = 0; dpass < 4; ++dpass, ++gpass) {
    const int shift = 24 - 8 * dpass;
    const int buf = gpass & 1;
    if (tid < 256) {
      S.hist_c[tid] = 0u;
      S.hist_w[tid] = 0ull;
    }
    __syncthreads();
    stream<kBF16>(g, S, pass, false, [&](int f, uint32_t wd, const float4& v) {
#pragma unroll 1
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
    });
    if (has_mod) {
      const int npen = sh.npen;
      for (int base = 0; base < npen; base += kThreads) {
        const int i = base + tid;
        bool pred = false;
        float y = -INFINITY;
        if (i < npen) {
          const float z = S.pz[i];
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
    for (int i = tid; i < 256 * g.C; i += kThreads) {
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
      if (weighted) pick_digit(S.mrg_w + buf * 256, target, &sh.digit, &sh.above, &sh.none);
      else pick_digit(S.mrg_c + buf * 256, target, &sh.digit, &sh.above, &sh.none);
    }
    __syncthreads();
    const bool none = sh.none != 0;
    const int dg = sh.digit;
    const unsigned long long ab = sh.above;
    // clear this buffer for its next use (two digits later, after another barrier)
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
}

// Rows without a usable bound (very large k, compaction overflow, top-p with an
// open-ended crossing bin): exact cluster-wide selects, then the race in place.
template <bool kBF16>
__device__ __noinline__ void route_slow(const LaunchParams& P, int& pass) {
  const Geo g = geo<kBF16>(P);
  const Smem S = carve(g.chunk);
  const clsample_args_t& a = P.a;
  const cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x;
  const RowParams q = sh.rp;
  const float m = sh.rs.m, invT = sh.rs.invT, lnS = sh.rs.lnS, L = sh.rs.L;
  const bool has_mod = a.hist_offs != nullptr || a.bias_offs != nullptr;
  const unsigned long long seed = q.seed, pos = q.pos;
  const int c0 = g.c0, C = g.C;
  const bool kfin = q.k >= 2;

  for (int i = tid; i < 2 * 256; i += kThreads) {
    S.mrg_c[i] = 0u;
    S.mrg_w[i] = 0ull;
  }
  cluster.sync();  // every merged copy is clear before the first push
  int gpass = 0;
  float tk = -INFINITY;
  if (kfin) {
    bool found;
    const float v = cluster_select<kBF16>(P, pass, gpass, false, -INFINITY, (unsigned long long)q.k, &found);
    if (found) tk = v;  // fewer than k candidates: top-k keeps them all
  }
  float tp = -INFINITY;
  if (q.p < 1.0f) {
    unsigned long long w = 0;
    stream<kBF16>(g, S, pass, false, [&](int f, uint32_t wd, const float4& v) {
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        if (!((wd >> j) & 1u)) continue;
        const float z = sanitize(comp(v, j));
        if (!(z > -INFINITY)) continue;
        const float y = y_of(z, m, invT);
        if (y >= tk) w += weight_fx(y);
      }
    });
    if (has_mod)
      for (int i = tid; i < sh.npen; i += kThreads) {
        const float z = S.pz[i];
        if (!(z > -INFINITY)) continue;
        const float y = y_of(z, m, invT);
        if (y >= tk) w += weight_fx(y);
      }
    w = block_sum_u64(w, sh.red_u);
    if (tid == 0) sh.x2_mine.w = w;
    __syncthreads();
    push_all(cluster, sh.x2, &sh.x2_mine, g.rank, C);
    cluster.sync();
    unsigned long long W = 0;
    for (int c = 0; c < C; ++c) W += sh.x2[c].w;
    bool found;
    const float v = cluster_select<kBF16>(P, pass, gpass, true, tk, ceil_scaled(W, q.p), &found);
    if (found) tp = v;
  }
  const float cut = fmaxf(tk, fmaxf(tp, L));
  Race race;
  race.init(sh.rs.s0);
  stream<kBF16>(g, S, pass, false, [&](int f, uint32_t wd, const float4& v) {
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
    if (!keep) return;
    const uint4 x = race_words((uint32_t)((c0 >> 2) + f), seed, pos);
#pragma unroll 1
    for (int j = 0; j < 4; ++j)
      if ((keep >> j) & 1u) race.add(y[j], c0 + 4 * f + j, pick_word(x, j));
  });
  if (has_mod)
    for (int i = tid; i < sh.npen; i += kThreads) {
      const float z = S.pz[i];
      if (!(z > -INFINITY)) continue;
      const float y = y_of(z, m, invT);
      if (!(y >= cut)) continue;
      const int gi = c0 + (int)S.pid[i];
      race.add(y, gi, pick_word(race_words_call((uint32_t)(gi >> 2), seed, pos), gi & 3));
    }
  block_reduce_race(race, sh.red_x);
  __syncthreads();
  if (tid == 0) {
    race.to(sh.x2_mine);
    sh.x2_mine.flags = sh.flags & kFlagRing;
  }
  __syncthreads();
  push_all(cluster, sh.x2, &sh.x2_mine, g.rank, C);
  cluster.sync();
  // the winner is the same in every CTA; its owner writes the outputs
  if (tid == 0) {
    Race r;
    r.init();
    for (int c = 0; c < C; ++c) r.merge(sh.x2[c]);
    const int owner = r.tok == INT_MAX ? 0 : r.tok / g.chunk;
    if (g.rank == owner) write_sampled(a, g.row, r, lnS, !(x2_flags(C) & kFlagRing));
  }
}

// ---------------------------------------------------------------- the kernel

template <bool kBF16>
__global__ void __launch_bounds__(kThreads, kMinBlocks) sampler_kernel(const __grid_constant__ LaunchParams P) {
  // DSMEM may only be touched once every CTA of the cluster runs: arrive now, wait just
  // before the first push (exchange1)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  prologue<kBF16>(P);
  pass_a<kBF16>(P);
  exchange1(P);
  if (finish_early(P)) return;
  plan_row(P);
  int pass = 1;
  const int plan = sh.rs.plan;
  if (plan == kPlanFast || plan == kPlanUntrunc) {
    if (route_fast<kBF16>(P, pass)) return;
  } else if (plan == kPlanTopP) {
    if (route_topp<kBF16>(P, pass)) return;
  }
  route_slow<kBF16>(P, pass);
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
  const uint4 x = race_words_call((uint32_t)((unsigned long long)t >> 2), seeds[i], (unsigned long long)pos[i]);
  u[i] = word_to_uniform(pick_word(x, (int)(t & 3)));
}

// ---------------------------------------------------------------- host side

// C = ceil(V / 2048) CTAs per row, at most the portable cluster size; slices are whole
// bitmask words.  Shared memory does not depend on the logits type.
Geometry geometry_for(int vocab) {
  Geometry g{0, 0, 0, 0};
  if (vocab <= 0) return g;
  int C = (vocab + 2047) / 2048;
  if (C > kMaxCluster) C = kMaxCluster;
  const int chunk = ((vocab + C - 1) / C + 31) / 32 * 32;
  if (chunk > kMaxChunk) return g;  // C = 0: vocabulary too large
  g.C = C;
  g.chunk = chunk;
  g.smem = (int)layout_for(chunk).total;
  g.cap = kCandCap;
  return g;
}

}  // namespace

namespace {

// Device scratch of one call: sized for max_batch rows of up to kMaxCluster slices.
struct Scratch {
  int max_batch;
  PenEntry* pen;  // penalised-token lists, [max_batch * C][kPenCap]
  int2* pen_n;    // their lengths and flags, [max_batch * C]
  Cand* cand;     // compacted candidates, [max_batch * C][kCandCap]
  int* rows;      // row classes and launch order, [2 * max_batch], then the ticket
};

// Checks the device (compute capability 10.3, enough shared memory) and raises the
// kernels' dynamic shared-memory limit to what the longest slice needs.
int setup_device(int dev) {
  int major = 0, minor = 0, optin = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return CLSAMPLE_ERR_CUDA;
  if (major != 10 || minor != 3) return CLSAMPLE_ERR_DEVICE;
  const int smem = (int)layout_for(kMaxChunk).total;
  if (smem > optin) return CLSAMPLE_ERR_DEVICE;
  const void* k32 = reinterpret_cast<const void*>(&sampler_kernel<false>);
  const void* k16 = reinterpret_cast<const void*>(&sampler_kernel<true>);
  if (cudaFuncSetAttribute(k32, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(k16, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return CLSAMPLE_ERR_CUDA;
  return CLSAMPLE_SUCCESS;
}

}  // namespace

struct clsample_handle {
  int max_batch;
  int vocab;
  int device;
  Geometry g;
  Scratch sc;
};

namespace {

// Scratch of clsample_apply_static: a fixed device array compiled into the library
// (zero at load, so the preparation kernel's ticket starts at 0), for kStaticRows rows.
constexpr int kStaticRows = 64;
constexpr size_t kStaticLists = (size_t)kStaticRows * kMaxCluster;
constexpr size_t kStaticOffPenN = align_up(kStaticLists * kPenCap * sizeof(PenEntry), 256);
constexpr size_t kStaticOffCand = kStaticOffPenN + align_up(kStaticLists * sizeof(int2), 256);
constexpr size_t kStaticOffRows = kStaticOffCand + align_up(kStaticLists * kCandCap * sizeof(Cand), 256);
constexpr size_t kStaticBytes = kStaticOffRows + align_up((2 * (size_t)kStaticRows + 1) * sizeof(int), 256);
static __device__ __align__(256) unsigned char g_static_scratch[kStaticBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mutex;
unsigned char* g_static_base[kMaxDevices];  // the array's address on each device, once set up

// The static scratch of device `dev` (its address taken and the kernels set up once per
// device); nullptr with *rc set on failure.
unsigned char* static_scratch(int dev, int* rc) {
  if (dev < 0 || dev >= kMaxDevices) {
    *rc = CLSAMPLE_ERR_DEVICE;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_static_mutex);
  if (!g_static_base[dev]) {
    *rc = setup_device(dev);
    if (*rc != CLSAMPLE_SUCCESS) return nullptr;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) {
      *rc = CLSAMPLE_ERR_CUDA;
      return nullptr;
    }
    g_static_base[dev] = static_cast<unsigned char*>(p);
  }
  *rc = CLSAMPLE_SUCCESS;
  return g_static_base[dev];
}

}  // namespace

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
  const int rc = setup_device(dev);
  if (rc != CLSAMPLE_SUCCESS) return rc;
  PenEntry* pen = nullptr;
  int2* pen_n = nullptr;
  Cand* cand = nullptr;
  int* rows = nullptr;
  if (max_batch > 0) {
    const size_t lists = (size_t)max_batch * (size_t)g.C;
    if (cudaMalloc(&pen, lists * kPenCap * sizeof(PenEntry)) != cudaSuccess ||
        cudaMalloc(&pen_n, lists * sizeof(int2)) != cudaSuccess ||
        cudaMalloc(&cand, lists * kCandCap * sizeof(Cand)) != cudaSuccess ||
        cudaMalloc(&rows, (2 * (size_t)max_batch + 1) * sizeof(int)) != cudaSuccess ||
        cudaMemset(rows, 0, (2 * (size_t)max_batch + 1) * sizeof(int)) != cudaSuccess) {
      if (pen) cudaFree(pen);
      if (pen_n) cudaFree(pen_n);
      if (cand) cudaFree(cand);
      if (rows) cudaFree(rows);
      return CLSAMPLE_ERR_CUDA;
    }
  }
  clsample_t* h = new clsample_t;
  h->max_batch = max_batch;
  h->vocab = vocab;
  h->device = dev;
  h->g = g;
  h->sc = Scratch{max_batch, pen, pen_n, cand, rows};
  *out = h;
  return CLSAMPLE_SUCCESS;
}

void clsample_destroy(clsample_t* h) {
  if (!h) return;
  if (h->sc.pen) cudaFree(h->sc.pen);
  if (h->sc.pen_n) cudaFree(h->sc.pen_n);
  if (h->sc.cand) cudaFree(h->sc.cand);
  if (h->sc.rows) cudaFree(h->sc.rows);
  delete h;
}

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

}  // extern "C"

namespace {

// Validates a call and fills the launch parameters (host only): the vocabulary must be
// `vocab`, the batch at most the scratch's rows, and `dev` the current device.
int make_params(const Geometry& g, int vocab, int dev, const Scratch& sc, const clsample_args_t* a,
                LaunchParams* P) {
  if (!a) return CLSAMPLE_ERR_NULL;
  if (a->B < 0 || a->B > sc.max_batch) return CLSAMPLE_ERR_BATCH;
  if (a->V != vocab) return CLSAMPLE_ERR_VOCAB;
  if (a->logits_dtype != CLSAMPLE_LOGITS_F32 && a->logits_dtype != CLSAMPLE_LOGITS_BF16) return CLSAMPLE_ERR_DTYPE;
  if (a->B == 0) return CLSAMPLE_SUCCESS;
  if (!a->logits || !a->tokens) return CLSAMPLE_ERR_NULL;
  if (a->hist_offs && !a->hist_ids) return CLSAMPLE_ERR_NULL;
  if (a->bias_offs && (!a->bias_ids || !a->bias_vals)) return CLSAMPLE_ERR_NULL;
  if (a->logits_row_stride < a->V) return CLSAMPLE_ERR_STRIDE;
  if (a->bitmask && a->bitmask_row_stride < (a->V + 31) / 32) return CLSAMPLE_ERR_STRIDE;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return CLSAMPLE_ERR_CUDA;
  if (cur != dev) return CLSAMPLE_ERR_DEVICE;
  const bool bf16 = a->logits_dtype == CLSAMPLE_LOGITS_BF16;
  const int esize = bf16 ? 2 : 4;
  P->a = *a;
  P->C = g.C;
  P->chunk = g.chunk;
  P->cap = g.cap;
  const uintptr_t base = reinterpret_cast<uintptr_t>(a->logits);
  P->vec_ok = (base % 16 == 0) && (((long long)a->logits_row_stride * esize) % 16 == 0);
  P->pen = sc.pen;
  P->pen_n = sc.pen_n;
  P->cand = sc.cand;
  P->row_class = sc.rows;
  P->row_order = sc.rows + sc.max_batch;
  P->ticket = reinterpret_cast<unsigned*>(sc.rows + 2 * (size_t)sc.max_batch);
  return CLSAMPLE_SUCCESS;
}

int make_params(const clsample_t* h, const clsample_args_t* a, LaunchParams* P) {
  if (!h) return CLSAMPLE_ERR_NULL;
  return make_params(h->g, h->vocab, h->device, h->sc, a, P);
}

int launch_prep(const LaunchParams& P, cudaStream_t st) {
  prep_kernel<<<(unsigned)(P.a.B * P.C), kPrepThreads, 0, st>>>(P);
  return cudaGetLastError() == cudaSuccess ? CLSAMPLE_SUCCESS : CLSAMPLE_ERR_CUDA;
}

int launch_sampler(const Geometry& g, const LaunchParams& P, cudaStream_t st) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  fill_launch(g, (unsigned)P.a.B, st, &cfg, attr);
  const cudaError_t err = P.a.logits_dtype == CLSAMPLE_LOGITS_BF16 ? cudaLaunchKernelEx(&cfg, sampler_kernel<true>, P)
                                                                    : cudaLaunchKernelEx(&cfg, sampler_kernel<false>, P);
  return err == cudaSuccess ? CLSAMPLE_SUCCESS : CLSAMPLE_ERR_CUDA;
}

}  // namespace

extern "C" {

int clsample_apply(clsample_t* h, const clsample_args_t* a, clsample_stream_t stream) {
  LaunchParams P;
  const int rc = make_params(h, a, &P);
  if (rc != CLSAMPLE_SUCCESS || a->B == 0) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int rp = launch_prep(P, st);
  return rp != CLSAMPLE_SUCCESS ? rp : launch_sampler(h->g, P, st);
}

int clsample_prepare(clsample_t* h, const clsample_args_t* a, clsample_stream_t stream) {
  LaunchParams P;
  const int rc = make_params(h, a, &P);
  if (rc != CLSAMPLE_SUCCESS || a->B == 0) return rc;
  return launch_prep(P, reinterpret_cast<cudaStream_t>(stream));
}

int clsample_sample(clsample_t* h, const clsample_args_t* a, clsample_stream_t stream) {
  LaunchParams P;
  const int rc = make_params(h, a, &P);
  if (rc != CLSAMPLE_SUCCESS || a->B == 0) return rc;
  return launch_sampler(h->g, P, reinterpret_cast<cudaStream_t>(stream));
}

int clsample_apply_static(const clsample_args_t* a, clsample_stream_t stream) {
  if (!a) return CLSAMPLE_ERR_NULL;
  const Geometry g = geometry_for(a->V);
  if (g.C == 0) return CLSAMPLE_ERR_VOCAB;
  if (a->B < 0 || a->B > kStaticRows) return CLSAMPLE_ERR_BATCH;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CLSAMPLE_ERR_CUDA;
  int rc = CLSAMPLE_SUCCESS;
  unsigned char* base = static_scratch(dev, &rc);
  if (!base) return rc;
  const Scratch sc{kStaticRows, reinterpret_cast<PenEntry*>(base), reinterpret_cast<int2*>(base + kStaticOffPenN),
                   reinterpret_cast<Cand*>(base + kStaticOffCand), reinterpret_cast<int*>(base + kStaticOffRows)};
  LaunchParams P;
  rc = make_params(g, a->V, dev, sc, a, &P);
  if (rc != CLSAMPLE_SUCCESS || a->B == 0) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  rc = launch_prep(P, st);
  return rc != CLSAMPLE_SUCCESS ? rc : launch_sampler(g, P, st);
}

int clsample_occupancy(clsample_t* h, int32_t logits_dtype, int32_t* max_active_clusters) {
  if (!h || !max_active_clusters) return CLSAMPLE_ERR_NULL;
  if (logits_dtype != CLSAMPLE_LOGITS_F32 && logits_dtype != CLSAMPLE_LOGITS_BF16) return CLSAMPLE_ERR_DTYPE;
  const bool bf16 = logits_dtype == CLSAMPLE_LOGITS_BF16;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  fill_launch(h->g, 1u, nullptr, &cfg, attr);
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
