// Batched constrained logits sampler for GB300 (sm_103a).
//
// A row's V logits are split into C slices of `chunk` tokens (a multiple of 32, so a
// slice owns whole bitmask words).  The sampler is one persistent kernel: every CTA
// (four per SM) takes work items from a global list, in order, with an atomic counter,
// and no CTA ever waits for another one's work except where the list says so.
//
//   P1 item   (row, slice): the slice's penalised / biased tokens from the row's
//             history and logit_bias lists, then pass A: the slice streams from HBM
//             through a 4-stage TMA ring (cp.async.bulk into shared memory, completing
//             on mbarriers) and gives its max, lowest argmax, online sum of
//             2^((z' - max) log2(e) / T), top-k bounds from per-thread maxima, and a
//             table of per-(thread, stage) maxima that later lets the row re-read only
//             the vectors that can hold candidates.  The slice record goes to global
//             memory and a per-row ticket counts the slices; the CTA that finishes the
//             row's last slice carries on with the row (no one waits for it).
//   row end   the last arriver combines the slice records, picks the truncation plan
//             and, for greedy and top-k / min-p rows, finishes the row alone: it reads
//             the tables, re-reads the few vectors above the top-k bound from L2,
//             compacts the candidates, finds top-k -> top-p -> min-p by exact selects
//             and runs the exponential race.
//   phases    rows that need every token a second time (top-p alone, min-p with top-p,
//             no truncation) get further per-slice items placed later in the list
//             (after about one wave of other items, so their first pass is done when
//             they are taken); an item of phase p waits, bounded, until the row's phase
//             p - 1 is complete, and the last arriver of each phase moves the row on.
//             Every wait is on items earlier in the list, which running CTAs took, so
//             the list cannot deadlock.
//
// A one-CTA kernel ahead of the sampler orders the rows heaviest first and writes the
// work list.  The arithmetic that decides integers (kept set, drawn id) is exact and
// identical on any IEEE machine (sampler_math.cuh).  Page references: "SGLang source
// teardown (10): Sampling, Grammar and structured output" (SGLang page) and "GLM-5.3
// inference (7): output side" (GLM page).

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

namespace {

using namespace clsample;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMinBlocks = 4;      // CTAs per SM the register budget is sized for
constexpr int kPenCap = 512;       // distinct penalised / biased ids per slice
constexpr int kCandCap = 4096;     // compacted candidates per slice segment (global scratch)
constexpr int kWhistBytes = 4096;  // top-p warp histograms (kWarps x 64 split counters)
constexpr int kMaxSlices = 8;      // slices per row
constexpr int kGatherCap = 4096;   // candidates the finishing CTA keeps in shared memory
constexpr int kMaxChunk = 32 * 1024;  // longest slice
constexpr int kStageBytes = 8192;     // one ring stage
constexpr int kStages = 4;            // ring depth
constexpr int kReload = 4;            // 16-byte loads in flight per thread when re-reading
constexpr int kTabMax = kMaxChunk * 4 / kStageBytes * kThreads;  // table entries per slice
constexpr int kOrderThreads = 512;
constexpr int kSmallRow = 2048;   // allowed tokens of a row that the row end takes all of
// penalised-token flags next to the history count
constexpr uint32_t kAllowedBit = 0x80000000u;
constexpr uint32_t kBiasBit = 0x40000000u;
constexpr uint32_t kCountMask = 0x3FFFFFFFu;
constexpr uint32_t kWaitLimit = 1u << 20;  // polls (<= 1 us apart) of a phase wait

enum : int { kRowOk = 0, kRowOverflow = 1, kRowInvalid = 2 };
enum : int { kFlagInvalid = 1, kFlagOverflow = 2, kFlagRing = 4 };  // kFlagRing: a wait gave up
enum : int { kPlanFast = 0, kPlanTopP = 1, kPlanUntrunc = 2, kPlanSlow = 3, kPlanDone = 4 };

struct Geometry {
  int C;      // slices per row
  int chunk;  // tokens per slice, multiple of 32
  int smem;   // dynamic shared memory per CTA
};

struct Cand {
  float y;
  int id;
};

// Lower bounds of the k-th largest z' come from maxima of disjoint token groups: each
// thread keeps one maximum per stage slot (kGroups groups), and the 32 maxima of one slot
// across a warp form a "group set".  A set whose j-th largest maximum is L guarantees j
// tokens at or above L.  For j = 2^i (i < kNJ) every slice reports the minimum of L over
// its sets that reach j maxima above -inf, and how many sets do; n such sets guarantee
// n*j tokens.
constexpr int kNJ = 6;  // j = 1, 2, 4, ..., 32

// Slice record of pass A.
struct X1 {
  float m;         // slice max of z' (-inf if no candidate)
  int arg;         // lowest id reaching m (INT_MAX if none)
  float s;         // sum over the slice's candidates of 2^((z' - m) * log2(e) / T)
  int flags;       // kFlag*
  float lk;        // max over warps of the warp's k-th largest thread max (k <= 32; else -inf)
  float lj[kNJ];   // min over the slice's groups reaching 2^i maxima of the 2^i-th largest
  unsigned char nj[8];  // how many groups reach 2^i (i < kNJ)
  int nallowed;    // allowed tokens of the slice
  int npen;        // penalised / biased tokens listed (at most kPenCap)
  int tab;         // 1: the table of vector maxima covers the slice's bulk part
};

// Slice record of a later phase.
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

// Row statistics and the truncation plan, set by the row's first phase end and read by
// its later phases.
struct RowState {
  float m;      // max z'
  int arg;      // lowest id reaching it
  float S;      // sum of 2^((z' - m) cS)
  int flags;
  float bound;  // lower bound of the k-th largest z' (-inf if none)
  int nallowed_max;  // the largest per-slice allowed-token count
  int nallowed_sum;  // allowed tokens of the row
  float lnS;
  float invT;
  float L;      // min-p cut in y: ln(min_p), or -inf
  float theta;  // lower bound of the kept set in y (kPlanFast)
  int plan;
  int needW;    // kPlanFast: the top-p mass is taken over the whole row
  int all;      // kPlanFast: every candidate of the row is compacted (theta = -inf)
  float s0;     // race score of the argmax token, which every kept set contains: a lower
                // bound of the winning score that seeds every race
  int bstar;    // top-p alone: the crossing bin
  unsigned long long above, cth;  // top-p alone: mass above the crossing bin; ceil(p W)
};

// One penalised / biased token of a slice, as the row preparation lists it.
constexpr uint32_t kPenBias = 0x80000000u;  // in PenEntry::id: a logit_bias entry applies
struct __align__(16) PenEntry {
  uint32_t id;     // local id | kPenBias
  uint32_t count;  // occurrences in the row's history (saturates at kCountMask)
  float bias;      // the last bias entry's value
  uint32_t pad;
};

struct LaunchParams {
  clsample_args_t a;
  int C;
  int chunk;
  int vec_ok;         // every row start is 16-byte aligned: slices stream through the TMA ring
  int gap;            // rows of the work list between a heavy row's phases
  // scratch (device)
  unsigned* ctl;      // [0] next item, [1] CTAs done, [2] work-list segments
  unsigned* ticket;   // [B][4] items of each phase of the row that have finished
  unsigned* phase_done;  // [B] the row's last completed phase
  unsigned* bad;      // [B] a phase wait of the row gave up
  unsigned* seg;      // [3 B] work list: row | phase << 24 | phases << 28, C items each
  int* order;         // [B] rows, heaviest class first
  RowState* rows;     // [B]
  X1* x1;             // [B * C]
  X2* x2;             // [B * C]
  PenEntry* plist;    // [B * C][kPenCap] penalised / biased tokens by id (row preparation)
  int2* plist_n;      // [B * C] their number, flags
  uint2* pen;         // [B * C][kPenCap] penalised tokens: local id, bits of z' (first phase)
  uint16_t* tab;      // [B * C][kTabMax] per-(stage, thread) maxima
  unsigned long long* phist;  // [B * C][kPBins] top-p bin masses
  Cand* cand;         // [B * C][kCandCap] compacted candidates
};

// ---------------------------------------------------------------- shared memory

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int kPBins = 64;
constexpr size_t kOffHistC = kWhistBytes;                                   // 4 KB
constexpr size_t kOffHistW = kOffHistC + sizeof(uint32_t) * 256;            // 5 KB
constexpr size_t kR2Bytes = 9 * 1024;

// Dynamic shared memory of one CTA (byte offsets):
//   ring      kStages x kStageBytes   the slice's stream (TMA destination); at a row end:
//                                     table hits, then the gathered candidates
//   live      u32[chunk/32]           allowed by the bitmask, inside the row, not penalised
//   mod       u32[chunk/32]           penalised / biased tokens
//   prank     u16[chunk/32]           rank of each mod word's first penalised token
//   pid/pcnt/pbias/pz [kPenCap]       the penalised tokens in token order: local id;
//                                     count | kBiasBit | kAllowedBit (pass A) ; bias
//                                     entry, then its value; raw logit in pass A, then the
//                                     final z'
//   r2 (9 KB) pass A: the table of vector maxima; later: top-p warp histograms [0, 4 KB),
//             hist_c u32[256] at 4 KB, hist_w u64[256] at 5 KB; at a row end the listed
//             penalised ids of every slice, then the bucket select
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
static_assert(sizeof(uint16_t) * kTabMax <= kR2Bytes, "table of vector maxima overflows r2");
static_assert(sizeof(uint16_t) * kPenCap * kMaxSlices <= kR2Bytes, "penalised ids overflow r2");
static_assert(kOffHistW + sizeof(unsigned long long) * 256 <= kR2Bytes, "r2 tables overflow");
static_assert(sizeof(unsigned long long) * 1024 <= kR2Bytes && sizeof(Cand) * 1024 <= kR2Bytes,
              "bucket select does not fit r2");
static_assert(2 * sizeof(uint32_t) * kWarps * kPBins <= kWhistBytes, "top-p histogram does not fit r2");
static_assert(sizeof(float) * kWarps * 4 * kNJ <= (size_t)kStages * kStageBytes, "group-set bounds overflow the ring");
static_assert(1024 % kThreads == 0, "bucket scan assumes whole buckets per thread");
static_assert(kStageBytes % (16 * kThreads) == 0, "a stage holds whole vectors per thread");
static_assert(kPenCap % kThreads == 0 && kPenCap <= 65536 && kMaxChunk <= 65536, "16-bit ids and ranks");
static_assert(kTabMax <= 4096 && kMaxSlices <= 16, "hit codes: slice << 16 | entry");

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
  s.gather = reinterpret_cast<Cand*>(b);
  return s;
}

// Static per-CTA state shared by the kernel's functions.
struct Shared {
  X1 x1[kMaxSlices];
  X2 x2[kMaxSlices];
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
  int poff[kMaxSlices + 1];
  float zth, res;
  int bstar, nl, flags, count, digit, none, npen, nallowed, nhits, last, ok;
  unsigned item;
  uint32_t seq;  // ring stages consumed by this CTA so far (fixes each buffer's parity)
  uint64_t policy;  // L2 policy of the current slice's stream
  unsigned long long tbar;  // the row end's table copies
  uint32_t tpar;     // its phase parity
  int tissued, tfail;  // copies issued and not yet waited for; a wait gave up
  uint32_t lean;       // pass A: stages whose tokens are all live or penalised
  unsigned long long above;
};
__shared__ Shared sh;

// The calling CTA's slice of a row.
struct Geo {
  int C, chunk, slice, row, c0, len, nvec;
  int bulk_tokens;  // tokens of the slice that stream through the ring (0: none)
  int nst;          // ring stages per pass
  const unsigned char* g;  // the slice's first logit
};

template <bool kBF16>
__device__ __forceinline__ Geo geo(const LaunchParams& P, int row, int slice) {
  constexpr int kEsize = kBF16 ? 2 : 4;
  Geo g;
  g.C = P.C;
  g.chunk = P.chunk;
  g.slice = slice;
  g.row = row;
  g.c0 = slice * g.chunk;
  g.len = max(0, min(P.a.V, g.c0 + g.chunk) - g.c0);
  g.nvec = g.chunk / 4;
  const int bulk = P.vec_ok ? (int)(((size_t)g.len * kEsize) & ~(size_t)15) : 0;
  g.bulk_tokens = bulk / kEsize;
  g.nst = (bulk + kStageBytes - 1) / kStageBytes;
  g.g = reinterpret_cast<const unsigned char*>(P.a.logits) +
        ((long long)row * P.a.logits_row_stride + g.c0) * kEsize;
  return g;
}

// ---------------------------------------------------------------- global memory between CTAs

// Data another CTA wrote during this launch is read at L2 (the L1 is not coherent).
template <typename T>
__device__ __forceinline__ void ldcg_copy(T* dst, const T* src) {
  static_assert(sizeof(T) % 4 == 0, "word copy");
  const uint32_t* s = reinterpret_cast<const uint32_t*>(src);
  uint32_t* d = reinterpret_cast<uint32_t*>(dst);
#pragma unroll
  for (int i = 0; i < (int)(sizeof(T) / 4); ++i) d[i] = __ldcg(s + i);
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// A candidate of a gathered array in shared memory or (when `global`) in the scratch.
__device__ __forceinline__ Cand ldcand(const Cand* G, int i, bool global) {
  if (global) {
    const float2 v = __ldcg(reinterpret_cast<const float2*>(G) + i);
    return Cand{v.x, __float_as_int(v.y)};
  }
  return G[i];
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
__device__ __forceinline__ float4 vload4(const unsigned char* base, int f) {
  if (kBF16) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(base) + f);
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                       __uint_as_float(w.y & 0xFFFF0000u));
  }
  return __ldg(reinterpret_cast<const float4*>(base) + f);
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

// Bitmask word w of a row's slice (32 tokens from c0 + 32 w), clipped to the row.
__device__ __forceinline__ uint32_t mask_word(const int32_t* bmrow, int c0, int len, int w) {
  const int e = 32 * w;
  if (e >= len) return 0u;
  uint32_t word = bmrow ? (uint32_t)__ldg(bmrow + (c0 >> 5) + w) : 0xFFFFFFFFu;
  const int rem = len - e;
  if (rem < 32) word &= (1u << rem) - 1u;
  return word;
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
__device__ __forceinline__ int pbin(float y) {
  const int b = __float2int_rz(__fmul_rn(-y, 4.0f));
  return b < kPBins - 1 ? b : kPBins - 1;
}

// Table entry of a group of tokens: 0 if none is live, else the top 16 bits of the
// order-preserving key of their largest z (so "entry >= top 16 bits of key(zth)" holds
// for every group with a live token at or above zth).
__device__ __forceinline__ uint16_t tab_entry(bool any, float vmax) {
  return (any && vmax > -INFINITY) ? (uint16_t)(fkey(vmax) >> 16) : (uint16_t)0;
}
__device__ __forceinline__ uint32_t tab_threshold(float zth) { return fkey(zth) >> 16; }

// ---------------------------------------------------------------- the TMA ring

// Issues stage k of the slice (stage sequence number s picks the buffer) on its barrier.
// Thread 0 only.
template <bool kBF16>
__device__ __forceinline__ void ring_issue(const Geo& g, const Smem& S, int k, uint32_t s) {
  constexpr int kEsize = kBF16 ? 2 : 4;
  const int off = k * kStageBytes;
  const uint32_t bytes = (uint32_t)min(kStageBytes, g.bulk_tokens * kEsize - off);
  const uint32_t slot = s % kStages;
  mbar_arrive_expect_tx(&sh.full[slot], bytes);
  bulk_copy_g2s_hint(S.ring + slot * kStageBytes, g.g + off, bytes, &sh.full[slot], sh.policy);
}

// Issues the first stages of the slice, continuing the CTA's stage sequence at seq0.
// Thread 0 only; the ring's previous contents (any proxy) are dead.
template <bool kBF16>
__device__ __forceinline__ void ring_start(const Geo& g, const Smem& S, uint32_t seq0) {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  for (int k = 0; k < min(kStages, g.nst); ++k) ring_issue<kBF16>(g, S, k, seq0 + (uint32_t)k);
}



// Waits (bounded, suspending) for ring stage s.  Thread 0 only; a stage that never lands
// marks the row OVERFLOW.
__device__ __forceinline__ void ring_wait(uint32_t s) {
  if (!mbar_wait_sleep(&sh.full[s % kStages], (s / kStages) & 1u)) atomicOr(&sh.flags, kFlagRing);
}

// Pass A's walk over the slice: body(t, f, wd, v) for every 4-token vector f (slot t of
// its stage), with its live bits wd and raw values v widened to f32, and stage_end(k)
// after every stage of the ring part.  Lanes without a vector get f = nvec (past the
// row) and wd = 0; every lane of a warp makes the same number of body calls.  A stage
// whose bit is set in `lean` (every token live or penalised) first gets patch(k, buf)
// (the penalised tokens leave the buffer), then lean(t, f, v) for every vector, with no
// per-token checks.  The ring part streams through the TMA ring (thread 0 started its
// first stages); the ragged tail and unaligned rows come in by plain loads (slot 0, no
// stage_end).
template <bool kBF16, class Body, class Lean, class Patch, class StageEnd>
__device__ __forceinline__ void stream_ring(const Geo& g, const Smem& S, uint32_t lean, Body&& body, Lean&& lean_body,
                                            Patch&& patch, StageEnd&& stage_end) {
  constexpr int kEsize = kBF16 ? 2 : 4;
  constexpr int kVecPerStage = kStageBytes / (4 * kEsize);
  constexpr int kVPT = kVecPerStage / kThreads;
  const int tid = threadIdx.x;
  const uint32_t seq0 = sh.seq;
#pragma unroll 1
  for (int k = 0; k < g.nst; ++k) {
    const uint32_t s = seq0 + (uint32_t)k;
    // thread 0 sleeps on the stage's barrier; the block barrier then also says that
    // every thread is done with stage k - 1, whose buffer is refilled at once
    if (tid == 0) ring_wait(s);
    __syncthreads();
    if (tid == 0 && k >= 1 && k - 1 + kStages < g.nst) ring_issue<kBF16>(g, S, k - 1 + kStages, s - 1 + kStages);
    (void)mbar_try_wait(&sh.full[s % kStages], (s / kStages) & 1u);  // this thread's acquire
    unsigned char* buf = S.ring + (s % kStages) * kStageBytes;
    if ((lean >> k) & 1u) {
      patch(k, buf);
#pragma unroll
      for (int t = 0; t < kVPT; ++t) {
        const int fl = t * kThreads + tid;
        lean_body(t, k * kVecPerStage + fl, sload4<kBF16>(buf, fl));
      }
    } else {
#pragma unroll
      for (int t = 0; t < kVPT; ++t) {
        const int fl = t * kThreads + tid;
        const int f = k * kVecPerStage + fl;
        const bool in = 4 * f < g.bulk_tokens;
        const uint32_t wd = in ? live4(S.live, f) : 0u;
        const float4 v = in ? sload4<kBF16>(buf, fl) : make_float4(0.f, 0.f, 0.f, 0.f);
        body(t, in ? f : g.nvec, wd, v);
      }
    }
    stage_end(k);
  }
  const int f_end = (g.len + 3) / 4;
#pragma unroll 1
  for (int base = g.bulk_tokens / 4; base < f_end; base += kThreads) {
    const int f = base + tid;
    const bool in = f < f_end;
    const uint32_t wd = in ? live4(S.live, f) : 0u;
    const float4 v = in ? gload4<kBF16>(g, f) : make_float4(0.f, 0.f, 0.f, 0.f);
    body(0, in ? f : g.nvec, wd, v);
  }
  __syncthreads();  // the ring is free; the bodies' shared writes are visible
  if (tid == 0) sh.seq = seq0 + (uint32_t)g.nst;
}

// A later pass over the slice, which is in L2 by now: body(f, wd, v) for every vector
// with a live token (plain 16-byte loads, kReload per thread in flight), lanes without
// one get f = nvec and wd = 0 (every lane of a warp makes the same number of calls).
template <bool kBF16, class Body>
__device__ __forceinline__ void stream_ldg(const Geo& g, const Smem& S, Body&& body) {
  const int tid = threadIdx.x;
  if (g.bulk_tokens > 0) {
    const int nv = g.bulk_tokens / 4;
#pragma unroll 1
    for (int base = 0; base < nv; base += kReload * kThreads) {
      float4 v[kReload];
      uint32_t wd[kReload];
#pragma unroll
      for (int u = 0; u < kReload; ++u) {
        const int f = base + u * kThreads + tid;
        const bool in = f < nv;
        wd[u] = in ? live4(S.live, f) : 0u;
        v[u] = wd[u] ? vload4<kBF16>(g.g, f) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kReload; ++u) {
        const int f = base + u * kThreads + tid;
        body(f < nv ? f : g.nvec, wd[u], v[u]);
      }
    }
  }
  const int f_end = (g.len + 3) / 4;
#pragma unroll 1
  for (int base = g.bulk_tokens / 4; base < f_end; base += kThreads) {
    const int f = base + tid;
    const bool in = f < f_end;
    const uint32_t wd = in ? live4(S.live, f) : 0u;
    const float4 v = in ? gload4<kBF16>(g, f) : make_float4(0.f, 0.f, 0.f, 0.f);
    body(in ? f : g.nvec, wd, v);
  }
  __syncthreads();
}

// A later-phase pass over the slice through the TMA ring: body(f, wd, v) for every
// vector, as stream_ldg gives them, but 32 KB in flight per CTA instead of kReload loads
// per thread.  Thread 0 started the ring (ring_start) before the pass.
template <bool kBF16, class Body>
__device__ __forceinline__ void stream_phase(const Geo& g, const Smem& S, Body&& body) {
  stream_ring<kBF16>(
      g, S, 0u, [&](int, int f, uint32_t wd, const float4& v) { body(f, wd, v); }, [](int, int, const float4&) {},
      [](int, unsigned char*) {}, [](int) {});
}

// ---------------------------------------------------------------- the work list

constexpr int kClasses = 5;
constexpr int kOrderPer = 8;  // rows per thread of the ordering kernel kept in registers

// Cost class of a row from its parameters alone (0 = heaviest: top-p alone, then
// untruncated or very large k, then large k or top-p over a min-p set, then the other
// sampling rows, then greedy or invalid rows; only the order of the work list uses it),
// and its work-list phases: rows that need every token a second time get one more
// per-slice pass (top-p mass over the whole row with min-p; the race over every token
// when nothing is truncated) or two (top-p alone: the mass histogram, then the race);
// every other row ends at the end of its first phase.
__device__ __forceinline__ void row_info(const clsample_args_t& a, int row, int* cls, int* nph) {
  const float T = a.temperatures ? __ldg(a.temperatures + row) : 1.0f;
  const int k = a.top_ks ? __ldg(a.top_ks + row) : -1;
  const float p = a.top_ps ? __ldg(a.top_ps + row) : 1.0f;
  const float mp = a.min_ps ? __ldg(a.min_ps + row) : 0.0f;
  if (!(T >= kGreedyEps) || k == 0 || k == 1 || k < -1) {
    *cls = 4;
    *nph = 1;
    return;
  }
  const bool kfin = k >= 2;
  if (!kfin && p < 1.0f && !(mp > 0.0f)) *cls = 0;
  else if ((!kfin && !(mp > 0.0f)) || k >= 512) *cls = 1;
  else if (k >= 64 || (!kfin && p < 1.0f)) *cls = 2;
  else *cls = 3;
  if (kfin) *nph = 1;
  else if (p < 1.0f) *nph = mp > 0.0f ? 2 : 3;
  else *nph = mp > 0.0f ? 1 : 2;
}

// Block-wide exclusive scan of one int per thread (kOrderThreads threads); returns the
// thread's offset, *total the sum.
__device__ int order_scan(int x, int* red, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  __syncthreads();
  if (lane == 31) red[warp] = incl;
  __syncthreads();
  int before = 0, tot = 0;
  for (int w = 0; w < kOrderThreads / 32; ++w) {
    if (w < warp) before += red[w];
    tot += red[w];
  }
  *total = tot;
  return before + incl - x;
}


constexpr int kRowPen = kPenCap * kMaxSlices;  // distinct penalised / biased ids of a row

// Shared memory of a row preparation CTA for a vocabulary of V tokens.
__host__ __device__ inline size_t prep_smem_bytes(int V) {
  const size_t W = (size_t)(V + 31) / 32;
  return sizeof(uint32_t) * 2 * W + sizeof(uint32_t) * 2 * kRowPen;
}

// Row preparation: one CTA of the ordering launch per row.  The row's history and
// logit_bias ids are marked in a bitmap of the vocabulary (shared memory), ranked in
// token order by a scan of the words' popcounts, counted (duplicates in a warp counted
// once: Zipf-like histories repeat their frequent ids many times), and every bias entry
// leaves its index at its id's rank, so that the last entry of an id wins (SGLang page,
// "Order semantics of the penalties" and "Why logit_bias is built from triples").  Then
// every slice gets its list of (local id, count, bias) in id order, with its length and
// flags: INVALID for ids outside [0, V), decreasing CSR offsets or NaN bias values,
// OVERFLOW for a slice with more than kPenCap distinct ids.
__device__ __noinline__ void prep_row(const LaunchParams& P, int row) {
  const clsample_args_t& a = P.a;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int W = (a.V + 31) / 32, C = P.C, chunk = P.chunk;
  uint32_t* bits = reinterpret_cast<uint32_t*>(smem_dyn);  // [W]
  uint32_t* prk = bits + W;                                 // [W] rank of each word's first id
  uint32_t* cnt = prk + W;                                  // [kRowPen]
  int* bidx = reinterpret_cast<int*>(cnt + kRowPen);        // [kRowPen]
  __shared__ int pcsr[4], pflags, ptot;
  __shared__ int pred[kOrderThreads / 32];
  const bool has_hist = a.hist_offs != nullptr, has_bias = a.bias_offs != nullptr;
  if (tid == 0) {
    pcsr[0] = has_hist ? a.hist_offs[row] : 0;
    pcsr[1] = has_hist ? a.hist_offs[row + 1] : 0;
    pcsr[2] = has_bias ? a.bias_offs[row] : 0;
    pcsr[3] = has_bias ? a.bias_offs[row + 1] : 0;
    pflags = 0;
  }
  for (int w = tid; w < W; w += kOrderThreads) bits[w] = 0u;
  for (int r = tid; r < kRowPen; r += kOrderThreads) {
    cnt[r] = 0u;
    bidx[r] = -1;
  }
  __syncthreads();
  int flags = 0;
  const int hlo = pcsr[0], hhi = pcsr[1], blo = pcsr[2], bhi = pcsr[3];
  if (hlo < 0 || hhi < hlo || blo < 0 || bhi < blo) flags |= kFlagInvalid;
  const bool hok = has_hist && hlo >= 0 && hhi >= hlo;
  const bool bok = has_bias && blo >= 0 && bhi >= blo;
  constexpr int kBatch = 8;
  if (hok) {
#pragma unroll 1
    for (int base = hlo; base < hhi; base += kBatch * kOrderThreads) {
      int ids[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int j = base + u * kOrderThreads + tid;
        ids[u] = j < hhi ? __ldg(a.hist_ids + j) : INT_MIN;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int id = ids[u];
        if (id == INT_MIN) continue;
        if (id < 0 || id >= a.V) {
          flags |= kFlagInvalid;
          continue;
        }
        const uint32_t bit = 1u << (id & 31);
        if (!(bits[id >> 5] & bit)) atomicOr(&bits[id >> 5], bit);
      }
    }
  }
  if (bok) {
    for (int j = blo + tid; j < bhi; j += kOrderThreads) {
      const int id = __ldg(a.bias_ids + j);
      const float b = __ldg(a.bias_vals + j);
      if (id < 0 || id >= a.V || b != b) flags |= kFlagInvalid;
      else atomicOr(&bits[id >> 5], 1u << (id & 31));
    }
  }
  if (flags) atomicOr(&pflags, flags);
  __syncthreads();
  // ranks: an exclusive scan of the words' popcounts, consecutive words per thread
  {
    const int per = (W + kOrderThreads - 1) / kOrderThreads;
    const int w0 = min(W, tid * per), w1 = min(W, w0 + per);
    int loc = 0;
    for (int w = w0; w < w1; ++w) loc += __popc(bits[w]);
    int x = loc;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += o;
    }
    if (lane == 31) pred[warp] = x;
    __syncthreads();
    int e = x - loc, tot = 0;
    for (int wp = 0; wp < kOrderThreads / 32; ++wp) {
      if (wp < warp) e += pred[wp];
      tot += pred[wp];
    }
    for (int w = w0; w < w1; ++w) {
      prk[w] = (uint32_t)e;
      e += __popc(bits[w]);
    }
    if (tid == 0) ptot = tot;
  }
  __syncthreads();
  auto rank_of = [&](int id) -> uint32_t {
    return prk[id >> 5] + __popc(bits[id >> 5] & ((1u << (id & 31)) - 1u));
  };
  if (hok) {
#pragma unroll 1
    for (int base = hlo; base < hhi; base += kBatch * kOrderThreads) {
      int ids[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int j = base + u * kOrderThreads + tid;
        ids[u] = j < hhi ? __ldg(a.hist_ids + j) : INT_MIN;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int id = ids[u];
        int r = -1;
        if (id >= 0 && id < a.V) {
          const uint32_t rr = rank_of(id);
          r = rr < (uint32_t)kRowPen ? (int)rr : -1;
        }
        const uint32_t peers = __match_any_sync(0xffffffffu, r);
        if (r >= 0 && lane == __ffs(peers) - 1) atomicAdd(&cnt[r], (uint32_t)__popc(peers));
      }
    }
  }
  if (bok) {
    for (int j = blo + tid; j < bhi; j += kOrderThreads) {
      const int id = __ldg(a.bias_ids + j);
      const float b = __ldg(a.bias_vals + j);
      if (id >= 0 && id < a.V && b == b) {
        const uint32_t r = rank_of(id);
        if (r < (uint32_t)kRowPen) atomicMax(&bidx[r], j);
      }
    }
  }
  __syncthreads();
  // the slices' lists, in id order
  PenEntry* out = P.plist + (size_t)row * C * kPenCap;
  for (int w = tid; w < W; w += kOrderThreads) {
    uint32_t b = bits[w];
    uint32_t r = prk[w];
    while (b) {
      const int bit = __ffs(b) - 1;
      b &= b - 1u;
      const int id = 32 * w + bit;
      const int sl = id / chunk;
      const uint32_t rs = prk[(sl * chunk) >> 5];
      const uint32_t p = r - rs;
      if (r < (uint32_t)kRowPen && p < (uint32_t)kPenCap) {
        const int bj = bidx[r];
        PenEntry en;
        en.id = (uint32_t)(id - sl * chunk) | (bj >= 0 ? kPenBias : 0u);
        en.count = min(cnt[r], kCountMask);
        en.bias = bj >= 0 ? __ldg(a.bias_vals + bj) : 0.0f;
        en.pad = 0u;
        out[(size_t)sl * kPenCap + p] = en;
      }
      ++r;
    }
  }
  if (tid < C) {
    const uint32_t r0 = prk[(tid * chunk) >> 5];
    const uint32_t r1 = tid + 1 < C ? prk[((tid + 1) * chunk) >> 5] : (uint32_t)ptot;
    int f = pflags;
    if (r1 - r0 > (uint32_t)kPenCap || r1 > (uint32_t)kRowPen) f |= kFlagOverflow;
    P.plist_n[(size_t)row * C + tid] = make_int2((int)min(r1 - r0, (uint32_t)kPenCap), f);
  }
}

// The ordering launch ahead of the sampler.  CTA 0 resets the scratch's counters, orders
// the rows by class (stable, heaviest first; order[] holds row | phases << 24) and writes
// the work list; CTAs 1 .. B (when the call has penalties or logit_bias) prepare the rows'
// penalised-token lists.
// List slot j holds the first phase of order[j], then the second phase of order[j - gap]
// and the third of order[j - 2 gap] where those rows have them (slots j >= B hold only
// those), so that a row's next phase comes about one wave of items after its previous
// one.
__global__ void __launch_bounds__(kOrderThreads, 2) order_kernel(const __grid_constant__ LaunchParams P) {
  // the sampler may be scheduled now: it waits for this grid's results (griddepcontrol.wait)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x > 0) {
    prep_row(P, (int)blockIdx.x - 1);
    return;
  }
  __shared__ int red[kOrderThreads / 32];
  const clsample_args_t& a = P.a;
  const int B = a.B, tid = threadIdx.x;
  for (int r = tid; r < B; r += kOrderThreads) {
    reinterpret_cast<uint4*>(P.ticket)[r] = make_uint4(0u, 0u, 0u, 0u);
    P.phase_done[r] = 0u;
    P.bad[r] = 0u;
  }
  if (tid == 0) {
    P.ctl[0] = 0u;
    P.ctl[1] = 0u;
  }
  // classes -> order: consecutive rows per thread, one scan per class
  {
    const int per = (B + kOrderThreads - 1) / kOrderThreads;
    const int r0 = min(B, tid * per), r1 = min(B, r0 + per);
    int cls[kOrderPer], nph[kOrderPer];
    int cnt[kClasses] = {0, 0, 0, 0, 0};
#pragma unroll
    for (int u = 0; u < kOrderPer; ++u)
      if (r0 + u < r1) {
        row_info(a, r0 + u, &cls[u], &nph[u]);
        ++cnt[cls[u]];
      }
    for (int r = r0 + kOrderPer; r < r1; ++r) {
      int c, n;
      row_info(a, r, &c, &n);
      ++cnt[c];
    }
    int base[kClasses], start = 0;
#pragma unroll
    for (int c = 0; c < kClasses; ++c) {
      int tot;
      base[c] = order_scan(cnt[c], red, &tot) + start;
      start += tot;
    }
#pragma unroll
    for (int u = 0; u < kOrderPer; ++u)
      if (r0 + u < r1) P.order[base[cls[u]]++] = (r0 + u) | (nph[u] << 24);
    for (int r = r0 + kOrderPer; r < r1; ++r) {
      int c, n;
      row_info(a, r, &c, &n);
      P.order[base[c]++] = r | (n << 24);
    }
  }
  __threadfence_block();
  __syncthreads();
  // the work list
  const int G = P.gap;
  const int J = B + 2 * G;
  const int per = (J + kOrderThreads - 1) / kOrderThreads;
  const int j0 = min(J, tid * per), j1 = min(J, j0 + per);
  auto entries = [&](int j, unsigned* out) -> int {
    int n = 0;
    const int o1 = j < B ? __ldcg(P.order + j) : -1;
    const int o2 = (j - G >= 0 && j - G < B) ? __ldcg(P.order + j - G) : -1;
    const int o3 = (j - 2 * G >= 0 && j - 2 * G < B) ? __ldcg(P.order + j - 2 * G) : -1;
    if (o1 >= 0) {
      if (out) out[n] = ((unsigned)o1 & 0xFFFFFFu) | (1u << 24) | ((unsigned)(o1 >> 24) << 28);
      ++n;
    }
    if (o2 >= 0 && (o2 >> 24) >= 2) {
      if (out) out[n] = ((unsigned)o2 & 0xFFFFFFu) | (2u << 24) | ((unsigned)(o2 >> 24) << 28);
      ++n;
    }
    if (o3 >= 0 && (o3 >> 24) >= 3) {
      if (out) out[n] = ((unsigned)o3 & 0xFFFFFFu) | (3u << 24) | ((unsigned)(o3 >> 24) << 28);
      ++n;
    }
    return n;
  };
  int mine = 0;
  for (int j = j0; j < j1; ++j) mine += entries(j, nullptr);
  int total;
  int pos = order_scan(mine, red, &total);
  for (int j = j0; j < j1; ++j) {
    unsigned e[3];
    const int n = entries(j, e);
    for (int i = 0; i < n; ++i) P.seg[pos++] = e[i];
  }
  if (tid == 0) P.ctl[2] = (unsigned)total;
}

// ---------------------------------------------------------------- first phase: setup

// Row parameters and their validity.
__device__ __forceinline__ RowParams load_params(const clsample_args_t& a, int row) {
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
  return q;
}

__device__ __forceinline__ bool params_greedy(const RowParams& q) {
  return (q.T < kGreedyEps) || q.k == 0 || q.k == 1;
}

// Exclusive scan of the mod words' popcounts into prank (token-order rank of each word's
// first penalised token); returns the total in every thread.
__device__ int rank_words(const Smem& S, int nw) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kPer = (kMaxChunk / 32) / kThreads;
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
  int excl = x - loc, total = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) excl += sh.red_i[w];
    total += sh.red_i[w];
  }
#pragma unroll
  for (int t = 0; t < kPer; ++t) {
    const int w = tid * kPer + t;
    if (w < nw) S.prank[w] = (uint16_t)excl;
    excl += cnt[t];
  }
  __syncthreads();
  return total;
}

// First phase of a slice, before pass A: thread 0 starts the slice's first ring stages,
// then the row parameters, the live bits (bitmask words clipped to the row) and the
// slice's penalised / biased tokens from the row preparation's list (in id order, so an
// entry's index is the token's rank); the bitmask's verdict on each moves into its entry
// and the token leaves the live set (pass A gives it its final value).
template <bool kBF16>
__device__ __noinline__ void setup_p1(const LaunchParams& P, int row, int slice, int nph) {
  const Geo g = geo<kBF16>(P, row, slice);
  const Smem S = carve(g.chunk);
  const clsample_args_t& a = P.a;
  const int tid = threadIdx.x, lane = tid & 31;
  const int nw = g.chunk / 32;
  const int32_t* bmrow = a.bitmask ? a.bitmask + (long long)row * a.bitmask_row_stride : nullptr;
  const bool has_mod = a.hist_offs != nullptr || a.bias_offs != nullptr;
  const size_t rc = (size_t)row * P.C + slice;
  (void)nph;
  if (tid == 0) {
    sh.flags = 0;
    sh.lean = 0u;
    sh.count = 0;
    sh.nallowed = 0;  // (sh.npen is thread 64's)
    ring_start<kBF16>(g, S, sh.seq);
  } else if (tid == 32) {
    sh.rp = load_params(a, row);
  } else if (tid == 64) {
    const int2 nf = has_mod ? P.plist_n[rc] : make_int2(0, 0);
    sh.npen = nf.x;
    sh.csr[0] = nf.y;  // the row preparation's flags
  }
  // the list is loaded whole (its length arrives with it): kPenCap / kThreads per thread
  PenEntry en[kPenCap / kThreads];
  if (has_mod) {
#pragma unroll
    for (int t = 0; t < kPenCap / kThreads; ++t) en[t] = P.plist[rc * kPenCap + t * kThreads + tid];
  }
  for (int w = tid; w < nw; w += kThreads) {
    S.live[w] = mask_word(bmrow, g.c0, g.len, w);
    S.mod[w] = 0u;
  }
  __syncthreads();
  if (!has_mod) {
    int na = 0;
    for (int w = tid; w < nw; w += kThreads) na += __popc(S.live[w]);
    na = __reduce_add_sync(0xffffffffu, na);
    if (lane == 0 && na) atomicAdd(&sh.nallowed, na);
    __syncthreads();
    return;
  }
  const int npen = sh.npen;
  if (tid == 0 && sh.csr[0]) sh.flags |= sh.csr[0];
#pragma unroll
  for (int t = 0; t < kPenCap / kThreads; ++t) {
    const int r = t * kThreads + tid;
    if (r >= npen) continue;
    const uint32_t l = en[t].id & ~kPenBias;
    const uint32_t bit = 1u << (l & 31);
    uint32_t c = min(en[t].count, kCountMask);
    if (en[t].id & kPenBias) c |= kBiasBit;
    if (S.live[l >> 5] & bit) c |= kAllowedBit;
    S.pid[r] = (uint16_t)l;
    S.pcnt[r] = c;
    S.pbias[r] = en[t].bias;
    atomicAnd(&S.live[l >> 5], ~bit);
    atomicOr(&S.mod[l >> 5], bit);
  }
  __syncthreads();
  (void)rank_words(S, nw);
  {
    int na = 0;
    for (int w = tid; w < nw; w += kThreads) na += __popc(S.live[w]);
    for (int r = tid; r < npen; r += kThreads) na += (S.pcnt[r] & kAllowedBit) ? 1 : 0;
    na = __reduce_add_sync(0xffffffffu, na);
    if (lane == 0 && na) atomicAdd(&sh.nallowed, na);
  }
  __syncthreads();
}

// ---------------------------------------------------------------- pass A

// Pass A: slice max, lowest argmax and online sum of 2^((z' - max) cS), cS = log2(e)/T_eff;
// per-warp lower bounds of the top-k cut from the per-thread maxima; the table of
// per-(stage, thread) maxima in r2.  Leaves the slice record in sh.x1_mine.
template <bool kBF16>
__device__ __noinline__ void pass_a(const LaunchParams& P, int row, int slice) {
  const Geo g = geo<kBF16>(P, row, slice);
  const Smem S = carve(g.chunk);
  const clsample_args_t& a = P.a;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RowParams q = sh.rp;
  const bool has_mod = a.hist_offs != nullptr || a.bias_offs != nullptr;
  const bool greedy = params_greedy(q);
  const float Teff = (q.T >= kGreedyEps) ? q.T : 1.0f;
  const float cS = 1.4426950408889634f / Teff;
  const int c0 = g.c0;
  constexpr int kGroups = kStageBytes / (4 * (kBF16 ? 2 : 4)) / kThreads;  // vectors per thread per stage
  static_assert(kGroups <= 4, "four group sets per warp at most");
  uint16_t* tab = reinterpret_cast<uint16_t*>(S.r2);

  constexpr int kTokPerStage = kStageBytes / (kBF16 ? 2 : 4);
  constexpr int kWordsPerStage = kTokPerStage / 32;
  const int nw = g.chunk / 32;

  // lean stages: every token live (allowed, inside the row) or penalised / biased, and
  // the whole stage inside the ring part (one warp per stage)
  for (int k = warp; k < g.nst; k += kWarps) {
    const int w0 = k * kWordsPerStage;
    bool all = (k + 1) * kTokPerStage <= g.bulk_tokens;
    for (int w = w0 + lane; w < w0 + kWordsPerStage; w += 32) all = all && (S.live[w] | S.mod[w]) == 0xFFFFFFFFu;
    if (__all_sync(0xffffffffu, all) && lane == 0) atomicOr(&sh.lean, 1u << k);
  }
  __syncthreads();
  uint32_t lean = sh.lean;

  // the thread's online state; a thread visits its tokens in increasing order, so the
  // first token reaching the running max is the lowest
  float sm, ss;
  int targ;
  // the maxima of the thread's vectors in each stage slot: kGroups disjoint token groups
  // per thread for the top-k bounds
  float gm[kGroups];
  float tmax;  // this stage's maximum (table)
  bool tany;
  float gmin;  // lean stages: the smallest vector maximum (-inf: a vector of -inf logits)
  for (;;) {
    sm = -INFINITY;
    ss = 0.0f;
    targ = INT_MAX;
#pragma unroll
    for (int t = 0; t < kGroups; ++t) gm[t] = -INFINITY;
    tmax = -INFINITY;
    tany = false;
    gmin = INFINITY;
    stream_ring<kBF16>(
        g, S, lean,
        [&](int t, int f, uint32_t wd, const float4& v) {
          if (has_mod && 4 * f < g.len) {
            // penalised / biased tokens: keep the raw logit (rank order) for the fold below
            const uint32_t mw = S.mod[f >> 3];
            const int sh4 = (f & 7) * 4;
            const uint32_t md = (mw >> sh4) & 0xFu;
            if (md) {
              int r = S.prank[f >> 3] + __popc(mw & ((1u << sh4) - 1u));
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if ((md >> j) & 1u) {
                  if (r < kPenCap) S.pz[r] = comp(v, j);
                  ++r;
                }
            }
          }
          if (!wd) return;
          float4 z = v;
          if (!(wd == 0xFu && finite4(v)))
            z = make_float4((wd & 1u) ? sanitize(v.x) : -INFINITY, (wd & 2u) ? sanitize(v.y) : -INFINITY,
                            (wd & 4u) ? sanitize(v.z) : -INFINITY, (wd & 8u) ? sanitize(v.w) : -INFINITY);
          const float fm = fmaxf(fmaxf(z.x, z.y), fmaxf(z.z, z.w));
          tany = true;
          tmax = fmaxf(tmax, fm);
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
        },
        // lean vector: no mask, penalty or finiteness checks (a non-finite logit shows in
        // ss or gmin, and the slice is then walked again with the checks)
        [&](int t, int f, const float4& v) {
          const float fm = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
          gmin = fminf(gmin, fm);
          tany = true;
          tmax = fmaxf(tmax, fm);
          gm[t] = fmaxf(gm[t], fm);
          if (fm > sm) {
            ss *= ex2_approx((sm - fm) * cS);
            sm = fm;
            targ = c0 + 4 * f + (v.x == fm ? 0 : v.y == fm ? 1 : v.z == fm ? 2 : 3);
          }
          const float e0 = ex2_approx((v.x - sm) * cS), e1 = ex2_approx((v.y - sm) * cS);
          const float e2 = ex2_approx((v.z - sm) * cS), e3 = ex2_approx((v.w - sm) * cS);
          ss += (e0 + e1) + (e2 + e3);
        },
        // a lean stage's penalised / biased tokens: raw logit to the fold below, -inf in
        // the buffer (a -inf lean token counts for nothing)
        [&](int k, unsigned char* buf) {
          if (!has_mod) return;
          const int w0 = k * kWordsPerStage, w1 = w0 + kWordsPerStage;
          const int r0 = S.prank[w0];
          const int r1 = w1 < nw ? (int)S.prank[w1] : (int)S.prank[nw - 1] + __popc(S.mod[nw - 1]);
          if (r1 <= r0) return;  // the same in every thread
          for (int r = r0 + tid; r < min(r1, kPenCap); r += kThreads) {
            const int i = (int)S.pid[r] - k * kTokPerStage;
            if (kBF16) {
              uint16_t* b16 = reinterpret_cast<uint16_t*>(buf);
              S.pz[r] = __uint_as_float((uint32_t)b16[i] << 16);
              b16[i] = (uint16_t)0xFF80u;
            } else {
              float* b32 = reinterpret_cast<float*>(buf);
              S.pz[r] = b32[i];
              b32[i] = -INFINITY;
            }
          }
          // the buffer is refilled by the async proxy later
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncthreads();
        },
        [&](int k) {
          tab[k * kThreads + tid] = tab_entry(tany, tmax);
          tany = false;
          tmax = -INFINITY;
        });
    // a lean stage saw NaN / +inf (ss is NaN) or a vector of -inf logits: walk the slice
    // again with every check (thread 0 restarts the ring)
    const bool bad = lean != 0u && (!(ss <= FLT_MAX) || gmin == -INFINITY);
    if (!__syncthreads_or(bad)) break;
    lean = 0u;
    if (tid == 0) ring_start<kBF16>(g, S, sh.seq);
  }
  // the penalised / biased tokens in token order: penalties, then bias, on the sanitised
  // raw logit (the mask applies to them too); the final z' replaces the raw one and joins
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
  // per group set, in the ring (free after the stream)
  float(*red_j)[kNJ] = reinterpret_cast<float(*)[kNJ]>(S.ring);
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
      sh.x1_mine.npen = has_mod ? sh.npen : 0;
      sh.x1_mine.tab = P.vec_ok;
    }
  }
  // the transformed logits, on request (debugging aid): plain values first, then the
  // penalised / biased tokens' final z'
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

// End of a first-phase item: the slice record, its penalised tokens (local id and final
// z', token order) and its table go to the scratch, then the row's ticket.  Returns true
// in every thread of the CTA that finished the row's last slice (the phase's ticket is
// reset for the next call).
template <bool kBF16>
__device__ __noinline__ bool publish_p1(const LaunchParams& P, int row, int slice) {
  const Geo g = geo<kBF16>(P, row, slice);
  const Smem S = carve(g.chunk);
  const int tid = threadIdx.x;
  const size_t idx = (size_t)row * P.C + slice;
  const RowParams q = sh.rp;
  const bool sampling = !params_greedy(q) && !q.invalid;  // only sampling rows read lists and tables again
  if (tid == 0) P.x1[idx] = sh.x1_mine;
  if (sampling) {
    const int npen = sh.x1_mine.npen;
    uint2* pl = P.pen + idx * kPenCap;
    for (int r = tid; r < npen; r += kThreads) pl[r] = make_uint2(S.pid[r], __float_as_uint(S.pz[r]));
    if (P.vec_ok && g.nst > 0) {
      const uint4* src = reinterpret_cast<const uint4*>(S.r2);
      uint4* dst = reinterpret_cast<uint4*>(P.tab + idx * kTabMax);
      const int n16 = g.nst * kThreads * (int)sizeof(uint16_t) / 16;
      for (int i = tid; i < n16; i += kThreads) dst[i] = src[i];
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const bool last = atomicAdd(P.ticket + 4 * row + 1, 1u) == (unsigned)P.C - 1u;
    if (last) P.ticket[4 * row + 1] = 0u;
    sh.last = last ? 1 : 0;
  }
  __syncthreads();
  if (!sh.last) return false;
  __threadfence();
  return true;
}

// ---------------------------------------------------------------- row end: combine and plan

// The last arriver of a row's first phase: the C slice records, combined in slice order
// (every float sum in a fixed order) into sh.rs.  The top-k bound is the larger of the
// warps' k-th largest thread maxima and, for each j = 2^i whose group sets guarantee k
// tokens (n * j >= k), the minimum over those sets of their j-th largest maximum.
__device__ __noinline__ void combine_row(const LaunchParams& P, int row) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = P.C;
  const RowParams q = sh.rp;
  const float Teff = (q.T >= kGreedyEps) ? q.T : 1.0f;
  const float cS = 1.4426950408889634f / Teff;
  if (tid < C) ldcg_copy(&sh.x1[tid], P.x1 + (size_t)row * C + tid);
  __syncthreads();
  if (warp == 0) {
    const bool in = lane < C;
    const float lm = in ? sh.x1[lane].m : -INFINITY;
    const int la = in ? sh.x1[lane].arg : INT_MAX;
    const float ls = in ? sh.x1[lane].s : 0.0f;
    int fl = in ? sh.x1[lane].flags : 0;
    float lk = in ? sh.x1[lane].lk : -INFINITY;
    int nal = in ? sh.x1[lane].nallowed : 0;
    const int nsum = __reduce_add_sync(0xffffffffu, nal);
    float m = lm;
#pragma unroll
    for (int d = 4; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
    m = __shfl_sync(0xffffffffu, m, 0);  // lanes >= 8 may hold their own partial maxima
    int arg = (in && lm == m) ? la : INT_MAX;
    const float term = (in && lm > -INFINITY) ? ls * ex2_approx((lm - m) * cS) : 0.0f;
#pragma unroll
    for (int d = 4; d > 0; d >>= 1) {
      arg = min(arg, __shfl_xor_sync(0xffffffffu, arg, d));
      fl |= __shfl_xor_sync(0xffffffffu, fl, d);
      lk = fmaxf(lk, __shfl_xor_sync(0xffffffffu, lk, d));
      nal = max(nal, __shfl_xor_sync(0xffffffffu, nal, d));
    }
    float bj = -INFINITY;
    if (lane < kNJ) {
      float lj = INFINITY;
      uint32_t n = 0;
      for (int c = 0; c < C; ++c) {
        lj = fminf(lj, sh.x1[c].lj[lane]);
        n += sh.x1[c].nj[lane];
      }
      if (n > 0 && (unsigned long long)n << lane >= (unsigned long long)max(q.k, 0)) bj = lj;
    }
    for (int d = 4; d > 0; d >>= 1) bj = fmaxf(bj, __shfl_xor_sync(0xffffffffu, bj, d));
    // the sum in a fixed order (slices 0 .. C-1)
    float tot = 0.0f;
#pragma unroll
    for (int r = 0; r < kMaxSlices; ++r) tot += __shfl_sync(0xffffffffu, term, r);
    if (lane == 0) {
      sh.rs.m = m;
      sh.rs.arg = arg;
      sh.rs.S = tot;
      sh.rs.flags = fl;
      sh.rs.bound = fmaxf(lk, bj);
      sh.rs.nallowed_max = nal;
      sh.rs.nallowed_sum = nsum;
      sh.rs.lnS = logf(tot);
    }
  }
  __syncthreads();
}

// Greedy, INVALID and OVERFLOW rows end after the first phase: the argmax (its y is 0,
// so its logprob is -ln S).  Returns true (in every thread) if the row ended.
__device__ __noinline__ bool finish_early(const LaunchParams& P, int row) {
  const RowParams q = sh.rp;
  const float m = sh.rs.m;
  const int fl = sh.rs.flags;
  int status = kRowOk;
  if (q.invalid || (fl & kFlagInvalid) || !(m > -INFINITY)) status = kRowInvalid;
  else if (fl & (kFlagOverflow | kFlagRing)) status = kRowOverflow;
  if (status == kRowOk && !params_greedy(q)) return false;
  if (threadIdx.x == 0) {
    const clsample_args_t& a = P.a;
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
//  * top-k rows: the row end compacts the tokens at or above a lower bound of the k-th
//    largest (the group-set bound, tightened by the table of group maxima);
//  * rows with few allowed tokens: the row end compacts all of them;
//  * min-p rows: K lies in {y >= ln min_p} (with top-p, its mass is taken over the whole
//    row in a later phase);
//  * untruncated rows and top-p alone: later phases over every slice.
__device__ __noinline__ void plan_row() {
  if (threadIdx.x == 0) {
    const RowParams q = sh.rp;
    RowState& rs = sh.rs;
    rs.invT = __frcp_rn(q.T);
    rs.L = q.mp > 0.0f ? (float)log((double)q.mp) : -INFINITY;  // min-p: y >= ln(min_p)
    const bool kfin = q.k >= 2;
    int plan = kPlanSlow, needW = 0, all = 0;
    float theta = -INFINITY;
    if (kfin) {
      plan = kPlanFast;  // every token of S_k has y >= y(bound)
      if (rs.bound > -INFINITY) theta = y_of(rs.bound, rs.m, rs.invT);
      if (q.p >= 1.0f) theta = fmaxf(theta, rs.L);
    } else if (rs.nallowed_sum <= kSmallRow) {
      plan = kPlanFast;  // few candidates: the row end sees all of them
      all = 1;
    } else if (q.mp > 0.0f) {
      plan = kPlanFast;  // K lies in {y >= ln min_p}
      theta = rs.L;
      needW = q.p < 1.0f;  // top-p renormalises over the whole row
    } else if (q.p >= 1.0f) {
      plan = kPlanUntrunc;  // K = every allowed token
    } else {
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

// Moves the row past phase `ph` (thread 0): the row's last listed phase resets its
// counter for the next call; otherwise the row state (plan kPlanDone when the row has
// ended) is published, then the phase number with release semantics.
__device__ void row_advance(const LaunchParams& P, int row, int ph, int nph, bool done) {
  if (threadIdx.x != 0) return;
  if (ph >= nph) {
    P.phase_done[row] = 0u;
    return;
  }
  if (done) sh.rs.plan = kPlanDone;
  P.rows[row] = sh.rs;
  __threadfence();
  st_release(P.phase_done + row, (unsigned)ph);
}

// ---------------------------------------------------------------- candidates and selects

// Appends (y, id) to a candidate array with a shared counter; the whole warp calls it.
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
// The same for one thread.
__device__ __forceinline__ void append1(Cand* cand, int cap, float y, int id) {
  const int p = atomicAdd(&sh.count, 1);
  if (p < cap) cand[p] = Cand{y, id};
}

// Radix select over a gathered set (entries with y >= ylo): the largest value v such
// that the count (or fixed-point weight) of entries >= v reaches `target`.
__device__ __noinline__ float local_select(int chunk, const Cand* G, int n, bool global, bool weighted, float ylo,
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
      const float y = ok ? ldcand(G, i, global).y : -INFINITY;
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

// Exact select over a gathered set, entries with y >= ylo, all within [lo, hi]: one
// 1024-bucket histogram (bucket order follows y), then the crossing bucket's entries are
// resolved by counting.  Falls back to local_select when that bucket holds more than
// 1024 entries (heavy ties).
__device__ __noinline__ float leader_select(int chunk, const Cand* G, int n, bool global, bool weighted, float lo,
                                            float hi, float ylo, unsigned long long target, bool* found) {
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
    const float y = ldcand(G, i, global).y;
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
    const Cand cd = ldcand(G, i, global);
    if (!(cd.y >= ylo) || bucket(cd.y) != bstar) continue;
    const int p = atomicAdd(&sh.nl, 1);
    if (p < 1024) Lb[p] = cd;
  }
  __syncthreads();
  const int nl = sh.nl;
  if (nl > 1024) {
    __syncthreads();
    return local_select(chunk, G, n, global, weighted, ylo, target, found);
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
__device__ __noinline__ Race leader_race(const Cand* G, int n, bool global, float cut, unsigned long long seed,
                                         unsigned long long pos) {
  Race r;
  r.init(sh.rs.s0);
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const Cand cd = ldcand(G, i, global);
    if (!(cd.y >= cut)) continue;
    r.add(cd.y, cd.id, pick_word(race_words_call((uint32_t)(cd.id >> 2), seed, pos), cd.id & 3));
  }
  block_reduce_race(r, sh.red_x);
  return r;
}

// Copies n candidates from the scratch into the gather area when they fit; returns the
// array the selects read and sets *global.
__device__ const Cand* gather_small(const Smem& S, const Cand* src, int n, bool* global) {
  if (n > kGatherCap) {
    *global = true;
    return src;
  }
  const float2* s = reinterpret_cast<const float2*>(src);
  float2* d = reinterpret_cast<float2*>(S.gather);
  for (int i = threadIdx.x; i < n; i += kThreads) d[i] = __ldcg(s + i);
  __syncthreads();
  *global = false;
  return S.gather;
}

// The per-slice segments of a later phase (counts in sh.x2), packed in slice order: into
// the gather area when they fit, else in place into the row's contiguous segments (each
// segment moves towards lower addresses, read whole first).
__device__ const Cand* collect_segments(const LaunchParams& P, const Smem& S, int row, int* n, bool* global) {
  const int tid = threadIdx.x, C = P.C;
  Cand* seg = P.cand + (size_t)row * C * kCandCap;
  int ntot = 0;
  for (int c = 0; c < C; ++c) ntot += sh.x2[c].count;
  *n = ntot;
  if (ntot <= kGatherCap) {
    int off = 0;
    for (int c = 0; c < C; ++c) {
      const int cnt = sh.x2[c].count;
      const float2* s = reinterpret_cast<const float2*>(seg + (size_t)c * kCandCap);
      float2* d = reinterpret_cast<float2*>(S.gather + off);
      for (int i = tid; i < cnt; i += kThreads) d[i] = __ldcg(s + i);
      off += cnt;
    }
    __syncthreads();
    *global = false;
    return S.gather;
  }
  int off = sh.x2[0].count;
  for (int c = 1; c < C; ++c) {
    const int cnt = sh.x2[c].count;
    float2 tmp[kCandCap / kThreads];
    const float2* s = reinterpret_cast<const float2*>(seg + (size_t)c * kCandCap);
#pragma unroll
    for (int t = 0; t < kCandCap / kThreads; ++t) {
      const int i = t * kThreads + tid;
      if (i < cnt) tmp[t] = __ldcg(s + i);
    }
    __syncthreads();
    float2* d = reinterpret_cast<float2*>(seg + off);
#pragma unroll
    for (int t = 0; t < kCandCap / kThreads; ++t) {
      const int i = t * kThreads + tid;
      if (i < cnt) d[i] = tmp[t];
    }
    __threadfence_block();
    __syncthreads();
    off += cnt;
  }
  *global = true;
  return seg;
}

// Top-k -> top-p -> min-p over the gathered candidates (an upper set of the row that
// holds every kept token; `Wrow` is the row's top-p mass when top-p renormalises over the
// whole row), then the race, then the outputs.  Thread 0 writes.
__device__ __noinline__ void leader_finish(const LaunchParams& P, int row, const Cand* G, int ntot, bool global,
                                           unsigned long long Wrow) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RowParams q = sh.rp;
  const float theta = sh.rs.theta, L = sh.rs.L, lnS = sh.rs.lnS;
  const bool kfin = q.k >= 2;
  // the bucket range: [theta, 0], or the gathered candidates' finite range
  float lo = theta;
  if (!(lo > -INFINITY)) {
    float ymin = INFINITY;
    for (int i = tid; i < ntot; i += kThreads) {
      const float y = ldcand(G, i, global).y;
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
    const float v = leader_select(P.chunk, G, ntot, global, false, lo, 0.0f, -INFINITY, (unsigned long long)q.k,
                                  &found);
    if (found) tk = v;
  }
  float tp = -INFINITY;
  if (q.p < 1.0f) {
    unsigned long long mset = 0;
    for (int i = tid; i < ntot; i += kThreads) {
      const float y = ldcand(G, i, global).y;
      if (y >= tk) mset += weight_fx(y);
    }
    mset = block_sum_u64(mset, sh.red_u);
    unsigned long long Wk = mset;  // top-k set (or every candidate) gathered: its mass
    if (!kfin && !sh.rs.all) Wk = Wrow;
    const unsigned long long cth = ceil_scaled(Wk, q.p);
    if (mset >= cth) {
      bool found;
      const float v = leader_select(P.chunk, G, ntot, global, true, lo, 0.0f, tk, cth, &found);
      if (found) tp = v;
    }
  }
  const float cut = fmaxf(tk, fmaxf(tp, L));
  const Race r = leader_race(G, ntot, global, cut, q.seed, q.pos);
  if (tid == 0) write_sampled(P.a, row, r, lnS, true);
}

// ---------------------------------------------------------------- re-reading a slice

// Slice state for a later pass over slice `slice`: the live bits (bitmask words clipped
// to the row, penalised tokens removed) and the first phase's list of penalised tokens
// with their final z'.  Needs sh.x1[slice].
template <bool kBF16>
__device__ __noinline__ void setup_re(const LaunchParams& P, int row, int slice) {
  const Geo g = geo<kBF16>(P, row, slice);
  const Smem S = carve(g.chunk);
  const clsample_args_t& a = P.a;
  const int tid = threadIdx.x;
  const int32_t* bmrow = a.bitmask ? a.bitmask + (long long)row * a.bitmask_row_stride : nullptr;
  const int npen = min(sh.x1[slice].npen, kPenCap);
  const uint2* pl = P.pen + ((size_t)row * P.C + slice) * kPenCap;
  __syncthreads();  // the previous user of these tables is done
  for (int w = tid; w < g.chunk / 32; w += kThreads) S.live[w] = mask_word(bmrow, g.c0, g.len, w);
  for (int r = tid; r < npen; r += kThreads) {
    const uint2 e = __ldcg(pl + r);
    S.pid[r] = (uint16_t)e.x;
    S.pz[r] = __uint_as_float(e.y);
  }
  __syncthreads();
  for (int r = tid; r < npen; r += kThreads) {
    const uint32_t l = S.pid[r];
    atomicAnd(&S.live[l >> 5], ~(1u << (l & 31)));
  }
  if (tid == 0) sh.npen = npen;
  __syncthreads();
}

// ---------------------------------------------------------------- fast rows at the row end

// Is local id l of slice s listed as penalised?  Binary search in the row end's copy of
// the slices' sorted id lists (r2).
__device__ __forceinline__ bool listed(const uint16_t* pids, int s, uint32_t l) {
  int lo = sh.poff[s], hi = sh.poff[s + 1];
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const uint32_t v = pids[mid];
    if (v == l) return true;
    if (v < l) lo = mid + 1;
    else hi = mid;
  }
  return false;
}

// Tokens of slice s's ring part (bulk); *len gets the slice's length.
template <bool kBF16>
__device__ __forceinline__ int bulk_of(const LaunchParams& P, int s, int* len) {
  constexpr int kEsize = kBF16 ? 2 : 4;
  const int c0 = s * P.chunk;
  *len = max(0, min(P.a.V, c0 + P.chunk) - c0);
  return P.vec_ok ? (int)(((size_t)*len * kEsize) & ~(size_t)15) / kEsize : 0;
}

// Shared-memory areas of the row end (the ring and the r2 tables are free).
constexpr int kHitList = 4096;                 // hit codes (u32) then their entries (u16)
constexpr int kCandSmem = (kStages * kStageBytes - kHitList * 6) / (int)sizeof(Cand);
constexpr int kPidsBytes = kPenCap * kMaxSlices * (int)sizeof(uint16_t);
static_assert(kCandSmem >= 1024, "row-end candidate area");
static_assert(kPidsBytes + 256 * (int)sizeof(uint32_t) <= (int)kR2Bytes, "row-end r2 tables");

// Appends (y, id) to the candidates: the shared copy while it fits, and the row's
// segments in the scratch; the whole warp calls it.
__device__ __forceinline__ void append2(Cand* sm, int smcap, Cand* gl, int glcap, bool keep, float y, int id) {
  const int lane = threadIdx.x & 31;
  const uint32_t bal = __ballot_sync(0xffffffffu, keep);
  if (!bal) return;
  const int leader = __ffs(bal) - 1;
  int basepos = 0;
  if (lane == leader) basepos = atomicAdd(&sh.count, __popc(bal));
  basepos = __shfl_sync(0xffffffffu, basepos, leader);
  if (keep) {
    const int p = basepos + __popc(bal & ((1u << lane) - 1u));
    if (p < smcap) sm[p] = Cand{y, id};
    if (p < glcap) gl[p] = Cand{y, id};
  }
}
__device__ __forceinline__ void append2_1(Cand* sm, int smcap, Cand* gl, int glcap, float y, int id) {
  const int p = atomicAdd(&sh.count, 1);
  if (p < smcap) sm[p] = Cand{y, id};
  if (p < glcap) gl[p] = Cand{y, id};
}


// A bound E on the table entries (at least k groups reach E, so the k-th largest z' is
// at least key^-1(E << 16)) in the y order the cuts use: y = fl(fl(z - m) (1/T)) can
// merge neighbouring z, so the tokens kept by top-k are those with z at or above the
// smallest z whose y reaches y(key^-1(E << 16)).  Warp 0 computes it into sh.res; every
// thread returns it after the barrier.
__device__ float entry_bound_z(uint32_t E, float m, float invT) {
  if (threadIdx.x < 32) {
    const float ye = y_of(key_to_float(E << 16), m, invT);
    const float zt = z_threshold_warp(fminf(ye, 0.0f), m, invT);
    if (threadIdx.x == 0) sh.res = zt;
  }
  __syncthreads();
  const float r = sh.res;
  __syncthreads();
  return r;
}

// The fallback of fast_serial (unaligned rows, tables too large for shared memory, too
// many listed groups, a table copy that never landed): every slice is re-read whole and
// its tokens with z >= zth (the exact z image of theta) are compacted, listed penalised
// tokens by their z'.  Then top-k -> top-p -> min-p and the race.  Returns false when
// the candidates overflow the row's segments.
template <bool kBF16>
__device__ __noinline__ bool fast_serial_global(const LaunchParams& P, int row) {
  const Smem S = carve(P.chunk);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = P.C;
  const float m = sh.rs.m, invT = sh.rs.invT, theta = sh.rs.theta;
  const int cap = C * kCandCap;
  Cand* seg = P.cand + (size_t)row * C * kCandCap;
  __syncthreads();
  if (warp == 0) {
    const float zt = z_threshold_warp(theta, m, invT);
    if (lane == 0) {
      sh.zth = zt;
      sh.count = 0;
    }
  }
  __syncthreads();
  const float zth = sh.zth;
#pragma unroll 1
  for (int s = 0; s < C; ++s) {
    setup_re<kBF16>(P, row, s);
    const Geo g = geo<kBF16>(P, row, s);
    stream_ldg<kBF16>(g, S, [&](int f, uint32_t wd, const float4& v) {
      float z[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) z[j] = ((wd >> j) & 1u) ? sanitize(comp(v, j)) : -INFINITY;
      const bool any = __any_sync(0xffffffffu, z[0] >= zth || z[1] >= zth || z[2] >= zth || z[3] >= zth);
      if (any) {
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          const bool keep = z[j] > -INFINITY && z[j] >= zth;
          append(seg, cap, keep, keep ? y_of(z[j], m, invT) : 0.0f, g.c0 + 4 * f + j);
        }
      }
    });
    for (int r = tid; r < sh.npen; r += kThreads) {
      const float z = S.pz[r];
      if (z > -INFINITY && z >= zth) append1(seg, cap, y_of(z, m, invT), g.c0 + (int)S.pid[r]);
    }
  }
  __threadfence_block();
  __syncthreads();
  const int n = sh.count;
  if (n > cap) return false;
  bool global;
  const Cand* G = gather_small(S, seg, n, &global);
  leader_finish(P, row, G, n, global, 0ull);
  return true;
}




// The row end's bulk copies of every slice's table into shared memory [0, C * tabstride),
// on the row end's barrier (thread 0).  The tables are other CTAs' ordinary stores
// (acquired through the ticket), read here by the async proxy: the proxy fence orders
// them (global and shared state spaces).
template <bool kBF16>
__device__ void tables_issue(const LaunchParams& P, int row) {
  constexpr int kEsize = kBF16 ? 2 : 4;
  const int C = P.C;
  const int nst_max = (int)(((size_t)P.chunk * kEsize + kStageBytes - 1) / kStageBytes);
  const int tabstride = nst_max * kThreads * (int)sizeof(uint16_t);
  asm volatile("fence.proxy.async;" ::: "memory");
  uint32_t bytes = 0;
  for (int s = 0; s < C; ++s) {
    const int c0 = s * P.chunk;
    const int len = max(0, min(P.a.V, c0 + P.chunk) - c0);
    const int bulk = P.vec_ok ? (int)(((size_t)len * kEsize) & ~(size_t)15) : 0;
    bytes += (uint32_t)((bulk + kStageBytes - 1) / kStageBytes * kThreads * 2);
  }
  mbar_arrive_expect_tx(&sh.tbar, bytes);
  for (int s = 0; s < C; ++s) {
    const int c0 = s * P.chunk;
    const int len = max(0, min(P.a.V, c0 + P.chunk) - c0);
    const int bulk = P.vec_ok ? (int)(((size_t)len * kEsize) & ~(size_t)15) : 0;
    const uint32_t b = (uint32_t)((bulk + kStageBytes - 1) / kStageBytes * kThreads * 2);
    if (b) bulk_copy_g2s(smem_dyn + (size_t)s * tabstride, P.tab + ((size_t)row * C + s) * kTabMax, b, &sh.tbar);
  }
  sh.tissued = 1;
}

// Waits for the table copies (thread 0, bounded) and moves the barrier to its next phase;
// returns false in every thread if they never landed.  Every thread calls it.
__device__ bool tables_wait() {
  if (threadIdx.x == 0 && !mbar_wait_sleep(&sh.tbar, sh.tpar)) sh.tfail = 1;
  __syncthreads();
  (void)mbar_try_wait(&sh.tbar, sh.tpar);
  const bool ok = !sh.tfail;
  __syncthreads();
  if (threadIdx.x == 0) {
    sh.tpar ^= 1u;
    sh.tissued = 0;
    sh.tfail = 0;
  }
  return ok;
}

// Whether a row's first-phase end is certain to gather candidates from the tables: top-k
// rows whose parameters are valid (their data can still end them early).
__device__ __forceinline__ bool tables_likely(const RowParams& q) {
  return !q.invalid && !params_greedy(q) && q.k >= 2;
}

// Candidates of a fast row (every token with z >= zth, the exact z image of theta, that
// can be kept), found by the CTA that ends the row's first phase:
//  1. one bulk copy (TMA) brings every slice's table of group maxima into shared memory
//     while the threads load the slices' listed penalised tokens (candidates by their
//     z') and ragged tails;
//  2. for a top-k row, a binary search over the table entries finds the largest E with
//     at least k entries >= E (at least k groups, hence k tokens, reach E, so every token
//     of the top-k set lies in a group whose entry reaches E); the groups whose entry
//     reaches the threshold are listed in table order by a block scan;
//  3. the listed groups' vectors are re-read from L2 with their bitmask words.
// Then top-k -> top-p -> min-p and the race.  Rows whose tables do not fit in shared
// memory take fast_serial_global.  Returns false when the candidates overflow the row's
// segments.
template <bool kBF16>
__device__ __noinline__ bool fast_serial(const LaunchParams& P, int row) {
  constexpr int kEsize = kBF16 ? 2 : 4;
  constexpr int kVecPerStage = kStageBytes / (4 * kEsize);
  constexpr int kVPT = kVecPerStage / kThreads;
  const Smem S = carve(P.chunk);
  const Layout Lo = layout_for(P.chunk);
  const clsample_args_t& a = P.a;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = P.C, chunk = P.chunk;
  const int nst_max = (int)(((size_t)chunk * kEsize + kStageBytes - 1) / kStageBytes);
  const int tabstride = nst_max * kThreads * (int)sizeof(uint16_t);  // bytes per slice
  const int tabbytes = C * tabstride;
  const int hitcap = ((int)Lo.r2 - tabbytes) / 4;
  if (!P.vec_ok || hitcap < kWarps * 128) {
    if (sh.tissued) (void)tables_wait();
    return fast_serial_global<kBF16>(P, row);
  }
  const RowParams q = sh.rp;
  const bool kfin = q.k >= 2;
  const float m = sh.rs.m, invT = sh.rs.invT, theta = sh.rs.theta;
  const int cap = C * kCandCap;
  const int csmcap = tabbytes / (int)sizeof(Cand);
  Cand* seg = P.cand + (size_t)row * C * kCandCap;
  unsigned char* tabs = smem_dyn;                                  // [0, tabbytes)
  uint32_t* hits = reinterpret_cast<uint32_t*>(smem_dyn + tabbytes);  // [tabbytes, r2)
  Cand* csm = reinterpret_cast<Cand*>(smem_dyn);                   // after the tables are done
  uint16_t* pids = reinterpret_cast<uint16_t*>(S.r2);
  const int32_t* bmrow = a.bitmask ? a.bitmask + (long long)row * a.bitmask_row_stride : nullptr;
  const unsigned char* lrow =
      reinterpret_cast<const unsigned char*>(a.logits) + (long long)row * a.logits_row_stride * kEsize;
  if (tid == 0) {
    if (!sh.tissued) tables_issue<kBF16>(P, row);
    sh.count = 0;
    int o = 0;
    for (int s = 0; s < C; ++s) {
      sh.poff[s] = o;
      o += min(sh.x1[s].npen, kPenCap);
    }
    sh.poff[C] = o;
  }
  if (warp == 1) {
    const float zt = z_threshold_warp(theta, m, invT);
    if (lane == 0) sh.zth = zt;
  }
  // this thread's tail token (threads < 8 C)
  float tz = -INFINITY;
  int tgi = -1;
  if (tid < C * 8) {
    const int s = tid >> 3;
    int len;
    const int l = bulk_of<kBF16>(P, s, &len) + (tid & 7);
    if (l < len) {
      const int gi = s * chunk + l;
      const bool allowed = !bmrow || (((uint32_t)__ldg(bmrow + (gi >> 5)) >> (gi & 31)) & 1u);
      tgi = gi;
      tz = allowed ? sanitize(gload1<kBF16>(lrow, gi)) : -INFINITY;
    }
  }
  __syncthreads();
  const float zth = sh.zth;
  // listed penalised tokens: ids for the check below, candidates by their z' (the
  // candidates go to the row's segments only until the tables are done)
  {
    const int npen_all = sh.poff[C];
    for (int base = 0; base < npen_all; base += 4 * kThreads) {
      uint2 e[4];
      int si[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = base + u * kThreads + tid;
        int s = 0;
        while (s + 1 < C && sh.poff[s + 1] <= i) ++s;
        si[u] = s;
        e[u] = i < npen_all ? __ldcg(P.pen + ((size_t)row * C + s) * kPenCap + (i - sh.poff[s])) : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = base + u * kThreads + tid;
        if (i >= npen_all) continue;
        pids[i] = (uint16_t)e[u].x;
        const float z = __uint_as_float(e[u].y);
        if (z > -INFINITY && z >= zth) append1(seg, cap, y_of(z, m, invT), si[u] * chunk + (int)e[u].x);
      }
    }
    __threadfence();  // read back below by other threads of the CTA
  }
  // the tables
  const bool tok = tables_wait();
  const int nch = tabbytes / 16;
  const uint4* t4 = reinterpret_cast<const uint4*>(tabs);
  float zcut = zth;  // candidates: z >= zcut (tightened for top-k rows below)
  uint32_t thr = tab_threshold(zth);
  if (kfin && tok) {
    // the k-th largest entry: per-warp histograms of the entries at or above thr (two
    // 16-bit counters a word, in the free area after the tables), merged per bin
    const uint32_t top = fkey(m) >> 16;
    int shift = 0;
    while (((top - min(top, thr)) >> shift) >= 256u) ++shift;
    uint32_t* wh = hits;  // kWarps x 128 words
    uint32_t* bins = reinterpret_cast<uint32_t*>(S.r2 + kPidsBytes);
    for (int i = tid; i < kWarps * 128; i += kThreads) wh[i] = 0u;
    __syncthreads();
    uint32_t* mine = wh + warp * 128;
    for (int i = tid; i < nch; i += kThreads) {
      const uint4 e = t4[i];
      const uint32_t w4[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t ent = (w4[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
        if (ent >= thr) {
          const uint32_t bin = min((ent - thr) >> shift, 255u);
          atomicAdd(&mine[bin >> 1], 1u << (16 * (bin & 1)));
        }
      }
    }
    __syncthreads();
    {
      uint32_t t = 0;
      for (int w = 0; w < kWarps; ++w) t += (wh[w * 128 + (tid >> 1)] >> (16 * (tid & 1))) & 0xFFFFu;
      bins[tid] = t;
    }
    __syncthreads();
    if (warp == 0) pick_digit(bins, (unsigned long long)q.k, &sh.digit, &sh.above, &sh.none);
    __syncthreads();
    if (!sh.none) {
      zcut = fmaxf(zth, entry_bound_z(thr + ((uint32_t)sh.digit << shift), m, invT));
      thr = tab_threshold(zcut);
    }
  }
  // the groups at or above the threshold, in table order
  int nh;
  {
    int c = 0;
    for (int i = tid; i < nch; i += kThreads) {
      const uint4 e = t4[i];
      const uint32_t w4[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) c += ((w4[j] & 0xFFFFu) >= thr) + ((w4[j] >> 16) >= thr);
    }
    int x = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += o;
    }
    __syncthreads();
    if (lane == 31) sh.red_i[warp] = x;
    __syncthreads();
    int pos = x - c;
    nh = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) pos += sh.red_i[w];
      nh += sh.red_i[w];
    }
    if (nh <= hitcap) {
      for (int i = tid; i < nch; i += kThreads) {
        const uint4 e = t4[i];
        const uint32_t w4[4] = {e.x, e.y, e.z, e.w};
        const int s = (i * 16) / tabstride, e0 = (i * 16 - s * tabstride) / 2;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t ent = (w4[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
          if (ent >= thr) hits[pos++] = ((uint32_t)s << 16) | (uint32_t)(e0 + j);
        }
      }
    }
  }
  __syncthreads();  // the tables are done: the candidate area is free
  if (nh > hitcap || !tok) return fast_serial_global<kBF16>(P, row);
  // the candidates found so far (listed penalised tokens) into the shared copy
  {
    const int n0 = sh.count;
    for (int i = tid; i < min(n0, csmcap); i += kThreads) {
      const float2 v = __ldcg(reinterpret_cast<const float2*>(seg) + i);
      csm[i] = Cand{v.x, __float_as_int(v.y)};
    }
  }
  if (tgi >= 0 && tz > -INFINITY && tz >= zth && !listed(pids, tgi / chunk, (uint32_t)(tgi % chunk)))
    append2_1(csm, csmcap, seg, cap, y_of(tz, m, invT), tgi);
  // the listed groups' vectors with their bitmask words
  constexpr int kHitBatch = 1;
#pragma unroll 1
  for (int h0 = 0; h0 < nh; h0 += kHitBatch * kThreads) {
    float4 v[kHitBatch][kVPT];
    uint32_t mw[kHitBatch][kVPT];
    int hs[kHitBatch], hf[kHitBatch];
#pragma unroll
    for (int b = 0; b < kHitBatch; ++b) {
      const int h = h0 + b * kThreads + tid;
      const bool valid = h < nh;
      const uint32_t code = valid ? hits[h] : 0u;
      const int s = (int)(code >> 16), e = (int)(code & 0xFFFFu);
      const int k = e / kThreads, tt = e % kThreads;
      const int c0s = s * chunk;
      int len;
      const int bulk = bulk_of<kBF16>(P, s, &len);
      hs[b] = s;
      hf[b] = k * kVecPerStage + tt;
#pragma unroll
      for (int u = 0; u < kVPT; ++u) {
        const int f = hf[b] + u * kThreads;
        const bool in = valid && 4 * f < bulk;
        v[b][u] = in ? vload4<kBF16>(lrow + (size_t)c0s * kEsize, f) : make_float4(0.f, 0.f, 0.f, 0.f);
        mw[b][u] = in ? ((bmrow ? (uint32_t)__ldg(bmrow + ((c0s + 4 * f) >> 5)) : 0xFFFFFFFFu) >> ((4 * f) & 31)) & 0xFu
                      : 0u;
      }
    }
#pragma unroll
    for (int b = 0; b < kHitBatch; ++b) {
#pragma unroll
      for (int u = 0; u < kVPT; ++u) {
        const int f = hf[b] + u * kThreads;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          bool keep = false;
          float z = -INFINITY;
          if ((mw[b][u] >> j) & 1u) {
            z = sanitize(comp(v[b][u], j));
            keep = z > -INFINITY && z >= zcut && !listed(pids, hs[b], (uint32_t)(4 * f + j));
          }
          append2(csm, csmcap, seg, cap, keep, keep ? y_of(z, m, invT) : 0.0f, hs[b] * chunk + 4 * f + j);
        }
      }
    }
  }
  __threadfence_block();
  __syncthreads();
  const int n = sh.count;
  if (n > cap) return false;
  const bool global = n > csmcap;
  leader_finish(P, row, global ? seg : csm, n, global, 0ull);
  return true;
}

// ---------------------------------------------------------------- later phases: slice passes

// Top-p alone, phase 2: the exact top-p mass of the slice and its histogram over
// quarter-unit y bins (warp-private split counters in r2, the open-ended last bin in
// registers), merged per bin into the slice's row of the scratch.
template <bool kBF16>
__device__ __noinline__ void topp_hist(const LaunchParams& P, int row, int slice) {
  const Geo g = geo<kBF16>(P, row, slice);
  const Smem S = carve(g.chunk);
  const int tid = threadIdx.x, warp = tid >> 5;
  const float m = sh.rs.m, invT = sh.rs.invT;
  const size_t idx = (size_t)row * P.C + slice;
  // warp-private split counters (two u32 per bin): a warp adds at most 4160 weights
  uint32_t* whist = reinterpret_cast<uint32_t*>(S.r2);
  for (int i = tid; i < 2 * kWarps * kPBins; i += kThreads) whist[i] = 0u;
  __syncthreads();
  unsigned long long w = 0, wlast = 0;
  uint32_t* mine = whist + 2 * warp * kPBins;
  stream_phase<kBF16>(g, S, [&](int f, uint32_t wd, const float4& v) {
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
  for (int i = tid; i < sh.npen; i += kThreads) {
    const float z = S.pz[i];
    if (!(z > -INFINITY)) continue;
    const float y = y_of(z, m, invT);
    const unsigned long long qw = weight_fx(y);
    if (!qw) continue;
    w += qw;
    split_add(mine + 2 * pbin(y), qw);
  }
  {
    const unsigned long long wl = warp_sum_u64(wlast);  // < 2^53: split_add holds it
    if ((tid & 31) == 0 && wl) split_add(mine + 2 * (kPBins - 1), wl);
  }
  w = block_sum_u64(w, sh.red_u);
  if (tid < kPBins) {
    unsigned long long t = 0;
    for (int wp = 0; wp < kWarps; ++wp) t += split_get(whist + 2 * (wp * kPBins + tid));
    P.phist[idx * kPBins + tid] = t;
  }
  if (tid == 0) {
    Race none;
    none.init();
    none.to(sh.x2_mine);
    sh.x2_mine.count = 0;
    sh.x2_mine.flags = 0;
    sh.x2_mine.w = w;
  }
}

// Top-p alone, phase 3: tokens above the crossing bin are certainly kept: raced here;
// tokens of the crossing bin go to the slice's candidate segment for the row end.
template <bool kBF16>
__device__ __noinline__ void topp_race(const LaunchParams& P, int row, int slice) {
  const Geo g = geo<kBF16>(P, row, slice);
  const Smem S = carve(g.chunk);
  const int tid = threadIdx.x;
  const RowParams q = sh.rp;
  const float m = sh.rs.m, invT = sh.rs.invT;
  const unsigned long long seed = q.seed, pos = q.pos;
  const int c0 = g.c0, cap = kCandCap;
  Cand* mycand = P.cand + ((size_t)row * P.C + slice) * kCandCap;
  const int bstar = sh.rs.bstar;
  const float yhi = -(float)bstar * 0.25f, ylo = -(float)(bstar + 1) * 0.25f;
  if (tid == 0) sh.count = 0;
  __syncthreads();
  Race race;
  race.init(sh.rs.s0);
  stream_phase<kBF16>(g, S, [&](int f, uint32_t wd, const float4& v) {
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
  {
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
  __syncthreads();
  if (tid == 0) {
    race.to(sh.x2_mine);
    sh.x2_mine.count = sh.count;
    sh.x2_mine.flags = sh.count > cap ? kFlagOverflow : 0;
    sh.x2_mine.w = 0ull;
  }
}

// Min-p with top-p over the whole row, phase 2: the slice's exact top-p mass and its
// tokens with z >= zth (the exact z image of ln min_p) into the slice's segment.
template <bool kBF16>
__device__ __noinline__ void minp_pass(const LaunchParams& P, int row, int slice) {
  const Geo g = geo<kBF16>(P, row, slice);
  const Smem S = carve(g.chunk);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float m = sh.rs.m, invT = sh.rs.invT, theta = sh.rs.theta;
  const int c0 = g.c0, cap = kCandCap;
  Cand* mycand = P.cand + ((size_t)row * P.C + slice) * kCandCap;
  if (warp == 0) {
    const float zt = z_threshold_warp(theta, m, invT);
    if (lane == 0) {
      sh.zth = zt;
      sh.count = 0;
    }
  }
  __syncthreads();
  const float zth = sh.zth;
  unsigned long long w = 0;
  stream_phase<kBF16>(g, S, [&](int f, uint32_t wd, const float4& v) {
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
#pragma unroll 1
      for (int j = 0; j < 4; ++j)
        if (z[j] > -INFINITY) w += weight_fx(y_of(z[j], m, invT));
    }
    const bool any = __any_sync(0xffffffffu, z[0] >= zth || z[1] >= zth || z[2] >= zth || z[3] >= zth);
    if (any) {
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        const bool keep = z[j] > -INFINITY && z[j] >= zth;
        append(mycand, cap, keep, keep ? y_of(z[j], m, invT) : 0.0f, c0 + 4 * f + j);
      }
    }
  });
  {
    const int npen = sh.npen;
    for (int base = 0; base < npen; base += kThreads) {
      const int i = base + tid;
      const float z = i < npen ? S.pz[i] : -INFINITY;
      const int gi = c0 + (i < npen ? (int)S.pid[i] : 0);
      const float y = z > -INFINITY ? y_of(z, m, invT) : -INFINITY;
      if (z > -INFINITY) w += weight_fx(y);
      append(mycand, cap, z > -INFINITY && z >= zth, y, gi);
    }
  }
  w = block_sum_u64(w, sh.red_u);
  if (tid == 0) {
    Race none;
    none.init();
    none.to(sh.x2_mine);
    sh.x2_mine.count = sh.count;
    sh.x2_mine.flags = sh.count > cap ? kFlagOverflow : 0;
    sh.x2_mine.w = w;
  }
}

// No truncation, phase 2: the race over every allowed token of the slice.  A vector
// whose every y is kGumbelMax below the best score so far cannot win and skips Philox.
template <bool kBF16>
__device__ __noinline__ void untrunc_pass(const LaunchParams& P, int row, int slice) {
  const Geo g = geo<kBF16>(P, row, slice);
  const Smem S = carve(g.chunk);
  const int tid = threadIdx.x;
  const RowParams q = sh.rp;
  const float m = sh.rs.m, invT = sh.rs.invT;
  const unsigned long long seed = q.seed, pos = q.pos;
  const int c0 = g.c0;
  Race race;
  race.init(sh.rs.s0);
  stream_phase<kBF16>(g, S, [&](int f, uint32_t wd, const float4& v) {
    if (!wd) return;
    float y[4];
    bool live_any = false, worth = false;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float z = ((wd >> j) & 1u) ? sanitize(comp(v, j)) : -INFINITY;
      y[j] = z > -INFINITY ? y_of(z, m, invT) : -INFINITY;
      if (z > -INFINITY) {
        live_any = true;
        worth |= y[j] + kGumbelMax >= race.s;
      }
    }
    if (worth) {
      const uint4 x = race_words((uint32_t)((c0 >> 2) + f), seed, pos);
#pragma unroll 1
      for (int j = 0; j < 4; ++j)
        if (y[j] > -INFINITY) race.add(y[j], c0 + 4 * f + j, pick_word(x, j));
    } else if (live_any) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (y[j] > -INFINITY) race.count_only(y[j]);
    }
  });
  for (int i = tid; i < sh.npen; i += kThreads) {
    const float z = S.pz[i];
    if (!(z > -INFINITY)) continue;
    const float y = y_of(z, m, invT);
    const int gi = c0 + (int)S.pid[i];
    race.add(y, gi, pick_word(race_words_call((uint32_t)(gi >> 2), seed, pos), gi & 3));
  }
  block_reduce_race(race, sh.red_x);
  __syncthreads();
  if (tid == 0) {
    race.to(sh.x2_mine);
    sh.x2_mine.count = 0;
    sh.x2_mine.flags = 0;
    sh.x2_mine.w = 0ull;
  }
}

// ---------------------------------------------------------------- rows without a usable bound

// Exact radix select over the whole row by one CTA (one pass over every slice per 8-bit
// digit): the largest value v such that the count (or fixed-point weight) of tokens with
// y >= v reaches `target`, among tokens with y >= ylo.  Needs sh.x1 of every slice.
template <bool kBF16>
__device__ __noinline__ float row_select(const LaunchParams& P, int row, bool weighted, float ylo,
                                         unsigned long long target, bool* found) {
  const Smem S = carve(P.chunk);
  const int tid = threadIdx.x, warp = tid >> 5;
  const float m = sh.rs.m, invT = sh.rs.invT;
  uint32_t prefix = 0u, pmask = 0u;
  for (int dpass = 0; dpass < 4; ++dpass) {
    const int shift = 24 - 8 * dpass;
    if (tid < 256) {
      S.hist_c[tid] = 0u;
      S.hist_w[tid] = 0ull;
    }
    for (int s = 0; s < P.C; ++s) {
      setup_re<kBF16>(P, row, s);
      const Geo g = geo<kBF16>(P, row, s);
      auto add = [&](bool live, float z) {
        bool pred = false;
        float y = -INFINITY;
        if (live && z > -INFINITY) {
          y = y_of(z, m, invT);
          pred = y >= ylo && (fkey(y) & pmask) == prefix;
        }
        const uint32_t digit = (fkey(y) >> shift) & 0xFFu;
        if (weighted) hist_add<true>(S.hist_c, S.hist_w, pred, digit, pred ? weight_fx(y) : 0ull);
        else hist_add<false>(S.hist_c, S.hist_w, pred, digit, 0ull);
      };
      stream_ldg<kBF16>(g, S, [&](int f, uint32_t wd, const float4& v) {
#pragma unroll 1
        for (int j = 0; j < 4; ++j) add(((wd >> j) & 1u) != 0u, sanitize(comp(v, j)));
      });
      const int npen = sh.npen;
      for (int base = 0; base < npen; base += kThreads) {
        const int i = base + tid;
        add(i < npen, i < npen ? S.pz[i] : -INFINITY);
      }
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

// Rows without a usable bound (very large k, candidate overflow, top-p with an
// open-ended crossing bin): exact selects over the whole row, then the race, all by the
// calling CTA.  Slow, and rare.  Needs sh.x1 of every slice.
template <bool kBF16>
__device__ __noinline__ void slow_serial(const LaunchParams& P, int row) {
  const Smem S = carve(P.chunk);
  const int tid = threadIdx.x;
  const RowParams q = sh.rp;
  const float m = sh.rs.m, invT = sh.rs.invT, lnS = sh.rs.lnS, L = sh.rs.L;
  const bool kfin = q.k >= 2;
  float tk = -INFINITY;
  if (kfin) {
    bool found;
    const float v = row_select<kBF16>(P, row, false, -INFINITY, (unsigned long long)q.k, &found);
    if (found) tk = v;  // fewer than k candidates: top-k keeps them all
  }
  float tp = -INFINITY;
  if (q.p < 1.0f) {
    unsigned long long w = 0;
    for (int s = 0; s < P.C; ++s) {
      setup_re<kBF16>(P, row, s);
      const Geo g = geo<kBF16>(P, row, s);
      stream_ldg<kBF16>(g, S, [&](int f, uint32_t wd, const float4& v) {
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          if (!((wd >> j) & 1u)) continue;
          const float z = sanitize(comp(v, j));
          if (!(z > -INFINITY)) continue;
          const float y = y_of(z, m, invT);
          if (y >= tk) w += weight_fx(y);
        }
      });
      for (int i = tid; i < sh.npen; i += kThreads) {
        const float z = S.pz[i];
        if (!(z > -INFINITY)) continue;
        const float y = y_of(z, m, invT);
        if (y >= tk) w += weight_fx(y);
      }
    }
    w = block_sum_u64(w, sh.red_u);
    bool found;
    const float v = row_select<kBF16>(P, row, true, tk, ceil_scaled(w, q.p), &found);
    if (found) tp = v;
  }
  const float cut = fmaxf(tk, fmaxf(tp, L));
  Race race;
  race.init(sh.rs.s0);
  for (int s = 0; s < P.C; ++s) {
    setup_re<kBF16>(P, row, s);
    const Geo g = geo<kBF16>(P, row, s);
    const int c0 = g.c0;
    stream_ldg<kBF16>(g, S, [&](int f, uint32_t wd, const float4& v) {
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
      const uint4 x = race_words((uint32_t)((c0 >> 2) + f), q.seed, q.pos);
#pragma unroll 1
      for (int j = 0; j < 4; ++j)
        if ((keep >> j) & 1u) race.add(y[j], c0 + 4 * f + j, pick_word(x, j));
    });
    for (int i = tid; i < sh.npen; i += kThreads) {
      const float z = S.pz[i];
      if (!(z > -INFINITY)) continue;
      const float y = y_of(z, m, invT);
      if (!(y >= cut)) continue;
      const int gi = c0 + (int)S.pid[i];
      race.add(y, gi, pick_word(race_words_call((uint32_t)(gi >> 2), q.seed, q.pos), gi & 3));
    }
  }
  block_reduce_race(race, sh.red_x);
  if (tid == 0) write_sampled(P.a, row, race, lnS, true);
  __syncthreads();
}

// ---------------------------------------------------------------- items

// A first-phase item; the CTA that finishes the row's last slice ends the row or hands
// it to the next phase.
template <bool kBF16>
__device__ __noinline__ void p1_item(const LaunchParams& P, int row, int slice, int nph) {
  setup_p1<kBF16>(P, row, slice, nph);
  pass_a<kBF16>(P, row, slice);
  if (!publish_p1<kBF16>(P, row, slice)) return;
  // a top-k row's end reads every table: their copies start before anything else
  if (threadIdx.x == 0 && tables_likely(sh.rp)) tables_issue<kBF16>(P, row);
  combine_row(P, row);
  if (finish_early(P, row)) {
    if (sh.tissued) (void)tables_wait();
    row_advance(P, row, 1, nph, true);
    return;
  }
  plan_row();
  const int plan = sh.rs.plan;
  if (plan == kPlanFast && !sh.rs.needW) {
    if (!fast_serial<kBF16>(P, row)) slow_serial<kBF16>(P, row);
    row_advance(P, row, 1, nph, true);
    return;
  }
  if (sh.tissued) (void)tables_wait();
  const int need = plan == kPlanTopP ? 3 : 2;  // phases the plan takes
  if (plan == kPlanSlow || nph < need) {
    slow_serial<kBF16>(P, row);
    row_advance(P, row, 1, nph, true);
    return;
  }
  row_advance(P, row, 1, nph, false);
}

// The last arriver of a later phase.  `what` is the pass the phase ran (0: none).
template <bool kBF16>
__device__ __noinline__ void phase_end(const LaunchParams& P, int row, int ph, int nph, int what) {
  const Smem S = carve(P.chunk);
  const int tid = threadIdx.x, C = P.C;
  const RowParams q = sh.rp;
  const bool bad = __ldcg(P.bad + row) != 0u;
  if (bad || !sh.ok) {
    // a wait gave up: the row's records are incomplete
    if (tid == 0 && !(sh.ok && sh.rs.plan == kPlanDone)) {
      Race r;
      r.init();
      write_sampled(P.a, row, r, 0.0f, false);
    }
    row_advance(P, row, ph, nph, true);
    return;
  }
  if (what == 0) {
    if (sh.rs.plan != kPlanDone) slow_serial<kBF16>(P, row);  // a plan without this phase: not reached
    row_advance(P, row, ph, nph, true);
    return;
  }
  int fl = 0;
  for (int c = 0; c < C; ++c) fl |= sh.x2[c].flags;
  if (what == 1) {
    // top-p alone: the crossing bin, where the running mass from the top first reaches
    // ceil(p W)
    unsigned long long W = 0;
    for (int c = 0; c < C; ++c) W += sh.x2[c].w;
    const unsigned long long cth = ceil_scaled(W, q.p);
    if (tid < kPBins) {
      unsigned long long t = 0;
      for (int c = 0; c < C; ++c) t += __ldcg(P.phist + ((size_t)row * C + c) * kPBins + tid);
      S.hist_w[tid] = t;
    }
    __syncthreads();
    if (tid == 0) {
      int bstar = kPBins - 1;
      unsigned long long above = 0, cum = 0;
      for (int b = 0; b < kPBins; ++b) {
        const unsigned long long nb = cum + S.hist_w[b];
        if (nb >= cth) {
          bstar = b;
          above = cum;
          break;
        }
        cum = nb;
      }
      sh.rs.bstar = bstar;
      sh.rs.above = above;
      sh.rs.cth = cth;
    }
    __syncthreads();
    if (sh.rs.bstar >= kPBins - 1) {
      slow_serial<kBF16>(P, row);
      row_advance(P, row, ph, nph, true);
    } else {
      row_advance(P, row, ph, nph, false);
    }
    return;
  }
  if (what == 4) {
    if (tid == 0) {
      Race r;
      r.init();
      for (int c = 0; c < C; ++c) r.merge(sh.x2[c]);
      write_sampled(P.a, row, r, sh.rs.lnS, true);
    }
    row_advance(P, row, ph, nph, true);
    return;
  }
  if (fl & kFlagOverflow) {
    slow_serial<kBF16>(P, row);
    row_advance(P, row, ph, nph, true);
    return;
  }
  int ntot = 0;
  bool global = false;
  const Cand* G = collect_segments(P, S, row, &ntot, &global);
  if (what == 2) {
    // top-p alone: the cut lies in the crossing bin: a weighted select over its tokens
    const int bstar = sh.rs.bstar;
    const float yhi = -(float)bstar * 0.25f, ylo = -(float)(bstar + 1) * 0.25f;
    bool found;
    const float vstar =
        leader_select(P.chunk, G, ntot, global, true, ylo, yhi, -INFINITY, sh.rs.cth - sh.rs.above, &found);
    Race r = leader_race(G, ntot, global, vstar, q.seed, q.pos);
    if (tid == 0) {
      for (int c = 0; c < C; ++c) r.merge(sh.x2[c]);
      write_sampled(P.a, row, r, sh.rs.lnS, found);
    }
  } else {
    unsigned long long W = 0;
    for (int c = 0; c < C; ++c) W += sh.x2[c].w;
    leader_finish(P, row, G, ntot, global, W);
  }
  row_advance(P, row, ph, nph, true);
}

// An item of a later phase: waits (bounded) until the row's previous phase is complete,
// runs the phase's pass over its slice, publishes the slice record and takes the ticket.
template <bool kBF16>
__device__ __noinline__ void phase_item(const LaunchParams& P, int row, int slice, int ph, int nph) {
  const int tid = threadIdx.x, C = P.C;
  const size_t idx = (size_t)row * C + slice;
  if (tid == 0) {
    unsigned v = ld_acquire(P.phase_done + row);
    for (uint32_t i = 0; v < (unsigned)(ph - 1) && i < kWaitLimit; ++i) {
      __nanosleep(i < 64u ? 100u : 1000u);
      v = ld_acquire(P.phase_done + row);
    }
    sh.ok = v >= (unsigned)(ph - 1) ? 1 : 0;
    sh.rp = load_params(P.a, row);
  }
  __syncthreads();
  if (tid == 0 && sh.ok) ldcg_copy(&sh.rs, P.rows + row);
  if (tid < C) ldcg_copy(&sh.x1[tid], P.x1 + (size_t)row * C + tid);
  __syncthreads();
  const bool ok = sh.ok != 0;
  if (!ok && tid == 0) atomicOr(P.bad + row, 1u);
  const int plan = ok ? sh.rs.plan : kPlanDone;
  int what = 0;
  if (plan == kPlanTopP && ph == 2) what = 1;
  else if (plan == kPlanTopP && ph == 3) what = 2;
  else if (plan == kPlanFast && sh.rs.needW && ph == 2) what = 3;
  else if (plan == kPlanUntrunc && ph == 2) what = 4;
  if (what) {
    if (tid == 0) ring_start<kBF16>(geo<kBF16>(P, row, slice), carve(P.chunk), sh.seq);
    setup_re<kBF16>(P, row, slice);
    if (what == 1) topp_hist<kBF16>(P, row, slice);
    else if (what == 2) topp_race<kBF16>(P, row, slice);
    else if (what == 3) minp_pass<kBF16>(P, row, slice);
    else untrunc_pass<kBF16>(P, row, slice);
    __syncthreads();
    if (tid == 0) P.x2[idx] = sh.x2_mine;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const bool last = atomicAdd(P.ticket + 4 * row + ph, 1u) == (unsigned)C - 1u;
    if (last) P.ticket[4 * row + ph] = 0u;
    sh.last = last ? 1 : 0;
  }
  __syncthreads();
  if (!sh.last) return;
  __threadfence();
  if (tid < C) ldcg_copy(&sh.x2[tid], P.x2 + (size_t)row * C + tid);
  __syncthreads();
  phase_end<kBF16>(P, row, ph, nph, what);
}

// ---------------------------------------------------------------- the kernel

template <bool kBF16>
__global__ void __launch_bounds__(kThreads, kMinBlocks) sampler_kernel(const __grid_constant__ LaunchParams P) {
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&sh.full[i], 1);
    mbar_init(&sh.tbar, 1);
    fence_mbar_init();
    sh.seq = 0u;
    // every ring copy's L2 policy (set before any item, first phase or later): the row
    // end or a later phase reads parts of the slice again soon, so normal lines
    sh.policy = make_policy_evict_normal();
    sh.tpar = 0u;
    sh.tissued = 0;
    sh.tfail = 0;
  }
  // the ordering launch ahead of this one (programmatic dependent launch) has finished and
  // its results are visible after this
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __syncthreads();
  const unsigned C = (unsigned)P.C;
  const unsigned nitems = P.ctl[2] * C;  // work-list segments (the ordering launch wrote them)
  for (;;) {
    if (tid == 0) sh.item = atomicAdd(P.ctl, 1u);
    __syncthreads();
    const unsigned item = sh.item;
    if (item >= nitems) break;
    const unsigned e = P.seg[item / C];
    const int row = (int)(e & 0xFFFFFFu), ph = (int)((e >> 24) & 0xFu), nph = (int)(e >> 28);
    const int slice = (int)(item % C);
    if (ph == 1) p1_item<kBF16>(P, row, slice, nph);
    else phase_item<kBF16>(P, row, slice, ph, nph);
    __syncthreads();
  }
  // the last CTA out resets the claim counter (a later launch may reuse the list)
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(P.ctl + 1, 1u) == gridDim.x - 1u) {
      P.ctl[0] = 0u;
      P.ctl[1] = 0u;
    }
  }
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

// C = ceil(V / 2048) slices per row, at most kMaxSlices; slices are whole bitmask words.
// Shared memory does not depend on the logits type.
Geometry geometry_for(int vocab) {
  Geometry g{0, 0, 0};
  if (vocab <= 0) return g;
  int C = (vocab + 2047) / 2048;
  if (C > kMaxSlices) C = kMaxSlices;
  const int chunk = ((vocab + C - 1) / C + 31) / 32 * 32;
  if (chunk > kMaxChunk) return g;  // C = 0: vocabulary too large
  g.C = C;
  g.chunk = chunk;
  g.smem = (int)layout_for(chunk).total;
  return g;
}

// Byte offsets of the scratch arrays for B rows of C slices (one allocation).
struct ScratchLayout {
  size_t ctl, ticket, phase_done, bad, seg, order, rows, x1, x2, plist, plist_n, pen, tab, phist, cand, total;
};

constexpr size_t take(size_t& off, size_t bytes) {
  const size_t o = off;
  off = align_up(off + bytes, 256);
  return o;
}

constexpr ScratchLayout scratch_layout(size_t B, size_t C) {
  ScratchLayout L{};
  size_t off = 0;
  L.ctl = take(off, 4 * sizeof(unsigned));
  L.ticket = take(off, 4 * B * sizeof(unsigned));
  L.phase_done = take(off, B * sizeof(unsigned));
  L.bad = take(off, B * sizeof(unsigned));
  L.seg = take(off, 3 * B * sizeof(unsigned));
  L.order = take(off, B * sizeof(int));
  L.rows = take(off, B * sizeof(RowState));
  L.x1 = take(off, B * C * sizeof(X1));
  L.x2 = take(off, B * C * sizeof(X2));
  L.plist = take(off, B * C * kPenCap * sizeof(PenEntry));
  L.plist_n = take(off, B * C * sizeof(int2));
  L.pen = take(off, B * C * kPenCap * sizeof(uint2));
  L.tab = take(off, B * C * kTabMax * sizeof(uint16_t));
  L.phist = take(off, B * C * kPBins * sizeof(unsigned long long));
  L.cand = take(off, B * C * kCandCap * sizeof(Cand));
  L.total = off;
  return L;
}

// Device scratch of one call: sized for max_batch rows of up to C slices.
struct Scratch {
  int max_batch;
  int C;
  unsigned char* base;
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
  const void* ko = reinterpret_cast<const void*>(&order_kernel);
  if (cudaFuncSetAttribute(ko, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)prep_smem_bytes(kMaxSlices * kMaxChunk)) !=
      cudaSuccess)
    return CLSAMPLE_ERR_CUDA;
  // every kernel asks for the largest shared-memory carveout, so that the SMs need not
  // change their L1 / shared split between the ordering kernel and the sampler
  if (cudaFuncSetAttribute(k32, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(k16, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(k32, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
          cudaSuccess ||
      cudaFuncSetAttribute(k16, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
          cudaSuccess ||
      cudaFuncSetAttribute(ko, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
          cudaSuccess)
    return CLSAMPLE_ERR_CUDA;
  return CLSAMPLE_SUCCESS;
}

// CTAs of the persistent sampler kernel: as many as can be resident on device `dev`.
int resident_ctas(const Geometry& g, bool bf16, int dev, int* out) {
  int sms = 0, per = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return CLSAMPLE_ERR_CUDA;
  const cudaError_t err =
      bf16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, sampler_kernel<true>, kThreads, (size_t)g.smem)
           : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, sampler_kernel<false>, kThreads, (size_t)g.smem);
  if (err != cudaSuccess) return CLSAMPLE_ERR_CUDA;
  *out = sms * (per > 0 ? per : 1);
  return CLSAMPLE_SUCCESS;
}

}  // namespace

struct clsample_handle {
  int max_batch;
  int vocab;
  int device;
  Geometry g;
  Scratch sc;
  int grid[2];  // resident CTAs for f32 and bf16 logits
};

namespace {

// Scratch of clsample_apply_static: a fixed device array compiled into the library
// (zero at load), for kStaticRows rows of up to kMaxSlices slices.
constexpr int kStaticRows = 64;
constexpr size_t kStaticBytes = scratch_layout(kStaticRows, kMaxSlices).total;
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

int clsample_geometry(int32_t vocab, int32_t* slices, int32_t* chunk, int32_t* smem_bytes) {
  const Geometry g = geometry_for(vocab);
  if (g.C == 0) return CLSAMPLE_ERR_VOCAB;
  if (slices) *slices = g.C;
  if (chunk) *chunk = g.chunk;
  if (smem_bytes) *smem_bytes = g.smem;
  return CLSAMPLE_SUCCESS;
}

int clsample_create(int32_t max_batch, int32_t vocab, clsample_t** out) {
  if (!out) return CLSAMPLE_ERR_NULL;
  *out = nullptr;
  if (max_batch < 0 || max_batch > (1 << 24) - 1) return CLSAMPLE_ERR_BATCH;
  const Geometry g = geometry_for(vocab);
  if (g.C == 0) return CLSAMPLE_ERR_VOCAB;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CLSAMPLE_ERR_CUDA;
  int rc = setup_device(dev);
  if (rc != CLSAMPLE_SUCCESS) return rc;
  int grid[2];
  if ((rc = resident_ctas(g, false, dev, &grid[0])) != CLSAMPLE_SUCCESS) return rc;
  if ((rc = resident_ctas(g, true, dev, &grid[1])) != CLSAMPLE_SUCCESS) return rc;
  unsigned char* base = nullptr;
  if (max_batch > 0) {
    const size_t bytes = scratch_layout((size_t)max_batch, (size_t)g.C).total;
    void* p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) return CLSAMPLE_ERR_CUDA;
    if (cudaMemset(p, 0, bytes) != cudaSuccess) {
      cudaFree(p);
      return CLSAMPLE_ERR_CUDA;
    }
    base = static_cast<unsigned char*>(p);
  }
  clsample_t* h = new clsample_t;
  h->max_batch = max_batch;
  h->vocab = vocab;
  h->device = dev;
  h->g = g;
  h->sc = Scratch{max_batch, g.C, base};
  h->grid[0] = grid[0];
  h->grid[1] = grid[1];
  *out = h;
  return CLSAMPLE_SUCCESS;
}

void clsample_destroy(clsample_t* h) {
  if (!h) return;
  if (h->sc.base) cudaFree(h->sc.base);
  delete h;
}

}  // extern "C"

namespace {

// Validates a call and fills the launch parameters (host only): the vocabulary must be
// `vocab`, the batch at most the scratch's rows, and `dev` the current device.
int make_params(const Geometry& g, int vocab, int dev, const Scratch& sc, int grid, const clsample_args_t* a,
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
  const uintptr_t lb = reinterpret_cast<uintptr_t>(a->logits);
  P->vec_ok = (lb % 16 == 0) && (((long long)a->logits_row_stride * esize) % 16 == 0);
  P->gap = grid / g.C > 1 ? grid / g.C : 1;
  const ScratchLayout L = scratch_layout((size_t)sc.max_batch, (size_t)sc.C);
  unsigned char* b = sc.base;
  P->ctl = reinterpret_cast<unsigned*>(b + L.ctl);
  P->ticket = reinterpret_cast<unsigned*>(b + L.ticket);
  P->phase_done = reinterpret_cast<unsigned*>(b + L.phase_done);
  P->bad = reinterpret_cast<unsigned*>(b + L.bad);
  P->seg = reinterpret_cast<unsigned*>(b + L.seg);
  P->order = reinterpret_cast<int*>(b + L.order);
  P->rows = reinterpret_cast<RowState*>(b + L.rows);
  P->x1 = reinterpret_cast<X1*>(b + L.x1);
  P->x2 = reinterpret_cast<X2*>(b + L.x2);
  P->plist = reinterpret_cast<PenEntry*>(b + L.plist);
  P->plist_n = reinterpret_cast<int2*>(b + L.plist_n);
  P->pen = reinterpret_cast<uint2*>(b + L.pen);
  P->tab = reinterpret_cast<uint16_t*>(b + L.tab);
  P->phist = reinterpret_cast<unsigned long long*>(b + L.phist);
  P->cand = reinterpret_cast<Cand*>(b + L.cand);
  return CLSAMPLE_SUCCESS;
}

int make_params(const clsample_t* h, const clsample_args_t* a, LaunchParams* P, int* grid) {
  if (!h) return CLSAMPLE_ERR_NULL;
  if (!a) return CLSAMPLE_ERR_NULL;
  *grid = h->grid[a->logits_dtype == CLSAMPLE_LOGITS_BF16 ? 1 : 0];
  return make_params(h->g, h->vocab, h->device, h->sc, *grid, a, P);
}

int launch_order(const LaunchParams& P, cudaStream_t st) {
  const bool has_mod = P.a.hist_offs != nullptr || P.a.bias_offs != nullptr;
  const unsigned grid = has_mod ? 1u + (unsigned)P.a.B : 1u;
  order_kernel<<<grid, kOrderThreads, has_mod ? prep_smem_bytes(P.a.V) : 0, st>>>(P);
  return cudaGetLastError() == cudaSuccess ? CLSAMPLE_SUCCESS : CLSAMPLE_ERR_CUDA;
}

// The sampler kernel, launched with programmatic stream serialisation: its CTAs may start
// while the ordering launch ahead of it finishes, and wait for it (griddepcontrol.wait)
// before they read the work list.
int launch_sampler(const Geometry& g, int grid, const LaunchParams& P, cudaStream_t st) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)g.smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err = P.a.logits_dtype == CLSAMPLE_LOGITS_BF16 ? cudaLaunchKernelEx(&cfg, sampler_kernel<true>, P)
                                                                    : cudaLaunchKernelEx(&cfg, sampler_kernel<false>, P);
  return err == cudaSuccess ? CLSAMPLE_SUCCESS : CLSAMPLE_ERR_CUDA;
}

}  // namespace

extern "C" {

int clsample_apply(clsample_t* h, const clsample_args_t* a, clsample_stream_t stream) {
  LaunchParams P;
  int grid = 0;
  const int rc = make_params(h, a, &P, &grid);
  if (rc != CLSAMPLE_SUCCESS || a->B == 0) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int ro = launch_order(P, st);
  return ro != CLSAMPLE_SUCCESS ? ro : launch_sampler(h->g, grid, P, st);
}

int clsample_prepare(clsample_t* h, const clsample_args_t* a, clsample_stream_t stream) {
  LaunchParams P;
  int grid = 0;
  const int rc = make_params(h, a, &P, &grid);
  if (rc != CLSAMPLE_SUCCESS || a->B == 0) return rc;
  return launch_order(P, reinterpret_cast<cudaStream_t>(stream));
}

int clsample_sample(clsample_t* h, const clsample_args_t* a, clsample_stream_t stream) {
  LaunchParams P;
  int grid = 0;
  const int rc = make_params(h, a, &P, &grid);
  if (rc != CLSAMPLE_SUCCESS || a->B == 0) return rc;
  return launch_sampler(h->g, grid, P, reinterpret_cast<cudaStream_t>(stream));
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
  const bool bf16 = a->logits_dtype == CLSAMPLE_LOGITS_BF16;
  int grid = 0;
  if ((rc = resident_ctas(g, bf16, dev, &grid)) != CLSAMPLE_SUCCESS) return rc;
  const Scratch sc{kStaticRows, kMaxSlices, base};
  LaunchParams P;
  rc = make_params(g, a->V, dev, sc, grid, a, &P);
  if (rc != CLSAMPLE_SUCCESS || a->B == 0) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  rc = launch_order(P, st);
  return rc != CLSAMPLE_SUCCESS ? rc : launch_sampler(g, grid, P, st);
}

int clsample_occupancy(clsample_t* h, int32_t logits_dtype, int32_t* resident_ctas_out) {
  if (!h || !resident_ctas_out) return CLSAMPLE_ERR_NULL;
  if (logits_dtype != CLSAMPLE_LOGITS_F32 && logits_dtype != CLSAMPLE_LOGITS_BF16) return CLSAMPLE_ERR_DTYPE;
  *resident_ctas_out = h->grid[logits_dtype == CLSAMPLE_LOGITS_BF16 ? 1 : 0];
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
