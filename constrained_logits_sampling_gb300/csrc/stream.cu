// Persistent streaming sampler for GB300 (sm_103a).
//
// One launch per call (per 1024 rows).  The grid is persistent: as many CTAs as fit at
// once (two per SM), each with three roles:
//
//   producer warp     takes tasks -- first from a global queue of tasks that became
//                     ready during the call, else the next entry of the call's static
//                     list -- and starts each data task's TMA bulk copies (the logits
//                     slice, its bitmask words, its listed penalised / biased tokens)
//                     into a three-deep ring of slice buffers, so that HBM keeps
//                     streaming while the consumers compute;
//   consumer warps    (eight) run the tasks in ring order;
//   coordinator warp  publishes finished slices: a ticket per row and pass, and the row
//                     step that the last slice of a pass triggers (combine the slice
//                     records, finish a greedy row, queue the next pass or the row end).
//
// A row of V tokens is cut into C slices of 8192.  Its tasks:
//
//   prep   (rows with penalties or logit_bias) one task lists the row's distinct
//          history ids with their counts and each id's last valid bias value, by slice;
//   P1     per slice: the transforms (sanitising, penalties, bias, the grammar mask),
//          the slice's max, lowest argmax and sum of exponentials; top-k rows with
//          k <= 1024 also compact a candidate superset of the slice's part of the top-k
//          set (bound from the warps' sorted per-thread maxima);
//   row    greedy rows end here; top-k rows finish from their candidates (a sorted
//          finisher: exact top-k, top-p by exact fixed-point mass, min-p, the race);
//   P2     rows whose cut needs the row max (top-p over the vocabulary, top-k beyond
//          1024, candidate overflow) take passes over the row (re-read through L2) that
//          count tokens, and sum exact top-p weights, in 64 bins of y; each pass narrows
//          the band that holds the cut until it is small enough to compact;
//   P3     one more pass races the surely-kept tokens (exponential race, exact scores
//          near the best) and compacts the band; the row end resolves the band exactly.
//
// No task ever waits for another CTA: a pass's last slice queues the next step, so no
// wait can deadlock, and the producers' polls of the queue are bounded.  The decisions
// that turn floats into integers use the exact arithmetic of sampler_math.cuh, so the
// result equals the slice-resident kernel's bit for bit.  Page references: "SGLang
// source teardown (10): Sampling, Grammar and structured output" (SGLang page) and
// "GLM-5.3 inference (7): output side" (GLM page).

#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "bulk_copy.cuh"
#include "clsample.h"
#include "sampler_math.cuh"
#include "stream.h"

namespace clsample_stream {
namespace {

using namespace clsample;

// ---------------------------------------------------------------- geometry and roles

constexpr int kCW = 8;                  // consumer warps
constexpr int kCT = kCW * 32;           // consumer threads
constexpr int kPW = kCW;                // the producer warp
constexpr int kBlock = kCT + 64;        // + producer and coordinator warps
constexpr int kNB = 3;                  // slice ring depth
constexpr int kSL = 8192;               // tokens per slice
constexpr int kBuf = kSL * 4;           // bytes per ring buffer (a slice widened to fp32)
constexpr int kMW = kSL / 32;           // bitmask words per slice
constexpr int kVPT = kSL / 4 / kCT;     // float4 vectors per consumer thread
constexpr int kMaxVocab = 262144;
constexpr int kMaxC = kMaxVocab / kSL;  // 32 slices at most (one per coordinator lane)
constexpr int kCand = 1024;             // light candidates per slice (global scratch)
constexpr int kItemCap = kBuf / 8;      // items a finisher sorts in its ring buffer
constexpr int kEnt = 512;               // listed tokens per (row, slice), header included
constexpr int kEntStage = 128;          // of which the producer copies into shared memory
constexpr int kBins = 64;
constexpr int kNQ = 16;                 // consumer -> coordinator notices
constexpr int kLightK = 1024;           // top-k rows with k <= this finish from candidates
constexpr int kLead = 32;               // rows whose lists are prepared ahead of their slices
constexpr int kMaxRounds = 12;          // bin passes per row before it reports OVERFLOW
constexpr int kPrepSlots = 4096;        // a preparation task's hash (8-byte slots in its buffer)
constexpr int kPrepMax = 3072;          // distinct listed tokens of a row before the slow path
constexpr uint32_t kPolls = 1u << 22;   // bounded polls (about a second with the naps)
constexpr int kMaxGrid = 1024;          // persistent CTAs at most (the grid is capped to this)

static_assert(kMaxC <= 32, "one slice per coordinator lane");
static_assert(kPrepSlots * 8 <= kBuf, "the preparation hash fits a ring buffer");
static_assert(kVPT * 4 * kCT == kSL, "whole vectors per thread");
static_assert(kMW + kCT >= 512, "the row end's digit masses fit the slice scratch");

enum : uint32_t { kP1 = 0, kP2 = 1, kP3 = 2, kFin = 3, kPrep = 4, kExit = 7 };
__host__ __device__ constexpr uint32_t tcode(uint32_t ph, uint32_t slice) { return ph | (slice << 4); }

// Row classes, in list order: rows with a whole-vocabulary top-p first (three passes),
// other rows of the general route, top-k rows with a large k (long row ends), other
// top-k rows, greedy rows, invalid rows.
enum : int { kClsTopP = 0, kClsGen = 1, kClsBigK = 2, kClsLight = 3, kClsGreedy = 4, kClsInvalid = 5, kNCls = 6 };

enum : unsigned {
  kFInvalid = 1,    // bad parameters, CSR offsets or ids
  kFOverflow = 2,   // a bounded wait or a scratch limit was hit
  kFNonFinite = 4,  // the slice held non-finite logits (later passes sanitise)
  kFSpill = 8,      // more candidates than the slice's area holds
  kFSlow = 16       // the row's lists could not be prepared: slices scan the CSRs
};

// Plan flags of a row's passes.
enum : unsigned {
  kPMass = 1,         // P2 sums exact weights and bins coarse masses (top-p)
  kPQuarter = 2,      // P2 bins are quarter units of y (else 64 equal key ranges)
  kPBandCompact = 4,  // P3 compacts the band
  kPBandRace = 8,     // P3 races the (single-value) band apart
  kPNeedAbove = 16,   // P3 sums the exact mass of the tokens above the band
  kPNonFinite = 32,   // sanitise per token (a slice held non-finite logits)
  kPWKnown = 64       // the row end takes W from the plan (else from its items)
};
enum : unsigned { kPhK = 0, kPhP = 1 };

struct Item {
  float z;
  int id;
};

struct Params {
  float T, invT, p, mp, L, rep, freq, pres;
  int k, cls, invalid, hlo, hhi, blo, bhi, pad;
  unsigned long long seed, pos;
};

struct Ctl {
  unsigned epoch;      // the last finished launch's epoch (this launch uses the next value)
  unsigned next;       // static list: next entry
  unsigned rr;         // task queues: entries handed out so far (entry t goes to CTA t % grid)
  unsigned pad0;
  unsigned rows_done;  // rows with outputs written
  unsigned exited;     // CTAs past their loops (wraps at grid - 1)
  unsigned err;
  unsigned pad;
};

// A queue entry, published with one 64-bit release store: epoch (low 32 bits), task code
// (bits 32..47), row (bits 48..63).  A reader that sees its launch's epoch sees the task.
using DSlot = unsigned long long;
__host__ __device__ constexpr DSlot make_slot(unsigned epoch, uint32_t code, uint32_t row) {
  return (unsigned long long)epoch | ((unsigned long long)(code & 0xFFFFu) << 32) | ((unsigned long long)row << 48);
}

// P1 record of a slice.
struct __align__(16) Rec1 {
  float m;      // max z' (-inf if no candidate)
  int arg;      // lowest id reaching it
  float s;      // sum of 2^((z' - m) log2(e) / T)
  float s1;     // the same at T = 1 (when the original logprob is requested)
  int nal;      // candidates (z' > -inf)
  float bound;  // light rows: candidate bound (-inf: every candidate)
  int ncand;    // light rows: candidates compacted
  unsigned flags;
};

// P3 record of a slice.
struct __align__(16) Rec3 {
  float rs;  // best race score of the kept tokens above the band
  int rid;
  float ry, rz;
  unsigned long long wabove;  // exact mass of the tokens above the band
  unsigned nabove, kabove;    // tokens above the band; of them, kept by min-p
  float miny, sume;           // smallest y and sum of e^y of the kept ones
  float bs;                   // the same race over a band raced apart
  int bid;
  float by, bz;
  unsigned bk;
  float bminy, bsume;
  unsigned pad;
};

struct __align__(16) RowState {
  float m, invT, lnS, lnS1;  // after the P1 combine
  int arg, nal;
  unsigned flags;
  int kcut;
  unsigned phase, round, lo, hi;   // current bin pass over keys (lo, hi]
  unsigned excl, blo, bhi, pflags; // tokens with key < excl are out; P3 band (blo, bhi]
  int krem;
  unsigned pad0;
  unsigned long long W;            // exact top-p mass when known
  unsigned t1, t2, t3, done;       // tickets per pass (wrap at C - 1); finish marker (epoch)
  unsigned long long accW, accMass;
  unsigned accCount, nitems, pad1[2];
  float rs;  // P3 combine, for the band finisher
  int rid;
  float ry, rz;
  unsigned long long wabove;
  unsigned nabove, kabove;
  float miny, sume;
  unsigned pad2[2];
};

struct RowBins {
  unsigned cnt[kBins];
  unsigned long long cm[kBins];  // sums of (weight >> the bin's shift)
};

// A listed token of a (row, slice): local id, history count (bit 15: has a bias value)
// and the bias value.  Entry 0 of a block is its header (lid = number of entries).
struct __align__(8) Ent {
  uint16_t lid;
  uint16_t cnt;
  float bias;
};

struct KP {
  clsample_args_t a;
  int B, C, esize, masked, lists, total, want_orig, want_kept;
  unsigned epoch;  // set on the device at entry (a launch may be replayed from a graph)
  unsigned dq_cap;
  Ctl* ctl;
  DSlot* dq;
  RowState* rs;
  RowBins* bins;
  Rec1* r1;
  Rec3* r3;
  Item* cand;  // [B][C][kCand]
  Item* band;  // [B][kItemCap]
  Ent* ent;    // [B][C][kEnt]
  unsigned long long* prep;  // [B] (kFInvalid / kFSlow found while listing) << 32 | epoch of the row's lists
};

struct Desc {
  uint32_t row, code;
  int slice, c0, n, plain, mplain;
  unsigned rflags, pflags;
  Params q;
  float m;
  unsigned lo, hi, excl, blo, bhi;
};

struct __align__(16) Sm {
  unsigned long long full[kNB], empty[kNB], nfull[kNQ], nempty[kNQ];
  Desc desc[kNB];
  uint32_t nrow[kNQ], ncode[kNQ];
  alignas(16) unsigned mask[kNB][kMW];  // bulk-copy destinations: 16-byte aligned
  alignas(16) Ent ents[kNB][kEntStage];
  union {
    struct {
      unsigned claim[kMW];  // slice tasks: listed tokens
      unsigned tkey[kCT];   // slice tasks: per-thread maxima
    };
    unsigned long long hmass[256];  // row end: masses per radix digit
  };
  unsigned bcnt[kBins], bcm[kBins], bshift[kBins];
  unsigned hist[256];
  float rf[kCW * 2];
  int ri[kCW * 2];
  unsigned long long ru[kCW * 2];
  int ci[16];
  float cf[16];
  unsigned long long cu[4];
  Rec1 recs[kMaxC];
  unsigned short order[kMaxRows];
  int cls_start[kNCls + 1];  // list positions where each row class starts
  int scnt[kMaxC];
  unsigned kcnt[kBins], kshift[kBins];
  unsigned long long kcm[kBins];
};

extern __shared__ __align__(128) unsigned char dyn[];
__shared__ Sm sm;

// ---------------------------------------------------------------- small helpers

__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ int cbar_or(int v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.or.pred p, 1, 256, p;\n\tselp.s32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(v)
      : "memory");
  return r;
}
__device__ __forceinline__ unsigned ld_acq(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_vol(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_rel(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_rel64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acq64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
template <class T>
__device__ __forceinline__ T ldcg_t(const T* p) {
  static_assert(sizeof(T) % 16 == 0, "16-byte records");
  T r;
  const int4* s = reinterpret_cast<const int4*>(p);
  int4* d = reinterpret_cast<int4*>(&r);
#pragma unroll
  for (int i = 0; i < (int)(sizeof(T) / 16); ++i) d[i] = __ldcg(s + i);
  return r;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(~0u, v, o));
  return v;
}
__device__ __forceinline__ float warp_min_f(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fminf(v, __shfl_xor_sync(~0u, v, o));
  return v;
}
template <class T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(~0u, v, o);
  return v;
}
__device__ __forceinline__ unsigned warp_or(unsigned v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v |= __shfl_xor_sync(~0u, v, o);
  return v;
}

// Block (consumer threads) reductions; every consumer thread gets the result.
template <class T>
__device__ T csum(T v, T* slot) {
  v = warp_sum(v);
  cbar();
  if ((threadIdx.x & 31) == 0) slot[threadIdx.x >> 5] = v;
  cbar();
  T r = slot[0];
  for (int i = 1; i < kCW; ++i) r += slot[i];
  return r;
}
__device__ float cmin_f(float v) {
  v = warp_min_f(v);
  cbar();
  if ((threadIdx.x & 31) == 0) sm.rf[threadIdx.x >> 5] = v;
  cbar();
  float r = sm.rf[0];
  for (int i = 1; i < kCW; ++i) r = fminf(r, sm.rf[i]);
  return r;
}
__device__ int cmin_i(int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(~0u, v, o));
  cbar();
  if ((threadIdx.x & 31) == 0) sm.ri[threadIdx.x >> 5] = v;
  cbar();
  int r = sm.ri[0];
  for (int i = 1; i < kCW; ++i) r = min(r, sm.ri[i]);
  return r;
}
__device__ int cmax_i(int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(~0u, v, o));
  cbar();
  if ((threadIdx.x & 31) == 0) sm.ri[threadIdx.x >> 5] = v;
  cbar();
  int r = sm.ri[0];
  for (int i = 1; i < kCW; ++i) r = max(r, sm.ri[i]);
  return r;
}
// Exclusive prefix sum over the consumer threads (thread order); *total gets the sum.
__device__ unsigned long long cscan_u64(unsigned long long x, unsigned long long* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  unsigned long long v = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(~0u, v, o);
    if (lane >= o) v += t;
  }
  cbar();
  if (lane == 31) sm.ru[w] = v;
  cbar();
  unsigned long long off = 0, tot = 0;
  for (int i = 0; i < kCW; ++i) {
    if (i < w) off += sm.ru[i];
    tot += sm.ru[i];
  }
  *total = tot;
  return off + v - x;
}

// Race argmax over the consumer threads: larger score, then lower id; the winner's y and
// z' come along.  Every consumer thread gets the result.
struct Race {
  float s;
  int id;
  float y, z;
};
__device__ __forceinline__ unsigned long long race_key(float s, int id) {
  return ((unsigned long long)fkey(s) << 32) | (unsigned)(~(unsigned)id);
}
__device__ Race crace(Race r) {
  unsigned long long k = r.id == INT_MAX ? 0ull : race_key(r.s, r.id);
#pragma unroll
  for (int o = 16; o; o >>= 1) k = max(k, __shfl_xor_sync(~0u, k, o));
  cbar();
  if ((threadIdx.x & 31) == 0) sm.ru[threadIdx.x >> 5] = k;
  cbar();
  unsigned long long b = sm.ru[0];
  for (int i = 1; i < kCW; ++i) b = max(b, sm.ru[i]);
  cbar();
  if (b != 0ull && r.id != INT_MAX && race_key(r.s, r.id) == b) {
    sm.cf[8] = r.s;
    sm.ci[8] = r.id;
    sm.cf[9] = r.y;
    sm.cf[10] = r.z;
  }
  cbar();
  Race w{-INFINITY, INT_MAX, 0.0f, 0.0f};
  if (b != 0ull) w = Race{sm.cf[8], sm.ci[8], sm.cf[9], sm.cf[10]};
  cbar();
  return w;
}

// Folds token (y, id, z) into a thread's running race: the fast score filters, only a
// token within kFastTol of the best pays for the exact score.
__device__ __forceinline__ void race_in(Race& r, float y, float z, int id, uint32_t x) {
  if (!(fast_race(y, x) >= r.s - kFastTol)) return;
  const float s = race_score(y, x);
  if (better(s, id, r.s, r.id)) r = Race{s, id, y, z};
}

// ---------------------------------------------------------------- row parameters

__device__ void load_params(const clsample_args_t& a, int row, Params& q) {
  q.T = a.temperatures ? a.temperatures[row] : 1.0f;
  q.k = a.top_ks ? a.top_ks[row] : -1;
  q.p = a.top_ps ? a.top_ps[row] : 1.0f;
  q.mp = a.min_ps ? a.min_ps[row] : 0.0f;
  q.rep = a.rep ? a.rep[row] : 1.0f;
  q.freq = a.freq ? a.freq[row] : 0.0f;
  q.pres = a.pres ? a.pres[row] : 0.0f;
  q.seed = a.seeds ? a.seeds[row] : 0ull;
  q.pos = (unsigned long long)(a.positions ? a.positions[row] : a.step);
  int inv = 0;
  if (q.T != q.T || q.T == INFINITY) inv = 1;
  if (q.k < -1) inv = 1;
  if (!(q.p > 0.0f && q.p <= 1.0f)) inv = 1;
  if (!(q.mp >= 0.0f && q.mp <= 1.0f)) inv = 1;
  if (!(q.rep > 0.0f) || q.rep == INFINITY || !isfinite(q.freq) || !isfinite(q.pres)) inv = 1;
  q.hlo = q.hhi = q.blo = q.bhi = 0;
  if (a.hist_offs) {
    const int lo = a.hist_offs[row], hi = a.hist_offs[row + 1];
    if (lo < 0 || hi < lo) inv = 1;
    else {
      q.hlo = lo;
      q.hhi = hi;
    }
  }
  if (a.bias_offs) {
    const int lo = a.bias_offs[row], hi = a.bias_offs[row + 1];
    if (lo < 0 || hi < lo) inv = 1;
    else {
      q.blo = lo;
      q.bhi = hi;
    }
  }
  q.invalid = inv;
  const float Teff = (q.T >= kGreedyEps) ? q.T : 1.0f;
  q.invT = __fdiv_rn(1.0f, Teff);
  q.L = q.mp > 0.0f ? (float)log((double)q.mp) : -INFINITY;
  const bool greedy = (q.T < kGreedyEps) || q.k == 0 || q.k == 1 || (a.mode & CLSAMPLE_MODE_SCORE_ONLY);
  if (inv) q.cls = kClsInvalid;
  else if (greedy) q.cls = kClsGreedy;
  else if (q.k >= 2 && q.k <= kLightK) q.cls = q.k > 128 ? kClsBigK : kClsLight;
  else q.cls = q.p < 1.0f ? kClsTopP : kClsGen;
}

// List rank of a row from its sampling parameters alone (a scheduling choice only).
__device__ int row_rank(const clsample_args_t& a, int row) {
  const float T = a.temperatures ? a.temperatures[row] : 1.0f;
  const int k = a.top_ks ? a.top_ks[row] : -1;
  const float p = a.top_ps ? a.top_ps[row] : 1.0f;
  if (T < kGreedyEps || k == 0 || k == 1 || (a.mode & CLSAMPLE_MODE_SCORE_ONLY)) return kClsGreedy;
  if (k < -1 || !(p > 0.0f && p <= 1.0f) || T != T) return kClsInvalid;
  if (k >= 2 && k <= kLightK) return k > 128 ? kClsBigK : kClsLight;
  return p < 1.0f ? kClsTopP : kClsGen;
}

// Candidates a light row's slice keeps at least: 1.5 times its expected share of the
// top-k set plus 10, at most 256 (the warps' sorted per-thread maxima give the bound).
// Whether they hold the slice's whole part of the top-k set is checked at the row end;
// rows whose top tokens crowd into few slices (a contiguous grammar range) fail the
// check and take the general route.
__device__ __forceinline__ int light_q(int k, int n, int V) {
  const float share = (float)n / (float)V;
  return min(min(k, 256), (int)ceilf(1.5f * (float)k * share) + 10);
}

// ---------------------------------------------------------------- list order (all threads)

// Every CTA orders the rows the same way: a stable partition by rank.
__device__ void build_order(const KP& P) {
  const int B = P.B, tid = threadIdx.x;
  const int per = (B + kBlock - 1) / kBlock;  // <= 4 rows per thread
  int rk[4], cnt[kNCls];
#pragma unroll
  for (int c = 0; c < kNCls; ++c) cnt[c] = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = tid * per + i;
    rk[i] = (i < per && r < B) ? row_rank(P.a, r) : -1;
    if (rk[i] >= 0) ++cnt[rk[i]];
  }
  int* red = sm.scnt;  // kBlock / 32 = 10 warp totals per rank, reused per rank
  int base[kNCls], start = 0;
  if (tid == 0) sm.cls_start[0] = 0;
  const int lane = tid & 31, w = tid >> 5;
  for (int c = 0; c < kNCls; ++c) {
    int v = cnt[c];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(~0u, v, o);
      if (lane >= o) v += t;
    }
    __syncthreads();
    if (lane == 31) red[w] = v;
    __syncthreads();
    int off = 0, tot = 0;
    for (int i = 0; i < kBlock / 32; ++i) {
      if (i < w) off += red[i];
      tot += red[i];
    }
    base[c] = start + off + v - cnt[c];
    start += tot;
    if (tid == 0) sm.cls_start[c + 1] = start;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (rk[i] >= 0) sm.order[base[rk[i]]++] = (unsigned short)(tid * per + i);
}

// Static list entry i: with lists, kLead preparation tasks first, then per row its C
// slices followed by the preparation of the row kLead places later.
__device__ void static_task(const KP& P, unsigned i, uint32_t* row, uint32_t* code, unsigned* lpos) {
  const unsigned C = (unsigned)P.C, B = (unsigned)P.B;
  unsigned pos;
  if (!P.lists) {
    pos = i / C;
    *code = tcode(kP1, i % C);
  } else {
    const unsigned L = min((unsigned)kLead, B);
    const unsigned G1 = (B - L) * (C + 1);
    if (i < L) {
      pos = i;
      *code = kPrep;
    } else if (i - L < G1) {
      const unsigned j = i - L, r = j % (C + 1);
      pos = j / (C + 1) + (r < C ? 0u : L);
      *code = r < C ? tcode(kP1, r) : kPrep;
    } else {
      const unsigned j2 = i - L - G1;
      pos = (B - L) + j2 / C;
      *code = tcode(kP1, j2 % C);
    }
  }
  *row = sm.order[pos];
  *lpos = pos;
}

// ---------------------------------------------------------------- task queue

// Entries per CTA queue: every CTA owns an equal segment of the queue area (the area
// holds at least kMaxGrid entries more than the launch can push, so the rounded-down
// segment still fits every CTA's share); entry t of the launch goes to CTA t % grid, at
// position t / grid of its segment.
__device__ __forceinline__ unsigned queue_seg(const KP& P) { return P.dq_cap / gridDim.x; }

// Appends C tasks (slices 0..C-1 of `ph`) or one task (slice 0) for `row`; single thread.
// The caller's earlier writes (row state, zeroed accumulators) are published first.
__device__ bool push_tasks(const KP& P, uint32_t row, uint32_t ph, int n) {
  __threadfence();
  const unsigned t0 = atomicAdd(&P.ctl->rr, (unsigned)n);
  const unsigned seg = queue_seg(P);
  for (int s = 0; s < n; ++s) {
    const unsigned t = t0 + (unsigned)s;
    const unsigned pos = t / gridDim.x;
    if (pos >= seg) {
      atomicOr(&P.ctl->err, 2u);
      return false;
    }
    DSlot* d = P.dq + (size_t)(t % gridDim.x) * seg + pos;
    // the fence above orders every earlier write before these entries: relaxed stores
    st_relaxed64(d, make_slot(P.epoch, tcode(ph, (uint32_t)s), row));
  }
  return true;
}

// ---------------------------------------------------------------- outputs

__device__ void write_out(const KP& P, int row, int status, int tok, float lp, int kept, float cut, float lp_orig,
                          float lp_kept) {
  const clsample_args_t& a = P.a;
  const bool bad = status != CLSAMPLE_ROW_OK;
  a.tokens[row] = bad ? -1 : tok;
  if (a.logprobs) a.logprobs[row] = bad ? -INFINITY : lp;
  if (a.logprobs_orig) a.logprobs_orig[row] = bad ? -INFINITY : lp_orig;
  if (a.logprobs_kept) a.logprobs_kept[row] = bad ? -INFINITY : lp_kept;
  if (a.row_status) a.row_status[row] = status;
  if (a.dbg_kept_count) a.dbg_kept_count[row] = bad ? 0 : kept;
  if (a.dbg_cut) a.dbg_cut[row] = bad ? -INFINITY : cut;
  P.rs[row].done = P.epoch;
  atomicAdd(&P.ctl->rows_done, 1u);
}

__device__ __forceinline__ void row_fail(const KP& P, int row, int status) {
  write_out(P, row, status, -1, -INFINITY, 0, -INFINITY, -INFINITY, -INFINITY);
}

// ---------------------------------------------------------------- bins of y

__device__ __forceinline__ int quarter_bin(float y) { return (int)fminf(-4.0f * y, 63.0f); }
// Key range (lo, hi] of bin b of a pass.
__device__ void bin_range(unsigned pflags, unsigned lo, unsigned hi, int b, unsigned* blo, unsigned* bhi) {
  if (pflags & kPQuarter) {
    *bhi = fkey(-0.25f * (float)b);
    *blo = b == kBins - 1 ? 0u : fkey(-0.25f * (float)(b + 1));
    return;
  }
  const unsigned long long W = (unsigned long long)(hi - lo);
  const unsigned long long a0 = ((unsigned long long)b * W + kBins - 1) / kBins;
  const unsigned long long a1 = ((unsigned long long)(b + 1) * W + kBins - 1) / kBins;
  *bhi = hi - (unsigned)a0;
  *blo = hi - (unsigned)a1;
}
__device__ __forceinline__ int lin_bin(unsigned key, unsigned lo, unsigned hi) {
  return (int)(((unsigned long long)(hi - key) * kBins) / (unsigned long long)(hi - lo));
}
// Shift of bin b's coarse masses: every token of the bin weighs at most the weight of
// the bin's largest y, so weight >> shift keeps about 16 bits of it (and a slice's sum
// fits 32 bits); the bin's exact mass lies in [cm << shift, (cm + cnt) << shift].
__device__ int bin_shift(unsigned pflags, unsigned lo, unsigned hi, int b) {
  unsigned blo, bhi;
  bin_range(pflags, lo, hi, b, &blo, &bhi);
  const float ytop = key_to_float(bhi);
  const unsigned long long w = ytop > 0.0f ? (1ull << 40) : weight_fx(ytop);
  const int bits = w ? 64 - __clzll((long long)w) : 0;
  return bits > 16 ? bits - 16 : 0;
}

// Starts the general route of a row (single thread): P3 alone when nothing needs the
// row's distribution (min-p only, or no truncation), else the first bin pass.
__device__ void start_general(const KP& P, int row, const Params& q, int nal, unsigned nonfinite) {
  RowState& R = P.rs[row];
  const int kcut = (q.k >= 2 && q.k < nal) ? q.k : 0;
  const bool pcut = q.p < 1.0f;
  R.kcut = kcut;
  R.excl = 0u;
  R.nitems = 0u;
  R.krem = 0;
  if (!kcut && !pcut) {
    R.blo = 0u;
    R.bhi = 0u;
    R.pflags = nonfinite;
    push_tasks(P, row, kP3, P.C);
    return;
  }
  R.phase = kcut ? kPhK : kPhP;
  R.round = 0u;
  R.lo = 0u;
  R.hi = fkey(0.0f);
  R.pflags = kPQuarter | (kcut ? 0u : kPMass) | nonfinite;
  R.accW = 0ull;
  R.accMass = 0ull;
  R.accCount = 0u;
  RowBins& G = P.bins[row];
  for (int b = 0; b < kBins; ++b) {
    G.cnt[b] = 0u;
    G.cm[b] = 0ull;
  }
  push_tasks(P, row, kP2, P.C);
}

// ---------------------------------------------------------------- slice front (consumers)

// Applies one listed token: sanitise, penalties, bias, overflow guard; marks it claimed.
// Returns 1 if an allowed token became -inf (the allowed count drops by one).
__device__ __forceinline__ int apply_entry(float* buf, const Desc& d, const unsigned* mw, int lid, unsigned cnt,
                                           bool hb, float bias) {
  float z = sanitize(buf[lid]);
  if (cnt) z = apply_penalties(z, cnt, d.q.freq, d.q.pres, d.q.rep);
  if (hb) z = __fadd_rn(z, bias);
  z = guard(z);
  buf[lid] = z;
  atomicOr(&sm.claim[lid >> 5], 1u << (lid & 31));
  const bool allowed = mw ? ((mw[lid >> 5] >> (lid & 31)) & 1u) : true;
  return (allowed && z == -INFINITY) ? 1 : 0;
}

// Slow path of the transforms (rows whose lists could not be prepared): every history
// id of the slice is counted by its first occurrence, each id's last valid bias entry
// found by a scan.  Quadratic in the history length; only pathological rows take it.
__device__ int slow_transforms(const KP& P, const Desc& d, float* buf, const unsigned* mw, unsigned* bad) {
  const clsample_args_t& a = P.a;
  const int c0 = d.c0, n = d.n, V = a.V;
  int ninf = 0;
  for (int j = d.q.hlo + threadIdx.x; j < d.q.hhi; j += kCT) {
    const int id = __ldg(a.hist_ids + j);
    if (id < 0 || id >= V) {
      *bad = 1;
      continue;
    }
    if (id < c0 || id >= c0 + n) continue;
    bool first = true;
    for (int i = d.q.hlo; i < j && first; ++i) first = __ldg(a.hist_ids + i) != id;
    if (!first) continue;
    unsigned c = 0;
    for (int i = j; i < d.q.hhi; ++i) c += __ldg(a.hist_ids + i) == id;
    int bj = -1;
    for (int i = d.q.blo; i < d.q.bhi; ++i) {
      const float bv = __ldg(a.bias_vals + i);
      if (__ldg(a.bias_ids + i) == id && bv == bv) bj = i;
    }
    ninf += apply_entry(buf, d, mw, id - c0, c, bj >= 0, bj >= 0 ? __ldg(a.bias_vals + bj) : 0.0f);
  }
  for (int j = d.q.blo + threadIdx.x; j < d.q.bhi; j += kCT) {
    const int id = __ldg(a.bias_ids + j);
    const float bv = __ldg(a.bias_vals + j);
    if (id < 0 || id >= V || bv != bv) {
      *bad = 1;
      continue;
    }
    if (id < c0 || id >= c0 + n) continue;
    bool in_hist = false;
    for (int i = d.q.hlo; i < d.q.hhi && !in_hist; ++i) in_hist = __ldg(a.hist_ids + i) == id;
    if (in_hist) continue;
    bool last = true;
    for (int i = j + 1; i < d.q.bhi && last; ++i) {
      const float v2 = __ldg(a.bias_vals + i);
      last = !(__ldg(a.bias_ids + i) == id && v2 == v2);
    }
    if (last) ninf += apply_entry(buf, d, mw, id - c0, 0u, true, bv);
  }
  return ninf;
}

// Brings the slice into its final transformed form in `buf` (fp32), except the grammar
// mask, which the caller applies per vector: plain copies where the producer could not
// use bulk copies, bf16 widening, the listed tokens.  Returns this thread's count of
// allowed tokens the transforms turned into -inf; sets *bad on an invalid id (slow path).
__device__ int slice_front(const KP& P, const Desc& d, int st, float* buf, unsigned* bad) {
  const clsample_args_t& a = P.a;
  const int n = d.n;
  unsigned* mw = P.masked ? sm.mask[st] : nullptr;
  for (int w = threadIdx.x; w < kMW; w += kCT) sm.claim[w] = 0u;
  if (d.plain) {
    if (P.esize == 4) {
      const float* src = static_cast<const float*>(a.logits) + (long long)d.row * a.logits_row_stride + d.c0;
      for (int i = threadIdx.x; i < n; i += kCT) buf[i] = __ldg(src + i);
    } else {
      const uint16_t* src = static_cast<const uint16_t*>(a.logits) + (long long)d.row * a.logits_row_stride + d.c0;
      for (int i = threadIdx.x; i < n; i += kCT) buf[i] = __uint_as_float((uint32_t)__ldg(src + i) << 16);
    }
  }
  if (mw && d.mplain) {
    const int32_t* src = a.bitmask + (long long)d.row * a.bitmask_row_stride + (d.c0 >> 5);
    for (int w = threadIdx.x; w < ((n + 31) >> 5); w += kCT) mw[w] = (uint32_t)__ldg(src + w);
  }
  if (P.esize == 2 && !d.plain) {
    // the raw bf16 slice sits in the upper half: read every element first, then widen
    const uint4* raw = reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned char*>(buf) + kBuf / 2);
    uint4 v[kSL / 8 / kCT];
#pragma unroll
    for (int u = 0; u < kSL / 8 / kCT; ++u) {
      const int f = threadIdx.x + u * kCT;
      v[u] = f * 8 < n ? raw[f] : make_uint4(0u, 0u, 0u, 0u);
    }
    cbar();
    float4* o = reinterpret_cast<float4*>(buf);
#pragma unroll
    for (int u = 0; u < kSL / 8 / kCT; ++u) {
      const int f = threadIdx.x + u * kCT;
      if (f * 8 < n) {
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        o[2 * f] = make_float4(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xFFFF0000u),
                               __uint_as_float(w[1] << 16), __uint_as_float(w[1] & 0xFFFF0000u));
        o[2 * f + 1] = make_float4(__uint_as_float(w[2] << 16), __uint_as_float(w[2] & 0xFFFF0000u),
                                   __uint_as_float(w[3] << 16), __uint_as_float(w[3] & 0xFFFF0000u));
      }
    }
  }
  // finite pads past the slice end (masked out below)
  if (threadIdx.x < 4 && (n & 3) && (n & ~3) + (int)threadIdx.x >= n) buf[(n & ~3) + threadIdx.x] = 0.0f;
  cbar();
  int ninf = 0;
  if (P.lists) {
    const unsigned rfl = d.rflags;
    if (rfl & kFSlow) {
      ninf = slow_transforms(P, d, buf, mw, bad);
    } else {
      const Ent* g = P.ent + ((size_t)d.row * P.C + d.slice) * kEnt;
      const Ent* s = sm.ents[st];
      const int nent = s[0].lid;  // the block's header
      for (int i = 1 + threadIdx.x; i <= nent; i += kCT) {
        Ent e;
        if (i < kEntStage) e = s[i];
        else {
          const int2 v = __ldcg(reinterpret_cast<const int2*>(g + i));
          memcpy(&e, &v, sizeof e);
        }
        ninf += apply_entry(buf, d, mw, e.lid, e.cnt & 0x7FFFu, (e.cnt >> 15) != 0, e.bias);
      }
    }
  }
  cbar();
  return ninf;
}

// Sanitises every unlisted token (listed ones already hold their final value) and
// applies the mask in place; for slices that held non-finite logits.
__device__ void checked_walk(const KP& P, const Desc& d, int st, float* buf) {
  const unsigned* mw = P.masked ? sm.mask[st] : nullptr;
  for (int l = threadIdx.x; l < kSL; l += kCT) {
    float z = -INFINITY;
    if (l < d.n) {
      const bool ok = mw ? ((mw[l >> 5] >> (l & 31)) & 1u) : true;
      const bool listed = (sm.claim[l >> 5] >> (l & 31)) & 1u;
      if (ok) z = listed ? buf[l] : sanitize(buf[l]);
    }
    buf[l] = z;
  }
  cbar();
}

__device__ __forceinline__ uint32_t mask_nibble(const unsigned* mw, int f) {
  return mw ? (mw[f >> 3] >> ((f & 7) * 4)) & 0xFu : 0xFu;
}

// Applies the mask (and the slice end) to vector f in place; returns the vector.
__device__ __forceinline__ float4 masked_vec(float* buf, const unsigned* mw, int f, int nv, uint32_t tail) {
  float4* b4 = reinterpret_cast<float4*>(buf);
  float4 v = b4[f];
  uint32_t bits = mask_nibble(mw, f);
  if (f == nv - 1) bits &= tail;
  if (bits != 0xFu) {
    if (!(bits & 1u)) v.x = -INFINITY;
    if (!(bits & 2u)) v.y = -INFINITY;
    if (!(bits & 4u)) v.z = -INFINITY;
    if (!(bits & 8u)) v.w = -INFINITY;
    b4[f] = v;
  }
  return v;
}

// ---------------------------------------------------------------- P1: statistics and candidates

__device__ void task_p1(const KP& P, const Desc& d, int st, float* buf) {
  const clsample_args_t& a = P.a;
  const int row = d.row, n = d.n, c0 = d.c0;
  const Params& q = d.q;
  if (q.cls == kClsInvalid && !a.dbg_transformed) {
    if (threadIdx.x == 0) {
      Rec1 r{-INFINITY, INT_MAX, 0.0f, 0.0f, 0, -INFINITY, 0, kFInvalid};
      P.r1[(size_t)row * P.C + d.slice] = r;
    }
    return;
  }
  unsigned bad = 0;
  const int ninf = slice_front(P, d, st, buf, &bad);
  const unsigned* mw = P.masked ? sm.mask[st] : nullptr;
  const int nv = (n + 3) >> 2;
  const uint32_t tail = (n & 3) ? ((1u << (n & 3)) - 1u) : 0xFu;
  const float c = __fmul_rn(1.4426950408889634f, q.invT);
  constexpr float l2e = 1.4426950408889634f;
  float4* b4 = reinterpret_cast<float4*>(buf);
  // the thread's vectors in registers: masked tokens and the slice end become -inf (and
  // are written back for the candidate and debug outputs); a running sum of the raw
  // values detects non-finite input
  float4 v[kVPT];
  float chk0 = 0.0f, chk1 = 0.0f;
  int nal = 0;
#pragma unroll
  for (int u = 0; u < kVPT; ++u) {
    const int f = threadIdx.x + u * kCT;
    float4 x = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    if (f < nv) {
      x = b4[f];
      if (u & 1) chk1 += (x.x + x.y) + (x.z + x.w);
      else chk0 += (x.x + x.y) + (x.z + x.w);
      uint32_t bits = mask_nibble(mw, f);
      if (f == nv - 1) bits &= tail;
      nal += __popc(bits);
      if (bits != 0xFu) {
        if (!(bits & 1u)) x.x = -INFINITY;
        if (!(bits & 2u)) x.y = -INFINITY;
        if (!(bits & 4u)) x.z = -INFINITY;
        if (!(bits & 8u)) x.w = -INFINITY;
        b4[f] = x;
      }
    }
    v[u] = x;
  }
  nal -= ninf;
  const int nonfinite = cbar_or(!(fabsf(chk0 + chk1) < INFINITY));
  if (nonfinite) {
    checked_walk(P, d, st, buf);
    nal = 0;
#pragma unroll
    for (int u = 0; u < kVPT; ++u) {
      const int f = threadIdx.x + u * kCT;
      v[u] = f < nv ? b4[f] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      nal += (v[u].x > -INFINITY) + (v[u].y > -INFINITY) + (v[u].z > -INFINITY) + (v[u].w > -INFINITY);
    }
  }
  // the thread's max, its first vector reaching it, then the sums against it
  float vm[kVPT];
  float tmax = -INFINITY;
#pragma unroll
  for (int u = 0; u < kVPT; ++u) {
    vm[u] = fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w));
    tmax = fmaxf(tmax, vm[u]);
  }
  int tf = INT_MAX;
#pragma unroll
  for (int u = kVPT - 1; u >= 0; --u)
    if (vm[u] == tmax) tf = threadIdx.x + u * kCT;
  float tsum = 0.0f, tsum1 = 0.0f;
  if (tmax > -INFINITY) {
    float p0 = 0.0f, p1 = 0.0f, p2 = 0.0f, p3 = 0.0f;
#pragma unroll
    for (int u = 0; u < kVPT; ++u) {
      p0 += ex2_approx((v[u].x - tmax) * c);
      p1 += ex2_approx((v[u].y - tmax) * c);
      p2 += ex2_approx((v[u].z - tmax) * c);
      p3 += ex2_approx((v[u].w - tmax) * c);
    }
    tsum = (p0 + p1) + (p2 + p3);
    if (P.want_orig) {
      p0 = p1 = p2 = p3 = 0.0f;
#pragma unroll
      for (int u = 0; u < kVPT; ++u) {
        p0 += ex2_approx((v[u].x - tmax) * l2e);
        p1 += ex2_approx((v[u].y - tmax) * l2e);
        p2 += ex2_approx((v[u].z - tmax) * l2e);
        p3 += ex2_approx((v[u].w - tmax) * l2e);
      }
      tsum1 = (p0 + p1) + (p2 + p3);
    }
  }
  sm.tkey[threadIdx.x] = tmax > -INFINITY ? fkey(tmax) : 0u;
  int arg = INT_MAX;
  if (tf != INT_MAX && tmax > -INFINITY) {
    const float4 x = b4[tf];
    const int j = x.x == tmax ? 0 : x.y == tmax ? 1 : x.z == tmax ? 2 : 3;
    arg = c0 + 4 * tf + j;
  }
  // combine: (max, lowest argmax) by 64-bit keys, then the sums rescaled to the max
  unsigned long long key = tmax > -INFINITY ? race_key(tmax, arg) : 0ull;
#pragma unroll
  for (int o = 16; o; o >>= 1) key = max(key, __shfl_xor_sync(~0u, key, o));
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) sm.ru[w] = key;
  bad = warp_or(bad);
  nal = warp_sum(nal);
  cbar();
  unsigned long long bk = sm.ru[0];
  for (int i = 1; i < kCW; ++i) bk = max(bk, sm.ru[i]);
  const float M = bk ? key_to_float((uint32_t)(bk >> 32)) : -INFINITY;
  float ws = (M > -INFINITY && tmax > -INFINITY) ? tsum * ex2_approx((tmax - M) * c) : 0.0f;
  float ws1 = (P.want_orig && M > -INFINITY && tmax > -INFINITY) ? tsum1 * ex2_approx((tmax - M) * l2e) : 0.0f;
  ws = warp_sum(ws);
  ws1 = warp_sum(ws1);
  if (lane == 0) {
    sm.rf[w] = ws;
    sm.rf[kCW + w] = ws1;
    sm.ri[w] = nal;
    sm.ri[kCW + w] = (int)bad;
  }
  cbar();
  Rec1 rec;
  rec.m = M;
  rec.arg = bk ? (int)~(uint32_t)bk : INT_MAX;
  rec.s = 0.0f;
  rec.s1 = 0.0f;
  rec.nal = 0;
  unsigned flags = (nonfinite ? kFNonFinite : 0u);
  for (int i = 0; i < kCW; ++i) {
    rec.s += sm.rf[i];
    rec.s1 += sm.rf[kCW + i];
    rec.nal += sm.ri[i];
    if (sm.ri[kCW + i]) flags |= kFInvalid;
  }
  rec.bound = -INFINITY;
  rec.ncand = 0;
  if (a.dbg_transformed) {
    float4* dst = reinterpret_cast<float4*>(a.dbg_transformed + (long long)row * a.V + c0);
    const bool vec = ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) && (n % 4 == 0);
#pragma unroll
    for (int u = 0; u < kVPT; ++u) {
      const int f = threadIdx.x + u * kCT;
      if (vec) {
        if (f < nv) dst[f] = v[u];
      } else {
        float* d1 = a.dbg_transformed + (long long)row * a.V + c0;
        const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (4 * f + j < n) d1[4 * f + j] = e[j];
      }
    }
  }
  if ((q.cls == kClsLight || q.cls == kClsBigK) && M > -INFINITY) {
    // candidate superset of the slice's part of the top-k set
    const int qn = light_q(q.k, n, a.V);
    uint32_t bkey = 0u;  // 0: take every candidate
    if (rec.nal > qn) {
      uint32_t kk = sm.tkey[threadIdx.x];
#pragma unroll
      for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          const uint32_t o = __shfl_xor_sync(~0u, kk, stride);
          const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
          kk = keep_max ? max(kk, o) : min(kk, o);
        }
      const int r = min(32, (qn + kCW - 1) / kCW) - 1;
      const uint32_t bw = __shfl_sync(~0u, kk, r);
      cbar();
      if (lane == 0) sm.ri[w] = (int)bw;
      cbar();
      bkey = (uint32_t)sm.ri[0];
      for (int i = 1; i < kCW; ++i) bkey = min(bkey, (uint32_t)sm.ri[i]);
    }
    const float bound = bkey ? key_to_float(bkey) : -INFINITY;
    if (threadIdx.x == 0) sm.ci[0] = 0;
    cbar();
    Item* dst = P.cand + ((size_t)row * P.C + d.slice) * kCand;
    // per thread: count, warp-aggregated slot, then write (from the registers)
    int mine = 0;
    if (tmax > -INFINITY && tmax >= bound) {
#pragma unroll
      for (int u = 0; u < kVPT; ++u)
        mine += (v[u].x >= bound && v[u].x > -INFINITY) + (v[u].y >= bound && v[u].y > -INFINITY) +
                (v[u].z >= bound && v[u].z > -INFINITY) + (v[u].w >= bound && v[u].w > -INFINITY);
    }
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(~0u, incl, o);
      if (lane >= o) incl += t;
    }
    int base = 0;
    if (lane == 31 && incl) base = atomicAdd(&sm.ci[0], incl);
    base = __shfl_sync(~0u, base, 31) + incl - mine;
    if (mine) {
      int pos = base;
#pragma unroll
      for (int u = 0; u < kVPT; ++u) {
        const int f = threadIdx.x + u * kCT;
        const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (e[j] >= bound && e[j] > -INFINITY) {
            if (pos < kCand) dst[pos] = Item{e[j], c0 + 4 * f + j};
            ++pos;
          }
      }
    }
    cbar();
    rec.ncand = sm.ci[0];
    rec.bound = bound;
    if (rec.ncand > kCand) flags |= kFSpill;
  }
  rec.flags = flags;
  if (threadIdx.x == 0) P.r1[(size_t)row * P.C + d.slice] = rec;
}

// ---------------------------------------------------------------- P2: bins

__device__ void task_p2(const KP& P, const Desc& d, int st, float* buf) {
  unsigned bad = 0;
  slice_front(P, d, st, buf, &bad);
  if (d.pflags & kPNonFinite) checked_walk(P, d, st, buf);
  for (int b = threadIdx.x; b < kBins; b += kCT) {
    sm.bcnt[b] = 0u;
    sm.bcm[b] = 0u;
    sm.bshift[b] = (unsigned)bin_shift(d.pflags, d.lo, d.hi, b);
  }
  cbar();
  const unsigned* mw = P.masked ? sm.mask[st] : nullptr;
  const int nv = (d.n + 3) >> 2;
  const uint32_t tail = (d.n & 3) ? ((1u << (d.n & 3)) - 1u) : 0xFu;
  const bool mass = d.pflags & kPMass, quarter = d.pflags & kPQuarter;
  const float m = d.m, invT = d.q.invT;
  unsigned long long Wt = 0ull, ma = 0ull;
  unsigned ca = 0u;
  for (int u = 0; u < kVPT; ++u) {
    const int f = threadIdx.x + u * kCT;
    if (f >= nv) break;
    const float4 v = masked_vec(buf, mw, f, nv, tail);
    const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (!(e[j] > -INFINITY)) continue;
      const float y = y_of(e[j], m, invT);
      const unsigned key = fkey(y);
      if (key < d.excl) continue;
      unsigned long long wx = 0ull;
      if (mass) {
        wx = weight_fx(y);
        Wt += wx;
      }
      if (key > d.hi) {
        ++ca;
        ma += wx;
      } else if (key > d.lo) {
        const int b = quarter ? quarter_bin(y) : lin_bin(key, d.lo, d.hi);
        atomicAdd(&sm.bcnt[b], 1u);
        if (mass) atomicAdd(&sm.bcm[b], (unsigned)(wx >> sm.bshift[b]));
      }
    }
  }
  Wt = csum(Wt, sm.ru);
  ma = csum(ma, sm.ru + kCW);
  ca = csum(ca, reinterpret_cast<unsigned*>(sm.ri));
  RowState& R = P.rs[d.row];
  RowBins& G = P.bins[d.row];
  if (threadIdx.x == 0) {
    if (Wt) atomicAdd(&R.accW, Wt);
    if (ma) atomicAdd(&R.accMass, ma);
    if (ca) atomicAdd(&R.accCount, ca);
  }
  for (int b = threadIdx.x; b < kBins; b += kCT) {
    if (sm.bcnt[b]) atomicAdd(&G.cnt[b], sm.bcnt[b]);
    if (sm.bcm[b]) atomicAdd(&G.cm[b], (unsigned long long)sm.bcm[b]);
  }
}

// ---------------------------------------------------------------- P3: race and band

__device__ void task_p3(const KP& P, const Desc& d, int st, float* buf) {
  unsigned bad = 0;
  slice_front(P, d, st, buf, &bad);
  if (d.pflags & kPNonFinite) checked_walk(P, d, st, buf);
  const unsigned* mw = P.masked ? sm.mask[st] : nullptr;
  const int nv = (d.n + 3) >> 2;
  const uint32_t tail = (d.n & 3) ? ((1u << (d.n & 3)) - 1u) : 0xFu;
  const float m = d.m, invT = d.q.invT, L = d.q.L;
  const bool need_above = d.pflags & kPNeedAbove, compact = d.pflags & kPBandCompact,
             braced = d.pflags & kPBandRace;
  const unsigned long long seed = d.q.seed, pos = d.q.pos;
  Race ra{-INFINITY, INT_MAX, 0.0f, 0.0f}, rb{-INFINITY, INT_MAX, 0.0f, 0.0f};
  unsigned long long wab = 0ull;
  unsigned nab = 0u, kab = 0u, bk = 0u;
  float miny = INFINITY, sume = 0.0f, bminy = INFINITY, bsume = 0.0f;
  const float l2e = 1.4426950408889634f;
  RowState& R = P.rs[d.row];
  Item* band = P.band + (size_t)d.row * kItemCap;
  for (int u = 0; u < kVPT; ++u) {
    const int f = threadIdx.x + u * kCT;
    if (f >= nv) break;
    const float4 v = masked_vec(buf, mw, f, nv, tail);
    const float e[4] = {v.x, v.y, v.z, v.w};
    float yy[4];
    unsigned cls[4];  // 0 out, 1 above, 2 band
    unsigned any_race = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      cls[j] = 0u;
      yy[j] = -INFINITY;
      if (!(e[j] > -INFINITY)) continue;
      yy[j] = y_of(e[j], m, invT);
      const unsigned key = fkey(yy[j]);
      if (key < d.excl) continue;
      if (key > d.bhi) cls[j] = 1u;
      else if (key > d.blo && (compact || braced)) cls[j] = 2u;
      if (cls[j] == 1u) {
        ++nab;
        if (need_above) wab += weight_fx(yy[j]);
      }
      if (cls[j] == 2u && compact) {
        const unsigned slot = atomicAdd(&R.nitems, 1u);
        if (slot < (unsigned)kItemCap) band[slot] = Item{e[j], d.c0 + 4 * f + j};
        cls[j] = 0u;
      }
      if (cls[j] && yy[j] >= L) {
        if (yy[j] + kGumbelMax >= (cls[j] == 1u ? ra.s : rb.s)) any_race |= 1u << j;
        if (cls[j] == 1u) {
          ++kab;
          miny = fminf(miny, yy[j]);
          sume += ex2_approx(yy[j] * l2e);
        } else {
          ++bk;
          bminy = fminf(bminy, yy[j]);
          bsume += ex2_approx(yy[j] * l2e);
        }
      }
    }
    if (any_race) {
      const int t0 = d.c0 + 4 * f;
      const uint4 x = race_words((uint32_t)t0 >> 2, seed, pos);
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (!((any_race >> j) & 1u)) continue;
        if (cls[j] == 1u) race_in(ra, yy[j], e[j], t0 + j, xs[j]);
        else race_in(rb, yy[j], e[j], t0 + j, xs[j]);
      }
    }
  }
  ra = crace(ra);
  rb = crace(rb);
  wab = csum(wab, sm.ru);
  nab = csum(nab, reinterpret_cast<unsigned*>(sm.ri));
  kab = csum(kab, reinterpret_cast<unsigned*>(sm.ri));
  bk = csum(bk, reinterpret_cast<unsigned*>(sm.ri));
  miny = cmin_f(miny);
  bminy = cmin_f(bminy);
  sume = csum(sume, sm.rf);
  bsume = csum(bsume, sm.rf);
  if (threadIdx.x == 0) {
    Rec3 r;
    r.rs = ra.s;
    r.rid = ra.id;
    r.ry = ra.y;
    r.rz = ra.z;
    r.wabove = wab;
    r.nabove = nab;
    r.kabove = kab;
    r.miny = miny;
    r.sume = sume;
    r.bs = rb.s;
    r.bid = rb.id;
    r.by = rb.y;
    r.bz = rb.z;
    r.bk = bk;
    r.bminy = bminy;
    r.bsume = bsume;
    r.pad = 0u;
    P.r3[(size_t)d.row * P.C + d.slice] = r;
  }
}

// ---------------------------------------------------------------- preparation of a row's lists

__device__ __forceinline__ unsigned prep_hash(int id) { return ((unsigned)id * 2654435761u) >> 20; }

__device__ void task_prep(const KP& P, const Desc& d, float* buf) {
  const clsample_args_t& a = P.a;
  const int row = d.row, V = a.V, C = P.C;
  // hash of the row's distinct ids: {id + 1, count (low 20 bits) | last bias entry + 1 - blo
  // (high 12 bits)}
  uint2* H = reinterpret_cast<uint2*>(buf);
  for (int i = threadIdx.x; i < kPrepSlots; i += kCT) H[i] = make_uint2(0u, 0u);
  if (threadIdx.x < kMaxC) sm.scnt[threadIdx.x] = 0;
  if (threadIdx.x == 0) {
    sm.ci[0] = 0;  // distinct ids
    // histories of 2^20 ids or more, or 4095 bias entries or more, do not fit the slots
    sm.ci[1] = (d.q.hhi - d.q.hlo >= (1 << 20) || d.q.bhi - d.q.blo >= 4095) ? (int)kFSlow : 0;
  }
  cbar();
  unsigned flags = 0u;
  auto insert = [&](int id) -> int {
    unsigned h = prep_hash(id);
    for (int t = 0; t < kPrepSlots; ++t) {
      const unsigned k = atomicCAS(&H[h].x, 0u, (unsigned)id + 1u);
      if (k == 0u) {
        atomicAdd(&sm.ci[0], 1);
        return (int)h;
      }
      if (k == (unsigned)id + 1u) return (int)h;
      h = (h + 1u) & (kPrepSlots - 1);
    }
    return -1;
  };
  if (!sm.ci[1]) {
    for (int j = d.q.hlo + threadIdx.x; j < d.q.hhi; j += kCT) {
      const int id = __ldg(a.hist_ids + j);
      if (id < 0 || id >= V) {
        flags |= kFInvalid;
        continue;
      }
      const int h = insert(id);
      if (h < 0) flags |= kFSlow;
      else atomicAdd(&H[h].y, 1u);
    }
  }
  cbar();
  // bias entries by one warp, in entry order, so the last valid entry of an id wins: in
  // each group of 32 the highest lane of an id writes
  if (!sm.ci[1] && threadIdx.x < 32) {
    const int lane = threadIdx.x;
    for (int j0 = d.q.blo; j0 < d.q.bhi; j0 += 32) {
      const int j = j0 + lane;
      int id = -1 - lane;
      bool ok = false;
      if (j < d.q.bhi) {
        const int bid = __ldg(a.bias_ids + j);
        const float bv = __ldg(a.bias_vals + j);
        ok = bid >= 0 && bid < V && bv == bv;
        if (!ok) flags |= kFInvalid;
        else id = bid;
      }
      const unsigned same = __match_any_sync(~0u, id);
      if (ok && (31 - __clz(same)) == lane) {
        const int h = insert(id);
        if (h < 0) flags |= kFSlow;
        else H[h].y = (H[h].y & 0xFFFFFu) | ((unsigned)(j - d.q.blo + 1) << 20);
      }
      __syncwarp();
    }
  }
  if (flags) atomicOr(reinterpret_cast<unsigned*>(&sm.ci[1]), flags);
  cbar();
  if (sm.ci[0] > kPrepMax) {
    if (threadIdx.x == 0) sm.ci[1] |= (int)kFSlow;
    cbar();
  }
  flags = (unsigned)sm.ci[1];
  if (!(flags & kFSlow)) {
    Ent* base = P.ent + (size_t)row * C * kEnt;
    for (int i = threadIdx.x; i < kPrepSlots; i += kCT) {
      const uint2 sl = H[i];
      if (!sl.x) continue;
      const int id = (int)sl.x - 1;
      const int sli = id / kSL;
      const int p = atomicAdd(&sm.scnt[sli], 1);
      const unsigned cnt = sl.y & 0xFFFFFu, bj = sl.y >> 20;
      if (cnt > 0x7FFFu) {
        atomicOr(reinterpret_cast<unsigned*>(&sm.ci[1]), kFSlow);
        continue;
      }
      if (p < kEnt - 1) {
        Ent e;
        e.lid = (uint16_t)(id - sli * kSL);
        e.cnt = (uint16_t)(cnt | (bj ? 0x8000u : 0u));
        e.bias = bj ? __ldg(a.bias_vals + d.q.blo + (int)bj - 1) : 0.0f;
        base[(size_t)sli * kEnt + 1 + p] = e;
      }
    }
    cbar();
    if (threadIdx.x < C) {
      const int nE = sm.scnt[threadIdx.x];
      if (nE > kEnt - 1) atomicOr(reinterpret_cast<unsigned*>(&sm.ci[1]), kFSlow);
      Ent h;
      h.lid = (uint16_t)min(nE, kEnt - 1);
      h.cnt = 0;
      h.bias = 0.0f;
      base[(size_t)threadIdx.x * kEnt] = h;
    }
    cbar();
    flags = (unsigned)sm.ci[1];
  }
  if (threadIdx.x == 0) {
    __threadfence();
    st_rel64(&P.prep[row], ((unsigned long long)flags << 32) | P.epoch);
  }
}

// ---------------------------------------------------------------- row end (consumers)

__device__ __forceinline__ unsigned long long item_key(float z, int id) {
  return ((unsigned long long)fkey(z) << 32) | (unsigned)(~(unsigned)id);
}
__device__ __forceinline__ float key_z(unsigned long long k) { return key_to_float((uint32_t)(k >> 32)); }
__device__ __forceinline__ int key_id(unsigned long long k) { return (int)~(uint32_t)k; }

constexpr int kIPT = kItemCap / kCT;  // row-end items per consumer thread (item i: thread i % kCT)

// Row-end items in shared memory: (order key of y) << 32 | ~id, so a larger entry is a
// larger y, then a lower id.
__device__ __forceinline__ uint32_t ikey(unsigned long long e) { return (uint32_t)(e >> 32); }
__device__ __forceinline__ int iid(unsigned long long e) { return (int)~(uint32_t)e; }

// The k-th largest (1-based) of the keys of the items x[0..n) with key >= lo, counting
// repeats: rounds of 8-bit digits from the highest bit in which kmin and kmax differ
// down (the bits above it are common to every key, and skipping them spreads the first
// round over its digits instead of piling the items onto one), each a count histogram
// over the items whose higher bits match.  Every consumer thread gets the key.
__device__ uint32_t select_kth(const unsigned long long* x, int n, uint32_t lo, uint32_t kmin, uint32_t kmax,
                               int k) {
  if (kmin == kmax) return kmin;
  // bits at or above `fixed` are known; each round takes the 8 (or fewer) bits below them
  int fixed = 32 - __clz(kmin ^ kmax);
  uint32_t prefix = fixed >= 32 ? 0u : (kmin & ~((1u << fixed) - 1u));
  int rem = k;
  const int lane = threadIdx.x & 31;
  while (fixed > 0) {
    const int sh = fixed > 8 ? fixed - 8 : 0;
    const uint32_t dm = (1u << (fixed - sh)) - 1u;
    const uint32_t hm = fixed >= 32 ? 0u : ~((1u << fixed) - 1u);
    sm.hist[threadIdx.x] = 0u;
    cbar();
    for (int i = threadIdx.x; i < n; i += kCT) {
      const uint32_t key = ikey(x[i]);
      if (key >= lo && (key & hm) == (prefix & hm)) atomicAdd(&sm.hist[(key >> sh) & dm], 1u);
    }
    cbar();
    if (threadIdx.x < 32) {
      // lane l owns digits 255 - 8l .. 248 - 8l; counts from the top
      unsigned c8[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c8[j] = sm.hist[255 - (lane * 8 + j)];
        tot += c8[j];
      }
      unsigned incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_up_sync(~0u, incl, o);
        if (lane >= o) incl += t;
      }
      unsigned above = incl - tot;
      if (above < (unsigned)rem && (unsigned)rem <= incl) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (above < (unsigned)rem && (unsigned)rem <= above + c8[j]) {
            sm.ci[12] = 255 - (lane * 8 + j);
            sm.ci[13] = rem - (int)above;
          }
          above += c8[j];
        }
      }
    }
    cbar();
    prefix |= (uint32_t)sm.ci[12] << sh;
    rem = sm.ci[13];
    fixed = sh;
  }
  return prefix;
}

// The top-p threshold among the items with key >= lo: the smallest key g of such an item
// with A (the mass of everything above the items) plus the mass of the items with a key
// above g below T.  Items with a key of at least g are kept: a tie group (one key) stays
// iff the mass strictly above it is below T.  Rounds of 8-bit digits with exact 64-bit
// digit masses, from the highest bit in which the keys differ.
__device__ uint32_t select_mass(const unsigned long long* x, int n, uint32_t lo, uint32_t kmin, uint32_t kmax,
                                unsigned long long A, unsigned long long T) {
  if (kmin == kmax) return A < T ? kmin : 0xFFFFFFFFu;
  int fixed = 32 - __clz(kmin ^ kmax);
  uint32_t prefix = fixed >= 32 ? 0u : (kmin & ~((1u << fixed) - 1u));
  const int lane = threadIdx.x & 31;
  while (fixed > 0) {
    const int sh = fixed > 8 ? fixed - 8 : 0;
    const uint32_t dm = (1u << (fixed - sh)) - 1u;
    const uint32_t hm = fixed >= 32 ? 0u : ~((1u << fixed) - 1u);
    sm.hist[threadIdx.x] = 0u;
    sm.hmass[threadIdx.x] = 0ull;
    cbar();
    for (int i = threadIdx.x; i < n; i += kCT) {
      const uint32_t key = ikey(x[i]);
      if (key >= lo && (key & hm) == (prefix & hm)) {
        const unsigned dg = (key >> sh) & dm;
        atomicAdd(&sm.hist[dg], 1u);
        atomicAdd(&sm.hmass[dg], weight_fx(key_to_float(key)));
      }
    }
    cbar();
    if (threadIdx.x < 32) {
      // the lowest non-empty digit whose mass above (A plus the higher digits) is below T
      unsigned long long m8[8], tot = 0;
      unsigned c8[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        m8[j] = sm.hmass[255 - (lane * 8 + j)];
        c8[j] = sm.hist[255 - (lane * 8 + j)];
        tot += m8[j];
      }
      unsigned long long incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(~0u, incl, o);
        if (lane >= o) incl += t;
      }
      unsigned long long before = A + incl - tot;
      int best = -1;
      unsigned long long best_before = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (c8[j] && before < T) {
          best = 255 - (lane * 8 + j);
          best_before = before;
        }
        before += m8[j];
      }
      // lanes hold descending digit ranges: the highest lane with a candidate has the lowest digit
      const unsigned has = __ballot_sync(~0u, best >= 0);
      if (has) {
        const int src = 31 - __clz(has);
        const int dgt = __shfl_sync(~0u, best, src);
        const unsigned long long bb = __shfl_sync(~0u, best_before, src);
        if (lane == 0) {
          sm.ci[12] = dgt;
          sm.cu[2] = bb;
        }
      } else if (lane == 0) {
        sm.ci[12] = -1;
      }
    }
    cbar();
    const int dgt = sm.ci[12];
    if (dgt < 0) return 0xFFFFFFFFu;  // nothing stays (cannot happen while A < T)
    prefix |= (uint32_t)dgt << sh;
    A = sm.cu[2];
    fixed = sh;
  }
  return prefix;
}

// z' of the token `tok` among the row's items in global memory (the drawn token's
// original logprob needs it); every consumer thread gets it.
__device__ float find_z(const Item* g, int n, int tok) {
  if (threadIdx.x == 0) sm.cf[11] = NAN;
  cbar();
  for (int i = threadIdx.x; i < n; i += kCT) {
    const int2 v = __ldcg(reinterpret_cast<const int2*>(g + i));
    if (v.y == tok) sm.cf[11] = __int_as_float(v.x);
  }
  cbar();
  return sm.cf[11];
}

// The row end of light rows (items = the slices' candidates) and of general-route rows
// with a compacted band (items = the band; the tokens above it were raced and summed by
// P3).  The cuts are thresholds on the key of y found by radix selects, no sort: top-k
// (every item with y at least the k-th largest), top-p (a tie group stays iff the mass
// strictly above it is below ceil(p W)), min-p; then the race over the kept items.
__device__ void task_fin(const KP& P, const Desc& d, float* buf) {
  const clsample_args_t& a = P.a;
  const int row = d.row, C = P.C;
  const Params& q = d.q;
  RowState& R = P.rs[row];
  if (threadIdx.x == 0) {
    sm.cf[0] = __ldcg(&R.m);
    sm.cf[1] = __ldcg(&R.lnS);
    sm.cf[2] = __ldcg(&R.lnS1);
    sm.ci[0] = __ldcg(&R.nal);
    sm.ci[1] = __ldcg(reinterpret_cast<const int*>(&R.pflags));
    sm.ci[2] = __ldcg(&R.krem);
    sm.ci[3] = (int)__ldcg(&R.nitems);
    sm.cu[0] = __ldcg(&R.W);
    sm.cu[1] = __ldcg(&R.wabove);
    sm.ci[4] = (int)__ldcg(&R.kabove);
    sm.cf[3] = __ldcg(&R.miny);
    sm.cf[4] = __ldcg(&R.sume);
    sm.cf[5] = __ldcg(&R.rs);
    sm.ci[5] = __ldcg(&R.rid);
    sm.cf[6] = __ldcg(&R.ry);
    sm.cf[7] = __ldcg(&R.rz);
    sm.ci[6] = (int)__ldcg(&R.flags);
  }
  if (threadIdx.x < C) sm.recs[threadIdx.x] = ldcg_t(P.r1 + (size_t)row * C + threadIdx.x);
  cbar();
  const float m = sm.cf[0], lnS = sm.cf[1], lnS1 = sm.cf[2];
  const int nal = sm.ci[0];
  const unsigned pf = (unsigned)sm.ci[1];
  const unsigned nf = ((unsigned)sm.ci[6] & kFNonFinite) ? kPNonFinite : 0u;
  // a light row's first row end takes the slices' candidates; every other row end (a
  // general-route row, or a light row that fell back to it) takes its compacted band
  const bool fromband = (pf & kPBandCompact) != 0;
  const bool light = !fromband;
  const float invT = q.invT;
  unsigned long long* x = reinterpret_cast<unsigned long long*>(buf);
  int n = 0, kk = 0;
  Race above{-INFINITY, INT_MAX, 0.0f, 0.0f};
  unsigned long long mass_above = 0ull;
  int kept_above = 0;
  float miny_above = INFINITY, sume_above = 0.0f;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  auto put = [&](int i, const Item* src) {
    const int2 v = __ldcg(reinterpret_cast<const int2*>(src));
    const uint32_t key = fkey(y_of(__int_as_float(v.x), m, invT));
    x[i] = ((unsigned long long)key << 32) | (unsigned)(~(unsigned)v.y);
    kmin = min(kmin, key);
    kmax = max(kmax, key);
  };
  if (fromband) {
    n = sm.ci[3];
    kk = sm.ci[2];
    mass_above = sm.cu[1];
    kept_above = sm.ci[4];
    miny_above = sm.cf[3];
    sume_above = sm.cf[4];
    above = Race{sm.cf[5], sm.ci[5], sm.cf[6], sm.cf[7]};
    const Item* g = P.band + (size_t)row * kItemCap;
    for (int i = threadIdx.x; i < n; i += kCT) put(i, g + i);
  } else {
    // light row: the candidates of every slice; fall back to the general route when they
    // do not fit, or when the kept set may hold tokens no slice compacted
    int total = 0, all_taken = 1;
    for (int s = 0; s < C; ++s) {
      const Rec1& r = sm.recs[s];
      if (r.flags & kFSpill) total = kItemCap + 1;
      total += r.ncand;
      if (r.bound > -INFINITY) all_taken = 0;
    }
    const int kcut = (q.k >= 2 && q.k < nal) ? q.k : 0;
    if (total > kItemCap || (!kcut && !all_taken)) {
      if (threadIdx.x == 0) start_general(P, row, q, nal, nf);
      return;
    }
    int off = 0;
    for (int s = 0; s < C; ++s) {
      const Item* g = P.cand + ((size_t)row * C + s) * kCand;
      const int c = sm.recs[s].ncand;
      for (int i = threadIdx.x; i < c; i += kCT) put(off + i, g + i);
      off += c;
    }
    n = off;
    kk = kcut;
  }
  // key range of the items (the radix selects skip the bits they all share)
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(~0u, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(~0u, kmax, o));
  }
  cbar();
  if ((threadIdx.x & 31) == 0) {
    sm.ri[threadIdx.x >> 5] = (int)kmin;
    sm.ri[kCW + (threadIdx.x >> 5)] = (int)kmax;
  }
  cbar();
  kmin = 0xFFFFFFFFu;
  kmax = 0u;
  for (int i = 0; i < kCW; ++i) {
    kmin = min(kmin, (uint32_t)sm.ri[i]);
    kmax = max(kmax, (uint32_t)sm.ri[kCW + i]);
  }
  // top-k: every item with y at least the kk-th largest
  uint32_t tk = 0u;
  if (kk > 0 && kk < n) {
    tk = select_kth(x, n, 0u, kmin, kmax, kk);
    if (light) {
      // the candidates hold the row's whole top-k set iff every slice whose bound was
      // below its top-k share left only tokens under y_k
      const float Yk = key_to_float(tk);
      int ok = 1;
      if (threadIdx.x < C) {
        const Rec1& r = sm.recs[threadIdx.x];
        const int nS = min(kSL, a.V - (int)threadIdx.x * kSL);
        if (r.bound > -INFINITY && light_q(q.k, nS, a.V) < q.k)
          ok = y_of(nextafterf(r.bound, -INFINITY), m, invT) < Yk;
      }
      if (cbar_or(!ok)) {
        if (threadIdx.x == 0) start_general(P, row, q, nal, nf);
        return;
      }
    }
  } else if (kk > 0 && light) {
    // fewer candidates than k: only valid when every slice took all of its candidates
    int all_taken = 1;
    for (int s = 0; s < C; ++s) all_taken &= !(sm.recs[s].bound > -INFINITY);
    if (!all_taken) {
      if (threadIdx.x == 0) start_general(P, row, q, nal, nf);
      return;
    }
  }
  // top-p over the top-k set (or the band, with the exact mass above it)
  uint32_t tp = 0u;
  if (q.p < 1.0f && n > 0) {
    unsigned long long W = sm.cu[0];
    if (!(pf & kPWKnown)) {
      unsigned long long mine = 0ull;
      for (int i = threadIdx.x; i < n; i += kCT) {
        const uint32_t key = ikey(x[i]);
        if (key >= tk) mine += weight_fx(key_to_float(key));
      }
      W = mass_above + csum(mine, sm.ru);
    }
    tp = select_mass(x, n, tk, max(kmin, tk), kmax, mass_above, ceil_scaled(W, q.p));
  }
  // min-p and the race over the kept items
  const uint32_t cut_key = max(tk, tp);
  Race r{-INFINITY, INT_MAX, 0.0f, 0.0f};
  float sk = 0.0f, ymin = INFINITY;
  int kept = 0;
  for (int i = threadIdx.x; i < n; i += kCT) {
    const unsigned long long it = x[i];
    const uint32_t key = ikey(it);
    const float y = key_to_float(key);
    if (key < cut_key || !(y >= q.L)) continue;
    const int id = iid(it);
    const uint4 w4 = race_words((uint32_t)id >> 2, q.seed, q.pos);
    const float sc = race_score(y, pick_word(w4, id & 3));
    if (better(sc, id, r.s, r.id)) r = Race{sc, id, y, 0.0f};
    sk += ex2_approx(y * 1.4426950408889634f);
    ymin = fminf(ymin, y);
    ++kept;
  }
  r = crace(r);
  sk = csum(sk, sm.rf);
  ymin = cmin_f(ymin);
  kept = csum(kept, sm.ri);
  if (r.id != INT_MAX && above.id != INT_MAX && better(above.s, above.id, r.s, r.id)) r = above;
  else if (r.id == INT_MAX) r = above;
  if (r.id != INT_MAX && P.want_orig && !(r.id == above.id && above.id != INT_MAX)) {
    // z' of a drawn item, from the items in global memory
    r.z = fromband ? find_z(P.band + (size_t)row * kItemCap, n, r.id) : 0.0f;
    if (!fromband) {
      float z = NAN;
      for (int s = 0; s < C && z != z; ++s) {
        const float zs = find_z(P.cand + ((size_t)row * C + s) * kCand, sm.recs[s].ncand, r.id);
        if (zs == zs) z = zs;
      }
      r.z = z;
    }
  }
  if (threadIdx.x == 0) {
    kept += kept_above;
    if (r.id == INT_MAX || kept == 0) {
      row_fail(P, row, CLSAMPLE_ROW_OVERFLOW);
    } else {
      const float cut = fminf(ymin, miny_above);
      const float lp = r.y - lnS;
      const float lpo = __fsub_rn(r.z, m) - lnS1;
      const float lpk = r.y - logf(sk + sume_above);
      write_out(P, row, CLSAMPLE_ROW_OK, r.id, lp, kept, cut, lpo, lpk);
    }
  }
}

// ---------------------------------------------------------------- coordinator: row steps

// After the last P1 slice of a row: combine the records (lane s holds slice s).
__device__ void after_p1(const KP& P, int row) {
  const int lane = threadIdx.x & 31, C = P.C;
  Rec1 r{-INFINITY, INT_MAX, 0.0f, 0.0f, 0, -INFINITY, 0, 0u};
  if (lane < C) r = ldcg_t(P.r1 + (size_t)row * C + lane);
  Params q;
  unsigned rfl = 0u;
  if (lane == 0) {
    load_params(P.a, row, q);
    if (P.lists) rfl = (unsigned)(__ldcg(P.prep + row) >> 32);
  }
  const float M = warp_max_f(r.m);
  const unsigned hit = __ballot_sync(~0u, r.m == M && M > -INFINITY);
  const int arg = hit ? __shfl_sync(~0u, r.arg, __ffs(hit) - 1) : INT_MAX;
  const int nal = warp_sum(r.nal);
  const unsigned flags = warp_or(r.flags);
  // sums rescaled to the row max (lane order, a fixed shuffle tree)
  const float invT_l = __shfl_sync(~0u, lane == 0 ? q.invT : 0.0f, 0);
  const float c = __fmul_rn(1.4426950408889634f, invT_l);
  float S = (M > -INFINITY && r.m > -INFINITY) ? r.s * ex2_approx((r.m - M) * c) : 0.0f;
  float S1 = (M > -INFINITY && r.m > -INFINITY) ? r.s1 * ex2_approx((r.m - M) * 1.4426950408889634f) : 0.0f;
  S = warp_sum(S);
  S1 = warp_sum(S1);
  if (lane != 0) return;
  const unsigned fl = flags | rfl;
  if (q.invalid || (fl & kFInvalid) || !(M > -INFINITY) || nal == 0) {
    row_fail(P, row, CLSAMPLE_ROW_INVALID);
    return;
  }
  if (fl & kFOverflow) {
    row_fail(P, row, CLSAMPLE_ROW_OVERFLOW);
    return;
  }
  const float lnS = logf(S), lnS1 = logf(S1);
  if (q.cls == kClsGreedy) {
    write_out(P, row, CLSAMPLE_ROW_OK, arg, 0.0f - lnS, 1, 0.0f, 0.0f - lnS1, 0.0f);
    return;
  }
  RowState& R = P.rs[row];
  R.m = M;
  R.invT = q.invT;
  R.lnS = lnS;
  R.lnS1 = lnS1;
  R.arg = arg;
  R.nal = nal;
  R.flags = fl;
  R.pflags = 0u;
  const unsigned nf = (fl & kFNonFinite) ? kPNonFinite : 0u;
  if ((q.cls == kClsLight || q.cls == kClsBigK) && !(fl & kFSpill)) {
    push_tasks(P, row, kFin, 1);
    return;
  }
  start_general(P, row, q, nal, nf);
}

// After the last P2 slice of a round: plan the next pass from the bins (lane 0).
__device__ void after_p2(const KP& P, int row) {
  const int lane = threadIdx.x & 31;
  const RowBins& G = P.bins[row];
  RowState& R = P.rs[row];
  {
    const unsigned pf0 = __ldcg(&R.pflags), lo0 = __ldcg(&R.lo), hi0 = __ldcg(&R.hi);
    for (int b = lane; b < kBins; b += 32) {
      sm.kcnt[b] = __ldcg(&G.cnt[b]);
      sm.kcm[b] = __ldcg(&G.cm[b]);
      sm.kshift[b] = (unsigned)bin_shift(pf0, lo0, hi0, b);
    }
  }
  __syncwarp();
  if (lane != 0) return;
  Params q;
  load_params(P.a, row, q);
  const unsigned phase = __ldcg(&R.phase), round = __ldcg(&R.round);
  const unsigned lo = __ldcg(&R.lo), hi = __ldcg(&R.hi);
  const unsigned pf = __ldcg(&R.pflags);
  const unsigned nf = pf & kPNonFinite;
  const int kcut = __ldcg(&R.kcut);
  const unsigned long long accW = __ldcg(&R.accW), accMass = __ldcg(&R.accMass);
  const unsigned accCount = __ldcg(&R.accCount);
  const bool pcut = q.p < 1.0f;
  if (round >= (unsigned)kMaxRounds) {
    row_fail(P, row, CLSAMPLE_ROW_OVERFLOW);
    return;
  }
  auto zero = [&]() {
    R.accW = 0ull;
    R.accMass = 0ull;
    R.accCount = 0u;
    RowBins& Gw = P.bins[row];
    for (int b = 0; b < kBins; ++b) {
      Gw.cnt[b] = 0u;
      Gw.cm[b] = 0ull;
    }
  };
  auto refine = [&](unsigned nlo, unsigned nhi, unsigned flags) {
    R.round = round + 1u;
    R.lo = nlo;
    R.hi = nhi;
    R.pflags = flags | nf;
    zero();
    push_tasks(P, row, kP2, P.C);
  };
  auto p3 = [&](unsigned blo, unsigned bhi, unsigned flags, int krem) {
    R.blo = blo;
    R.bhi = bhi;
    R.pflags = flags | nf;
    R.krem = krem;
    R.nitems = 0u;
    push_tasks(P, row, kP3, P.C);
  };
  if (phase == kPhK) {
    unsigned cum = accCount;
    int bk = -1;
    for (int b = 0; b < kBins; ++b) {
      if (cum + sm.kcnt[b] >= (unsigned)kcut) {
        bk = b;
        break;
      }
      cum += sm.kcnt[b];
    }
    if (bk < 0) {
      row_fail(P, row, CLSAMPLE_ROW_OVERFLOW);
      return;
    }
    unsigned blo, bhi;
    bin_range(pf, lo, hi, bk, &blo, &bhi);
    if (bhi - blo == 1u) {
      // the k-th largest y is resolved: every token at or above it is in S_k
      if (pcut) {
        R.phase = kPhP;
        R.excl = bhi;
        R.round = 0u;
        R.lo = 0u;
        R.hi = fkey(0.0f);
        R.pflags = kPQuarter | kPMass | nf;
        zero();
        push_tasks(P, row, kP2, P.C);
      } else {
        R.excl = bhi;
        p3(bhi - 1u, bhi - 1u, 0u, 0);
      }
      return;
    }
    if (!pcut && sm.kcnt[bk] <= (unsigned)kItemCap) {
      p3(blo, bhi, kPBandCompact, kcut - (int)cum);
      return;
    }
    if (pcut && cum + sm.kcnt[bk] <= (unsigned)kItemCap) {
      p3(blo, 0xFFFFFFFFu, kPBandCompact, kcut);
      return;
    }
    refine(blo, bhi, 0u);
    return;
  }
  // phase P: the top-p crossing, from exact counts and bracketed masses
  const unsigned long long T = ceil_scaled(accW, q.p);
  R.W = accW;
  unsigned long long lo_cum = accMass, hi_cum = accMass;
  int bf = -1, bl = -1, last_kept = -1;
  for (int b = 0; b < kBins; ++b) {
    const unsigned cnt = sm.kcnt[b];
    if (!cnt) continue;
    const unsigned long long cm = sm.kcm[b];
    const unsigned sh = sm.kshift[b];
    const unsigned long long a_lo = lo_cum + (cm << sh), a_hi = hi_cum + ((cm + cnt) << sh);
    const bool dropped = lo_cum >= T, kept = a_hi < T;
    if (kept) last_kept = b;
    if (!dropped && !kept) {
      if (bf < 0) bf = b;
      bl = b;
    }
    lo_cum = a_lo;
    hi_cum = a_hi;
  }
  if (bf < 0) {
    // the cut falls on a bin edge: everything in and above the last kept bin stays
    unsigned blo, bhi;
    if (last_kept < 0) {
      row_fail(P, row, CLSAMPLE_ROW_OVERFLOW);
      return;
    }
    bin_range(pf, lo, hi, last_kept, &blo, &bhi);
    p3(blo, blo, 0u, 0);
    return;
  }
  unsigned cnt_band = 0u;
  for (int b = bf; b <= bl; ++b) cnt_band += sm.kcnt[b];
  unsigned lo_b, hi_b, t0, t1;
  bin_range(pf, lo, hi, bl, &lo_b, &t0);
  bin_range(pf, lo, hi, bf, &t1, &hi_b);
  if (cnt_band <= (unsigned)kItemCap) {
    p3(lo_b, hi_b, kPBandCompact | kPNeedAbove | kPWKnown, 0);
    return;
  }
  if (hi_b - lo_b == 1u) {
    p3(lo_b, hi_b, kPBandRace | kPNeedAbove | kPWKnown, 0);
    return;
  }
  refine(lo_b, hi_b, kPMass);
}

// After the last P3 slice: combine the slices' races and sums; finish the row or queue
// its band end.
__device__ void after_p3(const KP& P, int row) {
  const int lane = threadIdx.x & 31, C = P.C;
  Rec3 r;
  r.rs = -INFINITY;
  r.rid = INT_MAX;
  r.ry = r.rz = 0.0f;
  r.wabove = 0ull;
  r.nabove = r.kabove = 0u;
  r.miny = INFINITY;
  r.sume = 0.0f;
  r.bs = -INFINITY;
  r.bid = INT_MAX;
  r.by = r.bz = 0.0f;
  r.bk = 0u;
  r.bminy = INFINITY;
  r.bsume = 0.0f;
  if (lane < C) r = ldcg_t(P.r3 + (size_t)row * C + lane);
  // best above and best in the band (score, then lower id)
  unsigned long long ka = r.rid == INT_MAX ? 0ull : race_key(r.rs, r.rid);
  unsigned long long kb = r.bid == INT_MAX ? 0ull : race_key(r.bs, r.bid);
  unsigned long long ma = ka, mb = kb;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    ma = max(ma, __shfl_xor_sync(~0u, ma, o));
    mb = max(mb, __shfl_xor_sync(~0u, mb, o));
  }
  const unsigned ha = __ballot_sync(~0u, ma != 0ull && ka == ma), hb = __ballot_sync(~0u, mb != 0ull && kb == mb);
  const int la = ha ? __ffs(ha) - 1 : 0, lb = hb ? __ffs(hb) - 1 : 0;
  Race A{__shfl_sync(~0u, r.rs, la), ma ? __shfl_sync(~0u, r.rid, la) : INT_MAX, __shfl_sync(~0u, r.ry, la),
         __shfl_sync(~0u, r.rz, la)};
  Race Bd{__shfl_sync(~0u, r.bs, lb), mb ? __shfl_sync(~0u, r.bid, lb) : INT_MAX, __shfl_sync(~0u, r.by, lb),
          __shfl_sync(~0u, r.bz, lb)};
  const unsigned long long wab = warp_sum(r.wabove);
  const unsigned kab = warp_sum(r.kabove), bk = warp_sum(r.bk);
  const float miny = warp_min_f(r.miny), bminy = warp_min_f(r.bminy);
  const float sume = warp_sum(r.sume), bsume = warp_sum(r.bsume);
  if (lane != 0) return;
  RowState& R = P.rs[row];
  const unsigned pf = __ldcg(&R.pflags);
  if (pf & kPBandCompact) {
    if (__ldcg(&R.nitems) > (unsigned)kItemCap) {
      row_fail(P, row, CLSAMPLE_ROW_OVERFLOW);
      return;
    }
    R.rs = A.s;
    R.rid = A.id;
    R.ry = A.y;
    R.rz = A.z;
    R.wabove = wab;
    R.kabove = kab;
    R.miny = miny;
    R.sume = sume;
    push_tasks(P, row, kFin, 1);
    return;
  }
  Race w = A;
  unsigned kept = kab;
  float cut = miny, sk = sume;
  if (pf & kPBandRace) {
    // a single-value band: all of it stays iff the mass strictly above it is below ceil(p W)
    const float p = P.a.top_ps ? P.a.top_ps[row] : 1.0f;
    const unsigned long long T = ceil_scaled(__ldcg(&R.W), p);
    if (wab < T) {
      if (Bd.id != INT_MAX && better(Bd.s, Bd.id, w.s, w.id)) w = Bd;
      kept += bk;
      cut = fminf(cut, bminy);
      sk += bsume;
    }
  }
  if (w.id == INT_MAX || kept == 0u) {
    row_fail(P, row, CLSAMPLE_ROW_OVERFLOW);
    return;
  }
  const float m = __ldcg(&R.m), lnS = __ldcg(&R.lnS), lnS1 = __ldcg(&R.lnS1);
  write_out(P, row, CLSAMPLE_ROW_OK, w.id, w.y - lnS, (int)kept, cut, __fsub_rn(w.z, m) - lnS1, w.y - logf(sk));
}

// ---------------------------------------------------------------- roles

__device__ void producer(const KP& P) {
  const int lane = threadIdx.x & 31;
  const clsample_args_t& a = P.a;
  const uint64_t pol_first = make_policy_evict_first(), pol_last = make_policy_evict_last();
  const unsigned G = gridDim.x, q = blockIdx.x, seg = queue_seg(P);
  const DSlot* myq = P.dq + (size_t)q * seg;
  unsigned my_pos = 0;  // next entry of this CTA's queue
  bool static_done = false;
  // the static list entry this producer takes next, claimed one task ahead so the
  // atomic's round trip overlaps the current task's loads
  unsigned next_static = 0xFFFFFFFFu;
  if (lane == 0) next_static = atomicAdd(&P.ctl->next, 1u);
  for (uint32_t s = 0;; ++s) {
    const int st = (int)(s % kNB);
    int ok = 1;
    if (lane == 0 && s >= (uint32_t)kNB) ok = mbar_wait_nap(&sm.empty[st], ((s / kNB) - 1u) & 1u);
    if (!__shfl_sync(~0u, ok, 0)) {
      if (lane == 0) atomicOr(&P.ctl->err, 8u);
      break;
    }
    uint32_t row = 0, code = kExit;
    if (lane == 0) {
      unsigned lpos = 0xFFFFFFFFu;
      for (uint32_t polls = 0;; ++polls) {
        // this CTA's queue first: tasks that became ready during the call
        const unsigned rr = ld_vol(&P.ctl->rr);
        const unsigned reserved = rr > q ? (rr - q - 1u) / G + 1u : 0u;
        if (my_pos < reserved) {
          const DSlot e = ld_acq64(myq + my_pos);
          if ((unsigned)e == P.epoch) {
            code = (uint32_t)(e >> 32) & 0xFFFFu;
            row = (uint32_t)(e >> 48);
            ++my_pos;
            break;
          }
        } else if (!static_done) {
          const unsigned i = next_static;
          if (i < (unsigned)P.total) {
            static_task(P, i, &row, &code, &lpos);
            next_static = atomicAdd(&P.ctl->next, 1u);
            break;
          }
          static_done = true;
          continue;
        } else if (ld_acq(&P.ctl->rows_done) >= (unsigned)P.B) {
          code = kExit;
          break;
        }
        if (polls > kPolls) {
          atomicOr(&P.ctl->err, 1u);
          code = kExit;
          break;
        }
        __nanosleep(polls < 64 ? 32 : 256);
      }
      Desc& d = sm.desc[st];
      const uint32_t ph = code & 15u;
      d.row = row;
      d.code = code;
      if (ph == kP1 || ph == kP2 || ph == kP3) {
        const int slice = (int)(code >> 4);
        const int c0 = slice * kSL, n = min(kSL, a.V - c0);
        d.slice = slice;
        d.c0 = c0;
        d.n = n;
        const unsigned char* src = static_cast<const unsigned char*>(a.logits) +
                                   ((long long)row * a.logits_row_stride + c0) * P.esize;
        const uint32_t bytes = (uint32_t)n * (uint32_t)P.esize;
        const bool bulk = ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) && (bytes % 16u == 0);
        d.plain = !bulk;
        unsigned char* dst = dyn + (size_t)st * kBuf + (P.esize == 2 ? kBuf / 2 : 0);
        // the slice's lines stay in L2 when the row takes more passes over it
        const bool keep = ph == kP2 || (ph == kP1 && lpos < (unsigned)sm.cls_start[kClsBigK]);
        if (bulk) {
          mbar_expect_tx(&sm.full[st], bytes);
          bulk_copy_g2s_hint(dst, src, bytes, &sm.full[st], keep ? pol_last : pol_first);
        }
        d.mplain = 0;
        if (P.masked) {
          const int32_t* msrc = a.bitmask + (long long)row * a.bitmask_row_stride + (c0 >> 5);
          const uint32_t mb = (uint32_t)((n + 31) >> 5) * 4u;
          if ((reinterpret_cast<uintptr_t>(msrc) & 15u) == 0 && mb % 16u == 0) {
            mbar_expect_tx(&sm.full[st], mb);
            bulk_copy_g2s_hint(sm.mask[st], msrc, mb, &sm.full[st], pol_first);
          } else {
            d.mplain = 1;
          }
        }
        // independent loads: the row's parameters, its plan (later passes), its lists' flag
        load_params(a, row, d.q);
        if (ph != kP1) {
          const RowState& R = P.rs[row];
          d.m = __ldcg(&R.m);
          d.lo = __ldcg(&R.lo);
          d.hi = __ldcg(&R.hi);
          d.excl = __ldcg(&R.excl);
          d.blo = __ldcg(&R.blo);
          d.bhi = __ldcg(&R.bhi);
          d.pflags = __ldcg(&R.pflags);
        }
        d.rflags = 0u;
        if (P.lists) {
          // the row's lists: the producer waits for them (never a consumer: a consumer
          // waiting in front of a preparation task in its own ring could wait forever)
          unsigned long long pw = ld_acq64(P.prep + row);
          for (uint32_t polls = 0; (unsigned)pw != P.epoch && polls < kPolls; ++polls) {
            __nanosleep(64);
            pw = ld_acq64(P.prep + row);
          }
          d.rflags = (unsigned)pw == P.epoch ? (unsigned)(pw >> 32) : kFSlow;
          if (!(d.rflags & kFSlow)) {
            // the lists were written by other CTAs' threads (generic proxy); the bulk
            // copy reads them through the async proxy
            asm volatile("fence.proxy.async.global;" ::: "memory");
            const Ent* eb = P.ent + ((size_t)row * P.C + slice) * kEnt;
            mbar_expect_tx(&sm.full[st], kEntStage * sizeof(Ent));
            bulk_copy_g2s_hint(sm.ents[st], eb, kEntStage * sizeof(Ent), &sm.full[st], pol_first);
          }
        }
      } else if (ph == kFin || ph == kPrep) {
        load_params(a, row, d.q);
      }
      mbar_arrive(&sm.full[st]);
    }
    code = __shfl_sync(~0u, code, 0);
    if ((code & 15u) == kExit) break;
  }
}

// Hands a finished slice to the coordinator.  False if the coordinator stopped taking
// notices (its bounded wait gave up): the caller then leaves, and the rows left report
// OVERFLOW at the end of the launch.
__device__ bool post_notice(uint32_t nq, uint32_t row, uint32_t code) {
  const int slot = (int)(nq % kNQ);
  if (nq >= (uint32_t)kNQ && !mbar_wait_nap(&sm.nempty[slot], ((nq / kNQ) - 1u) & 1u)) return false;
  sm.nrow[slot] = row;
  sm.ncode[slot] = code;
  mbar_arrive(&sm.nfull[slot]);
  return true;
}

__device__ void consumer(const KP& P) {
  uint32_t nq = 0;
  for (uint32_t s = 0;; ++s) {
    const int st = (int)(s % kNB);
    if (!mbar_wait_nap(&sm.full[st], (s / kNB) & 1u)) {
      // the producer stopped answering: leave (the rows left report OVERFLOW)
      if (threadIdx.x == 0) atomicOr(&P.ctl->err, 4u);
      break;
    }
    const Desc& d = sm.desc[st];
    // the task's identity, kept in registers: the descriptor belongs to the producer again
    // once the stage is released
    const uint32_t trow = d.row, tcode_ = d.code;
    const uint32_t ph = tcode_ & 15u;
    float* buf = reinterpret_cast<float*>(dyn + (size_t)st * kBuf);
    if (ph == kExit) {
      if (threadIdx.x == 0) post_notice(nq, 0u, kExit);
      break;
    }
    if (ph == kP1) task_p1(P, d, st, buf);
    else if (ph == kP2) task_p2(P, d, st, buf);
    else if (ph == kP3) task_p3(P, d, st, buf);
    else if (ph == kFin) task_fin(P, d, buf);
    else if (ph == kPrep) task_prep(P, d, buf);
    // this task's ordinary writes into the ring buffer are ordered before the bulk copy
    // that refills it (a different proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    cbar();
    int posted = 1;
    if (threadIdx.x == 0) {
      mbar_arrive(&sm.empty[st]);
      if (ph <= kP3) posted = post_notice(nq++, trow, tcode_);
      if (!posted) atomicOr(&P.ctl->err, 16u);
    }
    if (cbar_or(!posted)) break;
  }
}

__device__ void coordinator(const KP& P) {
  const int lane = threadIdx.x & 31;
  const unsigned C = (unsigned)P.C;
  for (uint32_t nq = 0;; ++nq) {
    const int slot = (int)(nq % kNQ);
    int ok = 1;
    if (lane == 0) ok = mbar_wait_nap(&sm.nfull[slot], (nq / kNQ) & 1u);
    if (!__shfl_sync(~0u, ok, 0)) break;
    const uint32_t row = sm.nrow[slot], code = sm.ncode[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.nempty[slot]);
    const uint32_t ph = code & 15u;
    if (ph == kExit) break;
    int last = 0;
    if (lane == 0) {
      __threadfence();
      unsigned* t = ph == kP1 ? &P.rs[row].t1 : ph == kP2 ? &P.rs[row].t2 : &P.rs[row].t3;
      last = atomicInc(t, C - 1u) == C - 1u;
      if (last) __threadfence();
    }
    last = __shfl_sync(~0u, last, 0);
    if (!last) continue;
    if (ph == kP1) after_p1(P, (int)row);
    else if (ph == kP2) after_p2(P, (int)row);
    else after_p3(P, (int)row);
    __syncwarp();
  }
}

__global__ void __launch_bounds__(kBlock, 2) stream_kernel(const __grid_constant__ KP P0) {
  const int warp = threadIdx.x >> 5;
  // this launch's epoch: one past the last finished launch's, never 0; the last CTA out
  // advances the device copy, after every CTA of this launch has read it
  __shared__ KP P;
  if (threadIdx.x == 0) {
    P = P0;
    const unsigned e = __ldcg(&P0.ctl->epoch) + 1u;
    P.epoch = e ? e : 1u;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNB; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < kNQ; ++i) {
      mbar_init(&sm.nfull[i], 1);
      mbar_init(&sm.nempty[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  build_order(P);
  __syncthreads();
  if (warp < kCW) consumer(P);
  else if (warp == kPW) producer(P);
  else coordinator(P);
  __syncthreads();
  // the last CTA out resets the call's counters; rows a failed poll left unfinished
  // report OVERFLOW
  // every write of this CTA (outputs, finish markers) is published before it counts out,
  // so the last CTA's sweep sees them
  if (threadIdx.x == 0) {
    __threadfence();
    sm.ci[0] = atomicInc(&P.ctl->exited, gridDim.x - 1u) == gridDim.x - 1u;
  }
  __syncthreads();
  if (sm.ci[0]) {
    __threadfence();
    for (int r = threadIdx.x; r < P.B; r += kBlock) {
      // tickets start the next launch at zero even if this one gave up on a row
      P.rs[r].t1 = 0u;
      P.rs[r].t2 = 0u;
      P.rs[r].t3 = 0u;
      if (__ldcg(&P.rs[r].done) != P.epoch) {
        const clsample_args_t& a = P.a;
        a.tokens[r] = -1;
        if (a.logprobs) a.logprobs[r] = -INFINITY;
        if (a.logprobs_orig) a.logprobs_orig[r] = -INFINITY;
        if (a.logprobs_kept) a.logprobs_kept[r] = -INFINITY;
        if (a.row_status) a.row_status[r] = CLSAMPLE_ROW_OVERFLOW;
        if (a.dbg_kept_count) a.dbg_kept_count[r] = 0;
        if (a.dbg_cut) a.dbg_cut[r] = -INFINITY;
      }
    }
    if (threadIdx.x == 0) {
      P.ctl->next = 0u;
      P.ctl->rr = 0u;
      P.ctl->rows_done = 0u;
      P.ctl->err = 0u;
      P.ctl->epoch = P.epoch;
    }
  }
}

// ---------------------------------------------------------------- host side

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
  size_t ctl, dq, rs, bins, r1, r3, cand, band, ent, prep, total;
  unsigned dq_cap;
};

constexpr size_t take(size_t& off, size_t bytes) {
  const size_t o = off;
  off = align_up(off + bytes, 256);
  return o;
}

Layout layout(size_t B, size_t C) {
  Layout L{};
  size_t off = 0;
  L.dq_cap = (unsigned)(B * (2 + (kMaxRounds + 2) * C) + kMaxGrid);
  L.ctl = take(off, sizeof(Ctl));
  L.dq = take(off, (size_t)L.dq_cap * sizeof(DSlot));
  L.rs = take(off, B * sizeof(RowState));
  L.bins = take(off, B * sizeof(RowBins));
  L.r1 = take(off, B * C * sizeof(Rec1));
  L.r3 = take(off, B * C * sizeof(Rec3));
  L.cand = take(off, B * C * kCand * sizeof(Item));
  L.band = take(off, B * kItemCap * sizeof(Item));
  L.ent = take(off, B * C * kEnt * sizeof(Ent));
  L.prep = take(off, B * sizeof(unsigned long long));
  L.total = off;
  return L;
}

int slices_for(int vocab) { return (vocab + kSL - 1) / kSL; }

std::mutex g_setup_mutex;
int g_grid[64];

}  // namespace

bool serves(const clsample_args_t* a) {
  return a && !a->tid_offs && !a->top_ns && !(a->mode & CLSAMPLE_MODE_JOINT_TOPK_TOPP) && a->V <= kMaxVocab;
}

size_t scratch_bytes(int max_batch, int vocab) {
  const int rows = max_batch < kMaxRows ? max_batch : kMaxRows;
  return layout((size_t)(rows > 0 ? rows : 1), (size_t)slices_for(vocab)).total;
}

int setup(int dev, int* grid) {
  if (dev < 0 || dev >= 64) return CLSAMPLE_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_grid[dev]) {
    const int smem = kNB * kBuf;
    if (cudaFuncSetAttribute(stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaFuncSetAttribute(stream_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
      return CLSAMPLE_ERR_CUDA;
    int sms = 0, per = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, stream_kernel, kBlock, (size_t)smem) != cudaSuccess)
      return CLSAMPLE_ERR_CUDA;
    if (per < 1) return CLSAMPLE_ERR_DEVICE;
    g_grid[dev] = sms * per;
  }
  *grid = g_grid[dev];
  return CLSAMPLE_SUCCESS;
}

int launch(const clsample_args_t* a, unsigned char* scratch, int max_batch, int grid, cudaStream_t st) {
  const int C = slices_for(a->V);
  const int rows_cap = max_batch < kMaxRows ? max_batch : kMaxRows;
  const Layout L = layout((size_t)(rows_cap > 0 ? rows_cap : 1), (size_t)C);
  for (int r0 = 0; r0 < a->B; r0 += kMaxRows) {
    const int B = a->B - r0 < kMaxRows ? a->B - r0 : kMaxRows;
    KP P;
    std::memset(&P, 0, sizeof P);
    P.a = *a;
    clsample_args_t& s = P.a;
    const int es = a->logits_dtype == CLSAMPLE_LOGITS_BF16 ? 2 : 4;
    s.B = B;
    s.logits = static_cast<const unsigned char*>(a->logits) + (size_t)r0 * a->logits_row_stride * es;
    auto off = [&](auto* p) { return p ? p + r0 : p; };
    s.temperatures = off(a->temperatures);
    s.top_ks = off(a->top_ks);
    s.top_ps = off(a->top_ps);
    s.min_ps = off(a->min_ps);
    s.rep = off(a->rep);
    s.freq = off(a->freq);
    s.pres = off(a->pres);
    s.hist_offs = off(a->hist_offs);
    s.bias_offs = off(a->bias_offs);
    s.bitmask = a->bitmask ? a->bitmask + (size_t)r0 * a->bitmask_row_stride : nullptr;
    s.seeds = off(a->seeds);
    s.positions = off(a->positions);
    s.tokens = off(a->tokens);
    s.logprobs = off(a->logprobs);
    s.row_status = off(a->row_status);
    s.dbg_transformed = a->dbg_transformed ? a->dbg_transformed + (size_t)r0 * a->V : nullptr;
    s.dbg_kept_count = off(a->dbg_kept_count);
    s.dbg_cut = off(a->dbg_cut);
    s.logprobs_orig = off(a->logprobs_orig);
    s.logprobs_kept = off(a->logprobs_kept);
    P.B = B;
    P.C = C;
    P.esize = es;
    P.masked = a->bitmask != nullptr;
    P.lists = (a->hist_offs || a->bias_offs) ? 1 : 0;
    P.total = P.lists ? B + B * C : B * C;
    P.want_orig = a->logprobs_orig != nullptr;
    P.want_kept = a->logprobs_kept != nullptr;
    P.dq_cap = L.dq_cap;
    P.ctl = reinterpret_cast<Ctl*>(scratch + L.ctl);
    P.dq = reinterpret_cast<DSlot*>(scratch + L.dq);
    P.rs = reinterpret_cast<RowState*>(scratch + L.rs);
    P.bins = reinterpret_cast<RowBins*>(scratch + L.bins);
    P.r1 = reinterpret_cast<Rec1*>(scratch + L.r1);
    P.r3 = reinterpret_cast<Rec3*>(scratch + L.r3);
    P.cand = reinterpret_cast<Item*>(scratch + L.cand);
    P.band = reinterpret_cast<Item*>(scratch + L.band);
    P.ent = reinterpret_cast<Ent*>(scratch + L.ent);
    P.prep = reinterpret_cast<unsigned long long*>(scratch + L.prep);
    const int tasks = P.total;
    int g = grid < tasks ? grid : tasks;
    if (g > kMaxGrid) g = kMaxGrid;
    stream_kernel<<<g, kBlock, (size_t)kNB * kBuf, st>>>(P);
    if (cudaGetLastError() != cudaSuccess) return CLSAMPLE_ERR_CUDA;
  }
  return CLSAMPLE_SUCCESS;
}

}  // namespace clsample_stream
