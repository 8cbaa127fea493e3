// Batched constrained logits sampler for GB300 (sm_103a).
//
// A row's V logits are split into C slices of `chunk` tokens (a multiple of 128).  Two
// launches per call:
//
//   order_kernel    the preparation launch.  CTA 0 orders the rows (heavy rows first,
//                   greedy last), resets the call's counters and sets "order ready";
//                   CTAs 1..B each list one row's distinct penalised and biased tokens by
//                   slice (a shared-memory hash of the history ids with their counts and
//                   each id's last valid bias entry), count its allowed tokens, and set
//                   the row's flag.
//   sampler_kernel  one CTA per (row, slice), launched with programmatic serialisation
//                   (its CTAs start once every preparation CTA has started and wait only
//                   on those flags).  A CTA takes its item from a global counter (items
//                   are taken in list order whatever order the hardware starts CTAs in),
//                   copies the slice into shared memory with one TMA bulk copy and keeps
//                   it there:
//
//   transforms  the slice's listed tokens get penalties, then bias, in place;
//   pass A      the grammar mask (written back as -inf), the slice's max, lowest argmax
//               and sum of 2^((z' - max) log2(e) / T);
//   candidates  light rows (top-k with k <= kKMax, min-p with p = 1) compact a superset
//               of the tokens their row can keep to global scratch: for top-k about
//               1.2 k times the slice's share of the row's allowed tokens, bounded by the
//               warps' sorted per-thread maxima; for min-p everything above the slice's
//               bound, with a rounding margin.  The CTA that finishes the row's last slice
//               (a ticket counter) finishes the row alone: it checks every slice's bound
//               exactly against the row's k-th largest y (redoing a slice that fails),
//               sorts the candidates, takes the top-k, top-p (exact fixed-point mass) and
//               min-p cuts as prefixes, and runs the exponential race.
//   heavy rows  rows whose kept set may span the whole vocabulary (top-p without a small
//               top-k, or no truncation) keep their C CTAs together: they are first in the
//               list, and each CTA waits (bounded) at two row barriers -- after pass A for
//               the row max, and after exact per-slice y-bin counts and masses -- so the
//               slices race their surely-kept tokens in place and compact only the band
//               that holds the cut; the last arriver resolves the cut exactly.
//
// A CTA only ever waits for CTAs that took earlier items of its own row (running), or
// for preparation CTAs (all started before this grid), so no wait can deadlock; every
// wait is bounded.  The arithmetic that decides integers (kept set, drawn id) is exact
// and identical on any IEEE machine (sampler_math.cuh).  Page references: "SGLang source
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
#include "bulk_copy.cuh"
#include "sampler_math.cuh"

namespace {

using namespace clsample;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSliceMax = 15360;   // longest slice (tokens, multiple of 128)
constexpr int kMaxVocab = 262144;
constexpr int kMaxSlices = (kMaxVocab + kSliceMax - 1) / kSliceMax;
constexpr int kKMax = 1024;        // top-k rows with k <= kKMax finish from candidates
constexpr int kCandCap = 2048;     // compacted candidates per slice (global scratch)
constexpr int kPen = 512;          // penalised / biased tokens applied per round
constexpr int kHList = 1024;       // the slice's history ids cached in shared memory
constexpr int kYBins = 64;         // heavy rows: quarter-unit y bins, the last one open-ended
constexpr int kDigitBins = 2048;   // radix selects: 11-bit digits
constexpr uint32_t kWaitPolls = 1u << 22;  // row-barrier polls (about 1 us apart at most)

enum : int { kRowOk = 0, kRowOverflow = 1, kRowInvalid = 2 };
enum : int { kRouteGreedy = 0, kRouteTopK = 1, kRouteMinP = 2, kRouteHeavy = 3 };
enum : int { kFlagInvalid = 1, kFlagOverflow = 2 };

constexpr int kTopNMax = 32;  // top-N logprobs: largest N per row

struct Item {
  float z;  // transformed logit z'
  int id;   // token id
};

// Per-slice record, written by the slice's CTA and read by the row's finisher (and, for
// heavy rows, by the row's other CTAs after a barrier).
struct SliceRec {
  float m;       // slice max of z' (-inf if no token is allowed)
  int arg;       // lowest id reaching m
  float s;       // sum of 2^((z' - m) log2(e) / T) over allowed tokens
  int nallowed;  // allowed tokens
  int flags;     // kFlag*
  int ncand;     // compacted items (candidates, or a heavy row's band); > kCandCap: spilled
  float zc;      // light rows: the slice's candidate bound in z (-inf: every allowed token)
  float dz;      // its rounding margin (the finisher checks it against the row max)
  float rs;      // heavy rows: best race score of the slice's surely-kept tokens
  int rtok;      // its id (INT_MAX if none)
  int kept;      // surely-kept tokens of the slice that pass min-p
  float ymin;    // their smallest y
  float ytok;    // y of rtok
  int spilled;   // the items are in the row's spill area (else in the slice's candidates)
  float s1;      // sum of 2^((z' - m) log2(e)) over allowed tokens (T = 1; when requested)
  float skept;   // heavy rows: sum of e^y over the slice's surely-kept tokens
  float ztok;    // heavy rows: z' of rtok
  int pad[3];
};

// Per-row control words (reset by the ordering kernel every call).
struct RowCtl {
  unsigned ticket;  // slices that finished their last phase
  unsigned bar;     // heavy rows: arrivals at the row barriers
  int spill;        // spill slot of the row + 1 (0: none; see row_spill_slot)
  unsigned pad;
};

// Heavy rows: exact per-slice y-bin counts and masses.
struct Bins {
  unsigned cnt[kYBins];
  unsigned long long mass[kYBins];
};
// The same in shared memory, masses as split 32-bit words.
struct SBins {
  uint32_t cnt[kYBins];
  uint32_t lo[kYBins];
  uint32_t hi[kYBins];
  unsigned long long mass[kYBins];  // the row's summed masses (after barrier 2)
};

struct RowParams {
  float T, Teff, invT, p, mp, L, rep, freq, pres;
  int k;
  int route;
  int invalid;  // kFlagInvalid from the parameters
  unsigned long long seed, pos;
  int hlo, hhi, blo, bhi;  // CSR ranges (hhi < hlo: none / invalid handled by flags)
};

// One penalised or biased token of a row, as the preparation launch lists it (the
// entries of a slice are contiguous).
struct __align__(16) PenEntry {
  int lid;       // id within its slice
  unsigned cnt;  // occurrences in the history
  int bj;        // the last valid logit_bias entry of the id (-1: none)
  int pad;
};
constexpr int kPenRowCap = 8192;   // listed tokens per row (more: the slices scan themselves)
constexpr int kHashSlots = 4096;   // the preparation CTA's hash of a row's ids

// Per-row facts from the preparation launch.
struct RowInfo {
  int flags;  // kFlagInvalid: bad CSR offsets, ids out of range, NaN bias values
  int nal;    // allowed tokens by the bitmask (V without one)
  int ready;  // the row's entries are listed (else each slice scans the CSRs itself)
  int pad;
};

struct SweepRec;

struct LaunchParams {
  clsample_args_t a;
  int C;
  int chunk;
  int vec_ok;  // every row start is 16-byte aligned: slices arrive by TMA bulk copies
  int spill_rows;
  // scratch (device)
  unsigned* ctl;      // [0] next item, [1] spill slots taken, [2] order ready, [3] rows finished
  unsigned* rflag;    // [B] the row's entries are listed (preparation launch)
  int* order;         // [B] rows in list order
  RowCtl* rowctl;     // [B]
  SliceRec* srec;     // [B * C]
  Bins* bins;         // [B * C]
  Item* cand;         // [B * C][kCandCap]
  Item* spill;        // [spill_rows][C * chunk]
  RowInfo* rinfo;     // [B]
  int* poff;          // [B][C + 1] each slice's first entry
  PenEntry* pent;     // [B][kPenRowCap]
  int lists;          // the preparation launch wrote rinfo / poff / pent (penalties, bias or a mask)
  Item* topn;         // [B * C][kTopNMax] each slice's most probable tokens (top-N logprobs)
  // the single-sweep path's scratch
  int sw_c;           // its slices per row
  SweepRec* sw_rec;   // [B][kSwMaxC] slice records
  Item* sw_cand;      // [B][kSwMaxC][kSwCand] race candidates (z', id)
  unsigned* sw_tick;  // [B] row tickets, zero between calls
};

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Dynamic shared memory of one CTA (byte offsets):
//   buf    f32[chunk]           the slice (z' after the transforms and the mask); at a
//                               row end: finisher items, then its digit histogram
//   claim  u32[chunk/32]        penalised / biased tokens of the slice
//   prefix u16[chunk/32]        rank of each claim word's first token
//   aux    kAuxBytes            transforms: rank -> id, counts, bias entries;
//                               later: the top-k histogram, heavy y bins
constexpr size_t kAuxBytes = 5120;
constexpr int kFinHistBytes = 2048 * (4 + 8);        // the finisher's two digit histograms
constexpr int kBufMin = kFinHistBytes + 1024 * 8;    // room for them and 1024 items
// Bytes of buf: the slice, and at least the finisher's area.
__host__ __device__ constexpr int buf_bytes(int chunk) { return chunk * 4 > kBufMin ? chunk * 4 : kBufMin; }
struct Layout {
  uint32_t claim, prefix, hlist, mask, aux, total;
};
__host__ __device__ inline Layout layout_for(int chunk) {
  Layout L;
  size_t off = (size_t)buf_bytes(chunk);
  L.claim = (uint32_t)off;
  off = align_up(off + sizeof(uint32_t) * (size_t)(chunk / 32), 16);
  L.prefix = (uint32_t)off;
  off = align_up(off + sizeof(uint16_t) * (size_t)(chunk / 32), 16);
  L.hlist = (uint32_t)off;
  off = align_up(off + sizeof(uint16_t) * (size_t)kHList, 16);
  L.mask = (uint32_t)off;
  off = align_up(off + sizeof(uint32_t) * (size_t)(chunk / 32), 16);
  L.aux = (uint32_t)off;
  L.total = (uint32_t)(off + kAuxBytes);
  return L;
}
static_assert(kPen * (2 + 4 + 4) <= (int)kAuxBytes, "transform tables overflow aux");
static_assert(kThreads * 8 <= (int)kAuxBytes, "per-thread maxima overflow aux");
static_assert(sizeof(SBins) <= kAuxBytes, "y bins overflow aux");
static_assert(kSliceMax % 128 == 0 && kSliceMax <= 65535, "16-bit local ids and ranks");
static_assert(kMaxSlices <= 31, "slice sets are 32-bit masks");
static_assert(kFinHistBytes == kDigitBins * 12, "digit histograms: u32 counts and u64 masses");

extern __shared__ __align__(128) unsigned char smem_dyn[];

struct Smem {
  float* buf;
  uint32_t* claim;
  uint16_t* prefix;
  uint16_t* hlist;      // the slice's history ids (local), in scan order
  uint32_t* mask;       // the slice's bitmask words
  uint16_t* pid;        // aux: rank -> local id
  uint32_t* pcnt;       // aux: rank -> history count
  int* pbias;           // aux: rank -> last bias entry (-1: none)
  uint32_t* hist;       // aux: top-k histogram
  SBins* bins;          // aux: heavy y bins
};

__device__ __forceinline__ Smem carve(int chunk) {
  const Layout L = layout_for(chunk);
  unsigned char* b = smem_dyn;
  Smem s;
  s.buf = reinterpret_cast<float*>(b);
  s.claim = reinterpret_cast<uint32_t*>(b + L.claim);
  s.prefix = reinterpret_cast<uint16_t*>(b + L.prefix);
  s.hlist = reinterpret_cast<uint16_t*>(b + L.hlist);
  s.mask = reinterpret_cast<uint32_t*>(b + L.mask);
  s.pid = reinterpret_cast<uint16_t*>(b + L.aux);
  s.pcnt = reinterpret_cast<uint32_t*>(b + L.aux + 2 * kPen);
  s.pbias = reinterpret_cast<int*>(b + L.aux + 6 * kPen);
  s.hist = reinterpret_cast<uint32_t*>(b + L.aux);
  s.bins = reinterpret_cast<SBins*>(b + L.aux);
  return s;
}

// Static per-CTA state.
struct Shared {
  RowParams rp;
  SliceRec rec;            // this CTA's slice record
  SliceRec row;            // combined record of the row (heavy rows, finisher)
  unsigned long long bar;  // the slice copy's mbarrier
  unsigned bar_uses;       // its completed phases
  uint32_t bulk;           // bytes of the slice copy in flight (issued at entry)
  RowInfo ri;              // the row's preparation facts (valid when ri_ok)
  int ri_ok, e0, ne;       // ... and this slice's entry range
  int ri_slice;            // the slice they were loaded for
  float red_f[kWarps * 2];
  float red_f2[kWarps];
  int red_i[kWarps * 2];
  unsigned long long red_u[kWarps];
  int row_id, slice;
  int ntouch, flag, cnt, last, spill;
  int nhist;    // history ids of the slice (cached in hlist while at most kHList)
  int nal_row;  // light top-k rows with a mask: allowed tokens of the whole row (by the mask)
  // heavy rows: the bin plan
  int blo, bhi;
  unsigned above_n;
  unsigned long long above_w, W;
  float lnS, lnS1;  // ln of the row's normaliser at T, and at T = 1
  float ztok;       // z' of the drawn token (original logprob)
  // finisher
  SliceRec recs[kMaxSlices];
  const Item* seg[2 * kMaxSlices];
  int segn[2 * kMaxSlices];
  int nseg, fin_smem, fin_n;
  float zmin;
  int digit;
  unsigned long long digit_above;
};
__shared__ Shared sh;

// ---------------------------------------------------------------- block reductions

__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait until *p == v (acquire); false on timeout.
__device__ bool wait_flag(const unsigned* p, unsigned v);

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned ld_relaxed(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Orders the loads that follow after a relaxed load that saw a released value.
__device__ __forceinline__ void fence_acquire() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Ticket increment that publishes this thread's earlier writes (and, through a preceding
// block barrier, the CTA's) and, for the thread that sees the final count, acquires the
// other CTAs' writes: one round trip instead of a fence and an atomic.
__device__ __forceinline__ unsigned atomic_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ bool wait_flag(const unsigned* p, unsigned v) {
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    if (ld_acquire(p) == v) return true;
    __nanosleep(64);
  }
  return false;
}


__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fminf(v, __shfl_xor_sync(~0u, v, o));
  return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(~0u, v, o);
  return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(~0u, v, o);
  return v;
}
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(~0u, v, o);
  return v;
}

// (value, id) argmax of the block: larger value, then lower id.  All threads get it.
__device__ void block_argmax(float& v, int& id) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float v2 = __shfl_xor_sync(~0u, v, o);
    const int i2 = __shfl_xor_sync(~0u, id, o);
    if (better(v2, i2, v, id)) {
      v = v2;
      id = i2;
    }
  }
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    sh.red_f[w] = v;
    sh.red_i[w] = id;
  }
  __syncthreads();
  v = sh.red_f[0];
  id = sh.red_i[0];
  for (int i = 1; i < kWarps; ++i)
    if (better(sh.red_f[i], sh.red_i[i], v, id)) {
      v = sh.red_f[i];
      id = sh.red_i[i];
    }
}

__device__ int block_sum_i(int v) {
  v = warp_sum_i(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh.red_i[threadIdx.x >> 5] = v;
  __syncthreads();
  int r = 0;
  for (int i = 0; i < kWarps; ++i) r += sh.red_i[i];
  return r;
}
__device__ unsigned long long block_sum_u64(unsigned long long v) {
  v = warp_sum_u64(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh.red_u[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long r = 0;
  for (int i = 0; i < kWarps; ++i) r += sh.red_u[i];
  return r;
}
__device__ float block_min_f(float v) {
  v = warp_min(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh.red_f[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = sh.red_f[0];
  for (int i = 1; i < kWarps; ++i) r = fminf(r, sh.red_f[i]);
  return r;
}

__device__ uint32_t block_min_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(~0u, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh.red_i[threadIdx.x >> 5] = (int)v;
  __syncthreads();
  uint32_t r = (uint32_t)sh.red_i[0];
  for (int i = 1; i < kWarps; ++i) r = min(r, (uint32_t)sh.red_i[i]);
  return r;
}

// Exclusive prefix sum over the block (thread order); *total gets the sum.
__device__ int block_scan_i(int x, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int v = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(~0u, v, o);
    if (lane >= o) v += t;
  }
  __syncthreads();
  if (lane == 31) sh.red_i[w] = v;
  __syncthreads();
  int off = 0, tot = 0;
  for (int i = 0; i < kWarps; ++i) {
    if (i < w) off += sh.red_i[i];
    tot += sh.red_i[i];
  }
  *total = tot;
  return off + v - x;
}

// Exact 64-bit mass sums in shared memory with 32-bit atomics: the low word takes the
// addend's low half and reports its own wrap-around as a carry into the high word.
__device__ __forceinline__ void add_mass(uint32_t* lo, uint32_t* hi, unsigned long long w) {
  const uint32_t wl = (uint32_t)w, wh = (uint32_t)(w >> 32);
  uint32_t carry = 0u;
  if (wl) {
    const uint32_t old = atomicAdd(lo, wl);
    carry = (old + wl < old) ? 1u : 0u;
  }
  if (wh + carry) atomicAdd(hi, wh + carry);
}
__device__ __forceinline__ unsigned long long get_mass(const uint32_t* lo, const uint32_t* hi) {
  return ((unsigned long long)*hi << 32) + *lo;
}

// ---------------------------------------------------------------- block sort

// Compare-exchange of a bitonic stage: element i keeps max(a, partner) if it is the pair's
// first element in a descending block (or the second in an ascending one), else the min.
__device__ __forceinline__ unsigned long long bitonic_pick(unsigned long long a, unsigned long long o, int i, int size,
                                                           int stride) {
  const bool keep_max = ((i & stride) == 0) == ((i & size) == 0);
  return keep_max ? (a > o ? a : o) : (a < o ? a : o);
}

// Sorts np = 256 * E 64-bit keys at k (shared memory) in descending order, bitonic:
// thread t holds keys [t E, t E + E) in registers; strides below E swap inside a
// thread, strides below 32 E between lanes by shuffles, wider ones through shared memory
// (the only stages with a block barrier).  The stage loops stay rolled (small code); the
// in-thread strides are dispatched to fixed register pairs.
template <int E>
__device__ void block_sort_desc(unsigned long long* k) {
  constexpr int np = kThreads * E;
  const int t = threadIdx.x;
  unsigned long long v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = k[t * E + e];
#pragma unroll 1
  for (int size = 2; size <= np; size <<= 1) {
#pragma unroll 1
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 32 * E) {
#pragma unroll
        for (int e = 0; e < E; ++e) k[t * E + e] = v[e];
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = bitonic_pick(v[e], k[(t * E + e) ^ stride], t * E + e, size, stride);
        __syncthreads();
      } else if (stride >= E) {
        const int lm = stride / E;
#pragma unroll
        for (int e = 0; e < E; ++e)
          v[e] = bitonic_pick(v[e], __shfl_xor_sync(~0u, v[e], lm), t * E + e, size, stride);
      } else {
        unsigned long long w[E];
#pragma unroll
        for (int st = 1; st < E; st <<= 1) {
          if (st != stride) continue;
#pragma unroll
          for (int e = 0; e < E; ++e) w[e] = bitonic_pick(v[e], v[e ^ st], t * E + e, size, st);
#pragma unroll
          for (int e = 0; e < E; ++e) v[e] = w[e];
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) k[t * E + e] = v[e];
  __syncthreads();
}

// Sorts n <= 2048 keys (padded with zeros to 256 E) descending.
__device__ void sort_desc(unsigned long long* k, int n) {
  int np = kThreads;
  while (np < n) np <<= 1;
  for (int i = n + threadIdx.x; i < np; i += kThreads) k[i] = 0ull;
  __syncthreads();
  if (np <= kThreads) block_sort_desc<1>(k);
  else if (np <= 2 * kThreads) block_sort_desc<2>(k);
  else if (np <= 4 * kThreads) block_sort_desc<4>(k);
  else block_sort_desc<8>(k);
}

// ---------------------------------------------------------------- row parameters

// A row's parameters as read from memory (loads only: a kernel may issue them early and
// decode them when it needs them).
struct RawRow {
  float T, p, mp, rep, freq, pres;
  int k, h0, h1, b0, b1;
  unsigned long long seed, pos;
};
__device__ __forceinline__ RawRow load_raw(const clsample_args_t& a, int row) {
  RawRow w;
  w.T = a.temperatures ? a.temperatures[row] : 1.0f;
  w.k = a.top_ks ? a.top_ks[row] : -1;
  w.p = a.top_ps ? a.top_ps[row] : 1.0f;
  w.mp = a.min_ps ? a.min_ps[row] : 0.0f;
  w.rep = a.rep ? a.rep[row] : 1.0f;
  w.freq = a.freq ? a.freq[row] : 0.0f;
  w.pres = a.pres ? a.pres[row] : 0.0f;
  w.seed = a.seeds ? a.seeds[row] : 0ull;
  w.pos = (unsigned long long)(a.positions ? a.positions[row] : a.step);
  w.h0 = a.hist_offs ? a.hist_offs[row] : 0;
  w.h1 = a.hist_offs ? a.hist_offs[row + 1] : 0;
  w.b0 = a.bias_offs ? a.bias_offs[row] : 0;
  w.b1 = a.bias_offs ? a.bias_offs[row + 1] : 0;
  return w;
}

// Parameters, greedy rule and route of a row from its loaded values (every CTA of the
// row computes the same).
__device__ void decode_params(const clsample_args_t& a, const RawRow& w, RowParams& q) {
  q.T = w.T;
  q.k = w.k;
  q.p = w.p;
  q.mp = w.mp;
  q.rep = w.rep;
  q.freq = w.freq;
  q.pres = w.pres;
  q.seed = w.seed;
  q.pos = w.pos;
  int inv = 0;
  if (q.T != q.T || q.T == INFINITY) inv = 1;
  if (q.k < -1) inv = 1;
  if (!(q.p > 0.0f && q.p <= 1.0f)) inv = 1;
  if (!(q.mp >= 0.0f && q.mp <= 1.0f)) inv = 1;
  if (!(q.rep > 0.0f) || q.rep == INFINITY || !isfinite(q.freq) || !isfinite(q.pres)) inv = 1;
  q.hlo = 0;
  q.hhi = 0;
  if (a.hist_offs) {
    if (w.h0 < 0 || w.h1 < w.h0) inv = 1;
    else {
      q.hlo = w.h0;
      q.hhi = w.h1;
    }
  }
  q.blo = 0;
  q.bhi = 0;
  if (a.bias_offs) {
    if (w.b0 < 0 || w.b1 < w.b0) inv = 1;
    else {
      q.blo = w.b0;
      q.bhi = w.b1;
    }
  }
  q.invalid = inv ? kFlagInvalid : 0;
  const bool greedy = (q.T < kGreedyEps) || q.k == 0 || q.k == 1 || (a.mode & CLSAMPLE_MODE_SCORE_ONLY);
  // joint top-k/top-p needs the whole row's exact mass: the co-resident row-group route
  const bool joint = (a.mode & CLSAMPLE_MODE_JOINT_TOPK_TOPP) && q.p < 1.0f;
  q.Teff = (q.T >= kGreedyEps) ? q.T : 1.0f;
  q.invT = __fdiv_rn(1.0f, q.Teff);
  q.L = q.mp > 0.0f ? (float)log((double)q.mp) : -INFINITY;
  if (inv || greedy) q.route = kRouteGreedy;
  else if (q.k >= 2 && q.k <= kKMax && !joint) q.route = kRouteTopK;
  else if (q.p == 1.0f && q.mp > 0.0f) q.route = kRouteMinP;
  else q.route = kRouteHeavy;
}

__device__ void load_params(const clsample_args_t& a, int row, RowParams& q) { decode_params(a, load_raw(a, row), q); }

// List order of a row: heavy rows first (their CTAs wait for each other and work longest),
// then top-k rows with a large k (their row ends take longest), top-k rows with a top-p
// cut, other rows that finish from candidates, greedy and invalid rows last (the
// cheapest).
constexpr int kClasses = 5;
__device__ __forceinline__ int route_rank(const RowParams& q) {
  if (q.route == kRouteHeavy) return 0;
  if (q.route == kRouteTopK && q.k > 128) return 1;
  if (q.route == kRouteTopK && q.p < 1.0f) return 2;  // a top-p cut lengthens the row end
  return q.route == kRouteGreedy ? 4 : 3;
}

// ---------------------------------------------------------------- ordering kernel

constexpr int kOrderThreads = 512;
constexpr int kClassCache = 4096;  // rows whose class the ordering CTA keeps in shared memory

constexpr size_t kPrepSmem = (size_t)kHashSlots * 14;  // keys, counts, bias entries, slot list

// Hash slot of id (an empty slot holds 0; a taken one id + 1), -1 if the table is full;
// *created tells whether this call took the slot.
__device__ __forceinline__ int hash_insert(uint32_t* key, int id, bool* created) {
  uint32_t h = ((uint32_t)id * 2654435761u) >> 20;  // 12 bits: kHashSlots
  *created = false;
  for (int probe = 0; probe < kHashSlots; ++probe) {
    const uint32_t k = atomicCAS(&key[h], 0u, (uint32_t)id + 1u);
    if (k == 0u) *created = true;
    if (k == 0u || k == (uint32_t)id + 1u) return (int)h;
    h = (h + 1u) & (kHashSlots - 1u);
  }
  return -1;
}

// Appends the slots the warp's lanes created to the slot list, one counter update per warp.
__device__ __forceinline__ void list_append(uint16_t* list, int* nlist, bool created, int h) {
  const int lane = threadIdx.x & 31;
  const unsigned b = __ballot_sync(~0u, created);
  if (!b) return;
  int base = 0;
  if (lane == 0) base = atomicAdd(nlist, __popc(b));
  base = __shfl_sync(~0u, base, 0);
  if (created) list[base + __popc(b & ((1u << lane) - 1u))] = (uint16_t)h;
}
static_assert(kHashSlots == 1 << 12, "hash of 12 bits");

// One CTA per row (preparation launch): the row's distinct history ids with their counts
// and the last valid logit_bias entry of each id, listed by slice; validity flags; the
// mask's allowed count.  A row whose entries do not fit is left to the slices (ready 0).
__device__ void prep_row_lists(const LaunchParams& P, int row) {
  uint32_t* key = reinterpret_cast<uint32_t*>(smem_dyn);
  unsigned* cnt = key + kHashSlots;
  int* bj = reinterpret_cast<int*>(cnt + kHashSlots);
  uint16_t* list = reinterpret_cast<uint16_t*>(bj + kHashSlots);
  __shared__ int scnt[kMaxSlices + 1], sfill[kMaxSlices];
  __shared__ int sflags, sover, snal, nlist;
  const int C = P.C, chunk = P.chunk, V = P.a.V;
  for (int h = threadIdx.x; h < kHashSlots; h += kOrderThreads) {
    key[h] = 0u;
    cnt[h] = 0u;
    bj[h] = -1;
  }
  if (threadIdx.x < kMaxSlices + 1) scnt[threadIdx.x] = 0;
  if (threadIdx.x < kMaxSlices) sfill[threadIdx.x] = 0;
  if (threadIdx.x == 0) {
    sflags = 0;
    sover = 0;
    nlist = 0;
  }
  __syncthreads();
  int bad = 0, over = 0;
  const int lane = threadIdx.x & 31;
  if (P.a.hist_offs) {
    const int lo = P.a.hist_offs[row], hi = P.a.hist_offs[row + 1];
    if (lo < 0 || hi < lo) bad = 1;
    else
      for (int j0 = lo; j0 < hi; j0 += 8 * kOrderThreads) {
        int ids[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = j0 + u * kOrderThreads + threadIdx.x;
          ids[u] = j < hi ? __ldg(P.a.hist_ids + j) : INT_MIN;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int id = ids[u];
          const bool ok = id >= 0 && id < V;
          if (id != INT_MIN && !ok) bad = 1;
          const unsigned peers = __match_any_sync(~0u, ok ? id : -1);
          bool created = false;
          int h = -1;
          if (ok && (__ffs(peers) - 1) == lane) {
            h = hash_insert(key, id, &created);
            if (h < 0) over = 1;
            else atomicAdd(&cnt[h], (unsigned)__popc(peers));
          }
          list_append(list, &nlist, created, h);
        }
      }
  }
  if (P.a.bias_offs) {
    const int lo = P.a.bias_offs[row], hi = P.a.bias_offs[row + 1];
    if (lo < 0 || hi < lo) bad = 1;
    else
      for (int j0 = lo; j0 < hi; j0 += kOrderThreads) {
        const int j = j0 + threadIdx.x;
        bool created = false;
        int h = -1;
        if (j < hi) {
          const int id = __ldg(P.a.bias_ids + j);
          const float b = __ldg(P.a.bias_vals + j);
          if (id < 0 || id >= V || b != b) {
            bad = 1;
          } else {
            h = hash_insert(key, id, &created);
            if (h < 0) over = 1;
            else atomicMax(&bj[h], j);
          }
        }
        list_append(list, &nlist, created, h);
      }
  }
  if (bad) sflags = kFlagInvalid;
  if (over) sover = 1;
  __syncthreads();
  const int nl = min(nlist, kHashSlots);
  const int lane2 = threadIdx.x & 31;
  for (int i0 = 0; i0 < nl; i0 += kOrderThreads) {
    const int i = i0 + threadIdx.x;
    const int sl = i < nl ? (int)(key[list[i]] - 1u) / chunk : -1;
    const unsigned peers = __match_any_sync(~0u, sl);
    if (sl >= 0 && (__ffs(peers) - 1) == lane2) atomicAdd(&scnt[sl], __popc(peers));
  }
  __syncthreads();
  int* poff = P.poff + (size_t)row * (C + 1);
  if (threadIdx.x == 0) {
    int t = 0;
    for (int s = 0; s < C; ++s) {
      const int c = scnt[s];
      scnt[s] = t;
      poff[s] = t;
      t += c;
    }
    poff[C] = t;
    if (t > kPenRowCap) sover = 1;
  }
  __syncthreads();
  if (!sover) {
    PenEntry* out = P.pent + (size_t)row * kPenRowCap;
    for (int i0 = 0; i0 < nl; i0 += kOrderThreads) {
      const int i = i0 + threadIdx.x;
      const int h = i < nl ? list[i] : 0;
      const int id = i < nl ? (int)(key[h] - 1u) : -1;
      const int sl = id >= 0 ? id / chunk : -1;
      // one counter update per slice and warp; each thread takes its rank among its peers
      const unsigned peers = __match_any_sync(~0u, sl);
      const int leader = __ffs(peers) - 1;
      int base = 0;
      if (sl >= 0 && leader == lane2) base = atomicAdd(&sfill[sl], __popc(peers));
      base = __shfl_sync(peers, base, leader);
      if (sl < 0) continue;
      const int pos = scnt[sl] + base + __popc(peers & ((1u << lane2) - 1u));
      PenEntry e;
      e.lid = id - sl * chunk;
      e.cnt = cnt[h];
      e.bj = bj[h];
      e.pad = 0;
      out[pos] = e;
    }
  }
  int nal = V;
  if (P.a.bitmask) {
    const int W = (V + 31) >> 5;
    const int32_t* mrow = P.a.bitmask + (long long)row * P.a.bitmask_row_stride;
    int c = 0;
    // eight words in flight per thread
    for (int w0 = 0; w0 < W; w0 += 8 * kOrderThreads) {
      uint32_t x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int w = w0 + u * kOrderThreads + threadIdx.x;
        x[u] = w < W ? (uint32_t)__ldg(mrow + w) : 0u;
        if (w == W - 1 && (V & 31)) x[u] &= (1u << (V & 31)) - 1u;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) c += __popc(x[u]);
    }
    if (threadIdx.x == 0) snal = 0;
    __syncthreads();
    atomicAdd(&snal, c);
    __syncthreads();
    nal = snal;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    RowInfo ri;
    ri.flags = sflags;
    ri.nal = nal;
    ri.ready = !sover;
    ri.pad = 0;
    P.rinfo[row] = ri;
    __threadfence();
    st_release(&P.rflag[row], 1u);
  }
}

// One CTA: classifies the rows, writes the list order (stable within a class) and resets
// the call's counters.
__global__ void __launch_bounds__(kOrderThreads) order_kernel(const __grid_constant__ LaunchParams P) {
  // Each CTA first clears the flag it will set (a stale one could be left by a
  // preparation that no sampler consumed), then lets the sampler grid launch: the sampler
  // starts only after every CTA of this grid has passed this point.
  if (threadIdx.x == 0) {
    if (blockIdx.x == 0) P.ctl[2] = 0u;
    else P.rflag[blockIdx.x - 1] = 0u;
    __threadfence();
  }
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x > 0) {
    prep_row_lists(P, blockIdx.x - 1);
    return;
  }
  __shared__ int cnt[kClasses][kOrderThreads / 32];
  __shared__ uint8_t cls_cache[kClassCache];  // classes of the first rows (read once)
  const int B = P.a.B;
  // (the item counter, spill counter and done counter were reset by the previous sampler
  // grid's last CTA, or are zero from the allocation)
  // totals per class first, so each class knows where it starts
  int tot[kClasses] = {0, 0, 0, 0, 0};
  for (int r0 = 0; r0 < B; r0 += kOrderThreads) {
    const int r = r0 + threadIdx.x;
    int c = -1;
    if (r < B) {
      RowParams q;
      load_params(P.a, r, q);
      c = route_rank(q);
      if (r < kClassCache) cls_cache[r] = (uint8_t)c;
      RowCtl rc;
      rc.ticket = 0;
      rc.bar = 0;
      rc.spill = 0;
      rc.pad = 0;
      P.rowctl[r] = rc;
    }
    for (int j = 0; j < kClasses; ++j) tot[j] += __syncthreads_count(c == j);
  }
  int start[kClasses];
  start[0] = 0;
  for (int j = 1; j < kClasses; ++j) start[j] = start[j - 1] + tot[j - 1];
  for (int r0 = 0; r0 < B; r0 += kOrderThreads) {
    const int r = r0 + threadIdx.x;
    int c = -1;
    if (r < B) {
      if (r < kClassCache) {
        c = cls_cache[r];
      } else {
        RowParams q;
        load_params(P.a, r, q);
        c = route_rank(q);
      }
    }
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int j = 0; j < kClasses; ++j) {
      const unsigned bal = __ballot_sync(~0u, c == j);
      if (lane == 0) cnt[j][w] = __popc(bal);
      __syncthreads();
      int off = 0, all = 0;
      for (int i = 0; i < kOrderThreads / 32; ++i) {
        if (i < w) off += cnt[j][i];
        all += cnt[j][i];
      }
      if (c == j) P.order[start[j] + off + __popc(bal & ((1u << lane) - 1u))] = r;
      start[j] += all;
      __syncthreads();
    }
  }
  // the sampler's CTAs (already running under programmatic serialisation) wait for this
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) st_release(&P.ctl[2], 1u);
}

// ---------------------------------------------------------------- slice load and transforms

__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Starts the slice copy into shared memory (fp32 slices at buf, bf16 slices in the upper
// half of buf, to be widened in place).  A TMA bulk copy takes the 16-byte-aligned bulk;
// the ragged tail and unaligned rows use plain loads.  Returns the bytes the mbarrier
// waits for (0: nothing to wait for).
template <bool kBF16>
__device__ uint32_t slice_load(const LaunchParams& P, const Smem& S, int row, int c0, int n) {
  constexpr int kEs = kBF16 ? 2 : 4;
  const unsigned char* g =
      reinterpret_cast<const unsigned char*>(P.a.logits) + ((long long)row * P.a.logits_row_stride + c0) * kEs;
  unsigned char* dst = reinterpret_cast<unsigned char*>(S.buf) + (kBF16 ? (size_t)P.chunk * 2 : 0);
  const uint32_t bulk = P.vec_ok ? (uint32_t)(((size_t)n * kEs) & ~(size_t)15) : 0u;
  if (threadIdx.x == 0) {
    if (sh.bar_uses == 0) {
      mbar_init(&sh.bar, 1);
      fence_mbar_init();
    }
    if (bulk) {
      mbar_arrive_expect_tx(&sh.bar, bulk);
      bulk_copy_g2s_hint(dst, g, bulk, &sh.bar, make_policy_evict_first());
    }
  }
  for (int i = (int)(bulk / kEs) + threadIdx.x; i < n; i += kThreads) {
    if (kBF16)
      reinterpret_cast<uint16_t*>(dst)[i] = __ldg(reinterpret_cast<const unsigned short*>(g) + i);
    else
      reinterpret_cast<float*>(dst)[i] = __ldg(reinterpret_cast<const float*>(g) + i);
  }
  return bulk;
}

// Bounded wait for the slice copy; false if it did not complete.
__device__ bool slice_wait(uint32_t bulk) {
  if (!bulk) return true;
  const bool ok = mbar_wait(&sh.bar, sh.bar_uses & 1u);
  __syncthreads();
  if (threadIdx.x == 0) ++sh.bar_uses;
  return ok;
}

// bf16 slices: widen [0, n) from the upper half of buf to fp32 at buf, in chunks that are
// read completely before they are written (an fp32 write never reaches bf16 data of a
// later chunk, see the index bound below).
__device__ void widen_bf16(const Smem& S, int chunk, int n) {
  const uint16_t* src = reinterpret_cast<const uint16_t*>(S.buf) + chunk;  // byte offset 2 * chunk
  for (int i0 = 0; i0 < n; i0 += kThreads * 8) {
    float v[8];
    const int i = i0 + threadIdx.x * 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = (i + j < n) ? bf16_to_f32(src[i + j]) : 0.0f;
    __syncthreads();
    // element e lives at bytes [2 chunk + 2e, +2) as bf16 and [4e, +4) as fp32; the fp32
    // writes of this chunk end below 4 (i0 + 8 kThreads) <= 2 chunk + 2 (i0 + 8 kThreads)
    // only while i0 + 8 kThreads <= chunk, and the elements of later chunks start there
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (i + j < n) S.buf[i + j] = v[j];
    __syncthreads();
  }
}

// Local rank of a claimed token (its position among the slice's claimed tokens).
__device__ __forceinline__ int claim_rank(const Smem& S, int l) {
  const uint32_t w = S.claim[l >> 5];
  return (int)S.prefix[l >> 5] + __popc(w & ((1u << (l & 31)) - 1u));
}

// Marks the slice's history and logit_bias ids in the claim bitmap and ranks them.
// Out-of-range ids and NaN bias values make the row INVALID (they are skipped).
__device__ void claim_tokens(const LaunchParams& P, const Smem& S, const RowParams& q, int c0, int n) {
  const int nw = (n + 31) >> 5;
  for (int w = threadIdx.x; w < nw; w += kThreads) S.claim[w] = 0u;
  __syncthreads();
  int bad = 0;
  const int V = P.a.V;
  if (threadIdx.x == 0) sh.nhist = 0;
  __syncthreads();
  // history ids, eight loads in flight per thread; the slice's ids are also listed
  for (int j0 = q.hlo; j0 < q.hhi; j0 += 8 * kThreads) {
    int ids[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u * kThreads + threadIdx.x;
      ids[u] = j < q.hhi ? __ldg(P.a.hist_ids + j) : INT_MIN;
    }
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int id = ids[u];
      if (id != INT_MIN && (id < 0 || id >= V)) bad = 1;
      const bool in = id != INT_MIN && (unsigned)(id - c0) < (unsigned)n;
      const unsigned inb = __ballot_sync(~0u, in);
      if (!inb) continue;
      // repeated ids of one warp (frequent tokens) mark the bitmap once
      const unsigned peers = __match_any_sync(~0u, in ? id : -1);
      if (in && (__ffs(peers & inb) - 1) == lane) atomicOr(&S.claim[(id - c0) >> 5], 1u << ((id - c0) & 31));
      int base = 0;
      if (lane == 0) base = atomicAdd(&sh.nhist, __popc(inb));
      base = __shfl_sync(~0u, base, 0);
      const int pos = base + __popc(inb & ((1u << lane) - 1u));
      if (in && pos < kHList) S.hlist[pos] = (uint16_t)(id - c0);
    }
  }
  for (int j = q.blo + threadIdx.x; j < q.bhi; j += kThreads) {
    const int id = __ldg(P.a.bias_ids + j);
    const float b = __ldg(P.a.bias_vals + j);
    if (id < 0 || id >= V || b != b) bad = 1;
    else if ((unsigned)(id - c0) < (unsigned)n) atomicOr(&S.claim[(id - c0) >> 5], 1u << ((id - c0) & 31));
  }
  if (bad) sh.rec.flags = kFlagInvalid;  // benign race: every writer stores the same value
  __syncthreads();
  // ranks: each thread owns a run of consecutive words
  const int per = (nw + kThreads - 1) / kThreads;
  const int w0 = threadIdx.x * per;
  int c = 0;
  for (int w = w0; w < min(nw, w0 + per); ++w) c += __popc(S.claim[w]);
  int total = 0;
  int r = block_scan_i(c, &total);
  for (int w = w0; w < min(nw, w0 + per); ++w) {
    S.prefix[w] = (uint16_t)r;
    r += __popc(S.claim[w]);
  }
  if (threadIdx.x == 0) sh.ntouch = total;
  __syncthreads();
}

// One round of the transforms, kPen claimed ranks from r0: rank -> local id, history
// counts and the last bias entry of each (needs no logits, so round 0 runs while the
// slice copy is in flight) ...
__device__ void transforms_prep(const LaunchParams& P, const Smem& S, const RowParams& q, int c0, int n, int r0) {
  const int nw = (n + 31) >> 5;
  for (int t = threadIdx.x; t < kPen; t += kThreads) {
    S.pcnt[t] = 0u;
    S.pbias[t] = -1;
  }
  for (int w = threadIdx.x; w < nw; w += kThreads) {
    uint32_t bits = S.claim[w];
    int r = S.prefix[w];
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1u;
      if (r >= r0 && r < r0 + kPen) S.pid[r - r0] = (uint16_t)(w * 32 + b);
      ++r;
    }
  }
  __syncthreads();
  const int V = P.a.V;
  const int nh = sh.nhist;
  if (nh <= kHList) {
    const int lane = threadIdx.x & 31;
    for (int i0 = 0; i0 < nh; i0 += kThreads) {
      const int i = i0 + threadIdx.x;
      int r = -1;
      if (i < nh) {
        r = claim_rank(S, S.hlist[i]) - r0;
        if ((unsigned)r >= (unsigned)kPen) r = -1;
      }
      // one atomic per distinct rank of the warp, adding its multiplicity
      const unsigned peers = __match_any_sync(~0u, r);
      if (r >= 0 && (__ffs(peers) - 1) == lane) atomicAdd(&S.pcnt[r], (unsigned)__popc(peers));
    }
  } else {
    for (int j0 = q.hlo; j0 < q.hhi; j0 += 8 * kThreads) {
      int ids[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u * kThreads + threadIdx.x;
        ids[u] = j < q.hhi ? __ldg(P.a.hist_ids + j) : -1;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int id = ids[u];
        if (id < 0 || id >= V || (unsigned)(id - c0) >= (unsigned)n) continue;
        const int r = claim_rank(S, id - c0) - r0;
        if ((unsigned)r < (unsigned)kPen) atomicAdd(&S.pcnt[r], 1u);
      }
    }
  }
  for (int j = q.blo + threadIdx.x; j < q.bhi; j += kThreads) {
    const int id = __ldg(P.a.bias_ids + j);
    const float b = __ldg(P.a.bias_vals + j);
    if (id < 0 || id >= V || b != b || (unsigned)(id - c0) >= (unsigned)n) continue;
    const int r = claim_rank(S, id - c0) - r0;
    if ((unsigned)r < (unsigned)kPen) atomicMax(&S.pbias[r], j);
  }
  __syncthreads();
}

// ... and its application to the slice in place (fp32): a claimed token's value is
// sanitised first, then penalised, biased and folded (guard: NaN -> -inf, +inf -> FLT_MAX).
__device__ void transforms_apply(const LaunchParams& P, const Smem& S, const RowParams& q, int r0) {
  const int nr = min(kPen, sh.ntouch - r0);
  for (int t = threadIdx.x; t < nr; t += kThreads) {
    const int l = S.pid[t];
    float z = sanitize(S.buf[l]);
    const uint32_t c = S.pcnt[t];
    if (c) z = apply_penalties(z, c, q.freq, q.pres, q.rep);
    const int bj = S.pbias[t];
    if (bj >= 0) z = __fadd_rn(z, __ldg(P.a.bias_vals + bj));
    S.buf[l] = guard(z);
  }
  __syncthreads();
}

// ---------------------------------------------------------------- pass A

__device__ __forceinline__ bool claimed(const Smem& S, int l) { return (S.claim[l >> 5] >> (l & 31)) & 1u; }

__device__ __forceinline__ uint32_t mask_nibble(const uint32_t* mw, int f) {
  return mw ? (mw[f >> 3] >> ((f & 7) * 4)) & 0xFu : 0xFu;
}

// The slice's max, lowest argmax, allowed count and sum of 2^((z' - max) c).  Writes the
// mask (and the tail past the slice end) into buf as -inf.  Fast walk: finite input is
// assumed and checked by a running sum; if any value was not finite the slice is redone
// with per-token sanitising (claimed tokens already hold their final value).
template <bool kT1>
__device__ void pass_a_t(const LaunchParams& P, const Smem& S, const RowParams& q, int row, int c0, int n) {
  const int nv = (n + 3) >> 2;
  const uint32_t* mw = P.a.bitmask ? S.mask : nullptr;
  const uint32_t tail = (n & 3) ? ((1u << (n & 3)) - 1u) : 0xFu;
  float4* b4 = reinterpret_cast<float4*>(S.buf);
  if (n & 3) {
    if (threadIdx.x == 0)
      for (int j = n; j < 4 * nv; ++j) S.buf[j] = 0.0f;  // pads: finite, masked below
    __syncthreads();
  }
  // one walk: max, first vector reaching it, and the sum of 2^((z' - tmax) c) against a
  // running per-thread max (rescaled when it grows)
  const float c = __fmul_rn(1.4426950408889634f, q.invT);
  const float c1 = 1.4426950408889634f;             // T = 1: the original distribution
  constexpr bool want1 = kT1;  // the second (T = 1) sum only when its logprob is requested
  float tmax = -INFINITY, tsum = 0.0f, tsum1 = 0.0f, chk = 0.0f;
  int tf = INT_MAX, nal = 0;
  for (int f = threadIdx.x; f < nv; f += kThreads) {
    float4 v = b4[f];
    chk += (v.x + v.y) + (v.z + v.w);
    uint32_t bits = mask_nibble(mw, f);
    if (f == nv - 1) bits &= tail;
    if (bits != 0xFu) {
      if (!(bits & 1u)) v.x = -INFINITY;
      if (!(bits & 2u)) v.y = -INFINITY;
      if (!(bits & 4u)) v.z = -INFINITY;
      if (!(bits & 8u)) v.w = -INFINITY;
      b4[f] = v;
    }
    nal += __popc(bits);
    const float a4 = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
    if (a4 > tmax) {
      tsum *= ex2_approx((tmax - a4) * c);
      if (want1) tsum1 *= ex2_approx((tmax - a4) * c1);
      tmax = a4;
      tf = f;
    }
    if (tmax > -INFINITY) {
      tsum += (ex2_approx((v.x - tmax) * c) + ex2_approx((v.y - tmax) * c)) +
              (ex2_approx((v.z - tmax) * c) + ex2_approx((v.w - tmax) * c));
      if (want1)
        tsum1 += (ex2_approx((v.x - tmax) * c1) + ex2_approx((v.y - tmax) * c1)) +
                 (ex2_approx((v.z - tmax) * c1) + ex2_approx((v.w - tmax) * c1));
    }
  }
  const int nonfinite = __syncthreads_or(!(fabsf(chk) < INFINITY));
  if (nonfinite) {
    // checked walk: sanitise unclaimed allowed tokens, mask, count
    tmax = -INFINITY;
    tf = INT_MAX;
    nal = 0;
    for (int l = threadIdx.x; l < 4 * nv; l += kThreads) {
      float z = -INFINITY;
      if (l < n) {
        const bool ok = mw ? ((mw[l >> 5] >> (l & 31)) & 1u) : true;
        if (ok) z = claimed(S, l) ? S.buf[l] : sanitize(S.buf[l]);
      }
      S.buf[l] = z;
    }
    __syncthreads();
    tsum = 0.0f;
    tsum1 = 0.0f;
    for (int f = threadIdx.x; f < nv; f += kThreads) {
      const float4 v = b4[f];
      nal += (v.x > -INFINITY) + (v.y > -INFINITY) + (v.z > -INFINITY) + (v.w > -INFINITY);
      const float a4 = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
      if (a4 > tmax) {
        tsum *= ex2_approx((tmax - a4) * c);
        if (want1) tsum1 *= ex2_approx((tmax - a4) * c1);
        tmax = a4;
        tf = f;
      }
      if (tmax > -INFINITY) {
        tsum += (ex2_approx((v.x - tmax) * c) + ex2_approx((v.y - tmax) * c)) +
                (ex2_approx((v.z - tmax) * c) + ex2_approx((v.w - tmax) * c));
        if (want1)
          tsum1 += (ex2_approx((v.x - tmax) * c1) + ex2_approx((v.y - tmax) * c1)) +
                   (ex2_approx((v.z - tmax) * c1) + ex2_approx((v.w - tmax) * c1));
      }
    }
  }
  S.hist[threadIdx.x] = tmax > -INFINITY ? fkey(tmax) : 0u;  // per-thread maxima for the top-k bound
  int arg = INT_MAX;
  if (tf != INT_MAX && tmax > -INFINITY) {
    const float4 v = b4[tf];
    const int j = v.x == tmax ? 0 : v.y == tmax ? 1 : v.z == tmax ? 2 : 3;
    arg = c0 + 4 * tf + j;
  }
  // one combine: each warp reduces (max, lowest argmax, allowed count, sum rescaled to
  // the warp max) with shuffles; thread 0 merges the warps in warp order
  float M = tmax;
  int am = arg;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float v2 = __shfl_xor_sync(~0u, M, o);
    const int i2 = __shfl_xor_sync(~0u, am, o);
    if (better(v2, i2, M, am)) {
      M = v2;
      am = i2;
    }
    nal += __shfl_xor_sync(~0u, nal, o);
  }
  float ws = (M > -INFINITY && tmax > -INFINITY) ? tsum * ex2_approx((tmax - M) * c) : 0.0f;
  ws = warp_sum_f(ws);
  float ws1 = (want1 && M > -INFINITY && tmax > -INFINITY) ? tsum1 * ex2_approx((tmax - M) * c1) : 0.0f;
  if (want1) ws1 = warp_sum_f(ws1);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    sh.red_f[w] = M;
    sh.red_i[w] = am;
    sh.red_u[w] = ((unsigned long long)(unsigned)nal << 32) | __float_as_uint(ws);
    sh.red_f2[w] = ws1;
  }
  __syncthreads();
  float s = 0.0f, s1 = 0.0f;
  if (threadIdx.x == 0) {
    float Mb = sh.red_f[0];
    int ab = sh.red_i[0];
    for (int i = 1; i < kWarps; ++i)
      if (better(sh.red_f[i], sh.red_i[i], Mb, ab)) {
        Mb = sh.red_f[i];
        ab = sh.red_i[i];
      }
    int nb = 0;
    for (int i = 0; i < kWarps; ++i) {
      const unsigned long long u = sh.red_u[i];
      nb += (int)(u >> 32);
      const float wsi = __uint_as_float((uint32_t)u);
      if (Mb > -INFINITY && sh.red_f[i] > -INFINITY) {
        s += wsi * ex2_approx((sh.red_f[i] - Mb) * c);
        s1 += sh.red_f2[i] * ex2_approx((sh.red_f[i] - Mb) * c1);
      }
    }
    M = Mb;
    arg = ab;
    nal = nb;
  }
  if (threadIdx.x == 0) {
    sh.rec.m = M;
    sh.rec.arg = M > -INFINITY ? arg : INT_MAX;
    sh.rec.s = s;
    sh.rec.s1 = s1;
    sh.rec.nallowed = nal;
  }
  if (P.a.dbg_transformed) {
    float* d = P.a.dbg_transformed + (long long)row * P.a.V + c0;
    for (int l = threadIdx.x; l < n; l += kThreads) d[l] = S.buf[l];
  }
  __syncthreads();
}

// Pass A, compiled once without and once with the T = 1 sum, so the common case carries
// no extra work in its walk.
__device__ __forceinline__ void pass_a(const LaunchParams& P, const Smem& S, const RowParams& q, int row, int c0,
                                       int n) {
  if (P.a.logprobs_orig) pass_a_t<true>(P, S, q, row, c0, n);
  else pass_a_t<false>(P, S, q, row, c0, n);
}

// ---------------------------------------------------------------- candidates of light rows

// The row's spill slot, taken once per row by the first slice that needs one.  The cell
// holds 0 (none yet: its state after a finished row and after allocation), -1 while that
// slice draws a slot, then slot + 1, or -2 if none was left.  Returns the slot, or -1 if
// the row has none.
__device__ int row_spill_slot(const LaunchParams& P, int row) {
  int* cell = &P.rowctl[row].spill;
  int cur = atomicCAS(cell, 0, -1);
  if (cur == 0) {
    const unsigned slot = atomicAdd(&P.ctl[1], 1u);
    const int v = slot < (unsigned)P.spill_rows ? (int)slot + 1 : -2;
    atomicExch(cell, v);
    return v > 0 ? v - 1 : -1;
  }
  for (uint32_t i = 0; i < kWaitPolls && cur == -1; ++i) {
    __nanosleep(64);
    cur = (int)ld_acquire(reinterpret_cast<const unsigned*>(cell));
  }
  return cur > 0 ? cur - 1 : -1;
}

__device__ __forceinline__ Item* spill_area(const LaunchParams& P, int slot, int slice) {
  return P.spill + ((size_t)slot * P.C + slice) * P.chunk;
}
__device__ __forceinline__ Item* cand_area(const LaunchParams& P, int row, int slice) {
  return P.cand + ((size_t)row * P.C + slice) * kCandCap;
}

// Items (z', id) of the slice's tokens with z' >= zc and z' > -inf, in token order per
// warp step; returns how many there are (only the first `cap` are written).
// `active` false: the calling thread's vectors hold no such token (its maximum is below),
// so a warp whose threads are all inactive skips the walk.
template <class Pred>
__device__ int compact_if(const Smem& S, int c0, int n, Pred&& keep, Item* dst, int cap, bool active = true) {
  const int nv = (n + 3) >> 2;
  const float4* b4 = reinterpret_cast<const float4*>(S.buf);
  if (threadIdx.x == 0) sh.cnt = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  const bool warp_active = __any_sync(~0u, active);
  for (int f0 = 0; warp_active && f0 < nv; f0 += kThreads) {
    const int f = f0 + threadIdx.x;
    const float4 v = f < nv ? b4[f] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    const float e[4] = {v.x, v.y, v.z, v.w};
    unsigned bal[4];
    int tot = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      bal[j] = __ballot_sync(~0u, active && e[j] > -INFINITY && keep(e[j]));
      tot += __popc(bal[j]);
    }
    if (!tot) continue;
    int base = 0;
    if (lane == 0) base = atomicAdd(&sh.cnt, tot);
    base = __shfl_sync(~0u, base, 0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if ((bal[j] >> lane) & 1u) {
        const int pos = base + __popc(bal[j] & lt);
        if (pos < cap) dst[pos] = Item{e[j], c0 + 4 * f + j};
      }
      base += __popc(bal[j]);
    }
  }
  __syncthreads();
  return sh.cnt;
}

// The same for the threshold z' >= zc: a warp step whose vectors all lie below it (their
// maxima) costs one vote and no per-token ballots.
__device__ int compact(const Smem& S, int c0, int n, float zc, Item* dst, int cap, bool active = true) {
  const int nv = (n + 3) >> 2;
  const float4* b4 = reinterpret_cast<const float4*>(S.buf);
  if (threadIdx.x == 0) sh.cnt = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  const bool warp_active = __any_sync(~0u, active);
  for (int f0 = 0; warp_active && f0 < nv; f0 += kThreads) {
    const int f = f0 + threadIdx.x;
    const float4 v = f < nv ? b4[f] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    const float vm = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
    const bool hit = active && vm > -INFINITY && vm >= zc;
    if (!__any_sync(~0u, hit)) continue;
    const float e[4] = {v.x, v.y, v.z, v.w};
    // the four ballots first, then one shared-memory atomic for the warp's whole step
    unsigned bal[4];
    int tot = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      bal[j] = __ballot_sync(~0u, hit && e[j] > -INFINITY && e[j] >= zc);
      tot += __popc(bal[j]);
    }
    int base = 0;
    if (lane == 0) base = atomicAdd(&sh.cnt, tot);
    base = __shfl_sync(~0u, base, 0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if ((bal[j] >> lane) & 1u) {
        const int pos = base + __popc(bal[j] & lt);
        if (pos < cap) dst[pos] = Item{e[j], c0 + 4 * f + j};
      }
      base += __popc(bal[j]);
    }
  }
  __syncthreads();
  return sh.cnt;
}

// Writes every allowed token of the slice to the row's spill area; returns the count, or
// -1 (and flags OVERFLOW) if no spill slot is left.
__device__ int spill_slice(const LaunchParams& P, const Smem& S, int row, int slice, int c0, int n) {
  if (threadIdx.x == 0) sh.spill = row_spill_slot(P, row);
  __syncthreads();
  const int slot = sh.spill;
  if (slot < 0) return -1;
  return compact(S, c0, n, -INFINITY, spill_area(P, slot, slice), P.chunk);
}

// Rounding margin of a candidate bound near `edge` in a slice whose max is M.
__device__ __forceinline__ float bound_margin(float M, float edge) {
  return (fabsf(M) + fabsf(edge) + 1.0f) * 0x1p-14f;
}

// Light rows: the slice's candidates.  Top-k: the tokens at or above a bound taken from
// the warps' sorted per-thread maxima, aiming at 1.2 k times the slice's share of the
// row's allowed tokens; whether that holds the row's whole top-k set is checked exactly
// at the row end (a failing slice is redone in full).  Min-p with p = 1: z' >=
// M + T ln(min_p) minus a rounding margin (the row max is at least M), a superset by
// construction.  Candidates past kCandCap spill the whole slice.
__device__ void light_candidates(const LaunchParams& P, const Smem& S, const RowParams& q, int row, int slice,
                                 int c0, int n) {
  const float M = sh.rec.m;
  float zc = -INFINITY, dz = 0.0f;
  int tnc = -1;  // top-k: candidates compacted while the bound was chosen (-1: none yet)
  if (M > -INFINITY && q.route == kRouteTopK) {
    const int nal = sh.rec.nallowed;
    const float share = P.a.bitmask ? (float)nal / (float)max(1, sh.nal_row) : (float)n / (float)P.a.V;
    int nc = -1;
    const int need = (int)ceilf(1.2f * (float)q.k * share) + 4;
    if (need < nal && need <= kThreads) {
      // each warp sorts its 32 per-thread maxima (shuffles only); the smallest over the
      // warps of their q-th largest, q = ceil(need / kWarps), has q tokens at or above it
      // in every warp
      const uint32_t mine = S.hist[threadIdx.x];  // this thread's maximum (order key)
      uint32_t key = mine;
      const int lane = threadIdx.x & 31;
      int qj = min(31, (need + kWarps - 1) / kWarps - 1);
      // qj <= 1 (small k): the warp's two largest by a pair reduction; else a full sort
      uint32_t t1 = mine, t2 = 0u;
      const bool small = qj <= 1;
      if (small) {
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const uint32_t a1 = __shfl_xor_sync(~0u, t1, o), a2 = __shfl_xor_sync(~0u, t2, o);
          const uint32_t hi = max(t1, a1);
          t2 = max(min(t1, a1), max(t2, a2));
          t1 = hi;
        }
      } else {
#pragma unroll
        for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
          for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const uint32_t o = __shfl_xor_sync(~0u, key, stride);
            const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
            key = keep_max ? max(key, o) : min(key, o);
          }
      }
      for (int tries = 0; tries < 3; ++tries) {
        const uint32_t thr = block_min_u32(small ? (qj == 0 ? t1 : t2) : __shfl_sync(~0u, key, qj));
        if (thr == 0u) break;  // a warp has fewer live threads: take every allowed token
        const float edge = key_to_float(thr);
        const int c = compact(S, c0, n, edge, cand_area(P, row, slice), kCandCap, mine >= thr);
        if (c <= kCandCap) {
          zc = edge;
          nc = c;
          break;
        }
        if (qj == 0) {
          nc = c;  // too many even at the warps' maxima: spill below
          break;
        }
        qj >>= 1;
      }
    }
    tnc = nc;  // uniform: every thread saw the same counts
  } else if (M > -INFINITY && q.route == kRouteMinP) {
    const float edge = M + q.L * q.Teff;
    dz = bound_margin(M, edge);
    zc = edge - dz;
  }
  int nc = 0;
  if (M > -INFINITY) {
    if (tnc >= 0) nc = tnc;  // compacted while the bound was chosen
    else nc = compact(S, c0, n, zc, cand_area(P, row, slice), kCandCap, !(zc > -INFINITY) || S.hist[threadIdx.x] >= fkey(zc));
    if (nc > kCandCap) {
      nc = spill_slice(P, S, row, slice, c0, n);
      if (threadIdx.x == 0) sh.rec.spilled = nc >= 0;
      if (nc < 0) {  // no spill slot left: the row reports OVERFLOW
        nc = 0;
        if (threadIdx.x == 0) sh.rec.flags |= kFlagOverflow;
      }
    }
  }
  if (threadIdx.x == 0) {  // the caller's barrier publishes the record
    sh.rec.ncand = nc;
    sh.rec.zc = zc;
    sh.rec.dz = dz;
  }
}

// ---------------------------------------------------------------- row end: records

__device__ __forceinline__ SliceRec ldcg_rec(const SliceRec* p) {
  SliceRec r;
  const int4* s = reinterpret_cast<const int4*>(p);
  int4* d = reinterpret_cast<int4*>(&r);
#pragma unroll
  for (int i = 0; i < (int)(sizeof(SliceRec) / 16); ++i) d[i] = __ldcg(s + i);
  return r;
}
static_assert(sizeof(SliceRec) % 16 == 0, "records move as 16-byte vectors");

__device__ __forceinline__ Item ldcg_item(const Item* p) {
  const int2 v = __ldcg(reinterpret_cast<const int2*>(p));
  return Item{__int_as_float(v.x), v.y};
}

// Publishes this CTA's record and everything the CTA wrote before: the block barrier
// orders every thread's writes before thread 0's, and thread 0's fence (cumulative) makes
// them visible device-wide before the ticket or barrier arrival that follows.
__device__ void publish_rec(const LaunchParams& P, int row, int slice) {
  __syncthreads();
  if (threadIdx.x == 0) {
    P.srec[(size_t)row * P.C + slice] = sh.rec;
    __threadfence();
  }
  __syncthreads();
}

// Reads the row's C records into shared memory and combines them (slice order, so the
// float sum does not depend on timing): max, lowest argmax, allowed tokens, flags and
// the normaliser S of 2^((z' - m) log2(e) / T) = sum of e^y.
__device__ void combine_row(const LaunchParams& P, int row, const RowParams& q) {
  const int C = P.C;
  if (threadIdx.x < C) sh.recs[threadIdx.x] = ldcg_rec(P.srec + (size_t)row * C + threadIdx.x);
  __syncthreads();
  if (threadIdx.x == 0) {
    SliceRec r = sh.recs[0];
    float m = -INFINITY;
    int arg = INT_MAX, nal = 0, flags = q.invalid;
    for (int s = 0; s < C; ++s) {
      const SliceRec& x = sh.recs[s];
      if (better(x.m, x.arg, m, arg)) {
        m = x.m;
        arg = x.arg;
      }
      nal += x.nallowed;
      flags |= x.flags;
    }
    float S = 0.0f, S1 = 0.0f;
    if (m > -INFINITY) {
      const float c = __fmul_rn(1.4426950408889634f, q.invT);
      for (int s = 0; s < C; ++s)
        if (sh.recs[s].m > -INFINITY) {
          S += sh.recs[s].s * ex2_approx((sh.recs[s].m - m) * c);
          S1 += sh.recs[s].s1 * ex2_approx((sh.recs[s].m - m) * 1.4426950408889634f);
        }
    }
    r.m = m;
    r.arg = arg;
    r.nallowed = nal;
    r.flags = flags;
    r.s = S;
    sh.row = r;
    sh.lnS = logf(S);
    sh.lnS1 = logf(S1);
  }
  __syncthreads();
}

// Writes a row's outputs.  lp_orig = z'_tok - m - ln S1 (T = 1); lp_kept = y_tok minus
// the log of the kept set's mass.
__device__ void write_row(const clsample_args_t& a, int row, int status, int tok, float lp, int kept, float cut,
                          float lp_orig = -INFINITY, float lp_kept = -INFINITY) {
  a.tokens[row] = status == kRowInvalid ? -1 : tok;
  if (a.logprobs) a.logprobs[row] = status == kRowInvalid ? -INFINITY : lp;
  if (a.logprobs_orig) a.logprobs_orig[row] = status == kRowInvalid ? -INFINITY : lp_orig;
  if (a.logprobs_kept) a.logprobs_kept[row] = status == kRowInvalid ? -INFINITY : lp_kept;
  if (a.row_status) a.row_status[row] = status;
  if (a.dbg_kept_count) a.dbg_kept_count[row] = status == kRowInvalid ? 0 : kept;
  if (a.dbg_cut) a.dbg_cut[row] = status == kRowInvalid ? -INFINITY : cut;
}

// Status of a combined row: INVALID (bad parameters or ids, no allowed token) or
// OVERFLOW (a scratch limit or a bounded wait was hit); else OK.
__device__ __forceinline__ int row_status_of(const SliceRec& r) {
  if ((r.flags & kFlagInvalid) || !(r.m > -INFINITY)) return kRowInvalid;
  return (r.flags & kFlagOverflow) ? kRowOverflow : kRowOk;
}

// ---------------------------------------------------------------- row end: exact selects

__device__ unsigned long long block_scan_u64(unsigned long long x, unsigned long long* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  unsigned long long v = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(~0u, v, o);
    if (lane >= o) v += t;
  }
  __syncthreads();
  if (lane == 31) sh.red_u[w] = v;
  __syncthreads();
  unsigned long long off = 0, tot = 0;
  for (int i = 0; i < kWarps; ++i) {
    if (i < w) off += sh.red_u[i];
    tot += sh.red_u[i];
  }
  *total = tot;
  return off + v - x;
}

// The finisher's items (y, id) in shared memory, and its two digit histograms, at the
// end of buf.
__device__ __forceinline__ Item* fin_items(const Smem& S) { return reinterpret_cast<Item*>(S.buf); }
__device__ __forceinline__ int fin_cap(int chunk) { return (buf_bytes(chunk) - kFinHistBytes) / (int)sizeof(Item); }
__device__ __forceinline__ uint32_t* fin_hc(const Smem& S, int chunk) {
  return reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(S.buf) + buf_bytes(chunk) - kFinHistBytes);
}
__device__ __forceinline__ unsigned long long* fin_hw(const Smem& S, int chunk) {
  return reinterpret_cast<unsigned long long*>(reinterpret_cast<unsigned char*>(S.buf) + buf_bytes(chunk) -
                                               kDigitBins * 8);
}

// Calls fn(y, id) for the finisher's items: from shared memory, or (when they did not
// fit) straight from the global segments with the prefilter z' >= zmin.
template <class Fn>
__device__ __forceinline__ void visit(const Smem& S, float m, float invT, Fn&& fn) {
  if (sh.fin_smem) {
    const Item* it = fin_items(S);
    for (int i = threadIdx.x; i < sh.fin_n; i += kThreads) fn(it[i].z, it[i].id);
  } else {
    for (int s = 0; s < sh.nseg; ++s) {
      const Item* g = sh.seg[s];
      const int n = sh.segn[s];
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const Item x = ldcg_item(g + i);
        if (x.z >= sh.zmin) fn(y_of(x.z, m, invT), x.id);
      }
    }
  }
}

// Copies the prefiltered items into shared memory as (y, id) if they fit.
__device__ void gather_items(const Smem& S, int chunk, float m, float invT) {
  const int cap = fin_cap(chunk);
  Item* it = fin_items(S);
  if (threadIdx.x == 0) sh.cnt = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const float zmin = sh.zmin;
  // one index space over the segments, eight loads in flight per thread
  int total = 0;
  for (int s = 0; s < sh.nseg; ++s) total += sh.segn[s];
  for (int i0 = 0; i0 < total; i0 += 8 * kThreads) {
    Item x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      int i = i0 + j * kThreads + threadIdx.x;
      x[j] = Item{-INFINITY, 0};
      if (i < total) {
        int s = 0;
        while (i >= sh.segn[s]) i -= sh.segn[s++];
        x[j] = ldcg_item(sh.seg[s] + i);
      }
    }
    // the eight ballots first, then one shared-memory atomic for the warp's step
    unsigned bal[8];
    int tot = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      bal[j] = __ballot_sync(~0u, x[j].z > -INFINITY && x[j].z >= zmin);
      tot += __popc(bal[j]);
    }
    if (!tot) continue;
    int base = 0;
    if (lane == 0) base = atomicAdd(&sh.cnt, tot);
    base = __shfl_sync(~0u, base, 0);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if ((bal[j] >> lane) & 1u) {
        const int pos = base + __popc(bal[j] & ((1u << lane) - 1u));
        if (pos < cap) it[pos] = Item{y_of(x[j].z, m, invT), x[j].id};
      }
      base += __popc(bal[j]);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    sh.fin_smem = sh.cnt <= cap;
    sh.fin_n = sh.cnt;
  }
  __syncthreads();
}

// Radix digits of the 32-bit order keys: 11 + 11 + 10 bits, high to low.
__device__ __forceinline__ int digit_shift(int r) { return r == 0 ? 21 : (r == 1 ? 10 : 0); }
__device__ __forceinline__ int digit_width(int r) { return r == 2 ? 10 : 11; }
__device__ __forceinline__ bool digit_match(uint32_t key, int r, uint32_t prefix) {
  return r == 0 || (key >> (digit_shift(r) + digit_width(r))) == prefix;
}
constexpr int kBPT = kDigitBins / kThreads;  // digit bins per thread
static_assert(kDigitBins % kThreads == 0, "whole digit bins per thread");

// Key of the krem-th largest y among the items (every item counted, ties by key).
__device__ uint32_t select_kth(const Smem& S, int chunk, float m, float invT, int krem) {
  uint32_t* hc = fin_hc(S, chunk);
  uint32_t prefix = 0;
  for (int r = 0; r < 3; ++r) {
    const int sft = digit_shift(r);
    const uint32_t dmask = (1u << digit_width(r)) - 1u;
    for (int t = threadIdx.x; t < kDigitBins; t += kThreads) hc[t] = 0u;
    __syncthreads();
    visit(S, m, invT, [&](float y, int) {
      const uint32_t key = fkey(y);
      if (digit_match(key, r, prefix)) atomicAdd(&hc[(key >> sft) & dmask], 1u);
    });
    __syncthreads();
    int c = 0;
    for (int d = kBPT * (int)threadIdx.x; d < kBPT * (int)threadIdx.x + kBPT; ++d) c += (int)hc[d];
    int tot = 0;
    const int pre = block_scan_i(c, &tot);
    const int above = tot - pre - c;  // items in the digits above this thread's eight
    if (above < krem && above + c >= krem) {
      int run = above;
      for (int d = kBPT * (int)threadIdx.x + kBPT - 1; d >= kBPT * (int)threadIdx.x; --d) {
        if (run + (int)hc[d] >= krem) {
          sh.digit = d;
          sh.cnt = run;
          break;
        }
        run += (int)hc[d];
      }
    }
    __syncthreads();
    krem -= sh.cnt;
    prefix = (prefix << digit_width(r)) | (uint32_t)sh.digit;
    __syncthreads();
  }
  return prefix;
}

// Top-p cut over the items with key >= tk: the smallest key c whose mass of strictly
// larger keys, A plus the items', is below thr (the tokens of equal y go in or out
// together).  Masses are exact 2^-40 fixed-point weights.
__device__ uint32_t select_mass(const Smem& S, int chunk, float m, float invT, uint32_t tk, unsigned long long A,
                                unsigned long long thr) {
  uint32_t* hc = fin_hc(S, chunk);
  uint32_t* hlo = reinterpret_cast<uint32_t*>(fin_hw(S, chunk));
  uint32_t* hhi = hlo + kDigitBins;
  uint32_t prefix = 0;
  for (int r = 0; r < 3; ++r) {
    const int sft = digit_shift(r);
    const uint32_t dmask = (1u << digit_width(r)) - 1u;
    for (int t = threadIdx.x; t < kDigitBins; t += kThreads) {
      hc[t] = 0u;
      hlo[t] = 0u;
      hhi[t] = 0u;
    }
    if (threadIdx.x == 0) sh.digit = INT_MAX;
    __syncthreads();
    visit(S, m, invT, [&](float y, int) {
      const uint32_t key = fkey(y);
      if (key >= tk && digit_match(key, r, prefix)) {
        const uint32_t d = (key >> sft) & dmask;
        atomicAdd(&hc[d], 1u);
        add_mass(&hlo[d], &hhi[d], weight_fx(y));
      }
    });
    __syncthreads();
    unsigned long long c = 0;
    for (int d = kBPT * (int)threadIdx.x; d < kBPT * (int)threadIdx.x + kBPT; ++d) c += get_mass(&hlo[d], &hhi[d]);
    unsigned long long tot = 0;
    const unsigned long long pre = block_scan_u64(c, &tot);
    const unsigned long long above = A + (tot - pre - c);
    unsigned long long run = above;
    int best = -1;
    for (int d = kBPT * (int)threadIdx.x + kBPT - 1; d >= kBPT * (int)threadIdx.x; --d) {
      if (hc[d] > 0u && run < thr) best = d;
      run += get_mass(&hlo[d], &hhi[d]);
    }
    if (best >= 0) atomicMin(&sh.digit, best);
    __syncthreads();
    const int ds = sh.digit;
    if (ds == INT_MAX) return tk;  // no key qualifies (cannot happen while A < thr)
    if (ds >= kBPT * (int)threadIdx.x && ds < kBPT * (int)threadIdx.x + kBPT) {
      unsigned long long cum = above;
      for (int d = kBPT * (int)threadIdx.x + kBPT - 1; d > ds; --d) cum += get_mass(&hlo[d], &hhi[d]);
      sh.digit_above = cum;
    }
    __syncthreads();
    A = sh.digit_above;
    prefix = (prefix << digit_width(r)) | (uint32_t)ds;
    __syncthreads();
  }
  return prefix;
}

// Race of a (y, id): Philox word id & 3 of counter (id / 4, position) under the seed.
__device__ __forceinline__ float race_of(float y, int id, unsigned long long seed, unsigned long long pos) {
  const uint4 w = race_words((uint32_t)id >> 2, seed, pos);
  return race_score(y, pick_word(w, id & 3));
}

// Block argmax of (score, id) that also hands out the winner's y.
__device__ void block_race(float& s, int& id, float& y) {
  const int mine = id;
  const float my_y = y;
  block_argmax(s, id);
  __syncthreads();
  if (mine == id && id != INT_MAX) sh.red_f[kWarps] = my_y;
  __syncthreads();
  y = sh.red_f[kWarps];
  __syncthreads();
}


// z' of token `tok` among the row's items (the global candidate / band segments, which
// hold z'); the caller knows the token is one of them.  Block-wide.
__device__ float find_item_z(int tok) {
  if (threadIdx.x == 0) sh.ztok = NAN;
  __syncthreads();
  for (int s = 0; s < sh.nseg; ++s) {
    const Item* g = sh.seg[s];
    const int n = sh.segn[s];
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const Item x = ldcg_item(g + i);
      if (x.id == tok) sh.ztok = x.z;
    }
  }
  __syncthreads();
  return sh.ztok;
}

// Sum over the block of per-thread floats (fixed order over the warps).
__device__ float block_sum_f2(float v) {
  v = warp_sum_f(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh.red_f2[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = 0.0f;
  for (int i = 0; i < kWarps; ++i) r += sh.red_f2[i];
  return r;
}

// ---------------------------------------------------------------- row end: sorted finisher

constexpr int kSortCap = 2048;  // items the sorted finisher takes (its masses fit the histogram area)
constexpr int kHeavySortMax = 1024;  // heavy rows without a top-k cut sort at most this many band items

// Sorts the n <= kSortCap smem items in place by (y descending, id ascending) as 64-bit
// composites (order key << 32 | ~id), bitonic, padded to a power of two with zeros.
__device__ void sort_items(const Smem& S, int chunk, int n) {
  unsigned long long* k = reinterpret_cast<unsigned long long*>(fin_items(S));
  if (n <= kThreads) {
    // rank sort with one item per thread
    unsigned long long mine = 0ull;
    if ((int)threadIdx.x < n) {
      const Item it = fin_items(S)[threadIdx.x];
      mine = ((unsigned long long)fkey(it.z) << 32) | (uint32_t)(~(uint32_t)it.id);
    }
    unsigned long long* tmp = reinterpret_cast<unsigned long long*>(fin_hc(S, chunk));
    if ((int)threadIdx.x < n) tmp[threadIdx.x] = mine;
    __syncthreads();
    int rank = 0;
    for (int j = 0; j < n; ++j) rank += tmp[j] > mine;
    if ((int)threadIdx.x < n) k[rank] = mine;
    __syncthreads();
    return;
  }
  if (n <= 2 * kThreads) {
    // rank sort: the composites are distinct, so each one's position is the number of
    // larger ones (every thread counts against all n, reading broadcast words)
    unsigned long long mine[2];
    int rank[2] = {0, 0};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int i = threadIdx.x + u * kThreads;
      mine[u] = 0ull;
      if (i < n) {
        const Item it = fin_items(S)[i];
        mine[u] = ((unsigned long long)fkey(it.z) << 32) | (uint32_t)(~(uint32_t)it.id);
      }
    }
    unsigned long long* tmp = reinterpret_cast<unsigned long long*>(fin_hc(S, chunk));
#pragma unroll
    for (int u = 0; u < 2; ++u)
      if (threadIdx.x + u * kThreads < n) tmp[threadIdx.x + u * kThreads] = mine[u];
    __syncthreads();
    for (int j = 0; j < n; ++j) {
      const unsigned long long o = tmp[j];
      rank[0] += o > mine[0];
      rank[1] += o > mine[1];
    }
#pragma unroll
    for (int u = 0; u < 2; ++u)
      if (threadIdx.x + u * kThreads < n) k[rank[u]] = mine[u];
    __syncthreads();
    return;
  }
  static_assert(kSortCap <= 8 * kThreads, "eight items per thread");
  unsigned long long v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int i = threadIdx.x + j * kThreads;
    v[j] = 0ull;
    if (i < n) {
      const Item it = fin_items(S)[i];
      v[j] = ((unsigned long long)fkey(it.z) << 32) | (uint32_t)(~(uint32_t)it.id);
    }
  }
  __syncthreads();  // every item is read before any composite overwrites it
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int i = threadIdx.x + j * kThreads;
    if (i < n) k[i] = v[j];
  }
  __syncthreads();
  sort_desc(k, n);
}

__device__ __forceinline__ int sorted_id(unsigned long long v) { return (int)~(uint32_t)v; }

// Finishes a row whose n <= kSortCap items are in shared memory: sort, then the top-k,
// top-p and min-p cuts are prefixes of the sorted order, and the race runs over the kept
// prefix.  Returns through the same outputs as the digit path.
template <class Above>
__device__ void finish_sorted(const LaunchParams& P, const Smem& S, const RowParams& q, int row, const Above& ab,
                              bool heavy, int status, const SliceRec& R, float lnS, bool sorted) {
  const int n = sh.fin_n;
  if (!sorted) sort_items(S, P.chunk, n);
  const unsigned long long* k = reinterpret_cast<const unsigned long long*>(fin_items(S));
  auto key_at = [&](int i) { return (uint32_t)(k[i] >> 32); };
  auto count_ge = [&](int lim, uint32_t key) {
    int c = 0;
    for (int i = threadIdx.x; i < lim; i += kThreads) c += key_at(i) >= key;
    return block_sum_i(c);
  };
  // top-k: the first nk items (every item tied with the k-th stays)
  const int kc = (q.k >= 2 && q.k < R.nallowed) ? q.k : 0;
  int nk = n;
  if (kc > 0) {
    const int krem = kc - (int)ab.n;
    if (krem >= 1 && krem <= n) nk = count_ge(n, key_at(krem - 1));
  }
  // top-p over the top-k set: item i stays iff the mass of strictly larger y is below
  // ceil(p W); with exclusive prefix masses w[i] that is a prefix of length c, extended
  // by the items tied with item c - 1
  int np = nk;
  if (q.p < 1.0f && nk > 0) {
    unsigned long long* w = fin_hw(S, P.chunk);
    unsigned long long loc[8], tsum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = 8 * (int)threadIdx.x + j;
      loc[j] = i < nk ? weight_fx(key_to_float(key_at(i))) : 0ull;
      tsum += loc[j];
    }
    unsigned long long tot = 0;
    unsigned long long run = ab.w + block_scan_u64(tsum, &tot);
    const bool whole = heavy && (kc == 0 || (P.a.mode & CLSAMPLE_MODE_JOINT_TOPK_TOPP));
    const unsigned long long W = whole ? ab.wall : ab.w + tot;
    const unsigned long long thr = ceil_scaled(W, q.p);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = 8 * (int)threadIdx.x + j;
      if (i < nk) w[i] = run;
      run += loc[j];
    }
    __syncthreads();
    int c = 0;
    for (int i = threadIdx.x; i < nk; i += kThreads) c += w[i] < thr;
    c = block_sum_i(c);
    np = c >= 1 ? count_ge(nk, key_at(c - 1)) : 0;
  }
  // min-p: y >= L, again a prefix
  int K = np;
  if (q.mp > 0.0f) {
    int c = 0;
    for (int i = threadIdx.x; i < np; i += kThreads) c += key_to_float(key_at(i)) >= q.L;
    K = block_sum_i(c);
  }
  // race over the kept prefix (and its mass, for the kept-set logprob)
  float bs = -INFINITY, by = 0.0f, sk = 0.0f;
  int bid = INT_MAX;
  const bool want_kept = P.a.logprobs_kept != nullptr;
  for (int i = threadIdx.x; i < K; i += kThreads) {
    const float y = key_to_float(key_at(i));
    const int id = sorted_id(k[i]);
    if (want_kept) sk += ex2_approx(y * 1.4426950408889634f);
    const uint4 wv = race_words((uint32_t)id >> 2, q.seed, q.pos);
    const uint32_t x = pick_word(wv, id & 3);
    if (fast_race(y, x) >= bs - kFastTol) {
      const float sc = race_score(y, x);
      if (better(sc, id, bs, bid)) {
        bs = sc;
        bid = id;
        by = y;
      }
    }
  }
  block_race(bs, bid, by);
  if (want_kept) sk = block_sum_f2(sk) + ab.skept;
  const bool from_above = ab.rtok != INT_MAX && better(ab.rs, ab.rtok, bs, bid);
  float ztok = 0.0f;
  if (P.a.logprobs_orig) ztok = from_above ? ab.ztok : (bid == INT_MAX ? R.m : find_item_z(bid));
  if (threadIdx.x == 0) {
    float ymin = K > 0 ? key_to_float(key_at(K - 1)) : INFINITY;
    if (from_above) {
      bs = ab.rs;
      bid = ab.rtok;
      by = ab.ytok;
    }
    ymin = fminf(ymin, ab.ymin);
    int st = status;
    if (bid == INT_MAX) st = kRowOverflow;
    write_row(P.a, row, st, bid == INT_MAX ? R.arg : bid, by - lnS, K + ab.kept, ymin,
              __fsub_rn(ztok, R.m) - sh.lnS1, by - logf(sk));
  }
}

// Narrows the finisher's items to those at or above the digit range that holds the
// krem-th largest key, once that set has at most kSortCap items (histogram rounds as in
// select_kth), and leaves them in fin_items as sorted composites (sh.fin_n, sh.fin_smem).
// The kept set of a row with a top-k cut lies inside that set.  False if no round gets
// the set small enough.
__device__ bool prefilter_kth(const Smem& S, int chunk, float m, float invT, int krem) {
  uint32_t* hc = fin_hc(S, chunk);
  uint32_t prefix = 0, lo_key = 0;
  int surv = -1, A = 0;  // A: items above the current digit range
  for (int r = 0; r < 3 && surv < 0; ++r) {
    const int sft = digit_shift(r);
    const uint32_t dmask = (1u << digit_width(r)) - 1u;
    for (int t = threadIdx.x; t < kDigitBins; t += kThreads) hc[t] = 0u;
    if (threadIdx.x == 0) sh.digit = -1;
    __syncthreads();
    visit(S, m, invT, [&](float y, int) {
      const uint32_t key = fkey(y);
      if (digit_match(key, r, prefix)) atomicAdd(&hc[(key >> sft) & dmask], 1u);
    });
    __syncthreads();
    int c = 0;
    for (int d = kBPT * (int)threadIdx.x; d < kBPT * (int)threadIdx.x + kBPT; ++d) c += (int)hc[d];
    int tot = 0;
    const int pre = block_scan_i(c, &tot);
    const int above = tot - pre - c;
    if (above < krem && above + c >= krem) {
      int run = above;
      for (int d = kBPT * (int)threadIdx.x + kBPT - 1; d >= kBPT * (int)threadIdx.x; --d) {
        if (run + (int)hc[d] >= krem) {
          sh.digit = d;
          sh.cnt = run;
          sh.flag = run + (int)hc[d];
          break;
        }
        run += (int)hc[d];
      }
    }
    __syncthreads();
    if (sh.digit < 0) return false;
    const int in_above = sh.cnt, in_incl = sh.flag;
    prefix = (prefix << digit_width(r)) | (uint32_t)sh.digit;
    if (A + in_incl <= kSortCap) {
      lo_key = prefix << sft;  // every item at or above this digit's lower edge
      surv = 1;
    }
    A += in_above;
    krem -= in_above;
    __syncthreads();
  }
  if (surv < 0) return false;
  // compact the survivors as composites into the histogram area, then sort them into place
  unsigned long long* tmp = reinterpret_cast<unsigned long long*>(hc);
  if (threadIdx.x == 0) sh.cnt = 0;
  __syncthreads();
  visit(S, m, invT, [&](float y, int id) {
    const uint32_t key = fkey(y);
    if (key >= lo_key) {
      const int pos = atomicAdd(&sh.cnt, 1);
      if (pos < kSortCap) tmp[pos] = ((unsigned long long)key << 32) | (uint32_t)(~(uint32_t)id);
    }
  });
  __syncthreads();
  const int n = min(sh.cnt, kSortCap);
  unsigned long long* k = reinterpret_cast<unsigned long long*>(fin_items(S));
  for (int i = threadIdx.x; i < n; i += kThreads) k[i] = tmp[i];
  __syncthreads();
  sort_desc(k, n);
  if (threadIdx.x == 0) {
    sh.fin_n = n;
    sh.fin_smem = 1;
  }
  __syncthreads();
  return sh.cnt <= kSortCap;
}
static_assert(kSortCap * 8 <= kFinHistBytes, "survivors fit the histogram area");

// ---------------------------------------------------------------- row end: finisher

template <bool kBF16>
__device__ void reprocess_slice(const LaunchParams& P, const Smem& S, const RowParams& q, int row, int s);

// Above-band aggregates of a heavy row (zero for light rows).
struct Above {
  unsigned n;             // tokens above the band (all allowed ones)
  unsigned long long w;   // their exact mass
  unsigned long long wall;  // mass of every allowed token (heavy rows without a top-k cut)
  float rs, ytok, ymin;   // best race among the surely-kept ones, its y, smallest kept y
  int rtok, kept;
  float skept, ztok;      // sum of e^y over the surely-kept ones; z' of rtok
};

// Requested token ids: every slice CTA stores z' of the ids inside its slice in the
// output slots (written before the slice's ticket, so the row end sees them) and flags
// the row INVALID if an id or the row's offsets are out of range.
__device__ __noinline__ void capture_tids(const LaunchParams& P, const Smem& S, int row, int c0, int n) {
  const int lo = P.a.tid_offs[row], hi = P.a.tid_offs[row + 1];
  int bad = lo < 0 || hi < lo;
  if (!bad)
    for (int j = lo + threadIdx.x; j < hi; j += kThreads) {
      const int id = __ldg(P.a.tid_ids + j);
      if (id < 0 || id >= P.a.V) bad = 1;
      else if (id >= c0 && id < c0 + n) P.a.tid_logprobs[j] = S.buf[id - c0];
    }
  if (__syncthreads_or(bad) && threadIdx.x == 0) sh.rec.flags |= kFlagInvalid;
}

// Row end of the requested ids: z' -> y - ln S in place (-inf for masked ids and for
// every id of an INVALID row).
__device__ __noinline__ void finish_tids(const LaunchParams& P, int row, int status, float m, float invT, float lnS) {
  const int lo = P.a.tid_offs[row], hi = P.a.tid_offs[row + 1];
  if (lo < 0 || hi < lo) return;  // nothing addressable: the row is INVALID
  for (int j = lo + threadIdx.x; j < hi; j += kThreads) {
    float v = -INFINITY;
    if (status != kRowInvalid) {
      const float z = __ldcg(P.a.tid_logprobs + j);
      if (z > -INFINITY) v = y_of(z, m, invT) - lnS;
    }
    P.a.tid_logprobs[j] = v;
  }
}

// Top-N logprobs.  The order is "more probable first": y is monotone in z', so tokens are
// ranked by z' descending and equal z' by id ascending -- a key no slice needs the row
// max for.  Larger key = ranked earlier; 0 is never a token's key.
__device__ __forceinline__ unsigned long long zid_key(float z, int id) {
  uint32_t u = __float_as_uint(z == 0.0f ? 0.0f : z);  // -0 and +0 are one value
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (0xFFFFFFFFu - (uint32_t)id);
}
__device__ __forceinline__ Item key_item(unsigned long long k) {
  uint32_t u = (uint32_t)(k >> 32);
  u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  return Item{__uint_as_float(u), (int)(0xFFFFFFFFu - (uint32_t)k)};
}
__device__ unsigned long long block_max_u64(unsigned long long v) {
  __shared__ unsigned long long red[kWarps];
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const unsigned long long t = __shfl_xor_sync(~0u, v, o);
    v = t > v ? t : v;
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long r = red[0];
  for (int i = 1; i < kWarps; ++i) r = red[i] > r ? red[i] : r;
  return r;
}
__device__ __forceinline__ bool top_n_ok(const LaunchParams& P, int N) {
  return N >= 0 && N <= kTopNMax && N <= P.a.top_n_stride;
}

// Each slice CTA writes its N highest-ranked allowed tokens (N rounds of a block-wide
// maximum below the previous one; z' = -inf marks an empty place) and flags the row
// INVALID for an N out of range.
__device__ __noinline__ void slice_top_n(const LaunchParams& P, const Smem& S, int row, int slice, int c0, int n) {
  const int N = P.a.top_ns[row];
  if (!top_n_ok(P, N)) {
    if (threadIdx.x == 0) sh.rec.flags |= kFlagInvalid;
    return;
  }
  Item* dst = P.topn + ((size_t)row * P.C + slice) * kTopNMax;
  unsigned long long prev = ~0ull;
  int r = 0;
  for (; r < N; ++r) {
    unsigned long long best = 0;
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const float z = S.buf[i];
      if (z > -INFINITY) {
        const unsigned long long k = zid_key(z, c0 + i);
        if (k < prev && k > best) best = k;
      }
    }
    best = block_max_u64(best);
    if (!best) break;  // uniform: the slice has no more allowed tokens
    if (threadIdx.x == 0) dst[r] = key_item(best);
    prev = best;
  }
  for (int j = r + (int)threadIdx.x; j < N; j += kThreads) dst[j] = Item{-INFINITY, -1};
}

// Row end of the top-N outputs: the slices' lists are ranked together in shared memory
// (each item's place = how many items rank above it) and the first N written with
// logprob y - ln S; places past the row's allowed tokens get -1 / -inf, as does every
// place of an INVALID row.
__device__ __noinline__ void finish_top_n(const LaunchParams& P, const Smem& S, int row, int status, float m,
                                          float invT, float lnS) {
  const int N = P.a.top_ns[row];
  if (!top_n_ok(P, N) || N == 0) return;  // nothing addressable (the row is INVALID) or wanted
  int32_t* oid = P.a.top_ids + (size_t)row * P.a.top_n_stride;
  float* olp = P.a.top_logprobs + (size_t)row * P.a.top_n_stride;
  for (int j = threadIdx.x; j < N; j += kThreads) {
    oid[j] = -1;
    olp[j] = -INFINITY;
  }
  if (status == kRowInvalid) return;
  const int C = P.C, tot = C * N;
  Item* it = reinterpret_cast<Item*>(S.buf);  // free at a row end: the finisher's items come later
  __syncthreads();
  for (int t = threadIdx.x; t < tot; t += kThreads)
    it[t] = ldcg_item(P.topn + ((size_t)row * C + t / N) * kTopNMax + t % N);
  __syncthreads();
  for (int t = threadIdx.x; t < tot; t += kThreads) {
    const Item x = it[t];
    if (!(x.z > -INFINITY)) continue;
    const unsigned long long k = zid_key(x.z, x.id);
    int rank = 0;
    for (int u = 0; u < tot; ++u) {
      const Item v = it[u];
      rank += (v.z > -INFINITY && zid_key(v.z, v.id) > k) ? 1 : 0;
    }
    if (rank < N) {
      oid[rank] = x.id;
      olp[rank] = y_of(x.z, m, invT) - lnS;
    }
  }
  __syncthreads();
}

// Finishes a row from its combined record (sh.row, sh.recs) and its items (candidates or
// band), exactly: top-k count select, top-p mass select over the top-k set, min-p, race.
template <bool kBF16>
__device__ void finish_row(const LaunchParams& P, const Smem& S, const RowParams& q, int row, const Above& ab,
                           bool heavy) {
  const SliceRec R = sh.row;
  int status = row_status_of(R);
  if (P.a.tid_offs) finish_tids(P, row, status, R.m, q.invT, sh.lnS);
  if (P.a.top_ns) finish_top_n(P, S, row, status, R.m, q.invT, sh.lnS);
  if (status == kRowInvalid) {
    if (threadIdx.x == 0) write_row(P.a, row, kRowInvalid, -1, -INFINITY, 0, -INFINITY);
    return;
  }
  const float m = R.m, invT = q.invT, lnS = sh.lnS;
  if (q.route == kRouteGreedy) {
    // z' of the argmax is m; a greedy row's kept set is the token alone
    if (threadIdx.x == 0) write_row(P.a, row, status, R.arg, -lnS, 1, 0.0f, -sh.lnS1, 0.0f);
    return;
  }
  const int C = P.C;
  const int kc = (q.k >= 2 && q.k < R.nallowed) ? q.k : 0;
  bool sorted = false;
  for (int attempt = 0;; ++attempt) {
    if (threadIdx.x == 0) {
      const int sc = atomicAdd(&P.rowctl[row].spill, 0);
      const int spill = sc > 0 ? sc - 1 : -1;
      int ns = 0;
      for (int s = 0; s < C; ++s) {
        const SliceRec& x = sh.recs[s];
        if (x.ncand <= 0) continue;
        if (!x.spilled) sh.seg[ns] = cand_area(P, row, s);
        else sh.seg[ns] = spill >= 0 ? spill_area(P, spill, s) : nullptr;
        sh.segn[ns] = sh.seg[ns] ? x.ncand : 0;
        ++ns;
      }
      float zmin = -INFINITY;
      if (!heavy && q.route == kRouteMinP) {
        const float edge = m + q.L * q.Teff;
        zmin = edge - bound_margin(m, edge);
      }
      sh.nseg = ns;
      sh.zmin = zmin;
    }
    __syncthreads();
    gather_items(S, P.chunk, m, invT);
    if (heavy || attempt > 0) break;
    // light rows: every token a slice left out must lie below the kept set -- y(zc) < Y_k
    // for top-k (all slices complete when there is no top-k cut), y(zc) < ln(min_p) for
    // min-p; slices that fail are redone in full (spilled) and the items gathered again
    float ybound = q.L;
    if (q.route == kRouteTopK) {
      ybound = -INFINITY;
      if (kc > 0 && kc <= sh.fin_n) {
        uint32_t key;
        if (sh.fin_smem && sh.fin_n <= kSortCap) {
          sort_items(S, P.chunk, sh.fin_n);
          sorted = true;
          key = (uint32_t)(reinterpret_cast<const unsigned long long*>(fin_items(S))[kc - 1] >> 32);
        } else if (prefilter_kth(S, P.chunk, m, invT, kc)) {
          sorted = true;  // the survivors (a superset of the top-k set) are sorted in place
          key = (uint32_t)(reinterpret_cast<const unsigned long long*>(fin_items(S))[kc - 1] >> 32);
        } else {
          key = select_kth(S, P.chunk, m, invT, kc);
        }
        ybound = key_to_float(key);
      }
    }
    if (threadIdx.x == 0) {
      int bad = 0;
      for (int s = 0; s < C; ++s) {
        const float zc = sh.recs[s].zc;
        if (zc > -INFINITY && !(y_of(zc, m, invT) < ybound)) bad |= 1 << s;
      }
      sh.flag = bad;
    }
    __syncthreads();
    const int bad = sh.flag;
    if (!bad) break;
    for (int s = 0; s < C; ++s)
      if ((bad >> s) & 1) reprocess_slice<kBF16>(P, S, q, row, s);
    sorted = false;
  }
  status = max(status, row_status_of(sh.row));  // a redone slice may have run out of spill room
  // many items and a top-k cut (heavy rows with k > kKMax): narrow them to a sortable set
  if (!sorted && !(sh.fin_smem && sh.fin_n <= kSortCap) && kc > 0) {
    const int krem = kc - (int)ab.n;
    if (krem >= 1 && krem <= sh.fin_n && prefilter_kth(S, P.chunk, m, invT, krem)) sorted = true;
  }
  // a heavy row without a top-k cut and many band items: its cut by radix mass selects
  // costs less than sorting them
  const bool by_digits = heavy && kc == 0 && !sorted && sh.fin_n > kHeavySortMax;
  if (sh.fin_smem && sh.fin_n <= kSortCap && !by_digits) {
    finish_sorted(P, S, q, row, ab, heavy, status, R, lnS, sorted);
    return;
  }
  int nitems = sh.fin_n;
  // top-k
  uint32_t tk = 0u;
  if (kc > 0) {
    const int krem = kc - (int)ab.n;
    if (krem >= 1 && krem <= nitems) tk = select_kth(S, P.chunk, m, invT, krem);
  }
  // top-p over the top-k set
  uint32_t cut = tk;
  if (q.p < 1.0f) {
    unsigned long long w = 0;
    visit(S, m, invT, [&](float y, int) {
      if (fkey(y) >= tk) w += weight_fx(y);
    });
    unsigned long long W = ab.w + block_sum_u64(w);
    // the base is the whole row without a top-k cut, and in the joint order
    if (heavy && (kc == 0 || (P.a.mode & CLSAMPLE_MODE_JOINT_TOPK_TOPP))) W = ab.wall;
    const unsigned long long thr = ceil_scaled(W, q.p);
    cut = select_mass(S, P.chunk, m, invT, tk, ab.w, thr);
  }
  // min-p and the race
  float bs = -INFINITY, by = 0.0f, ymin = INFINITY, sk = 0.0f;
  int bid = INT_MAX, kept = 0;
  const float L = q.L;
  const bool want_kept = P.a.logprobs_kept != nullptr;
  visit(S, m, invT, [&](float y, int id) {
    if (fkey(y) >= cut && y >= L) {
      ++kept;
      ymin = fminf(ymin, y);
      if (want_kept) sk += ex2_approx(y * 1.4426950408889634f);
      const float sc = race_of(y, id, q.seed, q.pos);
      if (better(sc, id, bs, bid)) {
        bs = sc;
        bid = id;
        by = y;
      }
    }
  });
  block_race(bs, bid, by);
  kept = block_sum_i(kept);
  ymin = block_min_f(ymin);
  if (want_kept) sk = block_sum_f2(sk) + ab.skept;
  const bool from_above = ab.rtok != INT_MAX && better(ab.rs, ab.rtok, bs, bid);
  float ztok = 0.0f;
  if (P.a.logprobs_orig) ztok = from_above ? ab.ztok : (bid == INT_MAX ? R.m : find_item_z(bid));
  if (threadIdx.x == 0) {
    if (from_above) {
      bs = ab.rs;
      bid = ab.rtok;
      by = ab.ytok;
    }
    kept += ab.kept;
    ymin = fminf(ymin, ab.ymin);
    int st = status;
    if (bid == INT_MAX) st = kRowOverflow;  // nothing kept: only if a limit was hit
    write_row(P.a, row, st, bid == INT_MAX ? R.arg : bid, by - lnS, kept, ymin,
              __fsub_rn(ztok, R.m) - sh.lnS1, by - logf(sk));
  }
}

// ---------------------------------------------------------------- heavy rows

// Arrive at the row barrier and wait (bounded) until `target` arrivals; false on timeout.
__device__ bool row_barrier(const LaunchParams& P, int row, unsigned target) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned* b = &P.rowctl[row].bar;
    atomicAdd(b, 1u);
    int ok = 0;
    for (uint32_t i = 0; i < kWaitPolls; ++i) {
      if (ld_acquire(b) >= target) {
        ok = 1;
        break;
      }
      __nanosleep(100);
    }
    sh.flag = ok;
  }
  __syncthreads();
  return sh.flag != 0;
}

__device__ __forceinline__ int ybin(float y) {
  const float t = -y * 4.0f;
  return t < (float)(kYBins - 1) ? (int)t : kYBins - 1;
}

// The C CTAs of a heavy row, after pass A: barrier 1 gives the row max; exact y-bin
// counts and masses (barrier 2) give the band of bins that holds the cut; each CTA races
// the tokens above the band in place and compacts the band.  `ab` gets the plan.
__device__ void heavy_slice(const LaunchParams& P, const Smem& S, const RowParams& q, int row, int slice, int c0,
                            int n, Above& ab) {
  const int C = P.C;
  publish_rec(P, row, slice);
  if (!row_barrier(P, row, (unsigned)C) && threadIdx.x == 0) sh.rec.flags |= kFlagOverflow;
  combine_row(P, row, q);
  ab = Above{0u, 0ull, 0ull, -INFINITY, 0.0f, INFINITY, INT_MAX, 0, 0.0f, 0.0f};
  if (threadIdx.x == 0) {
    sh.rec.ncand = 0;
    sh.rec.spilled = 0;
    sh.rec.rs = -INFINITY;
    sh.rec.rtok = INT_MAX;
    sh.rec.kept = 0;
    sh.rec.ymin = INFINITY;
    sh.rec.ytok = 0.0f;
  }
  const SliceRec R = sh.row;
  if (row_status_of(R) == kRowInvalid) {
    __syncthreads();
    return;
  }
  const float m = R.m, invT = q.invT;
  const int kc = (q.k >= 2 && q.k < R.nallowed) ? q.k : 0;
  const bool need_bins = kc > 0 || q.p < 1.0f;
  const int nv = (n + 3) >> 2;
  int blo = kYBins, bhi = -1;  // no band: every allowed token is surely kept
  if (need_bins) {
    SBins* B = S.bins;
    for (int t = threadIdx.x; t < kYBins; t += kThreads) {
      B->cnt[t] = 0u;
      B->lo[t] = 0u;
      B->hi[t] = 0u;
    }
    __syncthreads();
    const bool wm = q.p < 1.0f;
    // the open-ended last bin (most tokens of a wide row) is summed in registers
    unsigned clast = 0;
    unsigned long long wlast = 0;
    const float4* b4 = reinterpret_cast<const float4*>(S.buf);
    for (int f = threadIdx.x; f < nv; f += kThreads) {
      const float4 v = b4[f];
      const float zz[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (!(zz[j] > -INFINITY)) continue;
        const float y = y_of(zz[j], m, invT);
        const int b = ybin(y);
        const unsigned long long w = (wm && y > -28.0f) ? weight_fx(y) : 0ull;  // e^-28 < 2^-40
        if (b == kYBins - 1) {
          ++clast;
          wlast += w;
        } else {
          atomicAdd(&B->cnt[b], 1u);
          if (w) add_mass(&B->lo[b], &B->hi[b], w);
        }
      }
    }
    clast = (unsigned)warp_sum_i((int)clast);
    wlast = warp_sum_u64(wlast);
    if ((threadIdx.x & 31) == 0) {
      atomicAdd(&B->cnt[kYBins - 1], clast);
      add_mass(&B->lo[kYBins - 1], &B->hi[kYBins - 1], wlast);
    }
    __syncthreads();
    Bins* G = P.bins + (size_t)row * C + slice;
    for (int t = threadIdx.x; t < kYBins; t += kThreads) {
      G->cnt[t] = B->cnt[t];
      G->mass[t] = get_mass(&B->lo[t], &B->hi[t]);
    }
    if (!row_barrier(P, row, 2u * C) && threadIdx.x == 0) sh.rec.flags |= kFlagOverflow;
    // every CTA sums the row's bins and takes the same plan
    if (threadIdx.x < kYBins) {
      unsigned cs = 0;
      unsigned long long ws = 0;
      for (int s = 0; s < C; ++s) {
        const Bins* g = P.bins + (size_t)row * C + s;
        cs += __ldcg(&g->cnt[threadIdx.x]);
        ws += __ldcg(&g->mass[threadIdx.x]);
      }
      B->cnt[threadIdx.x] = cs;
      B->mass[threadIdx.x] = ws;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int bk = kYBins - 1;
      if (kc > 0) {
        unsigned cum = 0;
        for (int b = 0; b < kYBins; ++b) {
          cum += B->cnt[b];
          if (cum >= (unsigned)kc) {
            bk = b;
            break;
          }
        }
      }
      int lo = bk, hi = bk;
      if (q.p < 1.0f) {
        // sequential: a lower bound on the top-k set's mass (the bins above its band);
        // without a top-k cut, and in the joint order, the whole row's mass
        unsigned long long Wlo = 0;
        const int lim = (kc > 0 && !(P.a.mode & CLSAMPLE_MODE_JOINT_TOPK_TOPP)) ? bk : kYBins;
        for (int b = 0; b < lim; ++b) Wlo += B->mass[b];
        const unsigned long long thr = ceil_scaled(Wlo, q.p);
        int bp = kYBins - 1;
        unsigned long long cum = 0;
        for (int b = 0; b < kYBins; ++b) {
          cum += B->mass[b];
          if (cum >= thr) {
            bp = b;
            break;
          }
        }
        lo = kc > 0 ? min(bp, bk) : bp;
        // sequential: the top-p cut may lie anywhere up to the k-th token's bin.  Joint:
        // the kept set is the prefix up to the tighter of the two cuts, and every token
        // above either boundary bin passes both, so one bin decides
        hi = kc > 0 ? ((P.a.mode & CLSAMPLE_MODE_JOINT_TOPK_TOPP) ? lo : bk) : bp;
      }
      unsigned an = 0;
      unsigned long long aw = 0;
      for (int b = 0; b < lo; ++b) {
        an += B->cnt[b];
        aw += B->mass[b];
      }
      unsigned long long wall = 0;
      for (int b = 0; b < kYBins; ++b) wall += B->mass[b];
      sh.blo = lo;
      sh.bhi = hi;
      sh.above_n = an;
      sh.above_w = aw;
      sh.W = wall;
    }
    __syncthreads();
    blo = sh.blo;
    bhi = sh.bhi;
    ab.n = sh.above_n;
    ab.w = sh.above_w;
    ab.wall = sh.W;
  }
  // one walk: the surely-kept tokens (above the band, passing min-p) race in place, seeded
  // with the exact score of the row's argmax token (every kept set contains it), and the
  // band's tokens are compacted
  const float s0 = race_of(0.0f, R.arg, q.seed, q.pos);
  float bs = s0, by = 0.0f, ymin = INFINITY, bz = m, skept = 0.0f;
  int bid = R.arg, kept = 0;
  const float L = q.L;
  const bool band = bhi >= blo;
  const bool want_kept = P.a.logprobs_kept != nullptr;
  Item* cdst = cand_area(P, row, slice);
  if (threadIdx.x == 0) sh.cnt = 0;
  __syncthreads();
  {
    const float4* b4 = reinterpret_cast<const float4*>(S.buf);
    const int lane = threadIdx.x & 31;
    for (int f0 = 0; f0 < nv; f0 += kThreads) {
      const int f = f0 + threadIdx.x;
      const float4 v = f < nv ? b4[f] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      const float zz[4] = {v.x, v.y, v.z, v.w};
      float yy[4];
      unsigned km = 0, bm = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        yy[j] = -INFINITY;
        if (zz[j] > -INFINITY) {
          yy[j] = y_of(zz[j], m, invT);
          const int b = ybin(yy[j]);
          if (b < blo) {
            if (yy[j] >= L) {
              ++kept;
              ymin = fminf(ymin, yy[j]);
              if (want_kept) skept += ex2_approx(yy[j] * 1.4426950408889634f);
              // -ln(-ln U) <= kGumbelMax on the U grid: a token below bs - kGumbelMax cannot win
              if (yy[j] + kGumbelMax >= bs) km |= 1u << j;
            }
          } else if (b <= bhi) {
            bm |= 1u << j;
          }
        }
      }
      const int id0 = c0 + 4 * f;
      if (km) {
        const uint4 w = race_words((uint32_t)id0 >> 2, q.seed, q.pos);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (!((km >> j) & 1u)) continue;
          if (fast_race(yy[j], ww[j]) >= bs - kFastTol) {
            const float sc = race_score(yy[j], ww[j]);
            if (better(sc, id0 + j, bs, bid)) {
              bs = sc;
              bid = id0 + j;
              by = yy[j];
              bz = zz[j];
            }
          }
        }
      }
      if (band && __any_sync(~0u, bm != 0u)) {
        // the four ballots first, then one shared-memory atomic for the warp's step
        unsigned bal[4];
        int tot = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          bal[j] = __ballot_sync(~0u, (bm >> j) & 1u);
          tot += __popc(bal[j]);
        }
        int base = 0;
        if (lane == 0) base = atomicAdd(&sh.cnt, tot);
        base = __shfl_sync(~0u, base, 0);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if ((bal[j] >> lane) & 1u) {
            const int pos = base + __popc(bal[j] & ((1u << lane) - 1u));
            if (pos < kCandCap) cdst[pos] = Item{zz[j], id0 + j};
          }
          base += __popc(bal[j]);
        }
      }
    }
  }
  {
    // the winner's z' travels with its y (same owner thread)
    const int mine = bid;
    const float my_z = bz;
    block_race(bs, bid, by);
    if (mine == bid && bid != INT_MAX) sh.ztok = my_z;
  }
  kept = block_sum_i(kept);
  ymin = block_min_f(ymin);
  if (want_kept) {
    skept = warp_sum_f(skept);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sh.red_f2[threadIdx.x >> 5] = skept;
    __syncthreads();
    skept = 0.0f;
    for (int i = 0; i < kWarps; ++i) skept += sh.red_f2[i];
  }
  int nc = sh.cnt, spilled = 0;
  if (band && nc > kCandCap) {
    auto in_band = [&](float z) {
      const int b = ybin(y_of(z, m, invT));
      return b >= blo && b <= bhi;
    };
    if (threadIdx.x == 0) sh.spill = row_spill_slot(P, row);
    __syncthreads();
    if (sh.spill >= 0) {
      nc = compact_if(S, c0, n, in_band, spill_area(P, sh.spill, slice), P.chunk);
      spilled = 1;
    } else {
      nc = 0;
      if (threadIdx.x == 0) sh.rec.flags |= kFlagOverflow;
    }
  }
  if (threadIdx.x == 0) {
    sh.rec.rs = bs;
    sh.rec.rtok = bid;
    sh.rec.ytok = by;
    sh.rec.ztok = bid == R.arg ? m : sh.ztok;
    sh.rec.skept = skept;
    sh.rec.kept = kept;
    sh.rec.ymin = ymin;
    sh.rec.ncand = nc;
    sh.rec.spilled = spilled;
  }
  __syncthreads();
}

// Merges the heavy row's per-slice races into `ab` (after the final combine).
__device__ void heavy_above(Above& ab, int C) {
  ab.rs = -INFINITY;
  ab.rtok = INT_MAX;
  ab.ytok = 0.0f;
  ab.kept = 0;
  ab.ymin = INFINITY;
  ab.skept = 0.0f;
  ab.ztok = 0.0f;
  for (int s = 0; s < C; ++s) {
    const SliceRec& x = sh.recs[s];
    if (x.rtok != INT_MAX && better(x.rs, x.rtok, ab.rs, ab.rtok)) {
      ab.rs = x.rs;
      ab.rtok = x.rtok;
      ab.ytok = x.ytok;
      ab.ztok = x.ztok;
    }
    ab.kept += x.kept;
    ab.ymin = fminf(ab.ymin, x.ymin);
    ab.skept += x.skept;
  }
}

// ---------------------------------------------------------------- the sampler kernel

// Loads, transforms and masks slice `slice` of `row` into buf and runs pass A on it
// (sh.rec gets the slice statistics).
template <bool kBF16>
__device__ void slice_front(const LaunchParams& P, const Smem& S, const RowParams& q, int row, int slice, int c0,
                            int n, uint32_t bulk) {
  // the row's preparation facts, loaded at entry (a redone slice of a row end loads its
  // own; on a timeout the slices scan the CSRs themselves: ready stays 0)
  RowInfo ri{0, P.a.V, 0, 0};
  int e0 = 0, ne = 0;
  if (P.lists) {
    if (slice != sh.ri_slice) {
      if (threadIdx.x == 0) {
        sh.ri_ok = 0;
        sh.ri_slice = slice;
        if (wait_flag(P.rflag + row, 1u)) {
          const int4 v = __ldcg(reinterpret_cast<const int4*>(P.rinfo + row));
          const int* po = P.poff + (size_t)row * (P.C + 1) + slice;
          const int a0 = __ldcg(po), a1 = __ldcg(po + 1);
          sh.ri = RowInfo{v.x, v.y, v.z, v.w};
          sh.e0 = a0;
          sh.ne = a1 - a0;
          sh.ri_ok = 1;
        }
      }
      __syncthreads();
    }
    if (sh.ri_ok) {
      ri = sh.ri;
      e0 = sh.e0;
      ne = sh.ne;
    }
  }
  if (threadIdx.x == 0) {
    sh.rec.flags |= ri.flags;
    sh.nal_row = ri.nal;
  }
  if (ri.ready) {
    // the row's entries of this slice, listed by the preparation launch: mark them (the
    // checked walk of pass A must not sanitise them again) and keep up to two per thread
    // in registers until the logits have landed
    const PenEntry* seg = P.pent + (size_t)row * kPenRowCap + e0;
    const int nw = (n + 31) >> 5;
    for (int w = threadIdx.x; w < nw; w += kThreads) S.claim[w] = 0u;
    PenEntry mine[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int i = threadIdx.x + u * kThreads;
      mine[u].lid = -1;
      if (i < ne) {
        const int4 v = __ldcg(reinterpret_cast<const int4*>(seg + i));
        mine[u] = PenEntry{v.x, (unsigned)v.y, v.z, v.w};
      }
    }
    if (P.a.bitmask) {
      const int32_t* mrow = P.a.bitmask + (long long)row * P.a.bitmask_row_stride + (c0 >> 5);
      for (int w = threadIdx.x; w < nw; w += kThreads) S.mask[w] = (uint32_t)__ldg(mrow + w);
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 2; ++u)
      if (mine[u].lid >= 0) atomicOr(&S.claim[mine[u].lid >> 5], 1u << (mine[u].lid & 31));
    if (!slice_wait(bulk) && threadIdx.x == 0) sh.rec.flags |= kFlagOverflow;
    if (!bulk) __syncthreads();  // a slice of plain loads only (slice_wait did not sync)
    if (kBF16) widen_bf16(S, P.chunk, n);
    for (int i0 = 0; i0 < ne; i0 += 2 * kThreads) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        PenEntry e = mine[u];
        if (i0 > 0) {
          const int i = i0 + threadIdx.x + u * kThreads;
          e.lid = -1;
          if (i < ne) {
            const int4 v = __ldcg(reinterpret_cast<const int4*>(seg + i));
            e = PenEntry{v.x, (unsigned)v.y, v.z, v.w};
            atomicOr(&S.claim[e.lid >> 5], 1u << (e.lid & 31));
          }
        }
        if (e.lid < 0) continue;
        float z = sanitize(S.buf[e.lid]);
        if (e.cnt) z = apply_penalties(z, e.cnt, q.freq, q.pres, q.rep);
        if (e.bj >= 0) z = __fadd_rn(z, __ldg(P.a.bias_vals + e.bj));
        S.buf[e.lid] = guard(z);
      }
    }
    __syncthreads();
    pass_a(P, S, q, row, c0, n);
    return;
  }
  claim_tokens(P, S, q, c0, n);
  const int ntouch = sh.ntouch;
  if (ntouch > 0) transforms_prep(P, S, q, c0, n, 0);
  if (P.a.bitmask) {
    const int32_t* mrow = P.a.bitmask + (long long)row * P.a.bitmask_row_stride + (c0 >> 5);
    for (int w = threadIdx.x; w < ((n + 31) >> 5); w += kThreads) S.mask[w] = (uint32_t)__ldg(mrow + w);
  }
  if (!slice_wait(bulk) && threadIdx.x == 0) sh.rec.flags |= kFlagOverflow;
  if (!bulk) __syncthreads();  // a slice of plain loads only (slice_wait did not sync)
  if (kBF16) widen_bf16(S, P.chunk, n);
  for (int r0 = 0; r0 < ntouch; r0 += kPen) {
    if (r0 > 0) transforms_prep(P, S, q, c0, n, r0);
    transforms_apply(P, S, q, r0);
  }
  pass_a(P, S, q, row, c0, n);
}

// A light row's finisher redoes slice s whose candidate bound does not hold for the
// row max: the whole slice goes to the spill area.
template <bool kBF16>
__device__ void reprocess_slice(const LaunchParams& P, const Smem& S, const RowParams& q, int row, int s) {
  const int c0 = s * P.chunk;
  const int n = min(P.a.V - c0, P.chunk);
  slice_front<kBF16>(P, S, q, row, s, c0, n, slice_load<kBF16>(P, S, row, c0, n));
  const int nc = spill_slice(P, S, row, s, c0, n);
  if (threadIdx.x == 0) {
    if (nc < 0) {
      sh.recs[s].ncand = 0;
      sh.row.flags |= kFlagOverflow;
    } else {
      sh.recs[s].ncand = nc;
      sh.recs[s].spilled = 1;
    }
    sh.recs[s].zc = -INFINITY;
  }
  __syncthreads();
}

template <bool kBF16>
__global__ void __launch_bounds__(kThreads, 3) sampler_kernel(const __grid_constant__ LaunchParams P) {
  // No griddepcontrol.wait: this grid starts once every CTA of the preparation launch has
  // started (they trigger at entry), and waits only for the flags that launch sets.
  const Smem S = carve(P.chunk);
  const int C = P.C;
  if (threadIdx.x == 0) {
    // the counter is zero before the preparation launch runs, so the item is taken while
    // the order may still be in the making
    // the item and a first look at the order flag go out together; the flag's acquire
    // (a fence) follows once it reads set
    const unsigned item = atomicAdd(&P.ctl[0], 1u);
    const unsigned seen = ld_relaxed(&P.ctl[2]);
    if (seen == 1u) fence_acquire();
    sh.flag = seen == 1u || wait_flag(&P.ctl[2], 1u);
    // without the order (the wait gave up) the item's own row, which is below B, stands in
    sh.row_id = sh.flag ? __ldcg(P.order + item / (unsigned)C) : (int)(item / (unsigned)C);
    sh.slice = (int)(item % (unsigned)C);
    sh.bar_uses = 0;
  }
  __syncthreads();
  {
    // the slice copy starts before anything else is read
    const int c0 = sh.slice * P.chunk;
    sh.bulk = slice_load<kBF16>(P, S, sh.row_id, c0, min(P.a.V - c0, P.chunk));
  }
  if (threadIdx.x == 32) {
    // in parallel with the parameter loads: the row's preparation flag, then its facts
    // and this slice's entry range
    sh.ri_ok = 0;
    sh.ri_slice = sh.slice;
    if (P.lists && wait_flag(P.rflag + sh.row_id, 1u)) {
      const int4 v = __ldcg(reinterpret_cast<const int4*>(P.rinfo + sh.row_id));
      const int* po = P.poff + (size_t)sh.row_id * (P.C + 1) + sh.slice;
      const int a0 = __ldcg(po), a1 = __ldcg(po + 1);
      sh.ri = RowInfo{v.x, v.y, v.z, v.w};
      sh.e0 = a0;
      sh.ne = a1 - a0;
      sh.ri_ok = 1;
    }
  }
  if (threadIdx.x == 0) {
    load_params(P.a, sh.row_id, sh.rp);
    SliceRec z;
    memset(&z, 0, sizeof z);
    z.m = -INFINITY;
    z.arg = INT_MAX;
    z.flags = sh.rp.invalid | (sh.flag ? 0 : kFlagOverflow);
    z.zc = -INFINITY;
    z.rs = -INFINITY;
    z.rtok = INT_MAX;
    z.ymin = INFINITY;
    sh.rec = z;
  }
  __syncthreads();
  const int row = sh.row_id, slice = sh.slice;
  const RowParams& q = sh.rp;
  const int c0 = slice * P.chunk;
  const int n = min(P.a.V - c0, P.chunk);
  slice_front<kBF16>(P, S, q, row, slice, c0, n, sh.bulk);
  if (P.a.tid_offs) capture_tids(P, S, row, c0, n);
  if (P.a.top_ns) slice_top_n(P, S, row, slice, c0, n);
  Above ab{0u, 0ull, 0ull, -INFINITY, 0.0f, INFINITY, INT_MAX, 0, 0.0f, 0.0f};
  const bool heavy = q.route == kRouteHeavy;
  if (heavy) heavy_slice(P, S, q, row, slice, c0, n, ab);
  else if (q.route != kRouteGreedy) light_candidates(P, S, q, row, slice, c0, n);
  // publish the slice record (the barrier orders every thread's candidate writes before
  // thread 0's cumulative release) and take the row's ticket
  __syncthreads();
  if (threadIdx.x == 0) {
    P.srec[(size_t)row * P.C + slice] = sh.rec;
    sh.last = atomic_add_acq_rel(&P.rowctl[row].ticket, 1u) == (unsigned)(C - 1);
    sh.flag = 0;
  }
  __syncthreads();
  if (sh.last) {
    combine_row(P, row, q);
    if (heavy) heavy_above(ab, C);
    finish_row<kBF16>(P, S, q, row, ab, heavy);
    // the row's control words go back to their initial state (every CTA of the row is past
    // its ticket), so a sampler grid that runs without its preparation launch still finds
    // them clean; the last row to finish clears the preparation flags for the next call:
    // by then every CTA of the grid has taken its item and read the flags
    __syncthreads();
    if (threadIdx.x == 0) {
      P.rowctl[row] = RowCtl{0u, 0u, 0, 0u};
      sh.flag = atomicAdd(&P.ctl[3], 1u) == (unsigned)(P.a.B - 1);
    }
    __syncthreads();
  }
  if (sh.flag) {
    if (P.lists)
      for (int r = threadIdx.x; r < P.a.B; r += kThreads) P.rflag[r] = 0u;
    if (threadIdx.x == 0) {
      P.ctl[0] = 0u;
      P.ctl[1] = 0u;
      P.ctl[2] = 0u;
      P.ctl[3] = 0u;
    }
  }
}

// ---------------------------------------------------------------- single-sweep fast path

#include "sweep.cuh"

// ---------------------------------------------------------------- diagnostics

// Allowed-token lists -> grammar bitmask rows: one CTA per row clears the row's words,
// then sets the bit of every listed id; a row with an id outside [0, V) or an empty list
// ends all-zero (every token masked), which the sampler reports as INVALID.
__global__ void allowed_to_bitmask_kernel(const int32_t* __restrict__ offs, const int32_t* __restrict__ ids, int V,
                                          int32_t* bitmask, long long stride) {
  __shared__ int bad;
  const int row = blockIdx.x;
  const int W = (V + 31) >> 5;
  int32_t* words = bitmask + (long long)row * stride;
  const int lo = offs[row], hi = offs[row + 1];
  if (threadIdx.x == 0) bad = lo < 0 || hi < lo;
  for (int w = threadIdx.x; w < W; w += blockDim.x) words[w] = 0;
  __syncthreads();
  if (!bad)
    for (int j = lo + threadIdx.x; j < hi; j += blockDim.x) {
      const int id = ids[j];
      if (id < 0 || id >= V) bad = 1;
      else atomicOr(reinterpret_cast<unsigned*>(words + (id >> 5)), 1u << (id & 31));
    }
  __syncthreads();
  if (bad)
    for (int w = threadIdx.x; w < W; w += blockDim.x) words[w] = 0;
}

__global__ void debug_weights_kernel(const float* y, unsigned long long* w, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) w[i] = weight_fx(y[i]);
}

__global__ void debug_uniforms_kernel(const uint64_t* seeds, const int64_t* pos, const int64_t* tok, float* u, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    const uint4 w = race_words((uint32_t)((unsigned long long)tok[i] >> 2), seeds[i], (unsigned long long)pos[i]);
    u[i] = word_to_uniform(pick_word(w, (int)(tok[i] & 3)));
  }
}

// ---------------------------------------------------------------- host side

struct Geometry {
  int C;      // slices per row
  int chunk;  // tokens per slice, multiple of 128
  int smem;   // dynamic shared memory per CTA
};

// C = ceil(V / kSliceMax) slices of equal length (rounded up to 128 tokens); the last
// slice holds the rest.  Shared memory does not depend on the logits type.
Geometry geometry_for(int vocab) {
  Geometry g{0, 0, 0};
  if (vocab <= 0 || vocab > kMaxVocab) return g;
  const int c0 = (vocab + kSliceMax - 1) / kSliceMax;
  const int chunk = ((vocab + c0 - 1) / c0 + 127) / 128 * 128;
  g.C = (vocab + chunk - 1) / chunk;
  g.chunk = chunk;
  g.smem = (int)layout_for(chunk).total;
  return g;
}

// Byte offsets of the scratch arrays for B rows of C slices of `chunk` tokens.
struct ScratchLayout {
  size_t ctl, order, rowctl, srec, bins, cand, spill, rinfo, poff, pent, rflag, topn, sw_rec, sw_cand, sw_tick, total;
};

constexpr size_t take(size_t& off, size_t bytes) {
  const size_t o = off;
  off = align_up(off + bytes, 256);
  return o;
}

constexpr ScratchLayout scratch_layout(size_t B, size_t C, size_t chunk, size_t spill_rows) {
  ScratchLayout L{};
  size_t off = 0;
  L.ctl = take(off, 4 * sizeof(unsigned));
  L.order = take(off, B * sizeof(int));
  L.rowctl = take(off, B * sizeof(RowCtl));
  L.srec = take(off, B * C * sizeof(SliceRec));
  L.bins = take(off, B * C * sizeof(Bins));
  L.cand = take(off, B * C * kCandCap * sizeof(Item));
  L.spill = take(off, spill_rows * C * chunk * sizeof(Item));
  L.rinfo = take(off, B * sizeof(RowInfo));
  L.poff = take(off, B * (C + 1) * sizeof(int));
  L.pent = take(off, B * kPenRowCap * sizeof(PenEntry));
  L.rflag = take(off, B * sizeof(unsigned));
  L.topn = take(off, B * C * kTopNMax * sizeof(Item));
  L.sw_rec = take(off, B * kSwMaxC * sizeof(SweepRec));
  L.sw_cand = take(off, B * kSwMaxC * kSwCand * sizeof(Item));
  L.sw_tick = take(off, B * sizeof(unsigned));
  L.total = off;
  return L;
}


struct Scratch {
  int max_batch;
  int C;
  int chunk;
  int spill_rows;
  unsigned char* base;
};

// Checks the device (compute capability 10.3, enough shared memory) and sets the
// kernels' shared-memory limits.
int setup_device(int dev) {
  int major = 0, minor = 0, optin = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return CLSAMPLE_ERR_CUDA;
  if (major != 10 || minor != 3) return CLSAMPLE_ERR_DEVICE;
  const int smem = (int)layout_for(kSliceMax).total;
  if (smem > optin) return CLSAMPLE_ERR_DEVICE;
  const void* k32 = reinterpret_cast<const void*>(&sampler_kernel<false>);
  const void* k16 = reinterpret_cast<const void*>(&sampler_kernel<true>);
  const void* ko = reinterpret_cast<const void*>(&order_kernel);
  if (cudaFuncSetAttribute(ko, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrepSmem) != cudaSuccess ||
      cudaFuncSetAttribute(k32, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(k16, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(k32, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
          cudaSuccess ||
      cudaFuncSetAttribute(k16, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
          cudaSuccess)
    return CLSAMPLE_ERR_CUDA;
  return CLSAMPLE_SUCCESS;
}

// Resident CTAs of the sampler kernel on device `dev` (reported by clsample_occupancy).
int resident_ctas(const Geometry& g, bool bf16, int dev, int* out) {
  int sms = 0, per = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return CLSAMPLE_ERR_CUDA;
  const cudaError_t err =
      bf16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, sampler_kernel<true>, kThreads, (size_t)g.smem)
           : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, sampler_kernel<false>, kThreads, (size_t)g.smem);
  if (err != cudaSuccess) return CLSAMPLE_ERR_CUDA;
  *out = sms * per;
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
// (every device that loads the library holds it until the process exits), sized for
// kStaticRows rows of the longest slices and kStaticSpill spill rows.
constexpr int kStaticRows = 64;
constexpr int kStaticSpill = 4;
constexpr size_t kStaticBytes = scratch_layout(kStaticRows, kMaxSlices, kSliceMax, kStaticSpill).total;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mutex;
unsigned char* g_static_base[kMaxDevices];  // the array's device address on each device, once set up

// The static scratch of device `dev`: on the first call for a device (with that device
// current) the kernels are set up and the array's device address is looked up with
// cudaGetSymbolAddress; nullptr with *rc set on failure.
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
    case CLSAMPLE_ERR_MODE: return "unknown mode bit";
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
  // one spill row per batch row: a row takes at most one, so no valid row runs out
  const int spill_rows = max_batch;
  unsigned char* base = nullptr;
  if (max_batch > 0) {
    const size_t bytes = scratch_layout((size_t)max_batch, (size_t)g.C, (size_t)g.chunk, (size_t)spill_rows).total;
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
  h->sc = Scratch{max_batch, g.C, g.chunk, spill_rows, base};
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
int make_params(const Geometry& g, int vocab, int dev, const Scratch& sc, const clsample_args_t* a,
                LaunchParams* P) {
  if (!a) return CLSAMPLE_ERR_NULL;
  if (a->B < 0 || a->B > sc.max_batch) return CLSAMPLE_ERR_BATCH;
  if (a->V != vocab) return CLSAMPLE_ERR_VOCAB;
  if (a->logits_dtype != CLSAMPLE_LOGITS_F32 && a->logits_dtype != CLSAMPLE_LOGITS_BF16) return CLSAMPLE_ERR_DTYPE;
  if (a->mode & ~(CLSAMPLE_MODE_JOINT_TOPK_TOPP | CLSAMPLE_MODE_SCORE_ONLY | CLSAMPLE_MODE_FAST_SWEEP))
    return CLSAMPLE_ERR_MODE;
  // the single sweep has neither requested-id nor top-N logprobs
  if ((a->mode & CLSAMPLE_MODE_FAST_SWEEP) && (a->tid_offs || a->top_ns)) return CLSAMPLE_ERR_MODE;
  if (a->B == 0) return CLSAMPLE_SUCCESS;
  if (!a->logits || !a->tokens) return CLSAMPLE_ERR_NULL;
  if (a->hist_offs && !a->hist_ids) return CLSAMPLE_ERR_NULL;
  if (a->bias_offs && (!a->bias_ids || !a->bias_vals)) return CLSAMPLE_ERR_NULL;
  if (a->tid_offs && (!a->tid_ids || !a->tid_logprobs)) return CLSAMPLE_ERR_NULL;
  if (a->top_ns && (!a->top_ids || !a->top_logprobs)) return CLSAMPLE_ERR_NULL;
  if (a->top_ns && a->top_n_stride < 1) return CLSAMPLE_ERR_STRIDE;
  if (a->logits_row_stride < a->V) return CLSAMPLE_ERR_STRIDE;
  if (a->bitmask && a->bitmask_row_stride < (a->V + 31) / 32) return CLSAMPLE_ERR_STRIDE;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return CLSAMPLE_ERR_CUDA;
  if (cur != dev) return CLSAMPLE_ERR_DEVICE;
  const int esize = a->logits_dtype == CLSAMPLE_LOGITS_BF16 ? 2 : 4;
  P->a = *a;
  P->C = g.C;
  P->chunk = g.chunk;
  const uintptr_t lb = reinterpret_cast<uintptr_t>(a->logits);
  P->vec_ok = (lb % 16 == 0) && (((long long)a->logits_row_stride * esize) % 16 == 0);
  P->spill_rows = sc.spill_rows;
  const ScratchLayout L = scratch_layout((size_t)sc.max_batch, (size_t)sc.C, (size_t)sc.chunk, (size_t)sc.spill_rows);
  unsigned char* b = sc.base;
  P->ctl = reinterpret_cast<unsigned*>(b + L.ctl);
  P->order = reinterpret_cast<int*>(b + L.order);
  P->rowctl = reinterpret_cast<RowCtl*>(b + L.rowctl);
  P->srec = reinterpret_cast<SliceRec*>(b + L.srec);
  P->bins = reinterpret_cast<Bins*>(b + L.bins);
  P->cand = reinterpret_cast<Item*>(b + L.cand);
  P->spill = reinterpret_cast<Item*>(b + L.spill);
  P->rinfo = reinterpret_cast<RowInfo*>(b + L.rinfo);
  P->poff = reinterpret_cast<int*>(b + L.poff);
  P->pent = reinterpret_cast<PenEntry*>(b + L.pent);
  P->rflag = reinterpret_cast<unsigned*>(b + L.rflag);
  P->topn = reinterpret_cast<Item*>(b + L.topn);
  P->sw_c = (a->V + kSwSlice - 1) / kSwSlice;
  P->sw_rec = reinterpret_cast<SweepRec*>(b + L.sw_rec);
  P->sw_cand = reinterpret_cast<Item*>(b + L.sw_cand);
  P->sw_tick = reinterpret_cast<unsigned*>(b + L.sw_tick);
  P->lists = (a->hist_offs || a->bias_offs || a->bitmask) ? 1 : 0;
  return CLSAMPLE_SUCCESS;
}

int make_params(const clsample_t* h, const clsample_args_t* a, LaunchParams* P) {
  if (!h || !a) return CLSAMPLE_ERR_NULL;
  return make_params(h->g, h->vocab, h->device, h->sc, a, P);
}

// The preparation launch: CTA 0 orders the rows and resets the counters; with penalties,
// bias or a mask, CTAs 1..B list each row's entries.
int launch_order(const LaunchParams& P, cudaStream_t st) {
  const unsigned grid = P.lists ? 1u + (unsigned)P.a.B : 1u;
  order_kernel<<<grid, kOrderThreads, P.lists ? kPrepSmem : 0, st>>>(P);
  return cudaGetLastError() == cudaSuccess ? CLSAMPLE_SUCCESS : CLSAMPLE_ERR_CUDA;
}

// The single-sweep kernel: one CTA per (row, slice of kSwSlice tokens), no preparation.
int launch_sweep(const LaunchParams& P, cudaStream_t st) {
  const unsigned grid = (unsigned)(P.a.B * P.sw_c);
  if (P.a.logits_dtype == CLSAMPLE_LOGITS_BF16) sweep_kernel<true><<<grid, kSwThreads, 0, st>>>(P);
  else sweep_kernel<false><<<grid, kSwThreads, 0, st>>>(P);
  return cudaGetLastError() == cudaSuccess ? CLSAMPLE_SUCCESS : CLSAMPLE_ERR_CUDA;
}

// The sampler kernel (B x C CTAs), launched with programmatic stream serialisation: its
// CTAs may start while the ordering launch ahead of it finishes, and wait for it
// (griddepcontrol.wait) before they take items.
int launch_sampler(const Geometry& g, const LaunchParams& P, cudaStream_t st) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)(P.a.B * g.C), 1, 1);
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
  const int rc = make_params(h, a, &P);
  if (rc != CLSAMPLE_SUCCESS || a->B == 0) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (a->mode & CLSAMPLE_MODE_FAST_SWEEP) return launch_sweep(P, st);
  const int ro = launch_order(P, st);
  return ro != CLSAMPLE_SUCCESS ? ro : launch_sampler(h->g, P, st);
}

int clsample_prepare(clsample_t* h, const clsample_args_t* a, clsample_stream_t stream) {
  LaunchParams P;
  const int rc = make_params(h, a, &P);
  if (rc != CLSAMPLE_SUCCESS || a->B == 0) return rc;
  if (a->mode & CLSAMPLE_MODE_FAST_SWEEP) return CLSAMPLE_SUCCESS;  // the sweep has no preparation
  return launch_order(P, reinterpret_cast<cudaStream_t>(stream));
}

int clsample_sample(clsample_t* h, const clsample_args_t* a, clsample_stream_t stream) {
  LaunchParams P;
  const int rc = make_params(h, a, &P);
  if (rc != CLSAMPLE_SUCCESS || a->B == 0) return rc;
  if (a->mode & CLSAMPLE_MODE_FAST_SWEEP) return launch_sweep(P, reinterpret_cast<cudaStream_t>(stream));
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
  // the array is laid out for the longest slices; shorter geometries use a prefix of it
  const Scratch sc{kStaticRows, kMaxSlices, kSliceMax, kStaticSpill, base};
  LaunchParams P;
  rc = make_params(g, a->V, dev, sc, a, &P);
  if (rc != CLSAMPLE_SUCCESS || a->B == 0) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (a->mode & CLSAMPLE_MODE_FAST_SWEEP) return launch_sweep(P, st);
  rc = launch_order(P, st);
  return rc != CLSAMPLE_SUCCESS ? rc : launch_sampler(g, P, st);
}

int clsample_occupancy(clsample_t* h, int32_t logits_dtype, int32_t* resident_ctas_out) {
  if (!h || !resident_ctas_out) return CLSAMPLE_ERR_NULL;
  if (logits_dtype != CLSAMPLE_LOGITS_F32 && logits_dtype != CLSAMPLE_LOGITS_BF16) return CLSAMPLE_ERR_DTYPE;
  *resident_ctas_out = h->grid[logits_dtype == CLSAMPLE_LOGITS_BF16 ? 1 : 0];
  return CLSAMPLE_SUCCESS;
}

int clsample_allowed_to_bitmask(const int32_t* offs, const int32_t* ids, int32_t B, int32_t V, int32_t* bitmask,
                                int64_t bitmask_row_stride, clsample_stream_t stream) {
  if (B < 0 || B > (1 << 24) - 1) return CLSAMPLE_ERR_BATCH;
  if (V <= 0) return CLSAMPLE_ERR_VOCAB;
  if (bitmask_row_stride < (V + 31) / 32) return CLSAMPLE_ERR_STRIDE;
  if (B == 0) return CLSAMPLE_SUCCESS;
  if (!offs || !ids || !bitmask) return CLSAMPLE_ERR_NULL;
  allowed_to_bitmask_kernel<<<(unsigned)B, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      offs, ids, V, bitmask, (long long)bitmask_row_stride);
  return cudaGetLastError() == cudaSuccess ? CLSAMPLE_SUCCESS : CLSAMPLE_ERR_CUDA;
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
