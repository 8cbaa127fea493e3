// Single-sweep sampler (CLSAMPLE_MODE_FAST_SWEEP): for batches whose rows are all greedy
// or untruncated, the batch fast paths of the SGLang page ("Field groups": is_all_greedy,
// need_top_k/top_p/min_p_sampling; the sampler's simple-sampling branch) and the GLM
// page ("Sampling").  Such a row needs no select: a greedy row is the lowest-id argmax of
// z', an untruncated row the exponential race over every allowed token.  So one pass over
// the logits does all of it:
//
//   one CTA per (row, slice of kSwSlice tokens), each warp on a region of kSwRegion
//   tokens held in registers (coalesced vector loads, issued first);
//   while the loads fly, the row's history and bias lists are scanned for this slice's
//   tokens into a shared-memory table (count | bias entry), so no preparation launch; each
//   listed token's transformed value is then computed once, into its table entry;
//   the slice's transforms, mask, max / lowest argmax, allowed count and sums of
//   2^((z' - m_s) log2(e) / T) come from the registers; untruncated rows also race their
//   tokens with fast scores relative to the slice max and keep every token within
//   kSwTol of the slice's best fast score (the row's winner is among them, see below);
//   the CTA that takes a row's last ticket combines the slice records in slice order and
//   draws exactly from the candidates.
//
// Why the candidates hold the winner.  A token's exact score is y + G with y =
// fl(fl(z' - m) / T-form) against the row max m; its fast score is y_s + G~ with y_s the
// same against the slice max m_s.  Within a slice, y_s - y is the same constant up to
// rounding (< 2^-22 |y| invT-relative, about 5e-6 for any token that can win, whose y is
// above -20), and |G~ - G| < 1e-4 (fast_race).  So the row's winner, best in its slice by
// exact score, is within 2.1e-4 of the slice's best fast score; kSwTol is 2e-3.
//
// Included once by clsample.cu inside its anonymous namespace (it uses the row
// parameters, transforms and output helpers defined there).

constexpr int kSwThreads = 256;
constexpr int kSwWarps = kSwThreads / 32;
constexpr int kSwSlice = 8192;                   // tokens per CTA
constexpr int kSwRegion = kSwSlice / kSwWarps;   // tokens per warp
constexpr int kSwVec = kSwRegion / 128;          // vectors of 4 tokens per lane
constexpr int kSwMaxC = (kMaxVocab + kSwSlice - 1) / kSwSlice;
constexpr int kSwCand = 64;                      // race candidates a slice keeps
constexpr float kSwTol = 2e-3f;
constexpr unsigned kSwCountBits = 20;            // table entry: count | (bias entry + 1) << 20
constexpr unsigned kSwIneligible = 0x100;        // record flag: the row may not take this path
constexpr unsigned kSwSpill = 0x200;             // record flag: more candidates than kSwCand
static_assert(kSwVec * 128 * kSwWarps == kSwSlice, "whole vectors per lane");
static_assert(kSwMaxC <= kSwThreads, "one record per thread at the row end");

struct __align__(16) SweepRec {
  float m;         // max z' over the slice's allowed tokens (-inf: none)
  int arg;         // lowest id reaching it
  float s, s1;     // sums of 2^((z' - m) c) at T_eff and at T = 1
  float zmin;      // min allowed z'
  int nal;         // allowed tokens with z' > -inf
  int ncand;       // race candidates written
  unsigned flags;  // kFlagInvalid, kSwIneligible, kSwSpill
};


struct __align__(16) SweepShared {
  unsigned tab[kSwSlice];           // per token: history count | (bias entry + 1) << kSwCountBits
  unsigned listed[kSwSlice / 32];   // tokens with a table entry
  unsigned long long key[kSwWarps];
  float f[kSwWarps * 2];
  int i[kSwWarps * 2];
  unsigned flags, ncand;
  SweepRec rec[kSwMaxC];
  float lnS, lnS1;
};

// Row eligibility that needs only the parameters: greedy, or no top-p / min-p cut, and the
// table limits (2^20 history ids, 4095 bias entries).  A top-k that cuts is checked at the
// row end, where the allowed count is known.
__device__ __forceinline__ bool sweep_params_ok(const RowParams& q) {
  if (q.hhi - q.hlo >= (1 << kSwCountBits) || q.bhi - q.blo >= (1 << (32 - kSwCountBits)) - 1) return false;
  return q.route == kRouteGreedy || (q.p == 1.0f && q.mp == 0.0f);
}

__device__ __forceinline__ float sw_warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(~0u, v, o));
  return v;
}

template <bool kBF16>
__device__ __forceinline__ float4 sweep_load(const clsample_args_t& a, long long off, int t, int n, bool vec) {
  // tokens t .. t+3 of the slice (0 beyond its end: finite, masked later)
  if (kBF16) {
    const uint16_t* p = static_cast<const uint16_t*>(a.logits) + off + t;
    if (vec && t + 4 <= n) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
      return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                         __uint_as_float(w.y & 0xFFFF0000u));
    }
    float e[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) e[j] = t + j < n ? __uint_as_float((uint32_t)__ldg(p + j) << 16) : 0.0f;
    return make_float4(e[0], e[1], e[2], e[3]);
  } else {
    const float* p = static_cast<const float*>(a.logits) + off + t;
    if (vec && t + 4 <= n) return __ldg(reinterpret_cast<const float4*>(p));
    float e[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) e[j] = t + j < n ? __ldg(p + j) : 0.0f;
    return make_float4(e[0], e[1], e[2], e[3]);
  }
}

// The transforms of one listed token (sanitise, penalties, bias, overflow guard), in the
// order and arithmetic of the per-slice sampler.
__device__ __forceinline__ float sweep_transform(const clsample_args_t& a, const RowParams& q, float z, unsigned e) {
  z = sanitize(z);
  const unsigned c = e & ((1u << kSwCountBits) - 1u), bj = e >> kSwCountBits;
  if (c) z = apply_penalties(z, c, q.freq, q.pres, q.rep);
  if (bj) z = __fadd_rn(z, __ldg(a.bias_vals + q.blo + (int)bj - 1));
  return guard(z);
}

__device__ __forceinline__ float vget(const float4& v, int j) { return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w; }
__device__ __forceinline__ void vset(float4& v, int j, float z) {
  if (j == 0) v.x = z;
  else if (j == 1) v.y = z;
  else if (j == 2) v.z = z;
  else v.w = z;
}

template <bool kBF16>
__global__ void __launch_bounds__(kSwThreads, 4) sweep_kernel(const __grid_constant__ LaunchParams P) {
  __shared__ SweepShared X;
  __shared__ RowParams q;
  const clsample_args_t& a = P.a;
  const int C = P.sw_c;
  const int row = (int)blockIdx.x / C, slice = (int)blockIdx.x % C;
  const int c0 = slice * kSwSlice, n = min(kSwSlice, a.V - c0);
  const int wp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = wp * kSwRegion;
  const long long off = (long long)row * a.logits_row_stride + c0;
  // 1. the region's logits, all loads in flight before anything else
  float4 v[kSwVec];
  if (n == kSwSlice && P.vec_ok) {
    // a whole slice on aligned rows: plain vector loads, no tail
#pragma unroll
    for (int u = 0; u < kSwVec; ++u) v[u] = sweep_load<kBF16>(a, off, r0 + 4 * (lane + 32 * u), kSwSlice, true);
  } else {
#pragma unroll
    for (int u = 0; u < kSwVec; ++u) v[u] = sweep_load<kBF16>(a, off, r0 + 4 * (lane + 32 * u), n, P.vec_ok);
  }
  // the region's mask words, one per lane (word k covers tokens 32k .. 32k+31 of the region)
  unsigned mword = 0xFFFFFFFFu;
  if (a.bitmask && r0 + 32 * lane < n)
    mword = (unsigned)__ldg(a.bitmask + (long long)row * a.bitmask_row_stride + ((c0 + r0) >> 5) + lane);
  if (threadIdx.x == 0) {
    load_params(a, row, q);
    X.flags = q.invalid | (sweep_params_ok(q) ? 0u : kSwIneligible);
    X.ncand = 0;
  }
  const bool lists = a.hist_offs || a.bias_offs;
  // the row's first history ids and bias entries are loaded now, while the logits are in
  // flight (every thread reads the offsets itself, so nothing waits for thread 0)
  int h0 = 0, h1 = 0, b0 = 0, b1 = 0;
  if (a.hist_offs) {
    h0 = __ldg(a.hist_offs + row);
    h1 = __ldg(a.hist_offs + row + 1);
  }
  if (a.bias_offs) {
    b0 = __ldg(a.bias_offs + row);
    b1 = __ldg(a.bias_offs + row + 1);
  }
  // offsets that are bad or past the table's limits make the row INVALID or ineligible
  // (its parameters say so): no list is read then
  if (!(h0 >= 0 && h1 >= h0 && h1 - h0 < (1 << kSwCountBits))) h1 = h0;
  if (!(b0 >= 0 && b1 >= b0 && b1 - b0 < (1 << (32 - kSwCountBits)) - 1)) b1 = b0;
  int ids[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int j = h0 + u * kSwThreads + (int)threadIdx.x;
    ids[u] = j < h1 ? __ldg(a.hist_ids + j) : c0 - 1;
  }
  int bid = c0 - 1;
  float bval = 0.0f;
  if (b0 + (int)threadIdx.x < b1) {
    bid = __ldg(a.bias_ids + b0 + threadIdx.x);
    bval = __ldg(a.bias_vals + b0 + threadIdx.x);
  }
  if (lists) {
    uint4* t4 = reinterpret_cast<uint4*>(X.tab);
    for (int i = threadIdx.x; i < kSwSlice / 4; i += kSwThreads) t4[i] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x < kSwSlice / 32) X.listed[threadIdx.x] = 0u;
  }
  __syncthreads();
  // 2. this slice's part of the row's lists: history counts, and the last valid bias entry
  //    of each id (the largest entry index, kept in the high bits by a compare-and-swap
  //    whatever the order; the count in the low bits may change underneath: it retries)
  if (lists && !(X.flags & kSwIneligible)) {
    unsigned bad = 0;
    auto hist = [&](int id, int j) {
      if (j < h1 && (id < 0 || id >= a.V)) bad = 1;
      const int l = id - c0;
      if ((unsigned)l < (unsigned)n) {
        atomicAdd(&X.tab[l], 1u);
        atomicOr(&X.listed[l >> 5], 1u << (l & 31));
      }
    };
#pragma unroll
    for (int u = 0; u < 8; ++u) hist(ids[u], h0 + u * kSwThreads + (int)threadIdx.x);
    // longer histories: eight more ids in flight per thread each round
    for (int j0 = h0 + 8 * kSwThreads; j0 < h1; j0 += 8 * kSwThreads) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u * kSwThreads + (int)threadIdx.x;
        ids[u] = j < h1 ? __ldg(a.hist_ids + j) : c0 - 1;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) hist(ids[u], j0 + u * kSwThreads + (int)threadIdx.x);
    }
    for (int j = b0 + (int)threadIdx.x; j < b1; j += kSwThreads) {
      if (j != b0 + (int)threadIdx.x) {
        bid = __ldg(a.bias_ids + j);
        bval = __ldg(a.bias_vals + j);
      }
      if (bid < 0 || bid >= a.V || bval != bval) {
        bad = 1;
        continue;
      }
      const int l = bid - c0;
      if ((unsigned)l >= (unsigned)n) continue;
      const unsigned e = (unsigned)(j - b0 + 1);
      unsigned old = X.tab[l];
      while ((old >> kSwCountBits) < e) {
        const unsigned seen = atomicCAS(&X.tab[l], old, (old & ((1u << kSwCountBits) - 1u)) | (e << kSwCountBits));
        if (seen == old) break;
        old = seen;
      }
      atomicOr(&X.listed[l >> 5], 1u << (l & 31));
    }
    if (bad) atomicOr(&X.flags, kFlagInvalid);
    __syncthreads();
    // each listed token's transformed value, computed once from its raw logit (an L2 hit:
    // the slice was just loaded) and left in its table entry as float bits
    for (int wi = threadIdx.x; wi < kSwSlice / 32; wi += kSwThreads) {
      uint32_t bits = X.listed[wi];
      while (bits) {
        const int l = wi * 32 + __ffs(bits) - 1;
        bits &= bits - 1u;
        float z;
        if (kBF16) z = __uint_as_float((uint32_t)__ldg(static_cast<const uint16_t*>(a.logits) + off + l) << 16);
        else z = __ldg(static_cast<const float*>(a.logits) + off + l);
        X.tab[l] = __float_as_uint(sweep_transform(a, q, z, X.tab[l]));
      }
    }
    __syncthreads();
  }
  const unsigned lword = lists ? X.listed[(r0 >> 5) + lane] : 0u;
  // 3. raw check, sanitising (only when something was not finite), transforms, mask
  float chk = 0.0f;
#pragma unroll
  for (int u = 0; u < kSwVec; ++u) chk += (v[u].x + v[u].y) + (v[u].z + v[u].w);
  const bool nonfinite = __syncthreads_or(!(fabsf(chk) < INFINITY));
  int nal = 0;
  float tmax = -INFINITY;
  int tf = INT_MAX;
#pragma unroll
  for (int u = 0; u < kSwVec; ++u) {
    const int t = r0 + 4 * (lane + 32 * u);
    const int src = (lane >> 3) + 4 * u;
    const int sh4 = 4 * (lane & 7);
    uint32_t allow = (__shfl_sync(~0u, mword, src) >> sh4) & 0xFu;
    const uint32_t lst = (__shfl_sync(~0u, lword, src) >> sh4) & 0xFu;
    if (t + 4 > n) allow &= n > t ? (1u << (n - t)) - 1u : 0u;
    if (nonfinite) {
      v[u].x = (lst & 1u) ? v[u].x : sanitize(v[u].x);
      v[u].y = (lst & 2u) ? v[u].y : sanitize(v[u].y);
      v[u].z = (lst & 4u) ? v[u].z : sanitize(v[u].z);
      v[u].w = (lst & 8u) ? v[u].w : sanitize(v[u].w);
    }
    if (lst) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if ((lst >> j) & 1u) vset(v[u], j, __uint_as_float(X.tab[t + j]));
    }
    if (allow != 0xFu) {
      if (!(allow & 1u)) v[u].x = -INFINITY;
      if (!(allow & 2u)) v[u].y = -INFINITY;
      if (!(allow & 4u)) v[u].z = -INFINITY;
      if (!(allow & 8u)) v[u].w = -INFINITY;
    }
    nal += (v[u].x > -INFINITY) + (v[u].y > -INFINITY) + (v[u].z > -INFINITY) + (v[u].w > -INFINITY);
    const float vm = fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w));
    if (vm > tmax) {
      tmax = vm;
      tf = u;
    }
  }
  if (a.dbg_transformed) {
    float* d = a.dbg_transformed + (long long)row * a.V + c0;
#pragma unroll
    for (int u = 0; u < kSwVec; ++u) {
      const int t = r0 + 4 * (lane + 32 * u);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (t + j < n) d[t + j] = vget(v[u], j);
    }
  }
  // 4. slice max and lowest argmax (64-bit keys), allowed count
  int arg = INT_MAX;
  if (tmax > -INFINITY) {
#pragma unroll
    for (int u = 0; u < kSwVec; ++u)
      if (u == tf) {
        const int t = r0 + 4 * (lane + 32 * u);
        const int j = v[u].x == tmax ? 0 : v[u].y == tmax ? 1 : v[u].z == tmax ? 2 : 3;
        arg = c0 + t + j;
      }
  }
  unsigned long long key = tmax > -INFINITY ? ((unsigned long long)fkey(tmax) << 32) | (unsigned)(~(unsigned)arg) : 0ull;
#pragma unroll
  for (int o = 16; o; o >>= 1) key = max(key, __shfl_xor_sync(~0u, key, o));
  nal = warp_sum_i(nal);
  if (lane == 0) {
    X.key[wp] = key;
    X.i[wp] = nal;
  }
  __syncthreads();
  unsigned long long bkey = X.key[0];
  int snal = X.i[0];
  for (int i = 1; i < kSwWarps; ++i) {
    bkey = max(bkey, X.key[i]);
    snal += X.i[i];
  }
  const float ms = bkey ? key_to_float((uint32_t)(bkey >> 32)) : -INFINITY;
  // 5. sums against the slice max; the race of untruncated rows
  const float c = __fmul_rn(1.4426950408889634f, q.invT);
  const bool want1 = a.logprobs_orig != nullptr;
  float s = 0.0f, s1 = 0.0f, zmin = INFINITY;
  if (ms > -INFINITY) {
#pragma unroll
    for (int u = 0; u < kSwVec; ++u) {
      s += (ex2_approx((v[u].x - ms) * c) + ex2_approx((v[u].y - ms) * c)) +
           (ex2_approx((v[u].z - ms) * c) + ex2_approx((v[u].w - ms) * c));
      if (want1)
        s1 += (ex2_approx((v[u].x - ms) * 1.4426950408889634f) + ex2_approx((v[u].y - ms) * 1.4426950408889634f)) +
              (ex2_approx((v[u].z - ms) * 1.4426950408889634f) + ex2_approx((v[u].w - ms) * 1.4426950408889634f));
      if (a.dbg_cut) {
        const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (e[j] > -INFINITY) zmin = fminf(zmin, e[j]);
      }
    }
  }
  const bool race = q.route != kRouteGreedy && ms > -INFINITY && !(X.flags & kSwIneligible);
  float best = -INFINITY;  // this lane's best fast score
  if (race) {
#pragma unroll
    for (int u = 0; u < kSwVec; ++u) {
      float yy[4];
      unsigned any = 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float z = vget(v[u], j);
        yy[j] = z > -INFINITY ? y_of(z, ms, q.invT) : -INFINITY;
        if (yy[j] > -INFINITY && yy[j] + kGumbelMax >= best - kSwTol) any |= 1u << j;
      }
      if (any) {
        const int t0 = c0 + r0 + 4 * (lane + 32 * u);
        const uint4 x = race_words((uint32_t)t0 >> 2, q.seed, q.pos);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if ((any >> j) & 1u) best = fmaxf(best, fast_race(yy[j], pick_word(x, j)));
      }
    }
  }
  s = warp_sum_f(s);
  s1 = warp_sum_f(s1);
  zmin = warp_min(zmin);
  const float wbest = sw_warp_max(best);
  if (lane == 0) {
    X.f[wp] = s;
    X.f[kSwWarps + wp] = s1;
    X.i[kSwWarps + wp] = __float_as_int(zmin);
    X.key[wp] = (unsigned long long)__float_as_uint(wbest);
  }
  __syncthreads();
  float bs = -INFINITY;
  for (int i = 0; i < kSwWarps; ++i) bs = fmaxf(bs, __uint_as_float((uint32_t)X.key[i]));
  // 6. candidates: a lane whose best is within kSwTol of the slice's best walks its
  // tokens again and keeps every token within kSwTol
  if (race && best >= bs - kSwTol) {
    Item* dst = P.sw_cand + ((size_t)row * kSwMaxC + slice) * kSwCand;
#pragma unroll
    for (int u = 0; u < kSwVec; ++u) {
      const int t0 = c0 + r0 + 4 * (lane + 32 * u);
      const uint4 x = race_words((uint32_t)t0 >> 2, q.seed, q.pos);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float z = vget(v[u], j);
        if (!(z > -INFINITY)) continue;
        const float y = y_of(z, ms, q.invT);
        if (y + kGumbelMax < bs - kSwTol) continue;
        if (fast_race(y, pick_word(x, j)) >= bs - kSwTol) {
          const unsigned pos = atomicAdd(&X.ncand, 1u);
          if (pos < (unsigned)kSwCand) dst[pos] = Item{z, t0 + j};
        }
      }
    }
  }
  __syncthreads();
  // 7. the slice record, then the row's ticket
  if (threadIdx.x == 0) {
    SweepRec r;
    r.m = ms;
    r.arg = bkey ? (int)~(uint32_t)bkey : INT_MAX;
    r.s = 0.0f;
    r.s1 = 0.0f;
    r.zmin = INFINITY;
    for (int i = 0; i < kSwWarps; ++i) {
      r.s += X.f[i];
      r.s1 += X.f[kSwWarps + i];
      r.zmin = fminf(r.zmin, __int_as_float(X.i[kSwWarps + i]));
    }
    r.nal = snal;
    r.ncand = (int)min(X.ncand, (unsigned)kSwCand);
    r.flags = X.flags | (X.ncand > (unsigned)kSwCand ? kSwSpill : 0u);
    P.sw_rec[(size_t)row * kSwMaxC + slice] = r;
    X.flags = atomic_add_acq_rel(P.sw_tick + row, 1u) == (unsigned)(C - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (!X.flags) return;
  // 8. the row end (the CTA that took the last ticket)
  if (threadIdx.x < C) {
    const int4* src = reinterpret_cast<const int4*>(P.sw_rec + (size_t)row * kSwMaxC + threadIdx.x);
    int4* d = reinterpret_cast<int4*>(&X.rec[threadIdx.x]);
    d[0] = __ldcg(src);
    d[1] = __ldcg(src + 1);
  }
  if (threadIdx.x == 0) P.sw_tick[row] = 0u;  // every CTA of the row has taken its ticket
  __syncthreads();
  float m = -INFINITY, zm = INFINITY;
  int am = INT_MAX, nall = 0;
  unsigned fl = 0u;
  for (int i = 0; i < C; ++i) {
    const SweepRec& x = X.rec[i];
    if (better(x.m, x.arg, m, am)) {
      m = x.m;
      am = x.arg;
    }
    nall += x.nal;
    fl |= x.flags;
    zm = fminf(zm, x.zmin);
  }
  if (threadIdx.x == 0) {
    float S = 0.0f, S1 = 0.0f;
    if (m > -INFINITY)
      for (int i = 0; i < C; ++i)
        if (X.rec[i].m > -INFINITY) {
          S += X.rec[i].s * ex2_approx((X.rec[i].m - m) * c);
          S1 += X.rec[i].s1 * ex2_approx((X.rec[i].m - m) * 1.4426950408889634f);
        }
    X.lnS = logf(S);
    X.lnS1 = logf(S1);
  }
  const bool greedy = q.route == kRouteGreedy;
  int status = ((fl & kFlagInvalid) || q.invalid || !(m > -INFINITY)) ? kRowInvalid : kRowOk;
  // untruncated: no top-k cut either (k >= the allowed count keeps everything)
  if (status == kRowOk && !greedy && ((fl & kSwIneligible) || (q.k >= 2 && q.k < nall))) status = kRowInvalid;
  if (status == kRowOk && !greedy && (fl & kSwSpill)) status = kRowOverflow;
  // the exact race over the candidates
  float rs = -INFINITY, ry = 0.0f, rz = 0.0f;
  int rid = INT_MAX;
  if (status == kRowOk && !greedy) {
    for (int i = 0; i < C; ++i) {
      const Item* g = P.sw_cand + ((size_t)row * kSwMaxC + i) * kSwCand;
      for (int k = threadIdx.x; k < X.rec[i].ncand; k += kSwThreads) {
        const int2 it = __ldcg(reinterpret_cast<const int2*>(g + k));
        const float z = __int_as_float(it.x);
        const float y = y_of(z, m, q.invT);
        const uint4 x = race_words((uint32_t)it.y >> 2, q.seed, q.pos);
        const float sc = race_score(y, pick_word(x, it.y & 3));
        if (better(sc, it.y, rs, rid)) {
          rs = sc;
          rid = it.y;
          ry = y;
          rz = z;
        }
      }
    }
  }
  // block argmax of (score, id): 64-bit keys, then the owner publishes y and z'
  unsigned long long rk = rid == INT_MAX ? 0ull : ((unsigned long long)fkey(rs) << 32) | (unsigned)(~(unsigned)rid);
#pragma unroll
  for (int o = 16; o; o >>= 1) rk = max(rk, __shfl_xor_sync(~0u, rk, o));
  if (lane == 0) X.key[wp] = rk;
  __syncthreads();
  unsigned long long bk = X.key[0];
  for (int i = 1; i < kSwWarps; ++i) bk = max(bk, X.key[i]);
  if (bk && rid != INT_MAX && (((unsigned long long)fkey(rs) << 32) | (unsigned)(~(unsigned)rid)) == bk) {
    X.f[0] = ry;
    X.f[1] = rz;
    X.i[0] = rid;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const float lnS = X.lnS, lnS1 = X.lnS1;
    if (status == kRowInvalid) {
      write_row(a, row, kRowInvalid, -1, -INFINITY, 0, -INFINITY);
    } else if (greedy) {
      write_row(a, row, status, am, -lnS, 1, 0.0f, -lnS1, 0.0f);
    } else if (status == kRowOverflow || !bk) {
      write_row(a, row, kRowOverflow, -1, -INFINITY, 0, -INFINITY);
    } else {
      const float y = X.f[0], z = X.f[1];
      write_row(a, row, kRowOk, X.i[0], y - lnS, nall, y_of(zm, m, q.invT), __fsub_rn(z, m) - lnS1, y - lnS);
    }
  }
}
