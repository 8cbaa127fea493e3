"""Vocabulary-sharded sampling ("sample then gather"), simulated on the CPU.

When the LM head is split over tensor-parallel ranks, each rank holds the logits of a
contiguous range of the vocabulary.  The GLM page ("GLM-5.3 inference (7): output side",
its closing cost table) weighs gathering every row's full logits, O(B V), against each
shard sampling locally and merging per-shard results, O(B TP k), and names top-p's
global mass as the hard part.  This module states that protocol exactly, as a CPU
simulation (every GPU run here has one device): every rank holds columns [lo, lo + n)
of the transformed logits z' of all B rows and exchanges only per-row statistics, one
all-gather per round:

  1. the local max z' and its lowest id -> the row max m and the greedy token;
  2. with m, each token's tempered logit y = fl32(fl32(z' - m) * fl32(1/T)) and the local
     sum of e^y (the log-softmax normaliser), and by row class:
       top-k rows (k >= 2): the local top-k -- the tokens above the local k-th value and
         the group tied with it as (value, count, race winner); together they hold the
         row's top-k set, so the top-k cut, the top-p cut over the renormalised top-k
         set and the race need nothing more;
       top-p rows without a top-k cut: exact integer masses of 64 bins of the order key
         of y;
       min-p and untruncated rows: the local race winner among the kept tokens;
  3. top-p rows: bins are refined (64 sub-ranges of the bin that holds the cut) until
     the cut bin holds at most `band_cap` tokens or a single value of y, then those
     tokens are gathered and the cut is resolved exactly;
  4. top-p rows: the local race winner among the tokens at or above the cut.

Masses are integers (floor(e^y 2^52)), so sums do not depend on the order of shards or
tokens and every rank takes the same decisions; the race (the exponential race in its
Gumbel form, y - ln(-ln U) with U from Philox4x32-10 keyed by the row's seed and
position and counted by token id) is a max, order independent too.  The sharded result
therefore equals the one-shard result exactly for any split of the vocabulary.  The
arithmetic is float64 on the pages' definitions, not the CUDA kernel's fixed-point
exponential: rows where the two differ sit on a knife edge of the cut (see the tests).

Inputs are the transformed logits z' (penalties, bias and mask are per-token operations
each rank applies to its own columns); every row is assumed to have valid parameters.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Callable, List, Optional, Sequence

import numpy as np

F32 = np.float32
GREEDY_EPS = 1e-5
MASS_SHIFT = 52
NBINS = 64


# ----------------------------------------------------------------------------- race uniforms

_M0, _M1 = np.uint64(0xD2511F53), np.uint64(0xCD9E8D57)
_W0, _W1 = 0x9E3779B9, 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(ctr: np.ndarray, key: Sequence[int]) -> np.ndarray:
    """Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
    easy as 1, 2, 3", SC'11) on counters ctr[..., 4] (uint32) under one key (k0, k1)."""
    c = [ctr[..., i].astype(np.uint64) for i in range(4)]
    k0, k1 = int(key[0]) & 0xFFFFFFFF, int(key[1]) & 0xFFFFFFFF
    for i in range(10):
        if i:
            k0 = (k0 + _W0) & 0xFFFFFFFF
            k1 = (k1 + _W1) & 0xFFFFFFFF
        p0 = _M0 * c[0]
        p1 = _M1 * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c = [hi1 ^ c[1] ^ np.uint64(k0), lo1, hi0 ^ c[3] ^ np.uint64(k1), lo0]
    return np.stack([x.astype(np.uint32) for x in c], axis=-1)


def race_uniforms(seed: int, pos: int, ids: np.ndarray) -> np.ndarray:
    """U in (0, 1) of tokens `ids` of a row: word id & 3 of Philox at counter
    (id >> 2, position low, position high, 0) under the row's seed; (top 23 bits + 1/2) / 2^23."""
    ids = np.asarray(ids, np.int64)
    seed &= (1 << 64) - 1
    pos &= (1 << 64) - 1
    ctr = np.zeros(ids.shape + (4,), np.uint32)
    ctr[..., 0] = (ids >> 2).astype(np.uint32)
    ctr[..., 1] = pos & 0xFFFFFFFF
    ctr[..., 2] = pos >> 32
    x = philox4x32_10(ctr, (seed & 0xFFFFFFFF, seed >> 32))
    w = np.take_along_axis(x, (ids & 3)[..., None].astype(np.int64), axis=-1)[..., 0]
    return ((w >> np.uint32(9)).astype(np.float64) + 0.5) * 2.0 ** -23


# ----------------------------------------------------------------------------- rows

@dataclass
class RowParams:
    T: float
    k: int = -1
    p: float = 1.0
    mp: float = 0.0
    seed: int = 0
    pos: int = 0

    @property
    def greedy(self) -> bool:
        return self.T < GREEDY_EPS or self.k in (0, 1)

    @property
    def inv_t(self) -> F32:
        return F32(1.0) / F32(self.T if self.T >= GREEDY_EPS else 1.0)

    @property
    def L(self) -> float:
        """ln(min_p) rounded to single precision (the library's reading); -inf without min-p."""
        return float(F32(math.log(self.mp))) if self.mp > 0.0 else -math.inf


def _y(z: np.ndarray, m: float, inv_t: F32) -> np.ndarray:
    return ((z - F32(m)).astype(F32) * inv_t).astype(F32)


def _mass(y: np.ndarray) -> np.ndarray:
    return np.floor(np.exp(y.astype(np.float64)) * 2.0 ** MASS_SHIFT).astype(np.int64)


def _okey(y: np.ndarray) -> np.ndarray:
    """Order-preserving 32-bit key of float32 values (-0 folds onto +0)."""
    b = np.where(y == 0, F32(0), y).astype(F32).view(np.uint32).astype(np.uint64)
    return np.where(b & 0x80000000, (~b) & 0xFFFFFFFF, b | 0x80000000).astype(np.int64)


def _race_best(y: np.ndarray, ids: np.ndarray, q: RowParams):
    """(score, id, y) of the best race score among tokens ids (ties: lowest id), or None."""
    if len(ids) == 0:
        return None
    sc = y.astype(np.float64) - np.log(-np.log(race_uniforms(q.seed, q.pos, ids)))
    i = np.lexsort((ids, -sc))[0]
    return float(sc[i]), int(ids[i]), float(y[i])


def _better(a, b):
    if a is None:
        return False
    if b is None:
        return True
    return a[0] > b[0] or (a[0] == b[0] and a[1] < b[1])


def _ceil_p(W: int, p: float) -> int:
    """ceil(p W) exactly (p is a binary fraction)."""
    num, den = float(p).as_integer_ratio()
    return -((-W * num) // den)


# ----------------------------------------------------------------------------- per-shard rounds

class Shard:
    """One rank's columns [lo, lo + n) of z' for all rows."""

    def __init__(self, z: np.ndarray, lo: int, params: Sequence[RowParams]):
        self.z = np.asarray(z, F32)
        self.lo = lo
        self.q = list(params)
        self.ids = np.arange(lo, lo + self.z.shape[1], dtype=np.int64)

    def round1(self):
        """Per row: local max z' and its lowest id (None when no allowed token)."""
        out = []
        for r in range(self.z.shape[0]):
            z = self.z[r]
            ok = z > -np.inf
            if not ok.any():
                out.append(None)
                continue
            m = z[ok].max()
            out.append((float(m), int(self.ids[np.nonzero(z == m)[0][0]])))
        return out

    def round2(self, m: Sequence[Optional[float]], cls: Sequence[str]):
        out = []
        for r, q in enumerate(self.q):
            if m[r] is None:
                out.append(None)
                continue
            z = self.z[r]
            ok = z > -np.inf
            y = _y(z[ok], m[r], q.inv_t)
            ids = self.ids[ok]
            rec = {"S": float(np.exp(y.astype(np.float64)).sum()), "n": int(len(y))}
            if cls[r] == "greedy":
                pass  # only the normaliser of its logprob
            elif cls[r] == "topk":
                # the local top-k: the tokens above the local k-th value, and the group tied
                # with it as (value, count, its race winner) -- a flat row stays O(k)
                rec["tie"] = None
                if len(y) > q.k:
                    yk = np.sort(y)[::-1][q.k - 1]
                    above, tie = y > yk, y == yk
                    rec["cand"] = (y[above], ids[above])
                    rec["tie"] = (float(yk), int(tie.sum()), _race_best(y[tie], ids[tie], q))
                else:
                    rec["cand"] = (y, ids)
            elif cls[r] == "topp":
                key = _okey(y)
                rec["hist"] = _histogram(key, _mass(y), 0, 1 << 32)
            else:  # min-p or untruncated: race the kept tokens here
                keep = y >= q.L
                rec["race"] = _race_best(y[keep], ids[keep], q)
                rec["kept"] = int(keep.sum())
                rec["ymin"] = float(y[keep].min()) if keep.any() else math.inf
            out.append(rec)
        return out

    def refine(self, m, rows: dict):
        """Top-p rows: the histogram of key range [klo, khi) of each listed row, or the
        tokens there when `gather` is set."""
        out = {}
        for r, (klo, khi, gather) in rows.items():
            q = self.q[r]
            z = self.z[r]
            ok = z > -np.inf
            y = _y(z[ok], m[r], q.inv_t)
            key = _okey(y)
            sel = (key >= klo) & (key < khi)
            if gather:
                out[r] = (y[sel], self.ids[ok][sel])
            else:
                out[r] = _histogram(key[sel], _mass(y[sel]), klo, khi)
        return out

    def race_above(self, m, cuts: dict):
        """Top-p rows: the local race winner among tokens with y >= cut and y >= ln(min_p)."""
        out = {}
        for r, cut in cuts.items():
            q = self.q[r]
            z = self.z[r]
            ok = z > -np.inf
            y = _y(z[ok], m[r], q.inv_t)
            keep = (y >= cut) & (y >= q.L)
            out[r] = (_race_best(y[keep], self.ids[ok][keep], q), int(keep.sum()),
                      float(y[keep].min()) if keep.any() else math.inf)
        return out


def _edges(klo: int, khi: int) -> np.ndarray:
    return np.linspace(klo, khi, NBINS + 1).astype(np.int64)


def _histogram(key: np.ndarray, mass: np.ndarray, klo: int, khi: int):
    """Counts and integer masses of NBINS equal key ranges of [klo, khi), highest first."""
    e = _edges(klo, khi)
    b = np.clip(np.searchsorted(e, key, side="right") - 1, 0, NBINS - 1)
    cnt = np.bincount(b, minlength=NBINS)[::-1]
    ms = np.zeros(NBINS, dtype=object)
    for i in np.unique(b):
        ms[NBINS - 1 - i] = int(mass[b == i].astype(object).sum())
    return cnt.astype(np.int64), ms


# ----------------------------------------------------------------------------- the protocol

class LocalComm:
    """All ranks in one process: `allgather(fn)` runs fn(shard) for every shard."""

    def __init__(self, shards: List[Shard]):
        self.shards = shards

    def allgather(self, fn: Callable[[Shard], object]) -> list:
        return [fn(s) for s in self.shards]


class TorchComm:
    """One rank of a torch.distributed group: `allgather(fn)` runs fn on this rank's shard
    and all-gathers the (small) per-row statistics."""

    def __init__(self, shard: Shard, dist):
        self.shard = shard
        self.dist = dist

    def allgather(self, fn):
        out = [None] * self.dist.get_world_size()
        self.dist.all_gather_object(out, fn(self.shard))
        return out


def sample_sharded(params: Sequence[RowParams], comm, band_cap: int = 4096) -> dict:
    """Runs the protocol over `comm`; every rank returns the same per-row results:
    tokens, logprobs (y - ln sum e^y), kept_count, status (0 OK, 2 no allowed token) and
    the number of values exchanged per row (the communication volume)."""
    B = len(params)
    # round 1: row max and the lowest argmax
    r1 = comm.allgather(lambda s: s.round1())
    m, arg = [None] * B, [None] * B
    for shard_out in r1:
        for r, v in enumerate(shard_out):
            if v is not None and (m[r] is None or v[0] > m[r] or (v[0] == m[r] and v[1] < arg[r])):
                m[r], arg[r] = v
    cls = []
    for r, q in enumerate(params):
        if q.greedy:
            cls.append("greedy")
        elif q.k >= 2:
            cls.append("topk")  # a k at or above the allowed count keeps every candidate
        elif q.p < 1.0:
            cls.append("topp")
        else:
            cls.append("local")
    # round 2
    r2 = comm.allgather(lambda s: s.round2(m, cls))
    tokens = np.full(B, -1, np.int32)
    logp = np.full(B, -np.inf, np.float32)
    kept = np.zeros(B, np.int32)
    status = np.zeros(B, np.int32)
    volume = np.zeros(B, np.int64)
    S = np.zeros(B, np.float64)
    topp_rows = {}
    for r in range(B):
        if m[r] is None:
            status[r] = 2
            continue
        q = params[r]
        recs = [o[r] for o in r2 if o[r] is not None]
        S[r] = sum(x["S"] for x in recs)
        volume[r] += 2 * len(recs)
        if cls[r] == "greedy":
            tokens[r], logp[r], kept[r] = arg[r], -math.log(S[r]), 1
        elif cls[r] == "topk":
            tokens[r], kept[r], y_tok, vol = _merge_topk(recs, q)
            volume[r] += vol
            logp[r] = y_tok - math.log(S[r])
        elif cls[r] == "local":
            best = None
            for x in recs:
                if _better(x["race"], best):
                    best = x["race"]
            kept[r] = sum(x["kept"] for x in recs)
            volume[r] += 3 * len(recs)
            tokens[r], logp[r] = best[1], best[2] - math.log(S[r])
        else:
            cnt = sum(x["hist"][0] for x in recs)
            ms = np.array([sum(x["hist"][1][b] for x in recs) for b in range(NBINS)], dtype=object)
            volume[r] += 2 * NBINS * len(recs)
            topp_rows[r] = (0, 1 << 32, cnt, ms, 0, int(ms.sum()))
    # rounds 3 and 4 for top-p rows: refine the bin that holds the cut, then gather it
    cuts = {}
    while topp_rows:
        ask = {}
        for r, (klo, khi, cnt, ms, above, W) in topp_rows.items():
            thr = _ceil_p(W, params[r].p)
            e = _edges(klo, khi)[::-1]  # bin i (highest first) is keys [e[i+1], e[i])
            cum = above
            for i in range(NBINS):
                if cnt[i] and cum + int(ms[i]) >= thr:
                    break
                cum += int(ms[i])
            blo, bhi = int(e[i + 1]), int(e[i])
            if i == NBINS - 1:
                blo = klo
            if bhi - blo <= 1:
                # one value of y: a tie group whose mass above is below p W -- kept whole,
                # nothing to gather
                cuts[r] = _key_to_float(blo)
            else:
                ask[r] = (blo, bhi, bool(cnt[i] <= band_cap), cum, W)
        if not ask:
            break
        got = comm.allgather(lambda s: s.refine(m, {r: a[:3] for r, a in ask.items()}))
        nxt = {}
        for r, (blo, bhi, gather, cum, W) in ask.items():
            parts = [g[r] for g in got]
            volume[r] += (2 * NBINS if not gather else 2 * sum(len(p[1]) for p in parts)) * 1
            if gather:
                y = np.concatenate([p[0] for p in parts])
                ids = np.concatenate([p[1] for p in parts])
                keep = _topp_keep(y, ids, _mass(y), W, cum, params[r].p)
                # every token above the band is kept, and the band's first tie group (its
                # mass above is below p W), so the band's kept tokens end at the cut
                cuts[r] = float(y[keep].min())
            else:
                cnt2 = sum(p[0] for p in parts)
                ms2 = np.array([sum(p[1][b] for p in parts) for b in range(NBINS)], dtype=object)
                nxt[r] = (blo, bhi, cnt2, ms2, cum, W)
        topp_rows = nxt
    if cuts:
        got = comm.allgather(lambda s: s.race_above(m, cuts))
        for r in cuts:
            best = None
            kept[r] = 0
            for g in got:
                b, n, _ = g[r]
                kept[r] += n
                if _better(b, best):
                    best = b
            volume[r] += 3 * len(got)
            tokens[r], logp[r] = best[1], best[2] - math.log(S[r])
    return {"tokens": tokens, "logprobs": logp, "kept_count": kept, "status": status, "volume": volume}


def _merge_topk(recs, q: RowParams):
    """Top-k rows: the kept set from the shards' tokens above their local k-th values and
    their tie groups, then top-p over it (renormalised), min-p, and the race.  Returns
    (token, kept count, its y, values exchanged)."""
    ya = np.concatenate([x["cand"][0] for x in recs])
    ia = np.concatenate([x["cand"][1] for x in recs])
    ties = [x["tie"] for x in recs if x["tie"] is not None]
    vol = 2 * len(ia) + 5 * len(ties)
    # items: single tokens (count 1) and tie groups (count c), by value
    val = np.concatenate([ya.astype(np.float64), np.array([t[0] for t in ties], np.float64)])
    cnt = np.concatenate([np.ones(len(ya), np.int64), np.array([t[1] for t in ties], np.int64)])
    nal = int(sum(x["n"] for x in recs))
    keep = np.ones(len(val), bool)
    if q.k < nal:
        o = np.argsort(-val, kind="stable")
        cum = np.cumsum(cnt[o])
        yK = val[o][np.searchsorted(cum, q.k)]
        keep &= val >= yK
    if q.p < 1.0:
        # groups of equal value go in or out together; a group's mass is count x e^y
        v = val[keep]
        c = cnt[keep]
        mass = (_mass(v.astype(F32)).astype(object) * c.astype(object))
        W = int(mass.sum())
        thr = _ceil_p(W, q.p)
        order = np.argsort(-v, kind="stable")
        kv = np.zeros(len(v), bool)
        cum, i = 0, 0
        while i < len(order):
            j, g = i, 0
            while j < len(order) and v[order[j]] == v[order[i]]:
                g += mass[order[j]]
                j += 1
            if cum < thr:
                kv[order[i:j]] = True
            cum += g
            i = j
        kk = np.zeros(len(val), bool)
        kk[np.nonzero(keep)[0][kv]] = True
        keep = kk
    keep &= val >= q.L
    na = len(ya)
    best = _race_best(ya[keep[:na]], ia[keep[:na]], q)
    for t, kt in zip(ties, keep[na:]):
        if kt and _better(t[2], best):
            best = t[2]
    return best[1], int(cnt[keep].sum()), best[2], vol


def _key_to_float(k: int) -> float:
    b = np.uint32(k & 0x7FFFFFFF) if k & 0x80000000 else np.uint32(~k & 0xFFFFFFFF)
    return float(np.array([b], np.uint32).view(F32)[0])


def _topp_keep(y, ids, mass, W, above, p):
    """Top-p over tokens (y, ids) whose strictly larger neighbours outside them weigh
    `above`: keep a token iff the mass of the strictly more probable tokens is below p W
    (tokens of equal y go in or out together)."""
    thr = _ceil_p(W, p)
    o = np.lexsort((ids, -y))
    yo = y[o]
    mo = mass[o].astype(object)
    keep_o = np.zeros(len(o), bool)
    cum = above
    i = 0
    while i < len(o):
        j = i
        g = 0
        while j < len(o) and yo[j] == yo[i]:
            g += mo[j]
            j += 1
        if cum < thr:
            keep_o[i:j] = True
        cum += g
        i = j
    keep = np.zeros(len(o), bool)
    keep[o] = keep_o
    return keep


def split_vocab(V: int, tp: int) -> List[int]:
    """Column starts of `tp` near-equal contiguous shards of V tokens."""
    return [V * i // tp for i in range(tp + 1)]
