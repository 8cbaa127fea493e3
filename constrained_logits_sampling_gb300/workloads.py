"""Seeded synthetic sampler workloads.

This module only draws random inputs: logits, per-row sampling parameters, token
histories, logit_bias entries and grammar bitmasks.  It contains none of the
sampler's arithmetic, so both the CUDA path and the CPU oracle can consume the
same batches without sharing any of the method.

The five workloads mirror the sizes the pages use for the output side of a
serving stack (B=192 rows of a V=151936 vocabulary, "GLM-5.3 inference (7):
output side", section "From the last hidden state to a token id"), with the
parameter mix the pages list for SGLang's SamplingBatchInfo (temperature,
top_k int32, top_p, min_p, repetition / frequency / presence penalties,
logit_bias, grammar bitmask; "SGLang source teardown (10)", section
"SamplingBatchInfo").  No public dataset is involved: every value is drawn
from numpy's PCG64 generator seeded with ``1000 + workload number``.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np

VOCAB = 151936


@dataclasses.dataclass
class Batch:
    """One sampler call's inputs, all host numpy arrays.

    ``logits`` is float32 ``[B, V]`` or, when ``logits_bf16`` is set, uint16
    ``[B, V]`` holding bfloat16 bit patterns.  Optional fields are ``None``
    when the feature is off for the whole batch.
    """

    B: int
    V: int
    logits: np.ndarray
    logits_bf16: bool
    temperatures: Optional[np.ndarray] = None  # f32[B]
    top_ks: Optional[np.ndarray] = None  # i32[B]
    top_ps: Optional[np.ndarray] = None  # f32[B]
    min_ps: Optional[np.ndarray] = None  # f32[B]
    rep: Optional[np.ndarray] = None  # f32[B]
    freq: Optional[np.ndarray] = None  # f32[B]
    pres: Optional[np.ndarray] = None  # f32[B]
    hist_offs: Optional[np.ndarray] = None  # i32[B+1]
    hist_ids: Optional[np.ndarray] = None  # i32[nnz]
    bias_offs: Optional[np.ndarray] = None  # i32[B+1]
    bias_ids: Optional[np.ndarray] = None  # i32[nnz]
    bias_vals: Optional[np.ndarray] = None  # f32[nnz]
    bitmask: Optional[np.ndarray] = None  # i32[B, ceil(V/32)]
    seeds: Optional[np.ndarray] = None  # u64[B]
    positions: Optional[np.ndarray] = None  # i64[B]
    step: int = 0
    name: str = ""
    mode: int = 0  # bit 0: joint top-k/top-p; bit 1: score only (no draw)
    tid_offs: Optional[np.ndarray] = None  # i32[B+1]: requested token ids per row
    tid_ids: Optional[np.ndarray] = None  # i32[nnz]
    top_ns: Optional[np.ndarray] = None  # i32[B]: top-N logprobs wanted per row (0..32)
    top_n_stride: int = 0  # row stride of the top-N outputs (0: the largest N)

    def host_bytes(self) -> Dict[str, int]:
        out = {}
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            if isinstance(v, np.ndarray):
                out[f.name] = int(v.nbytes)
        return out

    def algorithmic_bytes(self) -> int:
        """Bytes a single sampler call must move at minimum: every input array
        read once (logits, bitmask, CSRs, per-row parameters) and the per-row
        outputs (token int32 + logprob float32) written once."""
        total = sum(self.host_bytes().values())
        return int(total + self.B * (4 + 4))

    def rows(self, idx) -> "Batch":
        """Sub-batch with the given row indices (CSR arrays re-based)."""
        idx = np.asarray(idx, dtype=np.int64)
        nb = Batch(B=len(idx), V=self.V, logits=np.ascontiguousarray(self.logits[idx]),
                   logits_bf16=self.logits_bf16, step=self.step, name=self.name + "[sub]", mode=self.mode,
                   top_n_stride=self.top_n_stride)
        for f in ("temperatures", "top_ks", "top_ps", "min_ps", "rep", "freq", "pres",
                  "seeds", "positions", "top_ns"):
            v = getattr(self, f)
            if v is not None:
                setattr(nb, f, np.ascontiguousarray(v[idx]))
        if self.bitmask is not None:
            nb.bitmask = np.ascontiguousarray(self.bitmask[idx])
        for offs_name, arrs in (("hist_offs", ("hist_ids",)),
                                ("bias_offs", ("bias_ids", "bias_vals")),
                                ("tid_offs", ("tid_ids",))):
            offs = getattr(self, offs_name)
            if offs is None:
                continue
            pieces = {a: [] for a in arrs}
            new_offs = [0]
            for r in idx:
                lo, hi = int(offs[r]), int(offs[r + 1])
                for a in arrs:
                    pieces[a].append(getattr(self, a)[lo:hi])
                new_offs.append(new_offs[-1] + hi - lo)
            setattr(nb, offs_name, np.asarray(new_offs, dtype=np.int32))
            for a in arrs:
                dt = getattr(self, a).dtype
                setattr(nb, a, np.concatenate(pieces[a]).astype(dt) if pieces[a] else np.zeros(0, dt))
        return nb


# ----------------------------------------------------------------------------- helpers

def splitmix64(x: int) -> int:
    """One step of the SplitMix64 mixer (Steele, Lea, Flood 2014); used only to
    derive per-row seeds from a workload seed."""
    x = (x + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
    return z ^ (z >> 31)


def row_seeds(base: int, B: int) -> np.ndarray:
    return np.array([splitmix64((base << 32) ^ r) for r in range(B)], dtype=np.uint64)


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def _peaked_normal(rng, B, V, sigma=3.0):
    z = rng.standard_normal((B, V), dtype=np.float32) * np.float32(sigma)
    for r in range(B):
        n = int(rng.integers(1, 21))
        ids = rng.choice(V, size=n, replace=False)
        z[r, ids] += rng.uniform(5.0, 12.0, size=n).astype(np.float32)
    return z


def _param_mix(rng, B, greedy_frac):
    T = rng.uniform(0.5, 1.2, size=B).astype(np.float32)
    greedy = rng.random(B) < greedy_frac
    T[greedy] = 0.0
    k = rng.choice(np.array([-1, 20, 50, 1000], dtype=np.int32), size=B)
    p = rng.choice(np.array([0.8, 0.95, 1.0], dtype=np.float32), size=B)
    mp = rng.choice(np.array([0.0, 0.05], dtype=np.float32), size=B)
    return T, k.astype(np.int32), p.astype(np.float32), mp.astype(np.float32)


def _grammar_row(rng, V):
    """One constrained row: allowed density 0.1%, 5% or 60%, as Bernoulli bits
    or one contiguous id range; at least one token allowed."""
    W = (V + 31) // 32
    density = float(rng.choice([0.001, 0.05, 0.6]))
    allowed = np.zeros(W * 32, dtype=bool)
    if rng.random() < 0.5:
        allowed[:V] = rng.random(V) < density
    else:
        n = max(1, int(round(density * V)))
        off = int(rng.integers(0, V - n + 1))
        allowed[off:off + n] = True
    if not allowed[:V].any():
        allowed[int(rng.integers(0, V))] = True
    bits = np.packbits(allowed.reshape(W, 32), axis=1, bitorder="little")
    return bits.view(np.uint32).reshape(W).view(np.int32)


def _masks(rng, B, V, frac):
    W = (V + 31) // 32
    m = np.full((B, W), -1, dtype=np.int32)
    rows = rng.random(B) < frac
    for r in np.nonzero(rows)[0]:
        m[r] = _grammar_row(rng, V)
    return m


def _zipf_history(rng, B, V, max_len=4096, s=1.1):
    """Per-row histories of U{0..max_len} ids drawn from a Zipf(s) law over
    ranks 1..V, mapped to token ids through a seeded permutation."""
    ranks = np.arange(1, V + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** (-s))
    cdf /= cdf[-1]
    perm = rng.permutation(V).astype(np.int32)
    lens = rng.integers(0, max_len + 1, size=B)
    offs = np.zeros(B + 1, dtype=np.int32)
    offs[1:] = np.cumsum(lens)
    u = rng.random(int(offs[-1]))
    ids = perm[np.minimum(np.searchsorted(cdf, u, side="right"), V - 1)]
    return offs, ids.astype(np.int32)


def _bias(rng, B, V, per_row=16):
    offs = np.arange(0, (B + 1) * per_row, per_row, dtype=np.int32)
    ids = np.concatenate([rng.choice(V, size=per_row, replace=False) for _ in range(B)]).astype(np.int32)
    vals = rng.uniform(-5.0, 5.0, size=B * per_row).astype(np.float32)
    return offs, ids, vals


# ----------------------------------------------------------------------------- workloads

WORKLOADS = {
    1: "tiny: B=4 V=32000 fp32, four fixed rows, no grammar, no penalties",
    2: "decode mix: B=64 V=151936 bf16-valued fp32 logits, 25% greedy, mixed top-k/top-p/min-p",
    3: "grammar-constrained: B=128 V=151936, 50% of rows bitmasked (0.1%/5%/60% density)",
    4: "penalties+bias: B=192 V=151936 fp32, Zipf histories, 16 logit_bias/row, 25% masked",
    5: "verify-scale: B=1024 (256 requests x 4 positions) V=151936 bf16 Student-t logits, all features",
    6: "all-greedy fast path: workload 4 with T=0 on every row (single sweep)",
    7: "all-untruncated fast path: workload 4 with T~U[0.5,1.2], no top-k/top-p/min-p (single sweep)",
}

MODE_FAST_SWEEP = 4  # clsample.h CLSAMPLE_MODE_FAST_SWEEP


def make_workload(n: int, B: Optional[int] = None, V: Optional[int] = None) -> Batch:
    """Build workload ``n`` (1..7).  ``B``/``V`` override the sizes for
    reduced parity cases; the value distributions stay the same.  Workloads 6
    and 7 are workload 4's logits, lists and masks with every row greedy, or
    every row sampled without truncation, marked for the single-sweep path."""
    if n in (6, 7):
        b = make_workload(4, B=B, V=V)
        rng = np.random.Generator(np.random.PCG64(1000 + n))
        if n == 6:
            b.temperatures = np.zeros(b.B, np.float32)
        else:
            b.temperatures = rng.uniform(0.5, 1.2, size=b.B).astype(np.float32)
            b.top_ks = np.full(b.B, -1, np.int32)
            b.top_ps = np.ones(b.B, np.float32)
            b.min_ps = np.zeros(b.B, np.float32)
        b.mode = MODE_FAST_SWEEP
        b.name = "all_greedy" if n == 6 else "all_untruncated"
        return b
    rng = np.random.Generator(np.random.PCG64(1000 + n))
    if n == 1:
        B = B or 4
        V = V or 32000
        z = rng.standard_normal((B, V), dtype=np.float32) * np.float32(3.0)
        for r in range(B):
            ids = rng.choice(V, size=5, replace=False)
            z[r, ids] += np.float32(10.0)
        T = np.ones(B, np.float32)
        k = np.full(B, -1, np.int32)
        p = np.ones(B, np.float32)
        mp = np.zeros(B, np.float32)
        fixed = [(0.0, -1, 1.0, 0.0), (0.7, 20, 1.0, 0.0), (1.0, -1, 0.9, 0.0), (0.8, 50, 0.95, 0.05)]
        for r in range(B):
            T[r], k[r], p[r], mp[r] = fixed[r % 4]
        return Batch(B=B, V=V, logits=z, logits_bf16=False, temperatures=T, top_ks=k, top_ps=p,
                     min_ps=mp, seeds=row_seeds(1001, B), step=7, name="tiny")
    if n in (2, 3):
        B = B or (64 if n == 2 else 128)
        V = V or VOCAB
        z = _peaked_normal(rng, B, V)
        z = bf16_bits_to_f32(round_to_bf16_bits(z)).reshape(B, V)
        T, k, p, mp = _param_mix(rng, B, 0.25)
        bm = _masks(rng, B, V, 0.5) if n == 3 else None
        return Batch(B=B, V=V, logits=z, logits_bf16=False, temperatures=T, top_ks=k, top_ps=p,
                     min_ps=mp, bitmask=bm, seeds=row_seeds(1000 + n, B),
                     positions=rng.integers(0, 1 << 20, size=B).astype(np.int64),
                     name="decode_mix" if n == 2 else "grammar")
    if n == 4:
        B = B or 192
        V = V or VOCAB
        z = _peaked_normal(rng, B, V)
        T, k, p, mp = _param_mix(rng, B, 0.25)
        hoffs, hids = _zipf_history(rng, B, V)
        boffs, bids, bvals = _bias(rng, B, V)
        return Batch(B=B, V=V, logits=z, logits_bf16=False, temperatures=T, top_ks=k, top_ps=p,
                     min_ps=mp,
                     rep=rng.uniform(1.0, 1.3, B).astype(np.float32),
                     freq=rng.uniform(0.0, 0.5, B).astype(np.float32),
                     pres=rng.uniform(0.0, 0.5, B).astype(np.float32),
                     hist_offs=hoffs, hist_ids=hids, bias_offs=boffs, bias_ids=bids, bias_vals=bvals,
                     bitmask=_masks(rng, B, V, 0.25), seeds=row_seeds(1004, B),
                     positions=rng.integers(0, 1 << 20, size=B).astype(np.int64),
                     name="penalties_bias")
    if n == 5:
        B = B or 1024
        V = V or VOCAB
        R = (B + 3) // 4  # requests of 4 draft positions each
        z = (rng.standard_t(3.0, size=(B, V)) * 3.0).astype(np.float32)
        bits = round_to_bf16_bits(z).reshape(B, V)
        Tq, kq, pq, mpq = _param_mix(rng, R, 0.20)
        rep_q = rng.uniform(1.0, 1.3, R).astype(np.float32)
        freq_q = rng.uniform(0.0, 0.5, R).astype(np.float32)
        pres_q = rng.uniform(0.0, 0.5, R).astype(np.float32)
        hoffs_q, hids_q = _zipf_history(rng, R, V)
        boffs_q, bids_q, bvals_q = _bias(rng, R, V)
        req = np.arange(B) // 4
        p0 = rng.integers(0, 1 << 20, size=R).astype(np.int64)
        positions = p0[req] + (np.arange(B) % 4)
        seeds_q = row_seeds(1005, R)
        # expand per-request CSRs to per-row CSRs (each row of a request repeats it)
        def expand(offs, *arrs):
            lens = np.diff(offs)[req]
            new_offs = np.zeros(B + 1, np.int32)
            new_offs[1:] = np.cumsum(lens)
            out = []
            for a in arrs:
                out.append(np.concatenate([a[offs[q]:offs[q + 1]] for q in req]).astype(a.dtype))
            return (new_offs, *out)
        hoffs, hids = expand(hoffs_q, hids_q)
        boffs, bids, bvals = expand(boffs_q, bids_q, bvals_q)
        return Batch(B=B, V=V, logits=bits, logits_bf16=True, temperatures=Tq[req], top_ks=kq[req],
                     top_ps=pq[req], min_ps=mpq[req], rep=rep_q[req], freq=freq_q[req],
                     pres=pres_q[req], hist_offs=hoffs, hist_ids=hids, bias_offs=boffs,
                     bias_ids=bids, bias_vals=bvals, bitmask=_masks(rng, B, V, 0.5),
                     seeds=seeds_q[req], positions=positions, name="verify_scale")
    raise ValueError(f"unknown workload {n}")
