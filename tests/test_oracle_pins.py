"""Pins of the CPU oracle to things other than itself.

Each test ties one part of the oracle to a published known-answer vector, a library
routine, a brute-force enumeration, a closed form or an invariant the pages state.
Page names: "SGLang source teardown (10)" for the sampling/grammar page, "GLM-5.3
output side" for the output-side page, "vLLM logits processors" for the design doc.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from constrained_logits_sampling_gb300.workloads import Batch, make_workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def batch(logits, **kw):
    z = np.ascontiguousarray(np.atleast_2d(np.asarray(logits, dtype=np.float32)))
    B, V = z.shape
    b = Batch(B=B, V=V, logits=z, logits_bf16=False)
    for k, v in kw.items():
        setattr(b, k, v)
    return b


def full(B, v, dt):
    return np.full(B, v, dtype=dt)


def mask_from_allowed(allowed_rows, V):
    W = (V + 31) // 32
    out = np.zeros((len(allowed_rows), W), np.uint32)
    for r, ids in enumerate(allowed_rows):
        for i in ids:
            out[r, i >> 5] |= np.uint32(1) << np.uint32(i & 31)
    return out.view(np.int32)


# ----------------------------------------------------------------------------- random numbers

def test_philox_known_answers(oracle):
    """Philox4x32-10 against the published known-answer vectors (Salmon et al., SC'11)."""
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(x, 16) for x in line.split()])
    assert len(rows) == 3
    for r in rows:
        got = oracle.philox4x32_10(r[0:4], r[4:6])
        assert [int(x) for x in got] == r[6:10]


def test_uniform_layout_and_range(oracle):
    """U = ((x >> 9) + 1/2) / 2^23 with x = word (token % 4) of Philox((token/4, pos, 0), seed)."""
    seed, pos = 0x0123456789ABCDEF, (5 << 32) + 77
    for tok in (0, 1, 2, 3, 4, 151935):
        x = oracle.philox4x32_10([tok >> 2, pos & 0xFFFFFFFF, pos >> 32, 0],
                                 [seed & 0xFFFFFFFF, seed >> 32])[tok & 3]
        assert oracle.uniform(seed, pos, tok) == ((int(x) >> 9) + 0.5) / 2 ** 23


def test_uniform_statistics(oracle):
    """Kolmogorov-Smirnov against U(0,1) over 200k draws of one request's stream,
    and independence of neighbouring positions (correlation near 0)."""
    from scipy import stats
    u = np.array([oracle.uniform(42, 1000 + (i // 2000), i % 2000) for i in range(200000)])
    assert u.min() > 0 and u.max() < 1
    assert stats.kstest(u, "uniform").pvalue > 1e-4
    a = np.array([oracle.uniform(7, p, 3) for p in range(20000)])
    b = np.array([oracle.uniform(7, p + 1, 3) for p in range(20000)])
    assert abs(np.corrcoef(a, b)[0, 1]) < 0.03


# ----------------------------------------------------------------------------- top-p arithmetic

def test_exp32_against_library_exp(oracle):
    """exp32 stays within 2 ulp of the correctly rounded exponential (numpy, float64)."""
    ys = np.concatenate([np.linspace(-32, 0, 40001, dtype=np.float32),
                         -np.logspace(-8, 1.5, 5001).astype(np.float32)])
    worst = 0
    for y in ys:
        got = oracle.exp32(float(y))
        ref = math.exp(float(y))
        ulp = np.spacing(np.float32(ref))
        worst = max(worst, abs(got - ref) / float(ulp))
    assert worst <= 2.0, worst
    assert oracle.exp32(0.0) == 1.0
    assert oracle.exp32(-33.0) == 0.0 and oracle.exp32(float("-inf")) == 0.0


def test_weight_fixed_point(oracle):
    assert oracle.weight_fx(0.0) == 2 ** 40
    y = -3.25
    assert oracle.weight_fx(y) == math.floor(Fraction(oracle.exp32(y)) * 2 ** 40)


def test_ceil_scaled_exact(oracle):
    """ceil(p * W) against exact rational arithmetic (fractions.Fraction)."""
    rng = np.random.default_rng(0)
    for _ in range(3000):
        W = int(rng.integers(1, 2 ** 58))
        p = F32(rng.random())
        if p <= 0:
            continue
        assert oracle.ceil_scaled(W, p) == math.ceil(Fraction(float(p)) * W)
    for p in (1.0, 0.5, 0.8, 0.95, 1e-30, 1e-45):
        for W in (1, 2 ** 40, 3 * 2 ** 40 + 17):
            assert oracle.ceil_scaled(W, p) == math.ceil(Fraction(float(F32(p))) * W)


# ----------------------------------------------------------------------------- transforms

def test_penalty_bias_mask_golden(oracle):
    """Hand-computed rows (golden/penalty_rows.json): penalties, bias dedup, mask."""
    with open(os.path.join(GOLDEN, "penalty_rows.json")) as f:
        g = json.load(f)
    V = g["V"]
    for row in g["rows"]:
        b = batch([g["logits"]], temperatures=full(1, 0.0, F32),
                  rep=full(1, row["rep"], F32), freq=full(1, row["freq"], F32),
                  pres=full(1, row["pres"], F32),
                  hist_offs=np.array([0, len(row["history"])], np.int32),
                  hist_ids=np.array(row["history"], np.int32),
                  bias_offs=np.array([0, len(row["bias"])], np.int32),
                  bias_ids=np.array([x[0] for x in row["bias"]], np.int32),
                  bias_vals=np.array([x[1] for x in row["bias"]], np.float32),
                  bitmask=mask_from_allowed([row["allowed"]], V))
        o = oracle.sample(b, want_transformed=True)
        exp = np.array([float(x) for x in row["expected_transformed"]], np.float32)
        assert np.array_equal(o["transformed"][0], exp), (row["name"], o["transformed"][0])
        assert o["tokens"][0] == row["expected_greedy"], row["name"]


def test_sanitize_non_finite(oracle):
    z = np.array([[1.0, np.nan, 0.5, np.inf, -np.inf, 2.0]], np.float32)
    o = oracle.sample(batch(z, temperatures=full(1, 0.0, F32)), want_transformed=True)
    t = o["transformed"][0]
    assert t[1] == -np.inf and t[3] == np.finfo(np.float32).max and t[4] == -np.finfo(np.float32).max
    assert o["tokens"][0] == 3
    # NaN is never drawn, even when every other logit is tiny
    z = np.array([[np.nan, -50.0, np.nan, -60.0]], np.float32)
    b = batch(np.repeat(z, 500, 0), positions=np.arange(500, dtype=np.int64),
              seeds=np.arange(500, dtype=np.uint64))
    o = oracle.sample(b)
    assert set(o["tokens"].tolist()) <= {1, 3}


def test_mask_commutes_with_penalties_and_bias(oracle):
    """-inf + c = -inf and -inf * r = -inf: masking last equals masking the
    unmasked result (SGLang teardown (10), 'Order semantics of the penalties')."""
    b = make_workload(4, B=6, V=3000)
    o_mask = oracle.sample(b, want_transformed=True)
    b.bitmask = None
    o_plain = oracle.sample(b, want_transformed=True)
    bm = make_workload(4, B=6, V=3000).bitmask
    bits = np.unpackbits(bm.view(np.uint8), axis=1, bitorder="little")[:, :3000].astype(bool)
    expect = np.where(bits, o_plain["transformed"], -np.inf).astype(np.float32)
    assert np.array_equal(o_mask["transformed"], expect)


def test_bias_duplicates_last_wins(oracle):
    z = np.random.default_rng(1).standard_normal((1, 64)).astype(np.float32)
    common = dict(temperatures=full(1, 0.0, F32))
    dup = oracle.sample(batch(z, bias_offs=np.array([0, 3], np.int32),
                              bias_ids=np.array([5, 9, 5], np.int32),
                              bias_vals=np.array([10.0, 1.0, -3.0], np.float32), **common),
                        want_transformed=True)
    one = oracle.sample(batch(z, bias_offs=np.array([0, 2], np.int32),
                              bias_ids=np.array([9, 5], np.int32),
                              bias_vals=np.array([1.0, -3.0], np.float32), **common),
                        want_transformed=True)
    assert np.array_equal(dup["transformed"], one["transformed"])


def test_all_ones_mask_equals_no_mask(oracle):
    """An unfilled bitmask row (every word -1) is unconstrained (SGLang teardown (10),
    'Bitmask: one int32 covers 32 tokens')."""
    b = make_workload(2, B=12, V=4000)
    o1 = oracle.sample(b, want_transformed=True)
    b.bitmask = np.full((12, 125), -1, np.int32)
    o2 = oracle.sample(b, want_transformed=True)
    for k in ("tokens", "logprobs", "kept_count", "cut", "transformed"):
        assert np.array_equal(o1[k], o2[k]), k


# ----------------------------------------------------------------------------- greedy

def test_greedy_is_argmax_lowest_id(oracle):
    rng = np.random.default_rng(2)
    z = rng.integers(-4, 4, size=(64, 50)).astype(np.float32)  # many exact ties
    o = oracle.sample(batch(z, temperatures=full(64, 0.0, F32)))
    assert np.array_equal(o["tokens"], np.argmax(z, axis=1))  # np.argmax: first maximum


def test_greedy_rules(oracle):
    """temperature < 1e-5 (GLM-5.3 output side) or top_k <= 1 (SGLang teardown (10))
    is greedy; top_k = -1 means the whole vocabulary and is not greedy."""
    rng = np.random.default_rng(3)
    z = rng.standard_normal((1, 300)).astype(np.float32) * 3
    arg = int(np.argmax(z))
    for T in (0.0, 1e-6, -1.0, 9.99e-6):
        o = oracle.sample(batch(z, temperatures=full(1, T, F32)))
        assert o["tokens"][0] == arg and o["kept_count"][0] == 1
    for k in (0, 1):
        for T in (0.3, 1.0, 5.0):
            o = oracle.sample(batch(z, temperatures=full(1, T, F32), top_ks=full(1, k, np.int32)))
            assert o["tokens"][0] == arg
    z2 = np.zeros((400, 300), np.float32)  # uniform row: -1 must sample broadly
    o = oracle.sample(batch(z2, top_ks=full(400, -1, np.int32), positions=np.arange(400, dtype=np.int64)))
    assert len(set(o["tokens"].tolist())) > 100


# ----------------------------------------------------------------------------- truncation

def test_no_truncation_keeps_every_allowed_token(oracle):
    b = make_workload(3, B=16, V=5000)
    b.top_ks[:] = -1
    b.top_ps[:] = 1.0
    b.min_ps[:] = 0.0
    b.temperatures[:] = 0.9
    o = oracle.sample(b)
    bits = np.unpackbits(b.bitmask.view(np.uint8), axis=1, bitorder="little")[:, :5000]
    assert np.array_equal(o["kept_count"], bits.sum(1))


def test_topk_counts_strictly_larger(oracle):
    """S_k = {i : rank(p_i) < k}, rank = number of strictly larger probabilities
    (SGLang teardown (10), 'The maths of the three cuts'); ties at the k-th value stay."""
    rng = np.random.default_rng(4)
    z = rng.integers(-6, 6, size=(40, 200)).astype(np.float32)
    ks = rng.integers(2, 60, size=40).astype(np.int32)
    o = oracle.sample(batch(z, top_ks=ks, temperatures=full(40, 1.0, F32)))
    for r in range(40):
        larger = (z[r][None, :] > z[r][:, None]).sum(1)
        assert o["kept_count"][r] == int((larger < ks[r]).sum())


def test_min_p_is_argmax_invariant(oracle):
    """Min-p never removes the most probable token (vLLM logits processors,
    argmax invariance); with min_p = 1 only the tokens tied with the maximum stay."""
    b = make_workload(2, B=32, V=6000)
    b.temperatures[:] = 0.0
    g0 = oracle.sample(b)["tokens"]
    for mp in (0.0, 0.05, 0.9):
        b.min_ps[:] = mp
        assert np.array_equal(oracle.sample(b)["tokens"], g0)
    b.temperatures[:] = 0.8
    b.top_ks[:] = -1
    b.top_ps[:] = 1.0
    b.min_ps[:] = 1.0
    o = oracle.sample(b)
    assert np.array_equal(o["tokens"], g0)
    zz = b.logits
    assert np.array_equal(o["kept_count"], (zz == zz.max(1, keepdims=True)).sum(1))


def test_top_p_ties_all_in_or_all_out(oracle):
    # Probabilities: 0.4025 (token 0), 4 x 0.1481 (tokens 1-4), 2 x 0.0027.  With
    # p = 0.5 a "smallest prefix" would stop after one of the tied tokens (0.55 >= 0.5),
    # but the definition keeps all four; at p = 0.999 the mass above the last pair is
    # 0.9946 < p, so it stays too.
    z = np.array([[2.0, 1.0, 1.0, 1.0, 1.0, -3.0, -3.0]], np.float32)
    for p, kept in ((0.2, 1), (0.3, 1), (0.5, 5), (0.99, 5), (0.999, 7), (1.0, 7)):
        o = oracle.sample(batch(z, top_ps=full(1, p, F32), temperatures=full(1, 1.0, F32)))
        assert o["kept_count"][0] == kept, (p, o["kept_count"][0])


def _brute_force_kept(y, allowed, k, p, mp):
    """Kept set at tiny V by enumeration: top-k by strictly-larger counts, top-p as
    the smallest subset closed under 'at least as probable' whose renormalised mass
    reaches p, min-p as p_i >= p_max * min_p.  Returns (kept mask, margin) where the
    margin is the distance of every threshold decision from its boundary."""
    V = len(y)
    cand = [i for i in range(V) if allowed[i]]
    w = {i: math.exp(y[i]) for i in cand}
    Sk = [i for i in cand if k < 2 or sum(y[j] > y[i] for j in cand) < k]
    Wk = sum(w[i] for i in Sk)
    margin = float("inf")
    if p < 1:
        best = None
        for n in range(1, len(Sk) + 1):
            for sub in itertools.combinations(Sk, n):
                s = set(sub)
                if any(y[j] >= y[i] and j not in s for i in s for j in Sk):
                    continue  # not closed upwards (ties included)
                mass = sum(w[i] for i in s) / Wk
                margin = min(margin, abs(mass - p))
                if mass >= p and (best is None or len(s) < len(best)):
                    best = s
        Sp = best
    else:
        Sp = set(Sk)
    kept = np.zeros(V, bool)
    for i in Sp:
        if mp == 0 or w[i] >= mp * max(w.values()):
            kept[i] = True
        if mp > 0:
            margin = min(margin, abs(w[i] / max(w.values()) - mp))
    return kept, margin


def test_sampling_law_brute_force_and_chi_square(oracle):
    """At V=8: the kept set equals the brute-force enumeration, and 1e5 draws over
    consecutive positions follow P(i) = w_i / sum_K w (chi-square)."""
    from scipy import stats
    rng = np.random.default_rng(5)
    n_draws = 100000
    cases = 0
    for trial in range(40):
        V = 8
        z = (rng.integers(-24, 24, size=V) / 8.0).astype(np.float32)  # dyadic: exact fp32 maths
        T = float(rng.choice([0.5, 1.0, 2.0]))
        k = int(rng.choice([-1, 2, 3, 5]))
        p = float(rng.choice([0.5, 0.8, 1.0]))
        mp = float(rng.choice([0.0, 0.1]))
        allowed = rng.random(V) < 0.8
        allowed[int(rng.integers(V))] = True
        zm = np.where(allowed, z, -np.inf)
        m = zm.max()
        y = [(float(zm[i]) - float(m)) / T if allowed[i] else -math.inf for i in range(V)]
        kept, margin = _brute_force_kept(y, allowed, k, p, mp)
        if margin < 1e-5:
            continue
        cases += 1
        b = batch(np.repeat(z[None], n_draws, 0), temperatures=full(n_draws, T, F32),
                  top_ks=full(n_draws, k, np.int32), top_ps=full(n_draws, p, F32),
                  min_ps=full(n_draws, mp, F32), bitmask=np.repeat(mask_from_allowed(
                      [np.nonzero(allowed)[0]], V), n_draws, 0),
                  seeds=full(n_draws, 1234 + trial, np.uint64),
                  positions=np.arange(n_draws, dtype=np.int64))
        o = oracle.sample(b)
        assert np.all(o["kept_count"] == kept.sum())
        counts = np.bincount(o["tokens"], minlength=V)
        assert counts[~kept].sum() == 0
        idx = np.nonzero(kept)[0]
        if len(idx) < 2:
            continue
        w = np.array([math.exp(y[i]) for i in idx])
        expected = w / w.sum() * n_draws
        assert stats.chisquare(counts[idx], expected).pvalue > 1e-4, (trial, counts[idx], expected)
    assert cases >= 20


# ----------------------------------------------------------------------------- logprob

def test_logprob_matches_library_log_softmax(oracle):
    """Logprob of the drawn token = log_softmax of the transformed logits at the row's
    temperature (SGLang teardown (10), 'Numerical consistency of logprobs'), checked
    against torch.log_softmax in float64 on the CPU."""
    import torch
    b = make_workload(4, B=24, V=20000)
    for r in range(24):
        b.temperatures[r] = (0.0, 1.0, 0.5)[r % 3]
    o = oracle.sample(b, want_transformed=True)
    for r in range(24):
        T = float(b.temperatures[r])
        Teff = T if T >= 1e-5 else 1.0
        z = torch.tensor(o["transformed"][r], dtype=torch.float64)
        ref = torch.log_softmax(z / Teff, dim=0)[int(o["tokens"][r])].item()
        assert abs(ref - o["logprobs"][r]) < 1e-5


def test_original_logprob_is_log_softmax_at_t1(oracle):
    """The original logprob (before temperature; SGLang teardown (10), 'Numerical
    consistency of logprobs') is log_softmax of the transformed logits at T = 1, checked
    against torch.log_softmax in float64; greedy rows with T < 1e-5 have it equal to the
    ordinary logprob."""
    import torch
    b = make_workload(4, B=24, V=20000)
    for r in range(24):
        b.temperatures[r] = (0.0, 1.3, 0.5)[r % 3]
    o = oracle.sample(b, want_transformed=True)
    for r in range(24):
        z = torch.tensor(o["transformed"][r], dtype=torch.float64)
        ref = torch.log_softmax(z, dim=0)[int(o["tokens"][r])].item()
        assert abs(ref - o["logprobs_orig"][r]) < 1e-5
        if b.temperatures[r] == 0.0:
            assert o["logprobs_orig"][r] == o["logprobs"][r]


def test_kept_logprob_brute_force(oracle):
    """The kept-set logprob (the distribution the token is drawn from; GLM page,
    'Sampling': processed logprobs) at V=8 equals log(w_tok / sum over the enumerated
    kept set of w); greedy rows give 0 (the kept set is the token alone)."""
    rng = np.random.default_rng(6)
    checked = 0
    for trial in range(60):
        V = 8
        z = (rng.integers(-24, 24, size=V) / 8.0).astype(np.float32)
        T = float(rng.choice([0.0, 0.5, 1.0, 2.0]))
        k = int(rng.choice([-1, 1, 2, 3, 5]))
        p = float(rng.choice([0.5, 0.8, 1.0]))
        mp = float(rng.choice([0.0, 0.1]))
        allowed = rng.random(V) < 0.8
        allowed[int(rng.integers(V))] = True
        b = batch(z[None].copy(), temperatures=full(1, T, F32), top_ks=full(1, k, np.int32),
                  top_ps=full(1, p, F32), min_ps=full(1, mp, F32),
                  bitmask=mask_from_allowed([np.nonzero(allowed)[0]], V), seeds=full(1, 77 + trial, np.uint64),
                  positions=np.arange(1, dtype=np.int64))
        o = oracle.sample(b)
        tok = int(o["tokens"][0])
        if T < 1e-5 or k in (0, 1):
            assert o["logprobs_kept"][0] == 0.0
            continue
        zm = np.where(allowed, z, -np.inf)
        m = float(zm.max())
        y = [(float(zm[i]) - m) / T if allowed[i] else -math.inf for i in range(V)]
        kept, margin = _brute_force_kept(y, allowed, k, p, mp)
        if margin < 1e-5:
            continue
        assert kept[tok]
        ref = y[tok] - math.log(sum(math.exp(y[i]) for i in range(V) if kept[i]))
        assert abs(ref - o["logprobs_kept"][0]) < 1e-6
        checked += 1
    assert checked >= 20


# ----------------------------------------------------------------------------- batching

def test_batch_composition_independence(oracle):
    """A row's draw depends only on its own data, seed and position (SGLang teardown
    (10): the position drives the seed so the stream does not depend on the batch)."""
    b = make_workload(4, B=20, V=3000)
    o = oracle.sample(b)
    perm = np.random.default_rng(6).permutation(20)
    o2 = oracle.sample(b.rows(perm))
    assert np.array_equal(o2["tokens"], o["tokens"][perm])
    assert np.array_equal(o2["logprobs"], o["logprobs"][perm])
    o3 = oracle.sample(b.rows([7]))
    assert o3["tokens"][0] == o["tokens"][7]


def test_invalid_rows(oracle):
    z = np.zeros((7, 40), np.float32)
    b = batch(z, temperatures=np.array([np.nan, 1, 1, 1, 1, 1, 1], F32),
              top_ks=np.array([-1, -2, -1, -1, -1, -1, -1], np.int32),
              top_ps=np.array([1, 1, 0.0, 1, 1, 1, 1], F32),
              min_ps=np.array([0, 0, 0, 1.5, 0, 0, 0], F32),
              hist_offs=np.array([0, 0, 0, 0, 0, 1, 1, 1], np.int32), hist_ids=np.array([40], np.int32),
              rep=np.array([1, 1, 1, 1, 1, 0.0, 1], F32),
              bitmask=np.array([[-1, -1]] * 6 + [[0, 0]], np.int32))
    o = oracle.sample(b)
    assert np.all(o["status"][:7] == 2) and np.all(o["tokens"] == -1)
    assert np.all(np.isneginf(o["logprobs"]))


# ----------------------------------------------------------------------------- joint top-k/top-p

def _joint_brute_force(y, allowed, k, p):
    """Joint order at tiny V by enumeration: the top-k set (strictly-larger counts)
    intersected with the smallest subset of ALL candidates, closed under 'at least as
    probable', whose mass reaches p of the whole candidate mass.  Returns (kept, margin)."""
    V = len(y)
    cand = [i for i in range(V) if allowed[i]]
    w = {i: math.exp(y[i]) for i in cand}
    W = sum(w.values())
    Sk = {i for i in cand if k < 2 or sum(y[j] > y[i] for j in cand) < k}
    margin = float("inf")
    best = set(cand)
    for n in range(1, len(cand) + 1):
        for sub in itertools.combinations(cand, n):
            s = set(sub)
            if any(y[j] >= y[i] and j not in s for i in s for j in cand):
                continue
            mass = sum(w[i] for i in s) / W
            margin = min(margin, abs(mass - p))
            if mass >= p and len(s) < len(best):
                best = s
    kept = np.zeros(V, bool)
    for i in best & Sk:
        kept[i] = True
    return kept, margin


def test_joint_worked_example(oracle):
    """Probabilities 0.4, 0.3, 0.2, 0.1 at T = 1.  Sequential (SGLang teardown (10), the
    top-k -> top-p order): top-p runs over the renormalised top-k set; joint
    (filter_apply_order 'joint'): top-p runs over the whole distribution and the result
    is intersected with top-k.  Hand-derived: k=2, p=0.5 keeps 1 token sequentially
    (0.4/0.7 >= 0.5) but 2 jointly (0.4 < 0.5); k=3, p=0.75 keeps 2 sequentially
    (0.7/0.9 >= 0.75) but 3 jointly (0.7 < 0.75)."""
    z = np.log(np.array([0.4, 0.3, 0.2, 0.1])).astype(np.float32)
    for k, p, seq, joint in ((2, 0.5, 1, 2), (3, 0.75, 2, 3), (-1, 0.75, 3, 3), (2, 1.0, 2, 2)):
        for mode, want in ((0, seq), (1, joint)):
            b = batch(z[None].copy(), top_ks=full(1, k, np.int32), top_ps=full(1, p, F32), mode=mode,
                      seeds=full(1, 5, np.uint64))
            o = oracle.sample(b)
            assert int(o["kept_count"][0]) == want, (k, p, mode)


def test_joint_brute_force_and_nesting(oracle):
    """Joint kept sets at V=8 match the enumeration above; on a larger workload the
    sequential kept set is inside the joint one, which is inside the top-k set, and the
    joint order equals the sequential one without a top-k cut."""
    rng = np.random.default_rng(12)
    checked = 0
    for trial in range(60):
        V = 8
        z = (rng.integers(-24, 24, size=V) / 8.0).astype(np.float32)
        T = float(rng.choice([0.5, 1.0, 2.0]))
        k = int(rng.choice([-1, 2, 3, 5]))
        p = float(rng.choice([0.3, 0.5, 0.8]))
        allowed = rng.random(V) < 0.8
        allowed[int(rng.integers(V))] = True
        b = batch(z[None].copy(), temperatures=full(1, T, F32), top_ks=full(1, k, np.int32),
                  top_ps=full(1, p, F32), bitmask=mask_from_allowed([np.nonzero(allowed)[0]], V),
                  seeds=full(1, 9 + trial, np.uint64), mode=1)
        o = oracle.sample(b)
        zm = np.where(allowed, z, -np.inf)
        m = float(zm.max())
        y = [(float(zm[i]) - m) / T if allowed[i] else -math.inf for i in range(V)]
        kept, margin = _joint_brute_force(y, allowed, k, p)
        if margin < 1e-5:
            continue
        assert int(o["kept_count"][0]) == int(kept.sum()), trial
        assert kept[int(o["tokens"][0])]
        checked += 1
    assert checked >= 30
    w = make_workload(2, B=48, V=6000)
    w.min_ps = np.zeros(48, np.float32)
    seq = oracle.sample(w)
    w.mode = 1
    jnt = oracle.sample(w)
    w.top_ps = np.ones(48, np.float32)
    topk = oracle.sample(w)
    ok = seq["status"] == 0
    assert (seq["kept_count"][ok] <= jnt["kept_count"][ok]).all()
    assert (jnt["kept_count"][ok] <= topk["kept_count"][ok]).all()
    assert (seq["kept_count"] < jnt["kept_count"]).any()
    nok = ok & ((w.top_ks <= 0) | (w.top_ks >= 6000))
    assert np.array_equal(seq["kept_count"][nok], jnt["kept_count"][nok])
    assert np.array_equal(seq["tokens"][nok], jnt["tokens"][nok])


# ----------------------------------------------------------------------------- requested ids, scoring

def _with_requests(b, per_row, rng):
    offs, ids = [0], []
    for r in range(b.B):
        n = int(rng.integers(0, per_row + 1))
        ids.extend(int(x) for x in rng.integers(0, b.V, size=n))
        offs.append(len(ids))
    b.tid_offs = np.asarray(offs, np.int32)
    b.tid_ids = np.asarray(ids, np.int32)
    return b


def test_requested_id_logprobs_match_library_log_softmax(oracle):
    """Logprobs of requested token ids (SGLang teardown (10), the output container's
    token-ids logprobs) are log_softmax of z'/T at those ids, checked against
    torch.log_softmax in float64; masked ids give -inf; a requested id equal to the drawn
    token gives the drawn token's logprob."""
    import torch
    rng = np.random.default_rng(21)
    b = _with_requests(make_workload(3, B=24, V=9000), 6, rng)
    # every row also asks for its drawn token
    o0 = oracle.sample(b)
    offs, ids = [0], []
    for r in range(b.B):
        ids.extend(b.tid_ids[b.tid_offs[r]:b.tid_offs[r + 1]].tolist() + [int(o0["tokens"][r])])
        offs.append(len(ids))
    b.tid_offs, b.tid_ids = np.asarray(offs, np.int32), np.asarray(ids, np.int32)
    o = oracle.sample(b, want_transformed=True)
    assert np.array_equal(o["tokens"], o0["tokens"])
    n_masked = 0
    for r in range(b.B):
        T = float(b.temperatures[r])
        Teff = T if T >= 1e-5 else 1.0
        z = torch.tensor(o["transformed"][r], dtype=torch.float64)
        ref = torch.log_softmax(z / Teff, dim=0)
        for j in range(b.tid_offs[r], b.tid_offs[r + 1]):
            i = int(b.tid_ids[j])
            if math.isinf(ref[i].item()):
                assert o["tid_logprobs"][j] == -math.inf
                n_masked += 1
            else:
                assert abs(ref[i].item() - o["tid_logprobs"][j]) < 1e-5
        assert o["tid_logprobs"][b.tid_offs[r + 1] - 1] == o["logprobs"][r]
    assert n_masked > 0


def test_requested_id_out_of_range_invalidates_row(oracle):
    """A requested id outside the vocabulary makes its row INVALID (like a bad history or
    bias id); the other rows are untouched."""
    b = make_workload(1, B=4, V=500)
    b.tid_offs = np.array([0, 1, 3, 3, 4], np.int32)
    b.tid_ids = np.array([3, 7, 500, 499], np.int32)
    o = oracle.sample(b)
    ref = oracle.sample(make_workload(1, B=4, V=500))
    assert list(o["status"]) == [0, 2, 0, 0]
    assert o["tokens"][1] == -1 and np.isneginf(o["tid_logprobs"][1:3]).all()
    assert np.array_equal(o["tokens"][[0, 2, 3]], ref["tokens"][[0, 2, 3]])


def test_score_only_mode(oracle):
    """Score-only mode (SGLang teardown (10), logprobs-only scoring: same preprocessing, no
    sampling): every row takes the greedy route whatever its parameters, so the seeds
    change nothing, the token is the lowest-id argmax of z', and the requested ids get the
    same logprobs as in sampling mode."""
    rng = np.random.default_rng(4)
    b = _with_requests(make_workload(4, B=16, V=7000), 5, rng)
    samp = oracle.sample(b)
    b.mode = 2
    o = oracle.sample(b, want_transformed=True)
    b.seeds = b.seeds[::-1].copy()
    o2 = oracle.sample(b)
    assert np.array_equal(o["tokens"], o2["tokens"])
    ok = o["status"] == 0
    assert np.array_equal(o["tokens"][ok], np.argmax(o["transformed"][ok], axis=1))
    assert (o["kept_count"][ok] == 1).all()
    assert np.array_equal(o["tid_logprobs"], samp["tid_logprobs"])


# ----------------------------------------------------------------------------- allowed ids, min tokens

def test_allowed_ids_bitmask_worked_example(oracle):
    """Allowed-id lists as bitmask words, hand-computed from the bit layout (bit i & 31 of
    word i >> 5): {0, 31, 32, 63, 64} over V = 70 -> 0x80000001, 0x80000001, 0x1; bad or
    empty rows are all zero, and such a row samples INVALID."""
    m = oracle.allowed_to_bitmask([0, 5, 5, 7, 8], [0, 31, 32, 63, 64, 3, 70, 69], 70).view(np.uint32)
    assert m.shape == (4, 3)
    assert [hex(int(x)) for x in m[0]] == ["0x80000001", "0x80000001", "0x1"]
    assert (m[1] == 0).all() and (m[2] == 0).all()
    assert [hex(int(x)) for x in m[3]] == ["0x0", "0x0", "0x20"]
    b = batch(np.zeros((4, 70), F32), bitmask=m.view(np.int32))
    o = oracle.sample(b)
    assert list(o["status"]) == [0, 2, 2, 0]
    assert int(o["tokens"][3]) == 69


def test_min_new_tokens_as_minus_inf_bias(oracle):
    """Min-new-tokens (SGLang teardown (10); vLLM logits processors, 'Min-tokens') read as
    a -inf logit_bias on the EOS ids: those ids are never drawn, even as the argmax, and
    the rest of the row is unchanged."""
    b = make_workload(2, B=16, V=5000)
    o = oracle.sample(b, want_transformed=True)
    eos = [int(t) for t in o["tokens"][:4]] + [int(np.argmax(o["transformed"][0]))]
    b.bias_offs = np.arange(0, 16 * len(eos) + 1, len(eos), dtype=np.int32)
    b.bias_ids = np.tile(np.asarray(eos, np.int32), 16)
    b.bias_vals = np.full(16 * len(eos), -np.inf, np.float32)
    o2 = oracle.sample(b, want_transformed=True)
    assert (o2["status"] == 0).all()
    assert not np.isin(o2["tokens"], eos).any()
    assert np.isneginf(o2["transformed"][:, eos]).all()
    keep = np.setdiff1d(np.arange(5000), eos)
    assert np.array_equal(o2["transformed"][:, keep], o["transformed"][:, keep])


# ----------------------------------------------------------------------------- top-N logprobs

def test_top_n_against_library_topk(oracle):
    """Top-N logprobs (SGLang teardown (10), the output container's top logprobs): the
    reported values are the N largest of torch.log_softmax(z'/T) in float64 (the values
    torch.topk returns), each reported id carries its own log_softmax value, and the
    order is by descending probability."""
    import torch
    b = make_workload(4, B=20, V=9000)
    b.top_ns = np.array([(0, 1, 5, 20, 32)[r % 5] for r in range(20)], np.int32)
    o = oracle.sample(b, want_transformed=True)
    assert o["top_ids"].shape == (20, 32)
    for r in range(20):
        n = int(b.top_ns[r])
        T = float(b.temperatures[r])
        Teff = T if T >= 1e-5 else 1.0
        ref = torch.log_softmax(torch.tensor(o["transformed"][r], dtype=torch.float64) / Teff, dim=0)
        vals = torch.topk(ref, n).values.numpy() if n else np.zeros(0)
        got = o["top_logprobs"][r, :n]
        assert np.allclose(got, vals, atol=1e-6, rtol=0)
        ids = o["top_ids"][r, :n]
        have = ids >= 0
        assert np.array_equal(have, np.isfinite(vals))  # -1 exactly past the candidates
        assert np.allclose(ref.numpy()[ids[have]], got[have], atol=1e-6, rtol=0)
        assert (np.diff(got[have]) <= 0).all()
        assert (o["top_ids"][r, n:] == -7).all()  # past N: untouched


def test_top_n_ties_and_short_rows(oracle):
    """Equal z' are reported lowest id first; a row with fewer candidates than N ends in
    -1 / -inf; N above 32 or above the stride makes the row INVALID."""
    V = 40
    z = np.zeros((4, V), F32)
    z[0, 17] = 1.0
    allowed = [np.arange(V), np.arange(V), np.array([3, 9]), np.arange(V)]
    b = batch(z, bitmask=mask_from_allowed(allowed, V), top_ns=np.array([4, 33, 4, 4], np.int32))
    b.top_n_stride = 4
    o = oracle.sample(b)
    assert list(o["top_ids"][0]) == [17, 0, 1, 2]
    assert list(o["status"]) == [0, 2, 0, 0]
    assert list(o["top_ids"][2]) == [3, 9, -1, -1] and np.isneginf(o["top_logprobs"][2, 2:]).all()
    assert abs(o["top_logprobs"][2, 0] - math.log(0.5)) < 1e-12
    assert list(o["top_ids"][3]) == [0, 1, 2, 3]
    assert abs(o["top_logprobs"][3, 0] - math.log(1 / 40)) < 1e-12
