"""Shared helpers of the GPU parity tests: run the CUDA path and the oracle on the same
seeded batch and compare them.

Acceptance bar (element by element):
  * transformed logits z' (penalties, bias, mask): bit-exact;
  * row status, kept-set size and cut (min y over the kept set): exact;
  * greedy and sampled token ids: exact, except rows whose two best race scores lie
    within 1e-5 relative (max(1, |best|)) of each other -- "ambiguous" rows, where fp32
    logs on the two machines may order the pair differently; there the GPU token must
    still be a kept token, and such rows must stay under 0.1% of the batch;
  * logprob of the drawn token: within 1e-5 absolute; so are the drawn token's logprob
    under the original (T = 1, untruncated) distribution and under the kept set, where
    both sides report them; so are the logprobs of requested token ids (with the same
    -inf pattern: masked ids and every id of an INVALID row), and the top-N lists (ids
    exact, logprobs within 1e-5).
"""
import numpy as np
import torch

LOGPROB_TOL = 1e-5
RACE_REL = 1e-5


def run_gpu(batch, debug=True, sampler=None):
    from constrained_logits_sampling_gb300.sampler import Sampler, batch_to_device
    s = sampler or Sampler(max(batch.B, 1), batch.V)
    kw = batch_to_device(batch, s.device)
    logits = kw.pop("logits")
    out = s(logits, debug=debug, **kw)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def run_oracle(batch, want_transformed=True):
    from oracle import oracle as O
    return O.sample(batch, nthreads=0, want_transformed=want_transformed)


def compare(batch, g, o, name="", max_ambiguous_frac=1e-3):
    B = batch.B
    assert np.array_equal(g["status"], o["status"]), (name, np.nonzero(g["status"] != o["status"]))
    if "transformed" in g and "transformed" in o:
        gt = g["transformed"].view(np.uint32)
        ot = o["transformed"].view(np.uint32)
        bad = np.nonzero((gt != ot).any(1))[0]
        assert len(bad) == 0, (name, "transformed differs in rows", bad[:10])
    ok = o["status"] == 0
    assert np.array_equal(g["kept_count"][ok], o["kept_count"][ok]), (
        name, "kept_count", np.nonzero(g["kept_count"] != o["kept_count"])[0][:10])
    assert np.array_equal(g["cut"][ok].view(np.uint32), o["cut"][ok].view(np.uint32)), (
        name, "cut", np.nonzero(g["cut"] != o["cut"])[0][:10])
    gap, best = o["race_gap"], o["race_best"]
    amb = ok & np.isfinite(gap) & np.isfinite(best) & (gap <= RACE_REL * np.maximum(1.0, np.abs(best)))
    same = g["tokens"] == o["tokens"]
    mism = np.nonzero(~same & ~amb)[0]
    assert len(mism) == 0, (name, "token mismatch rows", mism[:10], g["tokens"][mism[:10]], o["tokens"][mism[:10]])
    # ambiguous rows: the GPU's token must still be a kept token
    for r in np.nonzero(amb & ~same)[0]:
        t = int(g["tokens"][r])
        z = o["transformed"][r]
        assert z[t] > -np.inf, (name, r)
    n_amb = int(amb.sum())
    assert n_amb <= max(int(max_ambiguous_frac * B), 0) or n_amb == 0, (name, "ambiguous rows", n_amb)
    inval = ~ok
    assert np.all(g["tokens"][inval] == -1)
    assert np.all(np.isneginf(g["logprobs"][inval]))
    lp_err = np.abs(g["logprobs"][ok].astype(np.float64) - o["logprobs"][ok])
    assert (lp_err <= LOGPROB_TOL).all(), (name, "logprob", float(lp_err.max()), np.argmax(lp_err))
    for key in ("logprobs_orig", "logprobs_kept"):
        if key in g and key in o:
            rows = ok & same
            err = np.abs(g[key][rows].astype(np.float64) - o[key][rows])
            assert (err <= LOGPROB_TOL).all(), (name, key, float(err.max()), np.nonzero(rows)[0][np.argmax(err)])
            assert np.all(np.isneginf(g[key][inval])), (name, key, "invalid rows")
    if "tid_logprobs" in g and "tid_logprobs" in o:
        offs = np.asarray(batch.tid_offs, np.int64)
        owner = np.repeat(np.arange(B), np.diff(offs))
        gv, ov = g["tid_logprobs"].astype(np.float64), o["tid_logprobs"]
        assert np.array_equal(np.isneginf(gv), np.isneginf(ov)), (name, "tid -inf pattern")
        fin = np.isfinite(ov) & ok[owner]
        err = np.abs(gv[fin] - ov[fin])
        assert (err <= LOGPROB_TOL).all(), (name, "tid_logprobs", float(err.max()) if err.size else 0.0)
        assert np.all(np.isneginf(gv[~ok[owner]])), (name, "tid_logprobs of invalid rows")
    if "top_ids" in g and "top_ids" in o:
        N = np.asarray(batch.top_ns)
        for r in range(B):
            n = int(N[r])
            if not (0 <= n <= min(32, o["top_ids"].shape[1])):
                continue
            assert np.array_equal(g["top_ids"][r, :n], o["top_ids"][r, :n]), (name, "top_ids", r)
            gv, ov = g["top_logprobs"][r, :n].astype(np.float64), o["top_logprobs"][r, :n]
            assert np.array_equal(np.isneginf(gv), np.isneginf(ov)), (name, "top -inf pattern", r)
            fin = np.isfinite(ov)
            assert (np.abs(gv[fin] - ov[fin]) <= LOGPROB_TOL).all(), (name, "top_logprobs", r)
    return {"ambiguous": n_amb, "max_logprob_err": float(lp_err.max()) if lp_err.size else 0.0,
            "mismatch_ambiguous": int((amb & ~same).sum())}
