"""Vocabulary-sharded sampling (the GLM page's "sample then gather" over tensor-parallel
shards), simulated on the CPU: the protocol's result does not depend on how the
vocabulary is split, it agrees with the oracle row by row (outside knife edges of the
top-p cut), it runs across two gloo ranks, and it exchanges per-row statistics, not
logits."""
import math
import os
import socket
import sys
import tempfile

import numpy as np
import pytest

from constrained_logits_sampling_gb300.vocab_shard import (LocalComm, RowParams, Shard, philox4x32_10,
                                                           sample_sharded, split_vocab)
from constrained_logits_sampling_gb300.workloads import make_workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def params_of(b):
    return [RowParams(float(b.temperatures[r]), int(b.top_ks[r]), float(b.top_ps[r]), float(b.min_ps[r]),
                      int(b.seeds[r]), int(b.positions[r]) if b.positions is not None else int(b.step))
            for r in range(b.B)]


def run(z, ps, tp, band_cap=4096):
    e = split_vocab(z.shape[1], tp)
    return sample_sharded(ps, LocalComm([Shard(z[:, e[i]:e[i + 1]], e[i], ps) for i in range(tp)]),
                          band_cap=band_cap)


def transformed(b, oracle):
    return oracle.sample(b, nthreads=0, want_transformed=True)


def test_philox_known_answers():
    """The simulation's own Philox4x32-10 against the published known-answer vectors."""
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        rows = [[int(x, 16) for x in line.split()] for line in f if line.strip() and not line.startswith("#")]
    for r in rows:
        got = philox4x32_10(np.array([r[0:4]], np.uint32), r[4:6])[0]
        assert [int(x) for x in got] == r[6:10]


@pytest.fixture(scope="module")
def mixed(oracle):
    """Workload 2's row mix (greedy, top-k 20/50/1000, top-p 0.8/0.95, min-p) plus flat
    rows (one tie group) under top-p and top-k, at V = 20011."""
    b = make_workload(2, B=32, V=20011)
    b.logits[-3:] = 0.25
    b.temperatures[-3:] = 1.0
    b.top_ks[-3:] = np.array([-1, 7, -1], np.int32)
    b.top_ps[-3:] = np.array([0.5, 1.0, 1.0], F32)
    b.min_ps[-3:] = 0.0
    o = transformed(b, oracle)
    return b, o


@pytest.mark.parametrize("tp", [2, 3, 4, 7])
def test_result_does_not_depend_on_the_split(mixed, tp):
    b, o = mixed
    ps = params_of(b)
    one = run(o["transformed"], ps, 1)
    many = run(o["transformed"], ps, tp, band_cap=64)  # small bands: refinement rounds run
    for k in ("tokens", "kept_count", "status"):
        assert np.array_equal(one[k], many[k]), k
    assert np.allclose(one["logprobs"], many["logprobs"], rtol=0, atol=1e-12)


def knife_edge(y, ids, q, tol=1e-5):
    """Top-p rows whose mass above the cut lies within tol of p (the simulation's float64
    masses and the oracle's fixed-point ones may then decide differently)."""
    if q.p >= 1.0 or q.greedy:
        return False
    keep = np.ones(len(y), bool)
    if 2 <= q.k < len(y):
        keep &= y >= np.sort(y)[::-1][q.k - 1]
    yy = y[keep].astype(np.float64)
    w = np.exp(yy)
    o = np.lexsort((ids[keep], -yy))
    yo, wo = yy[o], w[o]
    start = np.r_[True, yo[1:] != yo[:-1]]
    above = (np.cumsum(wo) - wo)[np.nonzero(start)[0]] / w.sum()
    return bool(np.any(np.abs(above - q.p) < tol))


@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_agrees_with_the_oracle(n, oracle):
    b = make_workload(n, B=24, V=30011)
    o = transformed(b, oracle)
    ps = params_of(b)
    s = run(o["transformed"], ps, 4)
    assert np.array_equal(s["status"] != 0, o["status"] != 0)
    amb = 0
    for r in range(b.B):
        if o["status"][r] != 0:
            continue
        z = o["transformed"][r]
        ok = z > -np.inf
        y = ((z[ok] - z[ok].max()).astype(F32) * ps[r].inv_t).astype(F32)
        if knife_edge(y, np.nonzero(ok)[0], ps[r]):
            amb += 1
            continue
        assert s["tokens"][r] == o["tokens"][r], r
        assert s["kept_count"][r] == o["kept_count"][r], r
        assert abs(float(s["logprobs"][r]) - float(o["logprobs"][r])) <= 1e-5, r
    assert amb <= 2


def test_exchange_is_per_row_statistics(mixed):
    """Values exchanged per row: O(TP k) for top-k rows, O(TP) for min-p and untruncated
    rows, bins plus one band for top-p rows -- not O(V)."""
    b, o = mixed
    ps = params_of(b)
    tp = 4
    s = run(o["transformed"], ps, tp)
    for r, q in enumerate(ps):
        if q.greedy:
            assert s["volume"][r] <= 2 * tp
        elif 2 <= q.k <= 1000:
            assert s["volume"][r] <= 2 * tp + 2 * tp * (q.k + 64)
        assert s["volume"][r] < b.V


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_main(rank, world, port, path, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from constrained_logits_sampling_gb300.vocab_shard import RowParams, Shard, TorchComm, sample_sharded, split_vocab
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    d = np.load(path, allow_pickle=True)
    z, P = d["z"], d["params"]
    ps = [RowParams(float(t), int(k), float(p), float(mp), int(sd), int(pos)) for t, k, p, mp, sd, pos in P]
    e = split_vocab(z.shape[1], world)
    res = sample_sharded(ps, TorchComm(Shard(z[:, e[rank]:e[rank + 1]], e[rank], ps), dist))
    q.put((rank, res["tokens"].tolist(), res["kept_count"].tolist(), res["logprobs"].tolist()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks(mixed):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    b, o = mixed
    ps = params_of(b)
    one = run(o["transformed"], ps, 1)
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "shard_input.npz")
        P = np.array([(q.T, q.k, q.p, q.mp, q.seed, q.pos) for q in ps], dtype=object)
        np.savez(path, z=o["transformed"], params=P)
        ctx = mp.get_context("spawn")
        qu = ctx.Queue()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, path, qu)) for r in range(2)]
        for p in procs:
            p.start()
        res = sorted(qu.get(timeout=240) for _ in range(2))
        for p in procs:
            p.join(timeout=60)
            assert p.exitcode == 0
    for rank, tok, kept, lp in res:
        assert tok == one["tokens"].tolist() and kept == one["kept_count"].tolist()
        assert np.allclose(lp, one["logprobs"], rtol=0, atol=1e-12)
