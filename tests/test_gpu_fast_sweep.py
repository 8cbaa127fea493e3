"""GPU parity of the single-sweep fast path (CLSAMPLE_MODE_FAST_SWEEP): batches whose
rows are all greedy or untruncated, against the CPU oracle (which knows no such mode:
the flag must not change any result), plus the flag's own contract -- rows that break
the assertion are INVALID, and outputs it does not serve are refused on the host."""
import numpy as np
import pytest

from constrained_logits_sampling_gb300.workloads import MODE_FAST_SWEEP, Batch, make_workload

from parity import LOGPROB_TOL, compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
F32 = np.float32


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from constrained_logits_sampling_gb300 import build
    build.build()


def sweep_batch(z, bf16=False, **kw):
    z = np.ascontiguousarray(np.atleast_2d(z))
    b = Batch(B=z.shape[0], V=z.shape[1], logits=z, logits_bf16=bf16)
    for k, v in kw.items():
        setattr(b, k, v)
    b.mode = MODE_FAST_SWEEP
    return b


@pytest.mark.parametrize("w", [6, 7])
def test_fast_sweep_full_size(w):
    """All-greedy and all-untruncated batches at full size (B=192, V=151936, penalties,
    bias and masks), in the configuration the benchmark times."""
    b = make_workload(w)
    stats = compare(b, run_gpu(b), run_oracle(b), name=f"workload {w}")
    print(f"workload {w}: ambiguous={stats['ambiguous']} max|dlogprob|={stats['max_logprob_err']:.2e}")


@pytest.mark.parametrize("w", [6, 7])
@pytest.mark.parametrize("V", [23, 31, 4099, 8192, 8193, 40000])
def test_fast_sweep_ragged(w, V):
    """Vocabularies of a few vectors and a ragged one, exactly one slice, one token past
    it, and several slices with a ragged tail."""
    b = make_workload(w, B=12, V=V)
    compare(b, run_gpu(b), run_oracle(b), name=f"w{w} V={V}")


@pytest.mark.parametrize("V", [1, 2, 3, 5])
def test_fast_sweep_vocab_below_a_vector(V):
    rng = np.random.default_rng(V)
    z = rng.standard_normal((6, V)).astype(F32)
    b = sweep_batch(z, temperatures=np.array([0, 1, 0.5, 2, 0, 1], F32), positions=np.arange(6, dtype=np.int64))
    compare(b, run_gpu(b), run_oracle(b), name=f"V={V}")


def test_fast_sweep_bf16_and_mixed_rows():
    """bf16 logits with massive exact ties, greedy and untruncated rows in one batch,
    top_k at or above the allowed count (no cut), score-only rows."""
    b = make_workload(5, B=40, V=20011)
    b.temperatures[::3] = 0.0
    b.top_ks[:] = -1
    b.top_ks[1::5] = 25000  # >= the allowed tokens: untruncated
    b.top_ks[2::7] = 1      # greedy
    b.top_ps[:] = 1.0
    b.min_ps[:] = 0.0
    b.mode = MODE_FAST_SWEEP
    compare(b, run_gpu(b), run_oracle(b), name="bf16 mixed")


def test_fast_sweep_non_finite_masked_and_unaligned():
    from constrained_logits_sampling_gb300.sampler import Sampler, batch_to_device
    V = 9001
    rng = np.random.default_rng(5)
    z = (rng.standard_normal((8, V)) * 2).astype(F32)
    z[0, 10] = np.nan
    z[1, 20] = np.inf
    z[2, :] = -np.inf
    z[3, :] = np.nan  # every token out -> INVALID
    z[4, 100] = np.inf
    z[4, 8500] = np.inf  # two +inf in different slices: lowest id wins
    bm = np.full((8, (V + 31) // 32), -1, np.int32)
    bm[5, :] = 0  # nothing allowed -> INVALID
    bm[6, :] = 0
    bm[6, 280] = 1 << 7  # exactly one allowed token, in the second slice
    b = sweep_batch(z, bitmask=bm, temperatures=np.array([1, 0, 1, 1, 0, 1, 1, 0.5], F32),
                    positions=np.arange(8, dtype=np.int64))
    o = run_oracle(b)
    g = run_gpu(b)
    compare(b, g, o, name="non-finite")
    assert g["status"][3] == 2 and g["status"][5] == 2
    assert g["tokens"][1] == 20 and g["tokens"][4] == 100 and g["tokens"][6] == 280 * 32 + 7
    # rows that lose 16-byte alignment (scalar loads)
    s = Sampler(8, V)
    kw = batch_to_device(b, s.device)
    logits = kw.pop("logits")
    for pad in (1, 3):
        big = torch.full((8, V + pad), float("nan"), device="cuda")
        big[:, :V] = logits
        out = s(big[:, :V], debug=True, **kw)
        torch.cuda.synchronize()
        compare(b, {k: v.cpu().numpy() for k, v in out.items()}, o, name=f"pad {pad}")


def test_fast_sweep_penalties_in_one_slice():
    """Many distinct penalised ids and repeated bias ids (the last entry wins) in one slice."""
    V = 30000
    rng = np.random.default_rng(7)
    z = (rng.standard_normal((3, V)) * 3).astype(F32)
    hist = np.concatenate([np.arange(0, 4000), np.arange(0, 4000, 7), rng.integers(0, V, 300)]).astype(np.int32)
    offs = np.array([0, len(hist), len(hist) + 1, len(hist) + 1], np.int32)
    bias_ids = np.concatenate([np.arange(100, 1400, 3), np.arange(100, 400, 3)]).astype(np.int32)
    b = sweep_batch(z, hist_offs=offs, hist_ids=np.concatenate([hist, np.array([5], np.int32)]),
                    freq=np.full(3, 0.1, F32), pres=np.full(3, 0.2, F32), rep=np.full(3, 1.2, F32),
                    bias_offs=np.array([0, len(bias_ids), len(bias_ids), len(bias_ids)], np.int32),
                    bias_ids=bias_ids, bias_vals=rng.uniform(-3, 3, len(bias_ids)).astype(F32),
                    temperatures=np.array([0.0, 0.8, 1.0], F32), positions=np.arange(3, dtype=np.int64))
    compare(b, run_gpu(b), run_oracle(b), name="penalties")


def test_fast_sweep_equals_general_path():
    """The flag changes no result: the same untruncated batch through the general path."""
    b = make_workload(7, B=48, V=50021)
    g = run_gpu(b)
    b.mode = 0
    h = run_gpu(b)
    for k in ("tokens", "status", "kept_count", "transformed"):
        assert np.array_equal(g[k], h[k]), k
    ok = g["status"] == 0
    assert np.all(np.abs(g["logprobs"][ok].astype(np.float64) - h["logprobs"][ok]) <= LOGPROB_TOL)


def test_fast_sweep_rows_breaking_the_assertion_are_invalid():
    """A top-k that cuts, a top-p below 1 or a min-p above 0 on a sampled row makes that
    row INVALID; greedy rows with any truncation parameters stay valid."""
    V = 5000
    rng = np.random.default_rng(3)
    z = rng.standard_normal((6, V)).astype(F32)
    b = sweep_batch(z, temperatures=np.array([1, 1, 1, 1, 0, 1], F32),
                    top_ks=np.array([50, -1, -1, 5000, 50, -1], np.int32),
                    top_ps=np.array([1, 0.9, 1, 1, 0.5, 1], F32),
                    min_ps=np.array([0, 0, 0.05, 0, 0.1, 0], F32), positions=np.arange(6, dtype=np.int64))
    g = run_gpu(b)
    assert list(g["status"]) == [2, 2, 2, 0, 0, 0]
    o = run_oracle(b)
    for r in (3, 4, 5):
        assert g["tokens"][r] == o["tokens"][r]


def test_fast_sweep_refuses_requested_id_and_top_n_outputs():
    from constrained_logits_sampling_gb300.sampler import ClsampleError, Sampler, batch_to_device
    b = make_workload(6, B=4, V=1000)
    s = Sampler(4, 1000)
    kw = batch_to_device(b, s.device)
    logits = kw.pop("logits")
    with pytest.raises(ClsampleError):
        s(logits, top_ns=torch.full((4,), 3, dtype=torch.int32, device="cuda"), top_n_stride=3, **kw)
    s(logits, **kw)
    torch.cuda.synchronize()
