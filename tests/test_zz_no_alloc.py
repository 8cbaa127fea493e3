"""clsample_apply_static: the handle-free entry point whose scratch is a fixed device
array compiled into the library.  Two calls in a row must give exactly what the
handle-based clsample_apply gives, and oversized calls are rejected on the host.

The file name sorts last so that the static array is first touched after every other
GPU test has run."""
import numpy as np
import pytest

from constrained_logits_sampling_gb300.workloads import make_workload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from constrained_logits_sampling_gb300 import build, sampler
    build.build()
    return sampler


def _outputs(B):
    return {"tokens": torch.empty(B, dtype=torch.int32, device="cuda"),
            "logprobs": torch.empty(B, dtype=torch.float32, device="cuda"),
            "status": torch.empty(B, dtype=torch.int32, device="cuda")}


@pytest.mark.parametrize("n", [2, 4, 5])
def test_static_matches_handle_twice(lib, n):
    b = make_workload(n, B=48)  # <= 64 rows; penalties, bias and masks where the workload has them
    s = lib.Sampler(b.B, b.V)
    kw = lib.batch_to_device(b, "cuda")
    logits = kw.pop("logits")
    ref = s(logits, **kw)
    torch.cuda.synchronize()
    for call in range(2):
        out = _outputs(b.B)
        args = s.make_args(logits, tokens=out["tokens"], logprobs=out["logprobs"], row_status=out["status"], **kw)
        lib.apply_static(args)
        torch.cuda.synchronize()
        for key in ("tokens", "status"):
            assert torch.equal(out[key], ref[key]), (n, call, key)
        g = out["logprobs"].cpu().numpy()
        r = ref["logprobs"].cpu().numpy()
        assert np.array_equal(g.view(np.uint32), r.view(np.uint32)), (n, call, "logprobs")


def test_static_rejects_oversize(lib):
    b = make_workload(1, B=4)
    s = lib.Sampler(b.B, b.V)
    kw = lib.batch_to_device(b, "cuda")
    logits = kw.pop("logits")
    out = _outputs(b.B)
    args = s.make_args(logits, tokens=out["tokens"], logprobs=out["logprobs"], row_status=out["status"], **kw)
    args.B = 65
    with pytest.raises(lib.ClsampleError) as e:
        lib.apply_static(args)
    assert e.value.code == -2  # CLSAMPLE_ERR_BATCH
    args.B = b.B
    args.V = 262145
    with pytest.raises(lib.ClsampleError) as e:
        lib.apply_static(args)
    assert e.value.code == -3  # CLSAMPLE_ERR_VOCAB


def _static_vs_handle(lib, b):
    s = lib.Sampler(b.B, b.V)
    kw = lib.batch_to_device(b, "cuda")
    logits = kw.pop("logits")
    ref = s(logits, **kw)
    out = _outputs(b.B)
    args = s.make_args(logits, tokens=out["tokens"], logprobs=out["logprobs"], row_status=out["status"], **kw)
    lib.apply_static(args)
    torch.cuda.synchronize()
    return out, ref


def test_static_calls_of_different_sizes_in_a_row(lib):
    """Calls of different V (slice count and length) and B one after another on the one
    array: each uses a prefix of it laid out for the longest slices, and whatever a call
    leaves there is read back by the next.  Each call equals its own handle bit for bit."""
    for n, B, V in ((4, 48, None), (4, 8, 5003), (2, 64, None), (5, 16, 40001), (4, 48, None)):
        b = make_workload(n, B=B, V=V)
        out, ref = _static_vs_handle(lib, b)
        for key in ("tokens", "status"):
            assert torch.equal(out[key], ref[key]), (n, B, V, key)
        assert np.array_equal(out["logprobs"].cpu().numpy().view(np.uint32),
                              ref["logprobs"].cpu().numpy().view(np.uint32)), (n, B, V)


def test_static_spill_rows_are_four(lib):
    """Flat rows under top-k spill every slice; the static array holds 4 spill rows (the
    header states it), a handle one per batch row.  With 8 such rows the static call
    samples 4 of them exactly like the handle and reports the other 4 OVERFLOW; every
    other row matches."""
    V = 151936
    B = 12
    rng = np.random.default_rng(41)
    z = (rng.standard_normal((B, V)) * 3).astype(np.float32)
    z[:8] = 0.0
    from constrained_logits_sampling_gb300.workloads import Batch
    b = Batch(B=B, V=V, logits=z, logits_bf16=False)
    b.temperatures = np.ones(B, np.float32)
    b.top_ks = np.full(B, 50, np.int32)
    b.positions = np.arange(B, dtype=np.int64)
    out, ref = _static_vs_handle(lib, b)
    st, rs = out["status"].cpu().numpy(), ref["status"].cpu().numpy()
    assert np.all(rs == 0)
    assert np.all(st[8:] == 0) and (st[:8] == 1).sum() == 4 and (st[:8] == 0).sum() == 4
    ok = st == 0
    assert np.array_equal(out["tokens"].cpu().numpy()[ok], ref["tokens"].cpu().numpy()[ok])
