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
