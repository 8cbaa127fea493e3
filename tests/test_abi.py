"""The C-ABI library loads and exports every entry point include/clsample.h declares,
and the Python mirror of clsample_args_t has the header's layout.  No GPU needed:
only host-side entry points are called."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "clsample.h")


@pytest.fixture(scope="module")
def lib():
    from constrained_logits_sampling_gb300 import build, sampler
    build.build()
    return sampler.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(clsample_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "clsample_apply" in names and "clsample_create" in names
    for n in names:
        assert hasattr(lib, n), n
    from constrained_logits_sampling_gb300 import sampler
    assert set(sampler.EXPORTS) == set(names)


def test_nm_dynamic_symbols(lib):
    from constrained_logits_sampling_gb300 import sampler
    out = subprocess.run(["nm", "-D", "--defined-only", sampler.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    for n in declared_functions():
        assert re.search(rf"\bT {n}$", out, re.M), n


def test_strerror_and_geometry(lib):
    from constrained_logits_sampling_gb300 import sampler
    assert lib.clsample_strerror(0) == b"success"
    for code in range(-8, 0):
        assert lib.clsample_strerror(code) != b"unknown error"
    g = sampler.geometry(151936)
    assert g == {"slices": 10, "chunk": 15232, "smem_bytes": g["smem_bytes"]}
    assert g["smem_bytes"] <= 72 * 1024  # three CTAs per SM
    g = sampler.geometry(262144)
    assert g["slices"] == 18 and g["chunk"] % 128 == 0
    assert (g["slices"] - 1) * g["chunk"] < 262144 <= g["slices"] * g["chunk"]
    with pytest.raises(sampler.ClsampleError):
        sampler.geometry(262145)
    assert sampler.geometry(8)["slices"] == 1
    assert sampler.geometry(32000)["chunk"] * sampler.geometry(32000)["slices"] >= 32000
    with pytest.raises(sampler.ClsampleError):
        sampler.geometry(0)


def test_args_layout_matches_header(lib):
    """Compile a probe against the header with gcc and compare every field offset."""
    from constrained_logits_sampling_gb300.sampler import Args
    fields = [f for f, _ in Args._fields_]
    body = "\n".join(f'  printf("%s %zu\\n", "{f}", offsetof(clsample_args_t, {f}));' for f in fields)
    src = ("#include <stdio.h>\n#include <stddef.h>\n#include \"clsample.h\"\nint main(void){\n"
           f'  printf("sizeof %zu\\n", sizeof(clsample_args_t));\n{body}\n  return 0;\n}}\n')
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "probe.c")
        exe = os.path.join(d, "probe")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-o", exe, c], check=True)
        lines = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    got = dict(l.split() for l in lines if l)
    assert int(got["sizeof"]) == ctypes.sizeof(Args)
    for f in fields:
        assert int(got[f]) == getattr(Args, f).offset, f


def test_host_validation_without_gpu(lib):
    """Argument errors are reported on the host before any CUDA call."""
    from constrained_logits_sampling_gb300.sampler import Args
    assert lib.clsample_apply(None, None, None) == -1
    h = ctypes.c_void_p()
    assert lib.clsample_create(4, 100, None) == -1
    assert lib.clsample_create(-1, 100, ctypes.byref(h)) == -2
    assert lib.clsample_create(4, 0, ctypes.byref(h)) == -3
    assert lib.clsample_debug_weights(None, None, -1, None) == -2
    assert lib.clsample_debug_weights(None, None, 0, None) == 0
