"""Compile libclsample.so (sm_103a) in place with nvcc: each CUDA source to an object in
parallel, then one shared-library link.  Rebuilds when any source or header is newer
than the library."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, "clsample.cu")]
HEADERS = [os.path.join(ROOT, "include", "clsample.h")] + sorted(
    os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h")))
LIB = os.path.join(PKG, "libclsample.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC",
    "-Xptxas", "-v",
]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def build(force: bool = False, verbose: bool = False) -> str:
    newest = max(os.path.getmtime(p) for p in SOURCES + HEADERS)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest:
        return LIB
    tag = f".tmp{os.getpid()}"
    objs = [os.path.join(CSRC, os.path.basename(s) + tag + ".o") for s in SOURCES]
    procs = []
    for src, obj in zip(SOURCES, objs):
        cmd = [nvcc(), *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-c", src, "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)))
    report = []
    failed = None
    for cmd, p in procs:
        out, err = p.communicate()
        report.append(err)
        if p.returncode != 0 and failed is None:
            failed = (cmd, out + err)
    try:
        if failed:
            sys.stderr.write(failed[1])
            raise RuntimeError("nvcc failed: " + " ".join(failed[0]))
        tmp = LIB + tag
        link = [nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp, *objs, "-lcudart"]
        res = subprocess.run(link, capture_output=True, text=True)
        if res.returncode != 0:
            sys.stderr.write(res.stdout + res.stderr)
            raise RuntimeError("nvcc link failed: " + " ".join(link))
        with open(os.path.join(PKG, "ptxas_report.txt"), "w") as f:
            f.write("".join(report))
        if verbose:
            sys.stderr.write("".join(report))
        os.replace(tmp, LIB)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(LIB)
