"""ctypes front end of the CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline / reference arm are the only callers.  Nothing here imports the CUDA
library or its package code; inputs arrive as plain numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so in place with gcc (IEEE single/double, no fused
    multiply-adds, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=gnu11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
               "-pthread", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Args(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("V", ctypes.c_int32), ("logits_is_bf16", ctypes.c_int32),
        ("logits", ctypes.c_void_p), ("row_stride", ctypes.c_int64),
        ("temperatures", ctypes.c_void_p), ("top_ks", ctypes.c_void_p), ("top_ps", ctypes.c_void_p),
        ("min_ps", ctypes.c_void_p), ("rep", ctypes.c_void_p), ("freq", ctypes.c_void_p),
        ("pres", ctypes.c_void_p), ("hist_offs", ctypes.c_void_p), ("hist_ids", ctypes.c_void_p),
        ("bias_offs", ctypes.c_void_p), ("bias_ids", ctypes.c_void_p), ("bias_vals", ctypes.c_void_p),
        ("bitmask", ctypes.c_void_p), ("bitmask_row_stride", ctypes.c_int64),
        ("seeds", ctypes.c_void_p), ("positions", ctypes.c_void_p), ("step", ctypes.c_int64),
        ("tokens", ctypes.c_void_p), ("logprobs", ctypes.c_void_p), ("status", ctypes.c_void_p),
        ("transformed", ctypes.c_void_p), ("kept_count", ctypes.c_void_p), ("cut", ctypes.c_void_p),
        ("race_gap", ctypes.c_void_p), ("race_best", ctypes.c_void_p), ("nthreads", ctypes.c_int32),
        ("logprobs_orig", ctypes.c_void_p), ("logprobs_kept", ctypes.c_void_p),
        ("mode", ctypes.c_int32), ("tid_offs", ctypes.c_void_p), ("tid_ids", ctypes.c_void_p),
        ("tid_logprobs", ctypes.c_void_p), ("top_ns", ctypes.c_void_p), ("top_n_stride", ctypes.c_int32),
        ("top_ids", ctypes.c_void_p), ("top_logprobs", ctypes.c_void_p),
    ]


JOINT = 1       # top-p over the whole distribution, intersected with top-k
SCORE_ONLY = 2  # no draw: greedy route for every row; logprobs of requested ids


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            L.cls_oracle_sample.argtypes = [ctypes.POINTER(_Args)]
            L.cls_oracle_sample.restype = ctypes.c_int
            L.cls_oracle_philox4x32_10.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
            L.cls_oracle_philox4x32_10.restype = None
            L.cls_oracle_uniform.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64]
            L.cls_oracle_uniform.restype = ctypes.c_float
            L.cls_oracle_exp32.argtypes = [ctypes.c_float]
            L.cls_oracle_exp32.restype = ctypes.c_float
            L.cls_oracle_weight_fx.argtypes = [ctypes.c_float]
            L.cls_oracle_weight_fx.restype = ctypes.c_uint64
            L.cls_oracle_ceil_scaled.argtypes = [ctypes.c_uint64, ctypes.c_float]
            L.cls_oracle_ceil_scaled.restype = ctypes.c_uint64
            _lib = L
        return _lib


def _ptr(a: Optional[np.ndarray], dtype) -> Optional[int]:
    if a is None:
        return None
    assert a.dtype == np.dtype(dtype) and a.flags.c_contiguous, (a.dtype, dtype)
    return a.ctypes.data


def sample(batch, nthreads: int = 0, want_transformed: bool = False) -> Dict[str, np.ndarray]:
    """Run the oracle on a ``workloads.Batch`` (or any object with the same
    fields).  Returns tokens, logprobs (float64), logprobs_orig (T = 1),
    logprobs_kept (renormalised over the kept set), status, kept_count, cut,
    race_gap, race_best, threads, optionally the transformed logits z', and
    ``tid_logprobs`` when the batch carries requested ids (``tid_offs``,
    ``tid_ids``).  ``batch.mode`` holds the JOINT / SCORE_ONLY bits."""
    L = lib()
    B, V = int(batch.B), int(batch.V)
    logits = np.ascontiguousarray(batch.logits)
    if batch.logits_bf16:
        assert logits.dtype == np.uint16
    else:
        assert logits.dtype == np.float32
    keep = [logits]

    def arr(name, dtype):
        v = getattr(batch, name, None)
        if v is None:
            return None
        v = np.ascontiguousarray(v, dtype=dtype)
        keep.append(v)
        return v

    out = {
        "tokens": np.zeros(B, np.int32), "logprobs": np.zeros(B, np.float64),
        "status": np.zeros(B, np.int32), "kept_count": np.zeros(B, np.int32),
        "cut": np.zeros(B, np.float32), "race_gap": np.zeros(B, np.float32),
        "race_best": np.zeros(B, np.float32),
        "logprobs_orig": np.zeros(B, np.float64), "logprobs_kept": np.zeros(B, np.float64),
    }
    if want_transformed:
        out["transformed"] = np.zeros((B, V), np.float32)
    bm = arr("bitmask", np.int32)
    a = _Args()
    a.B, a.V, a.logits_is_bf16 = B, V, int(bool(batch.logits_bf16))
    a.logits = logits.ctypes.data
    a.row_stride = logits.shape[1] if logits.ndim == 2 else V
    for name, dt in (("temperatures", np.float32), ("top_ks", np.int32), ("top_ps", np.float32),
                     ("min_ps", np.float32), ("rep", np.float32), ("freq", np.float32),
                     ("pres", np.float32), ("hist_offs", np.int32), ("hist_ids", np.int32),
                     ("bias_offs", np.int32), ("bias_ids", np.int32), ("bias_vals", np.float32),
                     ("seeds", np.uint64), ("positions", np.int64)):
        setattr(a, name, _ptr(arr(name, dt), dt))
    a.bitmask = _ptr(bm, np.int32)
    a.bitmask_row_stride = bm.shape[1] if bm is not None else 0
    a.step = int(getattr(batch, "step", 0))
    a.tokens = out["tokens"].ctypes.data
    a.logprobs = out["logprobs"].ctypes.data
    a.status = out["status"].ctypes.data
    a.kept_count = out["kept_count"].ctypes.data
    a.cut = out["cut"].ctypes.data
    a.race_gap = out["race_gap"].ctypes.data
    a.race_best = out["race_best"].ctypes.data
    a.transformed = out["transformed"].ctypes.data if want_transformed else None
    a.nthreads = int(nthreads)
    a.logprobs_orig = out["logprobs_orig"].ctypes.data
    a.logprobs_kept = out["logprobs_kept"].ctypes.data
    a.mode = int(getattr(batch, "mode", 0) or 0)
    toffs, tids = arr("tid_offs", np.int32), arr("tid_ids", np.int32)
    if toffs is not None:
        a.tid_offs, a.tid_ids = toffs.ctypes.data, tids.ctypes.data
        out["tid_logprobs"] = np.zeros(max(int(toffs[-1]), 0), np.float64)
        a.tid_logprobs = out["tid_logprobs"].ctypes.data
    tns = arr("top_ns", np.int32)
    if tns is not None:
        stride = int(getattr(batch, "top_n_stride", 0) or max(int(tns.max()) if B else 1, 1))
        a.top_ns, a.top_n_stride = tns.ctypes.data, stride
        out["top_ids"] = np.full((B, stride), -7, np.int32)
        out["top_logprobs"] = np.full((B, stride), 7.0, np.float64)
        a.top_ids, a.top_logprobs = out["top_ids"].ctypes.data, out["top_logprobs"].ctypes.data
    out["threads"] = L.cls_oracle_sample(ctypes.byref(a))
    return out


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    o = np.zeros(4, np.uint32)
    lib().cls_oracle_philox4x32_10(c.ctypes.data, k.ctypes.data, o.ctypes.data)
    return o


def uniform(seed: int, position: int, token: int) -> float:
    return float(lib().cls_oracle_uniform(seed, position, token))


def exp32(y: float) -> float:
    return float(np.float32(lib().cls_oracle_exp32(float(np.float32(y)))))


def weight_fx(y: float) -> int:
    return int(lib().cls_oracle_weight_fx(float(np.float32(y))))


def ceil_scaled(W: int, p: float) -> int:
    return int(lib().cls_oracle_ceil_scaled(W, float(np.float32(p))))


def allowed_to_bitmask(offs, ids, V: int) -> np.ndarray:
    """Grammar-bitmask rows from allowed-token lists (vLLM page, "allowed token ids",
    expressed as the sampler's bitmask): bit i & 31 of word i >> 5 is set iff i is listed.
    A row with an id outside [0, V), a decreasing offset or an empty list is all zero
    (every token masked: the sampler reports the row INVALID)."""
    offs = np.asarray(offs, np.int64)
    ids = np.asarray(ids, np.int64)
    B, W = len(offs) - 1, (V + 31) // 32
    out = np.zeros((B, W), np.uint32)
    for r in range(B):
        lo, hi = int(offs[r]), int(offs[r + 1])
        if lo < 0 or hi < lo:
            continue
        row = ids[lo:hi]
        if ((row < 0) | (row >= V)).any():
            continue
        for i in row:
            out[r, i >> 5] |= np.uint32(1) << np.uint32(i & 31)
    return out.view(np.int32)
