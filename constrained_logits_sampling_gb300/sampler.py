"""Python binding of libclsample.so (ctypes).

Argument marshalling only: every step of the sampler runs in the CUDA library.  The
tensors must already live on the CUDA device of the handle; PyTorch supplies device
memory and the current stream.  There is no CPU fallback: if the library is missing,
``Sampler`` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Dict, Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libclsample.so")
_lock = threading.Lock()
_lib = None

LOGITS_F32, LOGITS_BF16 = 0, 1
MODE_JOINT_TOPK_TOPP, MODE_SCORE_ONLY, MODE_FAST_SWEEP = 1, 2, 4
ROW_OK, ROW_OVERFLOW, ROW_INVALID = 0, 1, 2


class Args(ctypes.Structure):
    """Mirror of clsample_args_t (include/clsample.h)."""
    _fields_ = [
        ("B", ctypes.c_int32), ("V", ctypes.c_int32), ("logits_dtype", ctypes.c_int32),
        ("mode", ctypes.c_int32),
        ("logits", ctypes.c_void_p), ("logits_row_stride", ctypes.c_int64),
        ("temperatures", ctypes.c_void_p), ("top_ks", ctypes.c_void_p), ("top_ps", ctypes.c_void_p),
        ("min_ps", ctypes.c_void_p), ("rep", ctypes.c_void_p), ("freq", ctypes.c_void_p),
        ("pres", ctypes.c_void_p), ("hist_offs", ctypes.c_void_p), ("hist_ids", ctypes.c_void_p),
        ("bias_offs", ctypes.c_void_p), ("bias_ids", ctypes.c_void_p), ("bias_vals", ctypes.c_void_p),
        ("bitmask", ctypes.c_void_p), ("bitmask_row_stride", ctypes.c_int64),
        ("seeds", ctypes.c_void_p), ("positions", ctypes.c_void_p), ("step", ctypes.c_int64),
        ("tokens", ctypes.c_void_p), ("logprobs", ctypes.c_void_p), ("row_status", ctypes.c_void_p),
        ("dbg_transformed", ctypes.c_void_p), ("dbg_kept_count", ctypes.c_void_p),
        ("dbg_cut", ctypes.c_void_p), ("logprobs_orig", ctypes.c_void_p), ("logprobs_kept", ctypes.c_void_p),
        ("tid_offs", ctypes.c_void_p), ("tid_ids", ctypes.c_void_p), ("tid_logprobs", ctypes.c_void_p),
        ("top_ns", ctypes.c_void_p), ("top_n_stride", ctypes.c_int32), ("reserved1", ctypes.c_int32),
        ("top_ids", ctypes.c_void_p), ("top_logprobs", ctypes.c_void_p),
    ]


EXPORTS = ("clsample_create", "clsample_destroy", "clsample_apply", "clsample_prepare", "clsample_sample",
           "clsample_apply_static", "clsample_strerror", "clsample_geometry", "clsample_occupancy",
           "clsample_debug_weights", "clsample_debug_uniforms", "clsample_allowed_to_bitmask")


def load_library(path: str = LIB_PATH):
    """Load libclsample.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it with "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(path)
            L.clsample_create.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_void_p)]
            L.clsample_create.restype = ctypes.c_int
            L.clsample_destroy.argtypes = [ctypes.c_void_p]
            L.clsample_destroy.restype = None
            for name in ("clsample_apply", "clsample_prepare", "clsample_sample"):
                getattr(L, name).argtypes = [ctypes.c_void_p, ctypes.POINTER(Args), ctypes.c_void_p]
                getattr(L, name).restype = ctypes.c_int
            L.clsample_apply_static.argtypes = [ctypes.POINTER(Args), ctypes.c_void_p]
            L.clsample_apply_static.restype = ctypes.c_int
            L.clsample_strerror.argtypes = [ctypes.c_int]
            L.clsample_strerror.restype = ctypes.c_char_p
            L.clsample_geometry.argtypes = [ctypes.c_int32, ctypes.POINTER(ctypes.c_int32),
                                            ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
            L.clsample_geometry.restype = ctypes.c_int
            L.clsample_occupancy.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]
            L.clsample_occupancy.restype = ctypes.c_int
            L.clsample_debug_weights.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
            L.clsample_debug_weights.restype = ctypes.c_int
            L.clsample_debug_uniforms.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int32, ctypes.c_void_p]
            L.clsample_debug_uniforms.restype = ctypes.c_int
            L.clsample_allowed_to_bitmask.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                                      ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64,
                                                      ctypes.c_void_p]
            L.clsample_allowed_to_bitmask.restype = ctypes.c_int
            _lib = L
        return _lib


class ClsampleError(RuntimeError):
    def __init__(self, code: int):
        msg = load_library().clsample_strerror(code).decode()
        super().__init__(f"clsample error {code}: {msg}")
        self.code = code


def _check(code: int):
    if code != 0:
        raise ClsampleError(code)


def geometry(vocab: int):
    L = load_library()
    c, k, s = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(L.clsample_geometry(vocab, ctypes.byref(c), ctypes.byref(k), ctypes.byref(s)))
    return {"slices": c.value, "chunk": k.value, "smem_bytes": s.value}


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _dptr(t: Optional[torch.Tensor], dtype: torch.dtype, n: Optional[int], name: str,
          device: torch.device) -> Optional[int]:
    if t is None:
        return None
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if n is not None and t.numel() != n:
        raise ValueError(f"{name} has {t.numel()} elements, expected {n}")
    return t.data_ptr()


class Sampler:
    """One handle of the C library: batches of up to ``max_batch`` rows over a
    vocabulary of ``vocab`` tokens, on the current CUDA device."""

    def __init__(self, max_batch: int, vocab: int):
        self._L = load_library()
        if not torch.cuda.is_available():
            raise RuntimeError("the sampler needs a CUDA device")
        self.device = torch.device("cuda", torch.cuda.current_device())
        h = ctypes.c_void_p()
        _check(self._L.clsample_create(int(max_batch), int(vocab), ctypes.byref(h)))
        self._h = h
        self.max_batch, self.vocab = int(max_batch), int(vocab)

    def resident_ctas(self, bf16: bool = False) -> int:
        """Resident CTAs of the sampler kernel on this device (``clsample_occupancy``)."""
        n = ctypes.c_int32()
        _check(self._L.clsample_occupancy(self._h, LOGITS_BF16 if bf16 else LOGITS_F32, ctypes.byref(n)))
        return n.value

    def close(self):
        if getattr(self, "_h", None):
            self._L.clsample_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def make_args(self, logits: torch.Tensor, *, temperatures=None, top_ks=None, top_ps=None,
                  min_ps=None, rep=None, freq=None, pres=None, hist_offs=None, hist_ids=None,
                  bias_offs=None, bias_ids=None, bias_vals=None, bitmask=None, seeds=None,
                  positions=None, step: int = 0, tokens=None, logprobs=None, row_status=None,
                  dbg_transformed=None, dbg_kept_count=None, dbg_cut=None, logprobs_orig=None,
                  logprobs_kept=None, mode: int = 0, tid_offs=None, tid_ids=None, tid_logprobs=None,
                  top_ns=None, top_n_stride: int = 0, top_ids=None, top_logprobs=None) -> Args:
        if logits.dim() != 2 or logits.stride(1) != 1:
            raise ValueError("logits must be [B, V] with unit column stride")
        if logits.dtype == torch.float32:
            dt = LOGITS_F32
        elif logits.dtype == torch.bfloat16:
            dt = LOGITS_BF16
        else:
            raise ValueError(f"unsupported logits dtype {logits.dtype}")
        B, V = logits.shape
        dev = self.device
        if logits.device != dev:
            raise ValueError(f"logits on {logits.device}, handle on {dev}")
        a = Args()
        a.B, a.V, a.logits_dtype, a.mode = B, V, dt, int(mode)
        a.logits = logits.data_ptr()
        a.logits_row_stride = logits.stride(0)
        f32, i32, i64 = torch.float32, torch.int32, torch.int64
        a.temperatures = _dptr(temperatures, f32, B, "temperatures", dev)
        a.top_ks = _dptr(top_ks, i32, B, "top_ks", dev)
        a.top_ps = _dptr(top_ps, f32, B, "top_ps", dev)
        a.min_ps = _dptr(min_ps, f32, B, "min_ps", dev)
        a.rep = _dptr(rep, f32, B, "rep", dev)
        a.freq = _dptr(freq, f32, B, "freq", dev)
        a.pres = _dptr(pres, f32, B, "pres", dev)
        a.hist_offs = _dptr(hist_offs, i32, B + 1, "hist_offs", dev)
        a.hist_ids = _dptr(hist_ids, i32, None, "hist_ids", dev)
        a.bias_offs = _dptr(bias_offs, i32, B + 1, "bias_offs", dev)
        a.bias_ids = _dptr(bias_ids, i32, None, "bias_ids", dev)
        a.bias_vals = _dptr(bias_vals, f32, None, "bias_vals", dev)
        if bitmask is not None:
            if bitmask.dim() != 2 or bitmask.shape[0] != B or bitmask.stride(1) != 1:
                raise ValueError("bitmask must be [B, W] with unit column stride")
            if bitmask.dtype != i32 or bitmask.device != dev:
                raise ValueError("bitmask must be int32 on the handle's device")
            a.bitmask = bitmask.data_ptr()
            a.bitmask_row_stride = bitmask.stride(0)
        if seeds is not None and seeds.dtype not in (i64, getattr(torch, "uint64", i64)):
            raise ValueError("seeds must be int64 or uint64 (64-bit keys)")
        a.seeds = _dptr(seeds, seeds.dtype if seeds is not None else i64, B, "seeds", dev)
        a.positions = _dptr(positions, i64, B, "positions", dev)
        a.step = int(step)
        a.tokens = _dptr(tokens, i32, B, "tokens", dev)
        a.logprobs = _dptr(logprobs, f32, B, "logprobs", dev)
        a.row_status = _dptr(row_status, i32, B, "row_status", dev)
        a.dbg_transformed = _dptr(dbg_transformed, f32, B * V, "dbg_transformed", dev)
        a.dbg_kept_count = _dptr(dbg_kept_count, i32, B, "dbg_kept_count", dev)
        a.dbg_cut = _dptr(dbg_cut, f32, B, "dbg_cut", dev)
        a.logprobs_orig = _dptr(logprobs_orig, f32, B, "logprobs_orig", dev)
        a.logprobs_kept = _dptr(logprobs_kept, f32, B, "logprobs_kept", dev)
        a.tid_offs = _dptr(tid_offs, i32, B + 1, "tid_offs", dev)
        a.tid_ids = _dptr(tid_ids, i32, None, "tid_ids", dev)
        a.tid_logprobs = _dptr(tid_logprobs, f32, None, "tid_logprobs", dev)
        a.top_ns = _dptr(top_ns, i32, B, "top_ns", dev)
        a.top_n_stride = int(top_n_stride)
        a.top_ids = _dptr(top_ids, i32, B * max(int(top_n_stride), 0), "top_ids", dev) if top_ids is not None else None
        a.top_logprobs = (_dptr(top_logprobs, f32, B * max(int(top_n_stride), 0), "top_logprobs", dev)
                          if top_logprobs is not None else None)
        return a

    def apply(self, args: Args, stream: Optional[torch.cuda.Stream] = None):
        """Enqueue one call (``clsample_apply``) on ``stream`` (default: current)."""
        _check(self._L.clsample_apply(self._h, ctypes.byref(args), _stream_ptr(stream)))

    def prepare(self, args: Args, stream: Optional[torch.cuda.Stream] = None):
        """Enqueue the ordering half of a call (``clsample_prepare``)."""
        _check(self._L.clsample_prepare(self._h, ctypes.byref(args), _stream_ptr(stream)))

    def sample(self, args: Args, stream: Optional[torch.cuda.Stream] = None):
        """Enqueue the sampler half of a call (``clsample_sample``); reads what the
        last ``prepare`` on this handle wrote."""
        _check(self._L.clsample_sample(self._h, ctypes.byref(args), _stream_ptr(stream)))

    def __call__(self, logits: torch.Tensor, *, debug: bool = False, variants: bool = False, stream=None,
                 **kw) -> Dict[str, torch.Tensor]:
        """Sample one token per row.  Returns a dict with ``tokens`` (int32),
        ``logprobs`` (float32) and ``status`` (int32); with ``debug`` also
        ``transformed`` [B, V], ``kept_count`` and ``cut``; with ``variants`` (or
        ``debug``) also ``logprobs_orig`` (T = 1) and ``logprobs_kept`` (renormalised
        over the kept set); with ``tid_offs``/``tid_ids`` (requested token ids, CSR)
        also ``tid_logprobs``; with ``top_ns`` (and ``top_n_stride``, default 32) also
        ``top_ids`` and ``top_logprobs`` [B, stride].  ``mode`` takes the MODE_* bits."""
        B, V = logits.shape
        dev = self.device
        out = {
            "tokens": torch.empty(B, dtype=torch.int32, device=dev),
            "logprobs": torch.empty(B, dtype=torch.float32, device=dev),
            "status": torch.empty(B, dtype=torch.int32, device=dev),
        }
        if debug:
            out["transformed"] = torch.empty(B, V, dtype=torch.float32, device=dev)
            out["kept_count"] = torch.empty(B, dtype=torch.int32, device=dev)
            out["cut"] = torch.empty(B, dtype=torch.float32, device=dev)
        if variants or debug:
            out["logprobs_orig"] = torch.empty(B, dtype=torch.float32, device=dev)
            out["logprobs_kept"] = torch.empty(B, dtype=torch.float32, device=dev)
        if kw.get("top_ns") is not None:
            stride = int(kw.setdefault("top_n_stride", 32))
            out["top_ids"] = torch.empty(B, stride, dtype=torch.int32, device=dev)
            out["top_logprobs"] = torch.empty(B, stride, dtype=torch.float32, device=dev)
        if kw.get("tid_offs") is not None:
            n = kw["tid_ids"].numel() if kw.get("tid_ids") is not None else 0
            out["tid_logprobs"] = torch.empty(max(n, 1), dtype=torch.float32, device=dev)[:n]
        args = self.make_args(logits, tokens=out["tokens"], logprobs=out["logprobs"],
                              row_status=out["status"], dbg_transformed=out.get("transformed"),
                              dbg_kept_count=out.get("kept_count"), dbg_cut=out.get("cut"),
                              logprobs_orig=out.get("logprobs_orig"), logprobs_kept=out.get("logprobs_kept"),
                              tid_logprobs=out.get("tid_logprobs"), top_ids=out.get("top_ids"),
                              top_logprobs=out.get("top_logprobs"), **kw)
        self.apply(args, stream)
        return out


def apply_static(args: Args, stream: Optional[torch.cuda.Stream] = None):
    """One call through ``clsample_apply_static`` (no handle, no allocation; at most 64
    rows; calls on one device must be ordered)."""
    _check(load_library().clsample_apply_static(ctypes.byref(args), _stream_ptr(stream)))


def allowed_to_bitmask(offs: torch.Tensor, ids: torch.Tensor, V: int, bitmask: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
    """Grammar-bitmask rows from allowed-token lists (CSR on the device), built by the
    library's kernel.  Returns (or fills) int32 [B, ceil(V/32)]."""
    L = load_library()
    B = offs.numel() - 1
    if bitmask is None:
        bitmask = torch.empty(max(B, 0), (V + 31) // 32, dtype=torch.int32, device=offs.device)
    if offs.dtype != torch.int32 or ids.dtype != torch.int32 or bitmask.dtype != torch.int32:
        raise ValueError("offs, ids and bitmask must be int32")
    if bitmask.dim() != 2 or bitmask.stride(1) != 1:
        raise ValueError("bitmask must be [B, W] with unit column stride")
    ids_ptr = ids.data_ptr() if ids.numel() else offs.data_ptr()  # an empty list is never read
    _check(L.clsample_allowed_to_bitmask(offs.contiguous().data_ptr(), ids_ptr, B, V, bitmask.data_ptr(),
                                         bitmask.stride(0), _stream_ptr(stream)))
    return bitmask


def debug_weights(y: torch.Tensor) -> torch.Tensor:
    """floor(exp32(y) * 2^40) computed by the library's device code."""
    L = load_library()
    y = y.contiguous()
    w = torch.empty(y.numel(), dtype=torch.int64, device=y.device)
    _check(L.clsample_debug_weights(y.data_ptr(), w.data_ptr(), y.numel(), _stream_ptr(None)))
    return w


def debug_uniforms(seeds: torch.Tensor, positions: torch.Tensor, tokens: torch.Tensor) -> torch.Tensor:
    """Race uniforms U(seed, position, token) computed by the library's device code."""
    L = load_library()
    n = seeds.numel()
    u = torch.empty(n, dtype=torch.float32, device=seeds.device)
    _check(L.clsample_debug_uniforms(seeds.contiguous().data_ptr(), positions.contiguous().data_ptr(),
                                     tokens.contiguous().data_ptr(), u.data_ptr(), n, _stream_ptr(None)))
    return u


def batch_to_device(batch, device) -> Dict[str, object]:
    """Move a ``workloads.Batch`` to the device as keyword arguments of ``Sampler``.
    (Host-to-device copies only; no arithmetic.)"""
    import numpy as np

    def t(x, dtype=None):
        if x is None:
            return None
        if x.dtype == np.uint64:
            return torch.from_numpy(x.view(np.int64)).to(device)
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)

    if batch.logits_bf16:
        logits = torch.from_numpy(batch.logits.view(np.int16)).to(device).view(torch.bfloat16)
    else:
        logits = torch.from_numpy(batch.logits).to(device)
    kw = dict(temperatures=t(batch.temperatures), top_ks=t(batch.top_ks), top_ps=t(batch.top_ps),
              min_ps=t(batch.min_ps), rep=t(batch.rep), freq=t(batch.freq), pres=t(batch.pres),
              hist_offs=t(batch.hist_offs), hist_ids=t(batch.hist_ids), bias_offs=t(batch.bias_offs),
              bias_ids=t(batch.bias_ids), bias_vals=t(batch.bias_vals), bitmask=t(batch.bitmask),
              seeds=t(batch.seeds), positions=t(batch.positions), step=int(batch.step))
    if getattr(batch, "mode", 0):
        kw["mode"] = int(batch.mode)
    if getattr(batch, "top_ns", None) is not None:
        kw["top_ns"] = t(np.asarray(batch.top_ns, np.int32))
        kw["top_n_stride"] = int(batch.top_n_stride or max(int(np.max(batch.top_ns)) if batch.B else 1, 1))
    if getattr(batch, "tid_offs", None) is not None:
        ids = np.asarray(batch.tid_ids, np.int32)
        # a device copy of an empty array may have no address: keep one padding slot
        kw["tid_offs"] = t(batch.tid_offs)
        kw["tid_ids"] = t(np.concatenate([ids, np.zeros(1, np.int32)]))[:ids.size]
    return {"logits": logits, **kw}
