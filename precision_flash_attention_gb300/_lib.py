"""ctypes binding of libpfa (include/pfa.h): argument marshalling only.

Each function takes torch CUDA tensors, checks dtype/device/layout, and passes
raw device pointers, sizes and the current CUDA stream to the C entry point of
the same name. All computation happens in libpfa's kernels; there is no other
code path. If the library has not been built the first call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_LIB = None

PFA_OK = 0
STATUS_NAMES = {0: "PFA_OK", -1: "PFA_ERR_INVALID_ARG", -2: "PFA_ERR_MISALIGNED",
                -3: "PFA_ERR_UNSUPPORTED", -4: "PFA_ERR_LAUNCH", -5: "PFA_ERR_DEVICE",
                -6: "PFA_ERR_TOO_LARGE"}

# Every entry point declared in include/pfa.h.
EXPORTS = ("pfa_attn_fwd", "pfa_attn_delta", "pfa_attn_delta_alt", "pfa_attn_bwd",
           "pfa_attn_bwd_accum", "pfa_attn_bwd_noalloc", "pfa_bwd_workspace_bytes", "pfa_status_string",
           "pfa_last_error", "pfa_device_error", "pfa_device_error_site", "pfa_wait_probe")


class PfaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = ""
        if status == -4:  # PFA_ERR_LAUNCH: name the CUDA error behind it
            detail = f" [{load().pfa_last_error().decode()}]"
        super().__init__(f"{where}: {status_string(status)} ({status}){detail}")


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libpfa.so (built in-tree by ``__graft_entry__.build()``)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or library_path()
    if not os.path.exists(p):
        raise RuntimeError(f"libpfa is not built ({p} missing): run __graft_entry__.build() first")
    lib = ctypes.CDLL(p)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.pfa_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, f, f, vp, vp]
    lib.pfa_attn_fwd.restype = i
    lib.pfa_attn_delta.argtypes = [vp, vp, vp, i, i, i, i, vp]
    lib.pfa_attn_delta.restype = i
    lib.pfa_attn_delta_alt.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.pfa_attn_delta_alt.restype = i
    lib.pfa_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.pfa_attn_bwd.restype = i
    lib.pfa_attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.pfa_attn_bwd_accum.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.pfa_attn_bwd_accum.restype = i
    lib.pfa_attn_bwd_noalloc.restype = i
    lib.pfa_bwd_workspace_bytes.argtypes = [i, i, i, i]
    lib.pfa_bwd_workspace_bytes.restype = sz
    lib.pfa_status_string.argtypes = [i]
    lib.pfa_status_string.restype = ctypes.c_char_p
    lib.pfa_last_error.argtypes = []
    lib.pfa_last_error.restype = ctypes.c_char_p
    lib.pfa_device_error_site.argtypes = []
    lib.pfa_device_error_site.restype = ctypes.c_longlong
    lib.pfa_device_error.argtypes = [i]
    lib.pfa_device_error.restype = i
    lib.pfa_wait_probe.argtypes = [vp]
    lib.pfa_wait_probe.restype = i
    if path is None:
        _LIB = lib
    return lib


def status_string(status: int) -> str:
    return load().pfa_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != PFA_OK:
        raise PfaError(status, where)


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _bhnd(t: torch.Tensor, name: str, dtype=torch.bfloat16, ndim=4) -> None:
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype or t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d {dtype} tensor")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def attn_fwd(q, k, v, o, lse, *, causal: bool, scale: float, fix_mode: int = 0,
             beta: float = 2.0, eps: float = 1e-3, counters=None, stream=None) -> None:
    """pfa_attn_fwd: O and lse of stabilised attention (see include/pfa.h)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _bhnd(t, n)
    _bhnd(lse, "lse", torch.float32, 3)
    if counters is not None:
        _bhnd(counters, "counters", torch.int64, 1)
        if counters.numel() != 3:
            raise ValueError("counters must hold 3 int64 values")
    B, Hq, N, d = q.shape
    st = load().pfa_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, k.shape[1], N,
                             d, int(bool(causal)), float(scale), int(fix_mode), float(beta),
                             float(eps), _ptr(counters) if counters is not None else None,
                             _stream(stream))
    _check(st, "pfa_attn_fwd")


def attn_delta(o, do, delta, *, stream=None) -> None:
    """pfa_attn_delta: delta = rowsum(dO o O)."""
    _bhnd(o, "o")
    _bhnd(do, "do")
    _bhnd(delta, "delta", torch.float32, 3)
    B, Hq, N, d = o.shape
    st = load().pfa_attn_delta(_ptr(o), _ptr(do), _ptr(delta), B, Hq, N, d, _stream(stream))
    _check(st, "pfa_attn_delta")


def attn_delta_alt(q, k, v, do, lse, delta, *, causal: bool, scale: float, stream=None) -> None:
    """pfa_attn_delta_alt: delta = rowsum(dP o P) with P, dP recomputed."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (do, "do")):
        _bhnd(t, n)
    _bhnd(lse, "lse", torch.float32, 3)
    _bhnd(delta, "delta", torch.float32, 3)
    B, Hq, N, d = q.shape
    st = load().pfa_attn_delta_alt(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse), _ptr(delta), B,
                                   Hq, k.shape[1], N, d, int(bool(causal)), float(scale),
                                   _stream(stream))
    _check(st, "pfa_attn_delta_alt")


def bwd_workspace_bytes(B: int, H_q: int, N: int, d: int) -> int:
    return int(load().pfa_bwd_workspace_bytes(B, H_q, N, d))


def attn_bwd(q, k, v, do, lse, delta, dq, dk, dv, dq_accum, *, causal: bool, scale: float,
             stream=None) -> None:
    """pfa_attn_bwd: dQ, dK, dV from lse and delta (dq_accum is the FP32 workspace)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (do, "do"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _bhnd(t, n)
    _bhnd(lse, "lse", torch.float32, 3)
    _bhnd(delta, "delta", torch.float32, 3)
    if dq_accum.device.type != "cuda" or dq_accum.dtype != torch.float32 or not dq_accum.is_contiguous():
        raise ValueError("dq_accum must be a contiguous float32 CUDA tensor")
    B, Hq, N, d = q.shape
    if dq_accum.numel() * 4 < bwd_workspace_bytes(B, Hq, N, d):
        raise ValueError("dq_accum is smaller than bwd_workspace_bytes()")
    st = load().pfa_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse), _ptr(delta), _ptr(dq),
                             _ptr(dk), _ptr(dv), _ptr(dq_accum), B, Hq, k.shape[1], N, d,
                             int(bool(causal)), float(scale), _stream(stream))
    _check(st, "pfa_attn_bwd")


def attn_bwd_accum(q, k, v, do, lse, delta, dq_accum, dk, dv, *, causal: bool, scale: float,
                   stream=None) -> None:
    """pfa_attn_bwd_accum: dq_accum (FP32 [B, H_q, N, d]) += alpha dS K; dk, dv written."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (do, "do"), (dk, "dk"), (dv, "dv")):
        _bhnd(t, n)
    _bhnd(lse, "lse", torch.float32, 3)
    _bhnd(delta, "delta", torch.float32, 3)
    _bhnd(dq_accum, "dq_accum", torch.float32)
    B, Hq, N, d = q.shape
    if dq_accum.shape != q.shape:
        raise ValueError("dq_accum must have the shape of q")
    st = load().pfa_attn_bwd_accum(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse), _ptr(delta),
                                   _ptr(dq_accum), _ptr(dk), _ptr(dv), B, Hq, k.shape[1], N, d,
                                   int(bool(causal)), float(scale), _stream(stream))
    _check(st, "pfa_attn_bwd_accum")


def attn_bwd_noalloc(q, k, v, do, lse, delta, dq, dk, dv, *, causal: bool, scale: float,
                     stream=None) -> None:
    """pfa_attn_bwd_noalloc: the backward pass without a caller workspace, for callers that
    may not allocate device memory; its dQ accumulation buffer is a fixed library-owned array
    (B * H_q * N * d <= 8,388,608), shared by all calls on a device."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (do, "do"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _bhnd(t, n)
    _bhnd(lse, "lse", torch.float32, 3)
    _bhnd(delta, "delta", torch.float32, 3)
    B, Hq, N, d = q.shape
    st = load().pfa_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse), _ptr(delta),
                                     _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, k.shape[1], N, d,
                                     int(bool(causal)), float(scale), _stream(stream))
    _check(st, "pfa_attn_bwd_noalloc")


def wait_probe(stream=None) -> None:
    """pfa_wait_probe: enqueue the bounded-wait self-test (sets PFA_DEVERR_TIMEOUT after
    about a second; see include/pfa.h)."""
    _check(load().pfa_wait_probe(_stream(stream)), "pfa_wait_probe")


def device_error(clear: bool = False) -> int:
    """pfa_device_error: the PFA_DEVERR_* bits of the current device (synchronises)."""
    st = load().pfa_device_error(int(bool(clear)))
    if st < 0:
        raise PfaError(st, "pfa_device_error")
    return st


def device_error_site() -> dict | None:
    """pfa_device_error_site, decoded: where the first timed-out wait was (None if none)."""
    w = int(load().pfa_device_error_site())
    if w < 0:
        raise PfaError(w, "pfa_device_error_site")
    if w == 0:
        return None
    return {"kernel": {1: "forward", 2: "backward", 3: "delta_alt", 4: "wait_probe"}.get((w >> 56) & 15, "?"),
            "drain": bool((w >> 55) & 1), "parity": (w >> 54) & 1,
            "barrier_offset": (w >> 32) & 0x3FFFFF, "block": w & 0xFFFFFFFF}
