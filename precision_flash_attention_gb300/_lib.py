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
# pfa_attn_fwd_ex flags and the monitor's size (include/pfa.h)
FWD_UNFUSED_BF16_PV = 1
FWD_PBAR_E4M3 = 2
FWD_PBAR_MXFP4 = 4
FWD_PAIR_CTA = 8
TIE_BINS = 8
MONITOR_WORDS = 1 + TIE_BINS
# bits of the device error word (pfa_device_error)
DEVERR_TIMEOUT = 1
DEVERR_SMEM_ALIGN = 2
# pfa_attn_bwd_ex flags (include/pfa.h)
BWD_DQ_DETERMINISTIC = 1
BWD_DQ_SPLIT = 2
BWD_WORKSPACE_ZEROED = 4
STATUS_NAMES = {0: "PFA_OK", -1: "PFA_ERR_INVALID_ARG", -2: "PFA_ERR_MISALIGNED",
                -3: "PFA_ERR_UNSUPPORTED", -4: "PFA_ERR_LAUNCH", -5: "PFA_ERR_DEVICE",
                -6: "PFA_ERR_TOO_LARGE"}

# Every entry point declared in include/pfa.h.
EXPORTS = ("pfa_attn_fwd", "pfa_attn_fwd_ex", "pfa_attn_delta", "pfa_attn_delta_zero", "pfa_attn_delta_alt", "pfa_attn_bwd",
           "pfa_attn_bwd_accum", "pfa_attn_bwd_ex", "pfa_attn_bwd_noalloc", "pfa_bwd_workspace_bytes", "pfa_status_string",
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
    lib.pfa_attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, f, f, vp, vp,
                                    ctypes.c_uint, vp]
    lib.pfa_attn_fwd_ex.restype = i
    lib.pfa_attn_delta.argtypes = [vp, vp, vp, i, i, i, i, vp]
    lib.pfa_attn_delta.restype = i
    lib.pfa_attn_delta_zero.argtypes = [vp, vp, vp, vp, i, i, i, i, vp]
    lib.pfa_attn_delta_zero.restype = i
    lib.pfa_attn_delta_alt.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.pfa_attn_delta_alt.restype = i
    lib.pfa_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.pfa_attn_bwd.restype = i
    lib.pfa_attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.pfa_attn_bwd_accum.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.pfa_attn_bwd_accum.restype = i
    lib.pfa_attn_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f,
                                    ctypes.c_uint, vp]
    lib.pfa_attn_bwd_ex.restype = i
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


def _layout(t, name: str, dtype=torch.bfloat16, ndim=4) -> None:
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch tensor")
    if t.dtype != dtype or t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d {dtype} tensor")


def _dims(q, k) -> tuple:
    """(B, H_q, H_kv, N, d) from q [B, H_q, N, d] and k [B, H_kv, N, d]."""
    B, Hq, N, d = q.shape
    if k.shape[0] != B or k.shape[2] != N or k.shape[3] != d:
        raise ValueError(f"k has shape {tuple(k.shape)}: expected [B, H_kv, N, d] with q's "
                         f"B={B}, N={N}, d={d}")
    Hkv = k.shape[1]
    if Hkv < 1 or Hq % Hkv != 0:
        raise ValueError(f"H_q={Hq} must be a multiple of H_kv={Hkv}")
    return B, Hq, Hkv, N, d


def _expect(t, name: str, shape) -> None:
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _on_device(*named) -> None:
    """Every tensor is a CUDA tensor on the current device (the one the call launches on)."""
    for t, name in named:
        if t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor")
    cur = torch.cuda.current_device()
    for t, name in named:
        if t.device.index != cur:
            raise ValueError(f"{name} is on cuda:{t.device.index}, but the current device is "
                             f"cuda:{cur}")


def _check_qkv(q, k, v, extra_q=(), extra_k=(), rows=(), also=()) -> tuple:
    """Layout, shape and device checks shared by the wrappers: q-shaped and k-shaped BF16
    tensors, [B, H_q, N] FP32 row tensors, and ``also``: (tensor, name) pairs whose own
    layout and shape the caller has checked, included in the device check. Raises
    ValueError before anything is launched; shapes are checked before devices."""
    named_q = [(q, "q")] + list(extra_q)
    named_k = [(k, "k"), (v, "v")] + list(extra_k)
    for t, n in named_q + named_k:
        _layout(t, n)
    for t, n in rows:
        _layout(t, n, torch.float32, 3)
    B, Hq, Hkv, N, d = _dims(q, k)
    for t, n in named_q:
        _expect(t, n, (B, Hq, N, d))
    for t, n in named_k:
        _expect(t, n, (B, Hkv, N, d))
    for t, n in rows:
        _expect(t, n, (B, Hq, N))
    _on_device(*(named_q + named_k + list(rows) + list(also)))
    return B, Hq, Hkv, N, d


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def attn_fwd(q, k, v, o, lse, *, causal: bool, scale: float, fix_mode: int = 0,
             beta: float = 2.0, eps: float = 1e-3, counters=None, stream=None) -> None:
    """pfa_attn_fwd: O and lse of stabilised attention (see include/pfa.h)."""
    also = []
    if counters is not None:
        _layout(counters, "counters", torch.int64, 1)
        if counters.numel() != 3:
            raise ValueError("counters must hold 3 int64 values")
        also = [(counters, "counters")]
    B, Hq, Hkv, N, d = _check_qkv(q, k, v, extra_q=[(o, "o")], rows=[(lse, "lse")], also=also)
    st = load().pfa_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N,
                             d, int(bool(causal)), float(scale), int(fix_mode), float(beta),
                             float(eps), _ptr(counters) if counters is not None else None,
                             _stream(stream))
    _check(st, "pfa_attn_fwd")


def attn_fwd_ex(q, k, v, o, lse, *, causal: bool, scale: float, fix_mode: int = 0,
                beta: float = 2.0, eps: float = 1e-3, counters=None, monitor=None, flags: int = 0,
                stream=None) -> None:
    """pfa_attn_fwd_ex: pfa_attn_fwd with the monitor (int64[9]: operational ones, then the
    8-bin tie-multiplicity histogram) and options (FWD_UNFUSED_BF16_PV, FWD_PBAR_E4M3,
    FWD_PBAR_MXFP4, FWD_PAIR_CTA)."""
    also = []
    for t, n, words in ((counters, "counters", 3), (monitor, "monitor", MONITOR_WORDS)):
        if t is not None:
            _layout(t, n, torch.int64, 1)
            if t.numel() != words:
                raise ValueError(f"{n} must hold {words} int64 values")
            also.append((t, n))
    B, Hq, Hkv, N, d = _check_qkv(q, k, v, extra_q=[(o, "o")], rows=[(lse, "lse")], also=also)
    st = load().pfa_attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d,
                                int(bool(causal)), float(scale), int(fix_mode), float(beta),
                                float(eps), _ptr(counters) if counters is not None else None,
                                _ptr(monitor) if monitor is not None else None, int(flags),
                                _stream(stream))
    _check(st, "pfa_attn_fwd_ex")


def attn_delta(o, do, delta, *, stream=None) -> None:
    """pfa_attn_delta: delta = rowsum(dO o O)."""
    _layout(o, "o")
    _layout(do, "do")
    _layout(delta, "delta", torch.float32, 3)
    B, Hq, N, d = o.shape
    _expect(do, "do", o.shape)
    _expect(delta, "delta", (B, Hq, N))
    _on_device((o, "o"), (do, "do"), (delta, "delta"))
    st = load().pfa_attn_delta(_ptr(o), _ptr(do), _ptr(delta), B, Hq, N, d, _stream(stream))
    _check(st, "pfa_attn_delta")


def attn_delta_zero(o, do, delta, dq_accum, *, stream=None) -> None:
    """pfa_attn_delta_zero: delta = rowsum(dO o O), and the first B*H_q*N*d values of the
    FP32 dQ workspace ``dq_accum`` zeroed in the same pass (then attn_bwd may skip its
    zeroing pass: ``workspace_zeroed=True``)."""
    _layout(o, "o")
    _layout(do, "do")
    _layout(delta, "delta", torch.float32, 3)
    B, Hq, N, d = o.shape
    _expect(do, "do", o.shape)
    _expect(delta, "delta", (B, Hq, N))
    if (not isinstance(dq_accum, torch.Tensor) or dq_accum.dtype != torch.float32
            or not dq_accum.is_contiguous()):
        raise ValueError("dq_accum must be a contiguous float32 tensor")
    if dq_accum.numel() < o.numel():
        raise ValueError("dq_accum is smaller than B*H_q*N*d values")
    _on_device((o, "o"), (do, "do"), (delta, "delta"), (dq_accum, "dq_accum"))
    st = load().pfa_attn_delta_zero(_ptr(o), _ptr(do), _ptr(delta), _ptr(dq_accum), B, Hq, N, d,
                                    _stream(stream))
    _check(st, "pfa_attn_delta_zero")


def attn_delta_alt(q, k, v, do, lse, delta, *, causal: bool, scale: float, stream=None) -> None:
    """pfa_attn_delta_alt: delta = rowsum(dP o P) with P, dP recomputed."""
    B, Hq, Hkv, N, d = _check_qkv(q, k, v, extra_q=[(do, "do")],
                                  rows=[(lse, "lse"), (delta, "delta")])
    st = load().pfa_attn_delta_alt(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse), _ptr(delta), B,
                                   Hq, Hkv, N, d, int(bool(causal)), float(scale),
                                   _stream(stream))
    _check(st, "pfa_attn_delta_alt")


def bwd_workspace_bytes(B: int, H_q: int, N: int, d: int) -> int:
    return int(load().pfa_bwd_workspace_bytes(B, H_q, N, d))


def attn_bwd(q, k, v, do, lse, delta, dq, dk, dv, dq_accum, *, causal: bool, scale: float,
             stream=None, workspace_zeroed: bool = False) -> None:
    """pfa_attn_bwd: dQ, dK, dV from lse and delta (dq_accum is the FP32 workspace).
    ``workspace_zeroed`` (pfa_attn_bwd_ex with BWD_WORKSPACE_ZEROED): the caller vouches that
    the workspace holds zeros (attn_delta_zero on the same stream), and the zeroing pass is
    skipped."""
    if (not isinstance(dq_accum, torch.Tensor) or dq_accum.dtype != torch.float32
            or not dq_accum.is_contiguous()):
        raise ValueError("dq_accum must be a contiguous float32 tensor")
    if q.dim() == 4 and dq_accum.numel() < q.numel():
        raise ValueError("dq_accum is smaller than bwd_workspace_bytes()")
    B, Hq, Hkv, N, d = _check_qkv(q, k, v, extra_q=[(do, "do"), (dq, "dq")],
                                  extra_k=[(dk, "dk"), (dv, "dv")],
                                  rows=[(lse, "lse"), (delta, "delta")], also=[(dq_accum, "dq_accum")])
    if workspace_zeroed:
        st = load().pfa_attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse), _ptr(delta),
                                    _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dq_accum), B, Hq, Hkv, N, d,
                                    int(bool(causal)), float(scale), BWD_WORKSPACE_ZEROED,
                                    _stream(stream))
        _check(st, "pfa_attn_bwd_ex")
        return
    st = load().pfa_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse), _ptr(delta), _ptr(dq),
                             _ptr(dk), _ptr(dv), _ptr(dq_accum), B, Hq, Hkv, N, d,
                             int(bool(causal)), float(scale), _stream(stream))
    _check(st, "pfa_attn_bwd")


def attn_bwd_ex(q, k, v, do, lse, delta, dq, dk, dv, dq_accum, *, causal: bool, scale: float,
                flags: int = 0, stream=None) -> None:
    """pfa_attn_bwd_ex: pfa_attn_bwd with options. ``flags`` 0 is attn_bwd (dq_accum the FP32
    workspace); BWD_DQ_DETERMINISTIC and/or BWD_DQ_SPLIT compute dQ by the query-outer pass
    (dq_accum unused, may be None)."""
    known = BWD_DQ_DETERMINISTIC | BWD_DQ_SPLIT | BWD_WORKSPACE_ZEROED
    if (flags & ~known) == 0 and (flags & (BWD_DQ_DETERMINISTIC | BWD_DQ_SPLIT)) == 0:
        attn_bwd(q, k, v, do, lse, delta, dq, dk, dv, dq_accum, causal=causal, scale=scale,
                 stream=stream, workspace_zeroed=bool(flags & BWD_WORKSPACE_ZEROED))
        return
    # The query-outer pass needs no workspace (unknown flag bits are the library's to refuse).
    B, Hq, Hkv, N, d = _check_qkv(q, k, v, extra_q=[(do, "do"), (dq, "dq")],
                                  extra_k=[(dk, "dk"), (dv, "dv")],
                                  rows=[(lse, "lse"), (delta, "delta")])
    st = load().pfa_attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse), _ptr(delta),
                                _ptr(dq), _ptr(dk), _ptr(dv), None, B, Hq, Hkv, N, d,
                                int(bool(causal)), float(scale), int(flags), _stream(stream))
    _check(st, "pfa_attn_bwd_ex")


def attn_bwd_accum(q, k, v, do, lse, delta, dq_accum, dk, dv, *, causal: bool, scale: float,
                   stream=None) -> None:
    """pfa_attn_bwd_accum: dq_accum (FP32 [B, H_q, N, d]) += dS K; dk, dv written."""
    _layout(dq_accum, "dq_accum", torch.float32)
    _layout(q, "q")
    _expect(dq_accum, "dq_accum", q.shape)
    B, Hq, Hkv, N, d = _check_qkv(q, k, v, extra_q=[(do, "do")], extra_k=[(dk, "dk"), (dv, "dv")],
                                  rows=[(lse, "lse"), (delta, "delta")], also=[(dq_accum, "dq_accum")])
    st = load().pfa_attn_bwd_accum(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse), _ptr(delta),
                                   _ptr(dq_accum), _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d,
                                   int(bool(causal)), float(scale), _stream(stream))
    _check(st, "pfa_attn_bwd_accum")


def attn_bwd_noalloc(q, k, v, do, lse, delta, dq, dk, dv, *, causal: bool, scale: float,
                     stream=None) -> None:
    """pfa_attn_bwd_noalloc: the backward pass without a caller workspace, for callers that
    may not allocate device memory; its dQ accumulation buffer is a fixed library-owned array
    (B * H_q * N * d <= 8,388,608), shared by all calls on a device."""
    B, Hq, Hkv, N, d = _check_qkv(q, k, v, extra_q=[(do, "do"), (dq, "dq")],
                                  extra_k=[(dk, "dk"), (dv, "dv")],
                                  rows=[(lse, "lse"), (delta, "delta")])
    st = load().pfa_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse), _ptr(delta),
                                     _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d,
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
    return {"kernel": {1: "forward", 2: "backward", 3: "delta_alt", 4: "wait_probe",
                       5: "dq_pass"}.get((w >> 56) & 15, "?"),
            "drain": bool((w >> 55) & 1), "parity": (w >> 54) & 1,
            "barrier_offset": (w >> 32) & 0x3FFFFF, "block": w & 0xFFFFFFFF}
