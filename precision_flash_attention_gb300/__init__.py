"""Stabilised BF16 flash attention (forward and backward) for one GB300 GPU.

The compute path is libpfa (hand-written sm_103a kernels behind the C ABI in
``include/pfa.h``); this package is its thin Python binding plus convenience
wrappers that allocate outputs with torch. There is no CPU or PyTorch fallback:
calls fail if libpfa has not been built or no sm_103 device is current.

The method is from Qiu & Yao, "Why Low-Precision Transformer Training Fails: An
Analysis on Flash Attention" (ICLR 2026): rows whose maximum score repeats get a
different softmax shift so that no BF16 exp(S - m) rounds to exactly 1.
"""
from __future__ import annotations

import math

import torch

from ._lib import (BWD_DQ_DETERMINISTIC, BWD_DQ_SPLIT, BWD_WORKSPACE_ZEROED, EXPORTS, FWD_PAIR_CTA, FWD_PBAR_E4M3,
                   FWD_PBAR_MXFP4, FWD_UNFUSED_BF16_PV, MONITOR_WORDS,
                   TIE_BINS, PfaError, attn_bwd, attn_bwd_accum, attn_bwd_ex, attn_bwd_noalloc,
                   attn_delta, attn_delta_alt, attn_delta_zero, attn_fwd, attn_fwd_ex, bwd_workspace_bytes,
                   device_error, device_error_site, load, status_string, wait_probe)

__all__ = [
    "BWD_DQ_DETERMINISTIC", "BWD_DQ_SPLIT", "BWD_WORKSPACE_ZEROED", "EXPORTS", "FWD_PAIR_CTA", "FWD_PBAR_E4M3",
    "FWD_PBAR_MXFP4",
    "FWD_UNFUSED_BF16_PV", "MONITOR_WORDS",
    "TIE_BINS", "PfaError", "attn_fwd", "attn_fwd_ex", "attn_delta", "attn_delta_zero",
    "attn_delta_alt", "attn_bwd", "attn_bwd_accum", "attn_bwd_ex", "attn_bwd_noalloc",
    "bwd_workspace_bytes", "device_error", "device_error_site", "load", "status_string", "wait_probe",
    "forward", "backward",
    "StabilizedAttention", "new_counters", "new_monitor",
]


def new_counters(device="cuda") -> torch.Tensor:
    """A zeroed int64[3] device buffer for (repeated_rows, ones, nonfinite_rows)."""
    return torch.zeros(3, dtype=torch.int64, device=device)


def new_monitor(device="cuda") -> torch.Tensor:
    """A zeroed int64[9] device buffer for the forward monitor: operational ones, then the
    tie-multiplicity histogram (multiplicity 1..7, >= 8)."""
    return torch.zeros(MONITOR_WORDS, dtype=torch.int64, device=device)


PBAR_FLAGS = {"bf16": 0, "e4m3": FWD_PBAR_E4M3, "mxfp4": FWD_PBAR_MXFP4}


def forward(q, k, v, *, causal=False, scale=None, fix_mode=0, beta=2.0, eps=1e-3, counters=None,
            monitor=None, unfused_bf16_pv=False, pbar="bf16", pair_cta=False, stream=None):
    """Allocate O and lse and run the forward pass (pfa_attn_fwd, or pfa_attn_fwd_ex with a
    monitor, the unfused BF16 study profile, a narrower Pbar format: ``pbar`` "e4m3" or
    "mxfp4", or ``pair_cta``: at d = 128 two CTAs share each product). Returns (o, lse)."""
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    flags = (FWD_UNFUSED_BF16_PV if unfused_bf16_pv else 0) | PBAR_FLAGS[pbar] | (FWD_PAIR_CTA if pair_cta else 0)
    if monitor is None and not flags:
        attn_fwd(q, k, v, o, lse, causal=causal, scale=scale, fix_mode=fix_mode, beta=beta, eps=eps,
                 counters=counters, stream=stream)
    else:
        attn_fwd_ex(q, k, v, o, lse, causal=causal, scale=scale, fix_mode=fix_mode, beta=beta,
                    eps=eps, counters=counters, monitor=monitor, flags=flags, stream=stream)
    return o, lse


DQ_MODES = {"atomic": 0, "deterministic": BWD_DQ_DETERMINISTIC,
            "split": BWD_DQ_DETERMINISTIC | BWD_DQ_SPLIT}


def backward(q, k, v, o, lse, do, *, causal=False, scale=None, delta_mode=0, dq_mode="atomic",
             stream=None, workspace=None):
    """delta (rowsum(dO o O), or rowsum(dP o P) with ``delta_mode=1``) then the backward pass.

    ``dq_mode``: "atomic" (pfa_attn_bwd: per-key-tile dQ sums reduce-added into an FP32
    workspace), "deterministic" (the query-outer dQ pass) or "split" (the query-outer pass
    with dS as a BF16 hi + lo pair). With "atomic" at d = 64 and delta = rowsum(dO o O), the
    delta pass also zeroes the workspace (pfa_attn_delta_zero) and the backward call skips
    its own zeroing pass. Returns (dq, dk, dv, delta)."""
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else scale
    flags = DQ_MODES[dq_mode]
    B, H, N, d = q.shape
    delta = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    fused_zero = flags == 0 and delta_mode == 0 and d == 64
    if flags == 0 and workspace is None:
        workspace = torch.empty(bwd_workspace_bytes(B, H, N, d) // 4, dtype=torch.float32,
                                device=q.device)
    if delta_mode == 0:
        if fused_zero:
            attn_delta_zero(o, do, delta, workspace, stream=stream)
        else:
            attn_delta(o, do, delta, stream=stream)
    else:
        attn_delta_alt(q, k, v, do, lse, delta, causal=causal, scale=scale, stream=stream)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if flags:
        attn_bwd_ex(q, k, v, do, lse, delta, dq, dk, dv, None, causal=causal, scale=scale,
                    flags=flags, stream=stream)
        return dq, dk, dv, delta
    attn_bwd(q, k, v, do, lse, delta, dq, dk, dv, workspace, causal=causal, scale=scale,
             stream=stream, workspace_zeroed=fused_zero)
    return dq, dk, dv, delta


class StabilizedAttention(torch.autograd.Function):
    """Autograd wrapper: ``StabilizedAttention.apply(q, k, v, causal, scale, fix_mode, beta, eps)``."""

    @staticmethod
    def forward(ctx, q, k, v, causal=False, scale=None, fix_mode=0, beta=2.0, eps=1e-3):
        o, lse = forward(q, k, v, causal=causal, scale=scale, fix_mode=fix_mode, beta=beta, eps=eps)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.scale = causal, scale
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv, _ = backward(q, k, v, o, lse, do.contiguous(), causal=ctx.causal,
                                 scale=ctx.scale)
        return dq, dk, dv, None, None, None, None, None
