"""Plain CPU definition of stabilised BF16 attention, forward and backward.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. It shares no code,
constant or helper with the CUDA path, and it reads nothing the CUDA path
writes.

Sources (cited by page title and section):

* PK = priors.kr post "BF16 플래시 어텐션은 왜 수천 스텝 뒤에 무너질까"
  (a summary of Qiu & Yao, ICLR 2026).
* BN = bud-325 note "Why Low-Precision Transformer Training Fails: An Analysis
  on Flash Attention".

What is computed, per batch b and query head h (key/value head h // (H_q/H_kv)),
over whole rows with no tiling (tiling is not the cause of the failure, BN "Key
claims", paper §3.2):

1. S = alpha * Q K^T; with ``causal`` key j is visible to query i iff j <= i.
2. r_m = rowmax(S); a row is *repeated* iff at least two of its entries lie
   within ``eps`` of r_m (PK "처방은 그 조건만 피한다", paper §4).
3. Shift m per row (PK paper §4 equation; BN "Method", Algorithm 1):
   mode 0 m = r_m; mode 1 on repeated rows m = beta*r_m if r_m > 0, 0 if
   r_m < 0 (and 2^-5 if r_m == 0, a reading: the pages give no value there);
   mode 2 on repeated rows m = r_m + 2^-5; every other row keeps m = r_m.
4. Pbar = exp(S - m), l = rowsum(Pbar), Obar = Pbar V, O = Obar / l,
   lse = m + ln l (PK "수식", paper §2.2 / §3).
5. Backward (PK "수식", paper §3.3.1): P = exp(S - lse), dP = dO V^T,
   delta = rowsum(dO o O) (or rowsum(dP o P), PK "방법", paper §3.2),
   dS = alpha P o (dP - delta), dQ = dS K, dK = dS^T Q, dV = P^T dO, with dK
   and dV summed over the query heads that share a key/value head.

Two precisions:

* ``emulate_bf16=False``: everything in float64 (the parity reference).
* ``emulate_bf16=True``: the cast points of a fused BF16 kernel with FP32
  accumulation: each dot product is formed exactly and rounded once to FP32
  (an order-free stand-in for an FP32 accumulator); Pbar is computed in FP32,
  rounded to BF16 and flushed to zero below the FP32 normal range; l sums the
  FP32 Pbar (before its BF16 cast, which only the Pbar V product sees); O, dQ,
  dK, dV are rounded to BF16 at the end. In the backward pass P = exp(S - lse)
  is FP32 (flushed to zero below the normal range), dS = P o (dP - delta) is
  formed in FP32 and, like P, rounded to BF16 before the products it feeds;
  alpha multiplies the FP32 results of the dQ and dK products (so the BF16 dS
  does not carry it). The pages fix the equation dS = alpha P o (dP - delta)
  but no rounding points; these are the backward kernel's.

Diagnostic counters (per call, summed over all rows): ``repeated_rows`` =
number of repeated rows; ``ones`` = number of entries whose BF16 Pbar under
the row's final shift equals 1.0 (the condition the fix removes, PK
"핵심 아이디어"); ``nonfinite_rows`` = rows whose l is 0 or not finite (the
underflow the pages warn about, PK "의심해볼 점" and paper App. C).

All inputs are numpy arrays of shape [B, H, N, d] holding the BF16 input
values as float64 (any float64 values are accepted in float64 mode).
"""
from __future__ import annotations

import numpy as np

from .bf16 import bf16_rne, e4m3_rne, fp32, ftz32, mx_e2m1

__all__ = [
    "EPS_SHIFT",
    "scores",
    "visible",
    "fix_shift",
    "attn_fwd_head",
    "attn_fwd",
    "attn_delta",
    "attn_delta_alt",
    "attn_bwd",
    "attn_bwd_rows",
    "attn_fwd_monitor",
    "attn_fwd_unfused",
    "attn_fwd_blockwise",
    "TIE_BINS",
]

# Bins of the tie-multiplicity histogram: multiplicity 1..7, and 8 or more.
TIE_BINS = 8

# The extra shift 2^-5 of mode 2 (BN "Key claims" and "Method", Algorithm 1).
EPS_SHIFT = 2.0 ** -5


def scores(qh: np.ndarray, kh: np.ndarray, scale: float, emulate_bf16: bool) -> np.ndarray:
    """S = scale * qh kh^T for one head (qh [R, d], kh [N, d]) -> [R, N].

    float64 mode: products and sums in float64. Emulation: the BF16 products are
    exact in float64 and the float64 dot product is rounded once to FP32, then
    multiplied by the FP32 scale with one FP32 rounding.
    """
    s = qh @ kh.T
    if emulate_bf16:
        return (fp32(s) * np.float32(scale)).astype(np.float64)
    return scale * s


def visible(rows: np.ndarray, n_keys: int, causal: bool) -> np.ndarray:
    """Boolean [R, N] mask of the keys a query row may attend to (j <= i if causal)."""
    cols = np.arange(n_keys)[None, :]
    if causal:
        return cols <= np.asarray(rows)[:, None]
    return np.ones((len(rows), n_keys), dtype=bool)


def fix_shift(r_m: np.ndarray, repeated: np.ndarray, fix_mode: int, beta: float,
              emulate_bf16: bool) -> np.ndarray:
    """The safe-softmax shift m per row (PK paper §4 equation; BN Algorithm 1).

    Rows that are not repeated, and every row in mode 0, subtract r_m itself.
    Mode 1, repeated rows: beta * r_m if r_m > 0; 0 if r_m < 0; 2^-5 if r_m == 0
    (the pages name only the two signed cases; 2^-5 keeps the largest exponent
    argument strictly negative, which is what PK says the rule guarantees).
    Mode 2, repeated rows: r_m + 2^-5.
    """
    if fix_mode not in (0, 1, 2):
        raise ValueError("fix_mode must be 0, 1 or 2")
    r_m = np.asarray(r_m, dtype=np.float64)
    m = r_m.copy()
    if fix_mode == 1:
        pos = repeated & (r_m > 0)
        neg = repeated & (r_m < 0)
        zero = repeated & (r_m == 0)
        m[pos] = beta * r_m[pos]
        m[neg] = 0.0
        m[zero] = EPS_SHIFT
    elif fix_mode == 2:
        m[repeated] = r_m[repeated] + EPS_SHIFT
    if emulate_bf16:
        m = fp32(m).astype(np.float64)
    return m


def attn_fwd_head(qh, kh, vh, *, causal=False, scale=None, fix_mode=0, beta=2.0,
                  eps=1e-3, emulate_bf16=False, rows=None) -> dict:
    """Forward pass of one (batch, query head), optionally for a subset of query rows.

    Returns a dict with ``o`` [R, d], ``lse`` [R], the per-row ``r_m``, ``m``,
    ``repeated`` (bool), ``ones`` (int) and ``nonfinite`` (bool).
    """
    n_q, d = qh.shape
    n_k = kh.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.arange(n_q) if rows is None else np.asarray(rows, dtype=np.int64)
    s = scores(qh[rows], kh, scale, emulate_bf16)
    vis = visible(rows, n_k, causal)
    s = np.where(vis, s, -np.inf)

    r_m = s.max(axis=1)
    repeated = (s >= (r_m - eps)[:, None]).sum(axis=1) >= 2
    m = fix_shift(r_m, repeated, fix_mode, beta, emulate_bf16)

    x = s - m[:, None]
    if emulate_bf16:
        p32 = ftz32(np.exp(fp32(x))).astype(np.float64)     # Pbar in FP32
        pbar = ftz32(bf16_rne(p32)).astype(np.float64)      # its BF16 cast, the Pbar V operand
        pbar_bf16 = pbar
    else:
        p32 = pbar = np.exp(x)
        pbar_bf16 = bf16_rne(fp32(pbar)).astype(np.float64)
    ones = (pbar_bf16 == 1.0).sum(axis=1)

    # l is the row sum of Pbar itself (before its BF16 cast), so lse = m + ln l keeps FP32
    # accuracy and P = exp(S - lse) in the backward pass sums to one.
    l = p32.sum(axis=1)
    obar = pbar @ vh
    with np.errstate(divide="ignore", invalid="ignore"):
        if emulate_bf16:
            l32 = fp32(l)
            o = bf16_rne(fp32(obar) / l32[:, None]).astype(np.float64)
            lse = fp32(fp32(m) + fp32(np.log(l32.astype(np.float64)))).astype(np.float64)
            l = l32.astype(np.float64)
        else:
            o = obar / l[:, None]
            lse = m + np.log(l)
    nonfinite = (l == 0) | ~np.isfinite(l)
    return {"o": o, "lse": lse, "r_m": r_m, "m": m, "repeated": repeated,
            "ones": ones, "nonfinite": nonfinite}


def _check_shapes(q, k, v=None):
    if q.ndim != 4 or k.ndim != 4:
        raise ValueError("expected [B, H, N, d] arrays")
    B, Hq, N, d = q.shape
    if k.shape[0] != B or k.shape[2] != N or k.shape[3] != d:
        raise ValueError("q and k disagree in B, N or d")
    if Hq % k.shape[1] != 0:
        raise ValueError("H_q must be a multiple of H_kv")
    if v is not None and v.shape != k.shape:
        raise ValueError("k and v must have the same shape")
    return B, Hq, k.shape[1], N, d


def attn_fwd(q, k, v, *, causal=False, scale=None, fix_mode=0, beta=2.0, eps=1e-3,
             emulate_bf16=False) -> dict:
    """Forward pass over all heads: ``o`` [B,H_q,N,d], ``lse`` [B,H_q,N] and counters.

    Also returns the per-row ``repeated`` flags and shifts ``m`` ([B,H_q,N]) for
    diagnosis.
    """
    B, Hq, Hkv, N, d = _check_shapes(q, k, v)
    group = Hq // Hkv
    o = np.zeros(q.shape, dtype=np.float64)
    lse = np.zeros((B, Hq, N), dtype=np.float64)
    rep = np.zeros((B, Hq, N), dtype=bool)
    shift = np.zeros((B, Hq, N), dtype=np.float64)
    counters = {"repeated_rows": 0, "ones": 0, "nonfinite_rows": 0}
    for b in range(B):
        for h in range(Hq):
            r = attn_fwd_head(q[b, h], k[b, h // group], v[b, h // group], causal=causal,
                              scale=scale, fix_mode=fix_mode, beta=beta, eps=eps,
                              emulate_bf16=emulate_bf16)
            o[b, h], lse[b, h], rep[b, h], shift[b, h] = r["o"], r["lse"], r["repeated"], r["m"]
            counters["repeated_rows"] += int(r["repeated"].sum())
            counters["ones"] += int(r["ones"].sum())
            counters["nonfinite_rows"] += int(r["nonfinite"].sum())
    return {"o": o, "lse": lse, "repeated": rep, "m": shift, "counters": counters}


def attn_delta(o, do, *, emulate_bf16=False) -> np.ndarray:
    """delta = rowsum(dO o O) ([B,H,N]) -- the backward preprocessing term where
    the error enters (PK "3줄 요약" and "방법", paper §3.2; BN "Key claims").
    Emulation rounds the exact sum of BF16 products once to FP32."""
    d = (np.asarray(o, dtype=np.float64) * np.asarray(do, dtype=np.float64)).sum(axis=-1)
    return fp32(d).astype(np.float64) if emulate_bf16 else d


def _probs(qh, kh, lse_h, causal, scale, emulate_bf16):
    """P = exp(S - lse) for one head with invisible entries set to 0."""
    n = qh.shape[0]
    s = scores(qh, kh, scale, emulate_bf16)
    vis = visible(np.arange(n), kh.shape[0], causal)
    x = s - np.asarray(lse_h, dtype=np.float64)[:, None]
    if emulate_bf16:
        p = ftz32(np.exp(fp32(x))).astype(np.float64)
    else:
        p = np.exp(x)
    return np.where(vis, p, 0.0)


def attn_delta_alt(q, k, v, do, lse, *, causal=False, scale=None, emulate_bf16=False) -> np.ndarray:
    """delta = rowsum(dP o P) with P = exp(S - lse) and dP = dO V^T: the
    mathematically equal alternative that the paper found stable (PK "방법",
    paper §3.2; BN "Key claims")."""
    B, Hq, Hkv, N, d = _check_shapes(q, k, v)
    group = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((B, Hq, N), dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            kv = h // group
            p = _probs(q[b, h], k[b, kv], lse[b, h], causal, scale, emulate_bf16)
            dp = do[b, h] @ v[b, kv].T
            if emulate_bf16:
                dp = fp32(dp).astype(np.float64)
                out[b, h] = fp32((p * dp).sum(axis=1))
            else:
                out[b, h] = (p * dp).sum(axis=1)
    return out


def attn_bwd(q, k, v, do, lse, delta, *, causal=False, scale=None, emulate_bf16=False) -> dict:
    """dQ, dK, dV from the saved lse and the given delta (PK "수식", paper §3.3.1).

    dS = scale * P o (dP - delta); dQ = dS K; dK = sum over the query heads of a
    group of dS^T Q; dV = sum over the group of P^T dO. The fix does not enter:
    the backward pass is unchanged (PK paper §4; BN "Results").
    """
    B, Hq, Hkv, N, d = _check_shapes(q, k, v)
    group = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(v.shape, dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            kv = h // group
            p = _probs(q[b, h], k[b, kv], lse[b, h], causal, scale, emulate_bf16)
            dp = do[b, h] @ v[b, kv].T
            dlt = np.asarray(delta[b, h], dtype=np.float64)[:, None]
            if emulate_bf16:
                # P o (dP - delta) in FP32 and cast to BF16 as the dQ / dK operand; alpha
                # multiplies the FP32 products afterwards, where the kernel applies it.
                dp = fp32(dp).astype(np.float64)
                ds_op = bf16_rne(fp32(p * fp32(dp - dlt))).astype(np.float64)
                p_op = bf16_rne(fp32(p)).astype(np.float64)
            else:
                ds_op = scale * p * (dp - dlt)
                p_op = p
            dq[b, h] = ds_op @ k[b, kv]
            dk[b, kv] += ds_op.T @ q[b, h]
            dv[b, kv] += p_op.T @ do[b, h]
    if emulate_bf16:
        a32 = np.float32(scale)
        dq, dk = (bf16_rne(fp32(fp32(x) * a32)).astype(np.float64) for x in (dq, dk))
        dv = bf16_rne(fp32(dv)).astype(np.float64)
    return {"dq": dq, "dk": dk, "dv": dv}


def attn_bwd_rows(qh, kh, vh, doh, lse_rows, delta_rows, rows, *, causal=False, scale=None) -> np.ndarray:
    """dQ of selected query rows of one head in float64 (qh, doh [R, d] the rows themselves;
    kh, vh [N, d]; ``rows`` their indices, for the causal range): over the visible keys,
    P_i = exp(S_i - lse_i), dP_i = dO_i V^T, dS_i = scale P_i o (dP_i - delta_i), dQ_i = dS_i K
    (PK "수식", paper §3.3.1). The rows of :func:`attn_bwd`'s dQ, without forming the other
    rows: long sequences are checked on sampled rows."""
    d = qh.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.asarray(rows, dtype=np.int64)
    s = scale * (qh @ kh.T)
    vis = visible(rows, kh.shape[0], causal)
    p = np.where(vis, np.exp(s - np.asarray(lse_rows, dtype=np.float64)[:, None]), 0.0)
    dp = doh @ vh.T
    ds = scale * p * (dp - np.asarray(delta_rows, dtype=np.float64)[:, None])
    return ds @ kh


def attn_fwd_monitor(q, k, v, *, causal=False, scale=None, fix_mode=0, beta=2.0, eps=1e-3,
                     tile=128, emulate_bf16=True) -> dict:
    """The training-time monitor of a tiled forward pass (the repeated maxima that PK "결과"
    (paper App. E.1, Fig. 13) tracks, and two views of them):

    * ``operational_ones``: over every row and every ``tile``-key block of its visible keys,
      in order, the entries whose BF16 Pbar equals 1.0 under the shift in use for that block:
      the shift rule (:func:`fix_shift`) applied to the row's maximum over the keys up to the
      block's end, with the repetition flag of those same keys (at least two of them within
      ``eps`` of that maximum). These are the exact ones a tiled kernel hands to the Pbar V
      product; rows whose maximum rises later can carry ones that the final shift no longer
      has.
    * ``tie_hist``: rows by the multiplicity of their maximum, #{j : S_ij >= r_m - eps}, in
      bins 1..7 and >= 8 (index multiplicity - 1, capped at 7).

    Scores, exponentials and the BF16 cast as in :func:`attn_fwd_head` (``emulate_bf16``
    selects FP32 scores and an FP32 exponential)."""
    B, Hq, Hkv, N, d = _check_shapes(q, k, v)
    group = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    ones = 0
    hist = np.zeros(TIE_BINS, dtype=np.int64)
    rows = np.arange(N)
    vis = visible(rows, N, causal)
    for b in range(B):
        for h in range(Hq):
            s = np.where(vis, scores(q[b, h], k[b, h // group], scale, emulate_bf16), -np.inf)
            r_m = s.max(axis=1)
            mult = (s >= (r_m - eps)[:, None]).sum(axis=1)
            hist += np.bincount(np.minimum(mult, TIE_BINS) - 1, minlength=TIE_BINS)
            for j0 in range(0, N, tile):
                seen = s[:, : j0 + tile]
                m1 = seen.max(axis=1)
                live = np.isfinite(m1)
                rep = (seen >= (m1 - eps)[:, None]).sum(axis=1) >= 2
                m = fix_shift(np.where(live, m1, 0.0), rep, fix_mode, beta, emulate_bf16)
                x = s[:, j0: j0 + tile] - m[:, None]
                if emulate_bf16:
                    pbar = ftz32(np.exp(fp32(x)))
                else:
                    pbar = fp32(np.exp(x))
                ones += int(((bf16_rne(pbar) == 1.0) & live[:, None]).sum())
    return {"operational_ones": ones, "tie_hist": hist}


def attn_fwd_unfused(q, k, v, *, causal=False, scale=None, fix_mode=0, beta=2.0, eps=1e-3,
                     block=512) -> dict:
    """The forward pass as an implementation that stores the unnormalised product Pbar V in
    BF16 computes it: the paper's analysed code, FlashAttention 2 written as PyTorch
    operations with blocks of 512 keys (PK "의심해볼 점"; the bias mechanism of PK
    "핵심 아이디어", paper §3.3.2, and BN "Results", Fig. 6). :func:`attn_fwd_blockwise`
    with a BF16 Pbar and BF16 accumulation."""
    return attn_fwd_blockwise(q, k, v, causal=causal, scale=scale, fix_mode=fix_mode, beta=beta,
                              eps=eps, block=block, pbar="bf16", accumulate="bf16")


def _round_pbar(p32, pbar):
    """The Pbar operand: BF16, FP8 E4M3, or MXFP4 (E2M1 with one power-of-two scale per 32
    consecutive keys, :func:`oracle.bf16.mx_e2m1`), from the FP32 Pbar of one key block."""
    if pbar == "bf16":
        return ftz32(bf16_rne(p32)).astype(np.float64)
    if pbar == "e4m3":
        return e4m3_rne(p32)
    if pbar == "mxfp4":
        return mx_e2m1(p32, axis=-1)
    raise ValueError("pbar must be 'bf16', 'e4m3' or 'mxfp4'")


def attn_fwd_blockwise(q, k, v, *, causal=False, scale=None, fix_mode=0, beta=2.0, eps=1e-3,
                       block=128, pbar="bf16", accumulate="bf16") -> dict:
    """Blockwise online softmax with a chosen Pbar format and Obar precision.

    Per row, per ``block`` of keys in order: the running maximum and the repetition flag of
    the keys so far give the shift m_b (:func:`fix_shift`); Pbar = ``pbar``(exp(S - m_b)) from
    an FP32 exponential (flushed to zero below the normal range); the block's product
    U_b = sum_j Pbar_j V_j is formed exactly and, with ``accumulate="bf16"``, rounded once to
    BF16 (an FP32-accumulating matrix product with a BF16 result, the accumulation model of
    the pages' worked traces, :func:`oracle.bf16.bf16_sum`) and accumulated as
    Obar = BF16(BF16(Obar * c_b) + U_b); with ``accumulate="fp32"``, Obar = FP32(Obar * c_b +
    U_b). c_b = exp(m_(b-1) - m_b) in FP32. l = FP32(l * c_b + sum of the rounded Pbar): the
    normaliser sums the weights the product used (a reading: the pages name only P V as
    stored in BF16). Finally O = BF16(Obar / l) and lse = m + ln l (FP32). Scores are FP32 (one
    rounding of the exact dot, times FP32 alpha).

    ``pbar`` "e4m3" and "mxfp4" are the narrower formats whose effect the pages leave open
    (PK "열린 질문"). Returns ``o``, ``lse``, ``obar`` (the accumulator before normalisation)
    and ``operational_ones`` (rounded Pbar entries equal to 1.0 handed to the products)."""
    B, Hq, Hkv, N, d = _check_shapes(q, k, v)
    if accumulate not in ("bf16", "fp32"):
        raise ValueError("accumulate must be 'bf16' or 'fp32'")
    group = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.arange(N)
    vis = visible(rows, N, causal)
    o = np.zeros(q.shape)
    obar_all = np.zeros(q.shape)
    lse = np.zeros((B, Hq, N))
    ones = 0
    for b in range(B):
        for h in range(Hq):
            kv = h // group
            s = np.where(vis, scores(q[b, h], k[b, kv], scale, True), -np.inf)
            m_prev = np.full(N, -np.inf)
            l = np.zeros(N)
            obar = np.zeros((N, d))
            for j0 in range(0, N, block):
                seen = s[:, : j0 + block]
                m1 = seen.max(axis=1)
                live = np.isfinite(m1)
                rep = (seen >= (m1 - eps)[:, None]).sum(axis=1) >= 2
                m = np.where(live, fix_shift(np.where(live, m1, 0.0), rep, fix_mode, beta, True),
                             -np.inf)
                with np.errstate(invalid="ignore"):
                    c = np.where(np.isfinite(m_prev), ftz32(np.exp(fp32(m_prev - m))), 0.0)
                with np.errstate(invalid="ignore"):
                    x = np.where(live[:, None], s[:, j0: j0 + block] - m[:, None], -np.inf)
                p = _round_pbar(ftz32(np.exp(fp32(x))), pbar)
                ones += int((p == 1.0).sum())
                l = fp32(l.astype(np.float64) * c + p.astype(np.float64).sum(axis=1))
                prod = p.astype(np.float64) @ v[b, kv, j0: j0 + block]
                if accumulate == "bf16":
                    u = bf16_rne(fp32(prod))
                    scaled = bf16_rne(fp32(obar.astype(np.float64) * c[:, None]))
                    obar = bf16_rne(fp32(scaled.astype(np.float64) + u.astype(np.float64)))
                else:
                    obar = fp32(obar.astype(np.float64) * c[:, None] + prod)
                m_prev = m
            with np.errstate(divide="ignore", invalid="ignore"):
                o[b, h] = bf16_rne(fp32(obar.astype(np.float64) / l.astype(np.float64)[:, None]))
                lse[b, h] = fp32(fp32(m_prev) + fp32(np.log(l.astype(np.float64))))
            obar_all[b, h] = obar
    return {"o": o, "lse": lse, "obar": obar_all, "operational_ones": ones}
