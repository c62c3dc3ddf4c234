"""BF16 / FP32 rounding primitives of the CPU oracle.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this module;
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.

Sources (cited by page title and section):

* PK = priors.kr post "BF16 플래시 어텐션은 왜 수천 스텝 뒤에 무너질까"
  (a summary of Qiu & Yao, "Why Low-Precision Transformer Training Fails: An
  Analysis on Flash Attention", ICLR 2026).
* BN = bud-325 note "Why Low-Precision Transformer Training Fails: An Analysis
  on Flash Attention".

PK, "왜 중요한가" (paper §2.1): BF16 keeps 7 stored mantissa bits, so values in
[1, 2) are spaced 1/128 apart. PK, "핵심 아이디어" (paper App. B): every BF16
operation rounds to the nearest representable value, ties to the even one.
PK "비트 수준에서는" (paper §3.3.2) and BN "Results" walk through two additions
where the running sum is held wider than BF16 (a BF16 value plus a small
residual) and rounded once: that is :func:`bf16_sum` below.

Every function works on numpy arrays (or scalars) and returns float32 arrays
whose values are exactly representable in BF16 unless stated otherwise.
"""
from __future__ import annotations

import numpy as np

__all__ = ["fp32", "bf16_rne", "ftz32", "bf16_sum", "BF16_ONE_THRESHOLD", "e4m3_rne", "e2m1_rne",
           "mx_e2m1", "E4M3_MAX", "E2M1_MAX", "MX_BLOCK"]

# Smallest FP32 value x with bf16_rne(x) == 1.0: the midpoint between 1 - 2^-8
# (the largest BF16 value below 1) and 1.0. A tie there rounds to 1.0 because
# 1.0 has the even (zero) last mantissa bit.
BF16_ONE_THRESHOLD = 1.0 - 2.0 ** -9


def fp32(x) -> np.ndarray:
    """Round (float64) values to the nearest binary32 value (numpy's cast is RNE)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def bf16_rne(x) -> np.ndarray:
    """Round binary32 values to bfloat16, round-to-nearest, ties-to-even.

    Written from the IEEE 754 definition: bfloat16 is the upper half of the
    binary32 bit pattern. The lower 16 bits are dropped; if they exceed half an
    ulp the kept part is incremented, if they are exactly half the kept part is
    incremented only when its last bit is odd. Adding 0x7FFF plus that last bit
    and truncating does both at once; a carry out of the mantissa correctly
    bumps the exponent (and turns the largest finite values into inf). NaN is
    mapped to the canonical quiet NaN so that the carry cannot turn it into inf.
    """
    a = np.array(x, dtype=np.float32, copy=True)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    r = r.astype(np.uint32)
    r = np.where(np.isnan(a), np.uint32(0x7FC00000), r).astype(np.uint32)
    return r.view(np.float32)


def ftz32(x) -> np.ndarray:
    """Flush binary32 subnormals to (signed) zero, as a flush-to-zero FP32 unit does."""
    a = np.asarray(x, dtype=np.float32)
    tiny = np.abs(a) < np.float32(2.0 ** -126)
    return np.where(tiny & (a != 0), np.copysign(np.float32(0.0), a), a).astype(np.float32)


def bf16_sum(terms) -> np.float32:
    """Add ``terms`` left to right in FP32, then round the total once to BF16.

    This is the accumulation model of the worked traces in PK "비트 수준에서는"
    (paper §3.3.2) and BN "Results": the partial sum carries the residual of the
    earlier small terms in bits below BF16 precision (the sticky bits), and only
    the final value is rounded to BF16.
    """
    s = np.float32(0.0)
    for t in terms:
        s = np.float32(s + np.float32(t))
    return np.float32(bf16_rne(s).reshape(()))


# --------------------------------------------------------------------------------------
# Narrower formats, for the question PK "열린 질문" leaves open: what the bias looks like
# when fewer mantissa bits carry the summed values (FP8, MXFP4).
# --------------------------------------------------------------------------------------
E4M3_MAX = 448.0   # largest finite FP8 E4M3 value: 1.75 x 2^8
E2M1_MAX = 6.0     # largest FP4 E2M1 value: 1.5 x 2^2
MX_BLOCK = 32      # elements sharing one scale in the MX formats


def _round_grid(a, exp_min, mbits):
    """Round non-negative float64 ``a`` to a binary grid with ``mbits`` stored mantissa bits
    and smallest exponent ``exp_min`` (subnormals below 2^exp_min), nearest, ties to even."""
    a = np.asarray(a, dtype=np.float64)
    out = np.zeros_like(a)
    nz = a > 0
    e = np.floor(np.log2(np.where(nz, a, 1.0)))
    e = np.maximum(e, exp_min)
    ulp = np.exp2(e - mbits)
    q = a / ulp
    r = np.round(q)             # numpy rounds halves to even
    out = np.where(nz, r * ulp, 0.0)
    return out


def e4m3_rne(x) -> np.ndarray:
    """Round to FP8 E4M3 (4 exponent bits with bias 7, 3 stored mantissa bits, no
    infinities): nearest, ties to even; magnitudes beyond the largest finite value 448
    saturate to it; subnormals are 2^-9 apart below 2^-6. Returns float64 values."""
    x = np.asarray(x, dtype=np.float64)
    y = np.minimum(_round_grid(np.abs(x), -6, 3), E4M3_MAX)
    return np.where(np.isnan(x), np.nan, np.copysign(y, x))


def e2m1_rne(x) -> np.ndarray:
    """Round to FP4 E2M1 (2 exponent bits with bias 1, 1 stored mantissa bit): the values
    0, 0.5, 1, 1.5, 2, 3, 4, 6; nearest, ties to even; saturating at 6."""
    x = np.asarray(x, dtype=np.float64)
    y = np.minimum(_round_grid(np.abs(x), 0, 1), E2M1_MAX)
    return np.copysign(y, x)


def mx_e2m1(x, axis=-1) -> np.ndarray:
    """MXFP4: blocks of 32 consecutive elements along ``axis`` share a power-of-two scale
    X = 2^(floor(log2(amax)) - 2) (2 = the largest exponent of E2M1), and each element
    becomes X * E2M1(v / X) (saturating). A block of zeros stays zero. Returns float64."""
    x = np.moveaxis(np.asarray(x, dtype=np.float64), axis, -1)
    n = x.shape[-1]
    pad = (-n) % MX_BLOCK
    xp = np.concatenate([x, np.zeros(x.shape[:-1] + (pad,))], axis=-1)
    blocks = xp.reshape(x.shape[:-1] + (-1, MX_BLOCK))
    amax = np.abs(blocks).max(axis=-1, keepdims=True)
    scale = np.where(amax > 0, np.exp2(np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2), 1.0)
    q = e2m1_rne(blocks / scale) * scale
    out = q.reshape(xp.shape)[..., :n]
    return np.moveaxis(out, -1, axis)
