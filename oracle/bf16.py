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

__all__ = ["fp32", "bf16_rne", "ftz32", "bf16_sum", "BF16_ONE_THRESHOLD"]

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
