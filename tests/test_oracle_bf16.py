"""Pins of the oracle's BF16 primitives against the pages' worked traces and a library cast."""
import math
import os

import numpy as np

import oracle
import pytest
import torch

from oracle import BF16_ONE_THRESHOLD, bf16_rne, bf16_sum, ftz32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "bf16_traces.txt")


def _traces():
    rows = []
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, r, b, rounded, true, src = line.split()
            rows.append((float(a), float(r), float(b), float(rounded), float(true), src))
    return rows


@pytest.mark.parametrize("trace", _traces(), ids=lambda t: t[5])
def test_worked_traces_bit_exact(trace):
    # Priors.kr core idea (paper §3.3.2) and bud-325 Results: the sum of a BF16 partial sum
    # carrying a small residual and another BF16 value rounds away from zero to `rounded`.
    a, r, b, rounded, true, _ = trace
    for x in (a, b, rounded):
        assert bf16_rne(np.float32(x)) == np.float32(x), "printed operands are BF16 values"
    got = bf16_sum([a, r, b])
    assert got == np.float32(rounded)
    # The printed true value is the exact sum (truncated when printed).
    assert abs((a + r + b) - true) < 1e-5


def test_trace1_error_magnitude():
    # Priors.kr: the error of trace 1 is about -0.0148 (computed minus true): the sticky
    # residual turns the tie into a rounding away from zero, towards the operands' sign.
    err = float(bf16_sum([-2.40625, -0.00087, -2.296875])) - (-2.40625 - 0.00087 - 2.296875)
    assert abs(err - (-0.0148)) < 1e-4


def test_trace2_error_magnitude():
    # bud-325 Results: |error| of trace 2 is about 0.000488 (= 2^-11). The note prints it as a
    # negative error (true minus computed); only the value and the magnitude are pinned.
    err = float(bf16_sum([-0.85546875, -2.0 ** -11, -0.0859375])) - (-0.94189453125)
    assert abs(abs(err) - 2.0 ** -11) < 1e-9


def test_no_residual_rounds_to_even():
    # Without the residual the same addition is an exact tie and goes to the even neighbour:
    # the small, opposite-sign error case of the priors.kr bit-level paragraph.
    assert bf16_sum([-2.40625, -2.296875]) == np.float32(-4.6875)


def test_rounding_after_every_add_does_not_reproduce_trace1():
    # The pages' model keeps the residual in wider bits; rounding the partial sum to BF16 after
    # every addition loses it and yields the tie-to-even value instead.
    s = np.float32(0.0)
    for t in (-2.40625, -0.00087, -2.296875):
        s = bf16_rne(np.float32(s + np.float32(t)))
    assert s == np.float32(-4.6875)


def test_spacing_and_ties():
    # Priors.kr "왜 중요한가" (paper §2.1): BF16 spacing in [1, 2) is 1/128.
    assert bf16_rne(np.float32(1 + 1 / 128)) == np.float32(1 + 1 / 128)
    assert bf16_rne(np.float32(1 + 1 / 256)) == np.float32(1.0)          # tie -> even (1.0)
    assert bf16_rne(np.float32(1 + 3 / 256)) == np.float32(1 + 2 / 128)  # tie -> even
    assert bf16_rne(np.float32(1 + 1 / 256 + 2 ** -20)) == np.float32(1 + 1 / 128)


def test_round_to_one_threshold():
    # BF16(exp(x)) == 1.0 exactly when exp(x) >= 1 - 2^-9 (the tie goes to 1.0).
    t = np.float32(BF16_ONE_THRESHOLD)
    assert bf16_rne(t) == np.float32(1.0)
    assert bf16_rne(np.nextafter(t, np.float32(0))) == np.float32(1.0 - 2.0 ** -8)
    # The mode-2 shift 2^-5 keeps the maximum strictly below 1 (bud-325, Method).
    assert bf16_rne(np.float32(math.exp(-2.0 ** -5))) == np.float32(0.96875)
    assert bf16_rne(np.float32(math.exp(-0.0019))) == np.float32(1.0)


def test_matches_library_cast():
    # A special case that reduces to a library routine: torch's float32 -> bfloat16 cast is RNE.
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 200000),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, -3.4e38, 1e-40, -1e-40, 1e-45], np.float32),
        rng.integers(0, 2 ** 32, 100000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ]).astype(np.float32)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).to(torch.float32).numpy()
    got = bf16_rne(x)
    nan = np.isnan(x)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_ftz():
    x = np.array([1e-39, -1e-39, 2.0 ** -126, -2.0 ** -126, 0.0, 1.0], np.float32)
    y = ftz32(x)
    assert y[0] == 0 and y[1] == 0 and np.signbit(y[1])
    assert y[2] == np.float32(2.0 ** -126) and y[3] == np.float32(-(2.0 ** -126))
    assert y[5] == 1.0


# ---------------------------------------------------------------- narrower formats
def test_e4m3_matches_the_library_cast_in_range():
    import torch
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(200000) * 10.0 ** rng.uniform(-4, 2.5, 200000),
                        rng.uniform(-440, 440, 20000), [0.0, -0.0, 1.0, 0.96875, 2.0 ** -9,
                                                        2.0 ** -10, 3 * 2.0 ** -11, 448.0]])
    x32 = x.astype(np.float32)
    x32 = x32[np.abs(x32) <= 448.0]   # the library cast gives NaN beyond the range; we saturate
    lib = torch.from_numpy(x32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.e4m3_rne(x32.astype(np.float64)), lib)


def test_e4m3_special_cases():
    # 1 - 2^-5 is the midpoint between 0.9375 and 1 and ties to the even 1.0: the mode-2 shift
    # exp(-2^-5) = 0.969 rounds back to exactly one in E4M3.
    assert oracle.e4m3_rne(1 - 2.0 ** -5) == 1.0
    assert oracle.e4m3_rne(float(np.exp(-2.0 ** -5))) == 1.0
    assert oracle.e4m3_rne(0.95) == 0.9375
    assert oracle.e4m3_rne(1000.0) == 448.0 and oracle.e4m3_rne(-1e9) == -448.0
    assert oracle.e4m3_rne(2.0 ** -10) == 0.0      # half the smallest subnormal: ties to zero
    assert oracle.e4m3_rne(3 * 2.0 ** -11) == 2.0 ** -9


def test_e2m1_is_the_nearest_grid_value_ties_to_even():
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    even = {0: True, 0.5: False, 1: True, 1.5: False, 2: True, 3: False, 4: True, 6: True}
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(0, 7, 5000), (grid[1:] + grid[:-1]) / 2])
    for v in x:
        d = np.abs(grid - v)
        best = grid[d == d.min()]
        want = best[0] if len(best) == 1 else [b for b in best if even[float(b)]][0]
        want = min(want, 6.0) if v <= 6 else 6.0
        assert oracle.e2m1_rne(v) == want, v
        assert oracle.e2m1_rne(-v) == -want


def test_mx_e2m1_block_scales():
    # A block whose largest magnitude is 1 gets the scale 2^-2, so 1 -> 4 X = 1 exactly and
    # 0.97 -> 3.88 X -> 4 X = 1: near-ones round to one. Blocks are 32 elements long.
    x = np.zeros(64)
    x[0], x[1], x[2] = 1.0, 0.97, 0.3
    x[32], x[33] = 0.01, 0.004
    q = oracle.mx_e2m1(x)
    assert q[0] == 1.0 and q[1] == 1.0 and q[2] == 0.25
    # second block: amax 0.01 -> floor(log2 0.01) = -7, X = 2^-9; 0.01 / X = 5.12 -> 6 (nearest
    # of 4 and 6 is 6); 0.004 / X = 2.048 -> 2
    assert q[32] == 6 * 2.0 ** -9 and q[33] == 2 * 2.0 ** -9
    assert np.all(q[34:] == 0)
