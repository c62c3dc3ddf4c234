"""Pins of the oracle's study functions: the forward pass of an implementation that stores
the unnormalised product Pbar V in BF16 (``attn_fwd_unfused``, the paper's analysed code)
and the tiled-kernel monitor (``attn_fwd_monitor``).

The unfused profile is pinned by the pages' two worked BF16 traces (its block product is
the rounding they walk through), by the float64 definition once every rounding is removed,
and by the bias the pages describe: two exact ones over negative-dominated values round
the sum one way, and the fix removes it. The monitor is pinned by brute force on small
integer inputs, a hand-worked row, and its agreement with the repeated-row counter."""
import numpy as np
import pytest

import oracle
import oracle.attention as oatt
from precision_flash_attention_gb300 import inputs


def _trace_row(acc, residual_v, addend):
    # One query row over three keys in one block: keys 0 and 2 score 0 (two exact maxima, so
    # mode 0 gives Pbar = 1 there), key 1 scores -0.69140625 (BF16 Pbar = 0.5); feature 0 of V
    # holds the trace's terms, so the block product is acc + 0.5 * residual_v + addend.
    q = np.zeros((1, 1, 3, 2))
    q[0, 0, :, 0] = 1.0
    k = np.zeros((1, 1, 3, 2))
    k[0, 0, 1, 0] = -0.69140625
    v = np.zeros((1, 1, 3, 2))
    v[0, 0, :, 0] = [acc, residual_v, addend]
    return q, k, v


@pytest.mark.parametrize("acc,residual_v,addend,expected", [
    # priors.kr post, bit-level paragraph of the core-idea section (paper §3.3.2): -2.40625,
    # a residual of about -0.00087 (here 0.5 * BF16(-0.00174) = -0.00086975...), and
    # -2.296875 round to -4.71875 against the exact -4.70399.
    (-2.40625, -0.001739501953125, -2.296875, -4.71875),
    # bud-325 note, Results: -0.85546875 + a small residual (-2^-11) + -0.0859375 round to
    # -0.94140625 instead of -0.94189453125.
    (-0.85546875, -2.0 ** -10, -0.0859375, -0.94140625),
])
def test_unfused_block_product_reproduces_the_worked_traces(acc, residual_v, addend, expected):
    q, k, v = _trace_row(acc, residual_v, addend)
    r = oracle.attn_fwd_unfused(q, k, v, scale=1.0, fix_mode=0, block=512)
    assert r["obar"][0, 0, 0, 0] == expected
    # Without the residual, the two BF16 terms alone land on a midpoint and tie to even
    # (the opposite-sign small error of the pages' single-add case).
    q, k, v = _trace_row(acc, 0.0, addend)
    r0 = oracle.attn_fwd_unfused(q, k, v, scale=1.0, fix_mode=0, block=512)
    assert r0["obar"][0, 0, 0, 0] == float(oracle.bf16_sum([acc, addend]))


def _identity(x):
    return np.asarray(x, dtype=np.float64)


@pytest.mark.parametrize("block", [16, 64])
@pytest.mark.parametrize("causal", [False, True])
def test_unfused_without_roundings_is_the_float64_pass(monkeypatch, block, causal):
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 2, 70, 8))
    k = rng.standard_normal((1, 1, 70, 8))
    v = rng.standard_normal((1, 1, 70, 8))
    k[0, 0, 5] = k[0, 0, 2]
    ref = oracle.attn_fwd(q, k, v, causal=causal, scale=0.375)   # alpha exact in FP32
    for name in ("fp32", "bf16_rne", "ftz32"):
        monkeypatch.setattr(oatt, name, _identity)
    for mode in (0, 1, 2):
        r = oracle.attn_fwd_unfused(q, k, v, causal=causal, scale=0.375, fix_mode=mode, block=block)
        np.testing.assert_allclose(r["o"], ref["o"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(r["lse"], ref["lse"], rtol=0, atol=1e-12)


def _bias_ulp(o, ref, first_row):
    ulp = 2.0 ** (np.floor(np.log2(np.abs(ref))) - 7)
    return float(((o - ref) / ulp)[..., first_row:, :].mean())


def test_unfused_profile_shows_the_pages_bias_and_the_fix_removes_it():
    # priors.kr post, core idea (paper §3.3.2): where two scores tie at the maximum, Pbar is
    # exactly 1 twice and the product's BF16 sum of two BF16 V values rounds one way on
    # negative-dominated features; the fix (paper §4) keeps every Pbar below 1. A single
    # maximum leaves no such bias.
    t2 = inputs.tie_probe(1, 4, 512, 64, ties=2, seed=1)
    t1 = inputs.tie_probe(1, 4, 512, 64, ties=1, seed=1)
    out = {}
    for name, t in (("two", t2), ("one", t1)):
        q, k, v = (t[n].double().numpy() for n in ("q", "k", "v"))
        ref = oracle.attn_fwd(q, k, v, causal=True, scale=0.125)["o"]
        for mode in (0, 1, 2):
            r = oracle.attn_fwd_unfused(q, k, v, causal=True, scale=0.125, fix_mode=mode, block=512)
            out[name, mode] = (_bias_ulp(r["o"], ref, 2),
                               float((np.sum(r["o"] - ref, axis=-1)[..., 2:] < 0).mean()))
    assert out["two", 0][0] < -0.08 and out["two", 0][1] > 0.9
    for mode in (1, 2):
        assert abs(out["two", mode][0]) < 0.03
    assert abs(out["one", 0][0]) < 0.03


# ---------------------------------------------------------------- monitor
def _brute_monitor(q, k, v, *, causal, scale, fix_mode, beta, eps, tile):
    """Pure-Python loops: the shift per tile from the keys up to its end, then the exact ones."""
    from oracle.bf16 import bf16_rne, fp32
    B, Hq, N, d = q.shape
    g = Hq // k.shape[1]
    ones = 0
    hist = [0] * oracle.TIE_BINS
    for b in range(B):
        for h in range(Hq):
            for i in range(N):
                keys = [j for j in range(N) if not causal or j <= i]
                s = {j: float(fp32(float(fp32(sum(q[b, h, i, c] * k[b, h // g, j, c] for c in range(d))))
                                   * float(np.float32(scale)))) for j in keys}
                r_m = max(s.values())
                mult = sum(1 for j in keys if s[j] >= r_m - eps)
                hist[min(mult, oracle.TIE_BINS) - 1] += 1
                for j0 in range(0, N, tile):
                    seen = [j for j in keys if j < j0 + tile]
                    if not seen:
                        continue
                    m1 = max(s[j] for j in seen)
                    rep = sum(1 for j in seen if s[j] >= m1 - eps) >= 2
                    m = m1
                    if rep and fix_mode == 1:
                        m = beta * m1 if m1 > 0 else (0.0 if m1 < 0 else 2.0 ** -5)
                    elif rep and fix_mode == 2:
                        m = m1 + 2.0 ** -5
                    m = float(fp32(m))
                    for j in seen:
                        if j >= j0:
                            p = float(fp32(np.exp(float(fp32(s[j] - m)))))
                            ones += int(float(bf16_rne(p)) == 1.0)
    return ones, np.array(hist)


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_monitor_matches_brute_force(mode, causal):
    t = inputs.integer_grid(1, 2, 1, 40, 8, causal=causal, n_planted=4, seed=mode + 3)
    q, k, v = (t[n].double().numpy() for n in ("q", "k", "v"))
    r = oracle.attn_fwd_monitor(q, k, v, causal=causal, scale=0.125, fix_mode=mode, tile=16)
    ones, hist = _brute_monitor(q, k, v, causal=causal, scale=0.125, fix_mode=mode, beta=2.0,
                                eps=1e-3, tile=16)
    assert r["operational_ones"] == ones
    assert np.array_equal(r["tie_hist"], hist)


def test_monitor_hand_worked_row():
    # Row 0 over two tiles of 4 keys: tile 0 holds a repeated maximum 1.0 (keys 0 and 1), tile
    # 1 a single larger maximum 2.0 (key 4). Mode 0: tile 0 hands two ones to the product
    # (shift 1.0), tile 1 one (shift 2.0): 3 operational ones, while the final shift has 1.
    # Mode 1: tile 0 is repeated (shift 2 x 1.0, no ones), tile 1 a single maximum (one): 1.
    # Rows 1..7 have q = 0: eight scores of 0, a maximum of multiplicity 8; mode 0 counts one
    # exact one per key (8 per row), mode 1 none (repeated, r_m = 0, shift 2^-5).
    q = np.zeros((1, 1, 8, 1))
    q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, 1, 8, 1))
    k[0, 0, :, 0] = [1.0, 1.0, -3.0, -3.0, 2.0, -3.0, -3.0, -3.0]
    v = np.zeros((1, 1, 8, 1))
    for mode, expect in ((0, 3 + 7 * 8), (1, 1)):
        r = oracle.attn_fwd_monitor(q, k, v, scale=1.0, fix_mode=mode, tile=4)
        assert r["operational_ones"] == expect, mode
        assert list(r["tie_hist"]) == [1, 0, 0, 0, 0, 0, 0, 7]
    assert oracle.attn_fwd(q, k, v, scale=1.0, fix_mode=0)["counters"]["ones"] == 1 + 7 * 8


@pytest.mark.parametrize("causal", [False, True])
def test_monitor_histogram_agrees_with_the_counters(causal):
    t = inputs.integer_grid(2, 2, 1, 150, 16, causal=causal, n_planted=8, seed=4)
    q, k, v = (t[n].double().numpy() for n in ("q", "k", "v"))
    for mode in (0, 1):
        r = oracle.attn_fwd_monitor(q, k, v, causal=causal, scale=0.125, fix_mode=mode)
        f = oracle.attn_fwd(q, k, v, causal=causal, scale=0.125, fix_mode=mode, emulate_bf16=True)
        assert r["tie_hist"].sum() == 2 * 2 * 150
        assert r["tie_hist"][1:].sum() == f["counters"]["repeated_rows"]
        if mode == 0:
            # Mode 0 never moves a shift away from the running maximum: every exact one of the
            # final shift was handed to the product in its own tile too.
            assert r["operational_ones"] >= f["counters"]["ones"]


# ---------------------------------------------------------------- narrower Pbar formats
def _tied_row(r_m):
    # Row 0 of a 4-key block: keys 0 and 1 score r_m (a repeated maximum), keys 2 and 3 far
    # below (-30); the other rows are copies. Scale 1.
    q = np.ones((1, 1, 4, 1))
    k = np.zeros((1, 1, 4, 1))
    k[0, 0, :, 0] = [r_m, r_m, -30.0, -30.0]
    v = np.ones((1, 1, 4, 1))
    return q, k, v


def test_e4m3_pbar_worked_cases():
    # Mode 2 subtracts 2^-5 on a repeated maximum: exp(-2^-5) = 0.9692 lies above the E4M3
    # midpoint 1 - 2^-5 between 0.9375 and 1, so Pbar rounds back to exactly 1 (two per row).
    q, k, v = _tied_row(1.0)
    r = oracle.attn_fwd_blockwise(q, k, v, scale=1.0, fix_mode=2, block=4, pbar="e4m3", accumulate="fp32")
    assert r["operational_ones"] == 2 * 4
    # Mode 1 with beta = 2 on a repeated maximum of 16: Pbar = e^-16 = 1.1e-7 lies below half
    # the smallest E4M3 subnormal (2^-10), so every weight is 0 and l = 0 (NaN output).
    q, k, v = _tied_row(16.0)
    r = oracle.attn_fwd_blockwise(q, k, v, scale=1.0, fix_mode=1, block=4, pbar="e4m3", accumulate="fp32")
    assert r["operational_ones"] == 0 and np.isnan(r["o"]).all()
    # In BF16 the same two cases keep every Pbar below 1 and finite.
    for mode, rm in ((2, 1.0), (1, 16.0)):
        q, k, v = _tied_row(rm)
        r = oracle.attn_fwd_blockwise(q, k, v, scale=1.0, fix_mode=mode, block=4, pbar="bf16",
                                      accumulate="fp32")
        assert r["operational_ones"] == 0 and np.isfinite(r["o"]).all()


def test_mxfp4_pbar_worked_case():
    # Mode 2 on a repeated maximum: both tied weights are 0.9692, the block's largest; the scale
    # is 2^(floor(log2 0.9692) - 2) = 1/8 and 0.9692 / (1/8) = 7.75 saturates at 6: Pbar = 0.75.
    # The far keys (e^-31) are below the smallest E2M1 step at that scale and become 0, so O is
    # V's mean over the two tied keys exactly, and no Pbar equals 1.
    q, k, v = _tied_row(1.0)
    v[0, 0, :, 0] = [2.0, 4.0, 100.0, 100.0]
    r = oracle.attn_fwd_blockwise(q, k, v, scale=1.0, fix_mode=2, block=4, pbar="mxfp4", accumulate="fp32")
    assert r["operational_ones"] == 0
    assert np.all(r["o"][0, 0, :, 0] == 3.0)
    assert np.all(r["obar"][0, 0, :, 0] == 0.75 * 6.0)


@pytest.mark.parametrize("pbar", ["e4m3", "mxfp4"])
@pytest.mark.parametrize("accumulate", ["bf16", "fp32"])
def test_blockwise_without_roundings_is_the_float64_pass(monkeypatch, pbar, accumulate):
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 2, 70, 8))
    k = rng.standard_normal((1, 1, 70, 8))
    v = rng.standard_normal((1, 1, 70, 8))
    k[0, 0, 9] = k[0, 0, 4]
    ref = oracle.attn_fwd(q, k, v, causal=True, scale=0.375)
    for name in ("fp32", "bf16_rne", "ftz32", "e4m3_rne", "mx_e2m1"):
        monkeypatch.setattr(oatt, name, lambda x, *a, **kw: np.asarray(x, dtype=np.float64))
    for mode in (0, 1, 2):
        r = oracle.attn_fwd_blockwise(q, k, v, causal=True, scale=0.375, fix_mode=mode, block=32,
                                      pbar=pbar, accumulate=accumulate)
        np.testing.assert_allclose(r["o"], ref["o"], rtol=0, atol=1e-12)
