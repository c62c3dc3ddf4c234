"""Pins of the oracle's forward pass: a library softmax, closed forms, shift invariance,
brute-force counts on integer-valued inputs, and the underflow the pages warn about."""
import math

import numpy as np
import pytest
import torch

import oracle
from precision_flash_attention_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _np(t):
    return t.to(torch.float64).numpy()


def _torch_reference(q, k, v, causal, scale):
    """softmax(scale * Q K^T + mask) V and logsumexp with torch CPU float64 ops."""
    group = q.shape[1] // k.shape[1]
    qt = torch.from_numpy(q)
    kt = torch.from_numpy(k).repeat_interleave(group, dim=1)
    vt = torch.from_numpy(v).repeat_interleave(group, dim=1)
    s = scale * qt @ kt.transpose(-1, -2)
    if causal:
        n = q.shape[2]
        s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
    return (torch.softmax(s, dim=-1) @ vt).numpy(), torch.logsumexp(s, dim=-1).numpy()


CASES = [
    # B, Hq, Hkv, N, d, causal
    (1, 1, 1, 64, 64, False),
    (2, 4, 2, 37, 16, True),
    (1, 3, 1, 100, 32, False),
    (1, 2, 2, 129, 8, True),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_matches_library_softmax(case, mode):
    B, Hq, Hkv, N, d, causal = case
    t = inputs.gaussian(B, Hq, Hkv, N, d, std_qkv=1.0, seed=1)
    q, k, v = _np(t["q"]), _np(t["k"]), _np(t["v"])
    scale = 1.0 / math.sqrt(d)
    r = oracle.attn_fwd(q, k, v, causal=causal, scale=scale, fix_mode=mode, beta=2.0, eps=1e-3)
    o_ref, lse_ref = _torch_reference(q, k, v, causal, scale)
    np.testing.assert_allclose(r["o"], o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["lse"], lse_ref, rtol=0, atol=1e-12)


def test_single_key_closed_form():
    # N = 1: the only weight is 1, so O = V and lse = S (for every mode).
    t = inputs.gaussian(2, 2, 1, 1, 16, seed=3)
    q, k, v = _np(t["q"]), _np(t["k"]), _np(t["v"])
    for mode in (0, 1, 2):
        r = oracle.attn_fwd(q, k, v, causal=True, scale=0.25, fix_mode=mode)
        for h in range(2):
            np.testing.assert_allclose(r["o"][:, h], v[:, 0], atol=1e-15)
            np.testing.assert_allclose(r["lse"][:, h, 0], 0.25 * (q[:, h, 0] * k[:, 0, 0]).sum(-1),
                                       atol=1e-14)


def test_causal_first_row():
    # Causal row 0 sees only key 0: O_0 = V_0.
    t = inputs.gaussian(1, 3, 3, 50, 32, seed=4)
    q, k, v = _np(t["q"]), _np(t["k"]), _np(t["v"])
    r = oracle.attn_fwd(q, k, v, causal=True, fix_mode=1)
    np.testing.assert_allclose(r["o"][0, :, 0], v[0, :, 0], atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_modes_agree_in_float64(causal):
    # Softmax is invariant to a per-row shift, so all three modes give the same O and lse in
    # exact arithmetic (priors.kr, the fix paragraph, paper §4; bud-325 Key claims).
    t = inputs.integer_grid(1, 2, 1, 80, 64, causal=causal, n_planted=12, seed=5)
    q, k, v = _np(t["q"]), _np(t["k"]), _np(t["v"])
    outs = [oracle.attn_fwd(q, k, v, causal=causal, scale=0.125, fix_mode=m, beta=3.0)
            for m in (0, 1, 2)]
    assert outs[0]["counters"]["repeated_rows"] >= 12
    for r in outs[1:]:
        np.testing.assert_allclose(r["o"], outs[0]["o"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(r["lse"], outs[0]["lse"], rtol=0, atol=1e-12)


def _brute_force_counts(q, k, causal, mode):
    """Pure-Python counts on integer-valued Q and K (scale 1/8, eps < 1/8).

    Scores are exact integers / 8, so a row is repeated iff its integer maximum occurs at
    least twice. Mode 0 keeps m = r_m: every maximum entry gives Pbar = 1 exactly and every
    other entry is at least 1/8 below, so the BF16 Pbar is below 1. In modes 1 and 2 a
    repeated row's shift moves the maximum exponent argument to at most -2^-5 (mode 2,
    or mode 1 with r_m = 0), -(beta-1) r_m <= -1/8 (r_m > 0) or r_m <= -1/8 (r_m < 0),
    all of which round below 1 in BF16; non-repeated rows keep exactly one 1.
    """
    B, Hq, N, d = q.shape
    group = Hq // k.shape[1]
    rep = ones = 0
    for b in range(B):
        for h in range(Hq):
            for i in range(N):
                qi = [int(x) for x in q[b, h, i]]
                dots = []
                for j in range(N):
                    if causal and j > i:
                        continue
                    kj = [int(x) for x in k[b, h // group, j]]
                    dots.append(sum(a * c for a, c in zip(qi, kj)))
                mx = max(dots)
                mult = sum(1 for x in dots if x == mx)
                rep += mult >= 2
                if mode == 0:
                    ones += mult
                else:
                    ones += 0 if mult >= 2 else 1
    return rep, ones


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("emulate", [False, True])
def test_counters_brute_force(causal, mode, emulate):
    t = inputs.integer_grid(1, 2, 1, 48, 16, causal=causal, n_planted=6, seed=7)
    q, k, v = _np(t["q"]), _np(t["k"]), _np(t["v"])
    r = oracle.attn_fwd(q, k, v, causal=causal, scale=0.125, fix_mode=mode, beta=2.0, eps=1e-3,
                        emulate_bf16=emulate)
    rep, ones = _brute_force_counts(q, k, causal, mode)
    assert rep >= 6
    assert r["counters"]["repeated_rows"] == rep
    assert r["counters"]["ones"] == ones
    assert r["counters"]["nonfinite_rows"] == 0


def test_tiny_grid_workload_counts():
    t = inputs.make("grid", seed=0)
    q, k, v = _np(t["q"]), _np(t["k"]), _np(t["v"])
    for mode in (0, 1, 2):
        r = oracle.attn_fwd(q, k, v, scale=0.125, fix_mode=mode)
        rep, ones = _brute_force_counts(q, k, False, mode)
        assert (r["counters"]["repeated_rows"], r["counters"]["ones"]) == (rep, ones)
        assert rep >= 8


@pytest.mark.parametrize("mode", [1, 2])
def test_fix_removes_repeated_ones(mode):
    # The fix's guarantee: on repeated-maximum rows no BF16 Pbar equals 1 (priors.kr, the fix
    # paragraph, paper §4; bud-325 Method). So no row has two or more entries equal to 1.0.
    t = inputs.integer_grid(1, 1, 1, 64, 64, n_planted=8, seed=11)
    q, k, v = _np(t["q"]), _np(t["k"]), _np(t["v"])
    h = oracle.attn_fwd_head(q[0, 0], k[0, 0], v[0, 0], scale=0.125, fix_mode=mode)
    assert h["repeated"].sum() >= 8
    assert (h["ones"][h["repeated"]] == 0).all()
    assert (h["ones"] <= 1).all()
    h0 = oracle.attn_fwd_head(q[0, 0], k[0, 0], v[0, 0], scale=0.125, fix_mode=0)
    assert (h0["ones"][h0["repeated"]] >= 2).all()


def test_shift_rule_cases():
    # priors.kr, the fix equation (paper §4), and bud-325 Algorithm 1.
    r_m = np.array([2.0, -3.0, 0.0, 1.5])
    rep = np.array([True, True, True, False])
    np.testing.assert_array_equal(oracle.fix_shift(r_m, rep, 0, 4.0, False), r_m)
    np.testing.assert_array_equal(oracle.fix_shift(r_m, rep, 1, 4.0, False), [8.0, 0.0, 2 ** -5, 1.5])
    np.testing.assert_array_equal(oracle.fix_shift(r_m, rep, 2, 4.0, False),
                                  [2.0 + 2 ** -5, -3.0 + 2 ** -5, 2 ** -5, 1.5])


def test_tie_tolerance_window():
    # A second score within eps of the maximum flags the row; one just outside does not.
    k = np.array([[1.0], [1.0 - 0.9e-3], [-2.0]])
    q = np.ones((1, 1))
    v = np.ones((3, 1))
    assert oracle.attn_fwd_head(q, k, v, scale=1.0, fix_mode=1, eps=1e-3)["repeated"][0]
    k[1, 0] = 1.0 - 1.1e-3
    assert not oracle.attn_fwd_head(q, k, v, scale=1.0, fix_mode=1, eps=1e-3)["repeated"][0]


def test_gap_between_eps_and_round_to_one():
    # eps = 1e-3 is below the BF16 round-to-one window (|x| <= 1.955e-3): a row whose top two
    # scores are 1.5e-3 apart is not flagged, yet both entries round to 1.0 in BF16.
    k = np.array([[1.0], [1.0 - 1.5e-3]])
    q = np.ones((1, 1))
    v = np.ones((2, 1))
    r = oracle.attn_fwd_head(q, k, v, scale=1.0, fix_mode=1, eps=1e-3)
    assert not r["repeated"][0] and r["ones"][0] == 2


def test_emulation_close_to_float64():
    t = inputs.sink_heavy(1, 2, 96, 16, seed=2)
    q, k, v = _np(t["q"]), _np(t["k"]), _np(t["v"])
    for mode in (0, 1, 2):
        a = oracle.attn_fwd(q, k, v, causal=True, scale=0.125, fix_mode=mode)
        e = oracle.attn_fwd(q, k, v, causal=True, scale=0.125, fix_mode=mode, emulate_bf16=True)
        rel = np.linalg.norm(e["o"] - a["o"]) / np.linalg.norm(a["o"])
        # The BF16 cast points stay inside the float tolerance the GPU path is held to.
        assert rel < 4e-3
        assert np.abs(e["o"] - a["o"]).max() < 1.5e-2
        assert np.abs(e["lse"] - a["lse"]).max() < 1.5e-2


def test_underflow_probe():
    # Mode 1 subtracts beta*r_m on repeated rows; with r_m = 200 every exponent argument falls
    # below the FP32 range and l underflows to 0 in FP32 (priors.kr caveats: logits in the
    # thousands push the shifted exponents out of FP32 range; paper App. C).
    big = inputs.underflow_probe(1, 1, 128, 64, logit=200.0)
    q, k, v = _np(big["q"]), _np(big["k"]), _np(big["v"])
    e = oracle.attn_fwd(q, k, v, scale=0.125, fix_mode=1, beta=2.0, emulate_bf16=True)
    assert e["counters"]["repeated_rows"] == 128
    assert e["counters"]["nonfinite_rows"] == 128
    assert np.isnan(e["o"]).all()
    f = oracle.attn_fwd(q, k, v, scale=0.125, fix_mode=1, beta=2.0)
    assert f["counters"]["nonfinite_rows"] == 0
    small = inputs.underflow_probe(1, 1, 128, 64, logit=10.0)
    q, k, v = _np(small["q"]), _np(small["k"]), _np(small["v"])
    e = oracle.attn_fwd(q, k, v, scale=0.125, fix_mode=1, beta=2.0, emulate_bf16=True)
    assert e["counters"]["repeated_rows"] == 128 and e["counters"]["nonfinite_rows"] == 0
    # Mode 2 only moves the shift by 2^-5 and never underflows here.
    e2 = oracle.attn_fwd(_np(big["q"]), _np(big["k"]), _np(big["v"]), scale=0.125, fix_mode=2,
                         emulate_bf16=True)
    assert e2["counters"]["nonfinite_rows"] == 0


def test_unconditional_beta_shift_is_rejected_variant():
    # priors.kr, the fix paragraph (paper App. C): applying beta*r_m to every row, not just
    # repeated ones, can zero the denominator on rows with a single large positive maximum.
    # The planted mistake lives here, on the CPU: flag every row and watch l underflow.
    s = np.array([[120.0, 3.0, -1.0]])
    r_m = s.max(1)
    m = oracle.fix_shift(r_m, np.array([True]), 1, 2.0, True)
    l = oracle.ftz32(np.exp(oracle.fp32(s - m[:, None]))).sum(1)
    assert l[0] == 0.0
    m_ok = oracle.fix_shift(r_m, np.array([False]), 1, 2.0, True)
    assert oracle.ftz32(np.exp(oracle.fp32(s - m_ok[:, None]))).sum(1)[0] > 0


# Planted tie patterns (inputs.TIE_PATTERNS): the flag each construction fixes by
# definition (two scores within eps = 0.05 of the row maximum, scale 1/8).
TIE_LABELS = {"jump_same_block": True, "jump_same_class": True, "jump_block_and_class": True,
              "jump_single": False, "jump_near_miss": False, "jump_exact_pair": True,
              "tie_below_running_max": True, "rise_within_eps": True}


@pytest.mark.parametrize("name", sorted(TIE_LABELS))
def test_planted_tie_patterns(name):
    t = inputs.tie_patterns([name])
    q, k, v = (t[n].double().numpy() for n in ("q", "k", "v"))
    r = oracle.attn_fwd(q, k, v, causal=False, scale=0.125, fix_mode=1, beta=2.0, eps=0.05)
    assert r["repeated"].all() if TIE_LABELS[name] else not r["repeated"].any()
    assert r["counters"]["repeated_rows"] == (256 if TIE_LABELS[name] else 0)


@pytest.mark.parametrize("sign", [-1, 0])
def test_signed_max_grid_has_the_promised_maxima(sign):
    # The generator's rows that see two planted keys have a repeated maximum of the stated
    # sign (negative, or exactly zero); the GPU tests rely on it to reach mode 1's r_m <= 0
    # branches.
    from precision_flash_attention_gb300 import inputs
    t = inputs.signed_max_grid(1, 2, 1, 200, 64, sign=sign, n_keys=3, seed=1)
    q, k, v = (t[n].double().numpy() for n in ("q", "k", "v"))
    f = oracle.attn_fwd(q, k, v, scale=0.125, fix_mode=0)
    assert f["repeated"].all()
    assert (f["m"] < 0).all() if sign < 0 else (f["m"] == 0).all()
    f1 = oracle.attn_fwd(q, k, v, scale=0.125, fix_mode=1)
    assert (f1["m"] == (0.0 if sign < 0 else 2.0 ** -5)).all()
    assert f1["counters"]["ones"] == 0
