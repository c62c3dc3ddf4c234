"""Pins of the oracle's BF16-emulating backward pass (``emulate_bf16=True``): a hand-worked
golden case that fixes every cast point bit for bit, planted mistakes in those cast points
that the golden values catch, and the emulation with every rounding removed, which must be
the float64 backward.

The equations are the pages' (priors.kr post "BF16 플래시 어텐션은 왜 수천 스텝 뒤에 무너질까",
equations, paper §3.3.1: dS = alpha P o (dP - delta), dQ = dS K); the rounding points are the
backward kernel's, as the golden file's header lists them."""
import os

import numpy as np
import pytest

import oracle
import oracle.attention as oatt
from oracle.bf16 import bf16_rne, fp32, ftz32

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "bwd_emulated_cast_points.txt")

# The inputs the golden file states.
Q = np.array([[1, 0], [0, 1], [1, 1]], dtype=np.float64)
K = np.array([[1, 2], [2, 1], [0, 1]], dtype=np.float64)
V = np.array([[1, 0.5], [0.25, 1], [0.5, 0.5]], dtype=np.float64)
DO = np.array([[1, 1], [1, -1], [1, 0]], dtype=np.float64)
ALPHA = float(np.float32(0.3))
LSE = np.array([1.0, 1.0, float(np.float32(89.4))])
DELTA = np.array([float(np.float32(0.496)), float(np.float32(0.249)), 0.5])


def _golden():
    out = {"dq": np.zeros((3, 2)), "dk": np.zeros((3, 2)), "dv": np.zeros((3, 2))}
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, row, a, b = line.split()
            out[name][int(row)] = [float(a), float(b)]
    return out


def _oracle(**kw):
    g = oracle.attn_bwd(Q[None, None], K[None, None], V[None, None], DO[None, None],
                        LSE[None, None], DELTA[None, None], causal=False, scale=ALPHA, **kw)
    return {n: g[n][0, 0] for n in ("dq", "dk", "dv")}


def test_golden_case_bit_exact():
    got, ref = _oracle(emulate_bf16=True), _golden()
    for n in ("dq", "dk", "dv"):
        assert np.array_equal(got[n], ref[n]), (n, got[n], ref[n])


def _variant(mistake=None):
    """The one-head emulated backward written out step by step, with one cast point moved
    (``mistake``); ``None`` restates the cast points the golden header lists."""
    s = fp32(fp32(Q @ K.T) * np.float32(ALPHA)).astype(np.float64)
    x = fp32(s - LSE[:, None])
    p = np.exp(x.astype(np.float64)).astype(np.float32)
    if mistake != "no_ftz":
        p = ftz32(p)
    p = p.astype(np.float64)
    dp = fp32(DO @ V.T).astype(np.float64)
    diff = dp - DELTA[:, None]
    diff = (bf16_rne(fp32(diff)) if mistake == "bf16_diff" else fp32(diff)).astype(np.float64)
    ds = fp32(p * diff).astype(np.float64)
    a = np.float32(ALPHA)
    if mistake == "alpha_before_cast":
        ds_op = bf16_rne(fp32(ds * a)).astype(np.float64)
        a = np.float32(1.0)
    else:
        ds_op = bf16_rne(fp32(ds)).astype(np.float64)
    p_op = p if mistake == "p_uncast" else bf16_rne(fp32(p)).astype(np.float64)
    dq = bf16_rne(fp32(fp32(ds_op @ K) * a)).astype(np.float64)
    dk = bf16_rne(fp32(fp32(ds_op.T @ Q) * a)).astype(np.float64)
    dv = bf16_rne(fp32(p_op.T @ DO)).astype(np.float64)
    return {"dq": dq, "dk": dk, "dv": dv}


def test_restated_cast_points_reproduce_the_golden_values():
    ref, got = _golden(), _variant(None)
    for n in ref:
        assert np.array_equal(got[n], ref[n]), n


@pytest.mark.parametrize("mistake,least", [("alpha_before_cast", 1), ("bf16_diff", 1),
                                           ("p_uncast", 1), ("no_ftz", 1)])
def test_planted_cast_mistakes_break_the_golden_values(mistake, least):
    # Each plausible slip in where the emulation rounds moves at least one golden value, so
    # the golden pin would catch it in the oracle.
    ref, got = _golden(), _variant(mistake)
    changed = sum(int((got[n] != ref[n]).sum()) for n in ref)
    assert changed >= least, mistake


def test_no_ftz_shows_in_dq_row_with_subnormal_probabilities():
    # Row 2's probabilities are FP32 subnormals: flushed, its dQ is exactly zero; kept, it is
    # a BF16 subnormal.
    assert np.all(_golden()["dq"][2] == 0.0)
    assert np.any(_variant("no_ftz")["dq"][2] != 0.0)


def _identity(x):
    return np.asarray(x, dtype=np.float64)


@pytest.mark.parametrize("causal", [False, True])
def test_emulation_without_roundings_is_the_float64_pass(monkeypatch, causal):
    # Remove every rounding of the emulation (FP32, BF16, flush to zero): what is left must be
    # the float64 definition, forward and backward, delta both ways.
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 4, 40, 8))
    k = rng.standard_normal((1, 2, 40, 8))
    v = rng.standard_normal((1, 2, 40, 8))
    do = rng.standard_normal((1, 4, 40, 8))
    k[0, 0, 3] = k[0, 0, 1]   # a planted tie so that the fix modes take their branches
    ref = {}
    for mode in (0, 1, 2):
        f = oracle.attn_fwd(q, k, v, causal=causal, scale=0.3, fix_mode=mode)
        d = oracle.attn_delta(f["o"], do)
        da = oracle.attn_delta_alt(q, k, v, do, f["lse"], causal=causal, scale=0.3)
        g = oracle.attn_bwd(q, k, v, do, f["lse"], d, causal=causal, scale=0.3)
        ref[mode] = (f, d, da, g)
    for name in ("fp32", "bf16_rne", "ftz32"):
        monkeypatch.setattr(oatt, name, _identity)
    for mode in (0, 1, 2):
        f = oracle.attn_fwd(q, k, v, causal=causal, scale=0.3, fix_mode=mode, emulate_bf16=True)
        d = oracle.attn_delta(f["o"], do, emulate_bf16=True)
        da = oracle.attn_delta_alt(q, k, v, do, f["lse"], causal=causal, scale=0.3,
                                   emulate_bf16=True)
        g = oracle.attn_bwd(q, k, v, do, f["lse"], d, causal=causal, scale=0.3, emulate_bf16=True)
        rf, rd, rda, rg = ref[mode]
        np.testing.assert_allclose(f["o"], rf["o"], rtol=0, atol=1e-6)
        np.testing.assert_allclose(f["lse"], rf["lse"], rtol=0, atol=1e-6)
        np.testing.assert_allclose(d, rd, rtol=0, atol=1e-6)
        np.testing.assert_allclose(da, rda, rtol=0, atol=1e-6)
        for n in ("dq", "dk", "dv"):
            np.testing.assert_allclose(g[n], rg[n], rtol=0, atol=1e-6)


def test_emulated_sink_heavy_dq_error_is_the_bf16_ds_cast():
    # On the sink-heavy input (+6 logit on key 0 carried by a feature of 48, its key copied
    # into other rows' visible keys) the BF16 cast of dS alone moves dQ by about 12% from
    # float64, while FP32 rounding of dP - delta moves it by 3e-5: the copies of the sink key
    # share the large feature and their dS nearly cancel along it.
    from precision_flash_attention_gb300 import inputs
    t = inputs.sink_heavy(1, 1, 512, 64, seed=0)
    q, k, v, do = (t[n].double().numpy() for n in ("q", "k", "v", "do"))
    f = oracle.attn_fwd(q, k, v, causal=True, scale=0.125)
    d = oracle.attn_delta(f["o"], do)
    g64 = oracle.attn_bwd(q, k, v, do, f["lse"], d, causal=True, scale=0.125)
    ge = oracle.attn_bwd(q, k, v, do, f["lse"], d, causal=True, scale=0.125, emulate_bf16=True)
    err = np.linalg.norm(ge["dq"] - g64["dq"]) / np.linalg.norm(g64["dq"])
    assert err > 2e-2
    for n in ("dk", "dv"):
        assert np.linalg.norm(ge[n] - g64[n]) / np.linalg.norm(g64[n]) < 1e-2
