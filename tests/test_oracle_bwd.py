"""Pins of the oracle's backward pass: central finite differences, the delta identity, a
library autograd reference, and planted mistakes that those pins must catch."""
import math

import numpy as np
import pytest
import torch

import oracle
from precision_flash_attention_gb300 import inputs


def _np(t):
    return t.to(torch.float64).numpy()


def _loss(q, k, v, do, causal, scale, mode):
    o = oracle.attn_fwd(q, k, v, causal=causal, scale=scale, fix_mode=mode, beta=2.0)["o"]
    return float((o * do).sum())


def _grads(q, k, v, do, causal, scale, mode, bwd_scale=None, delta=None):
    f = oracle.attn_fwd(q, k, v, causal=causal, scale=scale, fix_mode=mode, beta=2.0)
    dlt = oracle.attn_delta(f["o"], do) if delta is None else delta
    return oracle.attn_bwd(q, k, v, do, f["lse"], dlt, causal=causal,
                           scale=scale if bwd_scale is None else bwd_scale)


def _fd(q, k, v, do, causal, scale, mode, h=1e-6):
    out = {}
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        g = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            lp = _loss(q, k, v, do, causal, scale, mode)
            x[idx] = old - h
            lm = _loss(q, k, v, do, causal, scale, mode)
            x[idx] = old
            g[idx] = (lp - lm) / (2 * h)
        out[name] = g
    return out


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def _small(seed, n=7, causal=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, 2, n, 4))
    k = rng.standard_normal((1, 1, n, 4))
    v = rng.standard_normal((1, 1, n, 4))
    do = rng.standard_normal((1, 2, n, 4))
    if seed % 2 == 0:  # plant an exact tie in row n-1 so modes 1/2 take their branches
        k[0, 0, 1] = k[0, 0, 0]
    return q, k, v, do


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("seed", [0, 1])
def test_finite_differences(mode, causal, seed):
    # dS = alpha P o (dP - delta), dQ = dS K (priors.kr equations, paper §3.3.1); dK, dV the
    # standard flash-attention backward. L = sum(O o dO) so dL/dO = dO.
    q, k, v, do = _small(seed, causal=causal)
    scale = 0.7
    g = _grads(q, k, v, do, causal, scale, mode)
    fd = _fd(q, k, v, do, causal, scale, mode)
    for name in ("dq", "dk", "dv"):
        assert _rel(g[name], fd[name]) < 1e-6, name


def test_finite_differences_detect_planted_mistakes():
    # Each plausible slip in the backward formulas must break the finite-difference pin:
    # a dropped alpha in dS, a transposed operand (K and V swapped), a dropped delta.
    q, k, v, do = _small(2, causal=True)
    scale = 0.7
    fd = _fd(q, k, v, do, True, scale, 0)
    wrong_alpha = _grads(q, k, v, do, True, scale, 0, bwd_scale=1.0)
    assert _rel(wrong_alpha["dq"], fd["dq"]) > 1e-2
    f = oracle.attn_fwd(q, k, v, causal=True, scale=scale)
    swapped = oracle.attn_bwd(q, v, k, do, f["lse"], oracle.attn_delta(f["o"], do), causal=True,
                              scale=scale)
    assert _rel(swapped["dq"], fd["dq"]) > 1e-2
    no_delta = _grads(q, k, v, do, True, scale, 0, delta=np.zeros(q.shape[:3]))
    assert _rel(no_delta["dq"], fd["dq"]) > 1e-2


@pytest.mark.parametrize("causal", [False, True])
def test_matches_library_autograd(causal):
    t = inputs.gaussian(2, 4, 2, 33, 16, std_qkv=1.0, seed=9)
    q, k, v, do = (_np(t[n]) for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(16)
    g = _grads(q, k, v, do, causal, scale, 1)
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    kk, vv = kt.repeat_interleave(2, 1), vt.repeat_interleave(2, 1)
    s = scale * qt @ kk.transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(33, 33, dtype=torch.bool).triu(1), float("-inf"))
    o = torch.softmax(s, -1) @ vv
    (o * torch.from_numpy(do)).sum().backward()
    for name, ref in (("dq", qt.grad), ("dk", kt.grad), ("dv", vt.grad)):
        np.testing.assert_allclose(g[name], ref.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_delta_identity(causal):
    # rowsum(dO o O) == rowsum(dP o P) in exact arithmetic (priors.kr "방법", paper §3.2;
    # bud-325 Key claims): the two ways of computing the backward preprocessing term.
    t = inputs.sink_heavy(1, 2, 64, 16, seed=4)
    q, k, v, do = (_np(t[n]) for n in ("q", "k", "v", "do"))
    f = oracle.attn_fwd(q, k, v, causal=causal, scale=0.125)
    d1 = oracle.attn_delta(f["o"], do)
    d2 = oracle.attn_delta_alt(q, k, v, do, f["lse"], causal=causal, scale=0.125)
    np.testing.assert_allclose(d1, d2, rtol=0, atol=1e-12 * max(1.0, np.abs(d1).max()))


def test_emulated_backward_close_to_float64():
    t = inputs.gaussian(1, 2, 1, 96, 32, std_qkv=0.5, std_do=1e-2, seed=6)
    q, k, v, do = (_np(t[n]) for n in ("q", "k", "v", "do"))
    f = oracle.attn_fwd(q, k, v, causal=True)
    g = oracle.attn_bwd(q, k, v, do, f["lse"], oracle.attn_delta(f["o"], do), causal=True)
    fe = oracle.attn_fwd(q, k, v, causal=True, emulate_bf16=True)
    ge = oracle.attn_bwd(q, k, v, do, fe["lse"], oracle.attn_delta(fe["o"], do, emulate_bf16=True),
                         causal=True, emulate_bf16=True)
    for name in ("dq", "dk", "dv"):
        assert _rel(ge[name], g[name]) < 1e-2, name


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_rows_are_rows_of_the_full_backward(causal):
    # attn_bwd_rows is attn_bwd's dQ restricted to some rows (the sampled-row check of long
    # sequences); attn_bwd is pinned by finite differences and autograd above.
    t = inputs.gaussian(1, 2, 1, 70, 16, std_qkv=1.0, seed=12)
    q, k, v, do = (_np(t[n]) for n in ("q", "k", "v", "do"))
    f = oracle.attn_fwd(q, k, v, causal=causal, scale=0.25, fix_mode=1)
    dl = oracle.attn_delta(f["o"], do)
    g = oracle.attn_bwd(q, k, v, do, f["lse"], dl, causal=causal, scale=0.25)
    rows = np.array([0, 1, 17, 33, 69])
    for h in range(2):
        dq = oracle.attn_bwd_rows(q[0, h, rows], k[0, 0], v[0, 0], do[0, h, rows],
                                  f["lse"][0, h, rows], dl[0, h, rows], rows, causal=causal,
                                  scale=0.25)
        np.testing.assert_allclose(dq, g["dq"][0, h, rows], rtol=0, atol=1e-12)
