"""Seeded synthetic inputs for the attention workloads.

This module only draws numbers: it holds none of the attention arithmetic, and
both the CUDA path's tests and the CPU oracle's tests take their inputs from
it. Everything is drawn on the CPU with ``torch.Generator`` and returned as
contiguous BF16 CPU tensors in [B, H, N, d] layout (d innermost).

Workloads (the pages train GPT-2 Small on OpenWebText and inspect Llama 3.1 8B;
neither dataset nor weights are available, so these tensors stand in for the
shapes and value structure only):

* ``tiny``  B=1, H=1, N=64, d=64, non-causal; Q, K, V ~ N(0, 1).
* ``grid``  integer-valued Q, K in [-4, 4] with planted duplicated-maximum keys,
  so that every score is an exact multiple of 1/8 and ties are exact.
* ``gpt2``  GPT-2-small attention layer: B=8, H=12, N=1024, d=64, causal;
  Q, K, V ~ N(0, 1) * 0.5, dO ~ N(0, 1e-2^2).
* ``sink``  B=4, H=12, N=2048, d=64, causal; key 0 carries an exact +6 logit
  (through a reserved last feature), 10% of the rows get a copied argmax key,
  V features have negative means.
* ``long``  B=2, H=16, N=8192, d=128, causal; Q, K, V ~ N(0, 1) * 0.3.
* ``gqa``   Llama-3.1-8B-style GQA: B=1, H_q=32, H_kv=8, N=8192, d=128,
  causal; as ``long`` with 5% of the query rows scaled by 8.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = ["Workload", "WORKLOADS", "make", "gaussian", "integer_grid", "signed_max_grid",
           "sink_heavy", "tie_probe", "large_logit_rows", "underflow_probe"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H_q: int
    H_kv: int
    N: int
    d: int
    causal: bool
    modes: tuple = (0, 1, 2)
    beta: float = 2.0
    eps: float = 1e-3
    scale: float | None = None
    extra: dict = field(default_factory=dict)

    @property
    def alpha(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.d)

    def flops(self, which: str = "fwd+bwd") -> float:
        """Algorithmic FLOPs of the contractions: 4 B H_q N^2 d forward (S and
        Pbar V), 10 B H_q N^2 d backward (S, dP, dV, dK, dQ), halved if causal."""
        per = {"fwd": 4.0, "bwd": 10.0, "fwd+bwd": 14.0, "delta_alt": 4.0}[which]
        f = per * self.B * self.H_q * self.N * self.N * self.d
        return f / 2 if self.causal else f


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 1, 64, 64, False, scale=0.125),
    "gpt2": Workload("gpt2", 8, 12, 12, 1024, 64, True, modes=(0, 1), scale=0.125),
    "sink": Workload("sink", 4, 12, 12, 2048, 64, True, scale=0.125),
    "long": Workload("long", 2, 16, 16, 8192, 128, True, modes=(1,), beta=4.0),
    "gqa": Workload("gqa", 1, 32, 8, 8192, 128, True),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, g, mean=0.0) -> torch.Tensor:
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std + mean)


def gaussian(B, H_q, H_kv, N, d, *, std_qkv=1.0, std_do=1.0, seed=0) -> dict:
    """Q, K, V ~ N(0, std_qkv^2) and dO ~ N(0, std_do^2), rounded to BF16."""
    g = _gen(seed)
    q = _normal((B, H_q, N, d), std_qkv, g)
    k = _normal((B, H_kv, N, d), std_qkv, g)
    v = _normal((B, H_kv, N, d), std_qkv, g)
    do = _normal((B, H_q, N, d), std_do, g)
    return {n: t.to(torch.bfloat16).contiguous() for n, t in
            (("q", q), ("k", k), ("v", v), ("do", do))}


def integer_grid(B, H_q, H_kv, N, d, *, causal=False, n_planted=8, seed=0) -> dict:
    """Integer Q, K uniform in [-4, 4]; V, dO ~ N(0, 1).

    ``n_planted`` rows per query head get a duplicated maximum: two unused keys
    j1 != j2 (both <= i when causal) are set to 4*sign(q_i) (sign(0) = +1), the
    largest score any key in [-4, 4]^d can reach against q_i, so the row's
    maximum occurs at least twice. With scale 1/8 every score is an exact
    multiple of 1/8 in FP32 and FP64.
    """
    g = _gen(seed)
    q = torch.randint(-4, 5, (B, H_q, N, d), generator=g).to(torch.float32)
    k = torch.randint(-4, 5, (B, H_kv, N, d), generator=g).to(torch.float32)
    v = _normal((B, H_kv, N, d), 1.0, g)
    do = _normal((B, H_q, N, d), 1.0, g)
    group = H_q // H_kv
    for b in range(B):
        for h in range(H_q):
            kv = h // group
            used: set[int] = set()
            lo = 1 if causal else 0
            cand = torch.randperm(N - lo, generator=g)[: 4 * n_planted] + lo
            planted = 0
            for i in cand.tolist():
                if planted == n_planted:
                    break
                pool = [j for j in range(0, (i + 1) if causal else N) if j not in used]
                if len(pool) < 2:
                    continue
                pick = torch.randperm(len(pool), generator=g)[:2].tolist()
                j1, j2 = pool[pick[0]], pool[pick[1]]
                sgn = torch.where(q[b, h, i] >= 0, 4.0, -4.0)
                k[b, kv, j1] = sgn
                k[b, kv, j2] = sgn
                used.update((j1, j2))
                planted += 1
    return {"q": q.to(torch.bfloat16).contiguous(), "k": k.to(torch.bfloat16).contiguous(),
            "v": v.to(torch.bfloat16).contiguous(), "do": do.to(torch.bfloat16).contiguous()}


def signed_max_grid(B, H_q, H_kv, N, d, *, sign, n_keys=2, seed=0) -> dict:
    """Integer inputs whose row maxima are negative (``sign=-1``) or exactly zero (``sign=0``)
    and repeated.

    Q is binary ({0, 1}, feature 0 always 1 for ``sign=-1``) and K holds integers in
    [-3, -1], so every score q.k is negative. ``n_keys`` seed-chosen keys per key/value head
    become the row maximum for every query that sees them: the zero vector (score exactly 0)
    for ``sign=0``, the all -1 vector (score -(number of ones of q), the largest any key in
    [-3, -1]^d can reach) for ``sign=-1``. With a scale of 1/8 every score is an exact
    multiple of 1/8 in FP32 and FP64, so ties are exact. V, dO ~ N(0, 1).
    """
    if sign not in (-1, 0):
        raise ValueError("sign must be -1 or 0")
    g = _gen(seed)
    q = torch.randint(0, 2, (B, H_q, N, d), generator=g).to(torch.float32)
    if sign < 0:
        q[..., 0] = 1.0
    k = torch.randint(-3, 0, (B, H_kv, N, d), generator=g).to(torch.float32)
    for b in range(B):
        for h in range(H_kv):
            for j in torch.randperm(N, generator=g)[:n_keys].tolist():
                k[b, h, j] = 0.0 if sign == 0 else -1.0
    v = _normal((B, H_kv, N, d), 1.0, g)
    do = _normal((B, H_q, N, d), 1.0, g)
    return {n: t.to(torch.bfloat16).contiguous() for n, t in
            (("q", q), ("k", k), ("v", v), ("do", do))}


# Planted score patterns over two 128-key tiles (raw scores K / 8 for one-hot
# queries). Each entry: (keys of tile 0 set to a value, keys of tile 1 set to a
# value); every other key stays at or below 4 (score <= 0.5).
TIE_PATTERNS = {
    "jump_same_block": ({10: 8.0}, {128 + 3: 16.0, 128 + 5: 15.875}),
    "jump_same_class": ({10: 8.0}, {128 + 3: 16.0, 128 + 19: 15.875}),
    "jump_block_and_class": ({10: 8.0}, {128 + 3: 16.0, 128 + 40: 15.875}),
    "jump_single": ({10: 8.0}, {128 + 3: 16.0}),
    "jump_near_miss": ({10: 8.0}, {128 + 3: 16.0, 128 + 5: 15.5}),
    "jump_exact_pair": ({10: 8.0}, {128 + 3: 16.0, 128 + 4: 16.0}),
    "tie_below_running_max": ({10: 16.0}, {128 + 7: 15.875}),
    "rise_within_eps": ({10: 15.875}, {128 + 7: 16.0}),
}


def tie_patterns(names, N=256, d=64, *, seed=0) -> dict:
    """B=1, H=1 input whose query row i has the key scores of pattern names[i % len(names)]
    (TIE_PATTERNS): query i is one-hot on feature i % len(names), and feature f of the
    keys holds pattern f. Background keys are integers in [-16, 4]; V, dO ~ N(0, 1).
    With scale 1/8 the planted scores are 1.0, 2.0, 2.0 - 2^-6 and 2.0 - 2^-4, exact in
    BF16, FP32 and FP64."""
    assert N >= 256 and d >= len(names)
    g = _gen(seed)
    q = torch.zeros(1, 1, N, d)
    for i in range(N):
        q[0, 0, i, i % len(names)] = 1.0
    k = torch.randint(-16, 5, (1, 1, N, d), generator=g).to(torch.float32)
    for f, name in enumerate(names):
        t0, t1 = TIE_PATTERNS[name]
        for j, x in list(t0.items()) + list(t1.items()):
            k[0, 0, j, f] = x
    v = _normal((1, 1, N, d), 1.0, g)
    do = _normal((1, 1, N, d), 1.0, g)
    return {"q": q.to(torch.bfloat16).contiguous(), "k": k.to(torch.bfloat16).contiguous(),
            "v": v.to(torch.bfloat16).contiguous(), "do": do.to(torch.bfloat16).contiguous()}


def sink_heavy(B=4, H=12, N=2048, d=64, *, seed=0, dup_frac=0.10) -> dict:
    """The sink-heavy stress input (scale 1/8).

    * base Q, K, V ~ N(0, 0.25), dO ~ N(0, 1e-4);
    * an exact +6 logit on key 0: feature d-1 is reserved, Q[..., d-1] = 1,
      K[..., 0, d-1] = 48 (= 6 / (1/8), exact in BF16), K[..., j>0, d-1] = 0;
    * ``dup_frac`` of the rows i >= 1 (seed-chosen) get a duplicated maximum:
      the row's argmax key j* over the causal range is copied into a seed-chosen
      key j' <= i, j' != j* (sequentially; identical key rows tie exactly);
    * V feature f ~ N(mu_f, 0.25) with mu_f ~ N(-1, 0.01) (negative-dominated
      value features, as in the paper's feature 20).
    """
    g = _gen(seed)
    q = _normal((B, H, N, d), 0.5, g)
    k = _normal((B, H, N, d), 0.5, g)
    mu = _normal((B, H, 1, d), 0.1, g, mean=-1.0)
    v = _normal((B, H, N, d), 0.5, g) + mu
    do = _normal((B, H, N, d), 1e-2, g)
    q = q.to(torch.bfloat16).float()
    k = k.to(torch.bfloat16).float()
    q[..., d - 1] = 1.0
    k[..., d - 1] = 0.0
    k[..., 0, d - 1] = 48.0
    n_dup = max(1, int(round(dup_frac * (N - 1))))
    for b in range(B):
        for h in range(H):
            rows = (torch.randperm(N - 1, generator=g)[:n_dup] + 1).tolist()
            s = q[b, h, rows] @ k[b, h].T
            for r, i in enumerate(rows):
                js = int(torch.argmax(s[r, : i + 1]).item())
                jp = int(torch.randint(0, i, (1,), generator=g).item())
                if jp >= js:
                    jp += 1
                k[b, h, jp] = k[b, h, js]
    return {"q": q.to(torch.bfloat16).contiguous(), "k": k.to(torch.bfloat16).contiguous(),
            "v": v.to(torch.bfloat16).contiguous(), "do": do.to(torch.bfloat16).contiguous()}


def tie_probe(B=1, H=12, N=1024, d=64, *, ties=2, logit=16.0, seed=0) -> dict:
    """Rows whose maximum is a sink key repeated ``ties`` times (scale 1/8).

    * base Q, K ~ N(0, 0.25), dO ~ N(0, 1e-4);
    * key 0 carries an exact +``logit`` (feature d-1 reserved: Q[..., d-1] = 1,
      K[..., 0, d-1] = logit * 8, K[..., j>0, d-1] = 0), and keys 1 .. ties-1 are copies of
      key 0, so every row i >= ties - 1 has exactly ``ties`` tied maxima; with a logit of 16
      the other keys' weights are e^-16 each, so their sum stays far below a BF16 spacing
      of the output;
    * V feature f ~ N(mu_f, 0.25) with mu_f ~ N(-1, 0.01): negative-dominated features.
    """
    g = _gen(seed)
    q = _normal((B, H, N, d), 0.5, g)
    k = _normal((B, H, N, d), 0.5, g)
    mu = _normal((B, H, 1, d), 0.1, g, mean=-1.0)
    v = _normal((B, H, N, d), 0.5, g) + mu
    do = _normal((B, H, N, d), 1e-2, g)
    q = q.to(torch.bfloat16).float()
    k = k.to(torch.bfloat16).float()
    q[..., d - 1] = 1.0
    k[..., d - 1] = 0.0
    k[..., 0, d - 1] = logit * 8.0
    for t in range(1, ties):
        k[..., t, :] = k[..., 0, :]
    return {"q": q.to(torch.bfloat16).contiguous(), "k": k.to(torch.bfloat16).contiguous(),
            "v": v.to(torch.bfloat16).contiguous(), "do": do.to(torch.bfloat16).contiguous()}


def large_logit_rows(B=1, H_q=32, H_kv=8, N=8192, d=128, *, seed=0, frac=0.05,
                     factor=8.0) -> dict:
    """Q, K, V ~ N(0, 0.09), dO ~ N(0, 1e-4), with ``frac`` of the query rows
    (seed-chosen per head) multiplied by ``factor`` before rounding to BF16."""
    g = _gen(seed)
    t = gaussian(B, H_q, H_kv, N, d, std_qkv=0.3, std_do=1e-2, seed=seed + 1)
    sel = torch.rand((B, H_q, N, 1), generator=g) < frac
    q = t["q"].float()
    t["q"] = torch.where(sel, q * factor, q).to(torch.bfloat16).contiguous()
    return t


def underflow_probe(B=1, H=2, N=128, d=64, *, logit=200.0, seed=0) -> dict:
    """Rows with a repeated maximum of size ``logit`` and the rest far below it.

    Under mode 1 the shift beta*r_m then pushes every exponent argument below the
    FP32 range for ``logit`` large enough, so l underflows to 0 (paper App. C).
    Q row i = unit vector e_(i mod d) * sqrt(logit/scale), every key k_j = the
    same vector for two keys per row, small noise elsewhere.
    """
    g = _gen(seed)
    scale = 1.0 / math.sqrt(d)
    q = _normal((B, H, N, d), 0.01, g)
    k = _normal((B, H, N, d), 0.01, g)
    v = _normal((B, H, N, d), 1.0, g)
    do = _normal((B, H, N, d), 1.0, g)
    a = math.sqrt(logit / scale)
    for i in range(N):
        f = i % d
        q[:, :, i, :] = 0.0
        q[:, :, i, f] = a
    for f in range(min(d, N // 2)):
        k[:, :, 2 * f, :] = 0.0
        k[:, :, 2 * f + 1, :] = 0.0
        k[:, :, 2 * f, f] = a
        k[:, :, 2 * f + 1, f] = a
    return {n: t.to(torch.bfloat16).contiguous() for n, t in
            (("q", q), ("k", k), ("v", v), ("do", do))}


def make(name: str, seed: int = 0) -> dict:
    """Inputs of a named workload (``tiny``, ``grid``, ``gpt2``, ``sink``, ``long``, ``gqa``)."""
    if name == "tiny":
        return gaussian(1, 1, 1, 64, 64, std_qkv=1.0, std_do=1.0, seed=seed)
    if name == "grid":
        return integer_grid(1, 1, 1, 64, 64, causal=False, n_planted=8, seed=seed)
    if name == "gpt2":
        return gaussian(8, 12, 12, 1024, 64, std_qkv=0.5, std_do=1e-2, seed=seed)
    if name == "sink":
        return sink_heavy(4, 12, 2048, 64, seed=seed)
    if name == "long":
        return gaussian(2, 16, 16, 8192, 128, std_qkv=0.3, std_do=1e-2, seed=seed)
    if name == "gqa":
        return large_logit_rows(1, 32, 8, 8192, 128, seed=seed)
    raise KeyError(name)
