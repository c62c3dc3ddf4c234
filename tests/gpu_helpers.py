"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI, run the
oracle on the same seeded inputs, and compare with the float tolerances of the contract:
O and lse rel-L2 <= 4e-3 and max-abs <= 1.5e-2; dQ, dK, dV (and delta) rel-L2 <= 1e-2."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import precision_flash_attention_gb300 as pfa

TOL_FWD_REL = 4e-3
TOL_FWD_ABS = 1.5e-2
TOL_BWD_REL = 1e-2


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def to_dev(t: dict) -> dict:
    return {n: x.cuda() for n, x in t.items()}


def run_gpu(t: dict, *, causal, scale, fix_mode, beta=2.0, eps=1e-3, bwd=True, delta_mode=0,
            dq_mode="atomic", pair_cta=False):
    """Forward (+ delta + backward) on the GPU; returns numpy float64 results and counters.
    ``pair_cta``: the forward with two CTAs per product (d = 128)."""
    d = to_dev(t)
    cnt = pfa.new_counters()
    o, lse = pfa.forward(d["q"], d["k"], d["v"], causal=causal, scale=scale, fix_mode=fix_mode,
                         beta=beta, eps=eps, counters=cnt, pair_cta=pair_cta)
    out = {"o": o, "lse": lse}
    if bwd:
        dq, dk, dv, delta = pfa.backward(d["q"], d["k"], d["v"], o, lse, d["do"], causal=causal,
                                         scale=scale, delta_mode=delta_mode, dq_mode=dq_mode)
        out.update(dq=dq, dk=dk, dv=dv, delta=delta)
    torch.cuda.synchronize()
    assert pfa.device_error(clear=True) == 0
    res = {n: f64(x) for n, x in out.items()}
    c = cnt.cpu().tolist()
    res["counters"] = {"repeated_rows": c[0], "ones": c[1], "nonfinite_rows": c[2]}
    return res


def oracle_full(t: dict, *, causal, scale, fix_mode, beta=2.0, eps=1e-3, bwd=True):
    q, k, v, do = (f64(t[n]) for n in ("q", "k", "v", "do"))
    f = oracle.attn_fwd(q, k, v, causal=causal, scale=scale, fix_mode=fix_mode, beta=beta, eps=eps)
    out = {"o": f["o"], "lse": f["lse"], "counters": f["counters"]}
    if bwd:
        delta = oracle.attn_delta(f["o"], do)
        g = oracle.attn_bwd(q, k, v, do, f["lse"], delta, causal=causal, scale=scale)
        out.update(g, delta=delta)
    return out


def assert_fwd_close(got: dict, ref: dict, where: str = "") -> None:
    for n in ("o", "lse"):
        a, b = got[n], ref[n]
        assert np.isfinite(a).all(), f"{where} {n} has non-finite values"
        r = rel_l2(a, b)
        m = float(np.abs(a - b).max())
        assert r <= TOL_FWD_REL and m <= TOL_FWD_ABS, f"{where} {n}: rel-L2 {r:.3e}, max-abs {m:.3e}"


def assert_bwd_close(got: dict, ref: dict, where: str = "", names=("dq", "dk", "dv")) -> None:
    for n in names:
        a, b = got[n], ref[n]
        assert np.isfinite(a).all(), f"{where} {n} has non-finite values"
        r = rel_l2(a, b)
        assert r <= TOL_BWD_REL, f"{where} {n}: rel-L2 {r:.3e}"


def oracle_group(t: dict, b: int, hk: int, *, causal, scale, fix_mode, beta=2.0, eps=1e-3):
    """Oracle forward + backward restricted to batch b and key/value head hk with all the
    query heads that read it (dK and dV sum over exactly those heads)."""
    Hq, Hkv = t["q"].shape[1], t["k"].shape[1]
    g = Hq // Hkv
    hs = slice(hk * g, (hk + 1) * g)
    q = f64(t["q"][b:b + 1, hs])
    do = f64(t["do"][b:b + 1, hs])
    k = f64(t["k"][b:b + 1, hk:hk + 1])
    v = f64(t["v"][b:b + 1, hk:hk + 1])
    f = oracle.attn_fwd(q, k, v, causal=causal, scale=scale, fix_mode=fix_mode, beta=beta, eps=eps)
    delta = oracle.attn_delta(f["o"], do)
    gr = oracle.attn_bwd(q, k, v, do, f["lse"], delta, causal=causal, scale=scale)
    return {"o": f["o"][0], "lse": f["lse"][0], "delta": delta[0], "dq": gr["dq"][0],
            "dk": gr["dk"][0, 0], "dv": gr["dv"][0, 0], "counters": f["counters"], "heads": hs}


def oracle_group_emulated(t: dict, b: int, hk: int, *, causal, scale, fix_mode, beta=2.0, eps=1e-3,
                          delta_mode=0):
    """The BF16-emulating oracle (the kernel's cast points: FP32 scores, BF16 P / dS operands,
    BF16 outputs) on one key/value-head group; delta from the emulated O (delta_mode 0) or as
    rowsum(dP o P) (delta_mode 1)."""
    Hq, Hkv = t["q"].shape[1], t["k"].shape[1]
    g = Hq // Hkv
    hs = slice(hk * g, (hk + 1) * g)
    q = f64(t["q"][b:b + 1, hs])
    do = f64(t["do"][b:b + 1, hs])
    k = f64(t["k"][b:b + 1, hk:hk + 1])
    v = f64(t["v"][b:b + 1, hk:hk + 1])
    f = oracle.attn_fwd(q, k, v, causal=causal, scale=scale, fix_mode=fix_mode, beta=beta, eps=eps,
                        emulate_bf16=True)
    if delta_mode == 0:
        delta = oracle.attn_delta(f["o"], do, emulate_bf16=True)
    else:
        delta = oracle.attn_delta_alt(q, k, v, do, f["lse"], causal=causal, scale=scale,
                                      emulate_bf16=True)
    gr = oracle.attn_bwd(q, k, v, do, f["lse"], delta, causal=causal, scale=scale,
                         emulate_bf16=True)
    return {"o": f["o"][0], "lse": f["lse"][0], "dq": gr["dq"][0], "dk": gr["dk"][0, 0],
            "dv": gr["dv"][0, 0], "heads": hs}


def sampled_rows(N: int, n: int = 256, seed: int = 0) -> np.ndarray:
    """n query rows of a length-N sequence: the first and last 16 and a seeded random rest."""
    rng = np.random.default_rng(seed)
    edge = np.concatenate([np.arange(16), np.arange(N - 16, N)])
    mid = rng.choice(np.arange(16, N - 16), n - len(edge), replace=False)
    return np.sort(np.concatenate([edge, mid]))


def check_sampled_rows(t: dict, got: dict, rows, *, causal, scale, fix_mode, beta=2.0, eps=1e-3):
    """O, lse and dQ of the given rows of EVERY (batch, query head) against the float64 oracle
    (forward restricted to the rows, delta = rowsum(dO o O) of those rows, dQ rows)."""
    B, Hq = t["q"].shape[:2]
    g = Hq // t["k"].shape[1]
    acc = {n: ([], []) for n in ("o", "lse", "dq")}
    for b in range(B):
        for h in range(Hq):
            qh, doh = f64(t["q"][b, h]), f64(t["do"][b, h])
            kh, vh = f64(t["k"][b, h // g]), f64(t["v"][b, h // g])
            r = oracle.attn_fwd_head(qh, kh, vh, causal=causal, scale=scale, fix_mode=fix_mode,
                                     beta=beta, eps=eps, rows=rows)
            delta = oracle.attn_delta(r["o"][None, None], doh[rows][None, None])[0, 0]
            dq = oracle.attn_bwd_rows(qh[rows], kh, vh, doh[rows], r["lse"], delta, rows,
                                      causal=causal, scale=scale)
            for n, ref in (("o", r["o"]), ("lse", r["lse"]), ("dq", dq)):
                acc[n][0].append(got[n][b, h, rows])
                acc[n][1].append(ref)
    cat = {n: (np.concatenate(a), np.concatenate(r)) for n, (a, r) in acc.items()}
    assert_fwd_close({"o": cat["o"][0], "lse": cat["lse"][0]},
                     {"o": cat["o"][1], "lse": cat["lse"][1]}, "sampled rows")
    assert_bwd_close({"dq": cat["dq"][0]}, {"dq": cat["dq"][1]}, "sampled rows", names=("dq",))
