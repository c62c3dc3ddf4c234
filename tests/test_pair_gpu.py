"""GPU parity of the forward pass with the two CTAs of a cluster paired on every product
(PFA_FWD_PAIR_CTA, tcgen05 cta_group::2, d = 128): O and lse against the float64 oracle with
the contract's tolerances, the counters bit-exact on integer grids, and the outputs against the
one-CTA path on the same inputs. The shapes cover every remainder of the query-tile count
modulo four (an item is four query tiles, two per CTA), sequences shorter than one half key
tile, grouped heads and more items than clusters."""
import numpy as np
import pytest
import torch

import oracle
import precision_flash_attention_gb300 as pfa
from precision_flash_attention_gb300 import inputs
from gpu_helpers import assert_fwd_close, f64, sampled_rows, to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    pfa.device_error(clear=True)


def _both(t, **kw):
    """The paired and the one-CTA forward on the same device inputs."""
    d = to_dev(t)
    out = {}
    for name, pair in (("pair", True), ("one", False)):
        cnt = pfa.new_counters()
        o, lse = pfa.forward(d["q"], d["k"], d["v"], counters=cnt, pair_cta=pair, **kw)
        out[name] = (o, lse, cnt)
    torch.cuda.synchronize()
    assert pfa.device_error(clear=True) == 0
    res = {}
    for name, (o, lse, cnt) in out.items():
        c = cnt.cpu().tolist()
        res[name] = {"o": o, "lse": lse,
                     "counters": {"repeated_rows": c[0], "ones": c[1], "nonfinite_rows": c[2]}}
    return res


def _assert_matches_one_cta(res, where):
    # Each row's products add the same terms in the same order of the K dimension; the
    # pairing only changes which SM's tensor core holds the row.
    a, b = res["pair"], res["one"]
    assert torch.equal(a["o"].view(torch.int16), b["o"].view(torch.int16)), f"{where}: O differs"
    assert torch.equal(a["lse"].view(torch.int32), b["lse"].view(torch.int32)), f"{where}: lse differs"
    assert a["counters"] == b["counters"], (where, a["counters"], b["counters"])


# (B, H_q, H_kv, N, causal): query tiles modulo 4 = 1, 2, 3, 0, 1 (N < 64: the odd CTA's K
# half is past the end), 1 (N = 1), 0 with 8 tiles (two items per head), and GQA.
SHAPES = [(1, 2, 1, 300, True), (1, 2, 2, 129, True), (2, 4, 2, 640, True), (1, 2, 2, 512, False),
          (1, 1, 1, 50, False), (1, 2, 1, 1, True), (1, 4, 4, 1000, True), (2, 8, 2, 384, False)]


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}Hq{}Hkv{}N{}-{}".format(*s[:4], "causal" if s[4] else "full"))
def test_pair_matches_oracle(shape, mode):
    B, Hq, Hkv, N, causal = shape
    t = inputs.gaussian(B, Hq, Hkv, N, 128, std_qkv=0.8, std_do=1.0, seed=N + 7 * mode)
    kw = dict(causal=causal, scale=128 ** -0.5, fix_mode=mode, beta=2.0, eps=1e-3)
    res = _both(t, **kw)
    ref = oracle.attn_fwd(*(f64(t[n]) for n in ("q", "k", "v")), **kw)
    got = {n: f64(res["pair"][n]) for n in ("o", "lse")}
    assert_fwd_close(got, ref, f"pair {shape} mode {mode}")
    assert res["pair"]["counters"]["nonfinite_rows"] == 0
    _assert_matches_one_cta(res, f"{shape} mode {mode}")


@pytest.mark.parametrize("mode", [0, 2])
@pytest.mark.parametrize("shape", [(1, 2, 1, 300, True), (2, 2, 2, 777, True), (1, 3, 1, 640, False)],
                         ids=lambda s: "B{}Hq{}Hkv{}N{}".format(*s[:4]))
def test_pair_counters_bit_exact_on_integer_grids(shape, mode):
    B, Hq, Hkv, N, causal = shape
    t = inputs.integer_grid(B, Hq, Hkv, N, 128, causal=causal, n_planted=8, seed=N + mode)
    kw = dict(causal=causal, scale=0.125 * (64 / 128) ** 0.5, fix_mode=mode, beta=2.0, eps=1e-3)
    res = _both(t, **kw)
    ref = oracle.attn_fwd(*(f64(t[n]) for n in ("q", "k", "v")), **kw)
    assert res["pair"]["counters"] == ref["counters"]
    _assert_matches_one_cta(res, f"grid {shape} mode {mode}")


def test_pair_many_rounds_sampled_rows():
    # 2 x 16 heads x 4 items per head = 128 items: several serpentine rounds per cluster.
    B, Hq, Hkv, N = 2, 16, 4, 2048
    t = inputs.gaussian(B, Hq, Hkv, N, 128, std_qkv=0.8, std_do=1.0, seed=11)
    kw = dict(causal=True, scale=128 ** -0.5, fix_mode=1, beta=4.0, eps=1e-3)
    res = _both(t, **kw)
    _assert_matches_one_cta(res, "many rounds")
    rows = sampled_rows(N, 64, seed=3)
    o, lse = f64(res["pair"]["o"]), f64(res["pair"]["lse"])
    g = Hq // Hkv
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for b in range(B):
        for h in range(0, Hq, 3):
            r = oracle.attn_fwd_head(f64(t["q"][b, h]), f64(t["k"][b, h // g]), f64(t["v"][b, h // g]),
                                     rows=rows, **kw)
            got_o.append(o[b, h, rows])
            got_l.append(lse[b, h, rows])
            ref_o.append(r["o"])
            ref_l.append(r["lse"])
    assert_fwd_close({"o": np.concatenate(got_o), "lse": np.concatenate(got_l)},
                     {"o": np.concatenate(ref_o), "lse": np.concatenate(ref_l)}, "many rounds")


def test_pair_in_a_training_step():
    # The paired forward's O and lse feed the backward pass like the one-CTA path's.
    t = inputs.gaussian(1, 4, 2, 700, 128, std_qkv=0.8, std_do=1.0, seed=5)
    d = to_dev(t)
    kw = dict(causal=True, scale=128 ** -0.5)
    o, lse = pfa.forward(d["q"], d["k"], d["v"], fix_mode=1, pair_cta=True, **kw)
    grads = pfa.backward(d["q"], d["k"], d["v"], o, lse, d["do"], **kw)
    o1, lse1 = pfa.forward(d["q"], d["k"], d["v"], fix_mode=1, **kw)
    grads1 = pfa.backward(d["q"], d["k"], d["v"], o1, lse1, d["do"], dq_mode="deterministic", **kw)
    grads2 = pfa.backward(d["q"], d["k"], d["v"], o, lse, d["do"], dq_mode="deterministic", **kw)
    torch.cuda.synchronize()
    assert pfa.device_error(clear=True) == 0
    for a, b in zip(grads1, grads2):
        assert torch.equal(a, b)
    assert all(torch.isfinite(x.float()).all() for x in grads)


def test_pair_flag_is_refused_where_not_built():
    t = to_dev(inputs.gaussian(1, 1, 1, 64, 64, seed=0))
    o = torch.empty_like(t["q"])
    lse = torch.empty(t["q"].shape[:3], dtype=torch.float32, device="cuda")
    with pytest.raises(pfa.PfaError, match="UNSUPPORTED"):      # d = 64
        pfa.attn_fwd_ex(t["q"], t["k"], t["v"], o, lse, causal=False, scale=0.1, flags=pfa.FWD_PAIR_CTA)
    t = to_dev(inputs.gaussian(1, 1, 1, 64, 128, seed=0))
    o = torch.empty_like(t["q"])
    with pytest.raises(pfa.PfaError, match="UNSUPPORTED"):      # with the monitor
        pfa.attn_fwd_ex(t["q"], t["k"], t["v"], o, lse, causal=False, scale=0.1, monitor=pfa.new_monitor(),
                        flags=pfa.FWD_PAIR_CTA)
    assert pfa.device_error() == 0


def test_pair_forward_in_a_cuda_graph():
    # The paired forward is a cluster launch chained by programmatic dependent launch; it
    # captures into a CUDA graph with a backward call after it, and the replay gives the
    # eager results (dQ by the deterministic pass, so bit for bit).
    t = to_dev(inputs.gaussian(1, 4, 2, 700, 128, std_qkv=0.7, std_do=1.0, seed=13))
    q, k, v, do = t["q"], t["k"], t["v"], t["do"]
    o, lse = torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    delta = torch.empty_like(lse)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    kw = dict(causal=True, scale=128 ** -0.5)

    def step():
        pfa.attn_fwd_ex(q, k, v, o, lse, fix_mode=1, beta=2.0, eps=1e-3, flags=pfa.FWD_PAIR_CTA, **kw)
        pfa.attn_delta(o, do, delta)
        pfa.attn_bwd_ex(q, k, v, do, lse, delta, dq, dk, dv, None, flags=pfa.BWD_DQ_DETERMINISTIC, **kw)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [x.clone() for x in (o, lse, dq, dk, dv)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for x in (o, lse, dq, dk, dv):
        x.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert pfa.device_error(clear=True) == 0
    for a, b in zip(eager, (o, lse, dq, dk, dv)):
        assert torch.equal(a, b)
