"""GPU checks of the forward kernel's study variants against the oracle: the monitor (the
operational count of BF16 Pbar == 1 handed to the product and the tie-multiplicity
histogram, bit-exact on integer inputs) and the unfused BF16 profile (an implementation that
stores Pbar V in BF16, the paper's analysed code), whose rounding bias on tied maxima the
fix removes."""
import math

import numpy as np
import pytest
import torch

import oracle
import precision_flash_attention_gb300 as pfa
from precision_flash_attention_gb300 import inputs
from tests.gpu_helpers import assert_fwd_close, f64, rel_l2, to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    pfa.device_error(clear=True)


def _fwd(t, **kw):
    d = to_dev(t)
    cnt, mon = pfa.new_counters(), pfa.new_monitor()
    o, lse = pfa.forward(d["q"], d["k"], d["v"], counters=cnt, monitor=mon, **kw)
    o2, lse2 = pfa.forward(d["q"], d["k"], d["v"], counters=pfa.new_counters(),
                           **{n: x for n, x in kw.items() if n != "unfused_bf16_pv"})
    torch.cuda.synchronize()
    assert pfa.device_error(clear=True) == 0
    c = cnt.cpu().tolist()
    m = mon.cpu().tolist()
    return {"o": o, "lse": lse, "o_fused": o2, "lse_fused": lse2,
            "counters": {"repeated_rows": c[0], "ones": c[1], "nonfinite_rows": c[2]},
            "operational_ones": m[0], "tie_hist": np.array(m[1:])}


GRID_SHAPES = [(1, 1, 1, 64, 64, False), (1, 2, 1, 300, 64, True), (2, 4, 2, 200, 128, True),
               (1, 2, 2, 257, 128, False), (1, 3, 1, 512, 64, True)]


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("shape", GRID_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_monitor_bit_exact_on_integer_grids(shape, mode):
    B, Hq, Hkv, N, d, causal = shape
    t = inputs.integer_grid(B, Hq, Hkv, N, d, causal=causal, n_planted=8, seed=N + d + mode)
    kw = dict(causal=causal, scale=0.125, fix_mode=mode, beta=2.0, eps=1e-3)
    got = _fwd(t, **kw)
    q, k, v = (f64(t[n]) for n in ("q", "k", "v"))
    ref = oracle.attn_fwd_monitor(q, k, v, **kw)
    emu = oracle.attn_fwd(q, k, v, emulate_bf16=True, **kw)
    assert got["operational_ones"] == ref["operational_ones"]
    assert np.array_equal(got["tie_hist"], ref["tie_hist"])
    assert got["counters"] == emu["counters"]
    # The monitor counts alongside the fused computation: O and lse are the fused path's, bit
    # for bit (rows that underflow under the beta shift are NaN in both).
    assert torch.equal(got["o"].view(torch.int16), got["o_fused"].view(torch.int16))
    assert torch.equal(got["lse"].view(torch.int32), got["lse_fused"].view(torch.int32))


@pytest.mark.parametrize("sign", [-1, 0])
@pytest.mark.parametrize("mode", [1, 2])
def test_monitor_on_nonpositive_maxima(sign, mode):
    t = inputs.signed_max_grid(1, 2, 1, 300, 64, sign=sign, n_keys=3, seed=5)
    kw = dict(causal=True, scale=0.125, fix_mode=mode, beta=2.0, eps=1e-3)
    got = _fwd(t, **kw)
    ref = oracle.attn_fwd_monitor(*(f64(t[n]) for n in ("q", "k", "v")), **kw)
    assert got["operational_ones"] == ref["operational_ones"]
    assert np.array_equal(got["tie_hist"], ref["tie_hist"])


def test_monitor_on_gaussian_inputs_is_consistent():
    # On float inputs the histogram covers every row once, its repeated bins are the
    # repeated-row counter, and in mode 0 every exact one of the final shift was handed to the
    # product in its own tile.
    t = inputs.gaussian(2, 4, 4, 1000, 64, std_qkv=0.5, std_do=1e-2, seed=2)
    got = _fwd(t, causal=True, scale=0.125, fix_mode=0)
    assert got["tie_hist"].sum() == 2 * 4 * 1000
    assert got["tie_hist"][1:].sum() == got["counters"]["repeated_rows"]
    assert got["operational_ones"] >= got["counters"]["ones"]


# ---------------------------------------------------------------- unfused BF16 profile
def _bias_ulp(o, ref, first_row):
    ulp = 2.0 ** (np.floor(np.log2(np.abs(ref))) - 7)
    return float(((o - ref) / ulp)[..., first_row:, :].mean())


@pytest.mark.parametrize("shape", [(1, 2, 1, 300, 64, True), (1, 2, 2, 129, 64, False),
                                   (2, 2, 1, 700, 64, True)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_unfused_profile_matches_oracle(shape, mode):
    B, Hq, Hkv, N, d, causal = shape
    t = inputs.gaussian(B, Hq, Hkv, N, d, std_qkv=0.7, std_do=1.0, seed=N + mode)
    kw = dict(causal=causal, scale=0.125, fix_mode=mode, beta=2.0, eps=1e-3)
    got = _fwd(t, unfused_bf16_pv=True, **kw)
    q, k, v = (f64(t[n]) for n in ("q", "k", "v"))
    ref = oracle.attn_fwd_unfused(q, k, v, block=128, **kw)
    assert_fwd_close({"o": f64(got["o"]), "lse": f64(got["lse"])}, ref, f"profile {shape}")
    # Each tile's BF16 roundings happen on values within FP32 rounding of the oracle's: the
    # two differ in a few BF16 ulps of Obar at most.
    assert rel_l2(f64(got["o"]), ref["o"]) < 2e-3


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_unfused_profile_bias_and_its_removal(mode):
    # Rows whose maximum is a sink key repeated twice over negative-dominated value features:
    # the unfused profile's O carries a negative bias in mode 0 (two exact ones summed in
    # BF16, priors.kr core idea, paper §3.3.2) that modes 1 and 2 remove; the GPU profile
    # and the oracle's agree on it.
    t = inputs.tie_probe(1, 4, 1024, 64, ties=2, seed=0)
    kw = dict(causal=True, scale=0.125, fix_mode=mode, beta=2.0, eps=1e-3)
    got = _fwd(t, unfused_bf16_pv=True, **kw)
    q, k, v = (f64(t[n]) for n in ("q", "k", "v"))
    exact = oracle.attn_fwd(q, k, v, causal=True, scale=0.125)["o"]
    ref = oracle.attn_fwd_unfused(q, k, v, block=128, **kw)
    b_gpu, b_ref = _bias_ulp(f64(got["o"]), exact, 2), _bias_ulp(ref["o"], exact, 2)
    b_fused = _bias_ulp(f64(got["o_fused"]), exact, 2)
    emu = oracle.attn_fwd(q, k, v, emulate_bf16=True, **kw)
    b_emu = _bias_ulp(emu["o"], exact, 2)
    print(f"mode {mode}: mean O error in BF16 ulps -- unfused GPU {b_gpu:+.4f}, unfused oracle "
          f"{b_ref:+.4f}; fused GPU {b_fused:+.4f}, fused emulation {b_emu:+.4f}")
    assert abs(b_gpu - b_ref) < 0.02
    if mode == 0:
        assert b_gpu < -0.08
        # The fused path (FP32 accumulation, one rounding of O) keeps a smaller bias of its
        # own: (V_a + V_b) / 2 sits on a BF16 midpoint for half the features, and which way it
        # rounds is decided by the last bits of the tensor core's FP32 sum, which the oracle's
        # exact sum does not reproduce.
        assert abs(b_fused) < 0.5 * abs(b_gpu)
    else:
        assert abs(b_gpu) < 0.03
        # Mode 2 scales O by bf16(exp(-2^-5)) / exp(-2^-5) on these rows (l sums the FP32 Pbar,
        # the product uses its BF16 cast), a bias the emulation reproduces.
        assert abs(b_fused - b_emu) < 0.03


def test_unfused_profile_rejects_d128_and_unknown_flags():
    t = to_dev(inputs.gaussian(1, 1, 1, 64, 128, seed=0))
    o = torch.empty_like(t["q"])
    lse = torch.empty(t["q"].shape[:3], dtype=torch.float32, device="cuda")
    with pytest.raises(pfa.PfaError, match="UNSUPPORTED"):
        pfa.attn_fwd_ex(t["q"], t["k"], t["v"], o, lse, causal=False, scale=0.1, flags=1)
    with pytest.raises(pfa.PfaError, match="INVALID_ARG"):
        pfa.attn_fwd_ex(t["q"], t["k"], t["v"], o, lse, causal=False, scale=0.1, flags=16)
    with pytest.raises(pfa.PfaError, match="UNSUPPORTED"):
        pfa.attn_fwd_ex(t["q"], t["k"], t["v"], o, lse, causal=False, scale=0.1, flags=2)
    assert pfa.device_error() == 0


# ---------------------------------------------------------------- narrower Pbar formats
@pytest.mark.parametrize("profile", [False, True], ids=["fused", "unfused"])
@pytest.mark.parametrize("pbar", ["e4m3", "mxfp4"])
@pytest.mark.parametrize("shape", [(1, 2, 1, 300, 64, True), (1, 2, 2, 257, 64, False),
                                   (2, 2, 1, 700, 64, True)], ids=lambda s: "x".join(map(str, s)))
def test_narrow_pbar_matches_oracle(shape, pbar, profile):
    # Pbar rounded to FP8 E4M3 or MXFP4 before the product, Obar in FP32 (fused) or in BF16 per
    # key tile (the unfused profile), against the oracle's blockwise pass over 128-key blocks.
    B, Hq, Hkv, N, d, causal = shape
    t = inputs.gaussian(B, Hq, Hkv, N, d, std_qkv=0.7, std_do=1.0, seed=N + len(pbar))
    for mode in (0, 1, 2):
        kw = dict(causal=causal, scale=0.125, fix_mode=mode, beta=2.0, eps=1e-3)
        got = _fwd(t, unfused_bf16_pv=profile, pbar=pbar, **kw)
        q, k, v = (f64(t[n]) for n in ("q", "k", "v"))
        ref = oracle.attn_fwd_blockwise(q, k, v, block=128, pbar=pbar,
                                        accumulate="bf16" if profile else "fp32", **kw)
        assert_fwd_close({"o": f64(got["o"]), "lse": f64(got["lse"])}, ref, f"{pbar} {shape} {mode}")
        assert got["operational_ones"] == ref["operational_ones"]


@pytest.mark.parametrize("pbar", ["e4m3", "mxfp4"])
def test_narrow_pbar_on_tied_maxima(pbar):
    # The tie probe (a sink key repeated twice, logit 16): in E4M3 mode 2's shift exp(-2^-5)
    # rounds back to exactly 1, so the product sees as many ones as without the fix, and mode
    # 1's beta shift (e^-16) falls below E4M3's range, leaving l = 0; MXFP4's block scale keeps
    # mode 1 finite and saturates mode 2's 0.969 to 0.75. The GPU counts and NaN rows match the
    # oracle's.
    t = inputs.tie_probe(1, 2, 512, 64, ties=2, seed=4)
    q, k, v = (f64(t[n]) for n in ("q", "k", "v"))
    res = {}
    for mode in (0, 1, 2):
        kw = dict(causal=True, scale=0.125, fix_mode=mode, beta=2.0, eps=1e-3)
        got = _fwd(t, pbar=pbar, **kw)
        ref = oracle.attn_fwd_blockwise(q, k, v, block=128, pbar=pbar, accumulate="fp32", **kw)
        nan_g = np.isnan(f64(got["o"])).any(axis=-1)
        nan_r = np.isnan(ref["o"]).any(axis=-1)
        assert np.array_equal(nan_g, nan_r)
        assert got["operational_ones"] == ref["operational_ones"]
        res[mode] = (got["operational_ones"], int(nan_g.sum()))
    print(f"{pbar}: operational ones / NaN rows per mode {res}")
    if pbar == "e4m3":
        assert res[2][0] == res[0][0] > 0 and res[1][1] > 0.9 * 2 * 512
    else:
        assert res[2][0] < res[0][0] and res[1][1] == 0
