"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the same seeded
inputs. Float outputs within the contract tolerances; integer counters bit-exact on
integer-valued inputs, where every score is exact in FP32 and FP64."""
import math

import numpy as np
import pytest
import torch

import oracle
import precision_flash_attention_gb300 as pfa
from precision_flash_attention_gb300 import inputs
from tests.gpu_helpers import (TOL_BWD_REL, assert_bwd_close, assert_fwd_close, check_sampled_rows,
                               f64, oracle_full, oracle_group, oracle_group_emulated, rel_l2,
                               run_gpu, sampled_rows, to_dev)

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    pfa.device_error(clear=True)


# ---------------------------------------------------------------- tiny workload
@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("delta_mode", [0, 1])
def test_tiny_forward_backward(mode, delta_mode):
    t = inputs.make("tiny", seed=0)
    got = run_gpu(t, causal=False, scale=0.125, fix_mode=mode, delta_mode=delta_mode)
    ref = oracle_full(t, causal=False, scale=0.125, fix_mode=mode)
    assert_fwd_close(got, ref, f"tiny mode {mode}")
    assert_bwd_close(got, ref, f"tiny mode {mode} delta_mode {delta_mode}")
    assert rel_l2(got["delta"], ref["delta"]) <= TOL_BWD_REL


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 1, 64, 64), (2, 4, 2, 200, 64), (1, 2, 1, 384, 128),
                                   (1, 3, 3, 129, 128)])
def test_grid_counters_bit_exact(mode, causal, shape):
    # Integer Q, K in [-4, 4] with planted duplicated maxima: scores are exact multiples of 1/8.
    B, Hq, Hkv, N, d = shape
    t = inputs.integer_grid(B, Hq, Hkv, N, d, causal=causal, n_planted=8, seed=N + d + mode)
    got = run_gpu(t, causal=causal, scale=0.125, fix_mode=mode, beta=2.0, eps=1e-3, bwd=False)
    ref = oracle_full(t, causal=causal, scale=0.125, fix_mode=mode, beta=2.0, eps=1e-3, bwd=False)
    q, k, v = (f64(t[n]) for n in ("q", "k", "v"))
    emu = oracle.attn_fwd(q, k, v, causal=causal, scale=0.125, fix_mode=mode, beta=2.0, eps=1e-3,
                          emulate_bf16=True)
    assert ref["counters"]["repeated_rows"] >= 8
    # Tie and exact-one counts do not depend on the precision on these inputs; the underflow
    # count does: with d = 128 the beta shift of a planted maximum (about 140) leaves every
    # exponent argument below the FP32 range, as the pages warn, while float64 keeps it.
    for n in ("repeated_rows", "ones"):
        assert emu["counters"][n] == ref["counters"][n]
    assert got["counters"] == emu["counters"]
    bad = np.isnan(emu["o"]).any(axis=-1)
    assert np.array_equal(np.isnan(got["o"]).any(axis=-1), bad)
    assert_fwd_close({"o": got["o"][~bad], "lse": got["lse"][~bad]},
                     {"o": ref["o"][~bad], "lse": ref["lse"][~bad]}, "grid")
    if not bad.any():
        # Integer scores concentrate P on planted maxima; the BF16 cast of dS then puts dQ
        # within a hair of the float64 tolerance in the oracle's own emulation (0.6-1.0%),
        # so dQ is held to the emulating oracle and dK, dV to float64.
        got = run_gpu(t, causal=causal, scale=0.125, fix_mode=mode, beta=2.0, eps=1e-3)
        ref = oracle_full(t, causal=causal, scale=0.125, fix_mode=mode)
        assert_bwd_close(got, ref, "grid", names=("dk", "dv"))
        for b in range(B):
            for hk in range(Hkv):
                e = oracle_group_emulated(t, b, hk, causal=causal, scale=0.125, fix_mode=mode)
                assert_bwd_close({"dq": got["dq"][b, e["heads"]]}, e, "grid (emulated)",
                                 names=("dq",))


# ---------------------------------------------------------------- planted tie patterns
# The flag each construction fixes by definition (inputs.TIE_PATTERNS, eps = 0.05 in
# scaled units, scale 1/8): the repeated-maximum test in the jump tile must see a second
# entry in the same 16-column block, in the same column class, in neither, or none.
TIE_LABELS = {"jump_same_block": True, "jump_same_class": True, "jump_block_and_class": True,
              "jump_single": False, "jump_near_miss": False, "jump_exact_pair": True,
              "tie_below_running_max": True, "rise_within_eps": True}


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("name", sorted(TIE_LABELS))
def test_planted_tie_patterns(name, mode):
    t = inputs.tie_patterns([name])
    got = run_gpu(t, causal=False, scale=0.125, fix_mode=mode, beta=2.0, eps=0.05, bwd=False)
    ref = oracle_full(t, causal=False, scale=0.125, fix_mode=mode, beta=2.0, eps=0.05, bwd=False)
    assert ref["counters"]["repeated_rows"] == (256 if TIE_LABELS[name] else 0)
    assert got["counters"] == ref["counters"]
    assert_fwd_close(got, ref, name)


@pytest.mark.parametrize("mode", [1, 2])
def test_planted_tie_patterns_mixed(mode):
    # All eight patterns interleaved row by row: each warp holds rows that jump and rows
    # that do not, and rows whose second entry sits in different places.
    names = sorted(TIE_LABELS)
    t = inputs.tie_patterns(names, N=512)
    got = run_gpu(t, causal=False, scale=0.125, fix_mode=mode, beta=2.0, eps=0.05, bwd=False)
    ref = oracle_full(t, causal=False, scale=0.125, fix_mode=mode, beta=2.0, eps=0.05, bwd=False)
    assert ref["counters"]["repeated_rows"] == 512 * sum(TIE_LABELS.values()) // len(names)
    assert got["counters"] == ref["counters"]
    assert_fwd_close(got, ref, "mixed")


# ---------------------------------------------------------------- non-positive repeated maxima
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("sign", [-1, 0], ids=["r_m<0", "r_m=0"])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_nonpositive_repeated_maxima(mode, sign, causal, d):
    # Mode 1's shift for a repeated maximum that is not positive: m = 0 when r_m < 0 (the
    # priors.kr post's fix paragraph, paper §4 equation) and m = 2^-5 when r_m = 0 (a reading:
    # the pages name only the two signed cases); mode 2 subtracts r_m + 2^-5 in both. Integer
    # scores (multiples of 1/8) make the ties exact, so the counters must match bit for bit.
    B, Hq, Hkv, N = 1, 2, 1, 300
    t = inputs.signed_max_grid(B, Hq, Hkv, N, d, sign=sign, n_keys=3, seed=17 + d + sign)
    q, k, v = (f64(t[n]) for n in ("q", "k", "v"))
    kw = dict(causal=causal, scale=0.125, fix_mode=mode, beta=2.0, eps=1e-3)
    ref = oracle.attn_fwd(q, k, v, **kw)
    emu = oracle.attn_fwd(q, k, v, emulate_bf16=True, **kw)
    r_m = oracle.attn_fwd(q, k, v, causal=causal, scale=0.125, fix_mode=0)["m"]
    # Repeated rows with the intended sign of r_m (early causal rows that see no planted key
    # can also tie, at a negative integer maximum): the branch is really taken, many times.
    sel = ref["repeated"] & ((r_m < 0) if sign < 0 else (r_m == 0))
    assert sel.sum() >= (100 if causal else Hq * N)
    if mode == 1:
        assert (ref["m"][sel] == (0.0 if sign < 0 else 2.0 ** -5)).all()
    got = run_gpu(t, bwd=mode == 1, **kw)
    assert got["counters"] == emu["counters"] == ref["counters"]
    assert got["counters"]["nonfinite_rows"] == 0
    assert_fwd_close(got, ref, f"mode {mode} sign {sign}")
    if mode == 1:
        # The tied keys are identical, so dQ = dS K nearly cancels along their shared direction
        # and one BF16 rounding of dS moves it by percent: the default path's dQ is held to be
        # no worse than the BF16-emulating oracle's (same cast points), and the query-outer pass
        # with the hi + lo dS to the float64 tolerance. dK and dV are float64-close either way.
        full = oracle_full(t, **kw)
        assert_bwd_close(got, full, "signed maxima", names=("dk", "dv"))
        e = oracle_group_emulated(t, 0, 0, **kw)
        e_emu = rel_l2(e["dq"], full["dq"][0])
        e_gpu = rel_l2(got["dq"][0], full["dq"][0])
        assert e_gpu <= max(TOL_BWD_REL, 1.5 * e_emu), (e_gpu, e_emu)
        # With the query-outer pass the remaining error is delta's: rowsum(dO o O) from the
        # BF16 O moves dQ by percent here (the pages' point: the error enters through delta),
        # rowsum(dP o P) does not.
        split = run_gpu(t, dq_mode="split", delta_mode=1, **kw)
        assert_bwd_close(split, full, "signed maxima (split dS, delta from dP o P)")


# ---------------------------------------------------------------- ragged shapes
RAGGED = [
    # B, Hq, Hkv, N, d, causal
    (1, 1, 1, 1, 64, True),
    (1, 2, 1, 7, 64, False),
    (2, 2, 2, 65, 64, True),
    (1, 4, 2, 100, 128, True),
    (1, 1, 1, 129, 64, False),
    (1, 2, 2, 257, 128, False),
    (2, 3, 1, 300, 64, True),
    (1, 2, 1, 640, 128, True),
]


@pytest.mark.parametrize("shape", RAGGED, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_ragged_shapes(shape, mode):
    B, Hq, Hkv, N, d, causal = shape
    t = inputs.gaussian(B, Hq, Hkv, N, d, std_qkv=0.7, std_do=1.0, seed=7 * N + d)
    scale = 1.0 / math.sqrt(d)
    got = run_gpu(t, causal=causal, scale=scale, fix_mode=mode, beta=3.0)
    ref = oracle_full(t, causal=causal, scale=scale, fix_mode=mode, beta=3.0)
    assert_fwd_close(got, ref, f"{shape} mode {mode}")
    assert_bwd_close(got, ref, f"{shape} mode {mode}")
    assert got["counters"]["nonfinite_rows"] == 0


@pytest.mark.parametrize("N", [1, 2, 17])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_degenerate_lengths(N, d, causal):
    # Sequences shorter than one 128-row tile, down to a single key: row 0 of a causal row
    # sees only itself (one score, never repeated); everything past N is masked or zero-filled.
    t = inputs.gaussian(2, 2, 1, N, d, std_qkv=0.8, std_do=1.0, seed=N + d)
    scale = 1.0 / math.sqrt(d)
    for mode in (0, 1, 2):
        got = run_gpu(t, causal=causal, scale=scale, fix_mode=mode, beta=2.0)
        ref = oracle_full(t, causal=causal, scale=scale, fix_mode=mode, beta=2.0)
        assert_fwd_close(got, ref, f"N {N} d {d} mode {mode}")
        assert_bwd_close(got, ref, f"N {N} d {d} mode {mode}")
        # Float scores: a tie or a round-to-one decision may sit within FP32 rounding of its
        # threshold, so the counts may differ by one; nothing is non-finite.
        for n in ("repeated_rows", "ones"):
            assert abs(got["counters"][n] - ref["counters"][n]) <= 1, (n, got["counters"], ref["counters"])
        assert got["counters"]["nonfinite_rows"] == 0


@pytest.mark.parametrize("d", [64, 128])
def test_delta_zero_pass(d):
    # pfa_attn_delta_zero gives pfa_attn_delta's delta bit for bit and leaves the first
    # B*H*N*d values of the workspace zero (whatever they held), the rest untouched.
    t = to_dev(inputs.gaussian(2, 3, 3, 200, d, std_qkv=0.5, std_do=1.0, seed=d))
    o, lse = pfa.forward(t["q"], t["k"], t["v"], causal=True, scale=0.125)
    d1, d2 = torch.empty_like(lse), torch.empty_like(lse)
    ws = torch.full((t["q"].numel() + 64,), 7.0, dtype=torch.float32, device="cuda")
    pfa.attn_delta(o, t["do"], d1)
    pfa.attn_delta_zero(o, t["do"], d2, ws)
    torch.cuda.synchronize()
    assert pfa.device_error(clear=True) == 0
    assert torch.equal(d1, d2)
    assert int(torch.count_nonzero(ws[: t["q"].numel()])) == 0
    assert bool((ws[t["q"].numel():] == 7.0).all())


def test_delta_alt_equals_delta():
    # rowsum(dP o P) and rowsum(dO o O) agree (the identity of the paper's §3.2).
    t = inputs.gaussian(2, 4, 2, 333, 64, std_qkv=0.5, std_do=1.0, seed=3)
    d = to_dev(t)
    o, lse = pfa.forward(d["q"], d["k"], d["v"], causal=True, scale=0.125)
    d0 = torch.empty_like(lse)
    d1 = torch.empty_like(lse)
    pfa.attn_delta(o, d["do"], d0)
    pfa.attn_delta_alt(d["q"], d["k"], d["v"], d["do"], lse, d1, causal=True, scale=0.125)
    torch.cuda.synchronize()
    ref = oracle_full(t, causal=True, scale=0.125, fix_mode=0)["delta"]
    assert rel_l2(f64(d0), ref) <= TOL_BWD_REL
    assert rel_l2(f64(d1), ref) <= TOL_BWD_REL
    # delta from the GPU's own O is FP32 arithmetic on BF16 data: near-exact.
    exact = oracle.attn_delta(f64(o), f64(t["do"]))
    np.testing.assert_allclose(f64(d0), exact, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("shape", [(1, 2, 1, 300, 128, True), (2, 2, 2, 129, 128, False),
                                   (1, 4, 2, 640, 128, True)], ids=lambda s: "x".join(map(str, s)))
def test_delta_alt_d128(shape):
    # delta = rowsum(dP o P) from the d = 128 instantiation of the tcgen05 kernel, and the
    # backward pass fed with it, against the float64 oracle.
    B, Hq, Hkv, N, d, causal = shape
    t = inputs.gaussian(B, Hq, Hkv, N, d, std_qkv=0.5, std_do=1.0, seed=N)
    scale = 1.0 / math.sqrt(d)
    got = run_gpu(t, causal=causal, scale=scale, fix_mode=1, beta=2.0, delta_mode=1)
    ref = oracle_full(t, causal=causal, scale=scale, fix_mode=1, beta=2.0)
    assert rel_l2(got["delta"], ref["delta"]) <= TOL_BWD_REL
    assert_fwd_close(got, ref, f"{shape}")
    assert_bwd_close(got, ref, f"{shape} delta_mode 1")


# ---------------------------------------------------------------- full-size workloads
def test_gpt2_small_layer_all_heads():
    # B=8, H=12, N=1024, d=64, causal, modes 0 and 1 (beta=2): every head against the oracle.
    t = inputs.make("gpt2", seed=0)
    for mode in (0, 1):
        got = run_gpu(t, causal=True, scale=0.125, fix_mode=mode, beta=2.0)
        ref = oracle_full(t, causal=True, scale=0.125, fix_mode=mode, beta=2.0)
        assert_fwd_close(got, ref, f"gpt2 mode {mode}")
        assert_bwd_close(got, ref, f"gpt2 mode {mode}")
        assert got["counters"]["nonfinite_rows"] == 0
        # ones >= rows in mode 0: every row's maximum gives Pbar = 1 exactly.
        rows = 8 * 12 * 1024
        if mode == 0:
            assert got["counters"]["ones"] >= rows
        # the repeated-row count is the same tie detector in every mode (fp32 vs fp64 scores
        # may move a handful of borderline rows)
        assert abs(got["counters"]["repeated_rows"] - ref["counters"]["repeated_rows"]) <= 8


@pytest.mark.parametrize("d", [64, 128])
def test_three_rounds_of_key_tiles(d):
    # B = 4, H = 12, N = 1024, causal: 384 key-tile items (1 to 8 query tiles each) over 152
    # CTAs, three serpentine rounds with a partial last one. Every head against the oracle;
    # at d = 128 the kernel without its dQ product (the query-outer pass computes dQ).
    t = inputs.gaussian(4, 12, 12, 1024, d, std_qkv=0.7, std_do=1.0, seed=d)
    kw = dict(causal=True, scale=d ** -0.5, fix_mode=1, beta=2.0)
    got = run_gpu(t, **kw)
    ref = oracle_full(t, **kw)
    assert_fwd_close(got, ref, f"B4 H12 N1024 d={d}")
    assert_bwd_close(got, ref, f"B4 H12 N1024 d={d}")


def test_gpt2_shape_n2048_sampled_rows():
    # The GPT-2 shape at N = 2048 (a point of the bench's sweep): 768 forward items over
    # 152 CTAs, five serpentine rounds. Sampled rows of every head.
    B, H, N = 8, 12, 2048
    t = inputs.gaussian(B, H, H, N, 64, std_qkv=0.7, std_do=1.0, seed=21)
    kw = dict(causal=True, scale=0.125, fix_mode=1, beta=2.0)
    got = run_gpu(t, bwd=False, **kw)
    rows = sampled_rows(N, 48, seed=4)
    acc = ([], [], [], [])
    for b in range(B):
        for h in range(H):
            r = oracle.attn_fwd_head(f64(t["q"][b, h]), f64(t["k"][b, h]), f64(t["v"][b, h]), rows=rows, **kw)
            for lst, x in zip(acc, (got["o"][b, h, rows], r["o"], got["lse"][b, h, rows], r["lse"])):
                lst.append(x)
    cat = [np.concatenate(a) for a in acc]
    assert_fwd_close({"o": cat[0], "lse": cat[2]}, {"o": cat[1], "lse": cat[3]}, "gpt2 N=2048")
    assert got["counters"]["nonfinite_rows"] == 0


def _check_groups(t, got, groups, *, causal, scale, mode, beta, dq_emulated=False,
                  delta_mode=0):
    for b, hk in groups:
        r = oracle_group(t, b, hk, causal=causal, scale=scale, fix_mode=mode, beta=beta)
        hs = r["heads"]
        assert_fwd_close({"o": got["o"][b, hs], "lse": got["lse"][b, hs]}, r, f"group {b},{hk}")
        g = {"dq": got["dq"][b, hs], "dk": got["dk"][b, hk], "dv": got["dv"][b, hk]}
        if dq_emulated:
            assert_bwd_close(g, r, f"group {b},{hk}", names=("dk", "dv"))
            e = oracle_group_emulated(t, b, hk, causal=causal, scale=scale, fix_mode=mode,
                                      beta=beta, delta_mode=delta_mode)
            assert_bwd_close(g, e, f"group {b},{hk} (emulated)", names=("dq",))
        else:
            assert_bwd_close(g, r, f"group {b},{hk}")


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_sink_heavy(mode):
    # delta = rowsum(dP o P), the alternative the paper found stable (its §3.2), and dQ from the
    # query-outer pass with dS as a BF16 hi + lo pair: every output within the float64
    # tolerances of the contract, dQ included. (A single BF16 dS moves dQ by about 12% on this
    # input, in the oracle's own emulation as on the GPU: copies of the sink key share its
    # feature of 48 and their dS nearly cancel along it.)
    t = inputs.make("sink", seed=0)
    got = run_gpu(t, causal=True, scale=0.125, fix_mode=mode, beta=2.0, delta_mode=1,
                  dq_mode="split")
    _check_groups(t, got, [(0, 0), (3, 11), (1, 5)], causal=True, scale=0.125, mode=mode, beta=2.0)
    c = got["counters"]
    assert c["nonfinite_rows"] == 0
    assert c["repeated_rows"] > 0.1 * 4 * 12 * 2048  # the planted duplicates
    if mode > 0:
        # the fix leaves at most the single maximum of each non-repeated row at 1.0
        assert c["ones"] <= 4 * 12 * 2048 - c["repeated_rows"] + 64


def test_sink_heavy_single_bf16_ds_matches_emulation():
    # The default backward (one BF16 dS operand, dQ reduce-added per key tile): O, lse, dK and
    # dV within the float64 tolerances; dQ against the BF16-emulating oracle, which rounds dS
    # where the kernel does.
    t = inputs.make("sink", seed=0)
    got = run_gpu(t, causal=True, scale=0.125, fix_mode=1, beta=2.0, delta_mode=1)
    _check_groups(t, got, [(0, 0), (2, 7)], causal=True, scale=0.125, mode=1, beta=2.0,
                  dq_emulated=True, delta_mode=1)


def test_sink_heavy_delta_from_bf16_output():
    # delta = rowsum(dO o O) from the BF16 output: with a sink key the row's dP - delta is a
    # near-cancellation, so the BF16 rounding of O dominates dS on the sink column -- the
    # mechanism the pages trace the failure to (priors.kr three-line summary; bud-325 Key
    # claims). The float64 dQ is then out of reach of any BF16-O implementation: the oracle
    # itself, given delta from its own BF16-emulated O, lands as far from it. dK and dV stay
    # within tolerance, and the GPU's dQ is closer to that BF16-O oracle than to float64.
    t = inputs.make("sink", seed=0)
    got = run_gpu(t, causal=True, scale=0.125, fix_mode=1, beta=2.0, delta_mode=0)
    r = oracle_group(t, 0, 0, causal=True, scale=0.125, fix_mode=1, beta=2.0)
    assert_bwd_close({"dk": got["dk"][0, 0], "dv": got["dv"][0, 0]}, r, names=("dk", "dv"))
    q, k, v, do = (f64(t[n][0:1, 0:1]) for n in ("q", "k", "v", "do"))
    emu = oracle.attn_fwd(q, k, v, causal=True, scale=0.125, fix_mode=1, beta=2.0,
                          emulate_bf16=True)
    g_bf = oracle.attn_bwd(q, k, v, do, r["lse"][None], oracle.attn_delta(emu["o"], do),
                           causal=True, scale=0.125)
    err_oracle = rel_l2(g_bf["dq"][0, 0], r["dq"][0])
    err_gpu = rel_l2(got["dq"][0, 0], r["dq"][0])
    print(f"dQ rel-L2 vs float64: oracle with BF16 O {err_oracle:.3f}, GPU {err_gpu:.3f}, "
          f"GPU vs BF16-O oracle {rel_l2(got['dq'][0, 0], g_bf['dq'][0, 0]):.3f}")
    assert err_oracle > 0.3 and err_gpu > 0.3
    assert rel_l2(got["dq"][0, 0], g_bf["dq"][0, 0]) < err_gpu


def test_long_context():
    # B=2, H=16, N=8192, d=128, mode 1 with beta = 4: O, lse and dQ on 256 sampled rows of every
    # head (the first and last 16 rows included), dK and dV of three whole key/value heads.
    t = inputs.make("long", seed=0)
    scale = 1.0 / math.sqrt(128)
    got = run_gpu(t, causal=True, scale=scale, fix_mode=1, beta=4.0)
    check_sampled_rows(t, got, sampled_rows(8192), causal=True, scale=scale, fix_mode=1, beta=4.0)
    _check_groups(t, got, [(1, 15), (0, 0), (0, 9)], causal=True, scale=scale, mode=1, beta=4.0)
    assert got["counters"]["nonfinite_rows"] == 0


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_gqa_large_logits(mode):
    # B=1, H_q=32, H_kv=8, N=8192, d=128: sampled rows of all 32 query heads, and two whole
    # key/value groups (four query heads each) for dK and dV.
    t = inputs.make("gqa", seed=0)
    scale = 1.0 / math.sqrt(128)
    got = run_gpu(t, causal=True, scale=scale, fix_mode=mode, beta=2.0)
    check_sampled_rows(t, got, sampled_rows(8192, seed=mode), causal=True, scale=scale,
                       fix_mode=mode, beta=2.0)
    _check_groups(t, got, [(0, 3), (0, 7)], causal=True, scale=scale, mode=mode, beta=2.0)
    assert got["counters"]["nonfinite_rows"] == 0
    if mode == 0:
        assert got["counters"]["ones"] >= 32 * 8192


# ---------------------------------------------------------------- query-outer dQ pass
QOUTER_SHAPES = [(1, 1, 1, 1, 64, True), (1, 2, 1, 7, 64, False), (2, 4, 2, 300, 64, True),
                 (1, 2, 2, 257, 128, False), (1, 4, 2, 640, 128, True), (2, 3, 1, 129, 64, False)]


@pytest.mark.parametrize("dq_mode", ["deterministic", "split"])
@pytest.mark.parametrize("shape", QOUTER_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_query_outer_dq(shape, dq_mode):
    # dQ from the query-outer pass (pfa_attn_bwd_ex) against the float64 oracle, dK and dV from
    # the key-outer kernel without its dQ product; a second call gives the same bits.
    B, Hq, Hkv, N, d, causal = shape
    t = inputs.gaussian(B, Hq, Hkv, N, d, std_qkv=0.7, std_do=1.0, seed=3 * N + d)
    scale = 1.0 / math.sqrt(d)
    got = run_gpu(t, causal=causal, scale=scale, fix_mode=1, beta=2.0, dq_mode=dq_mode)
    ref = oracle_full(t, causal=causal, scale=scale, fix_mode=1, beta=2.0)
    assert_bwd_close(got, ref, f"{shape} {dq_mode}")
    again = run_gpu(t, causal=causal, scale=scale, fix_mode=1, beta=2.0, dq_mode=dq_mode)
    for n in ("dq", "dk", "dv"):
        assert np.array_equal(got[n], again[n]), n


def test_split_dq_is_closer_to_float64_than_single_bf16():
    # On a sink-heavy input (copies of a sink key whose large feature carries a +6 logit) the
    # single BF16 dS leaves dQ percent away from float64; the hi + lo pair removes that rounding.
    # delta = rowsum(dP o P) in both, so that delta from the BF16 O does not mask the effect.
    t = inputs.sink_heavy(1, 2, 512, 64, seed=3)
    ref = oracle_full(t, causal=True, scale=0.125, fix_mode=1)
    single = run_gpu(t, causal=True, scale=0.125, fix_mode=1, beta=2.0, delta_mode=1)
    split = run_gpu(t, causal=True, scale=0.125, fix_mode=1, beta=2.0, delta_mode=1, dq_mode="split")
    e1, e2 = rel_l2(single["dq"], ref["dq"]), rel_l2(split["dq"], ref["dq"])
    assert e1 > 2e-2 and e2 <= TOL_BWD_REL and e2 < 0.2 * e1, (e1, e2)


def test_bwd_ex_argument_errors():
    t = to_dev(inputs.make("tiny"))
    o, lse = pfa.forward(t["q"], t["k"], t["v"], scale=0.125)
    delta = torch.empty_like(lse)
    pfa.attn_delta(o, t["do"], delta)
    dq, dk, dv = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
    with pytest.raises(pfa.PfaError, match="INVALID_ARG"):   # an unknown flag bit
        pfa.attn_bwd_ex(t["q"], t["k"], t["v"], t["do"], lse, delta, dq, dk, dv, None, causal=False,
                        scale=0.125, flags=8)
    with pytest.raises(ValueError, match="dq_accum"):         # a zeroed workspace is still required
        pfa.attn_bwd_ex(t["q"], t["k"], t["v"], t["do"], lse, delta, dq, dk, dv, None, causal=False,
                        scale=0.125, flags=pfa.BWD_WORKSPACE_ZEROED)
    assert pfa.device_error() == 0


# ---------------------------------------------------------------- degenerate cases
def test_underflow_probe_matches_emulation():
    # Mode 1 with a repeated maximum of 200: beta*r_m pushes every exponent below FP32 range.
    for logit, expect_nonfinite in ((200.0, True), (10.0, False)):
        t = inputs.underflow_probe(1, 2, 128, 64, logit=logit)
        got = run_gpu(t, causal=False, scale=0.125, fix_mode=1, beta=2.0, bwd=False)
        q, k, v = (f64(t[n]) for n in ("q", "k", "v"))
        emu = oracle.attn_fwd(q, k, v, scale=0.125, fix_mode=1, beta=2.0, emulate_bf16=True)
        assert got["counters"] == emu["counters"]
        assert (got["counters"]["nonfinite_rows"] == 256) == expect_nonfinite
        if expect_nonfinite:
            assert np.isnan(got["o"]).all()
        else:
            assert np.isfinite(got["o"]).all()
        # mode 2 never underflows here
        got2 = run_gpu(t, causal=False, scale=0.125, fix_mode=2, bwd=False)
        assert got2["counters"]["nonfinite_rows"] == 0


def test_counters_accumulate_and_are_optional():
    t = to_dev(inputs.make("grid", seed=1))
    cnt = pfa.new_counters()
    for _ in range(2):
        pfa.forward(t["q"], t["k"], t["v"], scale=0.125, fix_mode=1, counters=cnt)
    o_nc, lse_nc = pfa.forward(t["q"], t["k"], t["v"], scale=0.125, fix_mode=1)
    o_c, lse_c = pfa.forward(t["q"], t["k"], t["v"], scale=0.125, fix_mode=1,
                             counters=pfa.new_counters())
    torch.cuda.synchronize()
    ref = oracle.attn_fwd(*(f64(t[n].cpu()) for n in ("q", "k", "v")), scale=0.125, fix_mode=1)
    assert cnt.cpu().tolist() == [2 * ref["counters"][n] for n in
                                  ("repeated_rows", "ones", "nonfinite_rows")]
    assert torch.equal(o_nc, o_c) and torch.equal(lse_nc, lse_c)


def test_invalid_arguments_raise():
    t = to_dev(inputs.make("tiny"))
    with pytest.raises(pfa.PfaError):
        pfa.forward(t["q"], t["k"], t["v"], scale=0.125, fix_mode=1, beta=0.5)
    with pytest.raises(ValueError):
        pfa.forward(t["q"].float(), t["k"], t["v"], scale=0.125)
    assert pfa.device_error() == 0


def test_stream_and_autograd_wrapper():
    t = to_dev(inputs.gaussian(1, 2, 2, 150, 64, std_qkv=0.5, seed=5))
    q, k, v = (t[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o = pfa.StabilizedAttention.apply(q, k, v, True, 0.125, 1, 2.0, 1e-3)
        o.backward(t["do"])
    torch.cuda.synchronize()
    ref = oracle_full({n: x.cpu() for n, x in t.items()}, causal=True, scale=0.125, fix_mode=1)
    assert_fwd_close({"o": f64(o), "lse": ref["lse"]}, ref)
    assert_bwd_close({"dq": f64(q.grad), "dk": f64(k.grad), "dv": f64(v.grad)}, ref)


@pytest.mark.parametrize("shape", [(1, 4, 2, 300, 64), (1, 2, 1, 200, 128)], ids=["d64-gqa", "d128"])
def test_bwd_accumulate_entry_point(shape):
    # pfa_attn_bwd_accum adds dS K (alpha is inside dS) into a caller's FP32 buffer and writes dK, dV;
    # two calls on one buffer give twice dQ, and dK, dV match pfa_attn_bwd.
    B, Hq, Hkv, N, d = shape
    t = to_dev(inputs.gaussian(B, Hq, Hkv, N, d, std_qkv=0.5, std_do=1.0, seed=7))
    scale = 1.0 / math.sqrt(d)
    o, lse = pfa.forward(t["q"], t["k"], t["v"], causal=True, scale=scale)
    dq, dk, dv, delta = pfa.backward(t["q"], t["k"], t["v"], o, lse, t["do"], causal=True, scale=scale)
    acc = torch.zeros(t["q"].shape, dtype=torch.float32, device="cuda")
    dk2, dv2 = torch.empty_like(dk), torch.empty_like(dv)
    for _ in range(2):
        pfa.attn_bwd_accum(t["q"], t["k"], t["v"], t["do"], lse, delta, acc, dk2, dv2, causal=True,
                           scale=scale)
    torch.cuda.synchronize()
    assert pfa.device_error(clear=True) == 0
    assert torch.equal(dk2, dk) and torch.equal(dv2, dv)
    half = acc / 2
    assert torch.isfinite(half).all()
    # The BF16 dQ of pfa_attn_bwd is the rounded FP32 accumulation of one call.
    assert rel_l2(f64(half.to(torch.bfloat16)), f64(dq)) < 1e-2
    ref = oracle_full({n: x.cpu() for n, x in t.items()}, causal=True, scale=scale, fix_mode=0)
    assert rel_l2(f64(half), ref["dq"]) <= TOL_BWD_REL
    # An argument error launches nothing and returns the code.
    lib = pfa.load()
    import ctypes
    st = lib.pfa_attn_bwd_accum(*([ctypes.c_void_p(t["q"].data_ptr())] * 6), None,
                                ctypes.c_void_p(dk2.data_ptr()), ctypes.c_void_p(dv2.data_ptr()),
                                B, Hq, Hkv, N, d, 1, scale, None)
    assert st == -1 and "INVALID_ARG" in pfa.status_string(st)


@pytest.mark.parametrize("d,B,H", [(64, 32, 512), (128, 16, 512)], ids=["d64", "d128"])
def test_maximum_size(d, B, H):
    # The largest problem the size checks accept: B * H * N * d just under 2^31 values per
    # tensor, 4 GiB of BF16, so the byte offsets of the last heads need 33 bits. P distinct
    # seeded heads are tiled over all B * H heads on the device; the first and last heads are
    # checked against the oracle of their pattern, and equal patterns must give equal bits
    # wherever the arithmetic does not depend on arrival order (O, lse, dK, dV).
    N, P = 2047, 4
    assert 2 ** 31 - 2 ** 21 < B * H * N * d < 2 ** 31
    small = inputs.gaussian(1, P, P, N, d, std_qkv=0.5, std_do=1.0, seed=5)
    full = {n: x.cuda().repeat(1, B * H // P, 1, 1).view(B, H, N, d) for n, x in small.items()}
    scale = 1.0 / math.sqrt(d)
    o, lse = pfa.forward(full["q"], full["k"], full["v"], causal=True, scale=scale, fix_mode=1)
    dq, dk, dv, _ = pfa.backward(full["q"], full["k"], full["v"], o, lse, full["do"], causal=True,
                                 scale=scale)
    torch.cuda.synchronize()
    assert pfa.device_error(clear=True) == 0
    del full
    ref = oracle_full(small, causal=True, scale=scale, fix_mode=1)
    n_heads = B * H
    for idx in (0, 1, 2, 3, n_heads // 2 + 1, n_heads - 4, n_heads - 3, n_heads - 2, n_heads - 1):
        b, h = divmod(idx, H)
        got = {n: f64(t[b, h]) for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
        want = {n: ref[n][0, idx % P] for n in ("o", "lse", "dq", "dk", "dv")}
        assert_fwd_close(got, want, f"head {idx}")
        assert_bwd_close(got, want, f"head {idx}")
    last = divmod(n_heads - P, H)
    for t in (o, lse, dk, dv):
        assert torch.equal(t[0, 0], t[last[0], last[1]])
    del o, lse, dq, dk, dv
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fused_zero", [False, True], ids=["separate-zeroing", "delta-zeroes"])
def test_cuda_graph_capture_matches_eager(fused_zero):
    # The calls allocate nothing and never synchronise, so a whole step (forward, delta,
    # backward with its zeroing and conversion, launched as programmatic dependents)
    # captures into a CUDA graph; replaying it gives the eager results bit for bit. With
    # fused_zero the delta pass zeroes the dQ workspace (pfa_attn_delta_zero) and the
    # backward call skips its zeroing pass, as pfa.backward does at d = 64.
    t = to_dev(inputs.gaussian(2, 4, 2, 384, 64, std_qkv=0.5, std_do=1.0, seed=11))
    q, k, v, do = t["q"], t["k"], t["v"], t["do"]
    o, lse = torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    delta = torch.empty_like(lse)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(pfa.bwd_workspace_bytes(*q.shape) // 4, dtype=torch.float32, device="cuda")

    def step():
        pfa.attn_fwd(q, k, v, o, lse, causal=True, scale=0.125, fix_mode=1, beta=2.0, eps=1e-3)
        if fused_zero:
            pfa.attn_delta_zero(o, do, delta, ws)
        else:
            pfa.attn_delta(o, do, delta)
        pfa.attn_bwd(q, k, v, do, lse, delta, dq, dk, dv, ws, causal=True, scale=0.125,
                     workspace_zeroed=fused_zero)

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
    for a, b in zip(eager[:2] + eager[3:], (o, lse, dk, dv)):
        assert torch.equal(a, b)
    # dQ sums reduce-adds in arrival order: equal up to FP32 rounding of that order.
    assert rel_l2(f64(dq), f64(eager[2])) < 1e-3


def test_cuda_graph_capture_deterministic_dq_is_bit_exact():
    # With the query-outer dQ pass every output, dQ included, replays bit for bit.
    t = to_dev(inputs.gaussian(2, 4, 2, 384, 64, std_qkv=0.5, std_do=1.0, seed=11))
    q, k, v, do = t["q"], t["k"], t["v"], t["do"]
    o, lse = torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    delta = torch.empty_like(lse)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def step():
        pfa.attn_fwd(q, k, v, o, lse, causal=True, scale=0.125, fix_mode=1, beta=2.0, eps=1e-3)
        pfa.attn_delta(o, do, delta)
        pfa.attn_bwd_ex(q, k, v, do, lse, delta, dq, dk, dv, None, causal=True, scale=0.125,
                        flags=pfa.BWD_DQ_DETERMINISTIC)

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
