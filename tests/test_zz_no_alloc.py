"""pfa_attn_bwd_noalloc: the backward pass for callers that may not allocate device memory.

Some callers cannot call cudaMalloc: runtimes that hand all device memory to their own pool
at start-up, real-time loops that cannot afford cudaMalloc's implicit synchronisation, or
plugins that only receive their inputs and outputs. For them the library keeps the dQ
accumulation buffer in a fixed array of its own. These tests call that entry point through
the C ABI and check that it returns what pfa_attn_bwd (with a caller workspace) returns,
within the backward tolerance the other GPU tests use (rel-L2 <= 1e-2), on two calls in a
row: the second call finds the first call's sums in the shared buffer and must clear them.
This file is collected last so that a run stopping at the first failure has run everything
else first; it also passes on its own in a fresh process.
"""
import ctypes
import math

import pytest
import torch

pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.fixture(scope="module")
def pfa():
    import __graft_entry__
    __graft_entry__.build()
    import precision_flash_attention_gb300 as mod
    mod.device_error(clear=True)
    return mod


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm())


@pytest.mark.parametrize("shape", [(2, 4, 2, 300, 64, True), (1, 2, 2, 257, 128, False),
                                   (8, 12, 12, 1024, 64, True)])
def test_noalloc_matches_workspace_entry_point(pfa, shape):
    from precision_flash_attention_gb300 import inputs
    B, Hq, Hkv, N, d, causal = shape
    t = {n: x.cuda() for n, x in inputs.gaussian(B, Hq, Hkv, N, d, std_qkv=0.5, std_do=1e-2,
                                                  seed=N + d).items()}
    scale = 1.0 / math.sqrt(d)
    o, lse = pfa.forward(t["q"], t["k"], t["v"], causal=causal, scale=scale, fix_mode=1)
    dq_ref, dk_ref, dv_ref, delta = pfa.backward(t["q"], t["k"], t["v"], o, lse, t["do"],
                                                 causal=causal, scale=scale)
    lib = pfa.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):  # two calls in a row share (and must re-clear) the library's buffer
        dq, dk, dv = (torch.full_like(x, float("nan")) for x in (t["q"], t["k"], t["v"]))
        p = [ctypes.c_void_p(x.data_ptr()) for x in (t["q"], t["k"], t["v"], t["do"], lse, delta,
                                                     dq, dk, dv)]
        st = lib.pfa_attn_bwd_noalloc(*p, B, Hq, Hkv, N, d, int(causal), scale, stream)
        assert st == 0, pfa.status_string(st)
        torch.cuda.synchronize()
        for got, ref in ((dq, dq_ref), (dk, dk_ref), (dv, dv_ref)):
            assert torch.isfinite(got).all()
            assert _rel(got, ref) <= TOL
    assert pfa.device_error() == 0


def test_noalloc_python_wrapper(pfa):
    # The same entry point through the package's binding, which checks shapes and devices.
    from precision_flash_attention_gb300 import inputs
    t = {n: x.cuda() for n, x in inputs.gaussian(1, 4, 2, 200, 64, std_qkv=0.5, std_do=1e-2,
                                                  seed=3).items()}
    o, lse = pfa.forward(t["q"], t["k"], t["v"], causal=True, scale=0.125, fix_mode=2)
    dq_ref, dk_ref, dv_ref, delta = pfa.backward(t["q"], t["k"], t["v"], o, lse, t["do"],
                                                 causal=True, scale=0.125)
    for _ in range(2):
        dq, dk, dv = (torch.full_like(x, float("nan")) for x in (t["q"], t["k"], t["v"]))
        pfa.attn_bwd_noalloc(t["q"], t["k"], t["v"], t["do"], lse, delta, dq, dk, dv, causal=True,
                             scale=0.125)
        torch.cuda.synchronize()
        for got, ref in ((dq, dq_ref), (dk, dk_ref), (dv, dv_ref)):
            assert _rel(got, ref) <= TOL
    with pytest.raises(ValueError):
        pfa.attn_bwd_noalloc(t["q"], t["k"], t["v"], t["do"], lse[:, :, :100].contiguous(), delta,
                             dq, dk, dv, causal=True, scale=0.125)
    assert pfa.device_error() == 0


def test_noalloc_rejects_problems_beyond_its_buffer(pfa):
    # 8 * 16 * 8192 * 128 = 134M values > 8,388,608: refused before anything is launched.
    lib = pfa.load()
    a = ctypes.c_void_p(1 << 20)
    st = lib.pfa_attn_bwd_noalloc(*([a] * 9), 8, 16, 16, 8192, 128, 1, 0.088, None)
    assert st == -6
    assert "PFA_ERR_TOO_LARGE" in pfa.status_string(st)
    # the limit itself is accepted: 1 * 1 * 65536 * 128 = 8,388,608 values
    x = torch.zeros((1, 1, 65536, 128), dtype=torch.bfloat16, device="cuda")
    s = torch.zeros((1, 1, 65536), dtype=torch.float32, device="cuda")
    p = [ctypes.c_void_p(y.data_ptr()) for y in (x, x, x, x, s, s)]
    outs = [torch.empty_like(x) for _ in range(3)]
    p += [ctypes.c_void_p(y.data_ptr()) for y in outs]
    st = lib.pfa_attn_bwd_noalloc(*p, 1, 1, 1, 65536, 128, 0, 0.088, None)
    assert st == 0, pfa.status_string(st)
    torch.cuda.synchronize()
    assert pfa.device_error() == 0
