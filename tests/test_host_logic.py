"""Host-side logic that needs no GPU: the product-text digest that keys the DRAM traffic
records, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

from precision_flash_attention_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _text(tmp_path, body):
    p = tmp_path / "k.cu"
    p.write_text(body)
    return build._product_text(str(p))


def test_product_text_ignores_comments_and_trace_only_code(tmp_path):
    base = "int f(int x) {\n  return x + 1;\n}\n"
    traced = ("// a comment\nint f(int x) {\n  /* block\n comment */\n"
              "  if (x == 0) PFA_BWD_TRACE(0, 1, x);\n"
              "#if defined(PFA_TRACE) && defined(PFA_TRACE_QOBS)\n  observe();\n#if 1\n#endif\n#endif\n"
              "  return x + 1;  // trailing\n}\n")
    strip = lambda b: b.replace(b" ", b"").replace(b"\n", b"")  # noqa: E731
    assert strip(_text(tmp_path, base)) == strip(_text(tmp_path, traced))


def test_product_text_sees_code_changes(tmp_path):
    assert _text(tmp_path, "int f(int x) { return x + 1; }\n") != _text(tmp_path, "int f(int x) { return x + 2; }\n")


def test_kernel_digest_is_per_kernel():
    d_bwd = build.kernel_source_digest("attn_bwd_kernel")
    d_fwd = build.kernel_source_digest("attn_fwd_kernel")
    assert d_bwd != d_fwd and len(d_bwd) == 64
    assert build.kernel_source_digest("convert_dq_kernel") == d_bwd   # same translation unit


def test_kernel_digest_follows_includes():
    # A kernel's digest covers the headers its translation unit (and the API file) include,
    # transitively, and no others: the forward kernel's header is not the backward kernel's.
    def names(tu):
        seen = []
        for f in (tu, "attn_api.cu"):
            build._local_includes(os.path.join(build.CSRC, f), seen)
        return {os.path.basename(p) for p in seen}
    bwd, fwd = names("attn_bwd.cu"), names("attn_fwd.cu")
    assert {"pfa_device.cuh", "pfa_internal.h", "pfa.h"} <= bwd and "attn_fwd.cuh" not in bwd
    assert {"attn_fwd.cuh", "pfa_device.cuh", "pfa_trace.cuh", "pfa.h"} <= fwd


def test_reference_arm_json_line():
    # The reference arm times the float64 oracle on the host; one short step is enough here.
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600, check=True).stdout
    line = json.loads(out.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["config"]["N"] == 1024 and line["config"]["d"] == 64
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_binding_rejects_mismatched_shapes_before_any_launch():
    # The wrappers check every tensor's shape against q and k before they look at devices or
    # call into the library, so these CPU tensors never reach a kernel.
    import pytest
    import torch

    from precision_flash_attention_gb300 import _lib

    bf = lambda *s: torch.zeros(s, dtype=torch.bfloat16)  # noqa: E731
    f32 = lambda *s: torch.zeros(s, dtype=torch.float32)  # noqa: E731
    q, k, v, do = bf(2, 4, 64, 64), bf(2, 2, 64, 64), bf(2, 2, 64, 64), bf(2, 4, 64, 64)
    lse, delta = f32(2, 4, 64), f32(2, 4, 64)
    dq, dk, dv = bf(2, 4, 64, 64), bf(2, 2, 64, 64), bf(2, 2, 64, 64)
    kw = dict(causal=True, scale=0.125)
    cases = [
        (dict(dq=bf(2, 4, 32, 64)), "dq"),          # dq smaller than q
        (dict(dk=bf(2, 4, 64, 64)), "dk"),          # dk shaped like q, not like k
        (dict(dv=bf(2, 2, 64, 32)), "dv"),
        (dict(lse=f32(2, 4, 63)), "lse"),
        (dict(delta=f32(2, 2, 64)), "delta"),
        (dict(k=bf(2, 3, 64, 64), v=bf(2, 3, 64, 64)), "multiple"),  # H_kv does not divide H_q
        (dict(v=bf(2, 2, 65, 64)), "v"),
    ]
    for change, what in cases:
        a = dict(q=q, k=k, v=v, do=do, lse=lse, delta=delta, dq=dq, dk=dk, dv=dv)
        a.update(change)
        with pytest.raises(ValueError, match=what):
            _lib.attn_bwd_noalloc(a["q"], a["k"], a["v"], a["do"], a["lse"], a["delta"], a["dq"],
                                  a["dk"], a["dv"], **kw)
    with pytest.raises(ValueError, match="o has shape"):
        _lib.attn_fwd(q, k, v, bf(2, 4, 64, 128), lse, **kw)
    with pytest.raises(ValueError, match="delta"):
        _lib.attn_delta(q, do, f32(2, 4, 32))
    with pytest.raises(ValueError, match="dq_accum"):
        _lib.attn_bwd_accum(q, k, v, do, lse, delta, f32(2, 4, 64, 32), dk, dv, **kw)
    # Shapes that agree get as far as the device check (CPU tensors are refused there).
    with pytest.raises(ValueError, match="CUDA"):
        _lib.attn_bwd_noalloc(q, k, v, do, lse, delta, dq, dk, dv, **kw)
