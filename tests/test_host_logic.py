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
