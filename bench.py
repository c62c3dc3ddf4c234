"""Benchmark: stabilised BF16 attention forward + backward TFLOP/s on GB300.

One step = forward (pfa_attn_fwd) + delta (pfa_attn_delta_zero, which also zeroes
the dQ workspace) + backward (pfa_attn_bwd_ex without its zeroing pass; it converts
the dQ workspace to BF16) over one batch
of the GPT-2-small attention layer (B=8, H=12, N=1024, d=64, causal), inputs
resident in HBM, L2 flushed between steps. Algorithmic FLOPs per step:
14 * B * H * N^2 * d / 2 (S, Pbar V forward; S, dP, dV, dK, dQ backward; causal).

Prints one JSON line (rank 0). ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "attention fwd+bwd TFLOP/s and % of GB300 BF16 peak (GPT-2 shape, N=1k–8k)"
WORKLOAD = dict(B=8, H=12, N=1024, d=64, causal=True, scale=0.125, beta=2.0, eps=1e-3)
L2_FLUSH_BYTES = 256 << 20
# The timed region spans at least this long, so the clock record holds several samples.
TIMED_REGION_MIN_S = 0.2
# Kernels of ours launched per step: attn_fwd, delta (which also zeroes the dQ
# workspace), attn_bwd and the dQ conversion.
LAUNCHES_PER_STEP = 4


def flops(B, H, N, d, causal, which="fwd+bwd"):
    per = {"fwd": 4.0, "bwd": 10.0, "fwd+bwd": 14.0}[which]
    f = per * B * H * N * N * d
    return f / 2 if causal else f


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p, encoding="utf-8") as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class _NoClock:
    """Stand-in for ClockSampler in profiling runs."""

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False

    def wait_first(self, *a):
        pass

    def mark_start(self):
        pass

    def mark_end(self):
        pass

    def summary(self):
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 10 ms by a reader thread
    that stamps each line with its arrival time. ``mark_start`` / ``mark_end``
    bracket the timed region; the summary uses the samples inside it, and only if a
    region is too short to hold one, the nearest sample on each side (both taken
    under the same load: warm-up before, an untimed tail of steps after)."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 10

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.samples = []          # (host time, line)
        self.t0 = self.t1 = None
        self._thread = None

    def _reader(self):
        for ln in self.proc.stdout:
            if ln.strip():
                self.samples.append((time.perf_counter(), ln.strip()))

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._thread = threading.Thread(target=self._reader, daemon=True)
            self._thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def wait_first(self, timeout_s=10.0):
        """Block until sampling is live (or the tool is missing)."""
        end = time.perf_counter() + timeout_s
        while self.proc is not None and not self.samples and time.perf_counter() < end:
            if self.proc.poll() is not None:
                break
            time.sleep(0.01)

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self._thread is not None:
                self._thread.join(timeout=5)

    @staticmethod
    def _parse(ln):
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) < 9:
            return None
        try:
            return float(parts[1]), float(parts[2]), parts[5:9]
        except ValueError:
            return None

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        parsed = [(t, self._parse(ln)) for t, ln in self.samples]
        parsed = [(t, p) for t, p in parsed if p is not None]
        if not parsed or self.t0 is None or self.t1 is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        inside = [p for t, p in parsed if self.t0 <= t <= self.t1]
        window = "timed region"
        if not inside:
            before = [p for t, p in parsed if t < self.t0][-1:]
            after = [p for t, p in parsed if t > self.t1][:1]
            inside = before + after
            window = "nearest samples around a timed region shorter than the sampling period"
        reasons = set()
        for _, _, flags in inside:
            for n, v in zip(names, flags):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(p[0] for p in inside), "sm_max_mhz": max(p[1] for p in inside),
                "reasons": sorted(reasons), "samples": len(inside), "window": window,
                "period_ms": self.PERIOD_MS}


def traffic_for(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the kernel's
    current sources (null otherwise)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        from precision_flash_attention_gb300 import build as _b
        with open(p, encoding="utf-8") as f:
            j = json.load(f)
        e = j.get(kernel)
        if not e or e.get("source_digest") != _b.kernel_source_digest(kernel):
            return None
        return e.get("dram_bytes_per_launch_full_workload")
    except (OSError, ValueError, KeyError):
        return None


_SI = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12}


def write_traffic(csv_path: str, kernel: str, command: str) -> dict:
    """Average DRAM bytes (read + write) per launch of `kernel` from an ncu --csv capture
    of dram__bytes_read.sum and dram__bytes_write.sum, stored in profiles/traffic.json
    under the digest of the kernel's current sources (so a later change to them reads as
    null)."""
    import csv
    from precision_flash_attention_gb300 import build as _b
    per_launch = {}
    with open(csv_path, encoding="utf-8") as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for row in csv.DictReader(lines):
        if kernel not in row.get("Kernel Name", ""):
            continue
        name = row.get("Metric Name", "")
        if name not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        val = float(row["Metric Value"].replace(",", "")) * _SI.get(row.get("Metric Unit", "byte"), 1.0)
        per_launch[row["ID"]] = per_launch.get(row["ID"], 0.0) + val
    if not per_launch:
        raise SystemExit(f"no dram__bytes rows for {kernel} in {csv_path}")
    p = os.path.join(ROOT, "profiles", "traffic.json")
    data = {}
    if os.path.exists(p):
        with open(p, encoding="utf-8") as f:
            data = json.load(f)
    data[kernel] = {"dram_bytes_per_launch_full_workload": sum(per_launch.values()) / len(per_launch),
                    "launches": len(per_launch), "source_digest": _b.kernel_source_digest(kernel),
                    "workload": dict(WORKLOAD), "command": command}
    with open(p, "w", encoding="utf-8") as f:
        json.dump(data, f, indent=1, sort_keys=True)
        f.write("\n")
    return data[kernel]


# ----------------------------------------------------------------------------- GPU arm
def make_inputs(device, B, H, N, d, seed=0):
    from precision_flash_attention_gb300 import inputs
    t = inputs.gaussian(B, H, H, N, d, std_qkv=0.5, std_do=1e-2, seed=seed)
    return {n: x.to(device) for n, x in t.items()}


class Step:
    """Buffers and launch sequence of one forward + backward step (GQA when k has fewer heads
    than q). ``delta_mode`` 0 takes delta = rowsum(dO o O), 1 delta = rowsum(dP o P)."""

    def __init__(self, t, *, causal, scale, fix_mode, beta, eps, delta_mode=0):
        import precision_flash_attention_gb300 as pfa
        self.pfa = pfa
        self.t = t
        q = t["q"]
        B, H, N, d = q.shape
        self.kw = dict(causal=causal, scale=scale)
        self.fkw = dict(fix_mode=fix_mode, beta=beta, eps=eps)
        self.delta_mode = delta_mode
        self.o = torch.empty_like(q)
        self.lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
        self.delta = torch.empty_like(self.lse)
        self.delta_alt = torch.empty_like(self.lse)
        self.dq, self.dk, self.dv = (torch.empty_like(t[n]) for n in ("q", "k", "v"))
        self.ws = torch.empty(pfa.bwd_workspace_bytes(B, H, N, d) // 4, dtype=torch.float32,
                              device=q.device)
        # As pfa.backward does: at d = 64 with delta = rowsum(dO o O), the delta pass also
        # zeroes the dQ workspace (pfa_attn_delta_zero) and the backward call skips its own
        # zeroing pass.
        self.fused_zero = delta_mode == 0 and d == 64

    def fwd(self):
        t = self.t
        self.pfa.attn_fwd(t["q"], t["k"], t["v"], self.o, self.lse, **self.kw, **self.fkw)

    def delta_(self):
        if self.delta_mode == 0:
            if self.fused_zero:
                self.pfa.attn_delta_zero(self.o, self.t["do"], self.delta, self.ws)
            else:
                self.pfa.attn_delta(self.o, self.t["do"], self.delta)
        else:
            self.delta_alt_(self.delta)

    def delta_alt_(self, out=None):
        t = self.t
        self.pfa.attn_delta_alt(t["q"], t["k"], t["v"], t["do"], self.lse,
                                self.delta_alt if out is None else out, **self.kw)

    def bwd(self):
        t = self.t
        self.pfa.attn_bwd(t["q"], t["k"], t["v"], t["do"], self.lse, self.delta, self.dq, self.dk,
                          self.dv, self.ws, workspace_zeroed=self.fused_zero, **self.kw)

    def bwd_ex(self, flags):
        """The backward call with pfa_attn_bwd_ex options (the query-outer dQ pass)."""
        t = self.t
        self.pfa.attn_bwd_ex(t["q"], t["k"], t["v"], t["do"], self.lse, self.delta, self.dq, self.dk,
                             self.dv, None, flags=flags, **self.kw)

    def bwd_kernel(self):
        """The backward kernel alone (pfa_attn_bwd_accum into the zeroed FP32 workspace)."""
        t = self.t
        self.pfa.attn_bwd_accum(t["q"], t["k"], t["v"], t["do"], self.lse, self.delta,
                                self.ws.view(t["q"].shape), self.dk, self.dv, **self.kw)

    def run(self):
        self.fwd()
        self.delta_()
        self.bwd()


def time_step(step, steps, warmup, flush, split=False):
    """CUDA-event timing of whole steps on the launching stream; L2 flushed before each
    step. The kernels of a step overlap their neighbours (programmatic dependent launch),
    so events go only at the step's ends; with `split` they also go between the calls,
    which serialises them, to give each call's own duration (and the backward kernel, and
    delta = rowsum(dP o P), each timed by itself)."""
    for _ in range(warmup):
        flush.fill_(1.0)
        step.run()
    torch.cuda.synchronize()
    rec = []
    for _ in range(steps):
        flush.fill_(1.0)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4 if split else 2)]
        e[0].record()
        step.fwd()
        if split:
            e[1].record()
        step.delta_()
        if split:
            e[2].record()
        step.bwd()
        e[-1].record()
        rec.append(e)
    torch.cuda.synchronize()
    out = {"step_ms": [a[0].elapsed_time(a[-1]) for a in rec]}
    if split:
        out.update(fwd_ms=[a[0].elapsed_time(a[1]) for a in rec],
                   delta_ms=[a[1].elapsed_time(a[2]) for a in rec],
                   bwd_ms=[a[2].elapsed_time(a[3]) for a in rec])

        def alone(fn, before=None):
            # One call by itself: L2 flushed (and `before` run) outside the events.
            kr = []
            for _ in range(steps):
                flush.fill_(1.0)
                if before is not None:
                    before()
                e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
                e[0].record()
                fn()
                e[1].record()
                kr.append(e)
            torch.cuda.synchronize()
            return [a[0].elapsed_time(a[1]) for a in kr]

        out["bwd_kernel_ms"] = alone(step.bwd_kernel, step.ws.zero_)
        out["delta_alt_ms"] = alone(step.delta_alt_)
        out["bwd_det_ms"] = alone(lambda: step.bwd_ex(1))
        out["bwd_split_ms"] = alone(lambda: step.bwd_ex(3))
    return out


def time_interleaved(steps_by_mode, k, flush):
    """Whole steps of each mode in turn, k rounds, L2 flushed before each step and CUDA
    events at each step's ends. Everything is enqueued before one synchronisation, so the
    host runs ahead of the GPU and its own launch work never shows in the device times.
    Returns the step times per mode (ms)."""
    rec = {m: [] for m in steps_by_mode}
    for _ in range(k):
        for m, st in steps_by_mode.items():
            flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            st.run()
            e1.record()
            rec[m].append((e0, e1))
    torch.cuda.synchronize()
    return {m: [a.elapsed_time(b) for a, b in v] for m, v in rec.items()}


def interleaved_step_ms(steps_by_mode, k, flush):
    """Median whole-step time per mode, the modes interleaved step by step (one step of each
    in turn, L2 flushed before each), so that they are compared under the same conditions."""
    for st in steps_by_mode.values():
        time_step(st, 1, 2, flush)
    times = time_interleaved(steps_by_mode, k, flush)
    return {m: statistics.median(v) for m, v in times.items()}


def measure_study(t, w, flush, k, peak):
    """Forward time of the study variants of pfa_attn_fwd_ex on the bench workload (mode 1):
    the fused kernel with its counters, the training-time monitor, the unfused BF16 Pbar V
    profile and the FP8 E4M3 / MXFP4 Pbar formats. The variants are interleaved one call at
    a time, L2 flushed before each, all enqueued before one synchronisation."""
    import precision_flash_attention_gb300 as pfa
    q = t["q"]
    B, H, N, d = q.shape
    o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    cnt, mon = pfa.new_counters(q.device), pfa.new_monitor(q.device)
    kw = dict(causal=True, scale=w["scale"], fix_mode=1, beta=w["beta"], eps=w["eps"])
    variants = {
        "fused": lambda: pfa.attn_fwd(q, t["k"], t["v"], o, lse, **kw),
        "fused + counters": lambda: pfa.attn_fwd(q, t["k"], t["v"], o, lse, counters=cnt, **kw),
        "monitor": lambda: pfa.attn_fwd_ex(q, t["k"], t["v"], o, lse, counters=cnt, monitor=mon, **kw),
        "unfused BF16 Pbar V profile": lambda: pfa.attn_fwd_ex(
            q, t["k"], t["v"], o, lse, monitor=mon, flags=pfa.FWD_UNFUSED_BF16_PV, **kw),
        "Pbar FP8 E4M3": lambda: pfa.attn_fwd_ex(q, t["k"], t["v"], o, lse, monitor=mon,
                                                 flags=pfa.FWD_PBAR_E4M3, **kw),
        "Pbar MXFP4": lambda: pfa.attn_fwd_ex(q, t["k"], t["v"], o, lse, monitor=mon,
                                              flags=pfa.FWD_PBAR_MXFP4, **kw),
    }
    for fn in variants.values():
        for _ in range(2):
            flush.fill_(1.0)
            fn()
    rec = {n: [] for n in variants}
    for _ in range(k):
        for n, fn in variants.items():
            flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            rec[n].append((e0, e1))
    torch.cuda.synchronize()
    f_fwd = flops(B, H, N, d, True, "fwd")
    med = {n: statistics.median(a.elapsed_time(b) for a, b in v) for n, v in rec.items()}
    return {n: {"fwd_ms": m, "fwd_tflops": f_fwd / m / 1e9, "fwd_frac_bf16_peak": f_fwd / m / 1e9 / peak,
                "vs_fused_pct": 100.0 * (m / med["fused"] - 1.0)} for n, m in med.items()}


def time_fwd_pair(t, wl, modes, flush, k):
    """Forward time of the CTA-paired variant (FWD_PAIR_CTA: the two CTAs of a cluster share
    every product, d = 128) and of the one-CTA fused forward, per mode, interleaved one call
    at a time, L2 flushed before each, all enqueued before one synchronisation."""
    import precision_flash_attention_gb300 as pfa
    q = t["q"]
    o, lse = torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    calls = {}
    for m in modes:
        kw = dict(causal=wl.causal, scale=wl.alpha, fix_mode=m, beta=wl.beta, eps=wl.eps)
        for pair in (False, True):
            calls[(m, pair)] = (lambda kw=kw, fl=pfa.FWD_PAIR_CTA if pair else 0:
                                pfa.attn_fwd_ex(q, t["k"], t["v"], o, lse, flags=fl, **kw))
    for fn in calls.values():
        for _ in range(2):
            flush.fill_(1.0)
            fn()
    rec = {c: [] for c in calls}
    for _ in range(k):
        for c, fn in calls.items():
            flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            rec[c].append((e0, e1))
    torch.cuda.synchronize()
    med = {c: statistics.median(a.elapsed_time(b) for a, b in v) for c, v in rec.items()}
    return {m: {"one": med[(m, False)], "pair": med[(m, True)]} for m in modes}


# The other configured workloads, each timed in every mode it lists (tests check them against
# the oracle; here they are measured). Mode 2 is added for the GPT-2 layer.
OTHER_WORKLOADS = [
    ("tiny", "C1 tiny: B=1 H=1 N=64 d=64 non-causal"),
    ("gpt2", "C2 GPT-2-small layer: B=8 H=12 N=1024 d=64 causal (all three modes)"),
    ("sink", "C3 sink-heavy: B=4 H=12 N=2048 d=64 causal, delta = rowsum(dP o P)"),
    ("long", "C4 long context: B=2 H=16 N=8192 d=128 causal, beta=4"),
    ("gqa", "C5 Llama-3.1-8B-style GQA: B=1 H_q=32 H_kv=8 N=8192 d=128 causal"),
]


def measure_workload(name, device, steps, flush, peaks):
    """fwd, delta, delta-alt, bwd and whole-step timings of one named workload (inputs from
    precision_flash_attention_gb300.inputs) in each of its modes, with algorithmic TFLOP/s
    and fractions of the measured peaks. The sink-heavy step takes delta = rowsum(dP o P)
    (the variant its parity test uses); delta = rowsum(dO o O) is timed too."""
    from precision_flash_attention_gb300 import inputs
    wl = inputs.WORKLOADS[name]
    t = {n: x.to(device) for n, x in inputs.make(name, seed=0).items()}
    B, Hq, N, d = t["q"].shape
    modes = (0, 1, 2) if name == "gpt2" else wl.modes
    peak, hbm = peaks["bf16_tflops"], peaks["hbm_gbs"]
    f_fwd, f_bwd, f_tot, f_alt = (wl.flops(w) for w in ("fwd", "bwd", "fwd+bwd", "delta_alt"))
    # delta reads O and dO and writes delta; at d = 64 the same pass zeroes the dQ workspace.
    dl_bytes = B * Hq * N * (4 * d + 4 + (4 * d if d == 64 else 0))
    out = {}
    sts = {m: Step(t, causal=wl.causal, scale=wl.alpha, fix_mode=m, beta=wl.beta, eps=wl.eps,
                   delta_mode=1 if name == "sink" else 0) for m in modes}
    splits = {m: time_step(sts[m], steps, 2, flush, split=True) for m in modes}
    step_ms_all = interleaved_step_ms(sts, steps, flush)
    pair = time_fwd_pair(t, wl, modes, flush, steps) if d == 128 else None
    for m in modes:
        r = splits[m]
        med = {k: statistics.median(v) for k, v in r.items()}
        step_ms = step_ms_all[m]
        e = {"fwd_ms": med["fwd_ms"], "bwd_call_ms": med["bwd_ms"], "bwd_kernel_ms": med["bwd_kernel_ms"],
             "step_ms": step_ms,
             "fwd_tflops": f_fwd / med["fwd_ms"] / 1e9,
             "bwd_tflops": f_bwd / med["bwd_ms"] / 1e9,
             "bwd_kernel_tflops": f_bwd / med["bwd_kernel_ms"] / 1e9,
             "total_tflops": f_tot / step_ms / 1e9}
        for k in ("fwd", "bwd", "bwd_kernel", "total"):
            e[k + "_frac_bf16_peak"] = e[k + "_tflops"] / peak
        e["delta_alt_ms"] = med["delta_alt_ms"]
        e["delta_alt_tflops"] = f_alt / med["delta_alt_ms"] / 1e9
        # The backward call with the query-outer dQ pass: deterministic dQ, and with the hi/lo
        # BF16 dS (algorithmic FLOPs as above; the pass recomputes S and dP).
        for k in ("det", "split"):
            e[f"bwd_{k}_ms"] = med[f"bwd_{k}_ms"]
            e[f"bwd_{k}_tflops"] = f_bwd / med[f"bwd_{k}_ms"] / 1e9
        if pair is not None:
            # The CTA-paired forward against the one-CTA forward timed beside it.
            e["fwd_pair_ms"] = pair[m]["pair"]
            e["fwd_pair_tflops"] = f_fwd / pair[m]["pair"] / 1e9
            e["fwd_pair_vs_one_cta_pct"] = 100.0 * (pair[m]["pair"] / pair[m]["one"] - 1.0)
        if name != "sink":
            e["delta_ms"] = med["delta_ms"]
            e["delta_gbs"] = dl_bytes / med["delta_ms"] / 1e6
            e["delta_frac_hbm_peak"] = e["delta_gbs"] / hbm
        else:
            e["step_note"] = "step = fwd + delta_alt + bwd; total_tflops counts fwd+bwd FLOPs only"
        out[f"mode {m}"] = e
    del sts, t
    torch.cuda.empty_cache()
    return {"shape": dict(B=B, H_q=Hq, H_kv=wl.H_kv, N=N, d=d, causal=wl.causal, alpha=wl.alpha,
                          beta=wl.beta, eps=wl.eps),
            "flops": {"fwd": f_fwd, "bwd": f_bwd, "fwd+bwd": f_tot, "delta_alt": f_alt},
            "delta_bytes": dl_bytes, "steps": steps, "modes": out}


def e2e_time(make_step, steps, warmup):
    """The step through the public API with every step's inputs copied in from pinned host
    memory and its outputs (O, lse, dQ, dK, dV) copied back, pipelined the way a training
    loop feeds a GPU: step k+1's inputs upload on one copy stream while step k computes,
    and step k's outputs download on another. Two sets of device buffers alternate.
    Returns ms per step (the span of the K steps / K) and the bytes copied per step."""
    bufs = [make_step(), make_step()]
    outs = lambda st: [st.o, st.lse, st.dq, st.dk, st.dv]  # noqa: E731
    host_in = {n: x.cpu().pin_memory() for n, x in bufs[0].t.items()}
    host_out = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in outs(bufs[0])]
    h2d = sum(x.numel() * x.element_size() for x in host_in.values())
    d2h = sum(x.numel() * x.element_size() for x in outs(bufs[0]))
    cmp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def run(n):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(cmp)
        s_in.wait_event(start)
        s_out.wait_event(start)
        ev_in, ev_done, ev_out = [None] * n, [None] * n, [None] * n

        def upload(k):
            b = bufs[k % 2]
            if k >= 2:
                s_in.wait_event(ev_done[k - 2])  # the buffer's last step has read its inputs
            with torch.cuda.stream(s_in):
                for name, x in host_in.items():
                    b.t[name].copy_(x, non_blocking=True)
            ev_in[k] = torch.cuda.Event()
            ev_in[k].record(s_in)

        upload(0)
        for k in range(n):
            b = bufs[k % 2]
            if k + 1 < n:
                upload(k + 1)
            cmp.wait_event(ev_in[k])
            if k >= 2:
                cmp.wait_event(ev_out[k - 2])  # the buffer's last outputs have been copied out
            b.run()
            ev_done[k] = torch.cuda.Event()
            ev_done[k].record(cmp)
            s_out.wait_event(ev_done[k])
            with torch.cuda.stream(s_out):
                for h, d in zip(host_out, outs(b)):
                    h.copy_(d, non_blocking=True)
            ev_out[k] = torch.cuda.Event()
            ev_out[k].record(s_out)
        cmp.wait_event(ev_out[n - 1])
        end.record(cmp)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / n

    run(max(2, warmup))
    return run(steps), h2d, d2h


def cpu_baseline(sample_heads=48, seed=0, min_seconds=0.0, max_reps=30):
    """The oracle (float64 numpy, as it stands) on a bounded sample of the workload:
    ``sample_heads`` (b, h) heads of the GPT-2 layer, forward + delta + backward,
    repeated until ``min_seconds`` of CPU work (at most ``max_reps`` passes)."""
    import oracle
    from precision_flash_attention_gb300 import inputs
    w = WORKLOAD
    t = inputs.gaussian(1, sample_heads, sample_heads, w["N"], w["d"], std_qkv=0.5, std_do=1e-2,
                        seed=seed)
    a = {n: x.to(torch.float64).numpy() for n, x in t.items()}
    reps, dt = 0, 0.0
    while reps < max_reps and (reps == 0 or dt < min_seconds):
        t0 = time.perf_counter()
        f = oracle.attn_fwd(a["q"], a["k"], a["v"], causal=True, scale=w["scale"], fix_mode=1,
                            beta=w["beta"], eps=w["eps"])
        dl = oracle.attn_delta(f["o"], a["do"])
        oracle.attn_bwd(a["q"], a["k"], a["v"], a["do"], f["lse"], dl, causal=True, scale=w["scale"])
        dt += time.perf_counter() - t0
        reps += 1
    fl = reps * flops(1, sample_heads, w["N"], w["d"], True)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{sample_heads} of 96 (b,h) heads of B=8,H=12,N=1024,d=64 causal, "
                      f"fwd(mode 1)+delta+bwd in float64 numpy, {reps} pass(es) in {dt:.2f} s",
            "seconds": dt}


def cpu_workloads():
    """The oracle (float64 numpy, as it stands) on one (batch, query head) slice of each
    other configured workload -- forward in the workload's last mode, delta and backward --
    and the time that scales linearly to the whole workload (every head costs the same)."""
    import oracle
    from precision_flash_attention_gb300 import inputs
    out = {}
    for name in ("tiny", "sink", "long", "gqa"):
        wl = inputs.WORKLOADS[name]
        t = inputs.make(name, seed=0)
        g = wl.H_q // wl.H_kv
        a = {n: x[:1, :1].to(torch.float64).numpy() for n, x in t.items() if n in ("q", "do")}
        a.update({n: x[:1, :1].to(torch.float64).numpy() for n, x in t.items() if n in ("k", "v")})
        t0 = time.perf_counter()
        f = oracle.attn_fwd(a["q"], a["k"], a["v"], causal=wl.causal, scale=wl.alpha,
                            fix_mode=wl.modes[-1], beta=wl.beta, eps=wl.eps)
        dl = oracle.attn_delta(f["o"], a["do"])
        oracle.attn_bwd(a["q"], a["k"], a["v"], a["do"], f["lse"], dl, causal=wl.causal,
                        scale=wl.alpha)
        dt = time.perf_counter() - t0
        heads = wl.B * wl.H_q
        fl = wl.flops() / heads
        out[name] = {"slice": f"1 of {heads} (b, h) heads" + (f" (group of {g} shares K, V)" if g > 1 else ""),
                     "slice_seconds": dt, "tflops": fl / dt / 1e12,
                     "extrapolated_seconds_full_workload": dt * heads}
    return out


def _progress(args, msg):
    if args.progress:
        print(f"[bench {time.strftime('%H:%M:%S')}] {msg}", file=sys.stderr, flush=True)


def run_gpu_arm(args):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    __graft_entry__.build()
    import precision_flash_attention_gb300 as pfa

    w = dict(WORKLOAD)
    if args.n:
        w["N"] = args.n
    if args.d:
        w["d"] = args.d
        w["scale"] = 1.0 / math.sqrt(args.d)
    peaks = load_peaks()
    t = make_inputs(dev, w["B"], w["H"], w["N"], w["d"], seed=rank)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    if args.fwd_pair:
        # Profiling run: the forward alone, the one-CTA and the CTA-paired kernel
        # alternating (warm-up calls included), L2 flushed before each; prints nothing.
        if w["d"] != 128:
            raise SystemExit("--fwd-pair needs --d 128")
        o = torch.empty_like(t["q"])
        lse = torch.empty(t["q"].shape[:3], dtype=torch.float32, device=dev)
        for _ in range(args.warmup + args.steps):
            for fl in (0, pfa.FWD_PAIR_CTA):
                flush.fill_(1.0)
                pfa.attn_fwd_ex(t["q"], t["k"], t["v"], o, lse, causal=w["causal"], scale=w["scale"],
                                fix_mode=args.mode, beta=w["beta"], eps=w["eps"], flags=fl)
        torch.cuda.synchronize()
        assert pfa.device_error() == 0, "device error word set during the forward run"
        return
    head = args.mode
    # Modes 0, 1 and 2 interleaved in the timed region: the headline is `head` (1 by
    # default), and the cost of each fix mode is read against mode 0 under the same load.
    steps = {m: Step(t, causal=w["causal"], scale=w["scale"], fix_mode=m, beta=w["beta"],
                     eps=w["eps"]) for m in sorted({0, 1, 2, head})}
    # Clocks are sampled from before the warm-up (so sampling is live when timing
    # starts) until after an untimed tail of the same steps; not under ncu.
    clk = _NoClock() if args.kernels_only else ClockSampler(local)
    with clk:
        clk.wait_first()
        for m in steps:
            _progress(args, f"warm-up mode {m}")
            time_step(steps[m], 1, args.warmup, flush)
            _progress(args, f"warm-up mode {m} done, device error word {pfa.device_error()}")
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        # Interleave the modes so the cost of the fix is measured under the same conditions.
        # One pass = K steps of each mode. The timed region repeats the pass until it spans
        # several clock-sampling periods (a pass of the bench workload takes a few ms, less
        # than one period); the line reports K and the number of passes.
        def one_pass(res, log):
            if log and args.progress:
                # Diagnostic run: one step at a time, each checked for a device error.
                for it in range(args.steps):
                    for m in steps:
                        r = time_step(steps[m], 1, 0, flush)
                        res[m]["step_ms"] += r["step_ms"]
                        err = pfa.device_error()
                        _progress(args, f"step {it} mode {m}: {r['step_ms'][0]:.3f} ms, error word {err}"
                                        + (f", first timeout at {pfa.device_error_site()}" if err else ""))
                return
            r = time_interleaved(steps, args.steps, flush)
            for m in r:
                res[m]["step_ms"] += r[m]

        passes = 1
        if not args.kernels_only:
            cal0 = time.perf_counter()
            one_pass({m: {"step_ms": []} for m in steps}, False)
            per_pass = time.perf_counter() - cal0
            passes = max(1, min(50, math.ceil(TIMED_REGION_MIN_S / max(per_pass, 1e-6))))
            if world > 1:
                t_p = torch.tensor([passes], dtype=torch.int64, device=dev)
                torch.distributed.all_reduce(t_p, op=torch.distributed.ReduceOp.MAX)
                passes = int(t_p.item())
        res = {m: {"step_ms": []} for m in steps}
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        clk.mark_start()
        wall0 = time.perf_counter()
        for _ in range(passes):
            one_pass(res, True)
        if world > 1:
            torch.distributed.barrier()
        wall = time.perf_counter() - wall0
        clk.mark_end()
        # Untimed tail under the same load, so a sample follows a short timed region.
        if not args.kernels_only:
            tail0 = time.perf_counter()
            for _ in range(2000):
                time_step(steps[head], 1, 0, flush)
                if time.perf_counter() - tail0 > 4 * ClockSampler.PERIOD_MS * 1e-3:
                    break
            torch.cuda.synchronize()
        # Each call's own duration: the same K steps again with events between the calls
        # (not part of the step time above).
        if not args.kernels_only:
            split = {m: time_step(steps[m], args.steps, 0, flush, split=True) for m in steps}
    assert pfa.device_error() == 0, "device error word set during the benchmark"
    if args.kernels_only:
        # Profiling run: the kernels above are all it launches (no sweep, copies or CPU work).
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    mean = lambda xs: sum(xs) / len(xs)  # noqa: E731
    ms = mean(res[head]["step_ms"])
    ms = max_over_ranks(ms, world, dev)
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    f_total = flops(B, H, N, d, True)
    value = world * f_total / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]

    fwd_ms, dl_ms, bwd_ms, bk_ms = (mean(split[head][k])
                                    for k in ("fwd_ms", "delta_ms", "bwd_ms", "bwd_kernel_ms"))
    f_fwd, f_bwd = flops(B, H, N, d, True, "fwd"), flops(B, H, N, d, True, "bwd")
    # delta reads O and dO and writes delta; at d = 64 the same pass zeroes the dQ workspace.
    dl_bytes = B * H * N * (4 * d + 4 + (4 * d if d == 64 else 0))
    kernels = {
        "attn_fwd": {"ms": fwd_ms, "TFLOP/s": f_fwd / fwd_ms / 1e9,
                     "frac_bf16_peak": f_fwd / fwd_ms / 1e9 / peak},
        "attn_delta": {"ms": dl_ms, "GB/s": dl_bytes / dl_ms / 1e6,
                       "frac_hbm_peak": dl_bytes / dl_ms / 1e6 / peaks["hbm_gbs"]},
        "attn_bwd": {"ms": bwd_ms, "TFLOP/s": f_bwd / bwd_ms / 1e9,
                     "frac_bf16_peak": f_bwd / bwd_ms / 1e9 / peak,
                     "note": "the backward call: kernel and dQ conversion (the delta pass zeroed the "
                             "workspace)"},
        "attn_bwd_kernel": {"ms": bk_ms, "TFLOP/s": f_bwd / bk_ms / 1e9,
                            "frac_bf16_peak": f_bwd / bk_ms / 1e9 / peak},
    }
    # Dominant kernel: the one with the largest share of the step, timed by itself.
    dom = "attn_bwd" if bwd_ms >= fwd_ms else "attn_fwd"
    ach = kernels["attn_bwd_kernel" if dom == "attn_bwd" else "attn_fwd"]["TFLOP/s"]
    roof = {"kernel": dom + "_kernel", "bound": "tensor", "achieved": ach, "peak": peak,
            "unit": "TFLOP/s", "frac": ach / peak,
            "peak_source": f"{peaks['source']} bf16 burst (cuBLAS), of measured"
            if peaks["source"] == "measured" else "fallback bf16 burst",
            "traffic": traffic_for(dom + "_kernel")}
    mode_tflops = {str(m): f_total / (mean(r["step_ms"]) * 1e-3) / 1e12 for m, r in res.items()}
    overhead = (100.0 * (mean(res[head]["step_ms"]) / mean(res[0]["step_ms"]) - 1.0)
                if head != 0 else None)
    overhead_all = {str(m): 100.0 * (mean(res[m]["step_ms"]) / mean(res[0]["step_ms"]) - 1.0)
                    for m in res if m != 0}

    sweep = {}
    _progress(args, f"timed steps done: {ms:.3f} ms per step")
    if args.sweep and rank == 0:
        for n_s in (2048, 4096, 8192, 16384):
            ts = make_inputs(dev, B, H, n_s, d, seed=1)
            k_s = max(3, args.steps // 2)
            sts = {m: Step(ts, causal=True, scale=w["scale"], fix_mode=m, beta=w["beta"], eps=w["eps"])
                   for m in (0, 1, 2)}
            split_s = {}
            for m in sts:
                _progress(args, f"sweep N={n_s} mode {m}")
                split_s[m] = time_step(sts[m], k_s, 2, flush, split=True)
            tot_ms = interleaved_step_ms(sts, k_s, flush)
            for m in (0, 1, 2):
                r = split_s[m]
                fm, bm, km = (statistics.median(r[k]) for k in ("fwd_ms", "bwd_ms", "bwd_kernel_ms"))
                sm = tot_ms[m]
                tot = flops(B, H, n_s, d, True) / sm / 1e9
                sweep[f"N={n_s},mode={m}"] = {
                    "fwd_tflops": flops(B, H, n_s, d, True, "fwd") / fm / 1e9,
                    "bwd_tflops": flops(B, H, n_s, d, True, "bwd") / bm / 1e9,
                    "bwd_kernel_tflops": flops(B, H, n_s, d, True, "bwd") / km / 1e9,
                    "total_tflops": tot, "total_frac_bf16_peak": tot / peak}
                if m > 0:
                    sweep[f"N={n_s},mode={m}"]["overhead_vs_mode0_pct"] = 100.0 * (sm / tot_ms[0] - 1.0)
            del sts, ts
    study = None
    if args.sweep and rank == 0 and w["d"] == 64:
        _progress(args, "study variants")
        study = measure_study(t, w, flush, max(5, args.steps // 2), peak)
    workloads = {}
    if args.sweep and rank == 0:
        for name, label in OTHER_WORKLOADS:
            _progress(args, f"workload {name}")
            workloads[label] = measure_workload(name, dev, max(5, args.steps // 2), flush, peaks)
        assert pfa.device_error() == 0, "device error word set while timing the workloads"

    _progress(args, f"sweep done, device error word {pfa.device_error()}")
    e2e = None
    if rank == 0:
        st0 = steps[head]
        e_ms_mean, h2d, d2h = e2e_time(
            lambda: Step({n: x.clone() for n, x in st0.t.items()}, causal=w["causal"], scale=w["scale"],
                         fix_mode=head, beta=w["beta"], eps=w["eps"]),
            args.steps, args.warmup)
        e2e = {"value": world * f_total / (e_ms_mean * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms_mean}

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    _progress(args, "e2e done; CPU baseline")
    cpu = cpu_baseline(sample_heads=48, min_seconds=10.0)
    if args.sweep:
        cpu["workloads"] = cpu_workloads()
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.25) Q/K/V, N(0,1e-4) dO)",
        "config": dict(workload_config(world, head, w), l2="flushed (256 MiB write) before every step"),
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": LAUNCHES_PER_STEP * args.steps * len(steps) * passes,
        "timed_passes": passes, "clocks": clk.summary(), "wall_s_timed_region": wall,
        "kernels": kernels, "mode_tflops": mode_tflops, "mode_overhead_pct": overhead,
        "mode_overhead_pct_all": overhead_all, "sweep": sweep, "workloads": workloads,
        "study": study,
        "peaks": peaks,
    }
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of the ranks' values (the slowest rank's step time sets the job's
    time); `x` itself on one rank. Every rank must call it."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def workload_config(world, mode, w=WORKLOAD):
    """The `config` object both arms report for the bench workload `w`."""
    return {"workload": "GPT-2-small attention layer fwd+bwd", "B": w["B"], "H": w["H"], "N": w["N"],
            "d": w["d"], "causal": w["causal"], "fix_mode": mode, "beta": w["beta"], "eps": w["eps"],
            "parallelism": f"replicas x{world}"}


def run_reference_arm(args):
    """The oracle as it stands on the host cores, one bounded sample per step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    for _ in range(args.warmup):
        cpu_baseline(sample_heads=4)
    vals, secs = [], []
    for _ in range(args.steps):
        c = cpu_baseline(sample_heads=4)
        vals.append(c["value"])
        secs.append(c["seconds"])
    v = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(world, args.mode),
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": "4 of 96 (b,h) heads per step, fwd+delta+bwd, float64 numpy"},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--mode", type=int, default=1, choices=[0, 1, 2])
    ap.add_argument("--no-sweep", dest="sweep", action="store_false")
    ap.add_argument("--n", type=int, default=0, help="override the sequence length (profiling)")
    ap.add_argument("--d", type=int, default=0, choices=[0, 64, 128],
                    help="override the head dimension, scale 1/sqrt(d) (profiling; d = 128 runs the "
                         "query-outer dQ pass)")
    ap.add_argument("--progress", action="store_true", help="log each stage to stderr")
    ap.add_argument("--fwd-pair", action="store_true",
                    help="run only the forward, one-CTA and CTA-paired alternating (with --d 128; "
                         "for ncu captures); prints nothing")
    ap.add_argument("--kernels-only", action="store_true",
                    help="launch only the timed steps (for ncu captures); prints nothing")
    ap.add_argument("--traffic-from", metavar="CSV",
                    help="store the attn_bwd_kernel DRAM bytes per launch of an ncu --csv capture "
                         "in profiles/traffic.json and exit (no GPU work)")
    ap.add_argument("--traffic-command", default="", help="the ncu command line of that capture")
    args = ap.parse_args()
    if args.traffic_from:
        print(json.dumps(write_traffic(args.traffic_from, "attn_bwd_kernel", args.traffic_command)))
        return
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        run_reference_arm(args)
    else:
        run_gpu_arm(args)


if __name__ == "__main__":
    main()
