"""Benchmark: stabilised BF16 attention forward + backward TFLOP/s on GB300.

One step = forward (pfa_attn_fwd) + delta (pfa_attn_delta) + backward
(pfa_attn_bwd, which also zeroes and converts its dQ workspace) over one batch
of the GPT-2-small attention layer (B=8, H=12, N=1024, d=64, causal), inputs
resident in HBM, L2 flushed between steps. Algorithmic FLOPs per step:
14 * B * H * N^2 * d / 2 (S, Pbar V forward; S, dP, dV, dK, dQ backward; causal).

Prints one JSON line (rank 0). ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
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
# Kernels of ours launched per step: attn_fwd, delta, attn_bwd, dQ convert (the
# workspace zeroing is a memset on the stream, not a kernel of this library).
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


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def traffic_for(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current
    sources (null otherwise)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        from precision_flash_attention_gb300 import build as _b
        with open(p, encoding="utf-8") as f:
            j = json.load(f)
        e = j.get(kernel)
        if not e or e.get("source_digest") != _b.source_digest():
            return None
        return e.get("dram_bytes_per_launch_full_workload")
    except (OSError, ValueError, KeyError):
        return None


# ----------------------------------------------------------------------------- GPU arm
def make_inputs(device, B, H, N, d, seed=0):
    from precision_flash_attention_gb300 import inputs
    t = inputs.gaussian(B, H, H, N, d, std_qkv=0.5, std_do=1e-2, seed=seed)
    return {n: x.to(device) for n, x in t.items()}


class Step:
    """Buffers and launch sequence of one forward + backward step."""

    def __init__(self, t, *, causal, scale, fix_mode, beta, eps):
        import precision_flash_attention_gb300 as pfa
        self.pfa = pfa
        self.t = t
        q = t["q"]
        B, H, N, d = q.shape
        self.kw = dict(causal=causal, scale=scale)
        self.fkw = dict(fix_mode=fix_mode, beta=beta, eps=eps)
        self.o = torch.empty_like(q)
        self.lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
        self.delta = torch.empty_like(self.lse)
        self.dq, self.dk, self.dv = (torch.empty_like(t[n]) for n in ("q", "k", "v"))
        self.ws = torch.empty(pfa.bwd_workspace_bytes(B, H, N, d) // 4, dtype=torch.float32,
                              device=q.device)

    def fwd(self):
        t = self.t
        self.pfa.attn_fwd(t["q"], t["k"], t["v"], self.o, self.lse, **self.kw, **self.fkw)

    def delta_(self):
        self.pfa.attn_delta(self.o, self.t["do"], self.delta)

    def bwd(self):
        t = self.t
        self.pfa.attn_bwd(t["q"], t["k"], t["v"], t["do"], self.lse, self.delta, self.dq, self.dk,
                          self.dv, self.ws, **self.kw)

    def run(self):
        self.fwd()
        self.delta_()
        self.bwd()


def time_step(step, steps, warmup, flush):
    """Per-phase CUDA-event timing on the launching stream; L2 flushed before each step."""
    for _ in range(warmup):
        flush.fill_(1.0)
        step.run()
    torch.cuda.synchronize()
    rec = []
    for _ in range(steps):
        flush.fill_(1.0)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record()
        step.fwd()
        e[1].record()
        step.delta_()
        e[2].record()
        step.bwd()
        e[3].record()
        rec.append(e)
    torch.cuda.synchronize()
    return {"fwd_ms": [a[0].elapsed_time(a[1]) for a in rec],
            "delta_ms": [a[1].elapsed_time(a[2]) for a in rec],
            "bwd_ms": [a[2].elapsed_time(a[3]) for a in rec],
            "step_ms": [a[0].elapsed_time(a[3]) for a in rec]}


def e2e_time(step, steps, warmup, flush):
    """Same step through the public API with the inputs copied from pinned host memory and
    the outputs (O, lse, dQ, dK, dV) copied back, all inside the timed region."""
    host_in = {n: x.cpu().pin_memory() for n, x in step.t.items()}
    outs = [step.o, step.lse, step.dq, step.dk, step.dv]
    host_out = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in outs]
    h2d = sum(x.numel() * x.element_size() for x in host_in.values())
    d2h = sum(x.numel() * x.element_size() for x in outs)

    def one():
        for n, x in host_in.items():
            step.t[n].copy_(x, non_blocking=True)
        step.run()
        for h, d in zip(host_out, outs):
            h.copy_(d, non_blocking=True)

    for _ in range(warmup):
        flush.fill_(1.0)
        one()
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        flush.fill_(1.0)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        one()
        b.record()
        ts.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ts], h2d, d2h


def cpu_baseline(sample_heads=48, seed=0):
    """The oracle (float64 numpy, as it stands) on a bounded sample of the workload:
    ``sample_heads`` (b, h) heads of the GPT-2 layer, forward + delta + backward."""
    import oracle
    from precision_flash_attention_gb300 import inputs
    w = WORKLOAD
    t = inputs.gaussian(1, sample_heads, sample_heads, w["N"], w["d"], std_qkv=0.5, std_do=1e-2,
                        seed=seed)
    a = {n: x.to(torch.float64).numpy() for n, x in t.items()}
    t0 = time.perf_counter()
    f = oracle.attn_fwd(a["q"], a["k"], a["v"], causal=True, scale=w["scale"], fix_mode=1,
                        beta=w["beta"], eps=w["eps"])
    dl = oracle.attn_delta(f["o"], a["do"])
    oracle.attn_bwd(a["q"], a["k"], a["v"], a["do"], f["lse"], dl, causal=True, scale=w["scale"])
    dt = time.perf_counter() - t0
    fl = flops(1, sample_heads, w["N"], w["d"], True)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{sample_heads} of 96 (b,h) heads of B=8,H=12,N=1024,d=64 causal, "
                      f"fwd(mode 1)+delta+bwd in float64 numpy, {dt:.2f} s",
            "seconds": dt}


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
    peaks = load_peaks()
    t = make_inputs(dev, w["B"], w["H"], w["N"], w["d"], seed=rank)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    head = args.mode
    steps = {m: Step(t, causal=w["causal"], scale=w["scale"], fix_mode=m, beta=w["beta"],
                     eps=w["eps"]) for m in sorted({0, head})}
    for m in steps:
        _progress(args, f"warm-up mode {m}")
        time_step(steps[m], 1, args.warmup, flush)
        _progress(args, f"warm-up mode {m} done, device error word {pfa.device_error()}")
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # Interleave the modes so the cost of the fix is measured under the same conditions.
    res = {m: {"fwd_ms": [], "delta_ms": [], "bwd_ms": [], "step_ms": []} for m in steps}
    wall0 = time.perf_counter()
    with ClockSampler(local) as clk:
        for it in range(args.steps):
            for m in steps:
                r = time_step(steps[m], 1, 0, flush)
                for k2 in r:
                    res[m][k2] += r[k2]
                if args.progress:
                    err = pfa.device_error()
                    _progress(args, f"step {it} mode {m}: {r['step_ms'][0]:.3f} ms, error word {err}"
                                    + (f", first timeout at {pfa.device_error_site()}" if err else ""))
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - wall0
    assert pfa.device_error() == 0, "device error word set during the benchmark"
    if args.kernels_only:
        # Profiling run: the kernels above are all it launches (no sweep, copies or CPU work).
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    mean = lambda xs: sum(xs) / len(xs)  # noqa: E731
    ms = mean(res[head]["step_ms"])
    if world > 1:
        tt = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        ms = float(tt.item())
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    f_total = flops(B, H, N, d, True)
    value = world * f_total / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]

    fwd_ms, dl_ms, bwd_ms = (mean(res[head][k]) for k in ("fwd_ms", "delta_ms", "bwd_ms"))
    f_fwd, f_bwd = flops(B, H, N, d, True, "fwd"), flops(B, H, N, d, True, "bwd")
    dl_bytes = B * H * N * (4 * d + 4)
    kernels = {
        "attn_fwd": {"ms": fwd_ms, "TFLOP/s": f_fwd / fwd_ms / 1e9,
                     "frac_bf16_peak": f_fwd / fwd_ms / 1e9 / peak},
        "attn_delta": {"ms": dl_ms, "GB/s": dl_bytes / dl_ms / 1e6,
                       "frac_hbm_peak": dl_bytes / dl_ms / 1e6 / peaks["hbm_gbs"]},
        "attn_bwd": {"ms": bwd_ms, "TFLOP/s": f_bwd / bwd_ms / 1e9,
                     "frac_bf16_peak": f_bwd / bwd_ms / 1e9 / peak},
    }
    # Dominant kernel: the one with the largest share of the step.
    dom = "attn_bwd" if bwd_ms >= fwd_ms else "attn_fwd"
    ach = kernels[dom]["TFLOP/s"]
    roof = {"kernel": dom + "_kernel", "bound": "tensor", "achieved": ach, "peak": peak,
            "unit": "TFLOP/s", "frac": ach / peak,
            "peak_source": f"{peaks['source']} bf16 burst (cuBLAS), of measured"
            if peaks["source"] == "measured" else "fallback bf16 burst",
            "traffic": traffic_for(dom + "_kernel")}
    mode_tflops = {str(m): f_total / (mean(r["step_ms"]) * 1e-3) / 1e12 for m, r in res.items()}
    overhead = (100.0 * (mean(res[head]["step_ms"]) / mean(res[0]["step_ms"]) - 1.0)
                if head != 0 else None)

    sweep = {}
    _progress(args, f"timed steps done: {ms:.3f} ms per step")
    if args.sweep and rank == 0:
        for n_s in (2048, 4096, 8192):
            ts = make_inputs(dev, B, H, n_s, d, seed=1)
            for m in sorted({0, head}):
                _progress(args, f"sweep N={n_s} mode {m}")
                st = Step(ts, causal=True, scale=w["scale"], fix_mode=m, beta=w["beta"], eps=w["eps"])
                r = time_step(st, max(3, args.steps // 2), 2, flush)
                fm, bm, sm = (statistics.median(r[k]) for k in ("fwd_ms", "bwd_ms", "step_ms"))
                tot = flops(B, H, n_s, d, True) / sm / 1e9
                sweep[f"N={n_s},mode={m}"] = {
                    "fwd_tflops": flops(B, H, n_s, d, True, "fwd") / fm / 1e9,
                    "bwd_tflops": flops(B, H, n_s, d, True, "bwd") / bm / 1e9,
                    "total_tflops": tot, "total_frac_bf16_peak": tot / peak}
            del ts

    _progress(args, f"sweep done, device error word {pfa.device_error()}")
    e2e = None
    if rank == 0:
        e_ms, h2d, d2h = e2e_time(steps[head], max(3, args.steps // 2), args.warmup, flush)
        e_ms_mean = mean(e_ms)
        e2e = {"value": world * f_total / (e_ms_mean * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms_mean}

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    _progress(args, "e2e done; CPU baseline")
    cpu = cpu_baseline(sample_heads=48)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.25) Q/K/V, N(0,1e-4) dO)",
        "config": {"workload": "GPT-2-small attention layer fwd+bwd", "B": B, "H": H, "N": N,
                   "d": d, "causal": True, "fix_mode": head, "beta": w["beta"], "eps": w["eps"],
                   "l2": "flushed (256 MiB write) before every step",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": LAUNCHES_PER_STEP * args.steps * len(steps),
        "clocks": clk.summary(), "wall_s_timed_region": wall,
        "kernels": kernels, "mode_tflops": mode_tflops, "mode_overhead_pct": overhead,
        "sweep": sweep, "peaks": peaks,
    }
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


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
        "data": "synthetic", "config": {"workload": "GPT-2-small attention layer fwd+bwd",
                                        "B": 8, "H": 12, "N": 1024, "d": 64, "causal": True,
                                        "fix_mode": args.mode},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": "4 of 96 (b,h) heads per step, fwd+delta+bwd, float64 numpy"},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--mode", type=int, default=1, choices=[0, 1, 2])
    ap.add_argument("--no-sweep", dest="sweep", action="store_false")
    ap.add_argument("--n", type=int, default=0, help="override the sequence length (profiling)")
    ap.add_argument("--progress", action="store_true", help="log each stage to stderr")
    ap.add_argument("--kernels-only", action="store_true",
                    help="launch only the timed steps (for ncu captures); prints nothing")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        run_reference_arm(args)
    else:
        run_gpu_arm(args)


if __name__ == "__main__":
    main()
