#!/usr/bin/env python
"""Benchmark of SageBwd-style low-bit attention (quantize + forward + backward)
on GB300: causal-adjusted fwd+bwd TOPS and the fraction of the tensor peak.

One step = the whole hot path on one batch: sage_attn_quantize, sage_attn_fwd,
sage_attn_bwd (8 kernel launches).  Inputs are synthetic, seeded, resident in
HBM; L2 is flushed (256 MiB write) between timed steps, outside the events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (launched by torch.distributed.run) every rank runs an independent
replica of the workload on its own GPU (the path has no cross-GPU exchange);
value = all ranks' work / the slowest rank's time.  --impl reference times the
CPU oracle (the reference arm of this library) on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd+bwd TOPS (causal-adjusted) and % of GB300 INT8/FP8 tensor peak"
UNIT = "TOPS"
KERNELS_PER_STEP = 8  # quantize: 2, forward: 1, backward: 5
FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--heads", type=int, default=None, help="run the workload with this many heads per batch "
                    "entry (a smaller case of the same kernels, for profiling)")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true", help="skip the per-kernel runs of the other "
                    "full-size workloads")
    return ap.parse_args()


def max_over_ranks(v: float, dist, device) -> float:
    """The largest of every rank's v (v itself without a process group): the job's time is
    its slowest rank's."""
    if dist is None:
        return v
    import torch
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"bf16": float(d["bf16_tflops"]), "bf16_sustained": float(d.get("bf16_tflops_sustained", 0) or 0),
                "hbm": float(d["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits", "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names[1:], parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------- profile summaries
def profiled_traffic(kernel: str, workload: str, source_file: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    kernel source as it is now (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
        sha = hashlib.sha256(open(source_file, "rb").read()).hexdigest()
        m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
        m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
        if m_sha and m_b and m_sha.group(1) == sha:
            return float(m_b.group(1))
    except OSError:
        pass
    return None


# ------------------------------------------------------------------ oracle
def oracle_flops(N, D, causal):
    f = 4.0 * N * N * D * (0.5 if causal else 1.0)
    return 3.5 * f


def oracle_sample_run(w, n_prefix: int, bh: int = 0):
    """Oracle quantize + forward + backward on the first n_prefix tokens of one head."""
    import numpy as np
    from bit_trainable_attention_sagebwd_gb300 import workloads as wl
    from oracle import oracle as orc
    hx = wl.head_inputs(w, bh)
    f = {n: wl.bf16_bits_to_f32(a[:n_prefix]).astype(np.float64) for n, a in hx.items()}
    orc.run_head(f["q"], f["k"], f["v"], f["do"], w.causal, w.sm_scale, w.qk_norm, w.k_smooth)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def pick_prefix(w, per_step_budget: float) -> int:
    """Largest sequence prefix (multiple of 128, <= N) whose oracle step fits the budget."""
    n = 128
    t0 = time.perf_counter()
    oracle_sample_run(w, n)
    t = time.perf_counter() - t0
    while n * 2 <= w.N and t * 4.2 <= per_step_budget:
        n *= 2
        t0 = time.perf_counter()
        oracle_sample_run(w, n)
        t = time.perf_counter() - t0
    return n


def cpu_baseline(w, budget_s: float) -> dict:
    """The oracle, as it stands, on a bounded sample of the workload."""
    from oracle import oracle as orc
    orc.build()
    heads, flops, elapsed = 0, 0.0, 0.0
    n = w.N
    # one full head first; if a head does not fit the budget, shrink to a prefix
    t0 = time.perf_counter()
    oracle_sample_run(w, n, 0)
    dt = time.perf_counter() - t0
    if dt > budget_s:
        n = pick_prefix(w, budget_s / 3)
        t0 = time.perf_counter()
        oracle_sample_run(w, n, 0)
        dt = time.perf_counter() - t0
    heads, flops, elapsed = 1, oracle_flops(n, w.D, w.causal), dt
    while elapsed + dt <= budget_s and heads < w.bh:
        t0 = time.perf_counter()
        oracle_sample_run(w, n, heads)
        elapsed += time.perf_counter() - t0
        heads += 1
        flops += oracle_flops(n, w.D, w.causal)
    return {"value": flops / elapsed / 1e12, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{heads} of {w.bh} heads, first {n} of {w.N} tokens each, quantize+fwd+bwd "
                      f"({elapsed:.1f} s, C oracle with OpenMP)"}


# ------------------------------------------------------------ reference arm
def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from oracle import oracle as orc
    orc.build()
    K, W = args.steps, args.warmup
    per_step = max(0.05, 150.0 / max(1, K + W))
    n = pick_prefix(w, per_step)
    for _ in range(W):
        oracle_sample_run(w, n)
    ts = []
    for k in range(K):
        t0 = time.perf_counter()
        oracle_sample_run(w, n, k % w.bh)
        ts.append(time.perf_counter() - t0)
    total = sum(ts)
    fl = oracle_flops(n, w.D, w.causal)
    value = fl * K / total / 1e12
    sample = f"per step: one head, first {n} of {w.N} tokens, quantize+fwd+bwd (C oracle, OpenMP)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": K,
        "warmup": W, "ms_per_step": 1e3 * total / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.note}", "B": w.B, "H": w.H, "N": w.N, "D": w.D,
                   "causal": w.causal, "sample_tokens": n},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------------- ours
def kernel_fractions(flops: dict, fwd_ms: float, bwd_main_ms: float, peaks: dict) -> dict:
    """Achieved TFLOP/s of fwd_kernel and bwd_main_kernel and their fractions of the FP8-equivalent
    peak (2 x measured bf16: the dense INT8/FP8 tensor rate the targets use) and of the executed formats
    (S, dP, dQ, dK on bf16 tensor cores; PV, dV on FP8)."""
    fp8 = 2.0 * peaks["bf16"]
    fa = flops["fwd"] / (fwd_ms * 1e-3) / 1e12
    ba = flops["bwd"] / (bwd_main_ms * 1e-3) / 1e12
    t_exec_fwd = (0.5 * flops["fwd"]) / (peaks["bf16"] * 1e12) + (0.5 * flops["fwd"]) / (fp8 * 1e12)
    t_exec_bwd = (0.8 * flops["bwd"]) / (peaks["bf16"] * 1e12) + (0.2 * flops["bwd"]) / (fp8 * 1e12)
    return {"fwd_kernel": {"achieved": fa, "frac": fa / fp8, "frac_executed_formats": t_exec_fwd / (fwd_ms * 1e-3),
                           "flops_per_launch": flops["fwd"], "avg_launch_ms": fwd_ms},
            "bwd_main_kernel": {"achieved": ba, "frac": ba / fp8,
                                "frac_executed_formats": t_exec_bwd / (bwd_main_ms * 1e-3),
                                "flops_per_launch": flops["bwd"], "avg_launch_ms": bwd_main_ms}}


def other_workload(sa, wl, name, dev, flush, peaks, steps=20):
    """Every launch group of another workload bracketed by events (after 3 warm-up steps, L2
    flushed before each step): per-group ms, step TOPS and the two main kernels' fractions."""
    import numpy as np
    import torch
    w = wl.WORKLOADS[name]
    B, H, N, D = w.B, w.H, w.N, w.D
    x = wl.all_inputs(w)
    t = {n: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev) for n, a in x.items()}
    del x
    ws, bws = sa.alloc_ws(B, H, N, D, dev), sa.alloc_bwd_ws(B, H, N, D, dev)
    o = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(o) for _ in range(3))

    def step():
        sa.quantize(t["q"], t["k"], t["v"], w.qk_norm, w.k_smooth, ws=ws)
        sa.forward(ws, B, H, N, D, w.causal, w.sm_scale, o=o, lse=lse, device=dev)
        sa.backward(t["q"], t["k"], t["v"], o, lse, t["do"], ws, w.causal, w.qk_norm, w.k_smooth, w.sm_scale,
                    bwd_ws=bws, dq=dq, dk=dk, dv=dv)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    groups = ("quantize", "fwd", "bwd_pre", "bwd_main", "bwd_dq")
    for g in groups:
        sa.sage_attn_timer_read(g)
    sa.sage_attn_timer_only(None)
    sa.sage_attn_timer_enable(1)
    for i in range(steps):
        flush.fill_(float(i))
        step()
    torch.cuda.synchronize()
    sa.sage_attn_timer_enable(0)
    if sa.get_status(ws) != sa.SAGE_OK:
        raise SystemExit(f"device status not ok after the {name} steps")
    ms = {g: (lambda r: r[0] / max(1, r[1]))(sa.sage_attn_timer_read(g)) for g in groups}
    ops = w.ops()
    step_ms = sum(ms.values())
    out = {"workload": f"{w.name}: {w.note}", "steps": steps, "kernel_ms_per_step": ms,
           "tops_sum_of_groups": ops["fwd_bwd"] / (step_ms * 1e-3) / 1e12}
    out.update(kernel_fractions(ops, ms["fwd"], ms["bwd_main"], peaks))
    return out


def run_ours(args, w):
    import numpy as np
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    from bit_trainable_attention_sagebwd_gb300 import build as sa_build
    sa_build.build()
    import bit_trainable_attention_sagebwd_gb300 as sa
    from bit_trainable_attention_sagebwd_gb300 import workloads as wl

    B, H, N, D = w.B, w.H, w.N, w.D
    x = wl.all_inputs(w)
    host = {n: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory() for n, a in x.items()}
    t = {n: v.to(dev) for n, v in host.items()}
    ws = sa.alloc_ws(B, H, N, D, dev)
    bws = sa.alloc_bwd_ws(B, H, N, D, dev)
    o = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(o) for _ in range(3))
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def step(q, k, v, do):
        sa.quantize(q, k, v, w.qk_norm, w.k_smooth, ws=ws)
        sa.forward(ws, B, H, N, D, w.causal, w.sm_scale, o=o, lse=lse, device=dev)
        sa.backward(q, k, v, o, lse, do, ws, w.causal, w.qk_norm, w.k_smooth, w.sm_scale, bwd_ws=bws,
                    dq=dq, dk=dk, dv=dv)

    for _ in range(max(3, args.warmup)):
        step(t["q"], t["k"], t["v"], t["do"])
    torch.cuda.synchronize()
    if sa.get_status(ws) != sa.SAGE_OK:
        raise SystemExit("device status not ok after warm-up")

    K = args.steps
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(gpu_id)
    for name in ("quantize", "fwd", "bwd_pre", "bwd_main", "bwd_dq"):
        sa.sage_attn_timer_read(name)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    # inside the timed steps only the dominant kernel is bracketed by events (an event
    # between two launches would end the overlap of each launch with its predecessor)
    sa.sage_attn_timer_only("bwd_main")
    sa.sage_attn_timer_enable(1)
    wall0 = time.perf_counter()
    for i in range(K):
        flush.fill_(float(i))  # 256 MiB write: evicts L2 between steps
        evs[i][0].record(stream)
        step(t["q"], t["k"], t["v"], t["do"])
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    sa.sage_attn_timer_enable(0)
    clk = clocks.stop()
    if dist:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = sum(step_ms)
    bwd_main_timed = sa.sage_attn_timer_read("bwd_main")
    if sa.get_status(ws) != sa.SAGE_OK:
        raise SystemExit("device status not ok after the timed steps")
    # per-group breakdown from a few more steps with every group bracketed (untimed)
    sa.sage_attn_timer_only(None)
    sa.sage_attn_timer_enable(1)
    for i in range(min(K, 20)):
        flush.fill_(float(i))
        step(t["q"], t["k"], t["v"], t["do"])
    torch.cuda.synchronize()
    sa.sage_attn_timer_enable(0)
    ktimes = {name: sa.sage_attn_timer_read(name) for name in ("quantize", "fwd", "bwd_pre", "bwd_main", "bwd_dq")}

    ops = w.ops()

    # ---- the same shape through grouped key/value heads and through Q-smoothing (not part of
    # `value`): median of 20 steps, L2 flushed before each
    def time_variant(fn, ws_status):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        for i in range(20):
            flush.fill_(float(i))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        if sa.get_status(ws_status) != sa.SAGE_OK:
            raise SystemExit("device status not ok after a variant's steps")
        ms = sorted(ts)[len(ts) // 2]
        return {"ms_per_step": ms, "tops": ops["fwd_bwd"] / (ms * 1e-3) / 1e12}

    variants = {}
    for hkv in sorted({H // 4, 1}, reverse=True):
        if hkv < 1 or H % hkv or hkv == H:
            continue
        kg, vg = t["k"][:, :hkv].contiguous(), t["v"][:, :hkv].contiguous()
        wsg, bwsg = sa.alloc_ws(B, H, N, D, dev, hkv), sa.alloc_bwd_ws(B, H, N, D, dev, hkv)
        dkg, dvg = torch.empty_like(kg), torch.empty_like(vg)

        def gstep():
            sa.quantize(t["q"], kg, vg, w.qk_norm, w.k_smooth, ws=wsg)
            sa.forward(wsg, B, H, N, D, w.causal, w.sm_scale, o=o, lse=lse, device=dev, hkv=hkv)
            sa.backward(t["q"], kg, vg, o, lse, t["do"], wsg, w.causal, w.qk_norm, w.k_smooth, w.sm_scale,
                        bwd_ws=bwsg, dq=dq, dk=dkg, dv=dvg)
        variants[f"kv_heads_{hkv}"] = dict(time_variant(gstep, wsg), query_heads_per_kv_head=H // hkv)
        del wsg, bwsg, kg, vg, dkg, dvg
    wsq = sa.alloc_ws(B, H, N, D, dev, None, True)

    def qstep():
        sa.quantize(t["q"], t["k"], t["v"], w.qk_norm, w.k_smooth, ws=wsq, q_smooth=True)
        sa.forward(wsq, B, H, N, D, w.causal, w.sm_scale, o=o, lse=lse, device=dev, q_smooth=True)
        sa.backward(t["q"], t["k"], t["v"], o, lse, t["do"], wsq, w.causal, w.qk_norm, w.k_smooth, w.sm_scale,
                    bwd_ws=bws, dq=dq, dk=dk, dv=dv, q_smooth=True)
    variants["q_smooth"] = time_variant(qstep, wsq)
    del wsq

    # NVFP4 PV (and P^ in the backward): the same step, and its quantize + forward alone
    ws4 = torch.empty(sa.sage_attn_fp4_ws_bytes(B, H, N, D), dtype=torch.uint8, device=dev)
    bws4 = torch.empty(sa.sage_attn_fp4_bwd_ws_bytes(B, H, N, D), dtype=torch.uint8, device=dev)

    def f4step():
        sa.fp4_quantize(t["q"], t["k"], t["v"], w.qk_norm, w.k_smooth, ws=ws4)
        sa.fp4_forward(ws4, B, H, N, D, w.causal, w.sm_scale, o=o, lse=lse, device=dev)
        sa.fp4_backward(t["q"], t["k"], t["v"], o, lse, t["do"], ws4, w.causal, w.qk_norm, w.k_smooth, w.sm_scale,
                        bwd_ws=bws4, dq=dq, dk=dk, dv=dv)

    def f4fwd():
        sa.fp4_quantize(t["q"], t["k"], t["v"], w.qk_norm, w.k_smooth, ws=ws4)
        sa.fp4_forward(ws4, B, H, N, D, w.causal, w.sm_scale, o=o, lse=lse, device=dev)
    variants["nvfp4"] = time_variant(f4step, ws4)
    f4f = time_variant(f4fwd, ws4)
    variants["nvfp4"]["forward_ms_per_step"] = f4f["ms_per_step"]
    variants["nvfp4"]["fwd_tops"] = ops["fwd"] / (f4f["ms_per_step"] * 1e-3) / 1e12
    del ws4, bws4

    # ThriftAttention (forward only, the page's 5 % budget) against the plain forward: quantize +
    # forward, median of 20 steps each, L2 flushed
    tws = None

    def pstep():
        sa.quantize(t["q"], t["k"], t["v"], w.qk_norm, w.k_smooth, ws=ws)
        sa.forward(ws, B, H, N, D, w.causal, w.sm_scale, o=o, lse=lse, device=dev)

    def tstep():
        nonlocal tws
        _, tws = sa.thrift_quantize(t["q"], t["k"], t["v"], w.causal, 0.05, w.qk_norm, w.k_smooth, ws=ws,
                                    tws=tws)
        sa.thrift_forward(ws, tws, B, H, N, D, w.causal, w.sm_scale, o=o, lse=lse, device=dev)
    plain_fwd = time_variant(pstep, ws)
    thr = time_variant(tstep, ws)
    # its launch groups, each bracketed by events over 5 more steps
    tgroups = ("quantize", "thrift_prepare", "fwd", "thrift_hp")
    for g in tgroups:
        sa.sage_attn_timer_read(g)
    sa.sage_attn_timer_only(None)
    sa.sage_attn_timer_enable(1)
    for i in range(5):
        flush.fill_(float(i))
        tstep()
    torch.cuda.synchronize()
    sa.sage_attn_timer_enable(0)
    tms = {g: (lambda r: r[0] / max(1, r[1]))(sa.sage_attn_timer_read(g)) for g in tgroups}
    fwd_ops = ops["fwd"]
    variants["thrift_5pct_forward"] = {
        "ms_per_step": thr["ms_per_step"], "fwd_tops": fwd_ops / (thr["ms_per_step"] * 1e-3) / 1e12,
        "plain_forward_ms_per_step": plain_fwd["ms_per_step"],
        "plain_fwd_tops": fwd_ops / (plain_fwd["ms_per_step"] * 1e-3) / 1e12,
        "kernel_ms_per_step": tms,
        "note": "quantize + forward; 5 % of the visible (query block, key tile) pairs in fp16"}
    del tws

    tmax = max_over_ranks(total_ms, dist, dev)
    value = world * ops["fwd_bwd"] * K / (tmax * 1e-3) / 1e12

    # ---- end to end through the public API, host buffers, copies inside the timed region:
    # sage_attn_step_host copies the host inputs in and the results out, overlapping the
    # copies of one head range with the computation of another
    pin_out = {"o": torch.empty(o.shape, dtype=o.dtype, pin_memory=True),
               "lse": torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True),
               "dq": torch.empty(dq.shape, dtype=dq.dtype, pin_memory=True),
               "dk": torch.empty(dk.shape, dtype=dk.dtype, pin_memory=True),
               "dv": torch.empty(dv.shape, dtype=dv.dtype, pin_memory=True)}
    scratch = sa.alloc_step_host(B, H, N, D, 0, dev)
    Ke = max(3, min(K, 30))
    e2e_ms = []
    for i in range(Ke + 2):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        sa.step_host(host["q"], host["k"], host["v"], host["do"], pin_out, scratch, w.causal, w.qk_norm,
                     w.k_smooth, w.sm_scale)
        b.record(stream)
        b.synchronize()
        if i >= 2:
            e2e_ms.append(a.elapsed_time(b))
    if sa.get_status(scratch) != sa.SAGE_OK:
        raise SystemExit("device status not ok after the end-to-end steps")
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in pin_out.values())
    e2e_total = max_over_ranks(sum(e2e_ms), dist, dev)
    e2e_value = world * ops["fwd_bwd"] * Ke / (e2e_total * 1e-3) / 1e12

    # ---- roofline of the dominant kernel (backward main: the five backward matmuls)
    peaks = measured_peaks()
    fp8_peak = 2.0 * peaks["bf16"]  # nominal fp8/bf16 dense ratio 4.5/2.25
    bm_ms, bm_n = bwd_main_timed
    fw_ms, fw_n = ktimes["fwd"]
    q_ms, q_n = ktimes["quantize"]
    bp_ms, _ = ktimes["bwd_pre"]
    bd_ms, _ = ktimes["bwd_dq"]
    bm_avg = bm_ms / max(1, bm_n)
    fw_avg = fw_ms / max(1, fw_n)
    bwd_flops = ops["bwd"]
    fwd_flops = ops["fwd"]
    achieved = bwd_flops / (bm_avg * 1e-3) / 1e12
    # executed formats: S, dP, dQ, dK on bf16 tensor cores (INT8 codes in bf16), dV on fp8
    t_exec_bwd = (0.8 * bwd_flops) / (peaks["bf16"] * 1e12) + (0.2 * bwd_flops) / (fp8_peak * 1e12)
    t_exec_fwd = (0.5 * fwd_flops) / (peaks["bf16"] * 1e12) + (0.5 * fwd_flops) / (fp8_peak * 1e12)
    traffic = profiled_traffic("bwd_main", w.name, os.path.join(ROOT, "bit_trainable_attention_sagebwd_gb300",
                                                                  "csrc", "bwd.cu"))
    roof = {"kernel": "bwd_main_kernel", "bound": "tensor", "achieved": achieved, "peak": fp8_peak,
            "unit": "TFLOP/s", "frac": achieved / fp8_peak, "traffic": traffic,
            "peak_note": f"{peaks['source']} bf16 {peaks['bf16']:.1f} TF/s (burst) x 2, the nominal fp8/bf16 ratio",
            "frac_executed_formats": t_exec_bwd / (bm_avg * 1e-3),
            "flops_per_launch": bwd_flops, "avg_launch_ms": bm_avg}
    # the forward kernel's block, from the breakdown steps (every launch group bracketed)
    ff = kernel_fractions(ops, fw_avg, bm_avg, peaks)["fwd_kernel"]
    roof_fwd = {"kernel": "fwd_kernel", "bound": "tensor", "achieved": ff["achieved"], "peak": fp8_peak,
                "unit": "TFLOP/s", "frac": ff["frac"],
                "traffic": profiled_traffic("fwd", w.name, os.path.join(ROOT, "bit_trainable_attention_sagebwd_gb300",
                                                                        "csrc", "fwd.cu")),
                "peak_note": roof["peak_note"], "frac_executed_formats": ff["frac_executed_formats"],
                "flops_per_launch": fwd_flops, "avg_launch_ms": fw_avg}
    others = {}
    if not args.no_other_workloads:
        for name in wl.WORKLOADS:
            if name in (w.name, "pr1_ref"):
                continue
            others[name] = other_workload(sa, wl, name, dev, flush, peaks)
            torch.cuda.empty_cache()
    fwd_tops = fwd_flops / ((q_ms + fw_ms) / max(1, fw_n) * 1e-3) / 1e12
    bk_ms, bk_n = ktimes["bwd_main"]
    bwd_tops = bwd_flops / ((bp_ms + bk_ms + bd_ms) / max(1, bk_n) * 1e-3) / 1e12
    detail = {
        "fwd_tops": fwd_tops, "bwd_tops": bwd_tops,
        "fwd_kernel_tops": fwd_flops / (fw_avg * 1e-3) / 1e12,
        "fwd_kernel_frac_fp8_peak": fwd_flops / (fw_avg * 1e-3) / 1e12 / fp8_peak,
        "fwd_kernel_frac_executed_formats": t_exec_fwd / (fw_avg * 1e-3),
        "bwd_main_frac_fp8_peak": achieved / fp8_peak,
        "fwd_bwd_frac_fp8_peak": value / world / fp8_peak,
        "kernel_ms_per_step": {n: ms / max(1, c) for n, (ms, c) in ktimes.items()},
        "kernel_ms_note": "per launch group, from 20 untimed steps with every group bracketed by events",
        "other_workloads": others,
        "other_workloads_note": "the other full-size workloads, 20 steps each after 3 warm-up, L2 flushed, "
                                "every launch group bracketed by events (not part of value)",
        "variants": variants,
        "variants_note": "the workload's shape with fewer key/value heads (grouped-query attention) and with "
                         "Q-smoothing: quantize + forward + backward, median of 20 steps, L2 flushed",
        "wall_s": wall,
    }

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_budget)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8/e4m3 (+bf16 dP)", "data": "synthetic",
            "config": {"workload": f"{w.name}: {w.note}", "B": B, "H": H, "N": N, "D": D, "causal": w.causal,
                       "qk_norm": w.qk_norm, "k_smooth": w.k_smooth, "sm_scale": w.sm_scale,
                       "l2": "flushed between timed steps (256 MiB write, outside the events)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": roof,
            "roofline_fwd": roof_fwd,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_total / Ke,
                    "api": "sage_attn_step_host (pinned host tensors; copies of one head range overlap the "
                           "computation of another)"},
            "gpu_launches": KERNELS_PER_STEP * K,
            "clocks": clk,
            "detail": detail,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    from bit_trainable_attention_sagebwd_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload or wl.BENCH_WORKLOAD]
    if args.heads:
        import dataclasses
        w = dataclasses.replace(w, H=args.heads, note=f"{w.note}, {args.heads} heads")
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
