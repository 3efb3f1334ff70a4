#!/usr/bin/env python3
"""Attention-forward throughput on GB300: one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

A step is one exact attention forward (softmax(scale*QK^T)V plus nothing
else) over the self-attention workload B=1, H=16, N=4096, D=512, bf16
inputs ~ N(0,1), non-causal (FFPA README "Quick Start" layout [B,H,N,D];
D=512 is the head dimension the pages benchmark).  TFLOPS follow the
pages' convention 4*B*Hq*Nq*Nkv*D (halved when causal).

* value / ms_per_step: device time of exactly K back-to-back steps, CUDA
  events on the launching stream, bracketed by barrier + synchronize; the
  inputs (256 MiB) are larger than the 129 MB L2.
* e2e: the same metric through the public API with pinned host buffers:
  every step copies Q, K, V host->device and O device->host; consecutive
  steps overlap on three streams (copy in / forward / copy out).
* roofline: the kernel against the dense bf16 tensor peak
  (MEASURED_PEAKS.json when present, else a recorded fallback).
* cpu_baseline: the float64 oracle on a bounded, seeded sample of rows of
  the same workload, on the host cores (rank 0, N = 1 only).
* --impl reference: the oracle alone, timed per step on bounded samples.
* --pass bwd: the backward instead (one ffpa_bwd call per step: the delta,
  dQ, dV and dK kernels) on the same workload, from device-resident Q, K, V,
  O, dO and LSE; TFLOPS in the usual 2.5x-forward convention.

Multi-GPU (torchrun): independent replicas, one per rank (the path has no
exchange step); value = all ranks' flops / max over ranks of the time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn fwd TFLOPS (bf16, D=512) and % of GB300 dense BF16 peak; oracle CPU s"
METRIC_FP8 = "attn fwd TFLOPS (e4m3 FP8 forward incl. quantisation, D=512) and % of GB300 dense FP8 peak"
FALLBACK_BF16_TFLOPS = 1900.0      # profiling recipe fallback (one earlier GB300 measurement)
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1000 * 1000


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="selfattn_b1_h16_n4096_d512")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--precision", choices=("bf16", "fp8"), default="bf16",
                    help="bf16 (default): the 16-bit forward; fp8: the e4m3 forward "
                         "(quantisation + attention, ffpa_fwd_fp8) on the same bf16 inputs")
    ap.add_argument("--pass", dest="which", choices=("fwd", "bwd"), default="fwd",
                    help="forward (default) or backward step")
    return ap.parse_args(argv)


def workload_by_name(name):
    from exact_headdim_attention_gb300 import workloads as wl
    for w in wl.all_workloads():
        if w.name == name:
            return w
    raise SystemExit(f"unknown workload {name}")


def config_of(w, flops):
    cfg = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Nq": w.Nq, "Nkv": w.Nkv,
           "D": w.D, "causal": w.causal, "mask": "additive f32" if w.additive_mask else None,
           "varlen": w.varlen, "flops_per_step": flops,
           "l2": "inputs larger than L2 (no flush between steps)"}
    return cfg


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            bf16 = d.get("bf16_tflops") or d.get("bf16_tflops_burst")
            sus = d.get("bf16_tflops_sustained")
            if bf16:
                return (float(bf16), "measured (MEASURED_PEAKS.json bf16_tflops, burst)",
                        float(sus) if sus else None)
        except (OSError, ValueError):
            pass
    return FALLBACK_BF16_TFLOPS, "fallback (profiling recipe: 1.9 PFLOP/s bf16 burst)", None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (every 100 ms) with host timestamps."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", self.gpu_id], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.monotonic(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        win = [p for t, p in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        if not win and self.samples:     # very short timed region: nearest sample
            mid = 0.5 * (t0 + t1)
            win = [min(self.samples, key=lambda s: abs(s[0] - mid))[1]]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in win if num(p[1]) is not None]
        mx = [num(p[2]) for p in win if num(p[2]) is not None]
        pw = [num(p[3]) for p in win if num(p[3]) is not None]
        reasons = sorted({name for p in win for name, val in zip(self.NAMES, p[5:9])
                          if val.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_median": statistics.median(pw) if pw else None,
                "reasons": reasons, "samples": len(win)}


def gpu_id_for(device_index: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(device_index)


# --------------------------------------------------------------- our arm
def make_step(w, x, dev, fp8=False):
    """Returns (device_step, e2e_step, e2e_start, e2e_finish, bytes_h2d, bytes_d2h, flops).

    device_step: one forward on device-resident inputs (torch's current stream).
    e2e_step: one end-to-end step through the public API: H2D copy of Q, K, V
    from pinned host memory, the forward, D2H copy of O into pinned host
    memory.  Consecutive steps are pipelined over three streams (copy in,
    compute, copy out) and two sets of device buffers, so step i's copies
    overlap step i-1's kernel; every step still moves all of its bytes.
    e2e_start / e2e_finish: make the pipeline's streams wait for torch's
    current stream / the current stream wait for all issued steps."""
    import torch
    import exact_headdim_attention_gb300 as pkg
    from exact_headdim_attention_gb300 import workloads as wl

    names = ("q", "k", "v")
    host = {n: x[n].pin_memory() for n in names}
    devt = {n: host[n].to(dev, non_blocking=False) for n in names}
    mask = None if w.varlen or x.get("mask") is None else x["mask"].to(dev)
    cq = x["cu_q"].to(dev) if w.varlen else None
    flops = wl.useful_flops(w, x["seqlens"]) if w.varlen else wl.useful_flops(w)

    ws = [None, None]
    if fp8:
        if w.varlen:
            raise SystemExit("--precision fp8 takes a dense workload")
        nbytes = pkg.fp8_workspace_bytes(w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.D)
        ws = [torch.empty(nbytes, dtype=torch.uint8, device=dev) for _ in range(2)]

    def forward(ins, out, lse, stream=None):
        if fp8:
            pkg.ffpa_fwd_fp8(ins["q"], ins["k"], ins["v"], attn_mask=mask, is_causal=w.causal,
                             enable_gqa=w.enable_gqa, out=out, stream=stream,
                             workspace=ws[0] if out is outs_ref[0] else ws[1])
        elif w.varlen:
            pkg.ffpa_fwd_varlen(ins["q"], ins["k"], ins["v"], cq, None, x["max_q"], x["max_k"],
                                causal=w.causal, enable_gqa=w.enable_gqa, return_lse=True,
                                out=out, lse=lse, stream=stream)
        else:
            pkg.ffpa_fwd(ins["q"], ins["k"], ins["v"], attn_mask=mask, is_causal=w.causal,
                         enable_gqa=w.enable_gqa, out=out, stream=stream)

    def new_lse():
        return (torch.empty(w.Hq, x["q"].shape[0], dtype=torch.float32, device=dev)
                if w.varlen else None)

    out = torch.empty_like(devt["q"])
    lse = new_lse()
    outs_ref = [out]

    def call():
        forward(devt, out, lse)

    # end to end: two buffer sets, three streams
    s_in, s_c, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ins = [devt, {n: torch.empty_like(devt[n]) for n in names}]
    outs = [out, torch.empty_like(out)]
    lses = [lse, new_lse()]
    o_host = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]      # inputs of buffer b landed
    ev_c = [torch.cuda.Event() for _ in range(2)]       # forward on buffer b done
    ev_out = [torch.cuda.Event() for _ in range(2)]     # O of buffer b copied out
    state = {"i": 0}

    def e2e():
        b = state["i"] & 1
        if state["i"] >= 2:
            s_in.wait_event(ev_c[b])          # the forward of step i-2 has read buffer b
        with torch.cuda.stream(s_in):
            for n in names:
                ins[b][n].copy_(host[n], non_blocking=True)
        ev_in[b].record(s_in)
        s_c.wait_event(ev_in[b])
        if state["i"] >= 2:
            s_c.wait_event(ev_out[b])         # O of step i-2 has left buffer b
        forward(ins[b], outs[b], lses[b], stream=s_c)
        ev_c[b].record(s_c)
        s_out.wait_event(ev_c[b])
        with torch.cuda.stream(s_out):
            o_host[b].copy_(outs[b], non_blocking=True)
        ev_out[b].record(s_out)
        state["i"] += 1

    def e2e_finish():
        cur = torch.cuda.current_stream(dev)
        for st in (s_in, s_c, s_out):
            cur.wait_stream(st)

    def e2e_start():
        cur = torch.cuda.current_stream(dev)
        for st in (s_in, s_c, s_out):
            st.wait_stream(cur)

    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = o_host[0].numel() * o_host[0].element_size()
    return call, e2e, e2e_start, e2e_finish, h2d, d2h, flops


def time_steps(fn, steps, dist_on, finish=None, start=None):
    """Device time of `steps` calls of fn: CUDA events on torch's current
    stream, bracketed by a barrier and a synchronize.  When fn issues work on
    other streams, `start` makes them wait for the start event and `finish`
    makes the current stream wait for them before the end event."""
    import torch
    import torch.distributed as dist
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    if dist_on:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.monotonic()
    s.record()
    if start is not None:
        start()
    for _ in range(steps):
        fn()
    if finish is not None:
        finish()
    e.record()
    torch.cuda.synchronize()
    t1 = time.monotonic()
    if dist_on:
        dist.barrier()
    return s.elapsed_time(e) / 1e3, t0, t1


def aggregate(elapsed_s: float, flops_per_step: float, steps: int, world: int, dist_on: bool,
              device=None):
    """Whole-job throughput: all ranks' flops / max over ranks of the time."""
    import torch
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    if dist_on:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    tmax = float(t.item())
    total = flops_per_step * steps * world
    return total / tmax / 1e12, tmax


def cpu_model() -> str:
    """Host CPU model (lscpu's "Model name", else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def oracle_tiny_one_core():
    """Seconds of the float64 oracle on the tiny B1 H1 N128 D320 case on one thread."""
    import oracle
    from exact_headdim_attention_gb300 import workloads as wl
    x = wl.materialize(wl.tiny_d320())
    orc = oracle.default()
    orc.attn_dense(x["q"], x["k"], x["v"], nthreads=1)
    t0 = time.perf_counter()
    orc.attn_dense(x["q"], x["k"], x["v"], nthreads=1)
    return time.perf_counter() - t0


def cpu_baseline(w, x, target_s: float, fp8: bool = False):
    """The float64 oracle (its FP8 reference with fp8) on a bounded seeded
    sample of rows of the workload."""
    import torch
    import oracle
    cores = oracle.host_threads()
    orc = oracle.default()
    attn = orc.attn_fp8 if fp8 else orc.attn_dense
    if w.varlen:
        raise SystemExit("cpu baseline for varlen workloads: use the dense workloads")
    per_row = 4.0 * w.Nkv * w.D / (2.0 if w.causal else 1.0)
    total_rows = w.B * w.Hq * w.Nq
    g = torch.Generator().manual_seed(w.seed + 17)

    def timed(n):
        rows = torch.randint(0, total_rows, (n,), generator=g)
        t0 = time.perf_counter()
        attn(x["q"], x["k"], x["v"], attn_mask=x.get("mask"), is_causal=w.causal, rows=rows,
             nthreads=cores)
        return max(time.perf_counter() - t0, 1e-6)

    # two calibration sizes separate the per-call cost (the FP8 reference quantises
    # all of Q, K and V first) from the per-row cost
    timed(cores)                                  # first call: library and thread start-up
    n1, n2 = cores, 4 * cores
    t1, t2 = timed(n1), timed(n2)
    per_row_s = max((t2 - t1) / (n2 - n1), 1e-9)
    fixed_s = max(t1 - n1 * per_row_s, 0.0)
    n = int(min(total_rows, max(cores, max(target_s - fixed_s, 0.5 * target_s) / per_row_s)))
    n = max(cores, (n // cores) * cores)
    dt = timed(n)
    flops = per_row * n
    full_s = fixed_s + (dt - fixed_s) * total_rows / n
    return {"value": flops / dt / 1e12, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
            "sample": f"{n} seeded random query rows of {total_rows} (all {w.Nkv} keys each), "
                      f"{dt:.1f} s; full workload would take ~{full_s:.0f} s",
            "seconds": dt, "rows": n, "full_workload_s": round(full_s, 1),
            "cpu_model": cpu_model(),
            "tiny_d320_one_core_s": round(oracle_tiny_one_core(), 4)}


def run_ours(args):
    import torch
    import torch.distributed as dist
    import exact_headdim_attention_gb300 as pkg
    from exact_headdim_attention_gb300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist_on = world > 1
    if dist_on:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkg.load_library()
    w = workload_by_name(args.workload)
    x = wl.materialize(w)
    fp8 = args.precision == "fp8"
    step, e2e, e2e_start, e2e_finish, h2d, d2h, flops = make_step(w, x, dev, fp8=fp8)
    assert args.warmup >= 3, "at least 3 warm-up steps"
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = pkg.ffpa_last_device_error()
    if st != pkg.FFPA_OK:
        raise SystemExit(f"device error during warm-up: {pkg.ffpa_status_string(st)}")
    sampler = ClockSampler(gpu_id_for(local))
    sampler.start()
    elapsed, t0, t1 = time_steps(step, args.steps, dist_on)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    value, tmax = aggregate(elapsed, flops, args.steps, world, dist_on, dev)
    # end to end through the public API with host buffers
    for _ in range(3):
        e2e()
    e2e_finish()
    n_e2e = max(3, min(args.e2e_steps, args.steps))
    e_el, _, _ = time_steps(e2e, n_e2e, dist_on, finish=e2e_finish, start=e2e_start)
    e_value, _ = aggregate(e_el, flops, n_e2e, world, dist_on, dev)
    st = pkg.ffpa_last_device_error()
    if st != pkg.FFPA_OK:
        raise SystemExit(f"device error: {pkg.ffpa_status_string(st)}")
    peak, peak_src, peak_sustained = read_peaks()
    if fp8:
        # e4m3 contraction: the bf16 figure times the nominal dense ratio (4.5 / 2.25 PFLOP/s)
        peak, peak_src = 2.0 * peak, peak_src + " x 2 (nominal e4m3 / bf16 dense ratio)"
        peak_sustained = 2.0 * peak_sustained if peak_sustained else None
    kname = "fp8" if fp8 else pkg.selected_kernel(w.D, w.varlen)
    if kname == "dual" and x.get("mask") is not None:
        kname = "single"   # the dual-tile kernel takes no mask
    vl, um = str(w.varlen).lower(), str(x.get("mask") is not None).lower()
    fp8_attn = ("ffpa_fwd_fp8_split_kernel" if w.D in (384, 512) else "ffpa_fwd_fp8_kernel")
    kernel = {"fp8": f"ffpa_fp8_quant_kernel + {fp8_attn}<{w.D // 128}, {um}>",
              "single": f"ffpa_fwd_kernel<{vl}, {um}>",
              "dual": f"ffpa_fwd_dual_kernel<{w.D // 64}>",
              "pair": f"ffpa_fwd_pair_kernel<{vl}, {w.D // 64}, {um}>",
              "split": (f"ffpa_fwd_split_kernel<{vl}, {w.D // 64}, {um}>" if w.D <= 512 else
                        f"ffpa_fwd_cluster_kernel<{vl}, {w.D // 64}, {um}, {w.D // 256}>")}[kname]
    per_launch_s = elapsed / args.steps
    achieved = flops / per_launch_s / 1e12
    line = {
        "metric": METRIC_FP8 if fp8 else METRIC, "value": round(value, 2), "unit": "TFLOPS",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tmax / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 (bf16 in and out)" if fp8 else "bf16",
        "data": "synthetic (seeded N(0,1) bf16, shapes of the pages' workloads)",
        "config": config_of(w, flops),
        "pct_of_peak": round(100.0 * achieved / peak, 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
                     "peak_source": peak_src, "kernel": kernel,
                     "frac_of_sustained": (round(achieved / peak_sustained, 4)
                                           if peak_sustained else None),
                     "algorithmic_flops_per_launch": flops},
        "e2e": {"value": round(e_value, 2), "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": n_e2e,
                "api": ("exact_headdim_attention_gb300.ffpa_fwd_fp8 (C ABI ffpa_fwd_fp8)" if fp8
                        else "exact_headdim_attention_gb300.ffpa_fwd (C ABI ffpa_fwd)"),
                "pipelining": "copy-in, forward and copy-out of consecutive steps on three "
                              "streams with two buffer sets"},
        "gpu_launches": (2 if fp8 else 1) * args.steps,
        "clocks": clocks,
        "impl": "ours",
    }
    if fp8:
        line["roofline"]["note"] = ("one step = two launches (quantisation, then attention); "
                                    "achieved = the step's useful flops over the step time")
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not w.varlen:
        line["cpu_baseline"] = cpu_baseline(w, x, args.cpu_seconds, fp8=fp8)
        line["oracle_cpu_s_full_workload_est"] = line["cpu_baseline"]["full_workload_s"]
    traffic = measured_traffic(w.name, key="fp8_dram_bytes_per_launch" if fp8 else "dram_bytes_per_launch")
    if traffic is not None:
        line["roofline"]["traffic"] = traffic
        if fp8:
            line["roofline"]["traffic_note"] = ("ncu DRAM bytes of the attention launch; the quantisation "
                                                "launch reads Q, K, V and writes their e4m3 codes")
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist_on:
        dist.destroy_process_group()


METRIC_BWD = "attn bwd TFLOPS (bf16, D=512; 2.5x forward flops) and % of GB300 dense BF16 peak"


def cpu_baseline_bwd(w, x, dout, target_s: float):
    """The float64 oracle's backward on a bounded seeded sample of dQ rows (each
    needs its row's softmax, dP and the dQ sum over all keys: 6*Nkv*D useful
    flops of the backward's 10*Nkv*D per query row)."""
    import torch
    import oracle
    cores = oracle.host_threads()
    orc = oracle.default()
    per_row = 6.0 * w.Nkv * w.D / (2.0 if w.causal else 1.0)
    total_rows = w.B * w.Hq * w.Nq
    g = torch.Generator().manual_seed(w.seed + 23)
    n = cores
    orc.attn_bwd_rows(x["q"], x["k"], x["v"], dout, [0], [], is_causal=w.causal, nthreads=cores)
    t0 = time.perf_counter()
    orc.attn_bwd_rows(x["q"], x["k"], x["v"], dout, torch.randint(0, total_rows, (n,), generator=g), [],
                      is_causal=w.causal, nthreads=cores)
    dt = max(time.perf_counter() - t0, 1e-6)
    n = int(min(total_rows, max(cores, n * target_s / dt)))
    n = max(cores, (n // cores) * cores)
    t0 = time.perf_counter()
    orc.attn_bwd_rows(x["q"], x["k"], x["v"], dout, torch.randint(0, total_rows, (n,), generator=g), [],
                      is_causal=w.causal, nthreads=cores)
    dt = time.perf_counter() - t0
    return {"value": per_row * n / dt / 1e12, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
            "sample": f"dQ of {n} seeded random query rows of {total_rows} (softmax, dP and dQ over "
                      f"all {w.Nkv} keys each), {dt:.1f} s", "seconds": dt, "rows": n,
            "cpu_model": cpu_model()}


def run_ours_bwd(args):
    """One backward per step; same timing, e2e and clock rules as the forward."""
    import torch
    import exact_headdim_attention_gb300 as pkg
    from exact_headdim_attention_gb300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world != 1:
        raise SystemExit("--pass bwd runs on one GPU")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pkg.load_library()
    w = workload_by_name(args.workload)
    if w.varlen or w.additive_mask:
        raise SystemExit("--pass bwd takes a dense workload without a mask")
    x = wl.materialize(w)
    g = torch.Generator().manual_seed(w.seed + 101)
    dout = torch.randn(x["q"].shape, generator=g).to(x["q"].dtype)
    names = ("q", "k", "v")
    host = {n: x[n].pin_memory() for n in names}
    host["dout"] = dout.pin_memory()
    devt = {n: host[n].to(dev) for n in host}
    o, lse = pkg.ffpa_fwd(devt["q"], devt["k"], devt["v"], is_causal=w.causal,
                          enable_gqa=w.enable_gqa, return_lse=True)
    host["o"] = o.cpu().pin_memory()
    host["lse"] = lse.cpu().pin_memory()
    devt["o"], devt["lse"] = o, lse
    flops = 2.5 * wl.useful_flops(w)

    def grads_like(t):
        return {"dq": torch.empty_like(t["q"]), "dk": torch.empty_like(t["k"]),
                "dv": torch.empty_like(t["v"]),
                "delta": torch.empty(t["lse"].shape, dtype=torch.float32, device=dev)}

    # The stored-tile workspace (P and dS of every visible tile), allocated
    # once: the timed steps and the end-to-end steps run on one stream at a
    # time, so they share it.
    B, Hq, Nq, D = x["q"].shape
    ws_bytes = pkg.bwd_workspace_bytes(B, Hq, x["k"].shape[1], Nq, x["k"].shape[2], D, w.causal)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None

    def backward(t, gr, stream=None):
        pkg.ffpa_bwd(t["dout"], t["q"], t["k"], t["v"], t["o"], t["lse"], is_causal=w.causal,
                     enable_gqa=w.enable_gqa, dq=gr["dq"], dk=gr["dk"], dv=gr["dv"],
                     delta=gr["delta"], workspace=ws, stream=stream)

    gr0 = grads_like(devt)

    def step():
        backward(devt, gr0)

    # end to end: inputs in, three gradients out; two buffer sets, three streams
    s_in, s_c, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ins = [devt, {n: torch.empty_like(devt[n]) for n in devt}]
    grs = [gr0, grads_like(devt)]
    out_host = [{n: torch.empty(grs[0][n].shape, dtype=grs[0][n].dtype, pin_memory=True)
                 for n in ("dq", "dk", "dv")} for _ in range(2)]
    ev_in, ev_c, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    state = {"i": 0}

    def e2e():
        b = state["i"] & 1
        if state["i"] >= 2:
            s_in.wait_event(ev_c[b])
        with torch.cuda.stream(s_in):
            for n in host:
                ins[b][n].copy_(host[n], non_blocking=True)
        ev_in[b].record(s_in)
        s_c.wait_event(ev_in[b])
        if state["i"] >= 2:
            s_c.wait_event(ev_out[b])
        backward(ins[b], grs[b], stream=s_c)
        ev_c[b].record(s_c)
        s_out.wait_event(ev_c[b])
        with torch.cuda.stream(s_out):
            for n in out_host[b]:
                out_host[b][n].copy_(grs[b][n], non_blocking=True)
        ev_out[b].record(s_out)
        state["i"] += 1

    def e2e_finish():
        cur = torch.cuda.current_stream(dev)
        for st in (s_in, s_c, s_out):
            cur.wait_stream(st)

    def e2e_start():
        cur = torch.cuda.current_stream(dev)
        for st in (s_in, s_c, s_out):
            st.wait_stream(cur)

    h2d = sum(host[n].numel() * host[n].element_size() for n in host)
    d2h = sum(t.numel() * t.element_size() for t in out_host[0].values())
    assert args.warmup >= 3, "at least 3 warm-up steps"
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = pkg.ffpa_last_device_error()
    if st != pkg.FFPA_OK:
        raise SystemExit(f"device error during warm-up: {pkg.ffpa_status_string(st)}")
    sampler = ClockSampler(gpu_id_for(0))
    sampler.start()
    elapsed, t0, t1 = time_steps(step, args.steps, False)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    value, tmax = aggregate(elapsed, flops, args.steps, 1, False, dev)
    for _ in range(3):
        e2e()
    e2e_finish()
    n_e2e = max(3, min(args.e2e_steps, args.steps))
    e_el, _, _ = time_steps(e2e, n_e2e, False, finish=e2e_finish, start=e2e_start)
    e_value, _ = aggregate(e_el, flops, n_e2e, 1, False, dev)
    st = pkg.ffpa_last_device_error()
    if st != pkg.FFPA_OK:
        raise SystemExit(f"device error: {pkg.ffpa_status_string(st)}")
    peak, peak_src, peak_sustained = read_peaks()
    achieved = value
    cfg = config_of(w, flops)
    cfg["pass"] = ("backward (delta, scores and contraction kernels; P and dS stored once per tile)"
                   if ws is not None else "backward (delta + dQ + dV + dK slice kernels)")
    cfg["bwd_workspace_bytes"] = ws_bytes
    line = {
        "metric": METRIC_BWD, "value": round(value, 2), "unit": "TFLOPS", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tmax / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q, K, V, dO; O and LSE from the forward)",
        "config": cfg,
        "pct_of_peak": round(100.0 * achieved / peak, 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
                     "peak_source": peak_src,
                     "kernel": (f"ffpa_bwd step: ffpa_bwd_delta_kernel + ffpa_bwd_scores_kernel<{D // 64}, false> "
                                f"+ ffpa_bwd_contract_kernel<{D // 64}>, one C call" if ws is not None else
                                "ffpa_bwd step: ffpa_bwd_delta_kernel + ffpa_bwd_kernel<0, false> (dQ) + "
                                "ffpa_bwd_kernel<1, false> (dV) + ffpa_bwd_kernel<2, false> (dK), one C call"),
                     "frac_of_sustained": (round(achieved / peak_sustained, 4)
                                           if peak_sustained else None),
                     "algorithmic_flops_per_launch": flops},
        "e2e": {"value": round(e_value, 2), "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": n_e2e,
                "api": "exact_headdim_attention_gb300.ffpa_bwd (C ABI ffpa_bwd_ws_ex)",
                "pipelining": "copy-in, backward and copy-out of consecutive steps on three "
                              "streams with two buffer sets"},
        "gpu_launches": (3 if ws is not None else 4) * args.steps,
        "clocks": clocks,
        "impl": "ours",
    }
    tb = measured_traffic_bwd(w.name) if ws is not None else None
    if tb is not None:
        line["roofline"]["traffic"] = tb["gradient_kernels_total"]
        line["roofline"]["traffic_note"] = ("ncu DRAM bytes of the scores and contraction launches of one "
                                            "step (delta kernel not captured)")
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_bwd(w, x, dout, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def strip_comments(src: str) -> str:
    """C/C++ source with comments removed and whitespace runs collapsed (string
    literals in these files hold no comment markers)."""
    import re
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


# The sources each recorded capture depends on: the kernel's own file, the
# shared device code and the host planner that sets its launch shape.
TRAFFIC_SOURCES = {
    "dram_bytes_per_launch": ("ffpa_split.cu", "ffpa_common.cuh", "ptx.cuh", "ffpa_api.cu"),
    "fp8_dram_bytes_per_launch": ("ffpa_fp8_split.cu", "ffpa_fp8.cu", "ffpa_common.cuh", "ptx.cuh",
                                  "ffpa_api.cu"),
    "bwd_dram_bytes_per_step": ("ffpa_bwd.cu", "ffpa_bwd_tiles.cu", "ffpa_bwd_common.cuh", "ffpa_common.cuh",
                                "ptx.cuh", "ffpa_api.cu"),
}


def kernel_source_sha(files=None) -> str:
    """Hash of kernel sources' code (comments and layout excluded), so that a
    recorded ncu capture stays attached to the code it measured.  files: the
    csrc file names to hash (all of them when None)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_headdim_attention_gb300", "csrc")
    for fn in sorted(files if files is not None else os.listdir(csrc)):
        with open(os.path.join(csrc, fn), encoding="utf-8") as f:
            h.update(fn.encode() + b"\0" + strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")


def _traffic_section(key, path):
    """Section `key` of the committed ncu summary (profiles/traffic.json), or None
    when it was captured on different code than the current sources."""
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    sec = d.get(key)
    if not isinstance(sec, dict) or sec.get("kernel_source_sha") != kernel_source_sha(TRAFFIC_SOURCES[key]):
        return None
    return sec


def measured_traffic_bwd(name, path=TRAFFIC_PATH):
    """DRAM bytes of one stored-tile backward step's scores and contraction launches
    from the committed ncu summary, or None when that capture was taken on
    different kernel code."""
    sec = _traffic_section("bwd_dram_bytes_per_step", path)
    return None if sec is None else sec.get(name)


def measured_traffic(name, path=TRAFFIC_PATH, key="dram_bytes_per_launch"):
    """DRAM bytes per launch from the committed ncu summary (profiles/traffic.json),
    or None when that capture was taken on a different kernel source.  key
    "fp8_dram_bytes_per_launch" holds the FP8 attention kernel's bytes."""
    sec = _traffic_section(key, path)
    return None if sec is None else sec.get(name)


# ---------------------------------------------------------- reference arm
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import torch
    import oracle
    from exact_headdim_attention_gb300 import workloads as wl
    w = workload_by_name(args.workload)
    x = wl.materialize(w)
    flops_full = wl.useful_flops(w)
    cores = oracle.host_threads()
    orc = oracle.default()
    per_row = 4.0 * w.Nkv * w.D / (2.0 if w.causal else 1.0)
    total_rows = w.B * w.Hq * w.Nq
    g = torch.Generator().manual_seed(w.seed + 29)
    # size each step so that warm-up + steps take about 90 s (the first call, which
    # loads the library and starts its threads, stays out of the probe)
    orc.attn_dense(x["q"], x["k"], x["v"], attn_mask=x.get("mask"), is_causal=w.causal,
                   rows=torch.zeros(1, dtype=torch.int64), nthreads=cores)
    probe = torch.randint(0, total_rows, (cores,), generator=g)
    t0 = time.perf_counter()
    orc.attn_dense(x["q"], x["k"], x["v"], attn_mask=x.get("mask"), is_causal=w.causal, rows=probe,
                   nthreads=cores)
    t_probe = max(time.perf_counter() - t0, 1e-6)
    per_step = 90.0 / (args.steps + args.warmup)
    n = max(cores, int(cores * per_step / t_probe) // cores * cores)
    for _ in range(args.warmup):
        orc.attn_dense(x["q"], x["k"], x["v"], attn_mask=x.get("mask"), is_causal=w.causal,
                       rows=torch.randint(0, total_rows, (n,), generator=g), nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.attn_dense(x["q"], x["k"], x["v"], attn_mask=x.get("mask"), is_causal=w.causal,
                       rows=torch.randint(0, total_rows, (n,), generator=g), nthreads=cores)
    dt = time.perf_counter() - t0
    value = per_row * n * args.steps / dt / 1e12
    sample = (f"each step: {n} seeded random query rows of {total_rows} (all keys), "
              f"float64 oracle on {cores} host threads")
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 inputs widened to float64)",
        "config": config_of(w, flops_full), "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    elif args.which == "bwd":
        run_ours_bwd(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
