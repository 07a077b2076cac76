"""Benchmark: attention forward + backward BF16 TFLOP/s on one GB300.

One step = one forward (O, LSE) and one backward (dQ, dK, dV) of the
long-context causal workload (B=1, Hq=Hkv=32, S=32768, d=128) through the
library's C ABI. Inputs (268 MB per tensor) are larger than the 129 MB L2, so
no flush is needed between steps. FLOPs: forward 4*B*Hq*Sq*Sk*d, halved for
causal; backward 2.5x forward.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --fp8 [--workload W]     # FP8 (e4m3) forward only, one GPU
  python bench.py --once [--workload W] [--bwd-mode M] [--fp8]
                                           # one step, no timing (profiler captures)
  python bench.py --once --head-dim D      # the same at B=1, H=16, S=16384, causal, d=D

Prints one JSON line (rank 0). N > 1 (torchrun) runs one independent replica
per GPU (the path has no exchange step) and reports the whole-job aggregate.
``--impl reference`` times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload.
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
sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd BF16 TFLOPs/s on 1 GB300; % of dense BF16 tensor peak"
WORKLOAD = "long_s32768_causal"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), "measured"
    return 1900.0, 1700.0, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Clocks:
    """Samples nvidia-smi SM clocks and throttle reasons every 50 ms. Started
    before the warm-up (nvidia-smi needs a moment for its first sample); the
    summary keeps the samples stamped inside the timed region."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="fa_clocks_", suffix=".csv")
        os.close(fd)

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self, t0=None, t1=None):
        """Median SM clock, max clock and throttle reasons of the samples taken
        between wall-clock times t0 and t1 (all samples when not given)."""
        import datetime
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            if t0 is not None:
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                if not (t0 <= ts <= t1):
                    continue
            rows.append(parts[1:])
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": reasons, "samples": len(rows)}


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step: float, steps: int, world: int, ms: float) -> float:
    """Whole-job throughput: every rank ran `steps` steps of `flops_per_step` in `ms` (max)."""
    return flops_per_step * steps * world / (ms * 1e-3) / 1e12


def profiled_traffic(kernel_file: str, profile: str):
    """DRAM bytes per launch recorded by an ncu capture, if the kernel source
    still matches the one profiled (else None)."""
    import hashlib
    try:
        text = open(os.path.join(ROOT, "profiles", profile)).read()
        src = open(os.path.join(ROOT, "exact_attention_smem_gb300", "csrc", kernel_file), "rb").read()
    except OSError:
        return None
    tb = [l for l in text.splitlines() if l.startswith("traffic_bytes_per_launch:")]
    sh = [l for l in text.splitlines() if l.startswith("source_sha256_16:")]
    if not tb or not sh:
        return None
    if hashlib.sha256(src).hexdigest()[:16] != sh[0].split(":")[1].split()[0]:
        return None
    return int(tb[0].split(":")[1])


def roofline_peak(peak_b, peak_s, kind, clocks):
    """The roofline denominator: the burst bf16 peak when the timed region ran
    at (nearly) the maximum SM clock, as a burst GEMM does; the sustained one
    when the clock sagged under the power cap (a long, throttled run). Without
    clock samples the burst peak (the larger, more conservative) is used."""
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    if sm is not None and smax and sm < 0.95 * smax:
        return peak_s, (f"{kind} sustained bf16 (median SM clock {sm:.0f} of {smax:.0f} MHz "
                        "in the timed region)")
    clk = f"median SM clock {sm:.0f} of {smax:.0f} MHz" if sm is not None else "no clock samples"
    return peak_b, f"{kind} burst bf16 ({clk} in the timed region)"


def l2_note(w):
    """How the timed steps avoid L2 reuse between iterations (GB300 L2: 129 MB)."""
    each = w.B * w.Sq * w.Hq * w.d * 2
    return (f"inputs ({each / 1e6:.0f} MB each) exceed L2" if each > 129e6 else
            f"inputs {each / 1e6:.0f} MB each (not above L2: a profiling case, not the bench line)")


def flops(w, lengths=None):
    from attn_inputs import flops_forward
    f = flops_forward(w, lengths)
    return f, 2.5 * f


def run_ours(args):
    import torch
    import torch.distributed as dist

    import exact_attention_smem_gb300 as fa
    from attn_inputs import WORKLOADS, make_inputs

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl")
    fa.load()
    w = WORKLOADS[WORKLOAD]
    x = make_inputs(w, "cuda")
    B, Hq, Hkv, S, d = w.B, w.Hq, w.Hkv, w.Sq, w.d
    scale = w.scale
    o = torch.empty_like(x.q)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(x.q), torch.empty_like(x.k), torch.empty_like(x.v)
    nbytes = fa.fa_bwd_workspace_bytes(B, Hq, S, d, 0)
    wsbuf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    f_fwd, f_bwd = flops(w)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        # ev: [pass start, fwd end / bwd start, pass end, bwd main kernels start, stop]
        if ev is not None:
            ev[0].record(stream)
        fa.fa_fwd(x.q, x.k, x.v, o, lse, B, Hq, Hkv, S, S, d, True, scale, None, stream)
        if ev is not None:
            ev[1].record(stream)
            fa.fa_debug_set_events(1, ev[3], ev[4])
        fa.fa_bwd(x.q, x.k, x.v, o, lse, x.do, dq, dk, dv, B, Hq, Hkv, S, S, d, True, scale, None,
                  wsbuf, nbytes, stream)
        if ev is not None:
            ev[2].record(stream)

    clk = Clocks(local).__enter__()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    t0.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    clk.__exit__(None, None, None)
    if ws > 1:
        dist.barrier()
    assert fa.fa_get_device_error() == 0
    ms = t0.elapsed_time(t1)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)      # the whole backward call
    bwd_kern_ms = statistics.mean(e[3].elapsed_time(e[4]) for e in evs)  # its two main kernels
    ms = max_over_ranks(ms, device="cuda")

    # end-to-end through the public API with host buffers (pinned), copies timed
    e2e = run_e2e(fa, w, x, args, stream) if rank == 0 else None

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    peak_b, peak_s, kind = _peaks()
    per_step = (f_fwd + f_bwd)
    value = job_tflops(per_step, args.steps, ws, ms)
    bwd_tf = f_bwd / (bwd_ms * 1e-3) / 1e12
    bwd_kern_tf = f_bwd / (bwd_kern_ms * 1e-3) / 1e12
    fwd_tf = f_fwd / (fwd_ms * 1e-3) / 1e12
    clocks = clk.summary(wall0, wall1)
    peak, peak_note = roofline_peak(peak_b, peak_s, kind, clocks)
    cpu = cpu_baseline(args) if not args.no_cpu else None
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": WORKLOAD, "B": B, "Hq": Hq, "Hkv": Hkv, "S": S, "d": d,
                   "causal": True, "step": "fwd+bwd", "l2": l2_note(w),
                   "parallelism": f"replicas x{ws}"},
        "fwd_tflops": round(fwd_tf, 1), "bwd_tflops": round(bwd_tf, 1),
        "fwd_ms": round(fwd_ms, 3), "bwd_ms": round(bwd_ms, 3),
        "fwd_frac_of_peak": round(fwd_tf / peak, 4), "bwd_frac_of_peak": round(bwd_tf / peak, 4),
        "frac_of_peak": round(value / ws / peak, 4),
        "frac_of_sustained_peak": {"peak": peak_s, "step": round(value / ws / peak_s, 4),
                                   "fwd": round(fwd_tf / peak_s, 4),
                                   "bwd": round(bwd_tf / peak_s, 4)},
        "roofline": {"bound": "tensor",
                     "kernel": "backward main kernels (dkdv_kernel + dq_kernel, tcgen05)",
                     "achieved": round(bwd_kern_tf, 1),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(bwd_kern_tf / peak, 4),
                     "peak_kind": peak_note,
                     "traffic": profiled_traffic("bwd_split.cu",
                                                 f"bwd_split_kernels_{WORKLOAD}.md"),
                     "fwd": {"achieved": round(fwd_tf, 1), "frac": round(fwd_tf / peak, 4),
                             "traffic": profiled_traffic("fwd.cu",
                                                         f"fwd_kernel_{WORKLOAD}.md")}},
        "e2e": e2e,
        "gpu_launches": 4 * args.steps,        # forward, preprocess, dK/dV pass, dQ pass
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(out))
    if ws > 1:
        dist.destroy_process_group()


def run_once(args):
    """One forward and one backward (or one FP8 forward) of the workload, no
    timing and no output line: the launch sequence a profiler capture selects
    kernels from (forward, preprocess, dK/dV pass, dQ pass)."""
    import torch

    import exact_attention_smem_gb300 as fa
    from attn_inputs import WORKLOADS, make_inputs

    torch.cuda.set_device(0)
    fa.load()
    w = WORKLOADS[WORKLOAD]
    if args.head_dim is not None:
        # the head-dim shape: B=1, H=16, S=16384, causal, seeded N(0,1) bf16
        import dataclasses
        from attn_inputs import random_inputs
        w = dataclasses.replace(w, B=1, Hq=16, Hkv=16, Sq=16384, Sk=16384, d=args.head_dim,
                                causal=True, scale=args.head_dim ** -0.5)
        x = random_inputs(B=1, Hq=16, Hkv=16, Sq=16384, Sk=16384, d=args.head_dim, seed=16,
                          device="cuda")
    else:
        x = make_inputs(w, "cuda")
    if args.fp8:
        q8, qs = fa.quantize_fp8(x.q, 0)
        k8, ks = fa.quantize_fp8(x.k, 0)
        v8, vs = fa.quantize_fp8(x.v, 1)
        fa.forward_fp8(q8, qs, k8, ks, v8, vs, causal=w.causal, scale=w.scale)
    else:
        o, lse = fa.forward(x.q, x.k, x.v, causal=w.causal, scale=w.scale,
                            cu_seqlens=x.cu_seqlens)
        fa.backward(x.q, x.k, x.v, o, lse, x.do, causal=w.causal, scale=w.scale,
                    cu_seqlens=x.cu_seqlens)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0


def run_fp8(args):
    """The FP8 (e4m3) forward on one GPU: Q, K, V quantized once before the
    timed region (codes resident in HBM), then K timed forward launches."""
    import torch

    import exact_attention_smem_gb300 as fa
    from attn_inputs import WORKLOADS, make_inputs

    ws, rank, local = _dist()
    if ws > 1:
        raise SystemExit("--fp8 runs on one GPU")
    torch.cuda.set_device(local)
    fa.load()
    w = WORKLOADS[WORKLOAD]
    x = make_inputs(w, "cuda")
    B, Hq, Hkv, S, d = w.B, w.Hq, w.Hkv, w.Sq, w.d
    stream = torch.cuda.current_stream()
    fa.quantize_fp8(x.q, 0), fa.quantize_fp8(x.v, 1)       # first launches (module loading)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record(stream)
    q8, qs = fa.quantize_fp8(x.q, 0)
    k8, ks = fa.quantize_fp8(x.k, 0)
    v8, vs = fa.quantize_fp8(x.v, 1)
    ev[1].record(stream)
    torch.cuda.synchronize()
    quant_ms = ev[0].elapsed_time(ev[1])
    o = torch.empty_like(x.q)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device="cuda")

    def step():
        fa.fa_fwd_fp8(q8, k8, v8, qs, ks, vs, o, lse, B, Hq, Hkv, S, S, d, True, w.scale, stream)

    clk = Clocks(local).__enter__()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert fa.fa_get_device_error() == 0
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    clk.__exit__(None, None, None)
    assert fa.fa_get_device_error() == 0
    ms = t0.elapsed_time(t1)
    f_fwd, _ = flops(w)
    value = job_tflops(f_fwd, args.steps, 1, ms)
    peak_b, peak_s, kind = _peaks()
    clocks = clk.summary(wall0, wall1)
    peak, peak_note = roofline_peak(peak_b, peak_s, kind, clocks)
    peak8 = 2.0 * peak                       # the nominal dense fp8 : bf16 ratio
    print(json.dumps({
        "metric": "attention fwd FP8 (e4m3) TFLOPs/s on 1 GB300", "value": round(value, 2),
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate)",
        "data": "synthetic (seeded N(0,1) bf16, quantized before the timed region)",
        "config": {"workload": WORKLOAD, "B": B, "Hq": Hq, "Hkv": Hkv, "S": S, "d": d,
                   "causal": True, "step": "fwd", "l2": l2_note(w)},
        "roofline": {"bound": "tensor", "kernel": "fwd_fp8_kernel (tcgen05 kind::f8f6f4)",
                     "achieved": round(value, 1), "peak": round(peak8, 1), "unit": "TFLOP/s",
                     "frac": round(value / peak8, 4),
                     "peak_kind": f"{peak_note} x 2 (nominal fp8:bf16 ratio)",
                     "traffic": profiled_traffic("fwd_fp8.cu", f"fwd_fp8_kernel_{WORKLOAD}.md")},
        "quantize_qkv_ms": round(quant_ms, 3),
        "gpu_launches": args.steps,
        "clocks": clocks,
    }))


def run_e2e(fa, w, x, args, stream):
    """The step through the C ABI with inputs and results in pinned host memory.

    Every step copies its inputs host->device and its results (O, LSE, dQ, dK,
    dV) device->host inside the timed region. The copies run on their own
    streams and device buffers are double-buffered, so step k's input copy and
    step k-1's result copy overlap step k-1's / k's kernels (a buffer set is
    reused only after the step that last used it has finished with it). Within
    a step the forward starts once Q, K, V are in (dO follows during the
    forward) and O, LSE go out during the backward."""
    import torch
    hq, hk, hv, hdo = (t.cpu().pin_memory() for t in (x.q, x.k, x.v, x.do))
    B, Hq, Hkv, S, d = w.B, w.Hq, w.Hkv, w.Sq, w.d
    ho, hlse = torch.empty_like(hq).pin_memory(), torch.empty(B, Hq, S).pin_memory()
    hdq, hdk, hdv = (torch.empty_like(t).pin_memory() for t in (hq, hk, hv))
    nbytes = fa.fa_bwd_workspace_bytes(B, Hq, S, d, 0)
    wsbuf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    sets = []
    for _ in range(2):
        q_, k_, v_, do_ = (torch.empty_like(t) for t in (x.q, x.k, x.v, x.do))
        sets.append({"in": (q_, k_, v_, do_),
                     "out": (torch.empty_like(x.q), torch.empty(B, Hq, S, dtype=torch.float32,
                                                                 device="cuda"),
                             torch.empty_like(x.q), torch.empty_like(x.k), torch.empty_like(x.v))})
    comp, h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_qkv = [torch.cuda.Event() for _ in range(2)]     # Q, K, V of the set copied in
    ev_in = [torch.cuda.Event() for _ in range(2)]      # all inputs of the set copied in
    ev_fwd = [torch.cuda.Event() for _ in range(2)]     # forward done (O, LSE final)
    ev_used = [torch.cuda.Event() for _ in range(2)]    # kernels done with the set
    ev_out = [torch.cuda.Event() for _ in range(2)]     # results of the set copied out
    for e in ev_used + ev_out:
        e.record(comp)

    def step(i):
        st = sets[i % 2]
        q_, k_, v_, do_ = st["in"]
        o_, lse_, dq_, dk_, dv_ = st["out"]
        h2d.wait_event(ev_used[i % 2])
        with torch.cuda.stream(h2d):
            for dst, src in ((q_, hq), (k_, hk), (v_, hv)):
                dst.copy_(src, non_blocking=True)
            ev_qkv[i % 2].record(h2d)
            do_.copy_(hdo, non_blocking=True)
        ev_in[i % 2].record(h2d)
        comp.wait_event(ev_qkv[i % 2])
        comp.wait_event(ev_out[i % 2])
        fa.fa_fwd(q_, k_, v_, o_, lse_, B, Hq, Hkv, S, S, d, True, w.scale, None, comp)
        ev_fwd[i % 2].record(comp)
        comp.wait_event(ev_in[i % 2])
        fa.fa_bwd(q_, k_, v_, o_, lse_, do_, dq_, dk_, dv_, B, Hq, Hkv, S, S, d, True, w.scale,
                  None, wsbuf, nbytes, comp)
        ev_used[i % 2].record(comp)
        d2h.wait_event(ev_fwd[i % 2])
        with torch.cuda.stream(d2h):
            for dst, src in ((ho, o_), (hlse, lse_)):
                dst.copy_(src, non_blocking=True)
        d2h.wait_event(ev_used[i % 2])
        with torch.cuda.stream(d2h):
            for dst, src in ((hdq, dq_), (hdk, dk_), (hdv, dv_)):
                dst.copy_(src, non_blocking=True)
        ev_out[i % 2].record(d2h)

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(1, args.steps)
    t0.record(h2d)
    for i in range(n):
        step(i)
    t1.record(d2h)                                      # after the last result copy
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / n
    f_fwd, f_bwd = flops(w)
    h2d_b = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
    d2h_b = sum(t.numel() * t.element_size() for t in (ho, hlse, hdq, hdk, hdv))
    return {"value": round((f_fwd + f_bwd) / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 3), "h2d_bytes_per_step": h2d_b, "d2h_bytes_per_step": d2h_b,
            "steps": n, "overlap": "copies on their own streams, device buffers double-buffered; "
                                   "the forward starts once Q, K, V are in, O and LSE go out "
                                   "during the backward"}


def _oracle_sample(w, x_cpu, rows=None):
    """fp64 oracle forward + backward of query head 0 of the workload, on its
    first `rows` query rows (all when None; causal rows [0, n) see only keys
    [0, n), so that prefix is itself an exact causal problem)."""
    import oracle
    n = x_cpu.q.shape[1] if rows is None else rows
    q = x_cpu.q[0, :n, 0]
    k = x_cpu.k[0, :n, 0]
    v = x_cpu.v[0, :n, 0]
    do = x_cpu.do[0, :n, 0]
    oracle.attend_head_backward(q, k, v, do, w.scale, w.causal)   # runs the forward inside


def cpu_baseline(args, reps=1):
    """Time the oracle (as it stands) on a bounded sample: one head of the workload."""
    from attn_inputs import WORKLOADS, make_inputs
    w = WORKLOADS[WORKLOAD]
    x = make_inputs(w, "cpu")
    f_fwd, f_bwd = flops(w)
    sample_flops = (f_fwd + f_bwd) / w.Hq
    t = time.perf_counter()
    for _ in range(reps):
        _oracle_sample(w, x)
    dt = (time.perf_counter() - t) / reps
    try:
        import numpy as np
        threads = np.__config__.show  # noqa: F841  (BLAS uses all cores by default)
    except Exception:
        pass
    return {"value": round(sample_flops / dt / 1e12, 6), "unit": "TFLOP/s",
            "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"query head 0 of {WORKLOAD} (1/{w.Hq} of the step's FLOPs), fp64 numpy "
                      f"fwd+bwd, {dt:.1f} s"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    from attn_inputs import WORKLOADS, make_inputs
    w = WORKLOADS[WORKLOAD]
    x = make_inputs(w, "cpu")
    f_fwd, f_bwd = flops(w)
    # each step: the first half of head 0's query rows (a quarter of the head's
    # causal FLOPs), so that --steps 10 --warmup 3 stays near a minute of CPU time
    rows = w.Sq // 2
    sample_flops = (f_fwd + f_bwd) / w.Hq * (rows / w.Sq) ** 2
    for _ in range(args.warmup):
        _oracle_sample(w, x, rows)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        _oracle_sample(w, x, rows)
        times.append(time.perf_counter() - t)
    dt = statistics.mean(times)
    value = sample_flops / dt / 1e12
    out = {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ws,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 1),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded N(0,1) bf16, upcast to fp64)", "impl": "reference",
           "config": {"workload": WORKLOAD, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.Sq,
                      "d": w.d, "causal": True,
                      "step": "fwd+bwd of query rows [0, S/2) of head 0 per step"},
           "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
                            "kind": "oracle",
                            "sample": f"query rows [0, {rows}) of head 0 of {WORKLOAD} per step "
                                      f"(causal: {sample_flops / (f_fwd + f_bwd):.5f} of the "
                                      "workload's FLOPs), fp64 numpy fwd+bwd"},
           "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 10; 50 with --fp8, whose steps are short)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline leg")
    ap.add_argument("--fp8", action="store_true", help="time the FP8 (e4m3) forward instead")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=["long_s32768_causal", "mha_s2048_causal", "gqa_s8192_causal",
                             "varlen16_causal"],
                    help="causal workload to run (the bench line is long_s32768_causal; the "
                         "others serve profiling captures and measurements)")
    ap.add_argument("--once", action="store_true",
                    help="run one forward + backward and exit (for profiler captures)")
    ap.add_argument("--head-dim", type=int, default=None, choices=[64, 128, 192, 256],
                    help="with --once: run B=1, H=16, S=16384, causal at this head dim instead")
    ap.add_argument("--bwd-mode", type=int, default=None, choices=[0, 1, 2],
                    help="backward form (fa_debug_set bwd_mode; default: the library's)")
    args = ap.parse_args()
    if args.workload == "varlen16_causal" and not args.once:
        ap.error("the packed workload runs with --once only")
    if args.head_dim is not None and (not args.once or args.fp8):
        ap.error("--head-dim goes with --once (bf16 forward + backward)")
    if args.bwd_mode is not None:
        import exact_attention_smem_gb300 as fa
        fa.fa_debug_set("bwd_mode", args.bwd_mode)
    if args.steps is None:
        args.steps = 50 if args.fp8 else 10
    globals()["WORKLOAD"] = args.workload
    if args.impl == "reference":
        run_reference(args)
    elif args.once:
        run_once(args)
    elif args.fp8:
        run_fp8(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
