#!/usr/bin/env python
"""Fused transformer MLP fwd+bwd throughput on GB300 (bf16 in, fp32 accumulate).

One step = one training forward (mlp_fwd) plus one backward (mlp_bwd from
saved preacts, or mlp_bwd_recompute) of the selected workload, on seeded
synthetic inputs already resident in HBM.  The L2 cache is flushed (a
512 MiB write) before every timed step, outside the step's events.  The
default workload is the largest, the Llama-3-8B-shaped MLP (8192 tokens,
4096 x 14336, backward recomputing the preacts), with its no-grad inference
forward beside it; the other four workloads (and, for the ReLU^2 one, the
FP8 step and the block with its neighbours) are measured for the breakdown
with a few steps each, and the inference forward of 1 to 512 tokens with the
same weights (decode sizes), unless --headline-only is given.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--headline-only]
    python bench.py --impl reference ...   # the fp64 CPU oracle, timed on the host cores

Prints one JSON line.  Under torchrun (N > 1) every rank runs an independent
replica of the workload (the MLP path has no collective of its own); the
step time is the maximum over ranks and `value` sums all ranks' work.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLP fwd+bwd TFLOP/s (bf16) and % of GB300 dense-BF16 peak, 1 GPU"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama3_8b_swiglu")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the other workloads' breakdown")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-trace", action="store_true")
    ap.add_argument("--fp8", action="store_true",
                    help="also time the FP8 forward and training step (ReLU^2 workloads)")
    ap.add_argument("--block", action="store_true",
                    help="also time the MLP block with its fused RMS norm and residual add")
    ap.add_argument("--sweep-m", action="store_true",
                    help="time the inference forward at decode-sized token counts even with "
                         "--headline-only (the default run includes it)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the workload's token count M (small cases for profiling)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def mode_of(w):
    return "bwd_recompute" if w.recompute else "bwd"


def flops_of(w, mode):
    """GEMM flops (2 x multiply-adds) of one pass; gated: fwd 6MHI, bwd 12MHI,
    recompute +4MHI; non-gated: 4, 8, +2."""
    mhi = float(w.M) * w.H * w.I
    g = w.gated
    if mode in ("fwd", "infer"):
        return (6 if g else 4) * mhi
    if mode == "bwd":
        return (12 if g else 8) * mhi
    if mode == "bwd_recompute":
        return (16 if g else 10) * mhi
    raise ValueError(mode)


def kernel_flops(w):
    """Algorithmic flops per launch of each kernel of a step."""
    mhi = float(w.M) * w.H * w.I
    g = w.gated
    return {
        "gate_up_act": (4 if g else 2) * mhi,
        "down_proj": 2 * mhi,
        "dgated": 2 * mhi,
        "dx": (4 if g else 2) * mhi,
        "wgrad": (6 if g else 4) * mhi,
        "dact_recompute": 4 * mhi,  # non-gated recompute: x W1^T and dout Wd
        "fwd_fused": (6 if g else 4) * mhi,  # gated forward: gate/up and down in one launch
    }


def code_text(src):
    """Source text without its comments and with whitespace runs collapsed,
    so that comment and layout edits leave the hash alone.  (The sources
    hold no string literal with a comment marker in it.)"""
    import re
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def csrc_hash(d=None):
    """Hash of the device code (kernel sources and the headers they include,
    comments aside; the host-side launch code in mlp_api.cu and
    mlp_noalloc.cu does not change what a kernel moves)."""
    h = hashlib.sha256()
    d = d or os.path.join(ROOT, "activated_mlp_gemms_gb300", "csrc")
    for n in sorted(os.listdir(d)):
        if n in ("mlp_api.cu", "mlp_noalloc.cu") or not n.endswith((".cu", ".cuh", ".h")):
            continue
        with open(os.path.join(d, n), encoding="utf-8") as f:
            h.update(n.encode())
            h.update(code_text(f.read()).encode())
    return h.hexdigest()[:16]


def load_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if taken on the
    current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(workload, {}).get(kernel)
        if e and e.get("csrc_hash") == csrc_hash():
            return e.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


class ClockSampler:
    """Samples SM clocks and throttle reasons during a timed region.

    One `nvidia-smi --query-gpu=timestamp,... -lms 20` process takes a sample
    every 20 ms from before the region starts until just after it ends, when
    it is stopped with SIGINT (nvidia-smi then exits normally).  Samples are
    attributed to the region by their own timestamps, so output buffering
    does not matter; the ones inside the region and the first one after it
    are kept.  If the loop yields nothing, one single query is taken."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 20

    def __init__(self, index, exe="nvidia-smi"):
        self.index = index
        self.exe = exe
        self.lines = []  # (sample time, fields) as read
        self.samples = []
        self._proc = None
        self._t = None
        self._first = threading.Event()
        self.t0 = self.t1 = None

    @staticmethod
    def _stamp(s):
        import datetime
        try:
            return datetime.datetime.strptime(s.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def _reader(self):
        for line in self._proc.stdout:
            f = [x.strip() for x in line.strip().split(",")]
            if len(f) >= 9:
                t = self._stamp(f[0])
                if t is not None:
                    self.lines.append((t, f[1:]))
                    self._first.set()

    def _single(self):
        try:
            r = subprocess.run([self.exe, "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                "--format=csv,noheader,nounits"], capture_output=True, text=True,
                               timeout=10)
            if r.returncode == 0 and r.stdout.strip():
                return [x.strip() for x in r.stdout.strip().splitlines()[0].split(",")]
        except (OSError, subprocess.SubprocessError):
            pass
        return None

    def __enter__(self):
        try:
            self._proc = subprocess.Popen(
                [self.exe, "-i", str(self.index), "--query-gpu=timestamp," + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._reader, daemon=True)
            self._t.start()
            self._first.wait(1.0)  # start once samples flow (or after 1 s if output is buffered)
        except OSError:
            self._proc = None
        self.t0 = time.time()
        return self

    def __exit__(self, *a):
        import signal
        self.t1 = time.time()
        if self._proc is not None:
            time.sleep(3 * self.PERIOD_MS / 1000.0)  # let one sample past the region be taken
            self._proc.send_signal(signal.SIGINT)
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
                self._proc.wait(timeout=5)
            self._t.join(timeout=5)
        inside = [f for t, f in self.lines if self.t0 <= t <= self.t1]
        after = [f for t, f in sorted(self.lines, key=lambda x: x[0]) if t > self.t1][:1]
        self.samples = inside + after
        if not self.samples:
            one = self._single()
            if one:
                self.samples = [one]

    def summary(self):
        if not self.samples:
            return None
        sm, mx = [], []
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in self.samples:
            try:
                sm.append(float(s[0]))
                mx.append(float(s[1]))
            except ValueError:
                continue
            for n, v in zip(names, s[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------- ours

def kernel_bytes(w):
    """Algorithmic DRAM bytes per launch of each kernel of a step (bf16
    tensors read or written once; the fused forward reads its postact back
    from L2), and of each kernel's epilogue alone (the [M,I] intermediates
    it reads and writes, and the [M,H] outputs of the down projection and
    dx).  Returns {kernel: (total, epilogue)}."""
    M, H, I = float(w.M), float(w.H), float(w.I)
    g = w.gated
    nw = 2 if g else 1                      # gate/up weights (or fc1)
    saved = not w.recompute
    pre = nw * 2 * M * I                    # the stored preacts G, U (or P)
    a = 2 * M * I                           # the postact
    gu_pre = pre if (saved or g) else 0.0   # gate/up kernel: forward saving, or recompute stage 0
    dw_out = (8 if w.fuse_grad_accum else 2) * (nw + 1) * H * I  # fp32 RMW or bf16 store
    return {
        "fwd_fused": (2 * M * H + 2 * nw * H * I + a + (pre if saved else 0.0) + 2 * H * I
                      + 2 * M * H, a + (pre if saved else 0.0) + 2 * M * H),
        "gate_up_act": (2 * M * H + 2 * nw * H * I + a + gu_pre, a + gu_pre),
        "down_proj": (a + 2 * H * I + 2 * M * H, 2 * M * H),
        "dgated": (2 * M * H + 2 * H * I + 2 * pre + (a if saved else 0.0),
                   2 * pre + (a if saved else 0.0)),
        "dact_recompute": (4 * M * H + 4 * H * I + 2 * a, 2 * a),
        "dx": (pre + 2 * nw * H * I + 2 * M * H, 2 * M * H),
        "wgrad": (pre + a + 2 * nw * M * H + 2 * M * H + dw_out, dw_out),
    }


class StepBuffers:
    """Device inputs, outputs and workspaces of one fwd + bwd step of a
    workload, and the step's two library calls."""

    def __init__(self, m, w, dev):
        import torch
        from activated_mlp_gemms_gb300.workloads import workload_inputs
        self.m, self.w, self.dev = m, w, dev
        t = workload_inputs(w)
        self.host = t
        self.g = {k: (v.to(dev) if v is not None else None) for k, v in t.items()}
        bf = torch.bfloat16
        M, H, I = w.M, w.H, w.I
        self.prob = m.problem(M, H, I, w.act, w.gate_mult, w.down_mult)
        self.out = torch.empty(M, H, dtype=bf, device=dev)
        self.dx = torch.empty(M, H, dtype=bf, device=dev)
        wdt = torch.float32 if w.fuse_grad_accum else bf
        self.dWg = torch.zeros(I, H, dtype=wdt, device=dev)
        self.dWu = torch.zeros(I, H, dtype=wdt, device=dev) if w.gated else None
        self.dWd = torch.zeros(H, I, dtype=wdt, device=dev)
        if w.fuse_grad_accum:
            self.dWg.copy_(t["dWg_prev"])
            self.dWd.copy_(t["dWd_prev"])
            if self.dWu is not None:
                self.dWu.copy_(t["dWu_prev"])
        self.saved = not w.recompute
        self.G = torch.empty(M, I, dtype=bf, device=dev) if self.saved else None
        self.U = torch.empty(M, I, dtype=bf, device=dev) if (self.saved and w.gated) else None
        self.ws_f = m.alloc_workspace(self.prob, m.MODE_FWD, dev)
        self.ws_b = m.alloc_workspace(self.prob, m.MODE_BWD_RECOMPUTE if w.recompute
                                      else m.MODE_BWD, dev)

    def fwd(self, x=None, out=None):
        g = self.g
        self.m.mlp_fwd(self.prob, g["x"] if x is None else x, g["Wg"], g["Wu"], g["Wd"],
                       self.out if out is None else out, self.G, self.U, ws=self.ws_f)

    def bwd(self, x=None, dout=None, dx=None):
        g, w = self.g, self.w
        x = g["x"] if x is None else x
        dout = g["dout"] if dout is None else dout
        dx = self.dx if dx is None else dx
        if self.saved:
            self.m.mlp_bwd(self.prob, dout, x, g["Wg"], g["Wu"], g["Wd"], self.G, self.U, dx,
                           self.dWg, self.dWu, self.dWd, fuse_grad_accum=w.fuse_grad_accum,
                           ws=self.ws_b)
        else:
            self.m.mlp_bwd_recompute(self.prob, dout, x, g["Wg"], g["Wu"], g["Wd"], dx, self.dWg,
                                     self.dWu, self.dWd, fuse_grad_accum=w.fuse_grad_accum,
                                     ws=self.ws_b)


def time_steps(st, K, warmup, flush, world=1, on_region=None):
    """Times K fwd + bwd steps of StepBuffers `st` with CUDA events on the
    launching stream, the L2 flushed before every step outside its events.
    Returns (fwd_ms list, bwd_ms list, wall seconds, device status)."""
    import torch
    import torch.distributed as dist
    m, dev = st.m, st.dev
    for _ in range(warmup):
        st.fwd()
        st.bwd()
    torch.cuda.synchronize(dev)
    if m.mlp_device_status(st.ws_b) != 0 or m.mlp_device_status(st.ws_f) != 0:
        raise RuntimeError("device status error during warm-up")
    stream = torch.cuda.current_stream(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ctx = on_region if on_region is not None else _Null()
    wall0 = time.perf_counter()
    with ctx:
        for i in range(K):
            flush.zero_()
            ev[i][0].record(stream)
            st.fwd()
            ev[i][1].record(stream)
            st.bwd()
            ev[i][2].record(stream)
        torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    status = m.mlp_device_status(st.ws_b)
    fwd_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    bwd_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    return fwd_ms, bwd_ms, wall, status


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def trace_kernels(st, steps, flush, peaks):
    """Per-kernel device times from a separate traced pass of L2-flushed
    steps (tracing brackets every launch with events and runs the kernels
    one after another), with each kernel's TFLOP/s and algorithmic GB/s.
    Returns (kernels dict, launches per step)."""
    import torch
    m, w = st.m, st.w
    m.mlp_trace_read()
    m.mlp_trace_enable(True)
    try:
        for _ in range(steps):
            flush.zero_()
            st.fwd()
            st.bwd()
        torch.cuda.synchronize(st.dev)
    finally:
        m.mlp_trace_enable(False)
    recs = m.mlp_trace_read(capacity=64 * (steps + 1))
    per = {}
    for name, ms in recs:
        per.setdefault(name, []).append(ms)
    kf, kb = kernel_flops(w), kernel_bytes(w)
    hbm = float(peaks["hbm_gbs"])
    kernels = {}
    for name, v in per.items():
        avg = sum(v) / len(v)
        fl = kf.get(name)
        tot, epi = kb.get(name, (None, None))
        kernels[name] = {
            "launches": len(v), "avg_ms": avg, "total_ms": sum(v),
            "tflops": (fl / (avg * 1e-3) / 1e12) if fl else None,
            "algorithmic_bytes": tot, "gbs": (tot / (avg * 1e-3) / 1e9) if tot else None,
            "hbm_frac": (tot / (avg * 1e-3) / 1e9 / hbm) if tot else None,
            "epilogue_bytes": epi, "epilogue_gbs": (epi / (avg * 1e-3) / 1e9) if epi else None}
    return kernels, len(recs) // max(1, steps)


def roofline_of(kernels, w, peaks, peaks_src, exact_workload):
    """The dominant kernel's tensor roofline (its flops per launch over its
    average traced duration, against the measured bf16 burst peak), with
    ncu's DRAM bytes per launch when a capture of the current device code
    exists; and the epilogue-heavy kernel's HBM figures (the derivative GEMM
    whose epilogue reads the preacts and writes their gradients)."""
    if not kernels:
        return None
    dom = max(kernels, key=lambda k: kernels[k]["total_ms"])
    d = kernels[dom]
    peak = float(peaks["bf16_tflops"])
    sus = float(peaks.get("bf16_tflops_sustained", 0.0)) or None
    ach = d["tflops"]
    traffic = load_traffic(dom, w.name) if exact_workload else None
    src = "MEASURED_PEAKS.json" if peaks_src == "measured" else "recipe fallback"
    roof = {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": peak, "unit": "TFLOP/s",
            "frac": (ach / peak) if ach else None, "traffic": traffic,
            "peak_sustained": sus, "frac_of_sustained": (ach / sus) if (ach and sus) else None,
            "peak_source": f"{peaks_src} bf16 burst ({src})"}
    epi_k = "dact_recompute" if "dact_recompute" in kernels else "dgated"
    if epi_k in kernels:
        e = kernels[epi_k]
        hbm = float(peaks["hbm_gbs"])
        tr = load_traffic(epi_k, w.name) if exact_workload else None
        roof["epilogue"] = {
            "kernel": epi_k, "epilogue_bytes": e["epilogue_bytes"],
            "achieved_gbs": e["epilogue_gbs"], "peak_gbs": hbm,
            "frac": e["epilogue_gbs"] / hbm if e["epilogue_gbs"] else None,
            "kernel_bytes": e["algorithmic_bytes"], "kernel_gbs": e["gbs"],
            "kernel_frac": e["hbm_frac"], "traffic": tr,
            "traffic_gbs": (tr / (e["avg_ms"] * 1e-3) / 1e9) if tr else None,
            "tflops": e["tflops"], "tensor_frac": e["tflops"] / peak if e["tflops"] else None,
            "peak_source": f"{peaks_src} HBM copy ({src})"}
    return roof


def measure_workload(m, w, dev, flush, steps, warmup, peaks, peaks_src):
    """A shorter measurement of another workload for the breakdown: its
    fwd + bwd step timed as the headline is, its per-kernel trace and its
    roofline."""
    import torch
    st = StepBuffers(m, w, dev)
    fwd_ms, bwd_ms, _, status = time_steps(st, steps, warmup, flush)
    kernels, per_step = trace_kernels(st, min(steps, 10), flush, peaks)
    f_fwd, f_bwd = flops_of(w, "fwd"), flops_of(w, mode_of(w))
    ms = (sum(fwd_ms) + sum(bwd_ms)) / steps
    peak = float(peaks["bf16_tflops"])
    res = {"M": w.M, "H": w.H, "I": w.I, "act": w.act, "gate_mult": w.gate_mult,
           "down_mult": w.down_mult,
           "backward": "recompute (save only x)" if w.recompute else "saved G/U",
           "fuse_grad_accum": w.fuse_grad_accum, "steps": steps, "warmup": warmup,
           "ms_per_step": ms, "tflops": (f_fwd + f_bwd) / (ms * 1e-3) / 1e12,
           "pct_of_peak": 100.0 * (f_fwd + f_bwd) / (ms * 1e-3) / 1e12 / peak,
           "model_tflops": (flops_of(w, "fwd") + flops_of(w, "bwd")) / (ms * 1e-3) / 1e12,
           "fwd_ms": sum(fwd_ms) / steps, "bwd_ms": sum(bwd_ms) / steps,
           "fwd_tflops": f_fwd / (sum(fwd_ms) / steps * 1e-3) / 1e12,
           "bwd_tflops": f_bwd / (sum(bwd_ms) / steps * 1e-3) / 1e12,
           "kernels": kernels, "launches_per_step": per_step, "device_status": status,
           "roofline": roofline_of(kernels, w, peaks, peaks_src, True)}
    del st
    torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world, local_rank):
    import torch

    import activated_mlp_gemms_gb300 as m
    from activated_mlp_gemms_gb300.workloads import WORKLOADS, workload_inputs

    w = WORKLOADS[args.workload]
    exact = True
    if args.tokens > 0:
        import dataclasses
        w = dataclasses.replace(w, M=args.tokens)
        exact = False
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    from activated_mlp_gemms_gb300 import _build
    _build.build()

    st = StepBuffers(m, w, dev)
    g, t = st.g, st.host
    bf = torch.bfloat16
    M, H, I = w.M, w.H, w.I
    prob = st.prob
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    K = args.steps
    cvd = [c for c in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if c.strip()]
    sampler = ClockSampler(cvd[local_rank] if local_rank < len(cvd) else local_rank)
    fwd_ms, bwd_ms, wall, status = time_steps(st, K, args.warmup, flush, world, sampler)
    peaks, peaks_src = load_peaks()
    # Per-kernel durations from a separate traced pass over the same steps:
    # tracing brackets every launch with events and runs the kernels one after
    # another, so it is kept out of the timed region above.
    k_tr = min(K, 50)
    kernels, per_step = trace_kernels(st, k_tr, flush, peaks) if not args.no_trace else ({}, 0)
    step_ms = [a + b for a, b in zip(fwd_ms, bwd_ms)]
    tot_ms = sum(step_ms)
    if world > 1:
        import torch.distributed as dist
        tt = torch.tensor([tot_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        tot_ms = float(tt.item())
    ms_per_step = tot_ms / K
    f_fwd = flops_of(w, "fwd")
    f_bwd = flops_of(w, mode_of(w))
    f_step = f_fwd + f_bwd
    value = world * f_step / (ms_per_step * 1e-3) / 1e12
    roof = roofline_of(kernels, w, peaks, peaks_src, exact)
    clocks = sampler.summary()
    out, dx = st.out, st.dx

    # End to end through the C ABI with host buffers.  Every step copies its
    # inputs x and dout from pinned host memory to the device and reads its
    # results out and dx back.  The steps are pipelined as a training loop
    # drives them: double-buffered device inputs and outputs, step i+1's
    # uploads and step i's read-backs on a copy stream under the compute.
    # The serial variant (x's upload and dx's read-back on each step's
    # critical path, dout and out overlapped within the step) is reported
    # beside it.
    e2e = None
    if not args.no_e2e:
        hx = t["x"].pin_memory()
        hd = t["dout"].pin_memory()
        ho = torch.empty(M, H, dtype=bf).pin_memory()
        hdx = torch.empty(M, H, dtype=bf).pin_memory()
        cs = torch.cuda.Stream(dev)
        ke = max(4, min(K, 50))
        nb = M * H * 2
        xb = [g["x"], torch.empty_like(g["x"])]
        db = [g["dout"], torch.empty_like(g["dout"])]
        ob = [out, torch.empty_like(out)]
        dxb = [dx, torch.empty_like(dx)]

        def pipelined(nsteps):
            ev_in = [torch.cuda.Event(), torch.cuda.Event()]
            ev_fwd = [torch.cuda.Event(), torch.cuda.Event()]
            ev_bwd = [torch.cuda.Event(), torch.cuda.Event()]
            ev_out = [torch.cuda.Event(), torch.cuda.Event()]
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            e0.record(stream)
            cs.wait_event(e0)
            with torch.cuda.stream(cs):
                xb[0].copy_(hx, non_blocking=True)
                db[0].copy_(hd, non_blocking=True)
                ev_in[0].record(cs)
            for i in range(nsteps):
                b = i % 2
                stream.wait_event(ev_in[b])
                if i >= 2:
                    stream.wait_event(ev_out[b])  # step i-2's read-backs of these buffers
                st.fwd(x=xb[b], out=ob[b])
                ev_fwd[b].record(stream)
                st.bwd(x=xb[b], dout=db[b], dx=dxb[b])
                ev_bwd[b].record(stream)
                with torch.cuda.stream(cs):
                    if i + 1 < nsteps:
                        if i >= 1:
                            cs.wait_event(ev_bwd[1 - b])  # step i-1 is done with its inputs
                        xb[1 - b].copy_(hx, non_blocking=True)
                        db[1 - b].copy_(hd, non_blocking=True)
                        ev_in[1 - b].record(cs)
                    cs.wait_event(ev_fwd[b])
                    ho.copy_(ob[b], non_blocking=True)
                    cs.wait_event(ev_bwd[b])
                    hdx.copy_(dxb[b], non_blocking=True)
                    ev_out[b].record(cs)
            stream.wait_event(ev_out[(nsteps - 1) % 2])
            e1.record(stream)
            torch.cuda.synchronize(dev)
            return e0.elapsed_time(e1) / nsteps

        pipelined(3)  # warm-up
        tms = pipelined(ke)

        # serial variant
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        ev_dout = torch.cuda.Event()
        ev_fwd = torch.cuda.Event()
        ev_out = torch.cuda.Event()
        tser = 0.0
        for i in range(ke + 2):
            flush.zero_()
            e0.record(stream)
            cs.wait_event(e0)
            g["x"].copy_(hx, non_blocking=True)
            with torch.cuda.stream(cs):
                g["dout"].copy_(hd, non_blocking=True)
                ev_dout.record(cs)
            st.fwd()
            ev_fwd.record(stream)
            with torch.cuda.stream(cs):
                cs.wait_event(ev_fwd)
                ho.copy_(out, non_blocking=True)
                ev_out.record(cs)
            stream.wait_event(ev_dout)
            st.bwd()
            hdx.copy_(dx, non_blocking=True)
            stream.wait_event(ev_out)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if i >= 2:
                tser += e0.elapsed_time(e1)
        tser /= ke
        if world > 1:
            import torch.distributed as dist
            tt = torch.tensor([tms, tser], device=dev, dtype=torch.float64)
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            tms, tser = float(tt[0].item()), float(tt[1].item())
        e2e = {"value": world * f_step / (tms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": tms,
               "h2d_bytes_per_step": 2 * nb, "d2h_bytes_per_step": 2 * nb,
               "schedule": "pipelined steps: the next step's x/dout uploads and this step's "
                           "out/dx read-backs on a copy stream under the compute; no L2 flush "
                           "(the weights exceed L2)",
               "serial": {"value": world * f_step / (tser * 1e-3) / 1e12, "ms_per_step": tser,
                          "schedule": "x upload and dx read-back on each step's critical path "
                                      "(dout/out overlapped within the step); L2 flushed"}}

    # extra: the no-grad inference forward of workloads that name it
    infer = None
    if w.infer:
        ei0 = torch.cuda.Event(enable_timing=True)
        ei1 = torch.cuda.Event(enable_timing=True)
        ws_i = m.alloc_workspace(prob, m.MODE_INFER, dev)
        for _ in range(3):
            m.mlp_fwd_infer(prob, g["x"], g["Wg"], g["Wu"], g["Wd"], out, ws=ws_i)
        ims = []
        for _ in range(max(3, min(K, 50))):
            flush.zero_()
            ei0.record(stream)
            m.mlp_fwd_infer(prob, g["x"], g["Wg"], g["Wu"], g["Wd"], out, ws=ws_i)
            ei1.record(stream)
            torch.cuda.synchronize(dev)
            ims.append(ei0.elapsed_time(ei1))
        im = sum(ims) / len(ims)
        infer = {"ms": im, "tflops": flops_of(w, "infer") / (im * 1e-3) / 1e12,
                 "pct_of_peak": 100.0 * flops_of(w, "infer") / (im * 1e-3) / 1e12
                 / float(peaks["bf16_tflops"])}

    # the decode-sized inference forward: part of the default single-GPU run
    do_sweep = args.sweep_m or (world == 1 and not args.headline_only)
    sweep = infer_m_sweep(m, w, g, dev, flush, peaks) if do_sweep else None
    block = block_step(m, w, g, dev, flush, K) if args.block else None
    fp8 = fp8_forward(m, w, g, dev, flush, K, peaks) if (args.fp8 and w.act == "relu_sq") else None
    launches = per_step * K if kernels else None
    del st, g, out, dx
    torch.cuda.empty_cache()

    # the other workloads, a few steps each (rank 0 of a single-GPU run only)
    workloads = None
    if world == 1 and not args.headline_only:
        workloads = {}
        ksub = max(3, min(K, 10))
        for name, ow in WORKLOADS.items():
            if name == w.name:
                continue
            r = measure_workload(m, ow, dev, flush, ksub, 3, peaks, peaks_src)
            if ow.act == "relu_sq":
                og = {k: (v.to(dev) if v is not None else None)
                      for k, v in workload_inputs(ow).items()}
                r["fp8"] = fp8_forward(m, ow, og, dev, flush, ksub, peaks)
                r["block"] = block_step(m, ow, og, dev, flush, ksub)
                del og
                torch.cuda.empty_cache()
            workloads[name] = r

    peak = float(peaks["bf16_tflops"])
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, nn.Linear Kaiming-uniform weights)",
        "config": {"workload": w.name, "M": M, "H": H, "I": I, "act": w.act,
                   "gate_mult": w.gate_mult, "down_mult": w.down_mult,
                   "backward": "recompute (save only x)" if w.recompute else "saved G/U",
                   "fuse_grad_accum": w.fuse_grad_accum,
                   "l2": "flushed before every timed step (512 MiB write, outside the step events)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "pct_of_peak": 100.0 * value / world / peak,
        "peak_tflops": peak, "peak_source": peaks_src,
        "breakdown": {"fwd_ms": sum(fwd_ms) / K, "bwd_ms": sum(bwd_ms) / K,
                      "fwd_tflops": f_fwd / (sum(fwd_ms) / K * 1e-3) / 1e12,
                      "bwd_tflops": f_bwd / (sum(bwd_ms) / K * 1e-3) / 1e12,
                      "model_flops_per_step": flops_of(w, "fwd") + flops_of(w, "bwd"),
                      "executed_flops_per_step": f_step,
                      "model_tflops": world * (flops_of(w, "fwd") + flops_of(w, "bwd"))
                      / (ms_per_step * 1e-3) / 1e12,
                      "kernels": kernels,
                      "kernels_timing": f"separate traced pass of {k_tr} L2-flushed steps, "
                                        "kernels serialised (no side stream, no PDL overlap)",
                      "infer": infer, "infer_m_sweep": sweep, "block": block, "fp8_forward": fp8,
                      "workloads": workloads},
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "device_status": status,
        "wall_s_timed_region": wall,
    }
    return res, w


def fp8_forward(m, w, g, dev, flush, K, peaks):
    """The e4m3 forward (mlp_fp8_fwd) on the workload's weights quantised with
    amax/448 scales and x with the page's static 2^-4, against the bf16
    inference forward; and the FP8 training step (the forward saving its
    bf16 preact, then mlp_fp8_bwd with e5m2 gradients: the static 2^-6 for
    dout, the delayed dpre scale as it settles) against the bf16 one
    (mlp_fwd saving the preact, mlp_bwd).  The codes of x and the weights
    are made once, outside the timing (the input's quantisation is timed on
    its own).  The 8-bit peak is the measured bf16 peak times the nominal
    ratio 2."""
    import torch
    M, H, I = w.M, w.H, w.I
    prob = m.problem(M, H, I, "relu_sq", w.gate_mult, w.down_mult)

    def quant(x, s):
        d = torch.empty(x.shape, dtype=torch.uint8, device=dev)
        m.mlp_fp8_quantize(x, torch.tensor([s], dtype=torch.float32, device=dev), d)
        return d
    s1 = float(g["Wg"].abs().max()) / 448.0
    s2 = float(g["Wd"].abs().max()) / 448.0
    x8, W1_8, W2_8 = quant(g["x"], 2.0 ** -4), quant(g["Wg"], s1), quant(g["Wd"], s2)
    # the post scale as the page's delayed one would settle: amax x 1.03 / 448
    pre = (g["x"][:256].float() @ g["Wg"].float().T).clamp(min=0) ** 2
    s_post = float(pre.max()) * w.gate_mult * 1.03 / 448.0
    bf = torch.bfloat16
    scales = torch.tensor([2.0 ** -4, s1, s2, s_post, 2.0 ** -6, 1.0], dtype=torch.float32,
                          device=dev)
    out = torch.empty(M, H, dtype=bf, device=dev)
    a8 = torch.empty(M, I, dtype=torch.uint8, device=dev)
    pre_s = torch.empty(M, I, dtype=bf, device=dev)
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    amax_d = torch.zeros(1, dtype=torch.float32, device=dev)
    dx = torch.empty(M, H, dtype=bf, device=dev)
    dW1 = torch.empty(I, H, dtype=bf, device=dev)
    dW2 = torch.empty(H, I, dtype=bf, device=dev)
    ws8 = m.alloc_workspace(prob, m.MODE_FP8_FWD, dev)
    wsb8 = m.alloc_workspace(prob, m.MODE_FP8_BWD, dev)
    wsi = m.alloc_workspace(prob, m.MODE_INFER, dev)
    wsb = m.alloc_workspace(prob, m.MODE_BWD, dev)
    sx_t = scales[:1]
    xq = torch.empty_like(x8)

    def fp8_fwd_train():
        m.mlp_fp8_fwd(prob, x8, W1_8, W2_8, scales, out, a8, amax, ws=ws8, pre_save=pre_s)

    def fp8_bwd():
        m.mlp_fp8_bwd(prob, g["dout"], x8, W1_8, W2_8, pre_s, a8, scales, dx, dW1, dW2, amax_d,
                      ws=wsb8)
    # the delayed dpre scale as it settles: the last step's amax x 1.25 / 57344
    fp8_fwd_train()
    fp8_bwd()
    torch.cuda.synchronize(dev)
    scales[5] = float(amax_d.item()) * 1.25 / 57344.0

    def bf16_train():
        m.mlp_fwd(prob, g["x"], g["Wg"], None, g["Wd"], out, pre_s, ws=wsb)
        m.mlp_bwd(prob, g["dout"], g["x"], g["Wg"], None, g["Wd"], pre_s, None, dx, dW1, None, dW2,
                  ws=wsb)
    def fp8_train_recompute():
        # the forward saves no preact; the backward's derivative GEMM recomputes it
        m.mlp_fp8_fwd(prob, x8, W1_8, W2_8, scales, out, a8, amax, ws=ws8)
        m.mlp_fp8_bwd(prob, g["dout"], x8, W1_8, W2_8, None, a8, scales, dx, dW1, dW2, amax_d,
                      ws=wsb8)
    runs = {"fp8_ms": lambda: m.mlp_fp8_fwd(prob, x8, W1_8, W2_8, scales, out, a8, amax, ws=ws8),
            "bf16_ms": lambda: m.mlp_fwd_infer(prob, g["x"], g["Wg"], None, g["Wd"], out, ws=wsi),
            "quantize_x_ms": lambda: m.mlp_fp8_quantize(g["x"], sx_t, xq),
            "fp8_bwd_ms": fp8_bwd,
            "fp8_train_ms": lambda: (fp8_fwd_train(), fp8_bwd()),
            "fp8_train_recompute_ms": fp8_train_recompute,
            "bf16_train_ms": bf16_train}
    res = {}
    for name, fn in runs.items():
        for _ in range(3):
            fn()
        ts = []
        for _ in range(max(5, min(K, 30))):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1))
        res[name] = sorted(ts)[len(ts) // 2]
    f = flops_of(w, "fwd")
    peak = 2.0 * float(peaks["bf16_tflops"])
    res["fp8_tflops"] = f / (res["fp8_ms"] * 1e-3) / 1e12
    res["bf16_tflops"] = f / (res["bf16_ms"] * 1e-3) / 1e12
    res["fp8_peak_tflops"] = peak
    res["fp8_frac"] = res["fp8_tflops"] / peak
    ft = flops_of(w, "fwd") + flops_of(w, "bwd")
    res["fp8_train_tflops"] = ft / (res["fp8_train_ms"] * 1e-3) / 1e12
    res["fp8_bwd_tflops"] = flops_of(w, "bwd") / (res["fp8_bwd_ms"] * 1e-3) / 1e12
    res["bf16_train_tflops"] = ft / (res["bf16_train_ms"] * 1e-3) / 1e12
    res["fp8_train_frac"] = res["fp8_train_tflops"] / peak
    # the same step recomputing the preact in the backward (model flops, as above)
    res["fp8_train_recompute_tflops"] = ft / (res["fp8_train_recompute_ms"] * 1e-3) / 1e12
    res["fp8_train_recompute_frac"] = res["fp8_train_recompute_tflops"] / peak
    res["peak_source"] = "measured bf16 burst x 2 (e4m3 / bf16 nominal ratio)"
    return res


def block_step(m, w, g, dev, flush, K):
    """fwd + bwd of the MLP block with its neighbours (RMS-normalised input,
    scaled residual add; saved preacts, bf16 weight gradients) against the
    plain MLP's fwd + bwd on the same inputs, L2 flushed before each step."""
    import torch
    bf = torch.bfloat16
    M, H, I = w.M, w.H, w.I
    prob = m.problem(M, H, I, w.act, w.gate_mult, w.down_mult)
    blk = m.block(1.1 ** 0.5, 0.8, 2.0 ** -7)
    G = torch.empty(M, I, dtype=bf, device=dev)
    U = torch.empty(M, I, dtype=bf, device=dev) if w.gated else None
    y = torch.empty(M, H, dtype=bf, device=dev)
    dx = torch.empty(M, H, dtype=bf, device=dev)
    dWg = torch.empty(I, H, dtype=bf, device=dev)
    dWu = torch.empty(I, H, dtype=bf, device=dev) if w.gated else None
    dWd = torch.empty(H, I, dtype=bf, device=dev)
    rstd = torch.empty(M, dtype=torch.float32, device=dev)
    wsf = m.alloc_workspace(prob, m.MODE_FWD, dev)
    wsb = m.alloc_workspace(prob, m.MODE_BWD, dev)

    def plain():
        m.mlp_fwd(prob, g["x"], g["Wg"], g["Wu"], g["Wd"], y, G, U, ws=wsf)
        m.mlp_bwd(prob, g["dout"], g["x"], g["Wg"], g["Wu"], g["Wd"], G, U, dx, dWg, dWu, dWd,
                  ws=wsb)

    def blk_step():
        m.mlp_block_fwd(prob, blk, g["x"], g["Wg"], g["Wu"], g["Wd"], y, G, U, rstd, ws=wsf)
        m.mlp_block_bwd(prob, blk, g["dout"], g["x"], g["Wg"], g["Wu"], g["Wd"], G, U, rstd, dx,
                        dWg, dWu, dWd, ws=wsb)

    res = {}
    for name, fn in (("plain_ms", plain), ("block_ms", blk_step)):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(max(5, min(K, 30))):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1))
        res[name] = sorted(ts)[len(ts) // 2]
    f = flops_of(w, "fwd") + flops_of(w, "bwd")
    res["block_tflops"] = f / (res["block_ms"] * 1e-3) / 1e12
    res["plain_tflops"] = f / (res["plain_ms"] * 1e-3) / 1e12
    res["overhead"] = res["block_ms"] / res["plain_ms"] - 1.0
    res["lambdas"] = {"resid_lambda": 1.1 ** 0.5, "post_lambda": 0.8, "eps": 2.0 ** -7}
    return res


def infer_m_sweep(m, w, g, dev, flush, peaks):
    """The no-grad forward at decode-sized token counts with the workload's
    weights: direct calls and CUDA-graph replays, CUDA events per call, L2
    flushed before each.  Reports time, TFLOP/s and the weight-streaming rate
    (the three weight matrices are read once per call)."""
    import torch
    bf = torch.bfloat16
    wbytes = (3 if w.gated else 2) * w.H * w.I * 2
    rows = []
    for M in (1, 2, 3, 4, 8, 16, 17, 32, 64, 128, 256, 512):
        prob = m.problem(M, w.H, w.I, w.act, w.gate_mult, w.down_mult)
        x = torch.randn(M, w.H, device=dev).to(bf)
        out = torch.empty(M, w.H, dtype=bf, device=dev)
        ws = m.alloc_workspace(prob, m.MODE_INFER, dev)

        def call():
            m.mlp_fwd_infer(prob, x, g["Wg"], g["Wu"], g["Wd"], out, ws=ws)
        for _ in range(3):
            call()
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call()
        res = {}
        for name, fn in (("direct", call), ("graph", graph.replay)):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            ts = []
            for _ in range(20):
                flush.zero_()
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize(dev)
                ts.append(e0.elapsed_time(e1))
            res[name] = sorted(ts)[len(ts) // 2] * 1e3  # median, us
        best = min(res.values())
        path = ("warp_mma_stream", "cuda_core_stream", "tensor_core_gemm")[
            [2, 1, 0].index(m.mlp_plan(prob, m.MODE_INFER)["decode"])]
        # the other weight stream on the same call, where both apply (1-4 tokens)
        alt_path, alt_us = None, None
        if path != "tensor_core_gemm" and M <= 4:
            alt = "cuda_core_stream" if path == "warp_mma_stream" else "warp_mma_stream"
            m.mlp_debug_set_flags(m.DEBUG_DECODE_FMA if alt == "cuda_core_stream"
                                  else m.DEBUG_DECODE_MMA)
            try:
                if m.mlp_plan(prob, m.MODE_INFER)["decode"] == (1 if alt == "cuda_core_stream" else 2):
                    alt_path = alt
                    for _ in range(3):
                        call()
                    torch.cuda.synchronize(dev)
                    g2 = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g2):
                        call()
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    ts = []
                    for _ in range(20):
                        flush.zero_()
                        e0.record()
                        g2.replay()
                        e1.record()
                        torch.cuda.synchronize(dev)
                        ts.append(e0.elapsed_time(e1))
                    alt_us = sorted(ts)[len(ts) // 2] * 1e3
            finally:
                m.mlp_debug_set_flags(0)
        rows.append({"M": M, "path": path, "direct_us": res["direct"], "graph_us": res["graph"],
                     "alt_path": alt_path, "alt_graph_us": alt_us,
                     "tflops": (6 if w.gated else 4) * M * w.H * w.I / (best * 1e-6) / 1e12,
                     "weight_gbs": wbytes / (best * 1e-6) / 1e9,
                     "hbm_frac": wbytes / (best * 1e-6) / 1e9 / float(peaks["hbm_gbs"])})
    return rows


# ------------------------------------------------------------ CPU oracle

def oracle_threads():
    """Threads the oracle's numpy BLAS calls run on."""
    try:
        from threadpoolctl import threadpool_info
        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except ImportError:
        pass
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(v, "").isdigit():
            return int(os.environ[v])
    return len(os.sched_getaffinity(0))


def oracle_sample(w, seconds, steps=1):
    """Time the fp64 oracle on a bounded token sample of the workload."""
    import numpy as np

    from activated_mlp_gemms_gb300.workloads import to_f64, workload_inputs
    from oracle import mlp_backward

    t = workload_inputs(w)
    a = {k: to_f64(v) for k, v in t.items() if v is not None}
    Wu = a.get("Wu")
    prev = None
    if w.fuse_grad_accum:
        prev = {"dWg": a["dWg_prev"], "dWu": a.get("dWu_prev"), "dWd": a["dWd_prev"]}

    def one(n):
        t0 = time.perf_counter()
        mlp_backward(a["dout"][:n], a["x"][:n], a["Wg"], Wu, a["Wd"], w.act, w.gate_mult,
                     w.down_mult, dW_prev=prev)  # runs the forward internally
        return time.perf_counter() - t0

    # calibrate on 16 tokens, then size the sample to the time budget per step
    n0 = min(16, w.M)
    t0 = one(n0)
    per_tok = t0 / n0
    n = int(max(8, min(w.M, seconds / max(per_tok, 1e-9))))
    times = [one(n) for _ in range(steps)]
    # flops of the oracle pass: forward + backward (saved-preact arithmetic)
    f = flops_of(type("W", (), {"M": n, "H": w.H, "I": w.I, "gated": w.gated})(), "fwd") + \
        flops_of(type("W", (), {"M": n, "H": w.H, "I": w.I, "gated": w.gated})(), "bwd")
    tpt = sum(times) / len(times)
    return {"value": f / tpt / 1e12, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
            "sample": f"{n} of {w.M} tokens (full H={w.H}, I={w.I}), oracle forward+backward in "
                      f"numpy fp64, {len(times)} pass(es), {tpt:.2f} s each",
            "seconds_per_pass": tpt, "tokens": n}, tpt


def run_reference(args, rank, world):
    from activated_mlp_gemms_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.tokens > 0:
        import dataclasses
        w = dataclasses.replace(w, M=args.tokens)
    K, W = args.steps, args.warmup
    budget = 150.0  # seconds for the whole reference run
    per_step = max(0.5, budget / max(1, K + W))
    cb, _ = oracle_sample(w, per_step, steps=1)
    n = cb["tokens"]
    import numpy as np  # noqa: F401

    from activated_mlp_gemms_gb300.workloads import to_f64, workload_inputs
    from oracle import mlp_backward
    t = workload_inputs(w)
    a = {k: to_f64(v) for k, v in t.items() if v is not None}
    prev = None
    if w.fuse_grad_accum:
        prev = {"dWg": a["dWg_prev"], "dWu": a.get("dWu_prev"), "dWd": a["dWd_prev"]}

    def step():
        mlp_backward(a["dout"][:n], a["x"][:n], a["Wg"], a.get("Wu"), a["Wd"], w.act, w.gate_mult,
                     w.down_mult, dW_prev=prev)

    for _ in range(W):
        step()
    t0 = time.perf_counter()
    for _ in range(K):
        step()
    sec = (time.perf_counter() - t0) / max(1, K)
    W_ = type("W", (), {"M": n, "H": w.H, "I": w.I, "gated": w.gated})()
    f = flops_of(W_, "fwd") + flops_of(W_, "bwd")
    val = f / sec / 1e12
    cpu = {"value": val, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
           "sample": f"{n} of {w.M} tokens per step (full H={w.H}, I={w.I}), oracle "
                     f"forward+backward in numpy fp64"}
    return {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "M": w.M, "H": w.H, "I": w.I, "act": w.act,
                       "gate_mult": w.gate_mult, "down_mult": w.down_mult,
                       "backward": "recompute (save only x)" if w.recompute else "saved G/U",
                       "fuse_grad_accum": w.fuse_grad_accum},
            "cpu_baseline": cpu,
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res, w = run_ours(args, rank, world, local_rank)
    if rank == 0 and not args.no_cpu_baseline:
        cb, _ = oracle_sample(w, args.cpu_seconds, steps=1)
        cb.pop("seconds_per_pass", None)
        cb.pop("tokens", None)
        res["cpu_baseline"] = cb
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
