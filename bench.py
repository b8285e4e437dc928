#!/usr/bin/env python
"""Benchmark of the NHA layer operator (forward + backward) on GB300.

One step = nha_forward + nha_backward over one batch of the chosen workload
(the backward given the forward's workspace, so it reuses the chunk states and
rotated q, k the forward formed, as a training step keeps them)
(default: the 1.3B-like layer, B4 H16 T2048 d128 m64 w512 C64, bf16), inputs
resident in HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl nha|reference]

Multi-GPU: one process per GPU under torchrun; every rank runs the same
per-GPU workload (heads are independent, so the work partitions over B x H
with no collective); value = tokens of all ranks / the slowest rank's time.

--impl reference times the fp64 CPU oracle (the method's plain definition) on
this machine's host cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
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
sys.path.insert(0, ROOT)

METRIC = "NHA layer fwd and fwd+bwd tokens/s on 1 GB300; fraction of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
L2_FLUSH_BYTES = 512 << 20


def workloads():
    from sliding_window_softmax_gb300 import synthetic as s

    out = {"1.3B": s.LAYER_1P3B, "340M": s.LAYER_340M, "tiny": s.TINY_F32,
           "1.3B-w0": s.LAYER_1P3B.with_(name="1.3B-like w=0", w=0),
           "1.3B-wT": s.LAYER_1P3B.with_(name="1.3B-like w=T", w=2048)}
    for T in s.LONG_CONTEXT_T:
        out[f"long{T}"] = s.long_context(T)
    for w in s.GRID_W:
        for m in s.GRID_M:
            out[f"grid-w{w}-m{m}"] = s.grid_point(w, m)
    return out


# ----------------------------------------------------------------------------------------
# Algorithmic work model: flops and bytes per launch, the roofline denominators.
def work_model(wl):
    T, d, m = wl.T, wl.d, wl.m
    w = min(wl.w, T)
    R = max(0, T - w)
    e = 2 if wl.dtype == "bf16" else 4
    n_sum = sum(min(t + 1, w) for t in range(T)) if w > 0 else 0  # window keys per head
    BH = wl.B * wl.H
    fwd_flops = BH * (4 * d * n_sum + 8 * m * d * R)
    fwd_bytes = BH * T * (4 * d * e + 4 * m + 4)
    bwd_bytes = BH * T * (8 * d * e + 8 * m + 4)
    # Per-kernel algorithmic bytes: every input a kernel reads and every output
    # it writes, once (the bf16 tensor-core kernels as designed).  Per token:
    # e-byte rows of width d, fp32 log_alpha rows (4m), bf16 slot rows (2m);
    # per 128-row tile, pairs of bf16 [m][d] chunk states (2 * 2 m d bytes).
    tiles = (R + 127) // 128
    pair = 2 * 2 * m * d  # one [2m][d] bf16 pair
    fwd_main = (BH * (4 * d * n_sum + 8 * m * d * R),
                BH * T * (6 * d * e + 4 * m + 4) + BH * tiles * 2 * pair)
    # q~, dout, o, k~, v in; dq and its correction partial out; D^, D_win
    wdq = (BH * 8 * d * n_sum, BH * T * (7 * d * e + 12))
    # q~, dout, k~, v, lse, D in; dk, dv partials out
    wkv = (BH * 8 * d * n_sum, BH * T * (6 * d * e + 8))
    # q, k, v, dout, dq partials, log_alpha, lse, D_win, D^ in; state pairs in;
    # dq, sigma dL, P_L (bf16), db1, D out; bf16 chunk adjoint contributions out
    sq = (BH * 12 * m * d * R,
          BH * T * (7 * d * e + 4 * m + 16) + BH * R * (2 * 2 * m + 4 * m) + BH * tiles * 2 * pair
          + BH * ((R + 63) // 64) * 2 * m * d * 2)
    # q, dout, k, v, dk / dv partials in; dk, dv out; log_alpha, sigma dL, P_L,
    # db1 in; dlog_alpha out; adjoint pairs in
    sk = (BH * 12 * m * d * R,
          BH * T * (8 * d * e + 4 * m + 4 * m) + BH * R * (2 * 2 * m + 4 * m) + BH * tiles * 2 * pair)
    k = {
        # name: (algorithmic flops, algorithmic bytes) per launch; the tensor-core
        # (bf16) and SIMT (fp32) kernels of the same step share a model
        "fwd_tc": fwd_main, "fwd_main": fwd_main,
        "state_chunk": (BH * 4 * m * d * R, BH * R * (2 * d * e + 4 * m)),
        # bf16 path: the chunk scan with the chunk coefficients formed inside
        # (K, V in; log_alpha in by the K and the V CTA; the bf16 states
        # entering each chunk out)
        "state_scan": (BH * 4 * m * d * R, BH * R * (2 * d * e + 8 * m) + BH * ((R + 63) // 64) * 4 * m * d),
        # reverse adjoint scan with the dlog_alpha carries: bf16 contributions
        # and bf16 states in, bf16 adjoints out, K and V
        "adj_scan": (BH * ((R + 63) // 64) * m * d * 4, BH * ((R + 63) // 64) * m * d * 12),
        # RoPE(q), RoPE(k) in bf16 and the (cos, sin) table: q, k in, copies out
        "rope_qk": (0, BH * T * 4 * d * e + T * d * 4),
        "bwd_wdq_tc": wdq, "bwd_window_dq": wdq,
        "bwd_wkv_tc": wkv, "bwd_window_dkdv": wkv,
        "bwd_sq_tc": sq, "bwd_slot_query": sq,
        "bwd_sk_tc": sk, "bwd_slot_key": sk,
    }
    # fwd + bwd flops: 3.5 x the forward (the FlashAttention convention: the
    # backward counts 2.5 forwards)
    return dict(fwd_flops=fwd_flops, fwd_bytes=fwd_bytes, step_flops=3.5 * fwd_flops,
                step_bytes=fwd_bytes + bwd_bytes, kernels=k, n_sum=n_sum, R=R)


def step_roofline(model, peaks, ms, backward=True):
    """Roofline of one whole step: the slower of the algorithmic flops at the
    dense bf16 peak and the algorithmic bytes at the HBM bandwidth.  Returns
    (t_roof seconds, roofline object) with frac = t_roof / measured time."""
    if backward:
        flops, nbytes = model["step_flops"], model["step_bytes"]
    else:
        flops, nbytes = model["fwd_flops"], model["fwd_bytes"]
    tc_peak = peaks["bf16_tflops"] * 1e12
    bw_peak = peaks["hbm_gbs"] * 1e9
    t_roof = max(flops / tc_peak, nbytes / bw_peak)
    sec = ms / 1e3
    if flops / tc_peak > nbytes / bw_peak:
        roof = {"bound": "tensor", "achieved": flops / sec / 1e12, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": nbytes / sec / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["algorithmic_bytes"] = nbytes
    roof["algorithmic_flops"] = flops
    roof["scope"] = "one whole step (" + ("fwd+bwd" if backward else "fwd") + ")"
    return t_roof, roof


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                "source": "measured"}
    return dict(FALLBACK_PEAKS, bf16_tflops_sustained=1700.0, source="fallback")


CSRC = os.path.join(ROOT, "sliding_window_softmax_gb300", "csrc")


def kernel_source_hash(kernel: str, reader=None) -> str:
    """Hash of the sources that define a kernel: the csrc .cu files that
    launch a kernel under that name and the csrc headers they include, transitively.
    ``reader(name) -> bytes`` reads a csrc file (default: the working tree)."""
    if reader is None:
        def reader(name):
            with open(os.path.join(CSRC, name), "rb") as fh:
                return fh.read()
    names = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    tag = ('NHA_LAUNCH("%s"' % kernel).encode()
    todo = [f for f in names if tag in reader(f)]
    if not todo:
        return "none"
    seen = []
    while todo:
        f = todo.pop()
        if f in seen:
            continue
        seen.append(f)
        for inc in re.findall(rb'#include "([^"]+)"', reader(f)):
            inc = inc.decode()
            if os.path.exists(os.path.join(CSRC, inc)):
                todo.append(inc)
    h = hashlib.sha256()
    for f in sorted(seen):
        h.update(f.encode() + b"\0" + reader(f))
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload_key: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the kernel's current sources (lines `traffic <kernel> <workload> <hash> <bytes>`,
    the hash from kernel_source_hash)."""
    p = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(p):
        return None
    cur = kernel_source_hash(kernel)
    with open(p) as f:
        for line in f:
            mm = re.match(r"\s*traffic\s+(\S+)\s+(\S+)\s+(\S+)\s+([0-9.eE+]+)", line)
            if mm and mm.group(1) == kernel and mm.group(2) == workload_key and mm.group(3) == cur:
                return float(mm.group(4))
    return None


def step_traffic(launches_per_step: dict, workload_key: str):
    """DRAM bytes of one whole step: the per-launch ncu traffic of every kernel
    the step launches times its launches per step, or None when a kernel has no
    capture on its current sources."""
    total = 0.0
    for k, n in launches_per_step.items():
        t = ncu_traffic(k, workload_key)
        if t is None:
            return None
        total += t * n
    return total


# ----------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples every 100 ms; summary() keeps those taken inside the
    timed region (or the three nearest to it when the region is shorter)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []  # (host time, csv line)
        self.window = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, t0: float, t1: float):
        """The timed region, in host time.time() seconds."""
        self.window = (t0, t1)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = self.lines
        if self.window is not None:
            inside = [x for x in lines if self.window[0] <= x[0] <= self.window[1]]
            if len(inside) < 3:  # too short a region: take the samples nearest to it
                mid = 0.5 * (self.window[0] + self.window[1])
                inside = sorted(lines, key=lambda x: abs(x[0] - mid))[:3]
            lines = inside
        for _, ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------------------
def oracle_sample(wl, heads, nthreads):
    """fwd + bwd of the fp64 oracle on `heads` heads (batch-major order); returns seconds."""
    import torch

    import oracle
    from sliding_window_softmax_gb300.synthetic import make_inputs

    x = make_inputs(wl)
    idx = [(i // wl.H, i % wl.H) for i in range(heads)]
    sel = {n: torch.stack([t[b, h] for b, h in idx])[None] for n, t in x.items()}
    t0 = time.perf_counter()
    oracle.forward(sel["q"], sel["k"], sel["v"], sel["log_alpha"], wl.w, nthreads=nthreads)
    if wl.backward:
        oracle.backward(sel["q"], sel["k"], sel["v"], sel["log_alpha"], sel["dout"], wl.w,
                        nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_baseline(wl, budget_s=20.0):
    import oracle

    cores = os.cpu_count() or 1
    oracle.build()
    t1 = oracle_sample(wl, 1, 1)
    heads = int(min(wl.B * wl.H, cores * max(1, math.floor(budget_s / max(t1, 1e-3)))))
    heads = max(1, min(heads, cores))
    sec = oracle_sample(wl, heads, min(cores, heads))
    tokens = heads * wl.T / wl.H  # a token is one position across all H heads
    return {"value": tokens / sec, "unit": "tokens/s", "cores": min(cores, heads), "kind": "oracle",
            "sample": f"{heads} of {wl.B * wl.H} heads of {wl.name}, "
                      f"{'fwd+bwd' if wl.backward else 'fwd'}, fp64, {sec:.2f} s wall"}


def run_reference(args, wl):
    """The reference arm: the oracle on the host cores, bounded sample per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    cores = os.cpu_count() or 1
    oracle.build()
    t1 = oracle_sample(wl, 1, 1)
    per_step = 150.0 / max(1, args.steps + args.warmup + 1)
    heads = max(1, min(cores, wl.B * wl.H, int(per_step / max(t1, 1e-3)) * cores))
    nth = min(cores, heads)
    for _ in range(args.warmup):
        oracle_sample(wl, heads, nth)
    times = [oracle_sample(wl, heads, nth) for _ in range(args.steps)]
    ms = 1e3 * statistics.mean(times)
    tokens = heads * wl.T / wl.H
    val = tokens / (ms / 1e3)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.B, "H": wl.H, "T": wl.T, "d": wl.d,
                       "m": wl.m, "w": wl.w, "C": wl.C, "pass": "fwd+bwd" if wl.backward else "fwd",
                       "sample_heads": heads},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": nth, "kind": "oracle",
                             "sample": f"{heads} of {wl.B * wl.H} heads per step"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------
def decode_bytes(dw):
    """Algorithmic bytes of one decode-step launch (one layer, all B*H heads)."""
    d, m, w = dw.d, dw.m, dw.w
    e = 2 if dw.dtype == "bf16" else 4
    per_head = (16 * m * d                 # S^K, S^V read and written back, fp32
                + 2 * d * e * max(w - 1, 0)  # window keys and values t-w+1 .. t-1 from the ring
                + (2 * d * e + 4 * m) * (1 if dw.t >= w and w > 0 else 0)  # leaving token
                + (2 * d * e + 4 * m) * (1 if w > 0 else 0)  # token t written into the ring
                + 4 * d * e + 4 * m)         # q, k, v, log_alpha in; o out
    return dw.B * dw.H * per_head


def decode_cpu_baseline(dw, layers=3):
    """The fp64 decode-step oracle on `layers` layer steps of the workload."""
    import numpy as np

    from oracle.decode import DecodeState, decode_step
    from sliding_window_softmax_gb300.synthetic import make_decode_layer

    secs = 0.0
    for layer in range(layers):
        x, state = make_decode_layer(dw, layer, device="cpu")
        st = DecodeState(dw.B, dw.H, dw.d, dw.m, dw.w)
        st.S_k, st.S_v, st.ring_k, st.ring_v, st.ring_la = (a.double().numpy() for a in state)
        xs = {n: t.double().numpy() for n, t in x.items()}
        t0 = time.perf_counter()
        decode_step(st, xs["q"], xs["k"], xs["v"], xs["log_alpha"], dw.t)
        secs += time.perf_counter() - t0
    per_layer = secs / layers
    return {"value": dw.B / (per_layer * dw.layers), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{layers} layer steps of all {dw.B * dw.H} heads (numpy fp64, one thread); "
                      f"value = B / ({dw.layers} x the mean layer-step time)"}


def run_decode(args, dev, stream, layers_override=None, batch_override=None):
    """One decode token for B sequences through every layer of the decode
    workload: one nha_decode_step launch per layer, the layers' launches
    captured in a CUDA graph and replayed.  Each layer keeps its own state,
    so a step reads several times the L2 capacity and no layer's state is
    still cached when its turn comes again."""
    import torch

    import sliding_window_softmax_gb300 as nha
    from sliding_window_softmax_gb300.synthetic import DECODE_1P3B, make_decode_layer

    dw = DECODE_1P3B
    if layers_override:
        dw = dataclasses.replace(dw, layers=layers_override,
                                 name=dw.name.replace(f"{dw.layers} layers", f"{layers_override} layers"))
    if batch_override:
        dw = dataclasses.replace(dw, B=batch_override, name=dw.name.replace(f"B{dw.B} ", f"B{batch_override} "))
    layers = [make_decode_layer(dw, i, device=dev) for i in range(dw.layers)]
    outs = [torch.empty_like(x["q"]) for x, _ in layers]

    # each layer's launch follows another layer's, which writes none of its
    # state: the launches may stream their states in early (one layer alone
    # follows itself and may not)
    overlap = dw.layers > 1

    def step():
        for (x, st), o in zip(layers, outs):
            nha.nha_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], dw.t, dw.w, st, o=o, overlap=overlap)

    side = torch.cuda.Stream(device=dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()  # eager once: validates the arguments
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    n0 = nha.launch_count()
    with torch.cuda.graph(graph):
        step()
    captured = nha.launch_count() - n0
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    K = max(10, min(args.steps, 200))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in ev:
        a.record(stream)
        graph.replay()
        b.record(stream)
    torch.cuda.synchronize()
    step_ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    per_launch_s = step_ms / 1e3 / dw.layers
    peaks = load_peaks()
    nbytes = decode_bytes(dw)
    achieved = nbytes / per_launch_s / 1e9
    return {
        "workload": dw.name, "B": dw.B, "H": dw.H, "d": dw.d, "m": dw.m, "w": dw.w, "t": dw.t,
        "layers": dw.layers, "dtype": dw.dtype, "overlapped_launches": overlap,
        "tokens_per_s": dw.B / (step_ms / 1e3), "ms_per_token_step": step_ms,
        "us_per_layer": per_launch_s * 1e6, "launches_per_step": captured, "steps": K,
        "timing": "CUDA graph of the layers' launches, median of replays; state of all layers "
                  f"{dw.layers * nbytes / 2**30:.2f} GiB of algorithmic traffic per step, above the L2 capacity",
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic("decode_step", "decode"),
                     "kernel": "decode_step", "bytes_per_launch": nbytes, "peak_source": peaks["source"]},
    }


def run_nha(args, wl, wl_key):
    import torch
    import torch.distributed as dist

    import sliding_window_softmax_gb300 as nha
    from sliding_window_softmax_gb300.dist import max_over_ranks
    from sliding_window_softmax_gb300.synthetic import make_inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()

    x = make_inputs(wl)
    d = {n: t.to(dev) for n, t in x.items()}
    B, H, T, D = d["q"].shape
    o, lse = torch.empty_like(d["q"]), torch.empty((B, H, T), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(d["q"]) for _ in range(3))
    dla = torch.empty_like(d["log_alpha"])
    wsf = torch.empty(max(1, nha.nha_workspace_bytes(B, H, T, D, wl.m, wl.w, wl.C, d["q"].dtype)),
                      dtype=torch.uint8, device=dev)
    # the backward reuses what the forward left in its workspace (chunk states,
    # rotated q and k): the saved-for-backward context of a training step
    wsb = torch.empty(max(1, nha.nha_workspace_bytes(B, H, T, D, wl.m, wl.w, wl.C, d["q"].dtype,
                                                     backward=True, reuse_forward=True)),
                      dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step(fwd_evt=None):
        nha.nha_forward(d["q"], d["k"], d["v"], d["log_alpha"], wl.w, wl.C, o=o, lse=lse,
                        workspace=wsf, stream=stream)
        if fwd_evt is not None:
            fwd_evt.record(stream)
        if wl.backward:
            nha.nha_backward(d["q"], d["k"], d["v"], d["log_alpha"], o, lse, d["dout"], wl.w,
                             wl.C, dq=dq, dk=dk, dv=dv, dlog_alpha=dla, workspace=wsb,
                             stream=stream, fwd_workspace=wsf)

    clk = ClockSampler(local).__enter__()
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    t_start = time.time()
    n0 = nha.launch_count()
    enq = []  # host time spent enqueuing each step (argument checks, tensor maps, launches)
    for i in range(K):
        flush.zero_()  # L2 flush between timed steps, outside the step's events
        ev[i][0].record(stream)
        h0 = time.perf_counter()
        step(ev[i][1])
        enq.append(time.perf_counter() - h0)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    launches = nha.launch_count() - n0
    clk.mark(t_start, time.time())
    clk.__exit__(None, None, None)
    wall = time.perf_counter() - wall0
    barrier()

    # per-kernel CUDA-event times, in a separate pass (the profiling session
    # records two extra events around every launch, so the headline steps
    # above run without it)
    KP = max(3, min(K, 20))
    nha.profile_begin()
    for i in range(KP):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    prof = nha.profile_end()
    step_ms = [ev[i][0].elapsed_time(ev[i][2]) for i in range(K)]
    fwd_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    ms = statistics.mean(step_ms)
    ms_fwd = statistics.mean(fwd_ms)
    ms_med = statistics.median(step_ms)
    ms, ms_fwd, ms_med = max_over_ranks([ms, ms_fwd, ms_med], device=dev)

    # the same steps back to back without the L2 flush (inputs may stay in L2)
    K2 = max(3, min(K, 100))
    ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K2)]
    barrier()
    torch.cuda.synchronize()
    for i in range(K2):
        ev2[i][0].record(stream)
        step(ev2[i][1])
        ev2[i][2].record(stream)
    torch.cuda.synchronize()
    ms_unfl = statistics.median(ev2[i][0].elapsed_time(ev2[i][2]) for i in range(K2))
    ms_unfl_fwd = statistics.median(ev2[i][0].elapsed_time(ev2[i][1]) for i in range(K2))
    ms_unfl, ms_unfl_fwd = max_over_ranks([ms_unfl, ms_unfl_fwd], device=dev)

    # ---- end to end through the public API with pinned host buffers
    hin = {n: t.pin_memory() for n, t in x.items()}
    hout = {n: torch.empty(t.shape, dtype=t.dtype).pin_memory()
            for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv, dlog_alpha=dla).items()}
    h2d = sum(t.numel() * t.element_size() for n, t in hin.items()
              if wl.backward or n != "dout")
    d2h = sum(t.numel() * t.element_size() for n, t in hout.items()
              if wl.backward or n in ("o", "lse"))
    outs = dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv, dlog_alpha=dla)

    def e2e_step():
        for n, t in hin.items():
            if wl.backward or n != "dout":
                d[n].copy_(t, non_blocking=True)
        step()
        for n, t in hout.items():
            if wl.backward or n in ("o", "lse"):
                t.copy_(outs[n], non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    E = max(3, min(K, 10))
    e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(E)]
    barrier()
    for i in range(E):
        flush.zero_()
        e_ev[i][0].record(stream)
        e2e_step()
        e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = statistics.mean(a.elapsed_time(b) for a, b in e_ev)
    (e2e_serial_ms,) = max_over_ranks([e2e_serial_ms], device=dev)

    # The same through a stream of steps as a training loop runs them: step i's
    # inputs are copied in on one copy stream while step i - 1 computes, and
    # its results copied out on another while step i + 1 computes (device
    # inputs and outputs double-buffered; every step still moves all of its
    # bytes across the host link, all inside the timed region, and the L2 is
    # flushed before every step's kernels).
    sets = [(d, outs)] + [({n: torch.empty_like(t) for n, t in d.items()},
                           {n: torch.empty_like(t) for n, t in outs.items()})]
    cin, cout = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def run_pipelined(n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_done = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        cin.wait_event(t0)
        cout.wait_event(t0)

        def copy_in(i):
            din, _ = sets[i % 2]
            with torch.cuda.stream(cin):
                if i >= 2:
                    cin.wait_event(ev_done[i - 2])  # step i - 2 no longer reads these inputs
                for nm, t in hin.items():
                    if wl.backward or nm != "dout":
                        din[nm].copy_(t, non_blocking=True)
                ev_in[i].record(cin)

        copy_in(0)
        for i in range(n):
            din, dout_set = sets[i % 2]
            if i + 1 < n:
                copy_in(i + 1)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])  # step i - 2's results copied out
            flush.zero_()
            nha.nha_forward(din["q"], din["k"], din["v"], din["log_alpha"], wl.w, wl.C, o=dout_set["o"],
                            lse=dout_set["lse"], workspace=wsf, stream=stream)
            if wl.backward:
                nha.nha_backward(din["q"], din["k"], din["v"], din["log_alpha"], dout_set["o"],
                                 dout_set["lse"], din["dout"], wl.w, wl.C, dq=dout_set["dq"],
                                 dk=dout_set["dk"], dv=dout_set["dv"], dlog_alpha=dout_set["dlog_alpha"],
                                 workspace=wsb, stream=stream, fwd_workspace=wsf)
            ev_done[i].record(stream)
            with torch.cuda.stream(cout):
                cout.wait_event(ev_done[i])
                for nm, t in hout.items():
                    if wl.backward or nm in ("o", "lse"):
                        t.copy_(dout_set[nm], non_blocking=True)
                ev_out[i].record(cout)
        stream.wait_event(ev_out[n - 1])
        stream.wait_event(ev_in[n - 1])
        t1.record(stream)
        return t0, t1

    run_pipelined(3)
    torch.cuda.synchronize()
    barrier()
    EP = max(3, min(K, 20))
    t0, t1 = run_pipelined(EP)
    torch.cuda.synchronize()
    e2e_ms = t0.elapsed_time(t1) / EP
    (e2e_ms,) = max_over_ranks([e2e_ms], device=dev)

    decode = None if args.no_decode else run_decode(args, dev, stream)

    if rank == 0:
        model = work_model(wl)
        peaks = load_peaks()
        tokens = world * B * T
        value = tokens / (ms / 1e3)
        # dominant kernel: the largest measured time per step among all the
        # library's kernels (the side stream's included)
        name, (cnt, tot) = max(prof.items(), key=lambda kv: kv[1][1])
        per_launch_ms = tot / cnt
        kflops, kbytes = model["kernels"].get(name, (0.0, 0.0))
        total_prof = sum(v[1] for v in prof.values())
        t_roof_fwd, _ = step_roofline(model, peaks, ms_fwd, backward=False)
        # the roofline object covers the whole step: the algorithmic bytes and
        # flops of one fwd (+ bwd) pass over the measured step time, so its frac
        # is step_roofline_frac
        t_roof_step, roof = step_roofline(model, peaks, ms, backward=wl.backward)
        s_bytes = roof["algorithmic_bytes"]
        launches_per_step = {k: c / KP for k, (c, _) in prof.items()}
        traffic = step_traffic(launches_per_step, wl_key)
        roof["traffic"] = traffic
        roof["traffic_over_algorithmic"] = None if traffic is None else traffic / s_bytes
        roof["peak_source"] = peaks["source"]
        roof["dominant_kernel"] = {
            "kernel": name, "ms_per_launch": per_launch_ms, "share": tot / total_prof,
            "model_bytes": kbytes, "model_flops": kflops,
            "model_gbs": kbytes / (per_launch_ms / 1e3) / 1e9,
            "model_tflops": kflops / (per_launch_ms / 1e3) / 1e12,
            "traffic": ncu_traffic(name, wl_key)}
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if wl.dtype == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": wl.name, "B": B, "H": H, "T": T, "d": D, "m": wl.m, "w": wl.w,
                       "C": wl.C, "pass": "fwd+bwd" if wl.backward else "fwd",
                       "l2": "flushed between timed steps (512 MB write)",
                       "parallelism": f"replicas x{world} over B*H (no collective)"},
            "fwd": {"ms": ms_fwd, "tokens_per_s": tokens / (ms_fwd / 1e3),
                    "roofline_frac": t_roof_fwd / (ms_fwd / 1e3)},
            "step_roofline_frac": t_roof_step / (ms / 1e3),
            "median_ms_per_step": ms_med,
            "unflushed": {"ms_per_step": ms_unfl, "fwd_ms": ms_unfl_fwd, "steps": K2,
                          "note": "median of back-to-back steps without the L2 flush"},
            "roofline": roof,
            "kernels": {k: {"launches_per_step": c / KP, "ms_per_launch": t / c, "share": t / total_prof,
                            "traffic": ncu_traffic(k, wl_key)}
                        for k, (c, t) in sorted(prof.items(), key=lambda kv: -kv[1][1])},
            "kernels_note": f"CUDA-event times per kernel from a separate pass of {KP} steps",
            "gpu_launches": int(launches),
            "e2e": {"value": tokens / (e2e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "ms_per_step": e2e_ms, "steps": EP,
                    "mode": "pipelined: step i's host-to-device copy beside step i - 1's kernels, its "
                            "device-to-host copy beside step i + 1's (double-buffered device tensors)",
                    "serial": {"value": tokens / (e2e_serial_ms / 1e3), "ms_per_step": e2e_serial_ms,
                               "note": "copy in, step, copy out on one stream, one step at a time"}},
            "clocks": clk.summary(),
            "wall_s_timed_region": wall,
            # median over the first steps: once the launch queue is full, an enqueue
            # waits for the device and the time measures the device instead
            "host_enqueue_ms_per_step": 1e3 * statistics.median(enq[:20]),
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(wl)
            if decode is not None:
                from sliding_window_softmax_gb300.synthetic import DECODE_1P3B

                decode["cpu_baseline"] = decode_cpu_baseline(DECODE_1P3B)
        if decode is not None:
            line["decode"] = decode
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="1.3B")
    ap.add_argument("--impl", default="nha", choices=["nha", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode-step measurement")
    ap.add_argument("--decode-only", action="store_true",
                    help="run only the decode-step measurement (one GPU) and print its object")
    ap.add_argument("--decode-layers", type=int, default=0, help="layers of the decode run (default 24)")
    ap.add_argument("--decode-batch", type=int, default=0, help="sequences of the decode run (default 16)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    wls = workloads()
    if args.workload not in wls:
        raise SystemExit(f"unknown workload {args.workload}; choose from {sorted(wls)}")
    wl = wls[args.workload]
    if args.decode_only:
        import torch

        torch.cuda.set_device(0)
        print(json.dumps(run_decode(args, torch.device("cuda", 0), torch.cuda.current_stream(),
                                    args.decode_layers or None, args.decode_batch or None)), flush=True)
        return
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_nha(args, wl, args.workload)


if __name__ == "__main__":
    main()
