#!/usr/bin/env python
"""Benchmark of the B300 Mixtral sparse-MoE layer (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                    [--workloads decode,prefill,...] [--no-cpu-baseline]

A step is one pass of the whole hot path - router, dispatch, grouped gate/up
GEMM with SwiGLU, grouped down GEMM, combine (and the RMSNorm prologue and
residual for the block workload) - over one batch of synthetic tokens, run
through the library's C ABI with every input already in HBM.  The headline
workload is Mixtral-shape decode (T=16); the other Mixtral workloads are
timed in the same run and reported under "workloads".

Timing: W untimed warm-up steps, then exactly K steps, each bracketed by CUDA
events on the launching stream, with an L2 flush (a 256 MiB write) between
steps outside the events; a barrier and a device synchronise on both sides.
Per-kernel events inside the step give the dominant kernel's roofline.
"e2e" runs moe_forward_host with pinned host activations (host->device copy,
the layer, device->host copy, synchronise) timed by the host clock.

Accuracy (part of the CPU-baseline leg, after the timed steps, skipped with
--no-cpu-baseline): every forward workload's routing and a sample of its
outputs are scored by the fp64 CPU oracle - near-tie tokens, those routed
differently, clear tokens routed differently (0), rel-L2 - and the line's
"targets" states the layer roofline fractions against the ones required.

Multi-GPU (torchrun): replicas only - every rank runs the same workload on its
own GPU with no collective on the data path; value = tokens of all ranks /
max over ranks of the timed region.  ``--impl reference`` times the fp64 CPU
oracle on the host cores (rank 0 only) on a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import moe_workloads as mw  # noqa: E402

METRIC = "MoE-layer tokens/s (Mixtral 4096/14336, E8 k2, bf16) + % of roofline"
HEADLINE = "decode"
ALL_BENCH = ["decode", "prefill", "skewed", "skewed_zero", "block", "decode_w8", "prefill_w8", "prefill_bwd"]
L2_FLUSH_BYTES = 256 << 20
KERNELS_PER_STEP = {False: 6, True: 7}  # router, rank, gather, gate_up, down, combine (+ rmsnorm)


# ---------------------------------------------------------------- peaks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ---------------------------------------------------------------- work model
def algorithmic(wl, counts):
    """Algorithmic FLOPs and bytes of one layer call, and of its gate/up GEMM.

    FLOP/token = k*6*d*F + 2*d*E.  Bytes = every used expert's three matrices
    + the gate + x in + out (+ gamma); permuted intermediates do not count.
    """
    T, d, F, E, k = wl.T, wl.d, wl.F, wl.E, wl.k
    used = int(sum(1 for c in counts if c > 0))
    flops = T * (k * 6 * d * F + 2 * d * E)
    if wl.w8:  # int8 codes + one fp32 scale per row
        expert_bytes, gu_expert_bytes = 3 * d * F + (2 * F + d) * 4, 2 * d * F + 2 * F * 4
    else:
        expert_bytes, gu_expert_bytes = 3 * d * F * 2, 2 * d * F * 2
    nbytes = used * expert_bytes + d * E * 2 + 2 * T * d * 2 + (d * 2 if wl.block else 0)
    gu_flops = T * k * 4 * d * F
    gu_bytes = used * gu_expert_bytes
    return flops, nbytes, gu_flops, gu_bytes


# ---------------------------------------------------------------- ncu traffic
def kernel_source_hash():
    h = hashlib.sha256()
    for name in ("ffn_tc.cu", "ffn_w8_wide.cu", "widen.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "sparse_mixture_experts_50_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """DRAM bytes (read + write) per gate/up launch from the committed ncu
    summary profiles/gemm_<workload>.md, if it was taken on the current
    kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"gemm_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_src = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_launch_full:\s*([0-9.e+]+)", text)
    if not (m_src and m_b) or m_src.group(1) != kernel_source_hash():
        return None
    return float(m_b.group(1))


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- the layer
class Layer:
    """Device-resident inputs, scratch and output of one workload.  step()
    runs the whole hot path as one moe_forward_ex call through the C ABI;
    with `ev` (5 CUDA events) the library records them before the router,
    after dispatch, after gate/up, after down and after combine.  The
    routing and intermediates are views into the scratch."""

    def __init__(self, wl, tensors, device):
        from sparse_mixture_experts_50_b300 import binding as B
        self.B = B
        self.wl = wl
        T, d, F, E, k = wl.T, wl.d, wl.F, wl.E, wl.k
        dev = torch.device(device)
        g = {n: v.to(dev, non_blocking=False) for n, v in tensors.items()}
        self.x, self.Wg, self.W1, self.W3, self.W2 = g["x"], g["Wg"], g["W1"], g["W3"], g["W2"]
        self.gamma = g.get("gamma")
        self.w8 = None
        if wl.w8:
            # Weight preparation (once, outside any timed region): per-row
            # int8 codes and fp32 scales on the GPU; the bf16 copies go.
            self.W1q, self.W1s = B.moe_quantize_int8(self.W1)
            self.W3q, self.W3s = B.moe_quantize_int8(self.W3)
            self.W2q, self.W2s = B.moe_quantize_int8(self.W2)
            self.W1 = self.W3 = self.W2 = None
            self.w8 = (self.W1q, self.W1s, self.W3q, self.W3s, self.W2q, self.W2s)
        dtype = B.MOE_DTYPE_BF16 if wl.dtype == "bf16" else B.MOE_DTYPE_F32
        self.ws = B.workspace(T, d, F, E, k, dtype, device=dev)
        v = B.workspace_views(self.ws, T, d, F, E, k, dtype)
        self.idx, self.w, self.counts, self.offsets = v["idx"], v["w"], v["counts"], v["offsets"]
        self.row_src, self.slot_pos, self.x_perm, self.h, self.y = (v["row_src"], v["slot_pos"], v["x_perm"], v["h"],
                                                                    v["y"])
        self.xn = v["xn"] if wl.block else None
        self.out = torch.empty((T, d), dtype=wl.torch_dtype, device=dev)

    def step(self, ev=None):
        wl = self.wl
        self.B.moe_forward_ex(self.x, self.Wg, wl.k, self.ws, W1=self.W1, W3=self.W3, W2=self.W2, gamma=self.gamma,
                              eps=wl.eps, w8=self.w8, out=self.out, events=ev)
        return self.out


class BwdLayer:
    """The backward of one workload.  The training forward
    (moe_forward_train_ws, which keeps the SwiGLU's local derivatives p and
    q) runs once at set-up with caller scratch (`saved`); step() runs
    moe_backward_ws through the C ABI into preallocated gradients;
    forward_step() re-runs that training forward."""

    def __init__(self, wl, tensors, device):
        from sparse_mixture_experts_50_b300 import binding as B
        self.B = B
        self.wl = wl
        T, d, F, E, k = wl.T, wl.d, wl.F, wl.E, wl.k
        g = {n: v.to(device) for n, v in tensors.items()}
        self.x, self.Wg, self.W1, self.W3, self.W2, self.dout = g["x"], g["Wg"], g["W1"], g["W3"], g["W2"], g["dout"]
        self.saved = B.workspace(T, d, F, E, k, B.MOE_DTYPE_BF16, device=device)
        self.out = torch.empty_like(self.x)
        self.keep = B.keep_buffer(T, F, k, device=device)
        self.forward_step()
        self.ws = torch.empty(B.moe_backward_workspace_bytes(T, d, F, E, k), dtype=torch.uint8, device=device)
        self.grads = B._grads(self.x, self.Wg, self.W1, self.W3, self.W2, None)

    def forward_step(self):
        self.B.moe_forward_train_ws(self.x, self.Wg, self.W1, self.W3, self.W2, self.wl.k, self.saved,
                                    keep=self.keep, out=self.out)

    def step(self, ev=None):
        if ev is not None:
            ev[0].record()
        self.B.moe_backward_ws(self.dout, self.x, self.Wg, self.W1, self.W3, self.W2, self.wl.k, self.saved, self.ws,
                               self.grads, keep=self.keep)
        if ev is not None:
            for e in ev[1:]:
                e.record()
        return self.grads


def make_tensors(wl, shared):
    """CPU tensors of a workload; the expert weights (which do not depend on
    T or the gate bias) are drawn once and shared across workloads."""
    key = (wl.d, wl.F, wl.E, wl.dtype, wl.init)
    if key not in shared:
        shared[key] = mw.make_inputs(wl, only=("W1", "W3", "W2"))
    rest = mw.make_inputs(wl, only=("x", "Wg", "gamma", "dout"))
    return {**rest, **shared[key]}


def time_layer(layer, steps, warmup, flush, dist_on):
    """K timed steps, each bracketed by CUDA events on the launching stream
    (an L2 flush between steps, outside the events), then up to 10 more steps
    with events recorded inside the call between its kernels, for the
    per-kernel split.  Only the first pass gives the step time: an event recorded between
    two kernels ends the overlap of the second kernel's launch and set-up with
    the first's tail (programmatic dependent launch)."""
    outer = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    for _ in range(warmup):
        layer.step()
        flush.zero_()
    torch.cuda.synchronize()
    if dist_on:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        outer[i][0].record()
        layer.step()
        outer[i][1].record()
        flush.zero_()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if dist_on:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in outer]
    # A short second pass: the dense workloads run at the power cap, and
    # every extra step heats the part for the workloads timed after it.
    evs = evs[:min(steps, 10)]
    for e in evs:
        layer.step(e)
        flush.zero_()
    torch.cuda.synchronize()
    parts = {
        "router_dispatch": [e[0].elapsed_time(e[1]) for e in evs],
        "gate_up": [e[1].elapsed_time(e[2]) for e in evs],
        "down": [e[2].elapsed_time(e[3]) for e in evs],
        "combine": [e[3].elapsed_time(e[4]) for e in evs],
    }
    return step_ms, parts, wall


def bench_backward(name, shared, args, device, peaks, dist_on):
    """The backward leg: T / (mean backward time); its tensor roofline uses
    the algorithmic 12*d*F FLOP per routed row (dh 2, dx 4, dW2 2, dW1+dW3 4;
    the forward's p and q, or a recomputation of a and b, are implementation
    work and not counted)."""
    wl = mw.get(name)
    layer = BwdLayer(wl, make_tensors(wl, shared), device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    layer.step()
    status = layer.B.moe_get_device_status(reset=True)
    if status != 0:
        raise RuntimeError(f"{name}: device status {status} after the first step")
    step_ms, _, wall = time_layer(layer, args.steps, args.warmup, flush, dist_on)
    status = layer.B.moe_get_device_status(reset=True)
    if status != 0:
        raise RuntimeError(f"{name}: device status {status} after the timed steps")
    ms = sum(step_ms) / len(step_ms)
    flops = wl.T * wl.k * 12 * wl.d * wl.F + wl.T * wl.k * 4 * wl.d * wl.E
    achieved = flops / (ms * 1e-3) / 1e12
    # The training forward that feeds it (p and q kept), timed the same way.
    fwd_ms = []
    for i in range(args.warmup + args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        layer.forward_step()
        b.record()
        flush.zero_()
        if i >= args.warmup:
            fwd_ms.append((a, b))
    torch.cuda.synchronize()
    fwd = sum(a.elapsed_time(b) for a, b in fwd_ms) / len(fwd_ms)
    return {
        "workload": name, "T": wl.T, "tokens_per_s": wl.T / (ms * 1e-3), "ms_per_step": ms,
        "ms_per_step_median": statistics.median(step_ms), "train_forward_ms": fwd,
        "layer_roofline_frac": achieved / peaks["bf16_tflops"], "bound": "tensor",
        "layer_roofline_frac_of_nominal": of_nominal("tensor", achieved),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"], "frac_of_nominal": of_nominal("tensor", achieved),
                     "kernel": "whole backward (moe_backward_ws)", "algorithmic_per_launch": flops, "traffic": None},
        "wall_s": wall,
    }, layer


# Nominal B300 figures, reported beside the fractions of the measured peaks:
# HBM3e ~8 TB/s and dense bf16 2.25 PFLOP/s.
NOMINAL = {"hbm_gbs": 8000.0, "bf16_tflops": 2250.0}


def of_nominal(bound, achieved):
    """achieved (GB/s for an HBM-bound kernel, TFLOP/s for a tensor-bound
    one) as a fraction of the nominal peak."""
    return achieved / (NOMINAL["hbm_gbs"] if bound == "hbm" else NOMINAL["bf16_tflops"])


def bench_workload(name, shared, args, device, peaks, dist_on):
    wl = mw.get(name)
    if wl.bwd:
        return bench_backward(name, shared, args, device, peaks, dist_on)
    layer = Layer(wl, make_tensors(wl, shared), device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    layer.step()
    status = layer.B.moe_get_device_status(reset=True)
    if status != 0:
        raise RuntimeError(f"{name}: device status {status} after the first step")
    counts = layer.counts.cpu().tolist()
    step_ms, parts, wall = time_layer(layer, args.steps, args.warmup, flush, dist_on)
    status = layer.B.moe_get_device_status(reset=True)
    if status != 0:
        raise RuntimeError(f"{name}: device status {status} after the timed steps")
    ms = sum(step_ms) / len(step_ms)
    flops, nbytes, gu_flops, gu_bytes = algorithmic(wl, counts)
    t_roof = max(flops / (peaks["bf16_tflops"] * 1e12), nbytes / (peaks["hbm_gbs"] * 1e9))
    t_nominal = max(flops / (NOMINAL["bf16_tflops"] * 1e12), nbytes / (NOMINAL["hbm_gbs"] * 1e9))
    bound = "hbm" if nbytes / (peaks["hbm_gbs"] * 1e9) > flops / (peaks["bf16_tflops"] * 1e12) else "tensor"
    gu_ms = sum(parts["gate_up"]) / len(parts["gate_up"])
    if bound == "hbm":
        achieved, peak, unit = gu_bytes / (gu_ms * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = gu_flops / (gu_ms * 1e-3) / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    res = {
        "workload": name, "T": wl.T, "tokens_per_s": wl.T / (ms * 1e-3), "ms_per_step": ms,
        "ms_per_step_median": statistics.median(step_ms),
        "layer_roofline_frac": t_roof / (ms * 1e-3), "bound": bound,
        "layer_roofline_frac_of_nominal": t_nominal / (ms * 1e-3),
        "layer_roofline_tokens_per_s": wl.T / t_roof,
        "kernel_ms": {p: sum(v) / len(v) for p, v in parts.items()},
        "expert_counts": counts,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                     "frac_of_nominal": of_nominal(bound, achieved),
                     "kernel": "grouped_gemm_tc_kernel<gate_up+SwiGLU%s>" % (", int8 weights" if wl.w8 else ""),
                     "algorithmic_per_launch": gu_bytes if bound == "hbm" else gu_flops,
                     "traffic": ncu_traffic(name)},
        "wall_s": wall,
    }
    return res, layer


def e2e_leg(layer, steps, warmup):
    """moe_forward_host with pinned host activations, host-clock timed."""
    B, wl = layer.B, layer.wl
    x_host = layer.x.cpu().pin_memory()
    out_host = torch.empty_like(x_host).pin_memory()
    ws = B.workspace(wl.T, wl.d, wl.F, wl.E, wl.k, B.MOE_DTYPE_BF16, device=layer.x.device, host=True)
    for _ in range(warmup):
        B.moe_forward_host(x_host, layer.Wg, layer.W1, layer.W3, layer.W2, wl.k, ws, out_host)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        B.moe_forward_host(x_host, layer.Wg, layer.W1, layer.W3, layer.W2, wl.k, ws, out_host)
    el = time.perf_counter() - t0
    nb = wl.T * wl.d * 2
    return {"value": wl.T * steps / el, "unit": "tokens/s", "h2d_bytes_per_step": nb, "d2h_bytes_per_step": nb}


def cpu_cores():
    try:
        import threadpoolctl
        return int(max((i.get("num_threads", 1) for i in threadpoolctl.threadpool_info()), default=1))
    except Exception:  # pragma: no cover
        return os.cpu_count() or 1


def oracle_time(name, tensors, tokens):
    """Seconds the fp64 CPU oracle takes for the layer on `tokens` rows."""
    import oracle.moe_oracle as O
    wl = mw.get(name)
    t = tensors
    x = t["x"][tokens]
    t0 = time.perf_counter()
    if wl.block:
        O.block_forward(x, t["gamma"], wl.eps, t["Wg"], t["W1"], t["W3"], t["W2"], wl.k)
    else:
        O.moe_forward(x, t["Wg"], t["W1"], t["W3"], t["W2"], wl.k)
    return time.perf_counter() - t0


def cpu_baseline(name, tensors, reps=3):
    """The oracle, as it stands, on the whole workload batch `reps` times
    (Mixtral decode: 16 tokens, ~4 s each on 8 cores)."""
    wl = mw.get(name)
    n = min(wl.T, 16)
    times = [oracle_time(name, tensors, slice(0, n)) for _ in range(reps)]
    el = statistics.median(times)
    return {"value": n / el, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{name}: tokens 0-{n - 1} of {wl.T}, whole layer in fp64 (numpy), median of {reps} runs, "
                      f"{el:.2f} s each"}


NEAR_TIE = 1e-3          # oracle logit gap below which a token's routing may legitimately differ
ACCURACY_SAMPLE = 64     # seeded tokens per workload whose outputs the oracle scores
# Layer roofline fractions the layer must reach (bound, target).
TARGETS = {"decode": ("hbm", 0.70), "skewed": ("tensor", 0.60), "skewed_zero": ("tensor", 0.60),
           "block": ("tensor", 0.60)}
_CODES = {}              # the oracle's int8 codes of an expert matrix, by (tensor id, expert)


class _OracleInt8Experts:
    """An [E, rows, cols] expert tensor as the int8 layer uses it: each
    expert quantised by the oracle and dequantised when indexed (one expert
    at a time; the codes are cached, the fp64 values are not)."""

    def __init__(self, W):
        self.W = W
        self.shape = tuple(W.shape)

    def __getitem__(self, e):
        import oracle.moe_oracle as O
        key = (id(self.W), int(e))
        if key not in _CODES:
            _CODES[key] = O.quantize_int8_rows(self.W[e])
        return O.dequantize_int8_rows(*_CODES[key])


def accuracy(layer, tensors, sample=ACCURACY_SAMPLE):
    """The GPU result of one workload scored by the fp64 oracle, after the
    timed steps (part of the CPU-baseline leg; nothing here is timed).

    Routing, on every token: the oracle's fp64 logits decide which tokens are
    near ties (a gap below 1e-3 among the k+1 largest logits; in the block
    form widened by the logit change of the rare normalised element the two
    sides round apart); counted are those tokens, those of them the GPU routed
    differently, and clear tokens the GPU routed differently (must be 0).
    Output: rel-L2 of the layer output over a seeded sample of tokens plus
    every near-tie token, against the oracle run on the GPU's routing where a
    near tie went the other way (block form: also of the MoE delta alone)."""
    import numpy as np

    import oracle.moe_oracle as O
    wl = layer.wl
    t0 = time.perf_counter()
    if wl.block:
        xin = O.block_normed_input(tensors["x"], tensors["gamma"], wl.eps)
        dl = (layer.xn.cpu().double().numpy() - xin) @ O.f64(tensors["Wg"]).T
        extra = np.max(np.abs(dl), axis=1)
    else:
        xin = O.f64(tensors["x"])
        extra = np.zeros(wl.T)
    ora_w, ora_idx, logits = O.router(xin, tensors["Wg"], wl.k)
    gi = layer.idx.cpu().numpy().astype(np.int64)
    top = -np.sort(-logits, axis=1)[:, : wl.k + 1]
    near = np.any(top[:, :-1] - top[:, 1:] < (NEAR_TIE + 2.0 * extra)[:, None], axis=1)
    differ = np.any(gi != ora_idx, axis=1)
    rng = np.random.default_rng(1)
    toks = set(rng.choice(wl.T, size=min(sample, wl.T), replace=False).tolist()) | set(np.nonzero(near)[0].tolist())
    s = np.array(sorted(toks))
    w_eff, idx_eff = ora_w[s].copy(), ora_idx[s].copy()
    for i, t in enumerate(s):
        if near[t] and differ[t]:
            idx_eff[i] = gi[t]
            w_eff[i] = O.softmax(logits[t, gi[t]])
    if wl.w8:
        W1, W3, W2 = (_OracleInt8Experts(tensors[n]) for n in ("W1", "W3", "W2"))
    else:
        W1, W3, W2 = tensors["W1"], tensors["W3"], tensors["W2"]
    t1 = time.perf_counter()
    delta = O.moe_forward_with_routing(xin[s], W1, W3, W2, w_eff, idx_eff)
    oracle_s = time.perf_counter() - t1

    def rel(got, ref):
        return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))

    out = layer.out.cpu().double().numpy()[s]
    res = {"near_tie_tokens": int(near.sum()), "near_tie_routed_differently": int((near & differ).sum()),
           "clear_tokens_routed_differently": int((~near & differ).sum()),
           "rel_l2": rel(out, delta + (O.f64(tensors["x"][s]) if wl.block else 0.0)),
           "rel_l2_bound": 5e-3, "scored_tokens": int(s.size)}
    if wl.block:
        gd = layer.B.moe_combine(layer.y, layer.slot_pos, layer.w, wl.T)
        res["rel_l2_moe_delta"] = rel(gd.cpu().double().numpy()[s], delta)
    res["oracle_tokens_per_s"] = s.size / oracle_s
    res["wall_s"] = time.perf_counter() - t0
    return res


def targets_of(results):
    """The layer roofline fractions the layer is held to, from this run."""
    out = {}
    for name, (bound, target) in TARGETS.items():
        r = results.get(name)
        if r is None:
            continue
        out[name] = {"bound": bound, "layer_frac": round(r["layer_roofline_frac"], 4), "target": target,
                     "met": bool(r["bound"] == bound and r["layer_roofline_frac"] >= target)}
    return out


def job_throughput(tokens_local, t_local, dist_on, device):
    """Whole-job tokens/s: the tokens every rank processed over the slowest
    rank's timed region (replicas: no collective touches the data path; this
    all-reduce of two numbers is control only)."""
    if not dist_on:
        return tokens_local / t_local, t_local
    import torch.distributed as dist
    t = torch.tensor([t_local], dtype=torch.float64, device=device)
    n = torch.tensor([tokens_local], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(n.item()) / float(t.item()), float(t.item())


def config_of(name, n_gpus):
    wl = mw.get(name)
    return {"workload": f"{name}: T={wl.T}, d={wl.d}, d_ff={wl.F}, E={wl.E}, top-{wl.k}, {wl.dtype}"
                        + (", int8 weight-only experts" if wl.w8 else "")
                        + (", RMSNorm + residual" if wl.block else "")
                        + (", skewed expert load" if wl.skew else ""),
            "T": wl.T, "d": wl.d, "d_ff": wl.F, "E": wl.E, "k": wl.k,
            "parallelism": f"replicas x{n_gpus}" if n_gpus > 1 else "single GPU",
            "l2": "flushed between timed steps (256 MiB write); expert weights (2.8 GB) also exceed L2"}


def ep_leg(args, name, world, rank, local):
    """The expert-parallel form of the layer (ExpertParallelMoE over NCCL):
    each of the `world` ranks holds E/world experts and its own batch of the
    workload's shape, and routes, exchanges, runs its experts and combines
    every step.  Host-clock timed (each step brings the exchange's counts to
    the host), barrier and device synchronise on both sides, slowest rank."""
    import torch.distributed as dist
    from sparse_mixture_experts_50_b300.expert_parallel import ExpertParallelMoE, TorchComm
    wl = mw.get(name)
    if wl.w8 or wl.bwd or wl.block or wl.dtype != "bf16" or wl.E % world:
        raise SystemExit(f"--expert-parallel runs a plain bf16 forward workload with E divisible by {world}")
    device = f"cuda:{local}"
    t = mw.make_inputs(wl, x_seed=1000 + rank)
    El = wl.E // world
    mine = slice(rank * El, (rank + 1) * El)
    g = {"x": t["x"].to(device), "Wg": t["Wg"].to(device)}
    for n in ("W1", "W3", "W2"):
        g[n] = t[n][mine].contiguous().to(device)
    del t
    layer = ExpertParallelMoE(g["Wg"], g["W1"], g["W3"], g["W2"], wl.k, TorchComm())
    for _ in range(args.warmup):
        layer.forward(g["x"])
    if layer.B.moe_get_device_status(reset=True) != 0:
        raise RuntimeError("expert-parallel: device status after the warm-up steps")
    clocks = ClockSampler(local)
    clocks.start()
    dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        layer.forward(g["x"])
    torch.cuda.synchronize()
    dist.barrier()
    el = time.perf_counter() - t0
    clk = clocks.stop()
    value, t_max = job_throughput(wl.T * args.steps, el, True, device)
    ms = t_max / args.steps * 1e3
    peaks = load_peaks()
    # Each rank streams its own experts' weights once per step (decode: all of them are used).
    local_bytes = El * 3 * wl.d * wl.F * 2
    achieved = local_bytes / (ms * 1e-3) / 1e9
    return {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**config_of(name, world),
                   "parallelism": f"expert-parallel x{world}: {El} experts per rank, NCCL all-to-all of counts and rows",
                   "l2": "not flushed (each step's exchange synchronises with the host)"},
        "impl": "native",
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                     "kernel": "whole expert-parallel step (this rank's expert weights per step time)"},
        "e2e": None, "cpu_baseline": None,
        # router, dispatch + row copy, regroup, gate/up + down, ungroup, combine
        "gpu_launches": 8 * args.steps,
        "clocks": clk,
    }


def flush_c_stdio():
    """Flush the C library's stdout buffers (NCCL prints its version line
    through them), so that the JSON line printed next stays the last line."""
    try:
        import ctypes
        ctypes.CDLL(None).fflush(None)
    except Exception:  # pragma: no cover
        pass


def ensure_built():
    from sparse_mixture_experts_50_b300 import binding
    if not os.path.exists(binding.LIB_PATH):
        from sparse_mixture_experts_50_b300.build import build
        build()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workloads", default=",".join(ALL_BENCH))
    ap.add_argument("--headline", default=HEADLINE, choices=[n for n in ALL_BENCH if not (mw.get(n).w8 or mw.get(n).bwd)],
                    help="workload of the JSON line's value (default: Mixtral-shape decode)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--expert-parallel", action="store_true",
                    help="time the expert-parallel layer (E/N experts per rank, NCCL all-to-alls) on the headline "
                         "workload instead of the replica bench")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    head_name = args.headline
    names = [n for n in args.workloads.split(",") if n]
    if head_name not in names:
        names.insert(0, head_name)

    if args.impl == "reference":
        # The fp64 CPU oracle timed on the host cores (rank 0 only).  Each
        # step is a bounded sample: the whole batch when there are few steps,
        # else 2 tokens (cycling through the batch), so any --steps run ends
        # within minutes.  Warm-up steps evaluate 1 token.
        if rank != 0:
            return
        wl = mw.get(head_name)
        t0 = time.perf_counter()
        tensors = make_tensors(wl, {})
        per = wl.T if args.steps <= 4 else min(2, wl.T)
        for i in range(args.warmup):
            oracle_time(head_name, tensors, slice(i % wl.T, i % wl.T + 1))
        el = 0.0
        for i in range(args.steps):
            a = (i * per) % wl.T
            el += oracle_time(head_name, tensors, slice(a, min(a + per, wl.T)))
        v = per * args.steps / el
        base = {"value": v, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                "sample": f"{head_name}: {per} token(s) per step, whole layer in fp64 (numpy)"}
        line = {"metric": METRIC, "value": v, "unit": "tokens/s", "impl": "reference", "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {**config_of(head_name, 1), "l2": "not applicable (host CPU)"},
                "cpu_baseline": base,
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "wall_s": time.perf_counter() - t0}
        print(json.dumps(line), flush=True)
        return

    if args.expert_parallel:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA GPU for the native implementation")
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", str(29600 + os.getpid() % 1000))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", rank=rank, world_size=world, device_id=torch.device(f"cuda:{local}"))
        try:
            ensure_built()
            line = ep_leg(args, head_name, world, rank, local)
            if rank == 0:
                flush_c_stdio()
                print(json.dumps(line), flush=True)
        finally:
            dist.destroy_process_group()
        return

    dist_on = world > 1
    if dist_on:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for the native implementation")
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    ensure_built()
    peaks = load_peaks()
    shared = {}
    results = {}
    e2e = None
    for name in names:
        # SM clocks are sampled during every workload: the dense ones run at
        # the power cap, below the maximum clock.
        clocks = ClockSampler(local)
        clocks.start()
        res, layer = bench_workload(name, shared, args, device, peaks, dist_on)
        res["clocks"] = clocks.stop()
        if name == head_name and not args.no_e2e:
            # Right after the headline's device-timed steps, before the
            # oracle's accuracy pass (whose host threads would share the
            # cores with this host-timed loop) and the other workloads.
            e2e = e2e_leg(layer, args.steps, args.warmup)
        if rank == 0 and not args.no_cpu_baseline and not mw.get(name).bwd:
            res["accuracy"] = accuracy(layer, make_tensors(mw.get(name), shared))
        del layer
        results[name] = res
        torch.cuda.empty_cache()

    head = results[head_name]
    # Whole job: tokens of all ranks over the slowest rank's timed region.
    t_local = head["ms_per_step"] * args.steps * 1e-3
    value, _ = job_throughput(mw.get(head_name).T * args.steps, t_local, dist_on, device)

    if dist_on and e2e is not None:
        # every rank ran the same number of host-timed steps
        T = mw.get(head_name).T
        e2e["value"], _ = job_throughput(T * args.steps, T * args.steps / e2e["value"], True, device)

    if rank == 0:
        cpu = None
        if not (args.no_cpu_baseline or dist_on):
            cpu = cpu_baseline(head_name, make_tensors(mw.get(head_name), shared))
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(head_name, world), "impl": "native",
            "roofline": {k: head["roofline"][k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")},
            "roofline_detail": {**head["roofline"], "peak_source": peaks["source"],
                                "layer_frac": head["layer_roofline_frac"],
                                "layer_frac_of_nominal": head["layer_roofline_frac_of_nominal"],
                                "nominal_peaks": NOMINAL},
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": KERNELS_PER_STEP[mw.get(head_name).block] * args.steps,
            "clocks": head.get("clocks"),
            "targets": targets_of(results),
            "accuracy": {n: {k: r["accuracy"][k] for k in ("near_tie_tokens", "near_tie_routed_differently",
                                                           "clear_tokens_routed_differently", "rel_l2")}
                         for n, r in results.items() if "accuracy" in r},
            "workloads": {n: {**{k: v for k, v in r.items() if k != "clocks"},
                              "sm_mhz": (r.get("clocks") or {}).get("sm_mhz")} for n, r in results.items()},
        }
        flush_c_stdio()
        print(json.dumps(line), flush=True)
    if dist_on:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
