#!/usr/bin/env python
"""Benchmark of the FP8 W8A8 linear-layer hot path on GB300.

Prints ONE JSON line (rank 0). The headline workload is the decode-shaped
block-scaled layer: M in {1, 4, 16} tokens through the four Llama-8B-like
projections (N, K) in {(4096,4096), (6144,4096), (28672,4096), (4096,14336)},
over a stack of layers with distinct weights so that every pass streams far
more weight bytes than the 129 MB L2 holds. One step = for every M, layer and
projection: dynamic 1x128 activation quantization + block-scaled GEMM, through
fp8_block_linear (a quantization launch and a GEMM launch per call, chained
by programmatic dependent launch). The metric is HBM GB/s of algorithmic
bytes (weights and scales, BF16 activations in, codes and scales out, BF16
output).

The same run also times, as extra sections, the prefill-shaped GEMMs
(TFLOPS vs the FP8 tensor peak), the per-tensor layer, the MoE grouped GEMM
and the quantizers.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the CPU oracle (the plain C reference of what the path
computes) on the host cores, on a bounded sample of the same workload.
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

import numpy as np  # noqa: E402

import synth  # noqa: E402

SHAPES = synth.LLAMA8B_SHAPES
DECODE_M = synth.DECODE_M
LAYERS = 8
SUSTAINED_S = 2.0  # seconds of replays in the sustained leg of the headline
CPU_SAMPLE_S = 8.0  # seconds of oracle work in each cpu_baseline leg (all cores, one core)
REF_TOTAL_S = 90.0  # target length of a whole --impl reference run
METRIC = "FP8 block-scaled GEMM TFLOPS (% FP8 peak); decode-M HBM GB/s (% of peak)"
FP8_OVER_BF16 = 2.0  # nominal dense FP8 / BF16 tensor throughput ratio


# ------------------------------------------------------------ bytes/flops --

def gemm_bytes(M, N, K):
    """Algorithmic bytes of one block-scaled GEMM: Qw + Sw + Qa + Sa + Y."""
    nb, kg = -(-N // 128), K // 128
    return N * K + 4 * nb * kg + M * K + 4 * M * kg + 2 * M * N


def act_quant_bytes(M, K):
    """BF16 read + E4M3 write + one FP32 scale per 128 values."""
    return 2 * M * K + M * K + 4 * M * (K // 128)


def linear_bytes(M, N, K):
    """Algorithmic bytes of one W8A8 linear call from BF16 activations: Qw + Sw,
    X (BF16) in, activation codes + scales out, Y (BF16) out."""
    nb, kg = -(-N // 128), K // 128
    return N * K + 4 * nb * kg + 2 * M * K + M * K + 4 * M * kg + 2 * M * N


def tensor_gemm_bytes(M, N, K):
    return N * K + M * K + 2 * M * N + 8


def whole_job(step_units: float, ms_per_step: float, world: int, dist=None, device="cpu"):
    """Whole-job throughput over all ranks: units every rank processed per step,
    summed, over the slowest rank's step time. Returns (units per second,
    max ms per step). With world > 1 it all-reduces through `dist`."""
    if world > 1:
        import torch
        t = torch.tensor([ms_per_step], dtype=torch.float64, device=device)
        u = torch.tensor([step_units], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(u, op=dist.ReduceOp.SUM)
        ms_per_step, step_units = t.item(), u.item()
    return step_units / (ms_per_step * 1e-3), ms_per_step


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples with host timestamps."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        self.thread = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                self.samples.append((time.time(), float(parts[0]), float(parts[1]), parts[3:7]))
            except ValueError:
                pass

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        sel = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed"
        if len(sel) < 3:
            sel = self.samples
            window = "whole run"
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in sel for i, v in enumerate(s[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(s[1] for s in sel), "sm_max_mhz": max(s[2] for s in sel),
                "reasons": reasons, "samples": len(sel), "window": window}


def _gpu_id(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def _traffic(kernel: str, algorithmic_bytes_per_launch: float):
    """DRAM bytes (read + write) per launch of `kernel`, from the committed ncu
    captures in profiles/traffic.json: the captured DRAM/algorithmic ratio
    (averaged over the captured shapes) times this launch's algorithmic bytes.
    None if the kernel's sources changed since the capture (sha256 check)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        e = json.load(f).get(kernel)
    if not e:
        return None
    d = hashlib.sha256()
    for src in e["sources"]:
        full = os.path.join(ROOT, src)
        if not os.path.exists(full):
            return None
        d.update(open(full, "rb").read())
    if d.hexdigest() != e["sha256"]:
        return None
    ratios = [c["ratio"] for c in e["captures"].values()]
    return sum(ratios) / len(ratios) * algorithmic_bytes_per_launch


# ------------------------------------------------------------ graph utils --

class Timed:
    """A captured CUDA graph of one step, optionally with external timing
    events around selected kernels (graph event-record nodes)."""

    def __init__(self, torch, fn, n_marks=0):
        self.torch = torch
        self.marks = []
        self.ext = False
        if n_marks:
            try:
                self.marks = [(torch.cuda.Event(enable_timing=True, external=True),
                               torch.cuda.Event(enable_timing=True, external=True)) for _ in range(n_marks)]
                self.ext = True
            except TypeError:
                self.marks = []
        fn(None)  # eager warm-up outside capture (one-time attribute setup etc.)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(self.graph, stream=s):
                fn(self.marks if self.ext else None)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()

    def replay(self):
        self.graph.replay()

    def mark_ms(self):
        return [a.elapsed_time(b) for a, b in self.marks]


def time_steps(torch, step, steps, warmup, sync_ranks=None):
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if sync_ranks:
        sync_ranks()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    t_host1 = time.time()
    if sync_ranks:
        sync_ranks()
    return e0.elapsed_time(e1), (t_host0, t_host1)


# --------------------------------------------------------------- sections --

def build_decode(torch, ops, dev, seed=0):
    """Quantized weights for LAYERS x 4 projections and per-(M, projection) activations."""
    layers = []
    for layer in range(LAYERS):
        per = []
        for (N, K) in SHAPES:
            w = synth.device_normal_bf16(N, K, seed, f"bench/W/{layer}/{N}x{K}", sigma=0.02, device=dev)
            qw, sw = ops.quant_weight_block(w)
            del w
            per.append((qw, sw))
        layers.append(per)
    acts = {}
    for M in DECODE_M:
        for (N, K) in SHAPES:
            cols = synth.pick(seed, f"bench/X/outliers/{K}", K, int(round(0.001 * K)))
            x = synth.device_normal_bf16(M, K, seed, f"bench/X/{M}x{K}", outlier_cols=cols, outlier_scale=50.0,
                                         device=dev)
            qa = torch.empty((M, K), dtype=torch.uint8, device=dev)
            sa = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
            ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(LAYERS)]
            acts[(M, N, K)] = (x, qa, sa, ys)
    torch.cuda.synchronize()
    return layers, acts


def decode_calls():
    return [(M, layer, i) for M in DECODE_M for layer in range(LAYERS) for i in range(len(SHAPES))]


def run_decode_section(torch, ops, dev, steps, warmup, peaks, sync_ranks):
    layers, acts = build_decode(torch, ops, dev)
    calls = decode_calls()

    def step(marks):
        for (M, layer, i) in calls:
            N, K = SHAPES[i]
            x, qa, sa, ys = acts[(M, N, K)]
            qw, sw = layers[layer][i]
            ops.fp8_block_linear(x, qa, sa, qw, sw, ys[layer])

    step_bytes = sum(linear_bytes(M, *SHAPES[i]) for M, _, i in calls)
    gemm_total_bytes = sum(gemm_bytes(M, *SHAPES[i]) for M, _, i in calls)
    timed = Timed(torch, step)
    ms, window = time_steps(torch, timed.replay, steps, warmup, sync_ranks)
    value = step_bytes * steps / (ms * 1e-3) / 1e9
    # Sustained: the same step replayed for at least SUSTAINED_S seconds
    # (whatever --steps is), so that the clocks are sampled under a long load.
    sus = None
    if SUSTAINED_S > 0:
        n_sus = max(steps, int(SUSTAINED_S / max(ms / steps * 1e-3, 1e-6)) + 1)
        ms_sus, window_sus = time_steps(torch, timed.replay, n_sus, 1, sync_ranks)
        sus = {"value": step_bytes * n_sus / (ms_sus * 1e-3) / 1e9, "unit": "GB/s", "steps": n_sus,
               "seconds": ms_sus * 1e-3, "ms_per_step": ms_sus / n_sus, "window": window_sus}

    # Dominant kernel: the same GEMM launches back to back in one graph (the
    # activation codes are already in place), timed with events around the
    # replays; average launch duration = time / launches.
    def gemms(marks, sel=None):
        for (M, layer, i) in (sel or calls):
            N, K = SHAPES[i]
            _, qa, sa, ys = acts[(M, N, K)]
            qw, sw = layers[layer][i]
            ops.fp8_block_gemm(qa, sa, qw, sw, ys[layer])

    g_all = Timed(torch, gemms)
    reps = max(5, steps // 2)
    ms_g, _ = time_steps(torch, g_all.replay, reps, warmup)
    launch_ms = ms_g / (reps * len(calls))
    roof = {"bound": "hbm", "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "peak_source": f"hbm_gbs of {peaks['source']}",
            "achieved": gemm_total_bytes / len(calls) / (launch_ms * 1e-3) / 1e9,
            "avg_launch_us": launch_ms * 1e3,
            "timing": "events around replays of a graph of the step's 96 GEMM launches"}
    roof["frac"] = roof["achieved"] / peaks["hbm_gbs"]
    roof["traffic"] = _traffic("gemm_decode_kernel", gemm_total_bytes / len(calls))
    roof["traffic_note"] = "ncu dram read+write per launch, captured ratio x this mix's algorithmic bytes"
    per_shape = {}
    for M in DECODE_M:
        for i, (N, K) in enumerate(SHAPES):
            sel = [(M, layer, i) for layer in range(LAYERS)]
            g = Timed(torch, lambda marks, sel=sel: gemms(marks, sel))
            t, _ = time_steps(torch, g.replay, reps, 3)
            us = t * 1e3 / (reps * LAYERS)
            per_shape[f"M{M}_N{N}_K{K}"] = {"us": us, "GBps": gemm_bytes(M, N, K) / (us * 1e-6) / 1e9}
    out = {"value": value, "ms_per_step": ms / steps, "roofline": roof, "per_shape": per_shape,
           "launches_per_step": 2 * len(calls), "window": window, "step_bytes": step_bytes, "sustained": sus}

    # End to end through the C entry point, as a C caller drives it: the step's
    # 96 activation inputs sit in one pinned host slab and its 96 outputs
    # come back into another; per step, one host->device copy of all inputs,
    # the 96 fp8_block_linear calls (pointers prepared once), one
    # device->host copy of all outputs, all inside the timed region.
    # Pipelined: two device slabs of each, the copies on streams of their own,
    # so that step i+1's inputs go up and step i-1's outputs come down while
    # step i computes (events keep each slab's copy and its calls in order).
    # The serial form (copies on the compute stream, in the chain) is timed
    # too and reported beside it.
    from fp8_w8a8_quantized_group_gb300 import _lib
    lib = _lib.load()
    x_elems = [M * SHAPES[i][1] for M, _, i in calls]
    y_elems = [M * SHAPES[i][0] for M, _, i in calls]
    x_dev = [torch.empty(sum(x_elems), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    y_dev = [torch.empty(sum(y_elems), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    x_host = torch.empty(sum(x_elems), dtype=torch.bfloat16, pin_memory=True)
    y_host = torch.empty(sum(y_elems), dtype=torch.bfloat16, pin_memory=True)
    args, xo, yo = ([], []), 0, 0
    for (M, layer, i), nx, ny in zip(calls, x_elems, y_elems):
        N, K = SHAPES[i]
        x, qa, sa, _ = acts[(M, N, K)]
        x_host[xo:xo + nx].copy_(x.reshape(-1).cpu())
        qw, sw = layers[layer][i]
        for p in range(2):
            args[p].append((x_dev[p][xo:].data_ptr(), qa.data_ptr(), sa.data_ptr(), qw.data_ptr(), sw.data_ptr(),
                            y_dev[p][yo:].data_ptr(), M, N, K))
        xo += nx
        yo += ny
    h2d = x_host.numel() * 2
    d2h = y_host.numel() * 2
    compute = torch.cuda.current_stream()
    handle = compute.cuda_stream
    linear = lib.fp8_block_linear

    def issue(p):
        for a in args[p]:
            st = linear(*a, handle)
            if st:
                raise RuntimeError(f"fp8_block_linear: status {st}")

    def serial_step():
        x_dev[0].copy_(x_host, non_blocking=True)
        issue(0)
        y_host.copy_(y_dev[0], non_blocking=True)

    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("x_ready", "x_free", "y_ready", "y_free")}
    count = [0]

    def pipelined_step():
        p = count[0] & 1
        count[0] += 1
        up.wait_event(ev["x_free"][p])  # the calls of two steps back have read this slab
        with torch.cuda.stream(up):
            x_dev[p].copy_(x_host, non_blocking=True)
        ev["x_ready"][p].record(up)
        compute.wait_event(ev["x_ready"][p])
        compute.wait_event(ev["y_free"][p])  # the outputs of two steps back have come down
        issue(p)
        ev["x_free"][p].record(compute)
        ev["y_ready"][p].record(compute)
        down.wait_event(ev["y_ready"][p])
        with torch.cuda.stream(down):
            y_host.copy_(y_dev[p], non_blocking=True)
        ev["y_free"][p].record(down)

    def time_pipelined(n, warm):
        for _ in range(warm):
            pipelined_step()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(compute)
        up.wait_event(e0)  # the first upload starts inside the timed region
        for _ in range(n):
            pipelined_step()
        compute.wait_stream(down)  # ... and the last download ends inside it
        e1.record(compute)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    e2e_steps = max(1, min(steps, 20))
    e2e_warm = max(1, min(warmup, 3))
    ms_e2e = time_pipelined(e2e_steps, e2e_warm)
    # The last step's outputs, as they came down, against the graph's.
    expect = torch.cat([acts[(M, *SHAPES[i])][3][layer].reshape(-1) for M, layer, i in calls]).cpu()
    match = bool(torch.equal(expect.view(torch.int16), y_host.view(torch.int16)))
    ms_serial, _ = time_steps(torch, serial_step, e2e_steps, e2e_warm)
    out["e2e"] = {"value": step_bytes * e2e_steps / (ms_e2e * 1e-3) / 1e9, "unit": "GB/s",
                  "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                  "ms_per_step": ms_e2e / e2e_steps, "outputs_match_graph": match,
                  "serial": {"value": step_bytes * e2e_steps / (ms_serial * 1e-3) / 1e9,
                             "ms_per_step": ms_serial / e2e_steps},
                  "note": "eager C-ABI calls of fp8_block_linear (no graph); per step one pinned "
                          "host->device copy of the 96 inputs and one device->host copy of the 96 outputs, "
                          "double-buffered on two copy streams so that they overlap the neighbouring steps' "
                          "calls; 'serial' has both copies on the compute stream"}
    del layers, acts
    return out


def run_prefill_section(torch, ops, dev, steps, warmup, peaks):
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    weights = []
    for (N, K) in SHAPES:
        w = synth.device_normal_bf16(N, K, 0, f"bench/W/0/{N}x{K}", sigma=0.02, device=dev)
        weights.append(ops.quant_weight_block(w))
        del w
    calls = []
    for M in synth.PREFILL_M:
        for i, (N, K) in enumerate(SHAPES):
            cols = synth.pick(0, f"bench/X/outliers/{K}", K, int(round(0.001 * K)))
            x = synth.device_normal_bf16(M, K, 0, f"bench/Xp/{M}x{K}", outlier_cols=cols, outlier_scale=50.0,
                                         device=dev)
            qa, sa = ops.quant_act_group(x)
            del x
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            calls.append((M, N, K, qa, sa, weights[i], y))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step(marks):
        for j, (M, N, K, qa, sa, (qw, sw), y) in enumerate(calls):
            flush.zero_()  # evict L2 between GEMMs (outside the kernel's events)
            if marks:
                marks[j][0].record()
            ops.fp8_block_gemm(qa, sa, qw, sw, y)
            if marks:
                marks[j][1].record()

    timed = Timed(torch, step, n_marks=len(calls))
    ms, _ = time_steps(torch, timed.replay, steps, warmup)
    per = {}
    total_flop = 0
    total_ms = 0.0
    if timed.ext:
        kms = timed.mark_ms()
        for j, (M, N, K, *_rest) in enumerate(calls):
            fl = 2.0 * M * N * K
            total_flop += fl
            total_ms += kms[j]
            per[f"M{M}_N{N}_K{K}"] = {"us": kms[j] * 1e3, "TFLOPS": fl / (kms[j] * 1e-3) / 1e12}
    achieved = total_flop / (total_ms * 1e-3) / 1e12 if total_ms else None
    out = {"metric": "FP8 block-scaled GEMM TFLOPS", "unit": "TFLOP/s", "value": achieved,
           "roofline": {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                        "frac": achieved / fp8_peak if achieved else None,
                        "peak_source": f"bf16_tflops of {peaks['source']} x {FP8_OVER_BF16} (nominal FP8/BF16)",
                        "traffic": _traffic("gemm_prefill_kernel", sum(
                            M * K + N * K + 2 * M * N + 4 * M * K // 128 for (M, N, K, *_r) in calls) / len(calls))},
           "per_shape": per, "ms_per_step_incl_l2_flush": ms / steps,
           "l2": "256 MB buffer written between GEMMs, outside the kernel events"}
    del calls, weights, flush
    return out


def run_tensor_section(torch, ops, dev, steps, warmup, peaks):
    """Per-tensor W8A8 layer, N = K = 8192, static weight scale, dynamic
    activation scale. M <= 16 is timed as the headline is: 8 layers of
    distinct weights (512 MB, far beyond L2) back to back in one graph, each
    call the per-tensor quantization of X chained to the decode GEMM; GB/s of
    the GEMM's algorithmic bytes over the GEMM launches alone, and of the
    whole layer. M >= 512 is timed per GEMM after a 256 MB L2 flush
    (TFLOP/s against the FP8 peak)."""
    N = K = 8192
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    layers = []
    for layer in range(LAYERS):
        w = synth.device_normal_bf16(N, K, layer, "bench/Wt", sigma=0.015,
                                     outlier_rows=synth.pick(0, "bench/Wt/rows", N, 8), outlier_scale=20.0,
                                     device=dev)
        qw, sw = ops.quant_per_tensor(w)          # load time: dynamic scale of W becomes its static scale
        qw, sw = ops.quant_per_tensor(w, scale=sw)
        layers.append((qw, sw))
        del w
    out = {"per_shape": {}}
    cols = synth.pick(0, f"bench/Xt/outliers/{K}", K, int(round(0.001 * K)))
    for M in [m for m in synth.PER_TENSOR_M if m <= 16]:
        x = synth.device_normal_bf16(M, K, 0, f"bench/Xt/{M}", outlier_cols=cols, outlier_scale=100.0, device=dev)
        qa = torch.empty((M, K), dtype=torch.uint8, device=dev)
        sa = torch.empty(1, dtype=torch.float32, device=dev)
        ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(LAYERS)]
        ops.fp8_quant_per_tensor(x, qa, sa, False)

        def gemms(marks, qa=qa, sa=sa, ys=ys):
            for layer, (qw, sw) in enumerate(layers):
                ops.fp8_tensor_gemm(qa, sa, qw, sw, ys[layer])

        def layer_calls(marks, x=x, qa=qa, sa=sa, ys=ys):
            for layer, (qw, sw) in enumerate(layers):
                ops.fp8_quant_per_tensor(x, qa, sa, False)
                ops.fp8_tensor_gemm(qa, sa, qw, sw, ys[layer])
        reps = max(5, steps)
        g = Timed(torch, gemms)
        ms_g, _ = time_steps(torch, g.replay, reps, warmup)
        g2 = Timed(torch, layer_calls)
        ms_l, _ = time_steps(torch, g2.replay, reps, warmup)
        us = ms_g * 1e3 / (reps * LAYERS)
        us_l = ms_l * 1e3 / (reps * LAYERS)
        nbytes = tensor_gemm_bytes(M, N, K)
        lbytes = nbytes + 2 * M * K + 2 * M * K  # + the activations, read twice by the dynamic per-tensor pass
        out["per_shape"][f"M{M}"] = {
            "us": us, "GBps": nbytes / (us * 1e-6) / 1e9,
            "roofline": {"bound": "hbm", "achieved": nbytes / (us * 1e-6) / 1e9, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"],
                         "peak_source": f"hbm_gbs of {peaks['source']}"},
            "layer_us": us_l, "layer_GBps": lbytes / (us_l * 1e-6) / 1e9,
            "timing": "8 distinct 64 MB weights back to back in a graph; layer = dynamic per-tensor "
                      "quantization of X + the GEMM"}
    qw, sw = layers[0]
    calls = []
    for M in [m for m in synth.PER_TENSOR_M if m > 16]:
        x = synth.device_normal_bf16(M, K, 0, f"bench/Xt/{M}", outlier_cols=cols, outlier_scale=100.0, device=dev)
        qa = torch.empty((M, K), dtype=torch.uint8, device=dev)
        sa = torch.empty(1, dtype=torch.float32, device=dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        calls.append((M, x, qa, sa, y))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step(marks):
        for j, (M, x, qa, sa, y) in enumerate(calls):
            flush.zero_()
            ops.fp8_quant_per_tensor(x, qa, sa, False)
            if marks:
                marks[j][0].record()
            ops.fp8_tensor_gemm(qa, sa, qw, sw, y)
            if marks:
                marks[j][1].record()

    timed = Timed(torch, step, n_marks=len(calls))
    time_steps(torch, timed.replay, steps, warmup)
    if timed.ext:
        for j, (M, *_r) in enumerate(calls):
            t = timed.mark_ms()[j] * 1e-3
            tf = 2.0 * M * N * K / t / 1e12
            out["per_shape"][f"M{M}"] = {
                "us": t * 1e6, "TFLOPS": tf, "GBps": tensor_gemm_bytes(M, N, K) / t / 1e9,
                "roofline": {"bound": "tensor", "achieved": tf, "peak": fp8_peak, "unit": "TFLOP/s",
                             "frac": tf / fp8_peak,
                             "peak_source": f"bf16_tflops of {peaks['source']} x {FP8_OVER_BF16}"},
                "timing": "the GEMM alone after a 256 MB L2 flush"}
    out["note"] = "M <= 16 is HBM-bound (GB/s), M >= 512 tensor-bound (TFLOPS)"
    del layers, calls, flush
    return out


def run_moe_section(torch, ops, dev, steps, warmup, peaks):
    """Mixture-of-experts layer: 8 experts [2048, 7168], 4096 tokens routed
    top-2 (8192 rows). Timed after a 256 MB L2 flush: the activation
    quantization of the routed rows, read through the routing index from the
    token-order X (no permuted copy), then the grouped GEMM."""
    tokens, E, N, K = 4096, 8, 2048, 7168
    token_of_row, offsets = synth.route_top2(tokens, E, seed=0)
    x = synth.device_normal_bf16(tokens, K, 0, "bench/moe/X", device=dev)
    ri = torch.from_numpy(token_of_row.astype(np.int32)).to(dev)
    qw = torch.empty((E, N, K), dtype=torch.uint8, device=dev)
    sw = torch.empty((E, N // 128, K // 128), dtype=torch.float32, device=dev)
    for e in range(E):
        w = synth.device_normal_bf16(N, K, 0, f"bench/moe/W{e}", sigma=0.02, device=dev)
        ops.fp8_quant_weight_block(w, qw[e], sw[e])
    M = ri.shape[0]
    qa = torch.empty((M, K), dtype=torch.uint8, device=dev)
    sa = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    off = torch.from_numpy(offsets).to(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step(marks):
        flush.zero_()
        if marks:
            marks[0][0].record()
        ops.fp8_quant_act_group_gather(x, ri, qa, sa)
        if marks:
            marks[1][0].record()
        ops.fp8_block_gemm(qa, sa, qw, sw, y, num_groups=E, group_offsets=off)
        if marks:
            marks[0][1].record()
            marks[1][1].record()

    timed = Timed(torch, step, n_marks=2)
    time_steps(torch, timed.replay, steps, warmup)
    out = {"counts": np.diff(offsets).tolist()}
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    fl = 2.0 * M * N * K
    if timed.ext:
        t_all, t_gemm = (v * 1e-3 for v in timed.mark_ms())
        out.update({"us": t_gemm * 1e6, "TFLOPS": fl / t_gemm / 1e12, "frac_fp8_peak": fl / t_gemm / 1e12 / fp8_peak,
                    "layer_us": t_all * 1e6, "layer_TFLOPS": fl / t_all / 1e12,
                    "quant_gather_GBps": (2 * M * K + M * K + 4 * M * K // 128) / (t_all - t_gemm) / 1e9,
                    "roofline": {"bound": "tensor", "achieved": fl / t_gemm / 1e12, "peak": fp8_peak,
                                 "unit": "TFLOP/s", "frac": fl / t_gemm / 1e12 / fp8_peak,
                                 "peak_source": f"bf16_tflops of {peaks['source']} x {FP8_OVER_BF16}"},
                    "note": "TFLOPS of the grouped GEMM; layer_* = routed-row activation quantization from "
                            "token-order X + the GEMM"})
    del x
    return out


def _cpu_quant_times(jobs_host):
    """The oracle's quantizers on the full shapes on all host cores (row slices
    of whole blocks per thread; the oracle's C calls release the GIL), each
    timed once. jobs_host: [(name, fn(lo, hi), rows, row_block)]."""
    import concurrent.futures as cf
    threads = os.cpu_count() or 1
    out = {}
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        for name, fn, rows, rb in jobs_host:
            blocks = -(-rows // rb)
            bounds = [rb * (blocks * i // threads) for i in range(threads + 1)]
            bounds[-1] = rows
            t0 = time.perf_counter()
            for f in [ex.submit(fn, a, b) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]:
                f.result()
            out[name] = {"us": (time.perf_counter() - t0) * 1e6, "threads": threads}
    return out


def run_quant_section(torch, ops, dev, steps, warmup, peaks, cpu=False):
    x = synth.device_normal_bf16(8192, 14336, 0, "bench/q/X", device=dev)
    qa = torch.empty(x.shape, dtype=torch.uint8, device=dev)
    sa = torch.empty((14336 // 128, 8192), dtype=torch.float32, device=dev)
    w = synth.device_normal_bf16(28672, 4096, 0, "bench/q/W", sigma=0.02, device=dev)
    qw = torch.empty(w.shape, dtype=torch.uint8, device=dev)
    sw = torch.empty((28672 // 128, 4096 // 128), dtype=torch.float32, device=dev)
    xt = synth.device_normal_bf16(4096, 8192, 0, "bench/q/Xt", device=dev)
    qt = torch.empty(xt.shape, dtype=torch.uint8, device=dev)
    st = torch.empty(1, dtype=torch.float32, device=dev)
    jobs = [("act_group 8192x14336", lambda: ops.fp8_quant_act_group(x, qa, sa), act_quant_bytes(8192, 14336)),
            ("weight_block 28672x4096", lambda: ops.fp8_quant_weight_block(w, qw, sw),
             3 * 28672 * 4096 + 4 * 224 * 32),
            ("per_tensor_dynamic 4096x8192", lambda: ops.fp8_quant_per_tensor(xt, qt, st, False),
             5 * 4096 * 8192 + 4)]
    out = {}
    for name, fn, nbytes in jobs:
        timed = Timed(torch, lambda marks, fn=fn: fn())
        ms, _ = time_steps(torch, timed.replay, steps, warmup)
        t = ms / steps * 1e-3
        out[name] = {"us": t * 1e6, "GBps": nbytes / t / 1e9, "frac_hbm": nbytes / t / 1e9 / peaks["hbm_gbs"]}
    out["note"] = ("inputs larger than L2 (235/235/64 MB); per_tensor_dynamic counts its two reads of the input "
                   "(amax pass + quantize pass)")
    if cpu:
        # The CPU oracle on the same full-size inputs (copied to the host
        # first, outside the timing), for scale: all host cores.
        import oracle
        oracle.build()
        xh = x.view(torch.int16).cpu().numpy().view(np.uint16)
        wh = w.view(torch.int16).cpu().numpy().view(np.uint16)
        cpu_t = _cpu_quant_times([
            ("act_group 8192x14336", lambda a, b: oracle.quant_act_group(xh[a:b]), xh.shape[0], 1),
            ("weight_block 28672x4096", lambda a, b: oracle.quant_weight_block(wh[a:b]), wh.shape[0], 128)])
        for name, v in cpu_t.items():
            out[name]["cpu_oracle"] = {**v, "GBps": [j for j in jobs if j[0] == name][0][2] / (v["us"] * 1e-6) / 1e9}
    return out


def run_rowwise_section(torch, ops, dev, steps, warmup, peaks):
    """Per-token activation x per-channel weight scales: decode shapes (M = 16,
    the four projections, 8 layers of distinct weights back to back, GB/s)
    and prefill shapes (M = 8192, each GEMM alone after an L2 flush, TFLOP/s)."""
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    out = {"decode": {}, "prefill": {}}
    weights = []
    for layer in range(LAYERS):
        per = []
        for (N, K) in SHAPES:
            w = synth.device_normal_bf16(N, K, 0, f"bench/rw/W/{layer}/{N}x{K}", sigma=0.02, device=dev)
            per.append(ops.quant_rowwise(w))
            del w
        weights.append(per)
    M = 16
    acts = {}
    for (N, K) in SHAPES:
        cols = synth.pick(0, f"bench/X/outliers/{K}", K, int(round(0.001 * K)))
        x = synth.device_normal_bf16(M, K, 0, f"bench/rw/X/{M}x{K}", outlier_cols=cols, outlier_scale=50.0,
                                     device=dev)
        qa, sa = ops.quant_rowwise(x)
        acts[(N, K)] = (qa, sa, [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(LAYERS)])
    reps = max(5, steps)
    total_bytes, total_us = 0.0, 0.0
    for i, (N, K) in enumerate(SHAPES):
        qa, sa, ys = acts[(N, K)]

        def g(marks, i=i, qa=qa, sa=sa, ys=ys):
            for layer in range(LAYERS):
                qw, sw = weights[layer][i]
                ops.fp8_rowwise_gemm(qa, sa, qw, sw, ys[layer])
        t = Timed(torch, g)
        ms, _ = time_steps(torch, t.replay, reps, warmup)
        us = ms * 1e3 / (reps * LAYERS)
        nbytes = N * K + 4 * N + M * K + 4 * M + 2 * M * N
        total_bytes += nbytes
        total_us += us
        out["decode"][f"M{M}_N{N}_K{K}"] = {"us": us, "GBps": nbytes / (us * 1e-6) / 1e9}
    ach = total_bytes / (total_us * 1e-6) / 1e9
    out["decode"]["roofline"] = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                 "frac": ach / peaks["hbm_gbs"], "peak_source": f"hbm_gbs of {peaks['source']}",
                                 "timing": "events around a graph of 8 back-to-back GEMMs per shape"}
    del weights, acts
    wq = []
    for (N, K) in SHAPES:
        w = synth.device_normal_bf16(N, K, 0, f"bench/rw/Wp/{N}x{K}", sigma=0.02, device=dev)
        wq.append(ops.quant_rowwise(w))
        del w
    calls = []
    for i, (N, K) in enumerate(SHAPES):
        Mp = 8192
        x = synth.device_normal_bf16(Mp, K, 0, f"bench/rw/Xp/{K}", device=dev)
        qa, sa = ops.quant_rowwise(x)
        del x
        calls.append((Mp, N, K, qa, sa, wq[i], torch.empty((Mp, N), dtype=torch.bfloat16, device=dev)))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step(marks):
        for j, (Mp, N, K, qa, sa, (qw, sw), y) in enumerate(calls):
            flush.zero_()
            if marks:
                marks[j][0].record()
            ops.fp8_rowwise_gemm(qa, sa, qw, sw, y)
            if marks:
                marks[j][1].record()
    timed = Timed(torch, step, n_marks=len(calls))
    time_steps(torch, timed.replay, steps, warmup)
    if timed.ext:
        kms = timed.mark_ms()
        fl_total, ms_total = 0.0, 0.0
        for j, (Mp, N, K, *_r) in enumerate(calls):
            fl = 2.0 * Mp * N * K
            fl_total += fl
            ms_total += kms[j]
            out["prefill"][f"M{Mp}_N{N}_K{K}"] = {"us": kms[j] * 1e3, "TFLOPS": fl / (kms[j] * 1e-3) / 1e12}
        ach = fl_total / (ms_total * 1e-3) / 1e12
        out["prefill"]["roofline"] = {"bound": "tensor", "achieved": ach, "peak": fp8_peak, "unit": "TFLOP/s",
                                      "frac": ach / fp8_peak,
                                      "peak_source": f"bf16_tflops of {peaks['source']} x {FP8_OVER_BF16}",
                                      "timing": "each GEMM alone after a 256 MB L2 flush"}
    del calls, wq, flush
    return out


def run_kv_section(torch, ops, dev, steps, warmup, peaks):
    """FP8 KV cache: store prefill batches of 8192 tokens (8 KV heads x 128,
    keys and values) into random slots of a 65536-slot cache, and gather-load
    all 65536 slots back to BF16. HBM GB/s of algorithmic bytes. The stores
    are timed as four distinct batches back to back in one graph (134 MB of
    inputs, more than L2), per store."""
    T, E, S, B = 8192, 1024, 65536, 4
    ks_in = [synth.device_normal_bf16(T, E, b, "bench/kv/k", device=dev) for b in range(B)]
    vs_in = [synth.device_normal_bf16(T, E, b, "bench/kv/v", device=dev) for b in range(B)]
    kc = torch.zeros((S, E), dtype=torch.uint8, device=dev)
    vc = torch.zeros((S, E), dtype=torch.uint8, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    perm = torch.randperm(S, generator=g, device=dev)
    slot_sets = [perm[b * T:(b + 1) * T].contiguous() for b in range(B)]
    all_slots = torch.randperm(S, generator=g, device=dev).contiguous()
    ks = torch.tensor([0.02], dtype=torch.float32, device=dev)
    vs = torch.tensor([0.015], dtype=torch.float32, device=dev)
    ko = torch.empty((S, E), dtype=torch.bfloat16, device=dev)
    vo = torch.empty((S, E), dtype=torch.bfloat16, device=dev)
    out = {}
    def stores():
        for b in range(B):
            ops.fp8_kv_cache_store(ks_in[b], vs_in[b], kc, vc, slot_sets[b], ks, vs)

    jobs = [("store 8192 tokens", stores, B, 2 * T * E * 3 + 8 * T),
            ("load 65536 slots", lambda: ops.fp8_kv_cache_load(kc, vc, ko, vo, all_slots, ks, vs), 1,
             2 * S * E * 3 + 8 * S)]
    for name, fn, calls, nbytes in jobs:
        timed = Timed(torch, lambda marks, fn=fn: fn())
        ms, _ = time_steps(torch, timed.replay, steps, warmup)
        t = ms / steps / calls * 1e-3
        out[name] = {"us": t * 1e6, "GBps": nbytes / t / 1e9, "frac_hbm": nbytes / t / 1e9 / peaks["hbm_gbs"]}
    out["note"] = ("E = 8 KV heads x 128; store reads BF16 K and V and writes E4M3 codes (3 B per element each), "
                   "timed per store over 4 distinct 8192-token batches in one graph (134 MB of inputs); load reads "
                   "codes and writes BF16 (134 MB of codes); both larger than the 129 MB L2")
    del ks_in, vs_in, kc, vc, ko, vo
    return out


# --------------------------------------------------------------- CPU legs --

_CPU_WEIGHTS = {}


def _cpu_weights(N, K, n):
    """Quantized weights of the first n rows of a projection for the CPU legs
    (generated and quantized once per process, outside every timed region)."""
    import oracle
    key = (N, K, n)
    if key not in _CPU_WEIGHTS:
        _CPU_WEIGHTS[key] = oracle.quant_weight_block(synth.weights(n, K, 0, f"cpu/W/{N}x{K}"))
    return _CPU_WEIGHTS[key]


def oracle_decode_sample(threads: int | None = None, ms=None, cols: int | None = None, min_seconds: float = 0.0):
    """Times the CPU oracle on one layer of the decode workload: for each M in
    `ms` and each projection, activation quantization of X [M, K] and the FP64
    dequantize-then-GEMM over the first `cols` output columns (all N by
    default). `threads` host threads split the output columns at 128-column
    boundaries (the oracle's C calls release the GIL). The layer is repeated
    until the timed total reaches `min_seconds` (at least once). Returns (GB/s
    of algorithmic bytes, description, seconds)."""
    import concurrent.futures as cf

    import oracle
    oracle.build()
    threads = threads or os.cpu_count() or 1
    ms = list(ms or DECODE_M)
    cases = [(N, K, min(N, cols) if cols else N) for (N, K) in SHAPES]
    xs = {(M, K): synth.activations(M, K, 0, f"cpu/X/{M}x{K}") for M in ms for (_, K, _) in cases}
    t_total, nbytes, passes = 0.0, 0.0, 0
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        while passes == 0 or t_total < min_seconds:
            for M in ms:
                for (N, K, n) in cases:
                    qw, sw = _cpu_weights(N, K, n)
                    blocks = -(-n // 128)
                    bounds = [128 * (blocks * i // threads) for i in range(threads + 1)]
                    bounds[-1] = n
                    t0 = time.perf_counter()
                    qa, sa = oracle.quant_act_group(xs[(M, K)])
                    futs = [ex.submit(oracle.gemm_block, qa, sa, qw[a:b], sw[a // 128:-(-b // 128)],
                                      with_absdot=False)
                            for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
                    for f in futs:
                        f.result()
                    t_total += time.perf_counter() - t0
                    nbytes += linear_bytes(M, n, K)
            passes += 1
    desc = (f"one layer of the decode step: M in {ms} x the four projections, activation quantization + FP64 GEMM "
            f"on the first {[n for (_, _, n) in cases]} output columns, C oracle on {threads} host thread(s)"
            + (f", {passes} passes" if passes > 1 else ""))
    return nbytes / t_total / 1e9, desc, t_total


def host_cpu() -> dict:
    """The host the CPU baseline ran on: logical CPUs, architecture and, where
    the platform reports it, the CPU model."""
    import platform
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return {"logical_cpus": os.cpu_count(), "machine": platform.machine(), "model": model}


def decode_workload() -> str:
    return (f"decode block-scaled W8A8: M in {DECODE_M} x projections {SHAPES} x {LAYERS} "
            "layers of distinct weights; step = act quant + GEMM for each")


def reference_arm(args):
    """--impl reference: the CPU oracle as it stands, on the decode workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    vals = []
    desc = ""
    threads = os.cpu_count() or 1
    # Size each step so that the whole run takes about REF_TOTAL_S: time a
    # 512-column slice of the layer once (untimed calibration), then scale the
    # columns (whole 128-column blocks, at most all of N).
    _, _, t512 = oracle_decode_sample(threads, cols=512)
    per_step = REF_TOTAL_S / max(1, args.warmup + args.steps)
    cols = max(128, int(512 * per_step / max(t512, 1e-6)) // 128 * 128)
    cols = None if cols >= max(N for N, _ in SHAPES) else cols
    for i in range(args.warmup + args.steps):
        v, desc, _ = oracle_decode_sample(threads, cols=cols)
        if i >= args.warmup:
            vals.append(v)
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded SplitMix64/Box-Muller)",
            "config": {"workload": decode_workload(), "parallelism": f"host, {threads} threads",
                       "sample": "each step the layer the GPU arm's cpu_baseline samples, on its first output "
                                 f"columns, sized so that the whole run takes about {REF_TOTAL_S:.0f} s"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": desc,
                             "host": host_cpu()},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ------------------------------------------------------------ single case --

def run_case(spec: str, launches: int):
    """One kernel on one shape, for profiling: KIND:M:N:K with KIND in
    decode|prefill|linear|tensor|rowwise|moe|act|weight|ptensor|kvstore|kvload (for the KV
    kinds M is the tokens, K the elements per token, N the cache slots). Prints
    per-launch times."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from fp8_w8a8_quantized_group_gb300 import ops
    kind, M, N, K = spec.split(":")
    M, N, K = int(M), int(N), int(K)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    x = synth.device_normal_bf16(M, K, 0, "case/X", device=dev)
    if kind in ("decode", "prefill"):
        qa, sa = ops.quant_act_group(x)
        qw, sw = ops.quant_weight_block(synth.device_normal_bf16(N, K, 0, "case/W", sigma=0.02, device=dev))
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        fn = lambda: ops.fp8_block_gemm(qa, sa, qw, sw, y)  # noqa: E731
    elif kind == "linear":
        qa = torch.empty((M, K), dtype=torch.uint8, device=dev)
        sa = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
        qw, sw = ops.quant_weight_block(synth.device_normal_bf16(N, K, 0, "case/W", sigma=0.02, device=dev))
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        fn = lambda: ops.fp8_block_linear(x, qa, sa, qw, sw, y)  # noqa: E731
    elif kind == "tensor":
        qa, sa = ops.quant_per_tensor(x)
        qw, sw = ops.quant_per_tensor(synth.device_normal_bf16(N, K, 0, "case/W", sigma=0.02, device=dev))
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        fn = lambda: ops.fp8_tensor_gemm(qa, sa, qw, sw, y)  # noqa: E731
    elif kind == "moe":
        E = 8
        tok, off = synth.route_top2(M // 2, E, seed=0)
        xp = x[: M // 2].index_select(0, torch.from_numpy(tok).to(dev))
        qa, sa = ops.quant_act_group(xp)
        qw = torch.empty((E, N, K), dtype=torch.uint8, device=dev)
        sw = torch.empty((E, N // 128, K // 128), dtype=torch.float32, device=dev)
        for e in range(E):
            ops.fp8_quant_weight_block(synth.device_normal_bf16(N, K, 0, f"case/W{e}", sigma=0.02, device=dev),
                                       qw[e], sw[e])
        y = torch.empty((xp.shape[0], N), dtype=torch.bfloat16, device=dev)
        offd = torch.from_numpy(off).to(dev)
        fn = lambda: ops.fp8_block_gemm(qa, sa, qw, sw, y, num_groups=E, group_offsets=offd)  # noqa: E731
    elif kind == "rowwise":
        qa, sa = ops.quant_rowwise(x)
        qw, sw = ops.quant_rowwise(synth.device_normal_bf16(N, K, 0, "case/W", sigma=0.02, device=dev))
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        fn = lambda: ops.fp8_rowwise_gemm(qa, sa, qw, sw, y)  # noqa: E731
    elif kind in ("kvstore", "kvload"):
        # M tokens of K elements each, N cache slots (a random permutation)
        kc = torch.zeros((N, K), dtype=torch.uint8, device=dev)
        vc = torch.zeros((N, K), dtype=torch.uint8, device=dev)
        g = torch.Generator(device=dev)
        g.manual_seed(5)
        sl = torch.randperm(N, generator=g, device=dev)[:M].contiguous()
        ks = torch.tensor([0.02], dtype=torch.float32, device=dev)
        xv = synth.device_normal_bf16(M, K, 1, "case/V", device=dev)
        if kind == "kvstore":
            fn = lambda: ops.fp8_kv_cache_store(x, xv, kc, vc, sl, ks, ks)  # noqa: E731
        else:
            fn = lambda: ops.fp8_kv_cache_load(kc, vc, x, xv, sl, ks, ks)  # noqa: E731
    elif kind == "act":
        qa = torch.empty((M, K), dtype=torch.uint8, device=dev)
        sa = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
        fn = lambda: ops.fp8_quant_act_group(x, qa, sa)  # noqa: E731
    elif kind == "weight":
        qw = torch.empty((M, K), dtype=torch.uint8, device=dev)
        sw = torch.empty((-(-M // 128), K // 128), dtype=torch.float32, device=dev)
        fn = lambda: ops.fp8_quant_weight_block(x, qw, sw)  # noqa: E731
    elif kind == "ptensor":
        q = torch.empty((M, K), dtype=torch.uint8, device=dev)
        s = torch.empty(1, dtype=torch.float32, device=dev)
        fn = lambda: ops.fp8_quant_per_tensor(x, q, s, False)  # noqa: E731
    else:
        raise SystemExit(f"unknown case kind {kind}")
    times = []
    for _ in range(launches):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3)
    # device time per launch: a graph of back-to-back launches, replayed
    reps = 20
    g = Timed(torch, lambda marks: [fn() for _ in range(reps)])
    ms, _ = time_steps(torch, g.replay, 5, 2)
    graph_us = ms * 1e3 / (5 * reps)
    code, site = ops.fp8_device_error()
    print(json.dumps({"case": spec, "us": times, "graph_us": graph_us, "device_error": code}))
    if code:
        raise SystemExit(1)


# ------------------------------------------------------------------- main --

def main():
    global SUSTAINED_S
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sections", default="prefill,tensor,moe,quant,rowwise,kv")
    ap.add_argument("--case", default=None, help="profile one kernel: KIND:M:N:K")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--sustained", type=float, default=SUSTAINED_S,
                    help="seconds of replays in the sustained leg of the headline (0: skip it)")
    args = ap.parse_args()
    if args.case:
        run_case(args.case, args.launches)
        return
    args.warmup = max(3, args.warmup)
    SUSTAINED_S = args.sustained
    if args.impl == "reference":
        reference_arm(args)
        return

    import torch
    import torch.distributed as dist

    import __graft_entry__
    __graft_entry__.build()
    from fp8_w8a8_quantized_group_gb300 import ops

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = _peaks()

    def sync_ranks():
        if world > 1:
            dist.barrier()

    sampler = ClockSampler(_gpu_id(torch, local))
    try:
        dec = run_decode_section(torch, ops, dev, args.steps, args.warmup, peaks, sync_ranks)
        sections = {}
        wanted = [s for s in args.sections.split(",") if s]
        sec_steps = max(5, min(args.steps, 30))
        for name, fn in [("prefill", run_prefill_section), ("tensor", run_tensor_section),
                         ("moe", run_moe_section), ("quant", run_quant_section),
                         ("rowwise", run_rowwise_section), ("kv", run_kv_section)]:
            if name in wanted:
                torch.cuda.empty_cache()
                kw = {"cpu": world == 1} if name == "quant" else {}
                sections[name] = fn(torch, ops, dev, sec_steps, 3, peaks, **kw)
        code, site = ops.fp8_device_error()
    finally:
        sampler.stop()
    clocks = sampler.summary(*dec["window"])
    if dec["sustained"] is not None:
        dec["sustained"]["clocks"] = sampler.summary(*dec["sustained"].pop("window"))

    # whole-job value: units of all ranks over the slowest rank's time
    bytes_per_s, ms_step = whole_job(dec["step_bytes"], dec["ms_per_step"], world, dist, dev)
    value = bytes_per_s / 1e9
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    cpu = None
    if world == 1:
        threads = os.cpu_count() or 1
        v, desc, secs = oracle_decode_sample(threads, min_seconds=CPU_SAMPLE_S)
        v1, desc1, secs1 = oracle_decode_sample(1, ms=[1], min_seconds=CPU_SAMPLE_S)
        cpu = {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": desc,
               "seconds": round(secs, 2), "host": host_cpu(),
               "one_core": {"value": v1, "sample": desc1, "seconds": round(secs1, 2)}}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3xe4m3->f32 (bf16 in/out)",
        "data": "synthetic (seeded; normal activations with 0.1% x50 outlier channels, N(0,0.02) weights)",
        "config": {"workload": decode_workload(),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2: {LAYERS} layers of FP8 weights "
                         f"({sum(N * K for N, K in SHAPES) * LAYERS / 1e9:.2f} GB) stream once per M per step",
                   "graph": "each step is one CUDA graph replay"},
        "roofline": dec["roofline"], "cpu_baseline": cpu, "e2e": dec["e2e"], "sustained": dec["sustained"],
        "gpu_launches": dec["launches_per_step"] * args.steps, "clocks": clocks,
        "decode_per_shape": dec["per_shape"], "sections": sections,
        "device_error": {"code": code, "site": site}, "peaks": peaks,
    }
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
