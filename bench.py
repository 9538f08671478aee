#!/usr/bin/env python3
"""Benchmark of the quantized linear layer on B300.

One step = one pass of the whole hot path over one batch of the 70B-shaped
down-projection workload (W [8192 x 28672]):
  1. qlin_quantize   X' bf16 [4096 x 28672] -> per-token INT8, where X' = X / s
                     carries the SmoothQuant factors (alpha = 0.5) folded into
                     the previous layer, as SmoothQuant deploys them
  2. qlin_gemm_w8a8  4096 x 8192 x 28672, INT32 sums, bf16 out
  3. qlin_gemm_w4a16 UINT4 asymmetric g=128 fp16 scales, M = 1, 8, 64, 256
  4. qlin_dequantize the INT8 activations back to bf16
The reported value is the step's fraction of the B300 roofline: the sum over
kernels of max(bytes / HBM peak, ops / tensor peak) divided by the measured
step time, summed over ranks (so N replicas report up to N x 100).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from activation_quantization_quantize_b300 import inputs, qlin  # noqa: E402

METRIC = "W8A8 GEMM TOPS and W4A16 decode weight-GB/s, as % of B300 roofline"
UNIT = "% of one B300 roofline (whole job)"
M8, N, K = 4096, 8192, 28672
W4_MS = (1, 8, 64, 256)
GROUP = 128
L2_BYTES = 126 * 1024 * 1024


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ------------------------------------------------------------------ roofline model
def kernel_bytes_flops():
    """Algorithmic bytes / ops of each kernel of one step."""
    d = {}
    # quantize: read X' bf16, write int8 codes + fp32 scales
    d["quantize"] = (M8 * K * 2 + M8 * K + M8 * 4, 0.0)
    # W8A8: read both operands once, write bf16 Y; 2*M*N*K integer ops
    d["gemm_w8a8"] = (M8 * K + N * K + M8 * 4 + N * 4 + M8 * N * 2, 2.0 * M8 * N * K)
    w4_bytes = N * K // 2 + N * (K // GROUP) * 2 + N * (K // GROUP) // 2
    for m in W4_MS:
        d["gemm_w4a16_m%d" % m] = (w4_bytes + m * K * 2 + m * N * 2, 2.0 * m * N * K)
    # dequantize: read int8 codes + scales, write bf16
    d["dequantize"] = (M8 * K + M8 * 4 + M8 * K * 2, 0.0)
    return d


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one W8A8 launch
# (the CTA-pair kernel k_w8a8_pair) at 4096 x 8192 x 28672, from a one-pass
# ncu capture, and a digest of the sources that kernel was built from: a
# changed kernel reports no traffic until it is captured again.
W8A8_TRAFFIC_BYTES = 1099.7e6 + 61.1e6
W8A8_TRAFFIC_SOURCES = ("activation_quantization_quantize_b300/csrc/gemm_w8a8.cu",
                        "activation_quantization_quantize_b300/csrc/tc_ptx.cuh",
                        "activation_quantization_quantize_b300/csrc/qlin_common.cuh")
W8A8_TRAFFIC_DIGEST = "50fb8b0ea150c4ba"


def w8a8_traffic_bytes():
    import hashlib
    h = hashlib.sha256()
    for f in W8A8_TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return W8A8_TRAFFIC_BYTES if h.hexdigest()[:16] == W8A8_TRAFFIC_DIGEST else None


def _queued_device_seconds(calls, hold_cycles=40_000_000):
    """Device time of a sequence of short calls: a spin kernel (about 20 ms at
    2 GHz) holds the stream while the host enqueues them, so launch gaps on
    the host are not counted."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    torch.cuda._sleep(hold_cycles)
    e0.record()
    for c in calls:
        c()
    e1.record()
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3


def roofline_seconds(nbytes, ops, peaks, int8_peak_tflops):
    t_mem = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_ops = ops / (int8_peak_tflops * 1e12) if ops else 0.0
    return max(t_mem, t_ops)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (200 ms) during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.t0 = self.t1 = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=timestamp," + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, begin):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [l for (t, l) in self.lines if self.t0 is not None and self.t0 - 0.1 <= t <= (self.t1 or t) + 0.1]
        if not rows:
            rows = [l for (_, l) in self.lines]
        sm, smax, reasons = [], [], set()
        for l in rows:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 10:
                continue
            try:
                sm.append(float(f[2]))
                smax.append(float(f[3]))
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for name, v in zip(names, f[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workload
class Step:
    """Device-resident inputs and the launch sequence of one step."""

    def __init__(self, dev, n_w4_copies=len(W4_MS)):
        torch.cuda.set_device(dev)
        self.dev = dev
        # activations and weights (seeded synthetic)
        x = inputs.downproj_activation(M8, outliers=True)
        w = inputs.downproj_weight()
        self.x = x.to(dev)
        wd = w.to(dev)
        del x, w
        # SmoothQuant factors (alpha = 0.5) from the channel maxima; the weights
        # are smoothed offline and 1/s is folded into the previous layer, so the
        # step's activations arrive as X' = bf16(X / s)
        xmax = qlin.absmax(self.x, qlin.QLIN_PER_COL)
        wmax = qlin.absmax(wd, qlin.QLIN_PER_COL)
        self.smooth = qlin.smooth_factors(xmax, wmax, 0.5)
        self.x = (self.x.float() / self.smooth[None, :]).to(torch.bfloat16)
        pw = qlin.make_params("s8", "row", smooth_mode=qlin.QLIN_SMOOTH_MULTIPLY)
        self.qw, self.sw, _ = qlin.quantize(wd, pw, smooth=self.smooth)
        # W4A16 weights (unsmoothed W), one packed copy per call so no call finds
        # its weights in L2
        p4 = qlin.make_params("u4", "group", group=GROUP, scale_f16=True)
        q4, s4, z4 = qlin.quantize(wd, p4)
        self.w4 = []
        for _ in range(n_w4_copies):
            self.w4.append(qlin.pack_w4(q4, s4, z4, N, K, GROUP))
        del q4, s4, z4, wd
        self.xs = [inputs.downproj_activation(m).to(dev) for m in W4_MS]
        # outputs / scratch
        self.px = qlin.make_params("s8", "row")
        self.qx = torch.empty((M8, K), dtype=torch.int8, device=dev)
        self.sx = torch.empty(M8, dtype=torch.float32, device=dev)
        nb = qlin.qlin_workspace_size(qlin.QLIN_OP_QUANTIZE, M8, K, 0, self.px)
        self.ws_q = torch.empty(max(nb, 16), dtype=torch.uint8, device=dev)
        self.ws_q_bytes = nb
        self.y8 = torch.empty((M8, N), dtype=torch.bfloat16, device=dev)
        self.y4 = [torch.empty((m, N), dtype=torch.bfloat16, device=dev) for m in W4_MS]
        # buffer sets of the step's inputs and outputs: set 0 is the above; the
        # end-to-end run adds a second so that copies overlap the compute
        self.sets = [(self.x, self.xs, self.y8, self.y4)]
        self.xhat = torch.empty((M8, K), dtype=torch.bfloat16, device=dev)
        self.ws4 = []
        for m in W4_MS:
            nb4 = qlin.qlin_workspace_size(qlin.QLIN_OP_GEMM_W4A16, m, N, K)
            self.ws4.append((torch.empty(max(nb4, 16), dtype=torch.uint8, device=dev), nb4))
        nb8 = qlin.qlin_workspace_size(qlin.QLIN_OP_GEMM_W8A8, M8, N, K)
        self.ws8 = torch.empty(max(nb8, 16), dtype=torch.uint8, device=dev)
        self.ws8_bytes = nb8
        torch.cuda.synchronize()

    names = ["quantize", "gemm_w8a8"] + ["gemm_w4a16_m%d" % m for m in W4_MS] + ["dequantize"]
    def launches_per_step(self):
        """Kernels one step launches: quantize (one per-token kernel), W8A8
        (plus the kernel that finishes K-split tail tiles, present when the
        workspace holds more than the INT32 drain tile), each W4A16 call (plus
        the split-K reduction when it needs a workspace), dequantize."""
        drain_bytes = (M8 * N * 4 + 15) // 16 * 16
        w8 = 1 + (1 if self.ws8_bytes > drain_bytes else 0)
        return 1 + w8 + sum(1 + (1 if nb4 > 0 else 0) for _, nb4 in self.ws4) + 1

    def add_buffer_set(self):
        dev = self.dev
        self.sets.append((torch.empty_like(self.x), [torch.empty_like(t) for t in self.xs],
                          torch.empty_like(self.y8), [torch.empty_like(t) for t in self.y4]))

    def run(self, stream, events=None, buf=0):
        """Enqueue one step on buffer set `buf`; events (len 8) bracket each
        kernel if given."""
        x, xs, y8, y4 = self.sets[buf]

        def ev(i):
            if events is not None:
                events[i].record(stream)
        ev(0)
        qlin.qlin_quantize(x, qlin.QLIN_BF16, M8, K, K, None, self.px, self.qx, self.sx, None,
                           self.ws_q, self.ws_q_bytes, stream)
        ev(1)
        qlin.qlin_gemm_w8a8(self.qx, self.sx, self.qw, self.sw, M8, N, K, y8, qlin.QLIN_BF16, None,
                            self.ws8, self.ws8_bytes, stream)
        ev(2)
        for i, m in enumerate(W4_MS):
            packed, hdr = self.w4[i % len(self.w4)]
            ws4, nb4 = self.ws4[i]
            qlin.qlin_gemm_w4a16(xs[i], packed, hdr, m, y4[i], ws4, nb4, stream)
            ev(3 + i)
        qlin.qlin_dequantize(self.qx, self.sx, None, self.px, M8, K, self.xhat, qlin.QLIN_BF16, stream)
        ev(7)


def measure_int8_reference_peak(dev):
    """Best torch._int_mm (cuBLASLt INT8) throughput on 8192^3, TFLOP/s."""
    try:
        a = torch.randint(-127, 128, (8192, 8192), dtype=torch.int8, device=dev)
        b = torch.randint(-127, 128, (8192, 8192), dtype=torch.int8, device=dev).t()
        for _ in range(3):
            torch._int_mm(a, b)
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._int_mm(a, b)
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1) / 1e3)
        del a, b
        return 2.0 * 8192 ** 3 / best / 1e12
    except Exception:  # noqa: BLE001 -- a missing INT8 library path is recorded as absent
        return None


# ------------------------------------------------------------------ the other configurations
def _time_calls(fn, n_iter=20, n_warm=3):
    """Mean seconds per call of fn(i) over n_iter calls (CUDA events)."""
    for i in range(n_warm):
        fn(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(n_iter):
        fn(i)
    e1.record()
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3 / n_iter


def _time_graph(fn, n_calls):
    """Mean seconds per call of fn(0) .. fn(n_calls - 1) replayed from one
    captured CUDA graph (no host launch cost between calls), as a decode loop
    would run them."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(3):
            fn(i)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n_calls):
            fn(i)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    e1.synchronize()
    del g
    return e0.elapsed_time(e1) / 1e3 / n_calls


def measure_other_configs(dev, peaks, int8_peak):
    """Time the remaining workloads outside the step: W4A16 decode 4096 x 4096
    (M = 1, 4, 16), W8A8 prefill 2048 x 11008 x 4096, and the quantize /
    dequantize sweep on [16384 x 4096] bf16.  Each timed call reads inputs
    larger than L2 or a distinct copy from a ring of >= 4 x L2."""
    hbm = peaks["hbm_gbs"] * 1e9
    out = {}
    ring_bytes = 4 * L2_BYTES
    # W4A16 decode: INT4 symmetric, g = 128, binary16 scales
    Nd, Kd = 4096, 4096
    wdec = inputs.to_bf16(inputs.normal((Nd, Kd), 0.02, 0)).to(dev)
    p4 = qlin.make_params("s4", "group", group=128, scale_f16=True)
    q4, s4, _ = qlin.quantize(wdec, p4)
    w_bytes = Nd * Kd // 2 + Nd * (Kd // 128) * 2
    copies = [qlin.pack_w4(q4, s4, None, Nd, Kd, 128) for _ in range(ring_bytes // w_bytes + 1)]
    dec = {}
    for m in (1, 4, 16):
        x = inputs.to_bf16(inputs.normal((m, Kd), 1.0, 1)).to(dev)
        y = torch.empty((m, Nd), dtype=torch.bfloat16, device=dev)
        nb = qlin.qlin_workspace_size(qlin.QLIN_OP_GEMM_W4A16, m, Nd, Kd)
        ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=dev)
        call = lambda i: qlin.qlin_gemm_w4a16(x, copies[i % len(copies)][0], copies[i % len(copies)][1], m,  # noqa: E731
                                               y, ws, nb, None)
        t_eager = _time_calls(call)
        t = _time_graph(call, len(copies))
        b = w_bytes + m * Kd * 2 + m * Nd * 2
        dec["M%d" % m] = {"us": t * 1e6, "weight_gbs": w_bytes / t / 1e9, "roofline_frac": b / hbm / t,
                          "us_eager": t_eager * 1e6, "timing": "CUDA graph of %d calls over distinct copies" % len(copies)}
    out["w4a16_decode_4096x4096_s4_g128"] = dec
    del copies, q4, s4, wdec
    # W8A8 prefill (SmoothQuant-smoothed X and W, per-token / per-channel INT8)
    x, w, _ = inputs.w8a8_prefill()
    xd, wd = x.to(dev), w.to(dev)
    sm = qlin.smooth_factors(qlin.absmax(xd, qlin.QLIN_PER_COL), qlin.absmax(wd, qlin.QLIN_PER_COL), 0.5)
    qx, sx, _ = qlin.quantize(xd, qlin.make_params("s8", "row", smooth_mode=qlin.QLIN_SMOOTH_DIVIDE), smooth=sm)
    qw, sw, _ = qlin.quantize(wd, qlin.make_params("s8", "row", smooth_mode=qlin.QLIN_SMOOTH_MULTIPLY), smooth=sm)
    Mp, Np, Kp = qx.shape[0], qw.shape[0], qx.shape[1]
    nrep = ring_bytes // ((Mp + Np) * Kp) + 1
    ring = [(qx.clone(), qw.clone()) for _ in range(nrep)]
    y = torch.empty((Mp, Np), dtype=torch.bfloat16, device=dev)
    nb = qlin.qlin_workspace_size(qlin.QLIN_OP_GEMM_W8A8, Mp, Np, Kp)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=dev)
    t = _time_calls(lambda i: qlin.qlin_gemm_w8a8(ring[i % nrep][0], sx, ring[i % nrep][1], sw, Mp, Np, Kp, y,
                                                  qlin.QLIN_BF16, None, ws, nb, None))
    ops = 2.0 * Mp * Np * Kp
    out["w8a8_prefill_%dx%dx%d" % (Mp, Np, Kp)] = {"us": t * 1e6, "tops": ops / t / 1e12,
                                                   "roofline_frac": ops / (int8_peak * 1e12) / t}
    del ring, qx, qw, xd, wd, x, w
    # quantize / dequantize sweep: every timed call reads a distinct copy of
    # its input from a ring of at least 4 x L2
    xs = inputs.sweep_tensor().to(dev)
    R_, C_ = xs.shape
    n_ring = -(-ring_bytes // (R_ * C_ * 2))
    xring = [xs] + [xs.clone() for _ in range(n_ring - 1)]
    sweep = {"ring": "%d input copies (%.0f MB) rotated per call" % (n_ring, n_ring * R_ * C_ * 2 / 1e6)}
    modes = [("s8", "tensor", 0), ("s8", "row", 0), ("s8", "col", 0), ("s8", "group", 32), ("s8", "group", 64),
             ("s8", "group", 128), ("s4", "tensor", 0), ("s4", "row", 0), ("s4", "group", 128), ("u8", "tensor", 0),
             ("u8", "row", 0), ("u8", "col", 0), ("u8", "group", 128)]
    for code, gran, g in modes:
        p = qlin.make_params(code, gran, group=g)
        q, s_, z_ = qlin.quantize(xs, p)
        nb = qlin.qlin_workspace_size(qlin.QLIN_OP_QUANTIZE, R_, C_, 0, p)
        ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=dev)
        t = _time_calls(lambda i: qlin.qlin_quantize(xring[i % n_ring], qlin.QLIN_BF16, R_, C_, C_, None, p, q, s_,
                                                     z_, ws, nb, None))
        b = R_ * C_ * 2 + q.numel() + s_.numel() * s_.element_size() + (0 if z_ is None else z_.numel() * 4)
        key = "quantize_%s_%s%s" % (code, gran, g if g else "")
        sweep[key] = {"us": t * 1e6, "gbs": b / t / 1e9, "roofline_frac": b / hbm / t}
        if gran in ("tensor", "col"):
            # a scope spanning rows needs its statistics before any code: the
            # input is read twice
            sweep[key]["roofline_frac_two_reads"] = (b + R_ * C_ * 2) / hbm / t
        if (code, gran) in (("s8", "row"), ("s4", "group")):
            yq = torch.empty((R_, C_), dtype=torch.bfloat16, device=dev)
            nq = -(-ring_bytes // q.numel())
            qring = [q] + [q.clone() for _ in range(nq - 1)]
            t = _time_calls(lambda i: qlin.qlin_dequantize(qring[i % nq], s_, z_, p, R_, C_, yq, qlin.QLIN_BF16,
                                                           None))
            del qring
            b = q.numel() + s_.numel() * s_.element_size() + R_ * C_ * 2
            sweep["dequantize_%s_%s%s" % (code, gran, g if g else "")] = {"us": t * 1e6, "gbs": b / t / 1e9,
                                                                           "roofline_frac": b / hbm / t}
    p = qlin.make_params("s8", "tensor", percentile=99.9)
    q, s_, z_ = qlin.quantize(xs, p)
    nb = qlin.qlin_workspace_size(qlin.QLIN_OP_QUANTIZE, R_, C_, 0, p)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=dev)
    t = _time_calls(lambda i: qlin.qlin_quantize(xring[i % n_ring], qlin.QLIN_BF16, R_, C_, C_, None, p, q, s_, z_,
                                                 ws, nb, None))
    b = R_ * C_ * 2 + q.numel() + 4
    sweep["quantize_s8_tensor_p99.9"] = {"us": t * 1e6, "gbs": b / t / 1e9, "roofline_frac": b / hbm / t,
                                         "roofline_frac_two_reads": (b + R_ * C_ * 2) / hbm / t}
    out["sweep_16384x4096_bf16"] = sweep
    del xring
    out.update(measure_next_rows(dev, peaks, int8_peak))
    return out


def measure_next_rows(dev, peaks, int8_peak):
    """W4A8 decode on the down-projection weight, the LLM.int8() decomposition
    on the prefill workload, and the SmoothQuant calibration sweep."""
    hbm = peaks["hbm_gbs"] * 1e9
    ring_bytes = 4 * L2_BYTES
    out = {}
    # W4A8: the step's UINT4 g = 128 weight (one packed copy per call from a
    # ring of >= 4 x L2), per-token INT8 activations
    w = inputs.downproj_weight().to(dev)
    p4 = qlin.make_params("u4", "group", group=GROUP, scale_f16=True)
    q4, s4, z4 = qlin.quantize(w, p4)
    del w
    w_bytes = N * K // 2 + N * (K // GROUP) * 2 + N * (K // GROUP) // 2
    copies = [qlin.pack_w4(q4, s4, z4, N, K, GROUP) for _ in range(-(-ring_bytes // w_bytes))]
    del q4, s4, z4
    dec = {}
    for m in (1, 8, 16):
        qx, sx, _ = qlin.quantize(inputs.downproj_activation(m, outliers=True).to(dev), qlin.make_params("s8", "row"))
        y = torch.empty((m, N), dtype=torch.bfloat16, device=dev)
        t = _time_calls(lambda i: qlin.qlin_gemm_w4a8(qx, sx, copies[i % len(copies)][0], copies[i % len(copies)][1],
                                                       m, y, qlin.QLIN_BF16, None, None, 0, None))
        b = w_bytes + m * K + m * 4 + m * N * 2
        dec["M%d" % m] = {"us": t * 1e6, "weight_gbs": w_bytes / t / 1e9, "roofline_frac": b / hbm / t,
                          "int_tops": 2.0 * m * N * K / t / 1e12}
    out["w4a8_decode_8192x28672_u4_g128"] = dec
    del copies
    # LLM.int8() on the prefill workload (1% outlier channels x U[20, 60])
    x, w, _ = inputs.w8a8_prefill()
    xd, wd = x.to(dev), w.to(dev)
    qw, sw, _ = qlin.quantize(wd, qlin.make_params("s8", "row"))
    Mp, Kp = xd.shape
    Np = qw.shape[0]
    nws = qlin.qlin_llmint8_workspace_size(Mp, Np, Kp, Kp // 32)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    y = torch.empty((Mp, Np), dtype=torch.bfloat16, device=dev)
    rep = torch.zeros(1 + Kp, dtype=torch.int32, device=dev)
    nrep = -(-ring_bytes // (Mp * Kp * 2 + Np * Kp)) + 1
    ring = [(xd.clone(), qw.clone()) for _ in range(nrep)]
    t = _time_calls(lambda i: qlin.qlin_gemm_llmint8(ring[i % nrep][0], qlin.QLIN_BF16, Mp, Kp, Kp, ring[i % nrep][1],
                                                     sw, Np, 6.0, Kp // 32, y, qlin.QLIN_BF16, rep, ws, nws, None))
    n_out = int(rep[0].item())
    ops = 2.0 * Mp * Np * Kp
    out["llmint8_%dx%dx%d" % (Mp, Np, Kp)] = {"us": t * 1e6, "outlier_channels": n_out, "tops": ops / t / 1e12,
                                              "roofline_frac": ops / (int8_peak * 1e12) / t, "threshold": 6.0}
    del ring, ws
    # SmoothQuant calibration: channel maxima over 4 batches, then the alpha
    # sweep (factors, smoothed per-token / per-channel INT8, error statistics)
    xmax = torch.zeros(Kp, dtype=torch.float32, device=dev)
    t_max = _time_calls(lambda i: qlin.absmax_update(xd, xmax), n_iter=20)
    wmax = qlin.absmax(wd, qlin.QLIN_PER_COL)
    px = qlin.make_params("s8", "row", smooth_mode=qlin.QLIN_SMOOTH_DIVIDE)
    pw = qlin.make_params("s8", "row", smooth_mode=qlin.QLIN_SMOOTH_MULTIPLY)
    qx = torch.empty((Mp, Kp), dtype=torch.int8, device=dev)
    sx = torch.empty(Mp, dtype=torch.float32, device=dev)
    qw2 = torch.empty((Np, Kp), dtype=torch.int8, device=dev)
    sw2 = torch.empty(Np, dtype=torch.float32, device=dev)
    errs = {}

    def sweep_once(i, record=False):
        for alpha in (0.3, 0.5, 0.7):
            s_ = qlin.smooth_factors(xmax, wmax, alpha)
            qlin.qlin_quantize(xd, qlin.QLIN_BF16, Mp, Kp, Kp, s_, px, qx, sx, None, None, 0, None)
            ex = qlin.quant_error(xd, px, qx, sx, None, smooth=s_)
            qlin.qlin_quantize(wd, qlin.QLIN_BF16, Np, Kp, Kp, s_, pw, qw2, sw2, None, None, 0, None)
            ew = qlin.quant_error(wd, pw, qw2, sw2, None, smooth=s_)
            if record:
                errs[alpha] = (ex, ew)
    t_sweep = _time_calls(sweep_once, n_iter=5, n_warm=1)
    sweep_once(0, record=True)
    tab = {}
    for alpha, (ex, ew) in errs.items():
        ex, ew = ex.cpu().numpy(), ew.cpu().numpy()
        tab["alpha_%.1f" % alpha] = {"act_rel_err": float(np.sqrt(ex[0] / ex[1])), "w_rel_err": float(np.sqrt(ew[0] / ew[1]))}
    del xd, wd, qx, qw2
    # KV cache (KIVI-style): Llama-7B attention shape, 32 heads x 128, a
    # 32768-token context, groups of 128 tokens, a 128-token bf16 window, INT4
    T_kv, C_kv, D_kv, G_kv, R_kv = 32768, 4096, 128, 128, 128
    cache = qlin.KVCache(T_kv, C_kv, D_kv, G_kv, R_kv, 4, device=dev)
    kf = inputs.to_bf16(inputs.normal((T_kv - 64, C_kv), 1.0, 91)).to(dev)
    vf = inputs.to_bf16(inputs.normal((T_kv - 64, C_kv), 1.0, 92)).to(dev)
    cache.append(kf, vf)                                 # prefill
    del kf, vf
    k1 = inputs.to_bf16(inputs.normal((64, C_kv), 1.0, 93)).to(dev)
    v1 = inputs.to_bf16(inputs.normal((64, C_kv), 1.0, 94)).to(dev)
    kq = inputs.to_bf16(inputs.normal((G_kv, C_kv), 1.0, 95)).to(dev)
    # group appends: 128 tokens into a full window, each quantizing one group;
    # a spin kernel holds the stream while the host enqueues the calls, so the
    # events see device time only
    n_grp = 16
    cache_g = qlin.KVCache((n_grp + 2) * G_kv + R_kv, C_kv, D_kv, G_kv, R_kv, 4, device=dev)
    cache_g.append(torch.cat([kq] * 2), torch.cat([kq] * 2))
    t_group = _queued_device_seconds([lambda: cache_g.append(kq, kq)] * n_grp) / n_grp
    del cache_g
    # decode steps, one token each (a group is quantized every 128th): device
    # time per call with the stream held as above, and the host-inclusive rate
    for i in range(8):
        cache.append(k1[i:i + 1], v1[i:i + 1])
    t_app = _queued_device_seconds([(lambda j: lambda: cache.append(k1[j:j + 1], v1[j:j + 1]))(8 + i)
                                    for i in range(28)]) / 28
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    for i in range(28):
        cache.append(k1[36 + i:37 + i], v1[36 + i:37 + i])
    torch.cuda.synchronize()
    t_app_host = (time.perf_counter() - h0) / 28
    k_out = torch.empty((T_kv, C_kv), dtype=torch.bfloat16, device=dev)
    v_out = torch.empty((T_kv, C_kv), dtype=torch.bfloat16, device=dev)
    t_read = _time_calls(lambda i: qlin.qlin_kv_read(cache.c, k_out, v_out, None), n_iter=10)
    T_now, tq = cache.c.length, cache.c.quantized
    rb = 2 * tq * C_kv // 2 + (tq // G_kv) * C_kv * 8 + tq * (C_kv // D_kv) * 8 + 2 * (T_now - tq) * C_kv * 2
    wb = 2 * T_now * C_kv * 2
    out["kv_cache_int4_32768x4096_g128_r128"] = {
        "append_us_per_token": t_app * 1e6, "append_us_per_token_host": t_app_host * 1e6,
        "append_timing": "device time with the host's enqueue hidden behind a spin kernel; _host: wall clock",
        "group_append_us": t_group * 1e6, "read_us": t_read * 1e6, "read_gbs": (rb + wb) / t_read / 1e9,
        "read_roofline_frac": (rb + wb) / hbm / t_read, "cache_bytes_per_token": 2 * C_kv // 2 + 8 * C_kv / G_kv
        + 8 * C_kv / D_kv, "bf16_bytes_per_token": 2 * C_kv * 2}
    del cache, k_out, v_out
    out["smoothquant_calibration_2048x4096_w11008"] = {
        "absmax_update_us": t_max * 1e6, "absmax_update_frac": Mp * Kp * 2 / hbm / t_max,
        "alpha_sweep_ms": t_sweep * 1e3, "errors": tab}
    return out


# ------------------------------------------------------------------ CPU baseline (oracle)
_SAMPLE_INPUTS = {}


def oracle_sample_seconds(rows_w8, threads):
    """Time the CPU oracle on a bounded sample of one step: rows_w8 of the
    4096 activation rows (quantize with the SmoothQuant divide, W8A8 int64
    sums and the binary64 epilogue against all 8192 weight rows, dequantize)
    and the same fraction of the 8192 W4 output channels (their dequantized
    weights and the binary64 products with M = 1, 8, 64, 256 tokens).
    Returns (seconds, fraction of the step's work, description)."""
    import oracle
    from activation_quantization_quantize_b300.inputs import normal

    used = oracle.set_threads(threads)
    frac = rows_w8 / M8
    n4 = max(1, int(round(N * frac)))
    if _SAMPLE_INPUTS.get("rows") != rows_w8:       # drawn once per process, outside the timing
        _SAMPLE_INPUTS.clear()
        _SAMPLE_INPUTS.update(
            rows=rows_w8, x=normal((rows_w8, K), 1.0, 101),
            sm=np.random.default_rng(102).uniform(0.2, 5, K).astype(np.float32),
            wq=np.random.default_rng(103).integers(-127, 128, (N, K)).astype(np.int8),
            sw=np.random.default_rng(104).uniform(1e-4, 1e-3, N).astype(np.float32),
            w4q=np.random.default_rng(105).integers(0, 16, (n4, K)).astype(np.int32),
            w4s=np.random.default_rng(106).uniform(1e-4, 1e-3, n4 * (K // GROUP)).astype(np.float32),
            w4z=np.random.default_rng(107).integers(0, 16, n4 * (K // GROUP)).astype(np.int32),
            xs=[normal((m, K), 1.0, 108 + m) for m in W4_MS])
    d = _SAMPLE_INPUTS
    x, sm, wq, sw, w4q, w4s, w4z, xs = d["x"], d["sm"], d["wq"], d["sw"], d["w4q"], d["w4s"], d["w4z"], d["xs"]
    t0 = time.perf_counter()
    qx, sx, _ = oracle.quantize(x, -127, 127, True, oracle.PER_ROW, smooth=sm, smooth_mode=oracle.SMOOTH_DIVIDE)
    acc = oracle.w8a8_acc(qx.astype(np.int8), wq)
    oracle.w8a8_out(acc, sx, sw)
    for _ in W4_MS:                       # each call of the step reads its own copy of the weight
        what = oracle.w4_dequant(w4q, w4s, w4z, GROUP)
    for xm in xs:
        oracle.matmul_f64(xm, what)
    oracle.dequantize(qx, sx, None, oracle.PER_ROW)
    sec = time.perf_counter() - t0
    desc = ("oracle on %d of %d activation rows (quantize, W8A8 int64 sums + binary64 epilogue, dequantize) "
            "and %d of %d W4 output channels (dequant + binary64 products at M = 1/8/64/256): %.4f of one "
            "step; OpenMP over rows in the W8A8 sums and binary64 products (%d threads), the quantize, "
            "dequantize and W4 dequant are single-threaded in the oracle" % (rows_w8, M8, n4, N, frac, used))
    return sec, frac, desc


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_rows(threads):
    """Activation rows of the oracle sample: two per thread (at least 32), so
    the row-parallel loops keep every core busy."""
    return 2 * max(16, threads)


# ------------------------------------------------------------------ main
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(v, world, dev):
    if world == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, world, rank):
    """The oracle as it stands on the host cores, one bounded sample of the
    step per timed step (the same sample as the cpu_baseline leg)."""
    if rank != 0:
        return
    peaks = load_peaks()
    bf = kernel_bytes_flops()
    int8_peak = peaks["bf16_tflops"]
    t_roof = sum(roofline_seconds(b, f, peaks, int8_peak) for b, f in bf.values())
    threads = cpu_threads()
    rows = cpu_rows(threads)
    for _ in range(args.warmup):
        oracle_sample_seconds(rows, threads)
    times = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sec, frac, sample = oracle_sample_seconds(rows, threads)
        times.append(sec)
    wall = time.perf_counter() - t0
    step = statistics.mean(times)
    value = 100.0 * frac * t_roof / step
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": step * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "int64+f64", "data": "synthetic",
           "config": {"workload": "70B down-projection W[8192x28672]: quantize+W8A8 M=4096, W4A16 M=1/8/64/256",
                      "step": "a %.4f sample of the step's work (same as cpu_baseline); value = roofline time "
                              "of that sample / its measured time" % frac,
                      "timed_wall_s": wall},
           "extrapolated_ms_per_full_step": step / frac * 1e3,
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


# ------------------------------------------------------------------ profiling cases
PROFILE_CASES = ("w8a8", "w8a8_full", "w4a16_m1", "w4a16_m64", "w4a16_m256", "quantize", "dequantize",
                 "sweep_row_s8", "sweep_row_u8", "sweep_group128_s8", "sweep_tensor_s8", "sweep_col_s8",
                 "sweep_col_u8", "sweep_tensor_u8", "sweep_tensorp999_s8", "w4a8_m1",
                 "llmint8", "kv_read")


def run_profile_case(name, dev):
    """One kernel on a bounded case larger than L2 (for ncu captures): two
    warm-up calls and one measured call, then exit."""
    torch.cuda.set_device(dev)
    if name.startswith("sweep_"):
        # the 16384 x 4096 sweep tensor: sweep_<gran>[g]_<code>; tensorp999:
        # per-tensor with the 99.9th-percentile clipping scale
        _, gran, code = name.split("_")
        g = int(gran[5:]) if gran.startswith("group") else 0
        pct = 99.9 if gran == "tensorp999" else 0.0
        xs = inputs.sweep_tensor().to(dev)
        p = qlin.make_params(code, "group" if g else ("tensor" if pct else gran), group=g, percentile=pct)
        fn = lambda: qlin.quantize(xs, p)  # noqa: E731
    elif name == "llmint8":
        x, w, _ = inputs.w8a8_prefill()
        xd = x.to(dev)
        qw, sw, _ = qlin.quantize(w.to(dev), qlin.make_params("s8", "row"))
        fn = lambda: qlin.gemm_llmint8(xd, qw, sw, threshold=6.0, max_outliers=128)  # noqa: E731
    elif name == "kv_read":
        cache = qlin.KVCache(8192, 4096, 128, 128, 128, 4, device=dev)
        kf = inputs.to_bf16(inputs.normal((8192, 4096), 1.0, 91)).to(dev)
        cache.append(kf, kf)
        del kf
        fn = lambda: cache.read()  # noqa: E731
    elif name == "w4a8_m1":
        w = inputs.downproj_weight().to(dev)
        p4 = qlin.make_params("u4", "group", group=GROUP, scale_f16=True)
        q4, s4, z4 = qlin.quantize(w, p4)
        packed, hdr = qlin.pack_w4(q4, s4, z4, N, K, GROUP)
        del w, q4
        qx, sx, _ = qlin.quantize(inputs.downproj_activation(1).to(dev), qlin.make_params("s8", "row"))
        fn = lambda: qlin.gemm_w4a8(qx, sx, packed, hdr)  # noqa: E731
    elif name.startswith("w8a8"):
        # 2048 x 4096 x 28672: 56 MiB + 112 MiB of int8 codes, quantized from
        # the down-projection activations (with outlier channels) and weights;
        # w8a8_full: the step's 4096 x 8192 x 28672 (for one-pass counters)
        Mp, Np = (M8, N) if name == "w8a8_full" else (2048, 4096)
        p8 = qlin.make_params("s8", "row")
        qx, sx, _ = qlin.quantize(inputs.downproj_activation(Mp, outliers=True).to(dev), p8)
        qw, sw, _ = qlin.quantize(inputs.downproj_weight(N=Np).to(dev), p8)
        fn = lambda: qlin.gemm_w8a8(qx, sx, qw, sw)  # noqa: E731
    elif name.startswith("w4a16"):
        m = int(name.split("_m")[1])
        w = inputs.downproj_weight().to(dev)
        p4 = qlin.make_params("u4", "group", group=GROUP, scale_f16=True)
        q4, s4, z4 = qlin.quantize(w, p4)
        packed, hdr = qlin.pack_w4(q4, s4, z4, N, K, GROUP)
        del w, q4
        x = inputs.downproj_activation(m).to(dev)
        fn = lambda: qlin.gemm_w4a16(x, packed, hdr)  # noqa: E731
    else:
        x = inputs.downproj_activation(M8, outliers=True).to(dev)
        px = qlin.make_params("s8", "row")
        qx, sx, _ = qlin.quantize(x, px)
        if name == "quantize":
            # as in the step: per-token INT8 of (folded) bf16 activations
            fn = lambda: qlin.quantize(x, px)  # noqa: E731
        else:
            fn = lambda: qlin.dequantize(qx, sx, None, px, M8, K)  # noqa: E731
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    if qlin.qlin_device_error() != 0:
        raise RuntimeError("device-side error")
    print(json.dumps({"profile_case": name, "ok": True}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile", choices=PROFILE_CASES, default=None,
                    help="run one kernel on a bounded case for an ncu capture, then exit")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the timings of the other workloads (decode, prefill, sweep)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    if args.profile:
        run_profile_case(args.profile, torch.device("cuda", 0))
        return
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    qlin.load()
    peaks = load_peaks()
    step = Step(dev)
    stream = torch.cuda.Stream(device=dev)
    int8_ref = measure_int8_reference_peak(dev)
    int8_peak = max(peaks["bf16_tflops"], int8_ref or 0.0)

    # warm-up
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step.run(stream)
    stream.synchronize()
    if qlin.qlin_device_error(stream) != 0:
        raise RuntimeError("device-side error during warm-up")

    # timed region: per-kernel events inside, whole-region events around
    uuid = str(getattr(torch.cuda.get_device_properties(dev), "uuid", "") or "")
    clocks = ClockSampler(("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else (uuid or local))
    clocks.start()
    time.sleep(0.4)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark(True)
    start.record(stream)
    for i in range(args.steps):
        step.run(stream, evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    clocks.mark(False)
    barrier(world)
    clock_info = clocks.stop()
    elapsed = start.elapsed_time(end) / 1e3
    elapsed = max_over_ranks(elapsed, world, dev)
    err = qlin.qlin_device_error(stream)
    if err != 0:
        raise RuntimeError("device-side error in timed region: %d" % err)

    per_kernel = {}
    for k, name in enumerate(Step.names):
        per_kernel[name] = statistics.mean(evs[i][k].elapsed_time(evs[i][k + 1]) for i in range(args.steps)) / 1e3
    bf = kernel_bytes_flops()
    t_roof = sum(roofline_seconds(bf[n][0], bf[n][1], peaks, int8_peak) for n in Step.names)
    ms_per_step = elapsed / args.steps * 1e3
    value = world * 100.0 * t_roof / (elapsed / args.steps)

    t8 = per_kernel["gemm_w8a8"]
    w8_tops = bf["gemm_w8a8"][1] / t8 / 1e12
    roofline = {"bound": "tensor", "achieved": w8_tops, "peak": int8_peak, "unit": "TFLOP/s",
                "frac": w8_tops / int8_peak, "traffic": w8a8_traffic_bytes(),
                "traffic_unit": "bytes per launch (DRAM read + write)",
                "kernel": "gemm_w8a8 (k_w8a8_pair, 4096x8192x28672 int8 ops)",
                "peak_source": "max(bf16 dense %s %.1f, torch._int_mm %s)" % (
                    peaks["source"], peaks["bf16_tflops"], "%.1f" % int8_ref if int8_ref else "n/a")}
    detail = {}
    for name in Step.names:
        b, f = bf[name]
        t = per_kernel[name]
        d = {"us": t * 1e6, "gbs": b / t / 1e9, "roofline_frac": roofline_seconds(b, f, peaks, int8_peak) / t}
        if f:
            d["tops"] = f / t / 1e12
        detail[name] = d
    w4_weight_bytes = N * K // 2 + N * (K // GROUP) * 2 + N * (K // GROUP) // 2
    detail["w4a16_decode_weight_gbs_m1"] = w4_weight_bytes / per_kernel["gemm_w4a16_m1"] / 1e9
    detail["w4a16_decode_frac_m1"] = detail["w4a16_decode_weight_gbs_m1"] / peaks["hbm_gbs"]

    # end to end through the C ABI with host buffers: every step copies its
    # activations in from pinned host memory and its outputs back.  Two
    # device buffer sets alternate, so the copies of step i+1's inputs (one
    # stream) and of step i-1's outputs (another stream) overlap step i.
    step.add_buffer_set()
    x_host = step.x.cpu().pin_memory()
    xs_host = [t.cpu().pin_memory() for t in step.xs]
    y8_host = torch.empty(step.y8.shape, dtype=step.y8.dtype).pin_memory()
    y4_host = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in step.y4]
    h2d = x_host.numel() * 2 + sum(t.numel() * 2 for t in xs_host)
    d2h = y8_host.numel() * 2 + sum(t.numel() * 2 for t in y4_host)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in_ready = [torch.cuda.Event() for _ in range(2)]
    ev_in_free = [torch.cuda.Event() for _ in range(2)]
    ev_out_ready = [torch.cuda.Event() for _ in range(2)]
    ev_out_free = [torch.cuda.Event() for _ in range(2)]

    def issue_h2d(i):
        b = i % 2
        x_d, xs_d, _, _ = step.sets[b]
        s_in.wait_event(ev_in_free[b])            # the step that last read set b is done
        with torch.cuda.stream(s_in):
            x_d.copy_(x_host, non_blocking=True)
            for d_, h_ in zip(xs_d, xs_host):
                d_.copy_(h_, non_blocking=True)
        ev_in_ready[b].record(s_in)

    def e2e_run(n):
        issue_h2d(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                issue_h2d(i + 1)
            stream.wait_event(ev_in_ready[b])
            stream.wait_event(ev_out_free[b])      # the outputs of step i-2 have left set b
            step.run(stream, buf=b)
            ev_in_free[b].record(stream)
            ev_out_ready[b].record(stream)
            s_out.wait_event(ev_out_ready[b])
            _, _, y8_d, y4_d = step.sets[b]
            with torch.cuda.stream(s_out):
                y8_host.copy_(y8_d, non_blocking=True)
                for h_, d_ in zip(y4_host, y4_d):
                    h_.copy_(d_, non_blocking=True)
            ev_out_free[b].record(s_out)
        stream.wait_stream(s_out)
        stream.wait_stream(s_in)

    e2e_run(3)
    stream.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    e2e_run(args.e2e_steps)
    e1.record(stream)
    stream.synchronize()
    e2e_t = max_over_ranks(e0.elapsed_time(e1) / 1e3 / args.e2e_steps, world, dev)
    e2e_value = world * 100.0 * t_roof / e2e_t
    # copy bandwidth alone (no compute), for the record
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(s_in)
    with torch.cuda.stream(s_in):
        for _ in range(3):
            step.sets[1][0].copy_(x_host, non_blocking=True)
    c1.record(s_in)
    s_in.synchronize()
    h2d_gbs = 3 * x_host.numel() * 2 / (c0.elapsed_time(c1) / 1e3) / 1e9

    configs = None
    if not args.no_configs:
        configs = measure_other_configs(dev, peaks, int8_peak)
        if qlin.qlin_device_error() != 0:
            raise RuntimeError("device-side error in the configuration measurements")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = cpu_threads()
        rows = cpu_rows(threads)
        sec = min(oracle_sample_seconds(rows, threads)[0] for _ in range(3))
        _, frac, sample = oracle_sample_seconds(rows, threads)
        sec1, _, _ = oracle_sample_seconds(rows, 1)
        cpu = {"value": 100.0 * frac * t_roof / sec, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": sample, "sample_seconds": sec, "sample_fraction": frac,
               "extrapolated_seconds_per_step": sec / frac,
               "single_thread": {"value": 100.0 * frac * t_roof / sec1, "sample_seconds": sec1, "cores": 1}}

    if rank == 0:
        out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
               "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "int8xint8->int32, bf16 (w4a16)",
               "data": "synthetic",
               "config": {"workload": "70B down-projection W[8192x28672]: per-token quantize of SmoothQuant-folded X + "
                                      "W8A8 M=4096 + W4A16 UINT4 g128 M=1/8/64/256 + dequantize",
                          "M_w8a8": M8, "N": N, "K": K, "w4_group": GROUP, "w4_M": list(W4_MS),
                          "l2": "every operand > L2 or read from a distinct copy (one packed W4 copy per call)",
                          "parallelism": "replicas" if world > 1 else "single GPU"},
               "roofline": roofline, "cpu_baseline": cpu,
               "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": e2e_t * 1e3, "steps": args.e2e_steps, "h2d_copy_gbs": h2d_gbs,
                       "overlap": "inputs of step i+1 and outputs of step i-1 copied on two side streams "
                                  "while step i computes (two device buffer sets)"},
               "gpu_launches": step.launches_per_step() * args.steps,
               "clocks": clock_info, "peaks": peaks, "int8_ref_tflops": int8_ref, "detail": detail,
               "configs": configs}
        print(json.dumps(out))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
