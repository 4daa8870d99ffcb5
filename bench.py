#!/usr/bin/env python3
"""Benchmark of the NVFP4 linear-layer path on B300.

One step = one training step of a 12B-class hybrid model's FFN
up-projection (8192 tokens, hidden 5120, FFN 20480), entirely through the
C ABI of libnvfp4:

  forward  (Y = X W^T):   amax X, 1x16 RNE quantise X; amax W, 16x16 RNE
                          quantise W emitting W and W^T; GEMM -> Y bf16
  dgrad    (dX = dY W):   amax dY, 1x16 Philox-SR quantise dY; GEMM with
                          W^T -> dX bf16
  wgrad    (dW = dY^T X): RHT-16 amax + RHT quantise of dY^T (SR) and X^T
                          (RNE), both read transposed (k = tokens); GEMM ->
                          dW bf16

Reported value: NVFP4 TFLOP/s of the whole step (3 GEMMs of 2*M*N*K each,
divided by the step time including all quantisation), plus GEMM-only
TFLOP/s and quantise GB/s (algorithmic bytes) measured with CUDA events on
the launching stream.  The step time is taken over replays of a CUDA graph of
the step's launches, captured once after the warm-up (--graph 0: eager
launches); the per-launch figures come from an eager pass with an event
around every launch.  L2 is flushed (256 MiB write) before every timed step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 GEMM TFLOPS and quantize GB/s (1×B300), % of roofline"
TOKENS, HIDDEN, FFN = 8192, 5120, 20480
GEMM_FLOPS = 2.0 * TOKENS * HIDDEN * FFN          # each of the three GEMMs
STEP_FLOPS = 3 * GEMM_FLOPS
SEED_X, SEED_W, SEED_DY = 2, 3, 3 + 7919
SR_SEED = 1003
RHT_SEED = 2004
WORKLOAD = ("linear-layer training step, 12B-hybrid FFN up-projection: X[8192x5120] "
            "W[20480x5120] dY[8192x20480]; fwd (1x16 RNE X, 16x16 W + W^T), dgrad (1x16 SR dY), "
            "wgrad (RHT-16 along tokens, SR dY^T, RNE X^T); bf16 outputs")

# algorithmic bytes per element (reads + writes) of each quantiser call: an
# amax reads 2 B; a 1x16 quantise reads 2 B and writes 0.5 B of codes and
# 1/16 B of scales; the 16x16 quantise with W^T and the dual-axis quantise
# read once and write two operands
B_AMAX, B_Q1D, B_Q2D_T, B_QDUAL = 2.0, 2.5625, 3.125, 3.125
# the dequantiser reads codes and scales (0.5625 B) and writes bf16 (2 B)
B_DEQ_BF16 = 2.5625
# dense FP4 tensor throughput of one B300 as NVIDIA lists it for HGX B300
# (108 PFLOP/s dense FP4 for 8 GPUs)
FP4_NOMINAL_TFLOPS = 13500.0


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6400.0, 1800.0, "fallback"


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [t.strip() for t in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                maxes.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms)}


# ------------------------------------------------------------- GPU step ----
class Step:
    """Device buffers and the launch sequence of one linear-layer step."""

    def __init__(self, nv, torch, host, path: str = "dual", sr_round=None, streams: int = 1):
        self.nv, self.torch = nv, torch
        self.sr_round = nv.NVFP4_SR if sr_round is None else sr_round
        # forward: the W chain (amax, 16x16 quantise) runs on a second stream beside
        # the X chain and joins the main stream before the forward GEMM
        self.side = torch.cuda.Stream() if (streams == 2 and path == "dual") else None
        self.fork = torch.cuda.Event()
        self.join = torch.cuda.Event()
        self.ev_start = torch.cuda.Event(enable_timing=True)
        self.ev_end = torch.cuda.Event(enable_timing=True)
        dev = "cuda"
        self.stream = torch.cuda.current_stream()
        self.x = torch.empty((TOKENS, HIDDEN), dtype=torch.bfloat16, device=dev)
        self.w = torch.empty((FFN, HIDDEN), dtype=torch.bfloat16, device=dev)
        self.dy = torch.empty((TOKENS, FFN), dtype=torch.bfloat16, device=dev)
        self.h2d(host)
        Q = nv.QTensor
        self.qx, self.qw, self.qwt = Q(TOKENS, HIDDEN), Q(FFN, HIDDEN, True), Q(HIDDEN, FFN, True)
        self.qdy, self.qdyt, self.qxt = Q(TOKENS, FFN), Q(FFN, TOKENS), Q(HIDDEN, TOKENS)
        self.amax = torch.empty((8,), dtype=torch.float32, device=dev)
        self.y = torch.empty((TOKENS, FFN), dtype=torch.bfloat16, device=dev)
        self.dx = torch.empty((TOKENS, HIDDEN), dtype=torch.bfloat16, device=dev)
        self.dw = torch.empty((FFN, HIDDEN), dtype=torch.bfloat16, device=dev)
        self.mask = nv.nvfp4_rht_mask_from_seed(RHT_SEED)
        self.flush_buf = torch.empty((256 << 20,), dtype=torch.uint8, device=dev)
        self.flush_rd = torch.zeros((256 << 20,), dtype=torch.uint8, device=dev)
        self.seq = self.phases(path)
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * len(self.seq))]
        self.launches_per_step = len(self.seq)

    def h2d(self, host):
        self.x.view(torch_int16(self.torch)).copy_(host["x"], non_blocking=True)
        self.w.view(torch_int16(self.torch)).copy_(host["w"], non_blocking=True)
        self.dy.view(torch_int16(self.torch)).copy_(host["dy"], non_blocking=True)

    def d2h(self, host):
        host["y"].copy_(self.y.view(torch_int16(self.torch)), non_blocking=True)
        host["dx"].copy_(self.dx.view(torch_int16(self.torch)), non_blocking=True)
        host["dw"].copy_(self.dw.view(torch_int16(self.torch)), non_blocking=True)

    def run_e2e(self, host):
        """One step end to end from and to pinned host buffers.  Uploads run on
        a copy-in stream and downloads on a copy-out stream, beside the compute
        on the main stream: X and W go up first, and dY's upload overlaps the
        forward pass; Y comes down once the forward GEMM is done, overlapping
        the backward pass; dX and dW come down at the end.  Every byte crosses
        inside the step; the main stream ends after the last download."""
        torch = self.torch
        main = torch.cuda.current_stream()
        i16 = torch_int16(torch)
        if not hasattr(self, "copy_in"):
            self.copy_in, self.copy_out = torch.cuda.Stream(), torch.cuda.Stream()
        cin, cout = self.copy_in, self.copy_out
        ev = [torch.cuda.Event() for _ in range(6)]
        ev[0].record(main)
        cin.wait_event(ev[0])
        with torch.cuda.stream(cin):
            self.x.view(i16).copy_(host["x"], non_blocking=True)
            self.w.view(i16).copy_(host["w"], non_blocking=True)
            ev[1].record(cin)
            self.dy.view(i16).copy_(host["dy"], non_blocking=True)
            ev[2].record(cin)
        split = [p[0] for p in self.seq].index("gemm_fwd") + 1
        main.wait_event(ev[1])
        for _, call, _, _ in self.seq[:split]:
            call()
        ev[3].record(main)
        cout.wait_event(ev[3])
        with torch.cuda.stream(cout):
            host["y"].copy_(self.y.view(i16), non_blocking=True)
        main.wait_event(ev[2])
        for _, call, _, _ in self.seq[split:]:
            call()
        ev[4].record(main)
        cout.wait_event(ev[4])
        with torch.cuda.stream(cout):
            host["dx"].copy_(self.dx.view(i16), non_blocking=True)
            host["dw"].copy_(self.dw.view(i16), non_blocking=True)
            ev[5].record(cout)
        main.wait_event(ev[5])

    def flush_l2(self):
        """Untimed preamble of a step: overwrite 256 MiB (> 126 MB of L2), then
        read another 256 MiB, so that the timed region starts with an L2 that
        holds none of its inputs and none of the flush's own dirty lines (whose
        write-back would otherwise share HBM with the first timed kernel); then
        hold the stream in a short device spin so the host enqueues the whole
        step before the GPU reaches it (launch gaps then never enter the
        events' intervals)."""
        self.flush_buf.fill_(1)
        self.flush_sink = self.flush_rd.sum(dtype=self.torch.int32)
        self.torch.cuda._sleep(3_000_000)

    def phases(self, path: str):
        """The launch sequence of one step: (name, call, algorithmic bytes,
        is_gemm).  "dual": X and dY are each read once for both of their
        operands (dual-axis amax and quantise); "separate": every operand by
        its own amax and quantiser call."""
        nv, a = self.nv, self.amax
        rne, sr = nv.NVFP4_RNE, self.sr_round
        x, w, dy = TOKENS * HIDDEN, FFN * HIDDEN, TOKENS * FFN
        fwd_w = [("amax_w", lambda: nv.nvfp4_amax(self.w, 0, a[1:2]), w * B_AMAX, False),
                 ("q2d_w", lambda: nv.nvfp4_quantize_2d(self.w, a[1:2], rne, 0, 0, self.qw, self.qwt),
                  w * B_Q2D_T, False)]
        gemm_fwd = ("gemm_fwd", lambda: nv.nvfp4_gemm(self.qx, self.qw, self.y), 0, True)
        gemm_dgrad = ("gemm_dgrad", lambda: nv.nvfp4_gemm(self.qdy, self.qwt, self.dx), 0, True)
        gemm_wgrad = ("gemm_wgrad", lambda: nv.nvfp4_gemm(self.qdyt, self.qxt, self.dw), 0, True)
        if path == "dual":
            # the W chain first (on the side stream when there is one), then the X chain
            return [
                *fwd_w,
                ("amax_dual_x", lambda: nv.nvfp4_amax_dual(self.x, self.mask, a[0:1], a[4:5]), x * B_AMAX, False),
                ("quant_dual_x", lambda: nv.nvfp4_quantize_dual(self.x, a[0:1], rne, 0, 0, self.qx, self.mask,
                                                                a[4:5], rne, 0, 0, self.qxt), x * B_QDUAL, False),
                gemm_fwd,
                ("amax_dual_dy", lambda: nv.nvfp4_amax_dual(self.dy, self.mask, a[2:3], a[3:4]), dy * B_AMAX, False),
                ("quant_dual_dy", lambda: nv.nvfp4_quantize_dual(self.dy, a[2:3], sr, SR_SEED, 1, self.qdy, self.mask,
                                                                 a[3:4], sr, SR_SEED, 2, self.qdyt), dy * B_QDUAL, False),
                gemm_dgrad, gemm_wgrad]
        return [
            ("amax_x", lambda: nv.nvfp4_amax(self.x, 0, a[0:1]), x * B_AMAX, False),
            ("q1d_x", lambda: nv.nvfp4_quantize_1d(self.x, a[0:1], rne, 0, 0, self.qx), x * B_Q1D, False),
            *fwd_w, gemm_fwd,
            ("amax_dy", lambda: nv.nvfp4_amax(self.dy, 0, a[2:3]), dy * B_AMAX, False),
            ("q1d_dy_sr", lambda: nv.nvfp4_quantize_1d(self.dy, a[2:3], sr, SR_SEED, 1, self.qdy), dy * B_Q1D, False),
            gemm_dgrad,
            # wgrad: k = tokens, both operands read transposed, RHT-16 along k
            ("amax_rht_dyt", lambda: nv.nvfp4_amax(self.dy, self.mask, a[3:4], transposed=True), dy * B_AMAX, False),
            ("rhtq_dyt_sr", lambda: nv.nvfp4_rht_quantize(self.dy, self.mask, a[3:4], sr, SR_SEED, 2, self.qdyt,
                                                          transposed=True), dy * B_Q1D, False),
            ("amax_rht_xt", lambda: nv.nvfp4_amax(self.x, self.mask, a[4:5], transposed=True), x * B_AMAX, False),
            ("rhtq_xt", lambda: nv.nvfp4_rht_quantize(self.x, self.mask, a[4:5], rne, 0, 0, self.qxt,
                                                      transposed=True), x * B_Q1D, False),
            gemm_wgrad]

    def run(self, timed: bool):
        """Enqueue one step.  With a side stream, the W-chain launches (amax_w,
        q2d_w) go to it after a fork event from the main stream, and the main
        stream waits for them before the forward GEMM; the step is timed by
        events on the main stream around everything."""
        torch, ev = self.torch, self.ev
        main = torch.cuda.current_stream()
        if timed:
            self.ev_start.record(main)
        if self.side is not None:
            self.fork.record(main)
            self.side.wait_event(self.fork)
        for j, (name, call, _, _) in enumerate(self.seq):
            s = self.side if (self.side is not None and name in ("amax_w", "q2d_w")) else main
            if name == "gemm_fwd" and self.side is not None:
                self.join.record(self.side)
                main.wait_event(self.join)
            with torch.cuda.stream(s):
                if timed:
                    ev[2 * j].record(s)
                call()
                if timed:
                    ev[2 * j + 1].record(s)
        if timed:
            self.ev_end.record(main)

    def phase_times(self):
        """ms of each launch of the last timed step."""
        return [self.ev[2 * j].elapsed_time(self.ev[2 * j + 1]) for j in range(len(self.seq))]


# single calls of the step, for kernel-level profiling (bench.py --profile-case)
PROFILE_CASES = {
    "gemm_fwd": lambda s: s.nv.nvfp4_gemm(s.qx, s.qw, s.y),
    "gemm_dgrad": lambda s: s.nv.nvfp4_gemm(s.qdy, s.qwt, s.dx),
    "gemm_wgrad": lambda s: s.nv.nvfp4_gemm(s.qdyt, s.qxt, s.dw),
    "amax_dy": lambda s: s.nv.nvfp4_amax(s.dy, 0, s.amax[2:3]),
    "q1d_x": lambda s: s.nv.nvfp4_quantize_1d(s.x, s.amax[0:1], s.nv.NVFP4_RNE, 0, 0, s.qx),
    "q1d_dy_sr": lambda s: s.nv.nvfp4_quantize_1d(s.dy, s.amax[2:3], s.nv.NVFP4_SR, SR_SEED, 1, s.qdy),
    "q2d_w": lambda s: s.nv.nvfp4_quantize_2d(s.w, s.amax[1:2], s.nv.NVFP4_RNE, 0, 0, s.qw, s.qwt),
    "rhtq_dyt_sr": lambda s: s.nv.nvfp4_rht_quantize(s.dy, s.mask, s.amax[3:4], s.nv.NVFP4_SR,
                                                      SR_SEED, 2, s.qdyt, transposed=True),
    "amax_rht_dyt": lambda s: s.nv.nvfp4_amax(s.dy, s.mask, s.amax[3:4], transposed=True),
    "amax_dual_dy": lambda s: s.nv.nvfp4_amax_dual(s.dy, s.mask, s.amax[2:3], s.amax[3:4]),
    "quant_dual_dy": lambda s: s.nv.nvfp4_quantize_dual(s.dy, s.amax[2:3], s.nv.NVFP4_SR, SR_SEED, 1, s.qdy, s.mask,
                                                        s.amax[3:4], s.nv.NVFP4_SR, SR_SEED, 2, s.qdyt),
    "quant_dual_dy_hw": lambda s: s.nv.nvfp4_quantize_dual(s.dy, s.amax[2:3], s.nv.NVFP4_SR_HW, SR_SEED, 1, s.qdy,
                                                           s.mask, s.amax[3:4], s.nv.NVFP4_SR_HW, SR_SEED, 2, s.qdyt),
    "quant_dual_x": lambda s: s.nv.nvfp4_quantize_dual(s.x, s.amax[0:1], s.nv.NVFP4_RNE, 0, 0, s.qx, s.mask,
                                                       s.amax[4:5], s.nv.NVFP4_RNE, 0, 0, s.qxt),
    # the library GEMM of the comparison (cuBLASLt through torch) on the forward operands
    "gemm_fwd_library": lambda s: library_gemm_call(s, s.qx, s.qw)(),
    "dequantize_x": lambda s: s.nv.nvfp4_dequantize(s.qx, dequant_out(s)),
}


def dequant_out(step):
    """The bf16 [tokens x hidden] output of the dequantiser's profile case,
    allocated on first use."""
    if not hasattr(step, "deq_out"):
        step.deq_out = step.torch.empty((TOKENS, HIDDEN), dtype=step.torch.bfloat16, device="cuda")
    return step.deq_out


def library_gemm_call(step, a, b):
    """cuBLASLt's NVFP4 GEMM (torch.nn.functional.scaled_mm, 1x16 E4M3 block
    scales in the same swizzled layout) of two quantised operands, bf16 out,
    as a callable.  Block scales only: the tensor scales (alpha) are left
    out, which does not change the work."""
    import torch
    import torch.nn.functional as F
    A = a.codes.view(torch.float4_e2m1fn_x2)
    B = b.codes.view(torch.float4_e2m1fn_x2).t()
    sa, sb = a.scales.view(torch.float8_e4m3fn), b.scales.view(torch.float8_e4m3fn)
    return lambda: F.scaled_mm(A, B, sa, F.ScalingType.BlockWise1x16, sb, F.ScalingType.BlockWise1x16,
                               F.SwizzleType.SWIZZLE_32_4_4, F.SwizzleType.SWIZZLE_32_4_4,
                               output_dtype=torch.bfloat16)


def torch_int16(torch):
    return torch.int16


def input_digests(**arrays) -> dict:
    """sha256 of each synthetic input's bytes (bf16 bit patterns), so a run's
    inputs can be matched against any other run's."""
    import hashlib
    return {k: hashlib.sha256(np.ascontiguousarray(v).tobytes()).hexdigest() for k, v in arrays.items()}


def make_host_inputs():
    import synth
    x = synth.activations(SEED_X)
    w = synth.weights(SEED_W)
    dy = synth.grad_output(SEED_DY)
    return x, w, dy


# ----------------------------------------------------------- CPU oracle ----
def oracle_step_sample(threads: int | None = None, rows: int = 16, pts: int = 256):
    """Time the CPU oracle on a bounded sample of the step and extrapolate
    to one full step.  Sample: `rows` rows of every quantised operand (of the
    8192..20480 rows) and `pts` output points of each GEMM (full K)."""
    import oracle
    import synth

    rng = np.random.default_rng(0)
    x = synth.activations(SEED_X, tokens=rows * 64)           # shape-compatible slices
    w = synth.weights(SEED_W, ffn=rows * 64)
    dy = synth.grad_output(SEED_DY, tokens=rows * 64)
    mask = oracle.rht_mask_from_seed(RHT_SEED)
    thr = threads or oracle.default_threads()
    t_quant = 0.0
    # (name, array, transposed, block2d, rht, sr, logical rows of the full tensor)
    jobs = [("X", x, False, False, 0, False, TOKENS), ("W", w, False, True, 0, False, FFN),
            ("dY", dy, False, False, 0, True, TOKENS), ("dYt", dy, True, False, mask, True, FFN),
            ("Xt", x, True, False, mask, False, HIDDEN)]
    for name, arr, tr, b2, m, s, full_rows in jobs:
        k_full = TOKENS if tr else (HIDDEN if name in ("X", "W") else FFN)
        k_here = arr.shape[0] if tr else arr.shape[1]
        t0 = time.perf_counter()
        am = oracle.amax(arr, tr, m)                       # whole slice, one thread
        t_amax = time.perf_counter() - t0
        t0 = time.perf_counter()
        oracle.quantize(arr, transposed=tr, rht_mask=m, block2d=b2, amax_v=am, sr=s, seed=SR_SEED,
                        threads=thr, rows_range=(0, rows))
        t_q = time.perf_counter() - t0
        full_elems = full_rows * k_full
        t_quant += t_amax * full_elems / arr.size + t_q * full_elems / (rows * k_here)
    t_gemm = 0.0
    for (M, N, K) in [(TOKENS, FFN, HIDDEN), (TOKENS, HIDDEN, FFN), (FFN, HIDDEN, TOKENS)]:
        ca, sa = synth.random_operand(64, K, 1)
        cb, sb = synth.random_operand(64, K, 2)
        ms = rng.integers(0, 64, pts)
        ns = rng.integers(0, 64, pts)
        swa, swb = oracle.swizzle_scales(sa, 64, K), oracle.swizzle_scales(sb, 64, K)
        t0 = time.perf_counter()
        oracle.gemm_points(ca, swa, 1.0, cb, swb, 1.0, 64, 64, K, ms, ns, threads=thr)
        t_gemm += (time.perf_counter() - t0) * (M * N) / pts
    t_step = t_quant + t_gemm
    q_bytes = (TOKENS * HIDDEN * 2 + FFN * HIDDEN + TOKENS * FFN * 2) * (B_AMAX + B_Q1D)
    return {"value": STEP_FLOPS / t_step / 1e12, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
            "sample": f"{rows} rows of each of the 5 quantised operands (amax over a {rows * 64}-row "
                      f"slice) and {pts} output points of each of the 3 GEMMs (full K), "
                      "extrapolated by element and output counts to one step",
            "quantize_gbs": q_bytes / t_quant / 1e9, "gemm_tflops": 3 * GEMM_FLOPS / t_gemm / 1e12,
            "seconds_per_step_extrapolated": t_step}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    t0 = time.perf_counter()
    vals = []
    for _ in range(args.warmup + args.steps):
        vals.append(oracle_step_sample())
    vals = vals[args.warmup:]
    v = statistics.median([c["value"] for c in vals])
    sec = statistics.median([c["seconds_per_step_extrapolated"] for c in vals])
    wall = time.perf_counter() - t0
    out = {"metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
           "impl": "reference",
           # the oracle cannot run a whole step in bench time: each timed step is a bounded
           # sample, and ms_per_step is the sample's time scaled by element and output counts
           "extrapolated": True,
           "sample_seconds_per_step": wall / max(1, args.warmup + args.steps),
           "config": main_config(args),
           "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": vals[0]["cores"], "kind": "oracle",
                            "sample": vals[0]["sample"], "quantize_gbs": vals[0]["quantize_gbs"],
                            "gemm_tflops": vals[0]["gemm_tflops"]},
           "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "wall_s": wall}
    print(json.dumps(out))
    return 0


def main_config(args, side_stream: bool = False) -> dict:
    """The `config` object of the JSON line (the same keys for both arms)."""
    return {"workload": WORKLOAD, "tokens": TOKENS, "hidden": HIDDEN, "ffn": FFN,
            "path": args.path,
            "streams": ("2: forward W chain on a second stream beside the X chain; phase_ms overlap"
                        if side_stream else "1"),
            "sr": ("NVFP4_SR_HW: random bits in the hardware SR conversion's layout" if args.sr == "hw"
                   else "NVFP4_SR: 16 independent Philox4x32-10 bits per element"),
            "l2": "flushed before each step, untimed: 256 MiB device write, then 256 MiB read (no dirty flush lines left)",
            "launch": ("CUDA graph of the step's launches, captured once and replayed each step"
                       if getattr(args, "graph", 0) else "eager launches"),
            "parallelism": f"replicas x{args.gpus}"}


# -------------------------------------------------------------------- main --
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-mx", action="store_true", help="skip the MXFP4 comparison timing")
    ap.add_argument("--no-sweep", action="store_true", help="skip the quantise-only sweep (2^20..2^30)")
    ap.add_argument("--path", default="dual", choices=["dual", "separate"],
                    help="dual: X and dY read once each for both operands; separate: one call per operand")
    ap.add_argument("--streams", type=int, default=1, choices=[1, 2],
                    help="2: the forward W chain (amax, 16x16 quantise) on a second stream beside the X chain "
                         "(dual path only; the persistent kernels each fill the GPU, so the gain is small)")
    ap.add_argument("--sr", default="philox16", choices=["philox16", "hw"],
                    help="rounding of dY: philox16 = NVFP4_SR (16 independent Philox bits per element), "
                         "hw = NVFP4_SR_HW (random bits in the hardware SR conversion's layout)")
    ap.add_argument("--graph", type=int, default=1, choices=[0, 1],
                    help="1: time the step as a CUDA graph of its launches, captured once after the warm-up "
                         "and replayed (per-launch figures still come from an eager pass); 0: eager launches")
    ap.add_argument("--profile-case", default=None, choices=sorted(PROFILE_CASES),
                    help="after one full untimed step, launch only this call --steps times "
                         "(a target for ncu -k; prints nothing)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    import nvfp4_block_scaled_29_b300 as nv

    xh, wh, dyh = make_host_inputs()
    digests = input_digests(x=xh, w=wh, dy=dyh)
    host = {"x": torch.from_numpy(xh.view(np.int16)).pin_memory(),
            "w": torch.from_numpy(wh.view(np.int16)).pin_memory(),
            "dy": torch.from_numpy(dyh.view(np.int16)).pin_memory()}
    host["y"] = torch.empty((TOKENS, FFN), dtype=torch.int16).pin_memory()
    host["dx"] = torch.empty((TOKENS, HIDDEN), dtype=torch.int16).pin_memory()
    host["dw"] = torch.empty((FFN, HIDDEN), dtype=torch.int16).pin_memory()
    step = Step(nv, torch, host, args.path, nv.NVFP4_SR_HW if args.sr == "hw" else nv.NVFP4_SR, args.streams)
    gemm_idx = [j for j, p in enumerate(step.seq) if p[3]]
    quant_idx = [j for j, p in enumerate(step.seq) if not p[3]]
    torch.cuda.synchronize()
    if args.profile_case:
        step.run(timed=False)
        for _ in range(args.steps):
            PROFILE_CASES[args.profile_case](step)
        torch.cuda.synchronize()
        st = nv.nvfp4_get_status()
        if st != nv.NVFP4_OK:
            raise SystemExit(f"device status: {nv.status_string(st)}")
        return 0

    for _ in range(max(3, args.warmup)):
        step.flush_l2()
        step.run(timed=False)
    torch.cuda.synchronize()
    st = nv.nvfp4_get_status()
    if st != nv.NVFP4_OK:
        raise SystemExit(f"device status after warm-up: {nv.status_string(st)}")

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # the step as a CUDA graph: the same launches on the same buffers, captured once
    graph = None
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step.run(timed=False)
        torch.cuda.synchronize()
        for _ in range(max(3, args.warmup)):
            step.flush_l2()
            graph.replay()
        torch.cuda.synchronize()
        st = nv.nvfp4_get_status()
        if st != nv.NVFP4_OK:
            raise SystemExit(f"device status after the graph warm-up: {nv.status_string(st)}")

    # ---- device-resident timed region: K eager steps with an event around
    # every launch (the per-launch figures), then, with --graph 1, K replays of
    # the step's graph (the step time)
    step_ms, gemm_ms, quant_ms = [], [], []
    graph_ms = []
    with ClockSampler(local) as clk:
        barrier()
        for _ in range(args.steps):
            step.flush_l2()
            step.run(timed=True)
            torch.cuda.synchronize()
            ph = step.phase_times()
            step_ms.append(step.ev_start.elapsed_time(step.ev_end))
            gemm_ms.extend(ph[j] for j in gemm_idx)
            quant_ms.append(sum(ph[j] for j in quant_idx))
        barrier()
        if graph is not None:
            main_stream = torch.cuda.current_stream()
            for _ in range(args.steps):
                step.flush_l2()
                step.ev_start.record(main_stream)
                graph.replay()
                step.ev_end.record(main_stream)
                torch.cuda.synchronize()
                graph_ms.append(step.ev_start.elapsed_time(step.ev_end))
            barrier()
    eager_total_ms = sum(step_ms)
    total_ms = sum(graph_ms) if graph is not None else eager_total_ms
    if world > 1:
        t = torch.tensor([total_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    st = nv.nvfp4_get_status()
    if st != nv.NVFP4_OK:
        raise SystemExit(f"device status after timing: {nv.status_string(st)}")

    # ---- end to end through the C ABI with host buffers
    e2e_ms = []
    h2d_bytes = sum(host[k].numel() * 2 for k in ("x", "w", "dy"))
    d2h_bytes = sum(host[k].numel() * 2 for k in ("y", "dx", "dw"))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    for _ in range(args.e2e_steps):
        step.flush_l2()
        e0.record()
        step.run_e2e(host)
        e1.record()
        torch.cuda.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    barrier()
    e2e_avg = statistics.mean(e2e_ms)
    if world > 1:
        t = torch.tensor([e2e_avg], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_avg = float(t.item())

    hbm_peak, bf16_peak, peak_src = load_peaks()
    fp4_peak = bf16_peak * 6.0        # dense FP4 : BF16 = 13.5 : 2.25 (nominal)
    ms_per_step = total_ms / args.steps
    eager_ms_per_step = eager_total_ms / args.steps
    gemm_avg_ms = statistics.mean(gemm_ms)
    gemm_tflops = GEMM_FLOPS / (gemm_avg_ms * 1e-3) / 1e12
    qbytes = sum(step.seq[j][2] for j in quant_idx)
    quant_gbs = qbytes / (statistics.mean(quant_ms) * 1e-3) / 1e9
    traffic = load_traffic()
    out = {
        "metric": METRIC,
        "value": world * STEP_FLOPS / (ms_per_step * 1e-3) / 1e12,
        "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "eager_ms_per_step": eager_ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp4-e2m1 x e4m3-scaled, fp32 accumulate (bf16 in/out)",
        "data": "synthetic (seeded N(0,1)+outliers, N(0,0.02^2), 1e-3*t3)",
        "inputs_sha256": digests,
        "config": main_config(args, step.side is not None),
        "gemm_tflops": gemm_tflops,
        "quantize_gbs": quant_gbs,
        "roofline": {"bound": "tensor", "achieved": gemm_tflops, "peak": fp4_peak, "unit": "TFLOP/s",
                     "frac": gemm_tflops / fp4_peak, "traffic": traffic.get("gemm_fwd"),
                     "peak_nominal": FP4_NOMINAL_TFLOPS, "frac_nominal": gemm_tflops / FP4_NOMINAL_TFLOPS,
                     "traffic_note": "forward-GEMM launch (8192x20480x5120); achieved is the mean of the 3 GEMMs",
                     "kernel": "k_gemm_nvfp4_2sm",
                     "peak_source": f"{peak_src} bf16 burst {bf16_peak} TFLOP/s x 6 (nominal dense FP4:BF16)"},
        "roofline_quantize": {"bound": "hbm", "achieved": quant_gbs, "peak": hbm_peak, "unit": "GB/s",
                              "frac": quant_gbs / hbm_peak,
                              "traffic": traffic.get(("quant_dual_dy_hw" if args.sr == "hw" else "quant_dual_dy")
                                                     if args.path == "dual" else "quant_sr_dy"),
                              "traffic_note": ("dual-axis SR quantise of dY (one launch)" if args.path == "dual"
                                               else "1x16 SR quantise of dY (one launch)"),
                              "peak_source": f"{peak_src} HBM copy"},
        "phase_ms": dict(zip([p[0] for p in step.seq], [round(v, 4) for v in step.phase_times()])),
        "e2e": {"value": world * STEP_FLOPS / (e2e_avg * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
                "ms_per_step": e2e_avg,
                "copies": "pinned host buffers; uploads and downloads on their own streams, dY's upload "
                          "overlapping the forward pass and Y's download the backward pass"},
        "gpu_launches": step.launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_mx:
        out["mxfp4"] = time_mxfp4(nv, torch, step)
        out["autograd"] = time_autograd(torch, step)
        if args.path == "dual" and args.sr == "philox16":
            out["sr_hw"] = time_sr_hw(nv, torch, step, out["phase_ms"], eager_ms_per_step)
    if world == 1:
        out["calls"] = time_calls(nv, torch, step, hbm_peak)
        out["library_gemm"] = time_library_gemm(torch, step)
        if not args.no_sweep:
            out["sweep"] = time_sweep(nv, torch, step, hbm_peak)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = oracle_step_sample(rows=96, pts=2048)
        out["cpu_baseline"].pop("seconds_per_step_extrapolated", None)
        one = oracle_step_sample(threads=1, rows=16, pts=256)
        out["cpu_baseline"]["single_thread"] = {k: one[k] for k in ("value", "quantize_gbs", "gemm_tflops",
                                                                      "cores", "sample")}
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        dist.destroy_process_group()
    return 0


def time_autograd(torch, step, reps: int = 10) -> dict:
    """The same training step through the autograd NVFP4 linear layer
    (forward + backward of NVFP4LinearFunction at the step's shapes), timed
    with CUDA events after an L2 flush."""
    import statistics as st
    from nvfp4_block_scaled_29_b300.linear import NVFP4LinearFunction
    x = step.x.detach().clone().requires_grad_(True)
    w = step.w.detach().clone().requires_grad_(True)
    dy = step.dy

    def once():
        y = NVFP4LinearFunction.apply(x, w, SR_SEED, step.mask)
        y.backward(dy)

    once()
    ts = []
    for _ in range(reps):
        x.grad = None
        w.grad = None
        step.flush_l2()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(); once(); e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    ms = st.median(ts)
    return {"ms_per_step": round(ms, 4), "tflops": STEP_FLOPS / (ms * 1e-3) / 1e12}


def time_sr_hw(nv, torch, step, phase_ms: dict, ms_per_step: float, reps: int = 10) -> dict:
    """The dual-axis quantise of dY with rounding mode NVFP4_SR_HW (the same
    rule, random bits in the hardware SR conversion's layout), CUDA events
    after an L2 flush, and the step time with that phase in place of the
    NVFP4_SR one."""
    import statistics as st
    a = step.amax

    def once():
        nv.nvfp4_quantize_dual(step.dy, a[2:3], nv.NVFP4_SR_HW, SR_SEED, 1, step.qdy, step.mask, a[3:4],
                               nv.NVFP4_SR_HW, SR_SEED, 2, step.qdyt)

    once()
    ts = []
    for _ in range(reps):
        step.flush_l2()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(); once(); e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    q_ms = st.median(ts)
    ms = ms_per_step - phase_ms["quant_dual_dy"] + q_ms
    return {"quant_dual_dy_ms": round(q_ms, 4), "step_ms": round(ms, 4),
            "step_tflops": STEP_FLOPS / (ms * 1e-3) / 1e12}


def time_mxfp4(nv, torch, step, reps: int = 10) -> dict:
    """The MXFP4 comparison path at the step's shapes: 1x32 quantise of X and
    dY (CUDA events, L2 flushed before each call) and the three GEMMs on
    MXFP4 operands of the forward, dgrad and wgrad shapes (operands made once,
    untimed)."""
    import statistics as st
    Q = nv.MxQTensor
    ops = {"x": (step.x, Q(TOKENS, HIDDEN)), "w": (step.w, Q(FFN, HIDDEN)), "dy": (step.dy, Q(TOKENS, FFN)),
           "wt": (step.w.t().contiguous(), Q(HIDDEN, FFN)), "dyt": (step.dy.t().contiguous(), Q(FFN, TOKENS)),
           "xt": (step.x.t().contiguous(), Q(HIDDEN, TOKENS))}
    for t, q in ops.values():
        nv.nvfp4_mx_quantize(t, 0, q)

    def timed(fn):
        ts = []
        for _ in range(reps):
            step.flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(); fn(); e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return st.median(ts)

    q_ms = {n: timed(lambda n=n: nv.nvfp4_mx_quantize(ops[n][0], 0, ops[n][1])) for n in ("x", "dy")}
    g_ms = [timed(lambda a=a, b=b, d=d: nv.nvfp4_mx_gemm(ops[a][1], ops[b][1], d))
            for a, b, d in (("x", "w", step.y), ("dy", "wt", step.dx), ("dyt", "xt", step.dw))]
    qbytes = {"x": TOKENS * HIDDEN, "dy": TOKENS * FFN}
    return {"gemm_ms": [round(v, 4) for v in g_ms],
            "gemm_tflops": GEMM_FLOPS / (st.mean(g_ms) * 1e-3) / 1e12,
            "quantize_ms": {n: round(v, 4) for n, v in q_ms.items()},
            "quantize_gbs": sum(qbytes[n] * (2 + 0.5 + 1 / 32) for n in q_ms) / (sum(q_ms.values()) * 1e-3) / 1e9}


def _timed_median(torch, step, fn, reps: int = 5) -> float:
    """Median CUDA-event time (ms) of fn() on the current stream, L2 flushed
    before each repetition."""
    fn()
    ts = []
    for _ in range(reps):
        step.flush_l2()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(); fn(); e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def time_calls(nv, torch, step, hbm_peak: float, reps: int = 5) -> dict:
    """Every call of the C ABI at the step's shapes, one at a time (L2
    flushed, median of `reps`): the separate-call path of the step (one amax
    and one quantiser per operand, the wgrad operands read transposed with
    the RHT), the dual-axis calls, the dequantiser and the three GEMMs.
    GB/s are algorithmic bytes over time; fractions are of the HBM peak."""
    rows = {}
    calls = step.phases("separate") + [p for p in step.phases("dual") if p[0].startswith(("amax_dual", "quant_dual"))]
    deq = torch.empty((TOKENS, HIDDEN), dtype=torch.bfloat16, device="cuda")
    calls.append(("dequantize_x", lambda: step.nv.nvfp4_dequantize(step.qx, deq), TOKENS * HIDDEN * B_DEQ_BF16,
                  False))
    for name, call, nbytes, is_gemm in calls:
        ms = _timed_median(torch, step, call, reps)
        if is_gemm:
            t = GEMM_FLOPS / (ms * 1e-3) / 1e12
            rows[name] = {"ms": round(ms, 4), "tflops": round(t, 1)}
        else:
            g = nbytes / (ms * 1e-3) / 1e9
            rows[name] = {"ms": round(ms, 4), "gbs": round(g, 1), "frac_hbm": round(g / hbm_peak, 3)}
    # reference for the write-dominated dequantiser: torch's fill kernel
    # writing the same 84 MB output (a write-only stream runs well below the
    # copy bandwidth on this part)
    wbytes = TOKENS * HIDDEN * 2
    ms = _timed_median(torch, step, lambda: deq.fill_(1.0), reps)
    g = wbytes / (ms * 1e-3) / 1e9
    rows["write_ref_x"] = {"ms": round(ms, 4), "gbs": round(g, 1), "frac_hbm": round(g / hbm_peak, 3),
                           "kernel": "torch fill_ (library), 84 MB bf16 write"}
    d = rows["dequantize_x"]
    d["write_gbs"] = round(wbytes / (d["ms"] * 1e-3) / 1e9, 1)
    d["frac_of_write_ref"] = round(d["write_gbs"] / g, 3)
    st = nv.nvfp4_get_status()
    if st != nv.NVFP4_OK:
        raise SystemExit(f"device status after the per-call timing: {nv.status_string(st)}")
    return rows


def time_library_gemm(torch, step, reps: int = 5) -> dict:
    """cuBLASLt's NVFP4 GEMM (through torch.nn.functional.scaled_mm, 1x16
    E4M3 block scales in the same swizzled layout) on the step's quantised
    operands, as a library comparison beside nvfp4_gemm.  Block scales only:
    the tensor scales (alpha) are left out, which does not change the work."""
    out = {}
    try:
        for name, a, b in (("fwd", step.qx, step.qw), ("dgrad", step.qdy, step.qwt), ("wgrad", step.qdyt, step.qxt)):
            ms = _timed_median(torch, step, library_gemm_call(step, a, b), reps)
            out[name] = {"ms": round(ms, 4), "tflops": round(GEMM_FLOPS / (ms * 1e-3) / 1e12, 1)}
        out["mean_tflops"] = round(statistics.mean(v["tflops"] for v in out.values()), 1)
        out["library"] = "cuBLASLt NVFP4 block-scaled GEMM via torch.nn.functional.scaled_mm"
    except Exception as e:                        # a torch without NVFP4 scaled_mm
        out = {"unavailable": f"{type(e).__name__}: {str(e)[:200]}"}
    return out


def time_sweep(nv, torch, step, hbm_peak: float, reps: int = 5) -> dict:
    """The quantise-only sweep: bf16 tensors of n = 2^20 .. 2^30 elements as
    [n/8192 x 8192], Student-t(3) (unscaled) and N(0,1) with 0.05% of the
    entries x100, quantised in every combination of {1x16, 16x16} x
    {RNE, NVFP4_SR} x {no RHT, RHT-16}: amax GB/s (2 B/element) per (size,
    RHT), quantise GB/s (amax given, 2.5625 B/element) per point, each the
    median of `reps` L2-flushed launches.  Inputs are drawn on the device
    (seeded) because the host generators take minutes at 2^30; the n-element
    tensor is the first n/8192 rows of the 2^30-element one."""
    import synth
    K = 8192
    rows_max = (1 << 30) // K
    amax = torch.empty((2,), dtype=torch.float32, device="cuda")
    cols = ["log2_n", "dist", "block", "round", "rht", "quant_ms", "quant_gbs", "quant_frac",
            "amax_ms", "amax_gbs", "amax_quant_gbs"]
    out_rows = []
    for dist in ("t3", "normal_outliers"):
        x = (synth.student_t_bf16_device((rows_max, K), 5, 1.0) if dist == "t3"
             else synth.normal_bf16_device((rows_max, K), 105, 1.0, 0.0005, 100.0))
        for e in range(20, 31):
            n = 1 << e
            v = x[: n // K]
            t_amax = {}
            for rht in (False, True):
                m = step.mask if rht else 0
                t_amax[rht] = _timed_median(torch, step, lambda: nv.nvfp4_amax(v, m, amax[0:1]), reps)
            for block2d in (False, True):
                q = nv.QTensor(n // K, K, block2d)
                for sr in (False, True):
                    rnd = nv.NVFP4_SR if sr else nv.NVFP4_RNE
                    for rht in (False, True):
                        m = step.mask if rht else 0
                        nv.nvfp4_amax(v, m, amax[0:1])
                        if rht:
                            f = lambda: nv.nvfp4_rht_quantize(v, m, amax[0:1], rnd, SR_SEED, 1, q)
                        elif block2d:
                            f = lambda: nv.nvfp4_quantize_2d(v, amax[0:1], rnd, SR_SEED, 1, q)
                        else:
                            f = lambda: nv.nvfp4_quantize_1d(v, amax[0:1], rnd, SR_SEED, 1, q)
                        tq = _timed_median(torch, step, f, reps)
                        gq = n * B_Q1D / (tq * 1e-3) / 1e9
                        ga = n * B_AMAX / (t_amax[rht] * 1e-3) / 1e9
                        both = n * (B_AMAX + B_Q1D) / ((tq + t_amax[rht]) * 1e-3) / 1e9
                        out_rows.append([e, dist, "16x16" if block2d else "1x16", "SR" if sr else "RNE",
                                         int(rht), round(tq, 4), round(gq, 1), round(gq / hbm_peak, 3),
                                         round(t_amax[rht], 4), round(ga, 1), round(both, 1)])
                del q
        del x
        torch.cuda.empty_cache()
    st = nv.nvfp4_get_status()
    if st != nv.NVFP4_OK:
        raise SystemExit(f"device status after the sweep: {nv.status_string(st)}")
    big = [r for r in out_rows if r[0] == 30]
    return {"columns": cols, "rows": out_rows, "unit": "GB/s", "hbm_peak_gbs": hbm_peak,
            "at_2^30": {"quant_gbs_min": min(r[6] for r in big), "quant_gbs_max": max(r[6] for r in big),
                        "quant_frac_median": statistics.median(r[7] for r in big),
                        "amax_gbs_min": min(r[9] for r in big)},
            "inputs": "seeded, drawn on the device (torch CUDA generator): t3 seed 5, normal seed 105",
            "l2": "flushed before each launch (256 MiB write, then 256 MiB read)"}


def load_traffic():
    """Per-launch DRAM bytes (read + write) from the committed ncu summaries
    (profiles/dram_traffic.txt: `key bytes note...` lines), if present."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    out = {}
    if os.path.exists(p):
        with open(p) as f:
            for line in f:
                t = line.split()
                if len(t) >= 2 and not line.startswith("#"):
                    out[t[0]] = int(t[1])
    return out


if __name__ == "__main__":
    sys.exit(main())
