#!/usr/bin/env python3
"""Benchmark of the MXFP4 training hot path on GB300.

One step = the whole path over one batch of the Llama-3.1-8B down-projection
layer (X[8192,14336], W[4096,14336], grad_out dY[8192,4096]; synthetic seeded
inputs standing in for the MaxText Llama-3.1-8B run the jax-aiter README
quotes):
  three dual casts  -- X (column copy with the 32-point Hadamard), W, dY
                       (column copy with the Hadamard);
  three MXFP4 GEMMs -- fwd Y = X W^T, dgrad dX = dY W, wgrad dW = dY^T X.
`value` is the step's GEMM TFLOP/s (3 x 2MNK per step over the step time,
casts included) with inputs resident in HBM.  A step is two launches: the
three casts in one mxfp4_cast_dual_grouped launch, then the three GEMMs in one
gemm_fp4_grouped launch (--separate-casts times four launches, the three casts
side by side on three streams or, with --serial-step, on one; --separate-gemms
six, with three gemm_fp4); `e2e` repeats it through the same
C-ABI calls with host buffers (pinned H2D of X, W, dY and D2H of Y, dX, dW of
every step inside the timed region, double-buffered so that one step's uploads
and downloads overlap its neighbours' compute).  `--impl reference` times the
CPU oracle instead.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
(for N > 1 launch one process per GPU with torch.distributed.run).
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from quantization_mxfp4_cast_gb300 import synth  # noqa: E402

M, N, K = 8192, 4096, 14336          # tokens, model dim (output of down-proj), FFN dim
X_SIGMA, W_SIGMA, DY_SIGMA = 0.02, 0.02, 1e-3
WORKLOAD = ("llama3.1-8b down-proj train step: X[8192,14336], W[4096,14336], dY[8192,4096] bf16; "
            "dual casts of X (col Hadamard), W, dY (col Hadamard) + MXFP4 fwd/dgrad/wgrad GEMMs, bf16 out")
METRIC = "MXFP4 fwd/dgrad/wgrad GEMM TFLOP/s at Llama shapes (train step, casts included)"
GEMM_FLOPS = [2.0 * M * N * K, 2.0 * M * K * N, 2.0 * N * K * M]   # fwd, dgrad, wgrad
STEP_FLOPS = sum(GEMM_FLOPS)
CAST_ELEMS = [M * K, N * K, M * N]                                  # X, W, dY
CAST_BYTES_PER_ELEM = 2 + 0.5 + 0.5 + 2.0 / 32                      # read bf16, write 2 x codes + 2 x scales
NOMINAL_FP4_OVER_BF16 = 13.5 / 2.25
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------------------- peaks
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {"bf16": float(d["bf16_tflops"]), "bf16_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "hbm": float(d["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16": FALLBACK_BF16_TFLOPS, "bf16_sustained": 1700.0, "hbm": FALLBACK_HBM_GBS,
                "source": "fallback"}


def strip_comments(src: str) -> str:
    """C++ source without its comments and blank lines (the sources hold no
    string literal with comment markers), so that a comment edit keeps the hash."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def gemm_source_hash():
    """sha256[:16] of the GEMM's code (gemm.cu and every header it includes,
    comments stripped)."""
    h = hashlib.sha256()
    for f in ("gemm.cu", "ptx.cuh", "quant.cuh", "internal.h"):
        text = open(os.path.join(ROOT, "quantization_mxfp4_cast_gb300", "csrc", f)).read()
        h.update(strip_comments(text).encode())
    return h.hexdigest()[:16]


def profiled_traffic(mode):
    """DRAM bytes per launch of the timed GEMM form ("grouped": the one
    grouped launch; "separate": mean of the three gemm_fp4 launches) from the
    committed ncu summary, if it was taken on the current GEMM source; else None."""
    p = os.path.join(ROOT, "profiles", "gemm_mxf4_llama8b_down_train_step.md")
    try:
        text = open(p).read()
    except OSError:
        return None
    src = re.search(r"gemm source sha256\[:16\]:\s*`?([0-9a-f]{16})", text)
    key = "grouped launch" if mode == "grouped" else "launch \\(mean of the three GEMMs\\)"
    tr = re.search(r"dram bytes per " + key + r":\s*([0-9.eE+]+)", text)
    if not src or not tr or src.group(1) != gemm_source_hash():
        return None
    return float(tr.group(1))


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                cur, mx = float(f[1]), float(f[2])
            except ValueError:
                continue
            smax = max(smax, mx)
            sm.append(cur)
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        loaded = [c for c in sm if c > 0.5 * smax] if smax else sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": smax or None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- GPU step
class Step:
    """Buffers and launches of one train step through the C ABI binding."""

    def __init__(self, m, dev):
        self.m = m
        x, w, dy = synth.linear_layer(M, N, K, X_SIGMA, W_SIGMA, DY_SIGMA)
        self.host = {"x": x.pin_memory(), "w": w.pin_memory(), "dy": dy.pin_memory()}
        self.x, self.w, self.dy = x.to(dev), w.to(dev), dy.to(dev)
        u8 = lambda n: torch.empty(n, dtype=torch.uint8, device=dev)
        sb = m.scales_bytes

        def dual(R, C):
            return (u8(R * C // 2).view(R, C // 2), u8(sb(R, C)), u8(C * R // 2).view(C, R // 2), u8(sb(C, R)))
        self.qx, self.qw, self.qdy = dual(M, K), dual(N, K), dual(M, N)
        bf = lambda r, c: torch.empty(r, c, dtype=torch.bfloat16, device=dev)
        self.y, self.dx, self.dw = bf(M, N), bf(M, K), bf(N, K)
        self.out_host = {"y": torch.empty(M, N, dtype=torch.bfloat16).pin_memory(),
                         "dx": torch.empty(M, K, dtype=torch.bfloat16).pin_memory(),
                         "dw": torch.empty(N, K, dtype=torch.bfloat16).pin_memory()}

    def launches(self, stream):
        m = self.m
        return [
            ("cast", lambda: m.mxfp4_cast_dual(self.x, hadamard_col=True, out=self.qx, stream=stream)),
            ("cast", lambda: m.mxfp4_cast_dual(self.w, out=self.qw, stream=stream)),
            ("cast", lambda: m.mxfp4_cast_dual(self.dy, hadamard_col=True, out=self.qdy, stream=stream)),
            ("gemm", lambda: m.gemm_fp4(self.qx[0], self.qx[1], self.qw[0], self.qw[1], M, N, K, c=self.y, stream=stream)),
            ("gemm", lambda: m.gemm_fp4(self.qdy[0], self.qdy[1], self.qw[2], self.qw[3], M, K, N, c=self.dx, stream=stream)),
            ("gemm", lambda: m.gemm_fp4(self.qdy[2], self.qdy[3], self.qx[2], self.qx[3], N, K, M, c=self.dw, stream=stream)),
        ]

    def run(self, stream, events=None):
        for i, (_, f) in enumerate(self.launches(stream)):
            if events is not None:
                events[i][0].record(stream)
            f()
            if events is not None:
                events[i][1].record(stream)

    def casts_grouped(self, stream, xs=None):
        """The dual casts of X and dY (column Hadamard) and W in one
        mxfp4_cast_dual_grouped launch."""
        x, w, dy = xs if xs is not None else (self.x, self.w, self.dy)
        return self.m.mxfp4_cast_dual_grouped([(x, False, True, self.qx), (w, False, False, self.qw),
                                               (dy, False, True, self.qdy)], stream=stream)

    def gemms_grouped(self, stream, outs=None):
        """fwd, dgrad and wgrad in one gemm_fp4_grouped launch."""
        m = self.m
        y, dx, dw = outs if outs is not None else (self.y, self.dx, self.dw)
        return m.gemm_fp4_grouped([
            (self.qx[0], self.qx[1], self.qw[0], self.qw[1], M, N, K, y),
            (self.qdy[0], self.qdy[1], self.qw[2], self.qw[3], M, K, N, dx),
            (self.qdy[2], self.qdy[3], self.qx[2], self.qx[3], N, K, M, dw)], stream=stream)

    def run_grouped(self, stream, side=None, casts_grouped=True):
        """The step as two launches: the casts of X, W and dY in one grouped
        launch, then the three GEMMs in one.  With casts_grouped=False, four:
        the three casts (side by side on three streams when `side` is given),
        then the grouped GEMM launch once all three are done."""
        if casts_grouped:
            self.casts_grouped(stream)
        elif side is None:
            for _, f in self.launches(stream)[:3]:
                f()
        else:
            s1, s2 = side
            s1.wait_stream(stream)
            s2.wait_stream(stream)
            for _, f in self.launches_streams((stream, s1, s2))[:3]:
                f()
            stream.wait_stream(s1)
            stream.wait_stream(s2)
        self.gemms_grouped(stream)

    def run_concurrent(self, stream, side):
        """The same six launches with the independent ones on three streams:
        the casts of X, W and dY side by side, then fwd (X, W), dgrad (dY, W)
        and wgrad (dY, X) each as soon as its two casts are done.  Every
        kernel fills the GPU; the overlap only fills the tail of one kernel
        with the start of the next."""
        s1, s2 = side
        s1.wait_stream(stream)
        s2.wait_stream(stream)
        fs = [f for _, f in self.launches_streams((stream, s1, s2))]
        fs[0]()                    # cast X  (stream)
        fs[1]()                    # cast W  (s1)
        fs[2]()                    # cast dY (s2)
        e_x, e_w, e_dy = stream.record_event(), s1.record_event(), s2.record_event()
        stream.wait_event(e_w)
        fs[3]()                    # fwd   (stream): X, W
        s1.wait_event(e_dy)
        fs[4]()                    # dgrad (s1): dY, W
        s2.wait_event(e_x)
        fs[5]()                    # wgrad (s2): dY, X
        stream.wait_stream(s1)
        stream.wait_stream(s2)

    def launches_streams(self, streams):
        s0, s1, s2 = streams
        m = self.m
        return [
            ("cast", lambda: m.mxfp4_cast_dual(self.x, hadamard_col=True, out=self.qx, stream=s0)),
            ("cast", lambda: m.mxfp4_cast_dual(self.w, out=self.qw, stream=s1)),
            ("cast", lambda: m.mxfp4_cast_dual(self.dy, hadamard_col=True, out=self.qdy, stream=s2)),
            ("gemm", lambda: m.gemm_fp4(self.qx[0], self.qx[1], self.qw[0], self.qw[1], M, N, K, c=self.y, stream=s0)),
            ("gemm", lambda: m.gemm_fp4(self.qdy[0], self.qdy[1], self.qw[2], self.qw[3], M, K, N, c=self.dx, stream=s1)),
            ("gemm", lambda: m.gemm_fp4(self.qdy[2], self.qdy[3], self.qx[2], self.qx[3], N, K, M, c=self.dw, stream=s2)),
        ]

    def e2e_buffers(self, dev):
        """A second set of bf16 inputs and outputs on the device, and two sets of
        pinned host outputs, for the double-buffered end-to-end pipeline."""
        bf = lambda r, c: torch.empty(r, c, dtype=torch.bfloat16, device=dev)
        self.e2e_in = [(self.x, self.w, self.dy), (bf(M, K), bf(N, K), bf(M, N))]
        self.e2e_out = [(self.y, self.dx, self.dw), (bf(M, N), bf(M, K), bf(N, K))]
        pin = lambda r, c: torch.empty(r, c, dtype=torch.bfloat16).pin_memory()
        self.e2e_host_out = [self.out_host, {"y": pin(M, N), "dx": pin(M, K), "dw": pin(N, K)}]

    def launches_on(self, xs, outs, stream, grouped=True):
        m = self.m
        x, w, dy = xs
        y, dx, dw = outs
        if grouped:  # one grouped cast launch and one grouped GEMM launch
            return [lambda: self.casts_grouped(stream, xs), lambda: self.gemms_grouped(stream, outs)]
        casts = [
            lambda: m.mxfp4_cast_dual(x, hadamard_col=True, out=self.qx, stream=stream),
            lambda: m.mxfp4_cast_dual(w, out=self.qw, stream=stream),
            lambda: m.mxfp4_cast_dual(dy, hadamard_col=True, out=self.qdy, stream=stream),
        ]
        return casts + [
            lambda: m.gemm_fp4(self.qx[0], self.qx[1], self.qw[0], self.qw[1], M, N, K, c=y, stream=stream),
            lambda: m.gemm_fp4(self.qdy[0], self.qdy[1], self.qw[2], self.qw[3], M, K, N, c=dx, stream=stream),
            lambda: m.gemm_fp4(self.qdy[2], self.qdy[3], self.qx[2], self.qx[3], N, K, M, c=dw, stream=stream),
        ]

    def run_e2e_pipelined(self, n_steps, streams, ev, grouped=True):
        """n_steps train steps from pinned host inputs to pinned host outputs.

        Every step copies its inputs host->device (copy-in stream), runs the
        casts and GEMMs (compute stream) and copies its three outputs
        device->host (copy-out stream).  Inputs and outputs are double-buffered
        so that step i+1's upload and step i-1's download overlap step i's
        compute; events order every reuse of a buffer.  (Measured: one copy
        stream per tensor and direction is slower than one per direction.)"""
        s_in, s_comp, s_out = streams
        h = self.host
        for i in range(n_steps):
            b = i % 2
            xs, outs, hout = self.e2e_in[b], self.e2e_out[b], self.e2e_host_out[b]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev["in_free"][b])      # step i-2's casts have read buffer b
                for dst, src in zip(xs, (h["x"], h["w"], h["dy"])):
                    dst.copy_(src, non_blocking=True)
                ev["in_ready"][b].record(s_in)
            s_comp.wait_event(ev["in_ready"][b])
            if i >= 2:
                s_comp.wait_event(ev["out_free"][b])       # step i-2's outputs have been downloaded
            fs = self.launches_on(xs, outs, s_comp, grouped)
            for f in fs[:3]:
                f()
            ev["in_free"][b].record(s_comp)
            for f in fs[3:]:
                f()
            ev["out_ready"][b].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["out_ready"][b])
                for name, src in zip(("y", "dx", "dw"), outs):
                    hout[name].copy_(src, non_blocking=True)
                ev["out_free"][b].record(s_out)

    def h2d_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.host.values())

    def d2h_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.out_host.values())


def host_link_rates(step, streams, dev, reps=5):
    """This box's pinned host<->device copy rates for the step's own tensors:
    uploads alone, downloads alone, and both directions at once on their two
    streams (no compute): the floor under the end-to-end leg."""
    s_in, _, s_out = streams
    h, xs = step.host, step.e2e_in[0]
    outs, hout = step.e2e_out[0], step.e2e_host_out[0]

    def up():
        with torch.cuda.stream(s_in):
            for dst, src in zip(xs, (h["x"], h["w"], h["dy"])):
                dst.copy_(src, non_blocking=True)

    def down():
        with torch.cuda.stream(s_out):
            for name, src in zip(("y", "dx", "dw"), outs):
                hout[name].copy_(src, non_blocking=True)

    def timed(fns):
        # the best of `reps` synchronized repetitions: a copy floor, so a slow
        # first use (or a neighbour's traffic) must not raise it
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for f in fns:
                f()
            torch.cuda.synchronize()
            best = min(best, time.perf_counter() - t0)
        return best

    up(), down()
    t_up, t_down, t_both = timed([up]), timed([down]), timed([up, down])
    bi, bo = step.h2d_bytes(), step.d2h_bytes()
    return {"h2d_gbs": bi / t_up / 1e9, "d2h_gbs": bo / t_down / 1e9,
            "both_directions_gbs": (bi + bo) / t_both / 1e9, "copy_floor_ms_per_step": t_both * 1e3,
            "upload_ms": t_up * 1e3, "download_ms": t_down * 1e3,
            "cuda_device_max_connections": os.environ.get("CUDA_DEVICE_MAX_CONNECTIONS", "unset (8)"),
            "what": "pinned copies of the step's inputs (H2D) and outputs (D2H), alone and both at once, "
                    f"best of {reps} synchronized repetitions each; copy_floor_ms_per_step is the time of one "
                    "step's copies with no compute"}


# ----------------------------------------------------------------------------- layer and FP8 legs
def time_loop(fn, iters, warm, stream):
    """Mean seconds per call of fn() on `stream` (CUDA events, after warm-up)."""
    with torch.cuda.stream(stream):
        for _ in range(warm):
            fn()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            fn()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3 / iters


def layer_leg(step, stream, iters=10):
    """The same train step through the layer API (MXFP4Linear: autograd
    forward + backward) with the weight's casts served by the workspace, as
    between two optimizer steps (micro-batches); gradients are dropped after
    each micro-batch, so no accumulation kernel runs."""
    from quantization_mxfp4_cast_gb300.layer import MXFP4Linear
    with torch.cuda.stream(stream):
        layer = MXFP4Linear(step.w.clone(), cache_name="down_proj")
        x = step.x.detach().clone().requires_grad_(True)
        dy = step.dy

        def micro_batch():
            y = layer(x)
            y.backward(dy)
            layer.weight.grad = None
            x.grad = None

        t = time_loop(micro_batch, iters, 2, stream)
    return {"value": STEP_FLOPS / t / 1e12, "unit": "TFLOP/s", "ms_per_micro_batch": t * 1e3,
            "weight_casts": layer.workspace.casts, "micro_batches": iters + 2,
            "what": "MXFP4Linear fwd + bwd (casts of X and dY, three GEMMs) with W's casts cached "
                    "in a WeightWorkspace across micro-batches"}


def fp8_wgrad_leg(step, stream, iters=20):
    """The FP8 alternative for the step's wgrad (dW = dY^T X over the tokens):
    MXFP8 (E4M3) column casts of dY and X with the Hadamard, then the
    kind::mxf8f6f4 GEMM, each timed on its own (CUDA events, back to back)."""
    m = step.m
    with torch.cuda.stream(stream):
        qdy = m.mxfp8_cast_cols(step.dy, hadamard=True, stream=stream)
        qx = m.mxfp8_cast_cols(step.x, hadamard=True, stream=stream)
        dw = torch.empty(N, K, dtype=torch.bfloat16, device=step.x.device)
        t_cast_dy = time_loop(lambda: m.mxfp8_cast_cols(step.dy, hadamard=True, out=qdy, stream=stream),
                              iters, 3, stream)
        t_cast_x = time_loop(lambda: m.mxfp8_cast_cols(step.x, hadamard=True, out=qx, stream=stream),
                             iters, 3, stream)
        t_gemm = time_loop(lambda: m.gemm_mxfp8(qdy[0], qdy[1], qx[0], qx[1], N, K, M, c=dw, stream=stream),
                           iters, 3, stream)
    cast_bytes = lambda r, c: r * c * (2 + 1) + r * c // 32  # bf16 in, E4M3 codes + scales out
    return {"gemm_tflops": 2.0 * M * N * K / t_gemm / 1e12, "gemm_us": t_gemm * 1e6,
            "cast_gbs": {"dY": cast_bytes(M, N) / t_cast_dy / 1e9, "X": cast_bytes(M, K) / t_cast_x / 1e9},
            "cast_us": {"dY": t_cast_dy * 1e6, "X": t_cast_x * 1e6},
            "wgrad_tflops_with_casts": 2.0 * M * N * K / (t_gemm + t_cast_dy + t_cast_x) / 1e12,
            "what": "MXFP8 wgrad recipe: column casts of dY and X (E4M3 + E8M0, Hadamard along M) "
                    "and the kind::mxf8f6f4 GEMM dW[N,K] = dY^T X"}


def cast_out_leg(step, stream, iters=20):
    """The dgrad GEMM with the next cast fused into its epilogue: dX = dY . W
    written as bf16 and, by the same kernel, as MXFP4 (row-wise, and column-wise
    with the Hadamard along M: the grad preset the layer below casts its
    grad_out with), against the same GEMM followed by a separate dual cast
    of dX.  Each variant timed on its own (CUDA events, back to back)."""
    m = step.m
    with torch.cuda.stream(stream):
        dx = torch.empty(M, K, dtype=torch.bfloat16, device=step.x.device)
        gemm = lambda: m.gemm_fp4(step.qdy[0], step.qdy[1], step.qw[2], step.qw[3], M, K, N, c=dx,
                                  stream=stream)
        gemm()
        qdx = m.mxfp4_cast_dual(dx, hadamard_col=True, stream=stream)
        cast = lambda: m.mxfp4_cast_dual(dx, hadamard_col=True, out=qdx, stream=stream)
        fused = lambda: m.gemm_fp4_cast_out(step.qdy[0], step.qdy[1], step.qw[2], step.qw[3], M, K, N,
                                            hadamard_col=True, c=dx, out=qdx, stream=stream)
        t_gemm = time_loop(gemm, iters, 3, stream)
        t_cast = time_loop(cast, iters, 3, stream)
        t_sep = time_loop(lambda: (gemm(), cast()), iters, 3, stream)
        t_fused = time_loop(fused, iters, 3, stream)
    flop = 2.0 * M * N * K
    return {"unit": "us", "dgrad_us": t_gemm * 1e6, "dual_cast_dx_us": t_cast * 1e6,
            "dgrad_then_cast_us": t_sep * 1e6, "dgrad_cast_out_us": t_fused * 1e6,
            "saved_us": (t_sep - t_fused) * 1e6,
            "dgrad_cast_out_tflops": flop / t_fused / 1e12,
            "what": "dX[8192,14336] = dY . W (MXFP4) plus the dual MXFP4 cast of dX (row; column with "
                    "Hadamard): separate cast kernel vs the cast written by the GEMM's epilogue"}


def fwd_with_casts_leg(m, dev, stream, iters=10):
    """The 8B gate/up forward from bf16 operands (X[8192, 4096] ~ N(0, 1),
    W[28672, 4096] ~ N(0, 0.02)) through gemm_fp4_bf16_fwd: both row-wise
    casts (one grouped launch), then the GEMM, against the GEMM alone on the
    operands already cast.  CUDA events, back to back."""
    M_, N_, K_, xs = synth.LLAMA_SHAPES["llama8b_gate_up"]
    x = synth.normal_bf16((M_, K_), xs, seed=81).to(dev)
    w = synth.normal_bf16((N_, K_), 0.02, seed=82).to(dev)
    with torch.cuda.stream(stream):
        y = torch.empty(M_, N_, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(m.workspace_bytes(m.MXFP4_OP_FWD, M_, N_, K_), dtype=torch.uint8, device=dev)
        qx, qw = m.mxfp4_cast(x, stream=stream), m.mxfp4_cast(w, stream=stream)
        full = lambda: m.gemm_fp4_bf16_fwd(x, w, y=y, ws=ws, stream=stream)
        gemm = lambda: m.gemm_fp4(qx[0], qx[1], qw[0], qw[1], M_, N_, K_, c=y, stream=stream)
        t_full = time_loop(full, iters, 3, stream)
        t_gemm = time_loop(gemm, iters, 3, stream)
    flop = 2.0 * M_ * N_ * K_
    return {"unit": "TFLOP/s", "with_casts_tflops": flop / t_full / 1e12, "with_casts_us": t_full * 1e6,
            "gemm_only_tflops": flop / t_gemm / 1e12, "gemm_only_us": t_gemm * 1e6,
            "casts_us": (t_full - t_gemm) * 1e6,
            "what": "Llama-3.1-8B gate/up forward Y[8192,28672] = X W^T from bf16 X and W: gemm_fp4_bf16_fwd "
                    "(row-wise casts of X and W in one grouped launch, then the GEMM) against gemm_fp4 on the "
                    "operands already cast (the weight cached)"}


def time_each(fn, iters, stream, flush):
    """Mean seconds of fn() launched alone on `stream`, L2 overwritten before
    each launch (the flush sits outside the timed events)."""
    with torch.cuda.stream(stream):
        for _ in range(2):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for e0, e1 in evs:
            flush.fill_(1.0)
            e0.record(stream)
            fn()
            e1.record(stream)
    torch.cuda.synchronize()
    return sum(e0.elapsed_time(e1) for e0, e1 in evs) / iters / 1e3


def cast_only_leg(m, dev, stream, hbm_gbs, iters=20):
    """The cast-only workload: bf16 activations [8192, 4096] ~ N(0,1) with 0.1%
    of the entries scaled by 50; the dual cast (row-wise + transposed) with
    the Hadamard off and on (both outputs), and the row-wise cast alone.
    Timed back to back over rotating input/output sets whose total is more
    than twice the L2, so every launch reads and writes HBM; the isolated time
    of one launch after an L2 overwrite is reported beside it."""
    x0 = synth.cast_input().to(dev)
    R, C = x0.shape
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_set = R * C * (2 + 1.0625)
    nsets = max(4, int(2 * l2 / per_set) + 1)
    xs = [x0.clone() for _ in range(nsets)]
    duals = [m.mxfp4_cast_dual(x, stream=stream) for x in xs]
    rows = [m.mxfp4_cast(x, stream=stream) for x in xs]
    runs = {
        "dual": (lambda k: m.mxfp4_cast_dual(xs[k], out=duals[k], stream=stream), 3.0625),
        "dual_hadamard_row_col": (lambda k: m.mxfp4_cast_dual(xs[k], hadamard_row=True, hadamard_col=True,
                                                               out=duals[k], stream=stream), 3.0625),
        "dual_hadamard_col": (lambda k: m.mxfp4_cast_dual(xs[k], hadamard_col=True, out=duals[k], stream=stream),
                              3.0625),
        "row_only": (lambda k: m.mxfp4_cast(xs[k], q=rows[k][0], sf=rows[k][1], stream=stream), 2.53125),
    }
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    out = {}
    for name, (fn, bpe) in runs.items():
        t = time_loop(lambda it=[0]: (fn(it[0] % nsets), it.__setitem__(0, it[0] + 1)), iters, 4, stream)
        t_iso = time_each(lambda: fn(0), 10, stream, flush)
        gbs = R * C * bpe / t / 1e9
        out[name] = {"us": t * 1e6, "gbs": gbs, "frac_of_measured_hbm": gbs / hbm_gbs, "frac_of_8tbs": gbs / 8000.0,
                     "isolated_us": t_iso * 1e6, "isolated_gbs": R * C * bpe / t_iso / 1e9}
    del flush, xs, duals, rows
    return {"shape": [R, C], "bytes_per_element": {"dual": 3.0625, "row_only": 2.53125}, **out,
            "what": f"cast-only workload (activations with 0.1% outliers x50): {iters} launches back to back over "
                    f"{nsets} rotating input/output sets ({nsets * per_set / 1e6:.0f} MB > 2x L2), CUDA events; "
                    "isolated_*: one launch alone after an L2 overwrite"}


def gemm_shapes_leg(m, dev, stream, iters=10):
    """Per-GEMM throughput at the Llama shapes: the 8B gate/up forward and the
    fwd / dgrad / wgrad of every 70B layer, on pre-quantized operands (random
    codes, scales 2^-9 .. 2^-6: the time does not depend on the values)."""
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    rnd = lambda n: torch.randint(0, 256, (n,), dtype=torch.uint8, device=dev, generator=g)
    sf = lambda r, k: torch.randint(0x76, 0x7A, (m.scales_bytes(r, k),), dtype=torch.uint8, device=dev,
                                    generator=g)
    cases = [("llama8b_gate_up", "fwd")] + [(n, d) for n in ("llama70b_qkv", "llama70b_o", "llama70b_gate_up",
                                                              "llama70b_down") for d in ("fwd", "dgrad", "wgrad")]
    out, flop_total, time_total = {}, 0.0, 0.0
    for name, which in cases:
        M_, N_, K_, _ = synth.LLAMA_SHAPES[name]
        mo, no, kc = {"fwd": (M_, N_, K_), "dgrad": (M_, K_, N_), "wgrad": (N_, K_, M_)}[which]
        a, b = rnd(mo * kc // 2), rnd(no * kc // 2)
        a_sf, b_sf = sf(mo, kc), sf(no, kc)
        c = torch.empty(mo, no, dtype=torch.bfloat16, device=dev)
        t = time_loop(lambda: m.gemm_fp4(a, a_sf, b, b_sf, mo, no, kc, c=c, stream=stream), iters, 3, stream)
        flop = 2.0 * mo * no * kc
        out[f"{name}.{which}"] = {"M": mo, "N": no, "K": kc, "tflops": flop / t / 1e12, "us": t * 1e6}
        flop_total += flop
        time_total += t
        del a, b, a_sf, b_sf, c
    # each 70B layer's fwd, dgrad and wgrad in one gemm_fp4_grouped launch
    grouped, gflop, gtime = {}, 0.0, 0.0
    for name in ("llama70b_qkv", "llama70b_o", "llama70b_gate_up", "llama70b_down"):
        M_, N_, K_, _ = synth.LLAMA_SHAPES[name]
        specs = [(M_, N_, K_), (M_, K_, N_), (N_, K_, M_)]
        descs = []
        for mo, no, kc in specs:
            descs.append((rnd(mo * kc // 2), sf(mo, kc), rnd(no * kc // 2), sf(no, kc), mo, no, kc,
                          torch.empty(mo, no, dtype=torch.bfloat16, device=dev)))
        t = time_loop(lambda: m.gemm_fp4_grouped(descs, stream=stream), iters, 3, stream)

        def three():
            for d in descs:
                m.gemm_fp4(*d[:7], c=d[7], stream=stream)
        t_sep = time_loop(three, iters, 3, stream)
        flop = sum(2.0 * mo * no * kc for mo, no, kc in specs)
        grouped[name] = {"tflops": flop / t / 1e12, "us": t * 1e6, "separate_us": t_sep * 1e6,
                         "separate_tflops": flop / t_sep / 1e12}
        gflop += flop
        gtime += t
        del descs
    return {"unit": "TFLOP/s", "gemms": out, "flop_weighted_tflops": flop_total / time_total / 1e12,
            "grouped_70b_layers": grouped, "grouped_flop_weighted_tflops": gflop / gtime / 1e12,
            "what": "gemm_fp4 at the 8B gate/up forward and the 70B layer shapes (M = 8192 tokens), "
                    "CUDA events, back to back; grouped_70b_layers: each 70B layer's fwd, dgrad and wgrad as "
                    "one gemm_fp4_grouped launch, against the same three as gemm_fp4 launches in a row "
                    "(both repeated, so both see the same L2 state)"}


def stack_leg(dev, stream, iters=10):
    """Two layers back to back at the 8B MLP shapes (up: 4096 -> 14336, then
    down: 14336 -> 4096; nothing between them), forward + backward with the
    weights' casts cached: MXFP4LinearStack (each GEMM casts its output for
    the next one in its epilogue, no bf16 intermediate) against a chain of
    two MXFP4Linear layers (bf16 intermediates, separate casts)."""
    from quantization_mxfp4_cast_gb300.layer import MXFP4Linear, MXFP4LinearStack
    w_up = synth.normal_bf16((K, N), 0.02, seed=71).to(dev)
    w_down = synth.normal_bf16((N, K), 0.02, seed=72).to(dev)
    x = synth.normal_bf16((M, N), 1.0, seed=73).to(dev)
    dy = synth.normal_bf16((M, N), 1e-3, seed=74).to(dev)
    with torch.cuda.stream(stream):
        stack = MXFP4LinearStack([w_up.clone(), w_down.clone()])
        chain = [MXFP4Linear(w_up.clone(), cache_name="up"), MXFP4Linear(w_down.clone(), cache_name="down")]
        xs = x.clone().requires_grad_(True)
        xc = x.clone().requires_grad_(True)

        def run_stack():
            stack(xs).backward(dy)
            xs.grad = None
            for p in stack.weights:
                p.grad = None

        def run_chain():
            h = xc
            for layer in chain:
                h = layer(h)
            h.backward(dy)
            xc.grad = None
            for layer in chain:
                layer.weight.grad = None

        t_stack = time_loop(run_stack, iters, 3, stream)
        t_chain = time_loop(run_chain, iters, 3, stream)
    flop = 2 * 3 * 2.0 * M * N * K
    return {"unit": "TFLOP/s", "stack_tflops": flop / t_stack / 1e12, "chain_tflops": flop / t_chain / 1e12,
            "stack_ms": t_stack * 1e3, "chain_ms": t_chain * 1e3, "saved_us": (t_chain - t_stack) * 1e6,
            "what": "x[8192,4096] -> up W[14336,4096] -> down W[4096,14336], fwd + bwd (6 GEMMs): "
                    "MXFP4LinearStack (casts fused into the producing GEMMs) vs two MXFP4Linear layers"}


def fp8_reference_leg(dev, stream, iters=20):
    """cuBLASLt FP8 (e4m3, per-tensor scales, bf16 out) through torch._scaled_mm
    on the step's three GEMM shapes, operands pre-quantized: context for the
    FP4 GEMMs on the same GPU.  Not part of any timed value."""
    try:
        f8 = torch.float8_e4m3fn
        out = {}
        one = torch.ones((), device=dev, dtype=torch.float32)
        for name, (mo, no, kc) in {"fwd": (M, N, K), "dgrad": (M, K, N), "wgrad": (N, K, M)}.items():
            a = (torch.randn(mo, kc, device=dev) * 0.5).to(f8)
            b = (torch.randn(no, kc, device=dev) * 0.5).to(f8)
            fn = lambda: torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            t = time_loop(fn, iters, 3, stream)
            out[name] = 2.0 * mo * no * kc / t / 1e12
            del a, b
        return {"unit": "TFLOP/s", "gemm_tflops": out,
                "what": "torch._scaled_mm (cuBLASLt) FP8 e4m3 x e4m3 -> bf16, per-tensor scales, "
                        "pre-quantized operands, same (M, N, K) as fwd / dgrad / wgrad"}
    except Exception as e:  # no FP8 GEMM in this torch build or on this device
        return {"unavailable": f"{type(e).__name__}: {e}"[:200]}


# ----------------------------------------------------------------------------- CPU oracle
_INPUTS = {}


def oracle_inputs():
    if not _INPUTS:
        import oracle
        x, w, dy = synth.linear_layer(M, N, K, X_SIGMA, W_SIGMA, DY_SIGMA)
        _INPUTS.update(x=oracle.as_bf16_bits(x), w=oracle.as_bf16_bits(w), dy=oracle.as_bf16_bits(dy))
    return _INPUTS["x"], _INPUTS["w"], _INPUTS["dy"]


def oracle_sample(rows_cast: int, out_rows: int, out_cols: int, nthreads: int):
    """Time the oracle on a slice of the step and extrapolate to a full step.

    cast part : dual cast (row + col, Hadamard as in the step) of the first
                `rows_cast` rows of X, W and dY;
    GEMM part : an out_rows x out_cols block of each of Y, dX, dW, from the
                oracle's cast of exactly the operand rows/columns it needs.
    Returns (estimated full-step seconds, seconds spent, description)."""
    import oracle
    bx, bw, bdy = oracle_inputs()
    t_all = time.perf_counter()
    t0 = time.perf_counter()
    n_cast = 0
    for arr, had in ((bx, True), (bw, False), (bdy, True)):
        sl = np.ascontiguousarray(arr[:rows_cast])
        oracle.cast_rows(sl)
        oracle.cast_cols(sl, hadamard=had)
        n_cast += sl.size
    t_cast = time.perf_counter() - t0
    t0 = time.perf_counter()
    ri, ci = np.arange(out_rows), np.arange(out_cols)
    a = oracle.cast_rows(np.ascontiguousarray(bx[ri]))
    b = oracle.cast_rows(np.ascontiguousarray(bw[ci]))
    oracle.gemm_mxfp4(*a, *b, nthreads=nthreads)                                   # Y block
    a = oracle.cast_rows(np.ascontiguousarray(bdy[ri]))
    b = oracle.cast_cols(np.ascontiguousarray(bw[:, ci]))
    oracle.gemm_mxfp4(*a, *b, nthreads=nthreads)                                   # dX block
    a = oracle.cast_cols(np.ascontiguousarray(bdy[:, ri]), hadamard=True)
    b = oracle.cast_cols(np.ascontiguousarray(bx[:, ci]), hadamard=True)
    oracle.gemm_mxfp4(*a, *b, nthreads=nthreads)                                   # dW block
    t_gemm = time.perf_counter() - t0
    sample_flops = 2.0 * out_rows * out_cols * (K + N + M)  # Y, dX, dW blocks contract over K, N, M
    full_cast = sum(CAST_ELEMS)
    est = t_cast * (full_cast / n_cast) + t_gemm * (STEP_FLOPS / sample_flops)
    desc = (f"oracle (scalar C quantizer, fp64 dot-product GEMM on {nthreads} threads): dual casts of the "
            f"first {rows_cast} rows of X, W, dY (cast single-threaded) and a {out_rows}x{out_cols} block of "
            f"each of Y, dX, dW with the operand casts it needs; extrapolated linearly to one full step")
    return est, time.perf_counter() - t_all, desc


def sample_idx(n, k, seed):
    """k distinct indices of range(n), the first and last always among them."""
    rng = np.random.default_rng(seed)
    idx = rng.choice(n, size=min(k, n), replace=False)
    idx[:2] = [0, n - 1]
    return np.unique(idx)


def gemm_within_tolerance(got, ref):
    """|gpu - oracle| <= 2^-8 |oracle| + 1e-3 rms(oracle) elementwise, rms over
    the sampled oracle values.  Returns (ok, worst excess over the bound)."""
    rms = float(np.sqrt(np.mean(ref ** 2)))
    excess = np.abs(got - ref) - (2.0 ** -8 * np.abs(ref) + 1e-3 * rms)
    return bool(np.isfinite(got).all() and (excess <= 0).all()), float(excess.max())


def parity_gate(step, nthreads, n_cast=64, n_out=64):
    """The step's own results against the oracle, before any number is
    reported: the row and column casts (codes and scales) of the first
    n_cast rows / columns of X, W and dY, and an n_out x n_out sample of each
    of Y, dX and dW (at the GEMM tolerance, rms over the sample's 4096 oracle
    values).  Returns a summary; 'ok' is False on any mismatch."""
    import oracle
    bx, bw, bdy = oracle_inputs()
    out = {"casts": {}, "gemms": {}}
    ok = True
    for name, arr, q, had in (("X", bx, step.qx, True), ("W", bw, step.qw, False), ("dY", bdy, step.qdy, True)):
        R, C = arr.shape
        cr, sr = oracle.cast_rows(np.ascontiguousarray(arr[:n_cast]))
        cc, sc = oracle.cast_cols(np.ascontiguousarray(arr[:, :n_cast]), hadamard=had)
        got_sr = oracle.sf_tile_to_linear(q[1].cpu().numpy(), R, C // 32)[:n_cast]
        got_sc = oracle.sf_tile_to_linear(q[3].cpu().numpy(), C, R // 32)[:n_cast]
        same = (np.array_equal(q[0][:n_cast].cpu().numpy(), cr) and np.array_equal(got_sr, sr)
                and np.array_equal(q[2][:n_cast].cpu().numpy(), cc) and np.array_equal(got_sc, sc))
        out["casts"][name] = "bit-exact" if same else "MISMATCH"
        ok &= same
    si, sj = sample_idx(M, n_out, 11), sample_idx(N, n_out, 12)
    sk, sn = sample_idx(K, n_out, 13), sample_idx(N, n_out, 14)
    cases = {
        "Y": (step.y, si, sj, oracle.cast_rows(np.ascontiguousarray(bx[si])),
              oracle.cast_rows(np.ascontiguousarray(bw[sj]))),
        "dX": (step.dx, si, sk, oracle.cast_rows(np.ascontiguousarray(bdy[si])),
               oracle.cast_cols(np.ascontiguousarray(bw[:, sk]))),
        "dW": (step.dw, sn, sk, oracle.cast_cols(np.ascontiguousarray(bdy[:, sn]), hadamard=True),
               oracle.cast_cols(np.ascontiguousarray(bx[:, sk]), hadamard=True)),
    }
    for name, (c, ri, ci, (ca, sa), (cb, sb)) in cases.items():
        ref = oracle.gemm_mxfp4(ca, sa, cb, sb, nthreads=nthreads)
        dev = c.device
        got = c[torch.from_numpy(ri).to(dev)][:, torch.from_numpy(ci).to(dev)].float().cpu().numpy().astype(np.float64)
        good, excess = gemm_within_tolerance(got, ref)
        out["gemms"][name] = {"ok": good, "worst_excess": excess, "samples": int(ref.size)}
        ok &= good
    out["ok"] = bool(ok)
    out["what"] = (f"before timing: casts of the first {n_cast} rows and columns of X, W, dY bit-exact against the "
                   f"oracle; {n_out}x{n_out} sampled outputs of Y, dX, dW within 2^-8|ref| + 1e-3 rms(ref)")
    return out


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------- main
def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, dev):
    if world <= 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def bench_config(world):
    """The workload description both arms print."""
    return {"workload": WORKLOAD, "M": M, "N": N, "K": K, "parallelism": f"replicas x{world}",
            "l2": "no flush: the step streams ~1.1 GB through HBM per iteration (inputs larger than the 129 MB L2)"}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    nthreads = cpu_threads()
    # calibrate once on a small slice, then size each step to fit the run's budget
    est_small, spent_small, _ = oracle_sample(32, 8, 32, nthreads)
    per_step_budget = min(20.0, 150.0 / max(1, args.steps + args.warmup))
    scale = max(1.0, per_step_budget / max(spent_small, 1e-3))
    rows_cast = int(min(M, max(32, 32 * scale)) // 32 * 32)
    out_rows = int(min(512, max(8, 8 * scale ** 0.5)))
    out_cols = int(min(2048, max(32, 32 * scale ** 0.5)))
    ests, desc = [], ""
    for i in range(args.warmup + args.steps):
        est, _, desc = oracle_sample(rows_cast, out_rows, out_cols, nthreads)
        if i >= args.warmup:
            ests.append(est)
    t_step = statistics.median(ests)
    value = STEP_FLOPS / t_step / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle; fp32 Hadamard)", "data": "synthetic",
            "config": bench_config(world),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
                             "sample": desc},
            "timing": {"ms_per_step": "median over the timed steps of the per-step estimate: each step times a "
                                      "bounded sample of the workload and extrapolates it linearly to one full "
                                      "step, so ms_per_step is far longer than the run's wall time"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the layer-API leg and the cuBLASLt FP8 reference GEMMs")
    ap.add_argument("--serial-step", action="store_true",
                    help="capture the step's launches on one stream instead of three")
    ap.add_argument("--separate-gemms", action="store_true",
                    help="time the step as six launches (three casts, three gemm_fp4)")
    ap.add_argument("--separate-casts", action="store_true",
                    help="time the step as four launches (three casts, one grouped GEMM launch) instead of two")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl != "reference":
        log("warmup raised to 3 (minimum)")
        args.warmup = 3

    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import quantization_mxfp4_cast_gb300 as m
    from quantization_mxfp4_cast_gb300 import build as _build
    _build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    step = Step(m, dev)
    torch.cuda.synchronize()

    side = (torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev))

    def timed_step():
        if args.separate_gemms:
            if args.serial_step:
                step.run(stream)
            else:
                step.run_concurrent(stream, side)
        else:
            step.run_grouped(stream, None if args.serial_step else side, casts_grouped=not args.separate_casts)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            timed_step()  # the form the timed region runs, so the parity gate checks its outputs
    stream.synchronize()
    if m.device_status() != 0:
        raise RuntimeError("device status word set during warm-up")
    # the warm-up steps' outputs against the oracle: no number without parity
    parity = parity_gate(step, cpu_threads())
    if not parity["ok"]:
        log("parity gate FAILED: " + json.dumps(parity))
        return 3

    # --------------------------------------------------------------- timed region (HBM-resident inputs)
    # One step (2 launches through the C ABI: one grouped cast launch and one
    # grouped GEMM launch; 4 with --separate-casts, 6 with --separate-gemms) is
    # captured once as a CUDA graph and replayed K times, so the host never
    # starves the GPU between launches.
    n_launch = len(step.launches(stream))
    n_launch_step = n_launch if args.separate_gemms else (4 if args.separate_casts else 2)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        timed_step()
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
    stream.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    smi_index = int(visible[local]) if len(visible) > local and visible[local].isdigit() else local
    with ClockSampler(smi_index) as clk:
        barrier(world)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            t_start.record(stream)
            for _ in range(args.steps):
                graph.replay()
            t_end.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        barrier(world)
    elapsed = max_over_ranks(t_start.elapsed_time(t_end) / 1e3, world, dev)
    if m.device_status() != 0:
        raise RuntimeError("device status word set in the timed region")
    value = world * STEP_FLOPS * args.steps / elapsed / 1e12
    ms_per_step = elapsed / args.steps * 1e3

    # --------------------------------------------------------------- per-kernel times
    # Eager launches with an event pair around each, all enqueued while the
    # stream is held by a GPU sleep, so the events time back-to-back GPU work.
    n_prof = min(args.steps, 20)
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_launch)]
           for _ in range(n_prof)]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        step.run(stream)
    stream.synchronize()
    host_per_step = time.perf_counter() - t0
    for attempt in range(3):
        sleep_s = 0.005 + 2.0 * n_prof * host_per_step * (2 ** attempt)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(int(sleep_s * 2.2e9))
            h0 = time.perf_counter()
            for i in range(n_prof):
                step.run(stream, evs[i])
            host_enqueue = time.perf_counter() - h0
        stream.synchronize()
        if host_enqueue < sleep_s:
            break
    # the grouped GEMM launch alone, eager, back to back behind a GPU sleep
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_prof)]
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int((0.005 + 2.0 * n_prof * host_per_step) * 2.2e9))
        for i in range(n_prof):
            gev[i][0].record(stream)
            step.gemms_grouped(stream)
            gev[i][1].record(stream)
    stream.synchronize()
    grouped_t = [a.elapsed_time(b) / 1e3 for a, b in gev]
    # the three casts back to back on one stream, events only around the
    # group: each cast's set-up overlaps the previous one's tail (programmatic
    # dependent launch), as in a step; an event between two launches stops that
    cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_prof)]
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int((0.005 + 2.0 * n_prof * host_per_step) * 2.2e9))
        for i in range(n_prof):
            cev[i][0].record(stream)
            for _, f in step.launches(stream)[:3]:
                f()
            cev[i][1].record(stream)
    stream.synchronize()
    cast_chain_t = [a.elapsed_time(b) / 1e3 for a, b in cev]
    # the three casts in one grouped launch, the step's form
    qev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_prof)]
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int((0.005 + 2.0 * n_prof * host_per_step) * 2.2e9))
        for i in range(n_prof):
            qev[i][0].record(stream)
            step.casts_grouped(stream)
            qev[i][1].record(stream)
    stream.synchronize()
    cast_grouped_t = [a.elapsed_time(b) / 1e3 for a, b in qev]
    kinds = [k for k, _ in step.launches(stream)]
    per = [[evs[i][j][0].elapsed_time(evs[i][j][1]) / 1e3 for j in range(n_launch)] for i in range(n_prof)]
    gemm_t = [sum(p[j] for j in range(n_launch) if kinds[j] == "gemm") for p in per]
    cast_t = [sum(p[j] for j in range(n_launch) if kinds[j] == "cast") for p in per]
    launch_mean = [statistics.mean(p[j] for p in per) for j in range(n_launch)]

    peaks = load_peaks()
    fp4_peak = peaks["bf16"] * NOMINAL_FP4_OVER_BF16
    if args.separate_gemms:
        gemm_launch_s = statistics.mean(gemm_t) / 3.0      # mean of the three gemm_fp4 launches
        achieved = (STEP_FLOPS / 3.0) / gemm_launch_s / 1e12
        traffic = profiled_traffic("separate")
        roof_kernel = "gemm_mxf4_pair_kernel (mean of the fwd/dgrad/wgrad gemm_fp4 launches)"
    else:
        gemm_launch_s = statistics.mean(grouped_t)          # the one grouped launch of the step
        achieved = STEP_FLOPS / gemm_launch_s / 1e12
        traffic = profiled_traffic("grouped")
        roof_kernel = "gemm_mxf4_pair_kernel (the grouped fwd + dgrad + wgrad launch)"
    cast_bytes = sum(CAST_ELEMS) * CAST_BYTES_PER_ELEM
    cast_gbs = cast_bytes / statistics.mean(cast_t) / 1e9
    gemm_names = ["fwd", "dgrad", "wgrad"]
    breakdown = {
        "gemm_tflops": {gemm_names[i]: GEMM_FLOPS[i] / launch_mean[3 + i] / 1e12 for i in range(3)},
        "gemm_us": {gemm_names[i]: launch_mean[3 + i] * 1e6 for i in range(3)},
        "gemm_separate_us_sum": sum(launch_mean[3:6]) * 1e6,
        "gemm_grouped_us": statistics.mean(grouped_t) * 1e6,
        "gemm_grouped_tflops": STEP_FLOPS / statistics.mean(grouped_t) / 1e12,
        "cast_gbs": {n: CAST_ELEMS[i] * CAST_BYTES_PER_ELEM / launch_mean[i] / 1e9 for i, n in enumerate(["X", "W", "dY"])},
        "cast_us": {n: launch_mean[i] * 1e6 for i, n in enumerate(["X", "W", "dY"])},
        "cast_gbs_all": cast_gbs,
        "cast_frac_of_hbm_measured": cast_gbs / peaks["hbm"],
        "cast_frac_of_8tbs": cast_gbs / 8000.0,
        "casts_back_to_back_us": statistics.mean(cast_chain_t) * 1e6,
        "casts_back_to_back_frac_of_hbm_measured": cast_bytes / statistics.mean(cast_chain_t) / 1e9 / peaks["hbm"],
        "casts_grouped_us": statistics.mean(cast_grouped_t) * 1e6,
        "casts_grouped_frac_of_hbm_measured": cast_bytes / statistics.mean(cast_grouped_t) / 1e9 / peaks["hbm"],
        "casts_what": "cast_us: each cast between its own event pair (no overlap with its neighbours); "
                      "casts_back_to_back: the three in a row with events only around them; "
                      "casts_grouped: the three in one mxfp4_cast_dual_grouped launch (the step's form)",
    }

    # --------------------------------------------------------------- e2e leg (host buffers)
    e2e = None
    if not args.no_e2e:
        k_e2e = max(3, min(args.steps, 20))
        step.e2e_buffers(dev)
        streams = (torch.cuda.Stream(device=dev), stream, torch.cuda.Stream(device=dev))
        ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in_ready", "in_free", "out_ready", "out_free")}
        grouped = not args.separate_gemms
        step.run_e2e_pipelined(2, streams, ev, grouped)  # warm-up
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for st in (streams[0], streams[2]):
            st.wait_event(e0)
        step.run_e2e_pipelined(k_e2e, streams, ev, grouped)
        for st in (streams[0], streams[2]):
            stream.wait_event(st.record_event())
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
        link = host_link_rates(step, streams, dev)
        ms_e2e = t_e2e / k_e2e * 1e3
        e2e = {"value": world * STEP_FLOPS * k_e2e / t_e2e / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": step.h2d_bytes(), "d2h_bytes_per_step": step.d2h_bytes(),
               "steps": k_e2e, "ms_per_step": ms_e2e,
               "pipeline": "double-buffered: upload of step i+1 and download of step i-1 overlap step i's compute",
               "host_link": link, "frac_of_copy_floor": link["copy_floor_ms_per_step"] / ms_e2e,
               "serialized_ms_per_step": link["upload_ms"] + link["download_ms"] + ms_per_step,
               "reading": "ms_per_step near copy_floor_ms_per_step: uploads, downloads and compute overlap; "
                          "near serialized_ms_per_step (upload + download + device step): they ran one after "
                          "another"}

    extra = {}
    if not args.no_extra:
        extra["layer"] = layer_leg(step, stream)
        extra["mxfp8_wgrad"] = fp8_wgrad_leg(step, stream)
        extra["fp8_cublaslt_reference"] = fp8_reference_leg(dev, stream)
        extra["dgrad_cast_out"] = cast_out_leg(step, stream)
        extra["cast_only"] = cast_only_leg(m, dev, stream, peaks["hbm"])
        extra["gemm_shapes"] = gemm_shapes_leg(m, dev, stream)
        extra["gate_up_fwd_with_casts"] = fwd_with_casts_leg(m, dev, stream)
        extra["stack"] = stack_leg(dev, stream)
        if m.device_status() != 0:
            raise RuntimeError("device status word set in the layer leg")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:  # the oracle baseline: one GPU only
        nthreads = cpu_threads()
        est, spent, desc = oracle_sample(8192, 256, 1536, nthreads)  # ~10-15 s of CPU work
        cpu = {"value": STEP_FLOPS / est / 1e12, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
               "sample": desc + f" ({spent:.1f} s of CPU work)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "mxfp4 (e2m1 x e2m1, e8m0 scales) -> f32 accum -> bf16",
            "data": "synthetic (seeded N(0,sigma) bf16: X,W ~ N(0,0.02), dY ~ N(0,1e-3))",
            "config": bench_config(world),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": fp4_peak, "unit": "TFLOP/s",
                         "frac": achieved / fp4_peak, "traffic": traffic,
                         "kernel": roof_kernel,
                         "peak_source": f"{peaks['source']} bf16 burst {peaks['bf16']:.1f} TFLOP/s x nominal "
                                        f"dense fp4/bf16 ratio {NOMINAL_FP4_OVER_BF16:.0f}"},
            "parity": parity,
            "breakdown": breakdown,
            "cpu_baseline": cpu,
            **({"extra": extra} if extra else {}),
            "e2e": e2e,
            "gpu_launches": n_launch_step * args.steps,
            "timing": {"timed_region": ("CUDA-graph replay of the captured step, K times, CUDA events on the launch stream; "
                                        + ("six launches (three casts, three gemm_fp4)" if args.separate_gemms else
                                           "four launches (three casts, one gemm_fp4_grouped of fwd, dgrad and wgrad)"
                                           if args.separate_casts else
                                           "two launches (one mxfp4_cast_dual_grouped of X, W and dY, one "
                                           "gemm_fp4_grouped of fwd, dgrad and wgrad)")
                                        + ("" if args.serial_step or not (args.separate_gemms or args.separate_casts)
                                           else ", the casts side by side on three streams")),
                       "per_kernel": f"{n_prof} eager steps of six launches, {n_prof} eager grouped GEMM launches, "
                                     f"{n_prof} runs of the three casts back to back and {n_prof} grouped cast launches, "
                                     "each enqueued behind a GPU sleep, an event pair per launch (per run for the "
                                     "casts back to back)"},
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
