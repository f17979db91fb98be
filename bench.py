"""Benchmark for the NVFP4 / FP8 weight-only matmul on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--quick]

Headline workload (one JSON line on rank 0): the NVFP4 decode GEMV of the
MTP-verify shape, M = 4, N = K = 5120, block_size 16, BF16 activations.  One
step is a chain of L = 32 such layers with 32 distinct weights (474 MB per
step, more than L2, so no layer reads its weight from L2), each layer's
output feeding the next layer's input, captured once as a CUDA graph and
replayed.  value = algorithmic bytes of all GEMV launches / device time
(GB/s).  Algorithmic bytes per launch = N*K/2 + N*K/16 + 2*M*K + 2*M*N + 4.

Also reported in the same line ("also"): the M = 1, 2, 8 sweep, the lm_head
GEMV (M = 4, N = 152064), the M = 8192 prefill GEMMs (TFLOP/s; L2 flushed
between timed launches), the standalone dequantize (GB/s) and the FP8 GEMV.

--impl reference times the CPU oracle (plain C++, float64) on the host cores
on a bounded sample of the same workload, as the reference arm.

Multi-GPU: every rank runs an independent replica of the workload on its own
GPU (weak scaling); the timed region is bracketed by a barrier and a device
synchronisation, and rank 0 reports the max time over ranks.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "NVFP4 W4A16 matmul: GEMV HBM GB/s (M≤8); prefill TFLOP/s (M=8192)"
UNIT = "GB/s"
LAYERS = 32


def gemv_bytes(M, N, K, bs=16, bias=False, kind="fp4"):
    S = (K + bs - 1) // bs
    if kind == "fp4":
        b = N * K // 2 + N * S + 2 * M * K + 2 * M * N + 4
    else:
        b = N * K + 4 * N * S + 2 * M * K + 2 * M * N
    return b + (2 * N if bias else 0)


def dequant_bytes(N, K, bs=16):
    return N * K // 2 + N * ((K + bs - 1) // bs) + 2 * N * K + 4


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "src": "fallback"}


# The sources a kernel is built from: its own translation unit (kernel and
# launcher) and the shared device and host headers.
KERNEL_SOURCES = {
    "gemv_decode_M4_N5120_K5120": ("wqmm_gemv.cu", "wqmm_device.cuh", "wqmm_internal.h"),
}


def csrc_hash(files=None):
    d = os.path.join(ROOT, "fp8_weight_only_nvfp4_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(files if files is not None else os.listdir(d)):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current sources of that kernel (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            rec = json.load(f)
        e = rec.get(kernel_key)
        if e and e.get("csrc_hash") == csrc_hash(KERNEL_SOURCES.get(kernel_key)):
            return e.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(values, dist=None, device=None):
    """Element-wise max of per-rank timings (the slowest rank decides)."""
    import torch
    t = torch.tensor(list(values), dtype=torch.float64,
                     device=device if device is not None else "cpu")
    if dist is not None and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def weak_scaling_value(per_rank_units, world, seconds):
    """Whole-job throughput: every rank processed per_rank_units in seconds."""
    return world * per_rank_units / seconds


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class Gpu:
    def __init__(self, device):
        import torch
        import fp8_weight_only_nvfp4_gb300 as wq
        self.torch = torch
        self.wq = wq
        self.dev = torch.device(device)
        torch.cuda.set_device(self.dev)
        self.stream = torch.cuda.Stream(self.dev)
        self.launches = 0

    def t(self, a, dtype=None):
        torch = self.torch
        x = torch.from_numpy(np.ascontiguousarray(a)).to(self.dev)
        if dtype is not None:
            x = x.view(dtype)
        return x

    def fp4_layers(self, M, N, K, L, seed0=100, log_uniform=False, ws2=0.0125, bias=False):
        torch = self.torch
        layers = []
        for i in range(L):
            Bp = wl.gen_fp4_packed(N, K, seed0 + i)
            ws = wl.gen_e4m3_scales(N, wl.scale_cols(K, 16), 2.0 ** (-6 if log_uniform else -4),
                                    4.0, log_uniform, seed0 + i)
            layers.append(dict(
                B=self.t(Bp), ws=self.t(ws),
                ws2=torch.tensor([ws2], dtype=torch.float32, device=self.dev),
                bias=(self.t(wl.gen_bias(N, 1, 0.02, seed0 + i).view(np.int16),
                             torch.bfloat16) if bias else None)))
        return layers

    def graph(self, fn):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(self.stream):
            fn()  # warm the library's one-time setup outside the capture
            self.stream.synchronize()
            with torch.cuda.graph(g, stream=self.stream):
                fn()
        return g

    def time_graph(self, g, steps, warmup, sync=None):
        torch = self.torch
        with torch.cuda.stream(self.stream):
            for _ in range(warmup):
                g.replay()
            self.stream.synchronize()
            if sync:
                sync()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            for _ in range(steps):
                g.replay()
            e1.record(self.stream)
            e1.synchronize()
            if sync:
                sync()
        return e0.elapsed_time(e1) / 1e3  # seconds

    def flush_l2(self):
        if not hasattr(self, "_flush"):
            self._flush = self.torch.empty(512 << 20, dtype=self.torch.uint8, device=self.dev)
        self._flush.fill_(1)

    def time_each(self, fn, reps, warmup, flush=True):
        """Median device time of single launches with L2 flushed between them."""
        torch = self.torch
        ts = []
        with torch.cuda.stream(self.stream):
            for i in range(warmup + reps):
                if flush:
                    self.flush_l2()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(self.stream)
                fn()
                e1.record(self.stream)
                e1.synchronize()
                if i >= warmup:
                    ts.append(e0.elapsed_time(e1) / 1e3)
        return statistics.median(ts)


def gemv_chain(gpu, M, N, K, L, kind="fp4", act="bf16", ws2=0.0125, feed=True):
    """L chained layers: layer i reads the previous layer's output (feed=True)
    or every layer reads the step's input (feed=False: for FP8 weights, which
    scale the activation by ~80 per layer and would leave the BF16 range; the
    launches are stream-ordered either way, each layer waiting for the
    previous one to complete, so the timing is the same)."""
    torch = gpu.torch
    wq = gpu.wq
    tdt = torch.bfloat16 if act == "bf16" else torch.float16
    if kind == "fp4":
        layers = gpu.fp4_layers(M, N, K, L, ws2=ws2)
    else:
        layers = []
        for i in range(L):
            layers.append(dict(B=gpu.t(wl.gen_fp8_weight(N, K, 300 + i)),
                               s=gpu.t(wl.gen_fp8_scale(N, wl.scale_cols(K, 128), 0.001, 0.02,
                                                        300 + i))))
    # bufs[0] holds the step's input and is never written, so every replay
    # starts from the same activation; the layers ping-pong between bufs[1]
    # and bufs[2] (N == K), layer i + 1 reading layer i's output.
    bufs = [gpu.t(wl.gen_activation(M, K, 1 if act == "bf16" else 0, 7).view(np.int16), tdt),
            torch.empty(M, N, dtype=tdt, device=gpu.dev),
            torch.empty(M, N, dtype=tdt, device=gpu.dev)]
    assert N == K

    def step():
        for i, ly in enumerate(layers):
            a = bufs[0] if (i == 0 or not feed) else bufs[1 + (i - 1) % 2]
            y = bufs[1 + i % 2]
            if kind == "fp4":
                wq.fp4_weight_matmul(a, ly["B"], ly["ws"], ly["ws2"], None, 16, out=y,
                                     stream=gpu.stream)
            else:
                wq.fp8_weight_matmul(a, ly["B"], ly["s"], None, 128, out=y, stream=gpu.stream)
    return step, bufs, layers


def bench_headline(gpu, args, rank, world, barrier_sync):
    torch = gpu.torch
    M, N, K, L = 4, 5120, 5120, LAYERS
    step, bufs, layers = gemv_chain(gpu, M, N, K, L)
    g = gpu.graph(step)
    per_launch = gemv_bytes(M, N, K)
    with ClockSampler(gpu.dev.index) as clk:
        dt = gpu.time_graph(g, args.steps, args.warmup, sync=barrier_sync)
    clocks = clk.summary()
    # e2e: through the same C-ABI calls, with the step's input copied from
    # pinned host memory and its result read back, every step.
    h_in = torch.from_numpy(wl.gen_activation(M, K, 1, 7).view(np.int16)).view(
        torch.bfloat16).pin_memory()
    h_out = torch.empty(M, N, dtype=torch.bfloat16).pin_memory()
    with torch.cuda.stream(gpu.stream):
        for _ in range(2):
            bufs[0].copy_(h_in, non_blocking=True)
            g.replay()
            h_out.copy_(bufs[1 + (L - 1) % 2], non_blocking=True)
        gpu.stream.synchronize()
        if barrier_sync:
            barrier_sync()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(gpu.stream)
        for _ in range(args.steps):
            bufs[0].copy_(h_in, non_blocking=True)
            g.replay()
            h_out.copy_(bufs[1 + (L - 1) % 2], non_blocking=True)
        e1.record(gpu.stream)
        e1.synchronize()
        wall = time.perf_counter() - t0
        if barrier_sync:
            barrier_sync()
    dt_e2e = max(e0.elapsed_time(e1) / 1e3, wall)
    return dict(dt=dt, per_launch=per_launch, launches=L, clocks=clocks, dt_e2e=dt_e2e,
                h2d=M * K * 2, d2h=M * N * 2)


def actq_bytes(M, K):
    """NVFP4 activation quantization: read A, write codes and scales."""
    return 2 * M * K + M * K // 2 + M * ((K + 15) // 16)


def bench_actq(gpu, args, hbm):
    """NVFP4 activation quantization of the 8K-token prefill activation
    (M = 8192, K = 5120, BF16): a graph of launches over two distinct inputs
    and outputs (215 MB, above L2), per launch."""
    torch = gpu.torch
    wq = gpu.wq
    M, K = 8192, 5120
    As = [torch.randn(M, K, device=gpu.dev, dtype=torch.bfloat16) for _ in range(2)]
    outs = [(torch.empty(M, K // 2, dtype=torch.uint8, device=gpu.dev),
             torch.empty(M, K // 16, dtype=torch.uint8, device=gpu.dev)) for _ in range(2)]

    def step():
        for A, (pc, sc) in zip(As, outs):
            wq.fp4_quantize_activation(A, out_packed=pc, out_scale=sc, stream=gpu.stream)
    g = gpu.graph(step)
    reps = max(5, args.steps // 5)
    dt = gpu.time_graph(g, reps, 2) / (reps * 2)
    gbs = actq_bytes(M, K) / dt / 1e9
    return {f"nvfp4_act_quantize_M{M}_K{K}": {"GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4),
                                                "us": round(dt * 1e6, 2)}}


def bench_also(gpu, args, peaks):
    torch = gpu.torch
    wq = gpu.wq
    out = {}
    hbm = peaks["hbm_gbs"]
    # M sweep of the decode GEMV chain.
    for M in (1, 2, 8):
        step, _, _ = gemv_chain(gpu, M, 5120, 5120, LAYERS)
        g = gpu.graph(step)
        dt = gpu.time_graph(g, max(5, args.steps // 2), 2)
        gbs = gemv_bytes(M, 5120, 5120) * LAYERS * max(5, args.steps // 2) / dt / 1e9
        out[f"gemv_M{M}_N5120_K5120"] = {"GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4)}
        del g
    # lm_head GEMV: 389 MB weight per launch (> L2), back-to-back launches.
    M, N, K = 4, 152064, 5120
    ly = gpu.fp4_layers(M, N, K, 1, seed0=500, log_uniform=True, ws2=0.01, bias=True)[0]
    A = gpu.t(wl.gen_activation(M, K, 1, 9).view(np.int16), torch.bfloat16)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=gpu.dev)
    g = gpu.graph(lambda: wq.fp4_weight_matmul(A, ly["B"], ly["ws"], ly["ws2"], ly["bias"], 16,
                                               out=Y, stream=gpu.stream))
    reps = 20
    dt = gpu.time_graph(g, reps, 3)
    gbs = gemv_bytes(M, N, K, bias=True) * reps / dt / 1e9
    out["lm_head_M4_N152064_K5120"] = {"GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4),
                                       "us": round(dt / reps * 1e6, 2)}
    # The same lm_head with FP16 activations and bias (the decode of each
    # weight pair folds its scale with one f16x2 multiply instead of two
    # mixed multiplies and a BF16 pack).
    A16 = gpu.t(wl.gen_activation(M, K, 0, 9).view(np.int16), torch.float16)
    b16 = gpu.t(wl.gen_bias(N, 0, 0.02, 500).view(np.int16), torch.float16)
    Y16 = torch.empty(M, N, dtype=torch.float16, device=gpu.dev)
    g16 = gpu.graph(lambda: wq.fp4_weight_matmul(A16, ly["B"], ly["ws"], ly["ws2"], b16, 16,
                                                 out=Y16, stream=gpu.stream))
    dt = gpu.time_graph(g16, reps, 3)
    gbs = gemv_bytes(M, N, K, bias=True) * reps / dt / 1e9
    out["lm_head_fp16_M4_N152064_K5120"] = {"GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4),
                                            "us": round(dt / reps * 1e6, 2)}
    # The M = 4 chain with FP16 activations (weight_scale_2 = 0.002 keeps the
    # chained values inside the FP16 range; the time does not depend on it).
    step, _, _ = gemv_chain(gpu, 4, 5120, 5120, LAYERS, act="fp16", ws2=0.002)
    gc = gpu.graph(step)
    nrep = max(5, args.steps // 2)
    dtc = gpu.time_graph(gc, nrep, 2)
    gbs = gemv_bytes(4, 5120, 5120) * LAYERS * nrep / dtc / 1e9
    out["gemv_fp16_M4_N5120_K5120"] = {"GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4),
                                       "us_per_layer": round(dtc / (nrep * LAYERS) * 1e6, 2)}
    del g, g16, gc, ly
    # Prefill GEMMs (tensor-bound), L2 flushed before each timed launch.
    tf_peak = peaks["bf16_tflops"]
    for shape, (N, K) in (("gate_up", (17408, 5120)), ("down", (5120, 17408))):
        M = 8192
        ly = gpu.fp4_layers(M, N, K, 1, seed0=700, bias=True)[0]
        A = torch.randn(M, K, device=gpu.dev, dtype=torch.bfloat16)
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=gpu.dev)
        fn = lambda: wq.fp4_weight_matmul(A, ly["B"], ly["ws"], ly["ws2"], ly["bias"], 16,
                                          out=Y, stream=gpu.stream)
        dt = gpu.time_each(fn, reps=5, warmup=2)
        tf = 2 * M * N * K / dt / 1e12
        out[f"prefill_{shape}_M8192_N{N}_K{K}"] = {"TFLOP/s": round(tf, 1),
                                                   "frac": round(tf / tf_peak, 4),
                                                   "ms": round(dt * 1e3, 3)}
        if shape == "gate_up":
            # Comparator arm: standalone dequant to scratch + cuBLAS (torch.matmul).
            W = torch.empty(N, K, dtype=torch.bfloat16, device=gpu.dev)
            dq = lambda: wq.fp4_dequantize(ly["B"], ly["ws"], ly["ws2"], 16, out=W,
                                           stream=gpu.stream)
            dt_dq = gpu.time_each(dq, reps=5, warmup=2)
            # Standalone dequantize: a graph of R launches over R distinct
            # weights and outputs (912 MB in total, far above L2), per launch.
            R = 4
            dls = gpu.fp4_layers(1, N, K, R, seed0=720)
            Ws = [torch.empty(N, K, dtype=torch.bfloat16, device=gpu.dev) for _ in range(R)]

            def dq_step():
                for d, w in zip(dls, Ws):
                    wq.fp4_dequantize(d["B"], d["ws"], d["ws2"], 16, out=w, stream=gpu.stream)
            gq = gpu.graph(dq_step)
            reps = max(5, args.steps // 5)
            dt_g = gpu.time_graph(gq, reps, 2) / (reps * R)
            gbs = dequant_bytes(N, K) / dt_g / 1e9
            out[f"dequant_N{N}_K{K}"] = {"GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4),
                                         "us": round(dt_g * 1e6, 2),
                                         "us_single_launch_l2_flushed": round(dt_dq * 1e6, 2)}
            del gq, dls, Ws
            mm = lambda: torch.matmul(A, W.t())
            with torch.cuda.stream(gpu.stream):
                dt_mm = gpu.time_each(mm, reps=5, warmup=2)
            out["comparator_dequant_plus_cublas_ms"] = round((dt_dq + dt_mm) * 1e3, 3)
            del W
        del ly, A, Y
    # FP8 decode GEMV chain (secondary format), M = 1, 4, 8.
    reps = max(5, args.steps // 2)
    for M in (1, 4, 8):
        step, _, _ = gemv_chain(gpu, M, 5120, 5120, LAYERS, kind="fp8", feed=False)
        g = gpu.graph(step)
        dt = gpu.time_graph(g, reps, 2)
        gbs = gemv_bytes(M, 5120, 5120, 128, kind="fp8") * LAYERS * reps / dt / 1e9
        out[f"fp8_gemv_M{M}_N5120_K5120"] = {"GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4)}
        del g
    # Mid-range M (8 < M <= 32) decode GEMV chain, NVFP4.
    for M in (16, 32):
        step, _, _ = gemv_chain(gpu, M, 5120, 5120, LAYERS)
        g = gpu.graph(step)
        dt = gpu.time_graph(g, reps, 2)
        gbs = gemv_bytes(M, 5120, 5120) * LAYERS * reps / dt / 1e9
        out[f"gemv_M{M}_N5120_K5120"] = {"GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4),
                                         "us_per_layer": round(dt / (reps * LAYERS) * 1e6, 2)}
        del g
    # Mid-range M (fused GEMM with a 64- or 128-token tile): R launches over
    # distinct weights per graph (more than L2 in total), TFLOP/s and weight
    # GB/s per launch.
    for (N, K, R) in ((17408, 5120, 4), (5120, 5120, 12)):
        lys = gpu.fp4_layers(8, N, K, R, seed0=800)
        for M in (64, 128):
            A = torch.randn(M, K, device=gpu.dev, dtype=torch.bfloat16)
            Y = torch.empty(M, N, dtype=torch.bfloat16, device=gpu.dev)

            def midm_step():
                for ly in lys:
                    wq.fp4_weight_matmul(A, ly["B"], ly["ws"], ly["ws2"], None, 16, out=Y,
                                         stream=gpu.stream)
            g = gpu.graph(midm_step)
            reps = max(5, args.steps // 5)
            dt = gpu.time_graph(g, reps, 2) / (reps * R)
            tf = 2 * M * N * K / dt / 1e12
            out[f"gemm_M{M}_N{N}_K{K}"] = {"TFLOP/s": round(tf, 1), "frac": round(tf / tf_peak, 4),
                                           "GB/s": round(gemv_bytes(M, N, K) / dt / 1e9, 1),
                                           "us": round(dt * 1e6, 2)}
            del g
        del lys
    out.update(bench_actq(gpu, args, hbm))
    # Whole decode step: one CUDA graph of 120 weight-only GEMVs shaped like a
    # 27B-class decoder (hidden 5120, MLP 17408): per layer four 5120 x 5120
    # projections, gate and up 17408 x 5120, down 5120 x 17408 (17 layers), then
    # the 152064 x 5120 lm_head; distinct synthetic weights per launch (3.6 GB,
    # far above L2).  Only the matmuls are timed: the attention core and the
    # activation function between them are not part of this path.
    out.update(decode_step(gpu, (4, 1), reps=max(3, args.steps // 10)))
    # FP8 prefill GEMM (secondary format), M = 8192, N = 17408, K = 5120, bs = 128.
    M, N, K = 8192, 17408, 5120
    B8 = gpu.t(wl.gen_fp8_weight(N, K, 900))
    s8 = gpu.t(wl.gen_fp8_scale(N, wl.scale_cols(K, 128), 0.001, 0.02, 900))
    A = torch.randn(M, K, device=gpu.dev, dtype=torch.bfloat16)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=gpu.dev)
    fn = lambda: wq.fp8_weight_matmul(A, B8, s8, None, 128, out=Y, stream=gpu.stream)
    dt = gpu.time_each(fn, reps=5, warmup=2)
    tf = 2 * M * N * K / dt / 1e12
    out[f"fp8_prefill_M{M}_N{N}_K{K}"] = {"TFLOP/s": round(tf, 1), "frac": round(tf / tf_peak, 4),
                                          "ms": round(dt * 1e3, 3)}
    # W8A8 prefill through the caller-workspace entry point: one pass that
    # quantize-dequantizes A to FP8 into the workspace, then the same GEMM.
    a_sc = torch.full((1,), 0.01, device=gpu.dev, dtype=torch.float32)
    ws = torch.empty(wq.fp8_w8a8_workspace_bytes(M, K), dtype=torch.uint8, device=gpu.dev)
    fn = lambda: wq.fp8_weight_matmul_w8a8_ws(A, a_sc, B8, s8, ws, None, 128, out=Y,
                                              stream=gpu.stream)
    dt_w = gpu.time_each(fn, reps=5, warmup=2)
    tf = 2 * M * N * K / dt_w / 1e12
    out[f"w8a8_prefill_M{M}_N{N}_K{K}"] = {"TFLOP/s": round(tf, 1), "frac": round(tf / tf_peak, 4),
                                           "ms": round(dt_w * 1e3, 3),
                                           "vs_weight_only": round(dt / dt_w, 3)}
    del B8, s8, A, Y, ws, a_sc
    # FP4 x FP4 prefill: the activation quantized to NVFP4 (timed separately
    # and together with the GEMM), then the block-scaled tensor-core GEMM.
    ly = gpu.fp4_layers(M, N, K, 1, seed0=700, bias=True)[0]
    A = torch.randn(M, K, device=gpu.dev, dtype=torch.bfloat16)
    qc, qs = wq.fp4_quantize_activation(A)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=gpu.dev)
    gemm = lambda: wq.fp4_fp4_matmul(qc, qs, ly["B"], ly["ws"], ly["ws2"], ly["bias"], out=Y,
                                     stream=gpu.stream)
    both = lambda: (wq.fp4_quantize_activation(A, out_packed=qc, out_scale=qs, stream=gpu.stream),
                    gemm())
    dt = gpu.time_each(gemm, reps=5, warmup=2)
    dt_q = gpu.time_each(both, reps=5, warmup=2)
    tf = 2 * M * N * K / dt / 1e12
    fp4_peak = 6 * tf_peak   # measured BF16 peak x the nominal FP4 : BF16 dense ratio
    out[f"f4f4_prefill_M{M}_N{N}_K{K}"] = {"TFLOP/s": round(tf, 1), "frac": round(tf / fp4_peak, 4),
                                           "peak_TFLOP/s": round(fp4_peak, 1),
                                           "ms": round(dt * 1e3, 3),
                                           "ms_with_activation_quantize": round(dt_q * 1e3, 3)}
    del ly, A, qc, qs, Y
    return out


def decode_step(gpu, Ms, reps, layers=17, hidden=5120, mlp=17408, vocab=152064):
    """120 chained GEMV launches of a synthetic 27B-class decode step, for
    each M in Ms (same weights)."""
    torch = gpu.torch
    wq = gpu.wq
    shapes = []
    for _ in range(layers):
        shapes += [(hidden, hidden)] * 4 + [(mlp, hidden), (mlp, hidden), (hidden, mlp)]
    shapes.append((vocab, hidden))
    # weight_scale_2 = 1 / (rms weight * sqrt(K)) keeps the chained
    # activations near unit scale through all 120 launches (the rms of an
    # E2M1 code times a scale uniform in [2^-4, 4] is about 6.8); the time
    # does not depend on it.
    ws = [gpu.fp4_layers(1, N, K, 1, seed0=2000 + i, ws2=1.0 / (6.8 * K ** 0.5))[0]
          for i, (N, K) in enumerate(shapes)]
    res = {}
    for M in Ms:
        # The step's input (never written) and two buffers per width.
        x_h = gpu.t(wl.gen_activation(M, hidden, 1, 11).view(np.int16), torch.bfloat16)
        bufs = {hidden: [torch.empty(M, hidden, dtype=torch.bfloat16, device=gpu.dev)
                         for _ in range(2)],
                mlp: [torch.empty(M, mlp, dtype=torch.bfloat16, device=gpu.dev) for _ in range(2)],
                vocab: [torch.empty(M, vocab, dtype=torch.bfloat16, device=gpu.dev)]}

        def step():
            cur = x_h
            for i, ((N, K), ly) in enumerate(zip(shapes, ws)):
                y = bufs[N][i % len(bufs[N])]
                if y is cur:
                    y = bufs[N][(i + 1) % len(bufs[N])]
                wq.fp4_weight_matmul(cur, ly["B"], ly["ws"], ly["ws2"], None, 16, out=y,
                                     stream=gpu.stream)
                # q, k, v, o, up and down feed the next launch; gate's output
                # is not consumed (up's output feeds down)
                if i >= 7 * layers or i % 7 != 4:
                    cur = y
        g = gpu.graph(step)
        dt = gpu.time_graph(g, reps, 2)
        per_step = dt / reps
        byts = sum(gemv_bytes(M, N, K) for (N, K) in shapes)
        res[f"decode_step_M{M}_{len(shapes)}_gemv"] = {
            "us_per_step": round(per_step * 1e6, 1), "GB/s": round(byts / per_step / 1e9, 1),
            "frac": round(byts / per_step / 1e9 / load_peaks()["hbm_gbs"], 4),
            "weight_GB": round(byts / 1e9, 2)}
        del g
    del ws
    return res


def cpu_oracle_baseline(budget_s=10.0):
    """The oracle, as it stands, on the host cores: full decode-GEMV layers
    (M=4, N=K=5120) repeated until about budget_s of CPU time."""
    import oracle
    p = wl.decode_gemv(M=4, seed=0)
    threads = oracle.hardware_threads()
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.fp4_matmul(p.A, p.B_packed, p.weight_scale, p.weight_scale_2, None, p.M, p.N, p.K,
                          16, p.dtype, threads=threads)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(gemv_bytes(4, 5120, 5120) * n / dt / 1e9, 4), "unit": UNIT,
            "cores": threads, "kind": "oracle",
            "sample": f"{n} full oracle calls of the M=4, N=K=5120 NVFP4 layer "
                      f"(float64, {threads} threads), {dt:.1f} s"}


def config(L=LAYERS):
    return {"workload": "NVFP4 decode GEMV (MTP verify) M=4 N=5120 K=5120 bs=16 BF16, "
                        f"chain of {L} layers with distinct weights, CUDA graph replay",
            "M": 4, "N": 5120, "K": 5120, "block_size": 16, "layers_per_step": L,
            "weight_bytes_per_step": L * (5120 * 2560 + 5120 * 320),
            "l2": "inputs larger than L2 (distinct weight per layer, 474 MB per step)",
            "parallelism": "replicas"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    p = wl.decode_gemv(M=4, seed=0)
    threads = oracle.hardware_threads()
    f = lambda: oracle.fp4_matmul(p.A, p.B_packed, p.weight_scale, p.weight_scale_2, None, p.M,
                                  p.N, p.K, 16, p.dtype, threads=threads)
    for _ in range(args.warmup):
        f()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        f()
    dt = time.perf_counter() - t0
    value = gemv_bytes(4, 5120, 5120) * args.steps / dt / 1e9
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "impl": "reference",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        # The same workload as the CUDA arm's line; each step is a bounded
        # sample of it (one of its layers, M = 4, N = K = 5120), and the value
        # counts the bytes of the layers actually processed.
        "config": config(),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads,
                         "kind": "oracle",
                         "sample": f"each step one layer of the {LAYERS}-layer chain (M=4, "
                                   f"N=K=5120, NVFP4, float64, {threads} threads); "
                                   f"{args.steps} timed steps"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_only(name, m, reps):
    """Run one workload a few times (for profilers); prints its device time."""
    import torch
    gpu = Gpu("cuda:0")
    wq = gpu.wq
    fn = None
    if name == "gemv":
        M, N, K = (m or 4), 5120, 5120
        ly = gpu.fp4_layers(M, N, K, 1, seed0=100)[0]
        A = gpu.t(wl.gen_activation(M, K, 1, 7).view(np.int16), torch.bfloat16)
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=gpu.dev)
        fn = lambda: wq.fp4_weight_matmul(A, ly["B"], ly["ws"], ly["ws2"], None, 16, out=Y,
                                          stream=gpu.stream)
        work = gemv_bytes(M, N, K) / 1e9, "GB/s"
    elif name == "lm_head":
        M, N, K = (m or 4), 152064, 5120
        ly = gpu.fp4_layers(M, N, K, 1, seed0=500, log_uniform=True, ws2=0.01, bias=True)[0]
        A = gpu.t(wl.gen_activation(M, K, 1, 9).view(np.int16), torch.bfloat16)
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=gpu.dev)
        fn = lambda: wq.fp4_weight_matmul(A, ly["B"], ly["ws"], ly["ws2"], ly["bias"], 16, out=Y,
                                          stream=gpu.stream)
        work = gemv_bytes(M, N, K, bias=True) / 1e9, "GB/s"
    elif name in ("prefill_gate_up", "prefill_down"):
        M = m or 8192
        N, K = (17408, 5120) if name == "prefill_gate_up" else (5120, 17408)
        ly = gpu.fp4_layers(M, N, K, 1, seed0=700, bias=True)[0]
        A = torch.randn(M, K, device=gpu.dev, dtype=torch.bfloat16)
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=gpu.dev)
        fn = lambda: wq.fp4_weight_matmul(A, ly["B"], ly["ws"], ly["ws2"], ly["bias"], 16, out=Y,
                                          stream=gpu.stream)
        work = 2 * M * N * K / 1e12, "TFLOP/s"
    elif name == "dequant":
        N, K = 17408, 5120
        ly = gpu.fp4_layers(1, N, K, 1, seed0=700)[0]
        W = torch.empty(N, K, dtype=torch.bfloat16, device=gpu.dev)
        fn = lambda: wq.fp4_dequantize(ly["B"], ly["ws"], ly["ws2"], 16, out=W, stream=gpu.stream)
        work = dequant_bytes(N, K) / 1e9, "GB/s"
    elif name == "actq":
        M, K = (m or 8192), 5120
        A = torch.randn(M, K, device=gpu.dev, dtype=torch.bfloat16)
        pc = torch.empty(M, K // 2, dtype=torch.uint8, device=gpu.dev)
        sc = torch.empty(M, K // 16, dtype=torch.uint8, device=gpu.dev)
        fn = lambda: wq.fp4_quantize_activation(A, out_packed=pc, out_scale=sc, stream=gpu.stream)
        work = actq_bytes(M, K) / 1e9, "GB/s"
    elif name == "fp8_gemv":
        M, N, K = (m or 4), 5120, 5120
        B = gpu.t(wl.gen_fp8_weight(N, K, 300))
        sc = gpu.t(wl.gen_fp8_scale(N, wl.scale_cols(K, 128), 0.001, 0.02, 300))
        A = gpu.t(wl.gen_activation(M, K, 1, 7).view(np.int16), torch.bfloat16)
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=gpu.dev)
        fn = lambda: wq.fp8_weight_matmul(A, B, sc, None, 128, out=Y, stream=gpu.stream)
        work = gemv_bytes(M, N, K, 128, kind="fp8") / 1e9, "GB/s"
    elif name == "w8a8_prefill":
        M, N, K = (m or 8192), 17408, 5120
        B = gpu.t(wl.gen_fp8_weight(N, K, 900))
        sc = gpu.t(wl.gen_fp8_scale(N, wl.scale_cols(K, 128), 0.001, 0.02, 900))
        A = torch.randn(M, K, device=gpu.dev, dtype=torch.bfloat16)
        a_sc = torch.full((1,), 0.01, device=gpu.dev, dtype=torch.float32)
        ws = torch.empty(wq.fp8_w8a8_workspace_bytes(M, K), dtype=torch.uint8, device=gpu.dev)
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=gpu.dev)
        fn = lambda: wq.fp8_weight_matmul_w8a8_ws(A, a_sc, B, sc, ws, None, 128, out=Y,
                                                  stream=gpu.stream)
        work = 2 * M * N * K / 1e12, "TFLOP/s"
    elif name == "f4f4_prefill":
        M, N, K = (m or 8192), 17408, 5120
        ly = gpu.fp4_layers(M, N, K, 1, seed0=700, bias=True)[0]
        A = torch.randn(M, K, device=gpu.dev, dtype=torch.bfloat16)
        qc, qs = wq.fp4_quantize_activation(A)
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=gpu.dev)
        fn = lambda: wq.fp4_fp4_matmul(qc, qs, ly["B"], ly["ws"], ly["ws2"], ly["bias"], out=Y,
                                       stream=gpu.stream)
        work = 2 * M * N * K / 1e12, "TFLOP/s"
    elif name == "decode_step":
        print(json.dumps(decode_step(gpu, (m or 4,), reps=reps)), flush=True)
        return
    else:
        raise SystemExit(f"unknown workload {name}")
    dt = gpu.time_each(fn, reps=reps, warmup=2, flush=True)
    print(json.dumps({"only": name, "M": m, "us": round(dt * 1e6, 2),
                      work[1]: round(work[0] / dt, 1)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="headline only (no extra workloads)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--only", default=None,
                    help="run one workload (gemv, lm_head, prefill_gate_up, prefill_down, "
                         "dequant, actq, fp8_gemv, decode_step) a few times, for profilers")
    ap.add_argument("--m", type=int, default=None, help="rows of A for --only")
    ap.add_argument("--reps", type=int, default=3, help="timed launches for --only")
    args = ap.parse_args()
    if args.only:
        run_only(args.only, args.m, args.reps)
        return
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    dist = None
    barrier_sync = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))

        def barrier_sync():
            dist.barrier()
            torch.cuda.synchronize()

    gpu = Gpu(f"cuda:{local}")
    peaks = load_peaks()
    h = bench_headline(gpu, args, rank, world, barrier_sync)
    dt = h["dt"]
    dt, dt_e2e = max_over_ranks([dt, h["dt_e2e"]], dist, gpu.dev if dist is not None else None)
    per_step = h["per_launch"] * h["launches"]
    value = weak_scaling_value(per_step * args.steps, world, dt) / 1e9
    avg_launch = dt / (args.steps * h["launches"])
    achieved = h["per_launch"] / avg_launch / 1e9
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config(),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": recorded_traffic("gemv_decode_M4_N5120_K5120"),
                     "peak_src": peaks["src"], "algorithmic_bytes_per_launch": h["per_launch"],
                     "avg_launch_us": round(avg_launch * 1e6, 3)},
        "e2e": {"value": round(weak_scaling_value(per_step * args.steps, world, dt_e2e) / 1e9, 1),
                "unit": UNIT,
                "h2d_bytes_per_step": h["h2d"], "d2h_bytes_per_step": h["d2h"]},
        "gpu_launches": h["launches"] * args.steps,
        "clocks": h["clocks"],
    }
    if not args.quick:
        line["also"] = bench_also(gpu, args, peaks)
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_oracle_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
