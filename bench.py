#!/usr/bin/env python3
"""Benchmark of the tiled block-32 quantized matmul hot path on GB300.

Headline workload: Q8_0 tiled matvec, K=4096, N=14336, batch 1 (an FFN up-projection shape).
One step = one pass of the hot path over one batch: dynamic Q8_0 quantization of the activation,
the matmul over the tiled weight and its fp32 output.  Decode shapes (up to 4 rows) run the step as
one kernel with the quantization fused in (qmm_matmul_f32); the two-call form (qmm_quantize_act +
qmm_matmul) is reported beside it; prefill shapes run qmm_quantize_act + the tensor-core GEMM.  The
weight is repacked once beforehand, as at model load.

  value   weight-tile bytes per step / device time per step (GB/s), inputs resident in HBM;
          K consecutive steps captured in one CUDA graph and timed with CUDA events on the launching
          stream, rotating through enough weight copies that the working set exceeds the 129 MB L2
          (no step hits a weight left in L2 by the previous one).
  e2e     the same metric through the C ABI with host buffers (eager launches): each step hands
          qmm_matmul_f32_ws its pinned host activation and output buffers (and a device workspace made
          once): x crosses NVLink-C2C once into the workspace, y is written over the link.  Beside it:
          qmm_matmul_f32 without a workspace, and explicit copies to and from device buffers.
  roofline  the decode matvec alone: algorithmic bytes (weight tiles + activation quants and
          scales + fp32 output) per launch / mean launch time (a graph of back-to-back launches
          timed with CUDA events), against the measured HBM copy bandwidth.
  other_configs  the remaining workloads, each as its own step (prefill GEMM in TFLOP/s).
  configs   last key of the line: the five quoted workloads -> kernel_us and roofline frac (HBM for
          the decode shapes, both HBM and bf16 tensor peak for the prefill shapes).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
HEADLINE = ("q8_0", 4096, 14336, 1)
OTHERS = [("q4_0", 4096, 4096, 1), ("iq4_nl", 4096, 4096, 8), ("q8_0", 4096, 128256, 1),
          ("q4_0", 4096, 14336, 512), ("q8_0", 4096, 128256, 128),
          # MXFP4 tiles (the next format of the pages' tile family), decode and prefill shapes
          ("mxfp4", 4096, 14336, 1), ("mxfp4", 4096, 14336, 512),
          # Q4_1 tiles (d and m per row)
          ("q4_1", 4096, 14336, 1), ("q4_1", 4096, 14336, 512),
          # Q4_K super-blocks (read through the Q4_1 tile)
          ("q4_k", 4096, 14336, 1),
          # flat (untiled) GGML rows, decode
          ("q4_0", 4096, 14336, 1, "flat"), ("q8_0", 4096, 14336, 1, "flat"), ("mxfp4", 4096, 14336, 1, "flat")]
METRIC = "tiled Q4_0/Q8_0 matvec weight GB/s (% HBM peak); prefill int8 GEMM TOPS"
# The five workloads the metric is quoted on (lm-head at batch 1 and 128), summarized at the end of
# the printed line: kernel time and roofline fraction of each.
SUMMARY = [("c1", ("q4_0", 4096, 4096, 1)), ("c2", HEADLINE), ("c3", ("iq4_nl", 4096, 4096, 8)),
           ("c4", ("q4_0", 4096, 14336, 512)), ("c5_b1", ("q8_0", 4096, 128256, 1)),
           ("c5_b128", ("q8_0", 4096, 128256, 128))]


def workload_name(type_, K, N, M, layout="tiled"):
    kind = "prefill_gemm" if M > 16 else ("matvec" if M == 1 else "matmul")
    if layout == "flat":
        kind = "flat_" + kind
    return f"{type_}_{kind}_K{K}_N{N}_M{M}"


def int8_library_tops(torch, n=8192, reps=5):
    """Reference point for the int8 tensor rate on this GPU: torch._int_mm (the vendor library's int8
    GEMM) on n x n x n, timed with CUDA events.  Context only; the prefill GEMM's roofline is the
    measured bf16 peak (there is no int8 tcgen05 on sm_103a)."""
    try:
        a = torch.randint(-127, 128, (n, n), dtype=torch.int8, device="cuda")
        b = torch.randint(-127, 128, (n, n), dtype=torch.int8, device="cuda")
        torch._int_mm(a, b)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            torch._int_mm(a, b)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        return {"tops": round(2.0 * n ** 3 / (ms * 1e-3) / 1e12, 1), "shape": f"{n}^3", "via": "torch._int_mm"}
    except Exception as exc:  # an int8 GEMM the library does not offer on this GPU
        return {"tops": None, "error": str(exc)[:120]}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
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
            for name, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons), "samples": len(sm)}


KERNEL_FILES = {"matvec": ("matvec.cu", "qmm_internal.cuh", "pipeline.cuh"),
                "gemm": ("gemm_fold.cu", "gemm_tc.cu", "tc_common.cuh", "qmm_internal.cuh", "pipeline.cuh")}


def kernel_kind(workload):
    return "gemm" if "prefill_gemm" in workload else "matvec"


def kernel_source_hash(kind="matvec"):
    """Hash of the sources a kernel family is compiled from, with comments and blank lines removed
    (a comment edit, or an edit of another kernel's file, does not change the kernels the recorded
    counters were taken on)."""
    import re

    h = hashlib.sha256()
    for name in KERNEL_FILES[kind]:
        with open(os.path.join(ROOT, "block_quantized_matmul_gb300", "csrc", name)) as f:
            text = re.sub(r"//[^\n]*", "", f.read())
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(name.encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """dram bytes per launch from a committed ncu capture, if it was taken on the current kernels."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
        ent = rec.get(workload)
        if ent and ent.get("source_hash") == kernel_source_hash(kernel_kind(workload)):
            return ent.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


class Workload:
    def __init__(self, torch, qmm, type_, K, N, M, layout="tiled", seed=0, copies=None):
        self.torch, self.qmm = torch, qmm
        self.type_, self.K, self.N, self.M = type_, K, N, M
        # flat: the decode matmul reads the GGML rows as they are (qmm_matmul_flat), no repack
        self.flat_layout = layout == "flat"
        self.tiled_bytes = qmm.flat_size(type_, K, N) if self.flat_layout else qmm.tiled_size(type_, K, N)
        g = torch.Generator(device="cuda")
        g.manual_seed(seed)
        # weights ~ N(0, 0.02^2), quantized and repacked once on the GPU (model-load path)
        flat = torch.empty(qmm.flat_size(type_, K, N), dtype=torch.uint8, device="cuda")
        rows = max(1, (256 << 20) // (4 * K))
        for r0 in range(0, N, rows):
            r1 = min(N, r0 + rows)
            w = torch.randn(r1 - r0, K, device="cuda", generator=g) * 0.02
            qmm.qmm_quantize_weight(type_, w, r1 - r0, K, K,
                                    flat[r0 * (K // 32) * qmm.block_size(type_):])
            del w
        self.copies = copies or max(2, -(-3 * L2_BYTES // self.tiled_bytes) if self.tiled_bytes < 3 * L2_BYTES else 2)
        self.tiled = []
        for _ in range(self.copies):
            t = torch.empty(self.tiled_bytes, dtype=torch.uint8, device="cuda")
            if self.flat_layout:
                t.copy_(flat)
            else:
                qmm.qmm_repack(type_, flat, K, N, t)
            self.tiled.append(t)
        del flat
        # activations ~ N(0,1), 1 % outliers x20 for the prefill workload
        self.n_act = 4
        xs = torch.randn(self.n_act, M, K, device="cuda", generator=g)
        if M > 16:
            mask = torch.rand(self.n_act, M, K, device="cuda", generator=g) < 0.01
            xs = torch.where(mask, xs * 20.0, xs)
        self.x = xs.contiguous()
        self.a_q = torch.empty((M, K), dtype=torch.int8, device="cuda")
        self.a_d = torch.empty((M, K // 32), dtype=torch.int16, device="cuda")
        self.y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        # prefill shapes take the tensor-core path with a caller workspace (qmm_matmul_ws)
        self.ws_bytes = qmm.matmul_workspace_size(M, K) if M > qmm.decode_max_m() else 0
        self.ws = torch.empty(self.ws_bytes + 256, dtype=torch.uint8, device="cuda") if self.ws_bytes else None
        self.ws_ptr = (self.ws.data_ptr() + (-self.ws.data_ptr()) % 256) if self.ws_bytes else None
        # decode shapes up to 4 tokens run the fused kernel (qmm_matmul_f32); from 5 tokens on the two
        # calls are faster (the fused kernel quantizes all M rows in every CTA)
        self.fused = M <= 4 and not self.flat_layout
        torch.cuda.synchronize()

    def step(self, i, stream):
        """One pass of the hot path: activation quantization + matmul + epilogue.  Decode shapes run
        it as one kernel (qmm_matmul_f32), prefill shapes as quantize + tensor-core GEMM."""
        if self.fused:
            self.qmm.qmm_matmul_f32(self.type_, self.tiled[i % self.copies], self.K, self.N, self.x[i % self.n_act],
                                    self.K, self.M, self.y, self.N, stream=stream)
        else:
            self.step_two_call(i, stream)

    def step_two_call(self, i, stream):
        self.qmm.qmm_quantize_act(self.x[i % self.n_act], self.M, self.K, self.K, self.a_q, self.a_d, stream=stream)
        self.matmul_only(i, stream)

    def kernel_only(self, i, stream):
        """The dominant kernel alone: the fused decode kernel, the decode kernel or the GEMM."""
        if self.fused:
            self.step(i, stream)
        else:
            self.matmul_only(i, stream)

    def matmul_only(self, i, stream):
        if self.flat_layout:
            self.qmm.qmm_matmul_flat(self.type_, self.tiled[i % self.copies], self.K, self.N, self.a_q, self.a_d,
                                     self.M, self.y, self.N, stream=stream)
        elif self.ws_bytes:
            self.qmm.qmm_matmul_ws(self.type_, self.tiled[i % self.copies], self.K, self.N, self.a_q, self.a_d, self.M,
                                   self.y, self.N, self.ws_ptr, self.ws_bytes, stream=stream)
        else:
            self.qmm.qmm_matmul(self.type_, self.tiled[i % self.copies], self.K, self.N, self.a_q, self.a_d, self.M,
                                self.y, self.N, stream=stream)

    def algorithmic_bytes(self):
        """Bytes the dominant kernel must move once: the weight tiles, its activation input (fp32 rows
        for the fused decode kernel, int8 quants + fp16 scales for the GEMM) and the fp32 output."""
        act = self.M * self.K * 4 if self.fused else self.M * self.K + self.M * (self.K // 32) * 2
        return self.tiled_bytes + act + self.M * self.N * 4

    def launches_per_step(self):
        """Kernels of this library launched by one step: the decode kernel once per 16-row group and K
        pass (K is split only beyond its 64 KB activation staging budget), plus the activation
        quantizer unless it is fused; or quantize + activation prepare + GEMM."""
        nkt = self.K // 32
        if self.flat_layout:       # groups of 4 rows, K passes of at most 384 blocks
            return 1 + -(-self.M // 4) * -(-nkt // min(nkt, 384))
        if self.M > 16:
            return 3
        n = 0 if self.fused else 1
        for m0 in range(0, self.M, 16):
            mm = min(16, self.M - m0)
            mt = mm if mm > 4 else (mm if mm <= 2 else 4)
            nkc = max(1, min(nkt, 65536 // (64 * mt)))
            n += -(-nkt // nkc)
        return n

    def flops(self):
        return 2.0 * self.M * self.N * self.K


def capture(torch, fn, n, stream):
    """CUDA graph of n consecutive calls fn(0..n-1) on `stream` (no host work left in the loop)."""
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            fn(i, stream)
    torch.cuda.synchronize()
    return g


def time_graph(torch, g, stream, n):
    """Device time per call of a captured graph of n calls: events on the launching stream."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n        # ms per call


def time_steps(torch, fn, steps, stream):
    """Eager loop (host launch overhead included), events on the launching stream."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(steps):
        fn(i, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps        # ms per step


def kernel_time(torch, wl, steps, stream):
    """Mean duration of the dominant kernel alone: a graph of `steps` back-to-back launches (rotating
    weight copies), timed with events on the launching stream."""
    g = capture(torch, wl.kernel_only, steps, stream)
    time_graph(torch, g, stream, steps)            # warm replay
    return time_graph(torch, g, stream, steps)


def run_gpu(args):
    import torch

    import block_quantized_matmul_gb300 as qmm
    from block_quantized_matmul_gb300 import build

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    build.build()
    hbm_peak, bf16_peak, peak_src = measured_peaks()
    stream = torch.cuda.Stream()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # ---------------- headline workload ----------------
    type_, K, N, M = HEADLINE
    wl = Workload(torch, qmm, type_, K, N, M)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            wl.step(i, stream)
    torch.cuda.synchronize()
    # The K timed steps run as one CUDA graph (act-quant + matmul per step, fused into one kernel for
    # this decode shape; rotating weights), so the measurement is the device time of the hot path,
    # not Python launch overhead.
    graph = capture(torch, wl.step, args.steps, stream)
    time_graph(torch, graph, stream, args.steps)         # warm-up replay
    with ClockSampler(local) as clk:
        barrier()
        ms = time_graph(torch, graph, stream, args.steps)
        barrier()
        # keep the GPU busy a little longer so the clock record is not empty on short runs
        t_end = time.time() + 0.5
        while time.time() < t_end:
            with torch.cuda.stream(stream):
                graph.replay()
            torch.cuda.synchronize()
    del graph
    if world > 1:
        t = torch.tensor([ms], device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    value = wl.tiled_bytes * world / (ms * 1e-3) / 1e9

    # roofline of the decode kernel
    kms = kernel_time(torch, wl, max(20, min(args.steps, 200)), stream)
    achieved = wl.algorithmic_bytes() / (kms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                "traffic": recorded_traffic(workload_name(*HEADLINE)), "kernel_us": round(kms * 1e3, 3)}

    # the same step as two calls (qmm_quantize_act, then qmm_matmul): for comparison only
    g2 = capture(torch, wl.step_two_call, args.steps, stream)
    time_graph(torch, g2, stream, args.steps)
    two_ms = time_graph(torch, g2, stream, args.steps)
    del g2
    two_call = {"ms_per_step": round(two_ms, 5), "value": round(wl.tiled_bytes / (two_ms * 1e-3) / 1e9, 1),
                "unit": "GB/s", "step": "qmm_quantize_act + qmm_matmul (two kernels)"}
    wl_launches = wl.launches_per_step()

    # end to end through the C ABI with host buffers (pinned), eager launches.  The call is given the
    # host buffers themselves and a device workspace (allocated once, as at start-up): a first kernel
    # copies x over NVLink-C2C into the workspace, the decode kernel writes y to host memory.  Beside
    # it: the same call without a workspace (the decode kernel reads x over the link, once per
    # thread-block cluster), and an explicit host-to-device copy, the call on device buffers and a
    # device-to-host copy.
    x_host = torch.empty((wl.n_act, M, K), dtype=torch.float32).pin_memory()
    x_host.copy_(wl.x.cpu())
    y_host = torch.empty((M, N), dtype=torch.float32).pin_memory()
    x_dev = torch.empty((M, K), dtype=torch.float32, device="cuda")
    ws_bytes = qmm.matmul_f32_workspace_size(M, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")

    def e2e_step(i, s):
        qmm.qmm_matmul_f32_ws(type_, wl.tiled[i % wl.copies], K, N, x_host[i % wl.n_act], K, M, y_host, N, ws,
                              ws_bytes, stream=s)

    def e2e_nows_step(i, s):
        qmm.qmm_matmul_f32(type_, wl.tiled[i % wl.copies], K, N, x_host[i % wl.n_act], K, M, y_host, N, stream=s)

    def e2e_copy_step(i, s):
        x_dev.copy_(x_host[i % wl.n_act], non_blocking=True)
        qmm.qmm_matmul_f32(type_, wl.tiled[i % wl.copies], K, N, x_dev, K, M, wl.y, N, stream=s)
        y_host.copy_(wl.y, non_blocking=True)

    def e2e_time(fn):
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                fn(i, stream)
            torch.cuda.synchronize()
            return time_steps(torch, fn, args.steps, stream)

    e2e_ms, e2e_nows_ms, e2e_copy_ms = e2e_time(e2e_step), e2e_time(e2e_nows_step), e2e_time(e2e_copy_step)
    e2e = {"value": round(wl.tiled_bytes * world / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
           "h2d_bytes_per_step": M * K * 4, "d2h_bytes_per_step": M * N * 4, "ms_per_step": round(e2e_ms, 5),
           "transfer": "qmm_matmul_f32_ws with pinned host x and y and a device workspace: one kernel copies x "
                       "over NVLink-C2C, the decode kernel writes y over it",
           "without_workspace": {"value": round(wl.tiled_bytes * world / (e2e_nows_ms * 1e-3) / 1e9, 1),
                                 "unit": "GB/s", "ms_per_step": round(e2e_nows_ms, 5),
                                 "transfer": "qmm_matmul_f32 with pinned host x and y: the decode kernel reads x "
                                             "over NVLink-C2C once per thread-block cluster"},
           "with_copies": {"value": round(wl.tiled_bytes * world / (e2e_copy_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                           "ms_per_step": round(e2e_copy_ms, 5),
                           "transfer": "cudaMemcpyAsync host-to-device, the call on device buffers, "
                                       "cudaMemcpyAsync device-to-host"}}

    # ---------------- other workloads ----------------
    others = []
    if not args.headline_only:
        del wl
        torch.cuda.empty_cache()
        for cfg in OTHERS:
            o = Workload(torch, qmm, *cfg)
            with torch.cuda.stream(stream):
                for i in range(max(3, args.warmup)):
                    o.step(i, stream)
            torch.cuda.synchronize()
            n = max(10, min(args.steps, 100 if cfg[3] > 16 else 1000))
            og = capture(torch, o.step, n, stream)
            time_graph(torch, og, stream, n)
            oms = time_graph(torch, og, stream, n)
            del og
            okms = kernel_time(torch, o, min(n, 200), stream)
            ent = {"workload": workload_name(*cfg), "ms_per_step": round(oms, 5), "kernel_us": round(okms * 1e3, 3),
                   "launches_per_step": o.launches_per_step(),
                   "weight_GBps": round(o.tiled_bytes / (oms * 1e-3) / 1e9, 1)}
            kbytes = o.algorithmic_bytes() / (okms * 1e-3) / 1e9
            ent["roofline_hbm"] = {"achieved": round(kbytes, 1), "peak": hbm_peak, "unit": "GB/s",
                                   "frac": round(kbytes / hbm_peak, 4)}
            if cfg[3] > 16:
                tf = o.flops() / (okms * 1e-3) / 1e12
                ent["TFLOPs"] = round(tf, 1)
                folded = cfg[0] in ("q4_0", "q8_0", "iq4_nl")
                note = ("folded-scale GEMM: block scales inside exact hi + lo fp16 operands, three fp16 tcgen05 "
                        "MMAs per K step (the tensor pipe executes 3x the algorithmic flops)" if folded else
                        "fp16 tcgen05 MMA on exact integer operands, per-block fp32 rescale")
                ent["roofline_tensor"] = {"achieved": round(tf, 1), "peak": bf16_peak, "unit": "TFLOP/s",
                                          "frac": round(tf / bf16_peak, 4),
                                          "note": note + " (no int8 tcgen05 on sm_103a); peak = measured bf16 burst"}
            others.append(ent)
            del o
            torch.cuda.empty_cache()
    status = qmm.qmm_device_status()

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8",
        "arith": "Q8_0 weights x int8 activations: exact integer block sums on fp16 tensor cores, fp32 scaling",
        "data": "synthetic (seeded: weights N(0,0.02^2) -> Q8_0 tiles, activations N(0,1))",
        "config": {"workload": workload_name(*HEADLINE), "type": type_, "K": K, "N": N, "M": M,
                   "step": "qmm_matmul_f32: activation quantization fused into the decode kernel",
                   "l2": f"{wl_copies_note(qmm, type_, K, N)}", "parallelism": f"replica x{world}"},
        "pct_hbm_peak": round(value / hbm_peak * 100, 2),
        "roofline": roofline,
        "e2e": e2e,
        "two_call_step": two_call,
        "gpu_launches": args.steps * wl_launches,
        "clocks": clk.summary(),
        "device_status": status,
        "other_configs": others,
        "int8_library_reference": None if args.headline_only else int8_library_tops(torch),
    }
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(HEADLINE, budget_s=args.cpu_seconds) if not args.no_cpu else None
        if line["cpu_baseline"] is not None:
            line["cpu_baseline"]["all_cores"] = cpu_baseline_all_cores(HEADLINE)
        line["configs"] = summary_configs(line)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def summary_configs(line):
    """Compact per-workload summary of SUMMARY from the headline roofline and other_configs."""
    by_name = {o["workload"]: o for o in line.get("other_configs") or []}
    out = {}
    for key, cfg in SUMMARY:
        name = workload_name(*cfg)
        if cfg == HEADLINE:
            r = line["roofline"]
            out[key] = {"workload": name, "kernel_us": r["kernel_us"], "frac": r["frac"], "of": "hbm"}
            continue
        o = by_name.get(name)
        if o is None:
            continue
        ent = {"workload": name, "kernel_us": o["kernel_us"], "frac": o["roofline_hbm"]["frac"], "of": "hbm"}
        if "roofline_tensor" in o:
            ent["tensor_frac"] = o["roofline_tensor"]["frac"]
        out[key] = ent
    return out


def wl_copies_note(qmm, type_, K, N):
    tb = qmm.tiled_size(type_, K, N)
    copies = max(2, -(-3 * L2_BYTES // tb) if tb < 3 * L2_BYTES else 2)
    return f"inputs larger than L2: {copies} rotating weight copies x {tb} B = {copies * tb} B > 129 MB L2"


# ---------------------------------------------------------------------------------------------
# CPU oracle timing (reported baseline; also the --impl reference arm)
# ---------------------------------------------------------------------------------------------
def _oracle_passes(cfg, budget_s, rows, seed):
    """One host process: the oracle's act-quant + matmul over a bounded sample, repeated for budget_s.
    Returns (tile bytes processed, seconds)."""
    import oracle
    from block_quantized_matmul_gb300 import synth

    type_, K, N, M = cfg
    w = synth.weights(rows, K, seed=seed)
    x = synth.activations(M, K)
    tiled = oracle.repack(type_, oracle.quantize_rows(type_, w), K, rows)
    bytes_per_pass = oracle.tiled_bytes(type_, K, rows)
    passes, t0 = 0, time.perf_counter()
    while True:
        a_q, a_d = oracle.quantize_act(x)
        oracle.matmul(type_, tiled, K, rows, a_q, a_d)
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s or passes >= 10000:
            return bytes_per_pass * passes, el


def _oracle_worker(job):
    return _oracle_passes(*job)


def cpu_baseline_all_cores(cfg, budget_s=1.5, rows=256):
    """The same oracle on every host core at once: one spawned process per core, each timing its own
    sample of `rows` weight rows for budget_s; aggregate bytes / the longest process's time."""
    import multiprocessing as mp

    import oracle

    oracle.build()
    n = os.cpu_count() or 1
    with mp.get_context("spawn").Pool(n) as pool:
        res = pool.map(_oracle_worker, [(cfg, budget_s, rows, 1000 + i) for i in range(n)])
    total = sum(b for b, _ in res)
    el = max(t for _, t in res)
    return {"value": round(total / el / 1e9, 5), "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"{workload_name(*cfg)}: {n} processes, each {rows} weight rows of act-quant + matmul "
                      f"for {budget_s} s (single-threaded C oracle per process)"}


def cpu_baseline(cfg, budget_s=15.0, rows=1024):
    import numpy as np

    import oracle
    from block_quantized_matmul_gb300 import synth

    type_, K, N, M = cfg
    rows = min(rows, N)
    w = synth.weights(rows, K)
    x = synth.activations(M, K)
    tiled = oracle.repack(type_, oracle.quantize_rows(type_, w), K, rows)
    bytes_per_pass = oracle.tiled_bytes(type_, K, rows)
    passes, t0 = 0, time.perf_counter()
    while True:
        a_q, a_d = oracle.quantize_act(x)
        oracle.matmul(type_, tiled, K, rows, a_q, a_d)
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s or passes >= 10000:
            break
    gbps = bytes_per_pass * passes / el / 1e9
    return {"value": round(gbps, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{workload_name(*cfg)}: first {rows} of {N} weight rows ({bytes_per_pass} tile bytes), "
                      f"{passes} passes of act-quant + matmul in {el:.1f} s, single-threaded C oracle",
            "host_cores_available": os.cpu_count()}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_baseline(HEADLINE, budget_s=per_step)
    t0 = time.perf_counter()
    vals = [cpu_baseline(HEADLINE, budget_s=per_step) for _ in range(args.steps)]
    el = time.perf_counter() - t0
    v = sum(r["value"] for r in vals) / len(vals)
    type_, K, N, M = HEADLINE
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 5), "unit": "GB/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64/f64",
            "data": "synthetic (seeded)",
            "config": {"workload": workload_name(*HEADLINE), "type": type_, "K": K, "N": N, "M": M},
            "cpu_baseline": {"value": round(v, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": vals[0]["sample"]},
            "e2e": {"value": round(v, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile(args):
    """Set up one workload and launch its dominant kernel warmup + steps times (for ncu captures)."""
    import torch

    import block_quantized_matmul_gb300 as qmm
    from block_quantized_matmul_gb300 import build

    torch.cuda.set_device(0)
    build.build()
    cfg = {workload_name(*c): c for c in [HEADLINE] + OTHERS}[args.profile]
    wl = Workload(torch, qmm, *cfg, copies=1)
    stream = torch.cuda.current_stream()
    wl.step(0, stream)
    for i in range(args.warmup + args.steps):
        wl.kernel_only(i, stream)
    torch.cuda.synchronize()
    print(json.dumps({"profile": args.profile, "launches": args.warmup + args.steps + 1,
                      "status": qmm.qmm_device_status()}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile", default=None, help="launch one workload's matmul kernel only (for ncu)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--headline-only", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
