#!/usr/bin/env python3
"""Benchmark of the Q8_0 hot path (row quantizer + qdot_t) on GB300.

A step is one pass of the path over one batch: quantize the activation rows
(pq_quantize_q8_0), then contract them with the resident Q8_0 weights
(pq_qdot_q8_0).  The headline workload is the decode projection
M=1, K=4096, N=4096; its metric is weight GB/s (stored weight bytes,
1.125 B per weight, per second).  The same line carries the prompt GEMM
(M=512, K=4096, N=14336) as int8-equivalent TOPS (2*M*N*K per second) and the
other workloads.

Timing: W warm-up steps, then exactly K steps captured in one CUDA graph and
replayed once (after one untimed launch of the same graph, which uploads it to
the device), bracketed by a barrier and torch.cuda.synchronize(); the step
time is taken with CUDA events on the launching stream, max over ranks.  Each
step reads the next of B rotating copies of the weights, with B * bytes
>= 2 x L2, so a step never finds its weights in L2.  External event nodes
around every kernel in the graph give each kernel's average duration for the
roofline.  SM clocks and throttle reasons are sampled through NVML during the
timed region.

``--impl reference`` times the CPU oracle (the plain C reference) on the same
workload and metric on the host cores instead.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gemm_q8_qdot_gb300 import workloads  # noqa: E402

METRIC = "Q8_0 matvec weight GB/s (M=1) & int8 GEMM TOPS (M=512), % of roofline"
HEADLINE = "decode_m1_k4096_n4096"
PROMPT = "prompt_m512_k4096_n14336"
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- helpers

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_digest(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


KERNEL_SOURCES = {
    "qdot_simt": ["gemm_q8_qdot_gb300/csrc/qdot_simt.cu", "gemm_q8_qdot_gb300/csrc/pq_device.cuh"],
    "qdot_tc": ["gemm_q8_qdot_gb300/csrc/qdot_tc.cu", "gemm_q8_qdot_gb300/csrc/tc_ptx.cuh",
                "gemm_q8_qdot_gb300/csrc/pq_device.cuh"],
    "quantize": ["gemm_q8_qdot_gb300/csrc/quantize.cu"],
    "qdot_fused": ["gemm_q8_qdot_gb300/csrc/qdot_simt.cu", "gemm_q8_qdot_gb300/csrc/pq_device.cuh"],
    "qdot_q50": ["gemm_q8_qdot_gb300/csrc/qdot_q50.cu", "gemm_q8_qdot_gb300/csrc/pq_device.cuh"],
    "qdot_mma": ["gemm_q8_qdot_gb300/csrc/qdot_mma.cu", "gemm_q8_qdot_gb300/csrc/pq_device.cuh"],
    "qdot_mmt": ["gemm_q8_qdot_gb300/csrc/qdot_mmt.cu", "gemm_q8_qdot_gb300/csrc/tc_ptx.cuh",
                 "gemm_q8_qdot_gb300/csrc/pq_device.cuh"],
    "qdot_q50_fused": ["gemm_q8_qdot_gb300/csrc/qdot_q50.cu", "gemm_q8_qdot_gb300/csrc/pq_device.cuh"],
    "qdot_tcw": ["gemm_q8_qdot_gb300/csrc/qdot_tcw.cu", "gemm_q8_qdot_gb300/csrc/tc_ptx.cuh",
                 "gemm_q8_qdot_gb300/csrc/pq_device.cuh"],
}


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from profiles/dram_traffic.md, if taken on the current source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.md")
    try:
        digest = source_digest(KERNEL_SOURCES[kernel])
        with open(path) as f:
            for line in f:
                cells = [c.strip() for c in line.strip().strip("|").split("|")]
                if len(cells) >= 4 and cells[0] == kernel and cells[1] == workload and cells[2] == digest:
                    return float(cells[3])
    except (OSError, ValueError, KeyError):
        pass
    return None


class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML in a thread."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device_index: int = 0, period_s: float = 0.002):
        self.samples: list[tuple[float, int, int]] = []
        self.period = period_s
        self.ok = False
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            import torch
            props = torch.cuda.get_device_properties(torch_device_index)
            bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0".encode()
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
                if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(torch_device_index), ctypes.byref(h)) != 0:
                    return
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            self.nv, self.h, self.ok = nv, h, True
        except Exception:
            self.ok = False

    def _sample(self):
        mhz = ctypes.c_uint()
        reasons = ctypes.c_ulonglong()
        self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz))
        fn = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
        fn(self.h, ctypes.byref(reasons))
        self.samples.append((time.perf_counter(), int(mhz.value), int(reasons.value)))

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    def stop(self):
        if self._thread:
            self._stop.set()
            self._thread.join()
            self._sample()

    def summary(self, t0: float, t1: float):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["nvml unavailable"]}
        inside = [s for s in self.samples if t0 <= s[0] <= t1] or self.samples[-2:]
        reasons = set()
        for _, _, r in inside:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(inside)}


def make_event():
    """A timing event that becomes an event-record node when captured in a graph."""
    import torch
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return _DriverEvent()


class _DriverEvent:
    """Driver-API event recorded with CU_EVENT_RECORD_EXTERNAL (for torch without `external`)."""
    _cu = None

    def __init__(self):
        if _DriverEvent._cu is None:
            _DriverEvent._cu = ctypes.CDLL("libcuda.so.1")
        self.ev = ctypes.c_void_p()
        assert self._cu.cuEventCreate(ctypes.byref(self.ev), 0) == 0

    def record(self, stream=None):
        import torch
        s = (stream or torch.cuda.current_stream()).cuda_stream
        assert self._cu.cuEventRecordWithFlags(self.ev, ctypes.c_void_p(s), 1) == 0

    def elapsed_time(self, other) -> float:
        ms = ctypes.c_float()
        fn = getattr(self._cu, "cuEventElapsedTime_v2", None) or self._cu.cuEventElapsedTime
        assert fn(ctypes.byref(ms), self.ev, other.ev) == 0
        return float(ms.value)


# ----------------------------------------------------------------------------- distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_units: float, per_rank_seconds: float, world: int, device=None):
    """Whole-job throughput: units of all ranks over the slowest rank's time."""
    t = max_over_ranks(per_rank_seconds, world, device)
    return per_rank_units * world / t, t


# ----------------------------------------------------------------------------- our arm

class Problem:
    """Device buffers of one workload: f32 activations, rotating Q8_0 weight copies, outputs.

    A step quantizes the activation rows and contracts them with the weights:
    for M <= 16 (M <= 8 with Q5_0 weights) through the one-call entry point
    (pq_quantize_qdot_q8_0, or pq_quantize_q50_qdot for Q5_0 weights, which
    also writes the quantized rows), otherwise pq_quantize_q8_0 then
    pq_qdot_q8_0 / pq_q50_qdot; `fused=False` forces the two-call sequence.
    """

    def __init__(self, pq, wl: workloads.Workload, device, fused: bool = True, split: tuple[int, int] = (0, 1)):
        import dataclasses

        import torch
        self.wl = wl
        self.pq = pq
        self.q50 = wl.w_format == "q5_0"
        self.fused = fused and wl.M <= (8 if self.q50 else 16)
        x = workloads.activations(wl)
        self.x_host = torch.from_numpy(x).pin_memory()
        # column split over `world` ranks: this rank holds the weight rows of its shard
        # of a layer world x N wide (drawn with a rank-dependent seed), x is replicated
        self.rank, self.world = split
        wl_w = dataclasses.replace(wl, index=wl.index + 1000 * self.rank) if self.rank else wl
        if self.q50:
            w5, ws = workloads.q50_weights(wl_w)
            W, WS = torch.from_numpy(w5).to(device), torch.from_numpy(ws).to(device)
        else:
            w = torch.from_numpy(workloads.weights(wl_w)).to(device)
            W, WS = pq.quantize_q8_0(w)
            del w
        wbytes = W.numel() + WS.numel() * 4
        self.copies = max(2, -(-2 * L2_BYTES // wbytes))
        self.W = [W] + [W.clone() for _ in range(self.copies - 1)]
        self.WS = [WS] + [WS.clone() for _ in range(self.copies - 1)]
        # the activation rows arrive after the weights are resident, as in a decode
        # loop where the previous operation has just written them
        self.x = self.x_host.to(device)
        self.A = torch.empty((wl.M, wl.K), dtype=torch.int8, device=device)
        self.AS = torch.empty((wl.M, wl.K // 32), dtype=torch.float32, device=device)
        self.C = torch.empty((wl.M, wl.N), dtype=torch.float32, device=device)
        # the gathered output of the column split: rank r's [M, N] block at rows
        # [r*M, (r+1)*M) (for M = 1 this is the row-major [1, world*N] result itself)
        self.C_all = torch.empty((self.world * wl.M, wl.N), dtype=torch.float32, device=device) \
            if self.world > 1 else None
        self.C_host = torch.empty((self.world * wl.M, wl.N), dtype=torch.float32).pin_memory()
        torch.cuda.synchronize()

    def step(self, t: int, events=None):
        self._step(t, events)
        if self.C_all is not None:  # the column split's exchange: all-gather of C (NCCL)
            import torch.distributed as dist
            dist.all_gather_into_tensor(self.C_all, self.C)

    def _step(self, t: int, events=None):
        c = t % self.copies
        if self.fused:
            if events is not None:
                events[0].record()
                events[1].record()
            if self.q50:
                self.pq.quantize_q50_qdot(self.x, self.W[c], self.WS[c], self.C, A=self.A, AS=self.AS)
            else:
                self.pq.quantize_qdot_q8_0(self.x, self.W[c], self.WS[c], self.C, A=self.A, AS=self.AS)
            if events is not None:
                events[2].record()
            return
        if events is not None:
            events[0].record()
        self.pq.quantize_q8_0(self.x, self.A, self.AS)
        if events is not None:
            events[1].record()
        self.qdot(c)
        if events is not None:
            events[2].record()

    def qdot(self, c: int):
        if self.q50:
            self.pq.q50_qdot(self.A, self.AS, self.W[c], self.WS[c], self.C)
        else:
            self.pq.qdot_q8_0(self.A, self.AS, self.W[c], self.WS[c], self.C)

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes the dominant kernel must move per launch.  qdot_t: W, WS, A, AS read
        once, C written once; the fused step reads x (f32) instead of A, AS and also
        writes A, AS."""
        wl = self.wl
        base = wl.weight_bytes + wl.M * wl.K + 4 * wl.M * (wl.K // 32) + 4 * wl.M * wl.N
        return base + 4 * wl.M * wl.K if self.fused else base


def _capture(prob: Problem, first: int, steps: int, stream, events=None, only_qdot=False):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for t in range(steps):
            if only_qdot:
                prob.qdot((first + t) % prob.copies)
            else:
                prob.step(first + t, events[t] if events else None)
    return g


# Cycles of a spin kernel enqueued ahead of a timed graph (~50 us at 2 GHz):
# it holds the stream until the graph launch has been submitted, so the timed
# region (start event to end event) holds the graph's K steps and not the
# host's launch latency, and the GPU does not idle meanwhile.
HOLD_CYCLES = 100_000


def _replay_ms(g, stream) -> float:
    import torch
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(HOLD_CYCLES)
        start.record(stream)
        g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def time_graph(prob: Problem, steps: int, warmup: int, world: int, sampler=None):
    """Times K steps captured in one graph; returns the step-region time and per-kernel durations.

    The timed graph holds the K steps and nothing else.  Per-kernel durations
    come from replaying the same K steps captured with an external timing event
    around each kernel (the event nodes add their own latency, so these
    durations are upper bounds); a graph of the K qdot launches alone gives a
    second figure (its launch gaps included).
    """
    import torch
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for t in range(2):
            prob.step(t)  # eager warm-up of the launch path
    stream.synchronize()
    g_warm = _capture(prob, 0, warmup, stream)
    g = _capture(prob, warmup, steps, stream)
    evs = [[make_event() for _ in range(3)] for _ in range(steps)]
    g_ev = _capture(prob, warmup, steps, stream, events=evs)
    g_qdot = _capture(prob, warmup, steps, stream, only_qdot=True)
    # the first launch of an instantiated graph also uploads it to the device:
    # launch every graph once, untimed, before any timed replay
    for gr in (g_warm, g, g_ev, g_qdot):
        with torch.cuda.stream(stream):
            gr.replay()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()  # before the warm replays: its thread start leaves no idle gap before timing
    # warm replays of the W warm-up steps and of the timed steps themselves right
    # before the timed replay, so that the GPU has no idle gap to fall out of its
    # load state in; then the barrier (a no-op for one rank) and a synchronize
    with torch.cuda.stream(stream):
        g_warm.replay()
        g.replay()
    stream.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ms = _replay_ms(g, stream)
    t1 = time.perf_counter()
    barrier(world)
    if sampler:
        sampler.stop()
    _replay_ms(g_ev, stream)
    quant_ms = statistics.fmean(e[0].elapsed_time(e[1]) for e in evs)
    qdot_ms = statistics.fmean(e[1].elapsed_time(e[2]) for e in evs)
    qdot_only_ms = _replay_ms(g_qdot, stream) / steps
    return ms, quant_ms, qdot_ms, qdot_only_ms, (t0, t1)


def time_reader(prob: Problem, steps: int, early: bool) -> float:
    """Mean time of the test-only streaming reader (the one-row step's weight traffic without
    its arithmetic) over the same rotating weight copies, K launches in one graph (ms)."""
    import torch
    out = torch.empty((prob.wl.N,), dtype=torch.float32, device=prob.x.device)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for t in range(2):
            prob.pq.debug_stream_read(prob.W[t % prob.copies], prob.WS[t % prob.copies], out, early=early)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for t in range(steps):
            prob.pq.debug_stream_read(prob.W[t % prob.copies], prob.WS[t % prob.copies], out, early=early)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    return _replay_ms(g, stream) / steps


def time_e2e(prob: Problem, steps: int, warmup: int):
    """Through the public API with host buffers, per step: the H2D copy of x from pinned host
    memory, the decode step, the D2H copy of C into pinned host memory (for Q8_0 weights one
    pq_quantize_qdot_q8_0_host call enqueues all three), then a synchronize."""
    import torch
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    for t in range(warmup + steps):
        if t == warmup:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
        if prob.q50 or prob.world > 1:
            prob.x.copy_(prob.x_host, non_blocking=True)
            prob.step(t)  # with the column split: the local step, then the all-gather of C
            prob.C_host.copy_(prob.C_all if prob.world > 1 else prob.C, non_blocking=True)
        else:
            c = t % prob.copies
            prob.pq.quantize_qdot_q8_0_host(prob.x_host, prob.W[c], prob.WS[c], prob.C_host)
        stream.synchronize()
    dt = time.perf_counter() - t0
    return dt, prob.x_host.numel() * 4, prob.C_host.numel() * 4


def set_host_path(pq, which: int) -> None:
    """Test hook of the host-buffer step: 0 host buffers in place (default), 1 copies."""
    lib = pq.load()
    lib.pq_debug_set_host_path.argtypes = [ctypes.c_int]
    lib.pq_debug_set_host_path.restype = ctypes.c_int
    if lib.pq_debug_set_host_path(int(which)) != 0:
        raise RuntimeError("pq_debug_set_host_path failed")


def fused_is_one_kernel(prob: Problem) -> bool:
    """Whether the one-call step runs as a single fused kernel for this shape:
    pq_quantize_qdot_q8_0 for one row (any N, its CTAs take further columns beyond
    one per SM; 9..16 rows are the quantizer and the TMA-fed warp-level MMA
    kernel); pq_quantize_q50_qdot for one row (32 columns per CTA, at most two
    waves)."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    if prob.q50:
        return prob.wl.M == 1 and -(-prob.wl.N // 32) <= 2 * sms
    return prob.wl.M == 1


def roofline_for(prob: Problem, qdot_ms: float, peaks, peak_src: str, one_kernel: bool = False):
    wl = prob.wl
    if wl.M <= 64:
        nbytes = prob.algorithmic_bytes if one_kernel else (
            wl.weight_bytes + wl.M * wl.K + 4 * wl.M * (wl.K // 32) + 4 * wl.M * wl.N)
        achieved = nbytes / (qdot_ms * 1e-3) / 1e9
        peak = float(peaks["hbm_gbs"])
        # the kernel the automatic path runs for this M (pq_api.cu: dp4a up to 8
        # rows, the TMA-fed warp-level MMA kernel for 9..16, tcgen05 above)
        kernel = ("qdot_q50_fused" if one_kernel else "qdot_q50") if prob.q50 else \
            ("qdot_fused" if one_kernel else "qdot_simt") if wl.M <= 8 else \
            "qdot_mmt" if wl.M <= 16 else "qdot_tc"
        traffic = recorded_traffic(kernel, wl.name)
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": kernel,
                "peak_source": f"{peak_src} hbm_gbs", "algorithmic_bytes": nbytes}
    achieved = wl.ops / (qdot_ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    # prompt shapes (Q8_0 and Q5_0 weights) run the kernel that applies the
    # scales in registers (qdot_tcw.cu)
    kernel = "qdot_tcw"
    traffic = recorded_traffic(kernel, wl.name)
    return {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": kernel,
            "peak_source": f"{peak_src} bf16_tflops (f16 operands: same dense rate)",
            "algorithmic_flops": wl.ops}


def run_workload(pq, name, steps, warmup, world, device, peaks, peak_src, sampler=None, e2e=False,
                 split: tuple[int, int] = (0, 1)):
    wl = workloads.WORKLOADS[name]
    prob = Problem(pq, wl, device, split=split)
    ms, quant_ms, qdot_ms, qdot_only_ms, window = time_graph(prob, steps, warmup, world, sampler)
    per_rank_s = ms * 1e-3
    if wl.M == 1 or wl.M <= 64:
        units, unit = wl.weight_bytes * steps, "GB/s"
        scale = 1e9
    else:
        units, unit = wl.ops * steps, "TOPS"
        scale = 1e12
    value, t_max = aggregate(units, per_rank_s, world, device)
    kernel_ms = {"qdot_graph_only": round(qdot_only_ms, 5)}
    if prob.fused:
        kernel_ms["quantize_qdot_fused"] = round(qdot_ms, 5)
    else:
        kernel_ms.update({"quantize": round(quant_ms, 5), "qdot": round(qdot_ms, 5)})
    # duration of the dominant kernel: a step that is one kernel (the fused decode
    # step) is timed exactly by the step time;
    # otherwise the mean launch of a graph
    # of that kernel alone (event-record nodes between kernels add their own
    # latency, so the in-graph event figure is an upper bound, reported beside it)
    one_kernel = prob.fused and fused_is_one_kernel(prob)
    dom_ms = (ms / steps) if one_kernel else qdot_only_ms
    if prob.world > 1:  # the step also holds the all-gather: the kernel's own event-bracketed time
        dom_ms = qdot_ms
    kernel_ms["dominant"] = round(dom_ms, 5)
    res = {"value": round(value / scale, 3), "unit": unit, "ms_per_step": round(t_max * 1e3 / steps, 5),
           "step": (("pq_quantize_q50_qdot" if prob.q50 else "pq_quantize_qdot_q8_0") +
                    (" (one kernel)" if one_kernel else " (two kernels)"))
           if prob.fused else ("pq_quantize_q8_0 + pq_q50_qdot" if prob.q50 else "pq_quantize_q8_0 + pq_qdot_q8_0"),
           "kernel_ms": kernel_ms,
           "roofline": roofline_for(prob, dom_ms, peaks, peak_src, one_kernel), "weight_copies": prob.copies,
           "window": window}
    if wl.M == 1 and not prob.q50 and split[1] == 1:
        # the floor launch chaining sets: the same weight traffic with no arithmetic
        res["stream_reader_ms"] = {"chained": round(time_reader(prob, steps, False), 5),
                                   "early": round(time_reader(prob, steps, True), 5)}
    if prob.fused and split[1] == 1:
        # the same step as two calls (quantizer, then qdot_t), for comparison
        two = Problem(pq, wl, device, fused=False)
        ms2, _, q2, _, _ = time_graph(two, steps, warmup, world)
        res["two_call"] = {"ms_per_step": round(ms2 / steps, 5), "qdot_ms": round(q2, 5),
                           "value": round(units / (ms2 * 1e-3) / scale, 3)}
        del two
    if e2e:
        dt, h2d, d2h = time_e2e(prob, steps, warmup)
        ev, _ = aggregate(units, dt, world, device)
        # x is copied in, C written in place into page-locked host memory over the
        # chip-to-chip link; the bytes still cross between host and device
        res["e2e"] = {"value": round(ev / scale, 3), "unit": unit, "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h}
        if not prob.q50 and prob.world == 1:
            set_host_path(pq, 1)
            try:
                dt2, _, _ = time_e2e(prob, steps, warmup)
            finally:
                set_host_path(pq, 0)
            res["e2e_copies"] = {"value": round(units / dt2 / scale, 3), "unit": unit}
    del prob
    import torch
    torch.cuda.empty_cache()
    return res


def int8_library_rate():
    """The GPU's practical dense int8 tensor rate: cuBLASLt's int8 GEMM (torch._int_mm) at 8192^3.

    A context figure for the prompt GEMM, which computes int8 x int8 block sums on the f16
    tensor path (the int8 MMA kind is not available on sm_103a); not part of any step."""
    import torch
    try:
        n = 8192
        a = torch.randint(-127, 128, (n, n), dtype=torch.int8, device="cuda")
        b = torch.randint(-127, 128, (n, n), dtype=torch.int8, device="cuda").t()
        for _ in range(2):
            torch._int_mm(a, b)
        torch.cuda.synchronize()
        ts = []
        for _ in range(3):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            torch._int_mm(a, b)
            e.record()
            torch.cuda.synchronize()
            ts.append(s.elapsed_time(e))
        del a, b
        torch.cuda.empty_cache()
        return round(2 * n ** 3 / (sorted(ts)[1] * 1e-3) / 1e12, 1)
    except Exception:  # torch without _int_mm, or no int8 GEMM for this device
        return None


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the Arm part code)."""
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    if "CPU part" in fields:
        return f"implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    return "unknown"


def _oracle_rate(wl, omp: bool, budget_s: float):
    """One bounded sample of the workload on the oracle: the activation rows quantized and
    contracted with the first n weight rows, n grown until one step takes about budget_s / 3;
    returns (units per second in the workload's unit, n, steps, seconds)."""
    import oracle
    x = workloads.activations(wl)
    per_col = 1.125 * wl.K if wl.M <= 64 else 2.0 * wl.M * wl.K  # weight bytes or ops per column
    scale = 1e9 if wl.M <= 64 else 1e12
    n = min(wl.N, 16)
    while True:
        if wl.w_format == "q5_0":
            w5, ws = workloads.q50_weights(wl, N=n)
        else:
            qw, sw = oracle.quantize_q8_0(workloads.weights(wl, N=n), omp=omp)
        t0 = time.perf_counter()
        qa, sa = oracle.quantize_q8_0(x, omp=omp)
        if wl.w_format == "q5_0":
            oracle.qdot_q5_0(qa, sa, w5, ws, omp=omp)
        else:
            oracle.qdot(qa, sa, qw, sw, omp=omp)
        dt = time.perf_counter() - t0
        if dt >= budget_s / 3 or n == wl.N:
            break
        n = min(wl.N, max(n + 1, int(n * min(16.0, budget_s / 3 / max(dt, 1e-6)))))
    steps, t0 = 0, time.perf_counter()
    while True:
        qa, sa = oracle.quantize_q8_0(x, omp=omp)
        if wl.w_format == "q5_0":
            oracle.qdot_q5_0(qa, sa, w5, ws, omp=omp)
        else:
            oracle.qdot(qa, sa, qw, sw, omp=omp)
        steps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s * 2 / 3:
            break
    unit_bytes = wl.weight_bytes / wl.N if wl.M <= 64 else per_col
    return unit_bytes * n * steps / dt / scale, n, steps, dt


def oracle_threads():
    """(True, threads) when the oracle's OpenMP build loads, else (False, 1)."""
    import oracle
    try:
        return True, oracle.threads(True)
    except Exception:  # no OpenMP runtime: the single-thread build is the baseline
        return False, 1


def cpu_baseline(name: str, budget_s: float = 4.0):
    """The oracle, as it stands, on a bounded sample of the workload (rank 0, host cores):
    the OpenMP build on every host core (the reported value) and the single-thread build
    beside it."""
    wl = workloads.WORKLOADS[name]
    omp, cores = oracle_threads()
    v_all, n_all, st_all, dt_all = _oracle_rate(wl, omp, budget_s)
    v_one, n_one, st_one, dt_one = _oracle_rate(wl, False, budget_s)
    unit = "GB/s" if wl.M <= 64 else "TOPS"
    return {"value": round(v_all, 5), "unit": unit, "cores": cores, "kind": "oracle",
            "cpu": cpu_model(), "single_thread": round(v_one, 5),
            "sample": f"{name}: x quantized + contracted with the first {n_all} of {wl.N} weight rows, "
                      f"{st_all} steps in {dt_all:.1f} s on every core; single thread {n_one} rows, "
                      f"{st_one} steps in {dt_one:.1f} s"}


def reference_arm(args):
    """--impl reference: the CPU oracle (OpenMP build, every host core) on the headline
    workload and metric, a bounded sample of weight rows per step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    omp, cores = oracle_threads()
    wl = workloads.WORKLOADS[args.workload]
    x = workloads.activations(wl)
    qw, sw = oracle.quantize_q8_0(workloads.weights(wl), omp=omp)
    # calibrate one full step; sample columns so that W + K steps stay near 60 s
    t0 = time.perf_counter()
    qa, sa = oracle.quantize_q8_0(x, omp=omp)
    oracle.qdot(qa, sa, qw, sw, omp=omp)
    full = time.perf_counter() - t0
    budget = 60.0
    frac = min(1.0, budget / max(1e-9, full * (args.steps + args.warmup)))
    ncols = max(1, int(wl.N * frac))
    qw_s, sw_s = qw[:ncols], sw[:ncols]
    for _ in range(args.warmup):
        qa, sa = oracle.quantize_q8_0(x, omp=omp)
        oracle.qdot(qa, sa, qw_s, sw_s, omp=omp)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        qa, sa = oracle.quantize_q8_0(x, omp=omp)
        oracle.qdot(qa, sa, qw_s, sw_s, omp=omp)
    dt = time.perf_counter() - t0
    if wl.M <= 64:
        units, unit, scale = ncols * wl.K + 4 * ncols * (wl.K // 32), "GB/s", 1e9
    else:
        units, unit, scale = 2 * wl.M * ncols * wl.K, "TOPS", 1e12
    value = units * args.steps / dt / scale
    sample = f"{ncols} of {wl.N} weight rows per step ({args.steps} steps, {cores} threads)"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64/f64",
            "data": "synthetic", "config": {"workload": wl.name, "M": wl.M, "K": wl.K, "N": wl.N},
            "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": cores, "kind": "oracle",
                             "cpu": cpu_model(), "sample": sample},
            "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


WORKLOAD_FIELDS = ["value", "unit", "ms_per_step", "roofline_frac", "cpu_baseline_value"]


def compact(res: dict, cpu: dict | None = None):
    """One workload's figures for the final line, in the order of WORKLOAD_FIELDS."""
    if "error" in res:
        return {"error": res["error"][:80]}
    return [res["value"], res["unit"], res["ms_per_step"], round(res["roofline"]["frac"], 4),
            float(f"{cpu['value']:.4g}") if cpu else None]


def final_line(head: dict, others: dict, cpus: dict, args, world: int, clocks: dict) -> dict:
    """The one JSON line: the contract's keys for the headline workload, then the prompt GEMM
    (the metric's second half) and a compact figure per workload as the last keys, so that
    the end of the line carries every workload."""
    wl = workloads.WORKLOADS[args.workload]
    launches_per_step = 1 if head["step"].endswith("(one kernel)") else 2
    line = {"metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic",
            "config": {"workload": args.workload, "M": wl.M, "K": wl.K, "N": wl.N,
                       "parallelism": head.get("parallelism", "single"),
                       "l2": f"{head['weight_copies']} rotating weight copies (>= 2x L2)",
                       "timing": "K steps in one CUDA graph, events on the launching stream"},
            "roofline": head["roofline"], "e2e": head["e2e"], "step": head["step"],
            "gpu_launches": launches_per_step * args.steps, "clocks": clocks}
    if args.workload in cpus:
        line["cpu_baseline"] = cpus[args.workload]
    variants = {}
    if "stream_reader_ms" in head:
        variants["reader_chained_ms"] = head["stream_reader_ms"]["chained"]
        variants["reader_early_ms"] = head["stream_reader_ms"]["early"]
    if "e2e_copies" in head:
        variants["e2e_with_copies"] = head["e2e_copies"]["value"]
    if variants:
        line["step_variants"] = variants
    prompt = head if args.workload == PROMPT else others.get(PROMPT)
    if prompt and "roofline" in prompt:
        rl = {k: prompt["roofline"][k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
        for k in ("int8_library_tops", "frac_of_int8_library"):
            if k in prompt["roofline"]:
                rl[k] = prompt["roofline"][k]
        line["prompt"] = {"workload": PROMPT, "value": prompt["value"], "unit": prompt["unit"],
                          "ms_per_step": prompt["ms_per_step"], "roofline": rl}
    allres = {args.workload: head, **others}
    line["workloads"] = {"fields": WORKLOAD_FIELDS,
                         **{n: compact(r, cpus.get(n)) for n, r in allres.items()}}
    return line


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=list(workloads.WORKLOADS))
    ap.add_argument("--no-others", action="store_true", help="time only the headline workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--parallel", choices=["colsplit", "replicas"], default="colsplit",
                    help="with N > 1 ranks: each rank holds an N-column shard of a layer N x wider "
                         "and C is all-gathered every step (colsplit), or each rank runs an "
                         "independent copy of the workload (replicas)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init(world, "nccl")
    import gemm_q8_qdot_gb300 as pq
    pq.load()
    peaks, peak_src = load_peaks()
    sampler = ClockSampler(local)
    split = (rank, world) if world > 1 and args.parallel == "colsplit" else (0, 1)
    head = run_workload(pq, args.workload, args.steps, args.warmup, world, device, peaks, peak_src,
                        sampler=sampler, e2e=True, split=split)
    head["parallelism"] = (f"colsplit{world}: each rank holds {workloads.WORKLOADS[args.workload].N} weight rows "
                           f"of a {world}x wider layer, C all-gathered over NCCL every step"
                           if split[1] > 1 else f"replicas{world}" if world > 1 else "single")
    clocks = sampler.summary(*head.pop("window"))
    others = {}
    if not args.no_others and split[1] == 1:
        for name in (PROMPT, "ffn_up_m1_k4096_n14336", "ffn_down_m1_k14336_n4096",
                     "smallm_m4_k4096_n11008", "smallm_m16_k4096_n11008", "smallm_m64_k4096_n11008",
                     "q50_decode_m1_k4096_n4096", "q50_prompt_m512_k4096_n14336"):
            if name == args.workload:
                continue
            try:
                r = run_workload(pq, name, args.steps, args.warmup, world, device, peaks, peak_src)
                r.pop("window")
                others[name] = r
            except pq.PQError as e:
                others[name] = {"error": str(e)}
    prompt_res = head if args.workload == PROMPT else others.get(PROMPT, {})
    if "roofline" in prompt_res:
        rate = int8_library_rate()
        if rate:
            rl = prompt_res["roofline"]
            rl["int8_library_tops"] = rate
            rl["frac_of_int8_library"] = round(rl["achieved"] / rate, 3)
    cpus = {}
    if rank == 0 and not args.no_cpu_baseline:
        for name in [args.workload] + [n for n in others if "error" not in others[n]]:
            cpus[name] = cpu_baseline(name, 6.0 if name == args.workload else 2.0)
    line = final_line(head, others, cpus, args, world, clocks)
    if rank == 0:
        # every figure of every workload, on stderr; stdout carries the one line
        print("bench detail: " + json.dumps({"headline": {args.workload: head}, "others": others,
                                             "cpu_baseline": cpus}), file=sys.stderr, flush=True)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
