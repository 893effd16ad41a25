"""Benchmark: Conv2d dgrad over the ResNet-50 v1.5 bottleneck convolutions
(all but conv1) at batch 256, NHWC bf16, fp32 accumulation, on one GB300.

One step = one dgrad of each of the 22 layers (one launch each), inputs
resident in HBM.  Prints one JSON line:
  value        aggregate useful TFLOP/s (sum of 2*N*P*Q*K*C*R*S over the 22
               layers / device time of the step), whole job over all ranks
  per_layer    each layer's TFLOP/s and its fraction of the slower-of
               (tensor, HBM) roofline, from a separate pass that launches
               each layer back to back over rotating buffer copies (working
               set >= 2x L2) with events around the run only; the time with
               one event pair around every launch is printed beside it
               (ms_event_pair, ~3 us of event overhead more); the tensor peak is the burst bf16
               figure when the SM clock held its maximum during the timed
               region, else the sustained one (roofline.peak_basis), and the
               fraction on the other basis is printed beside it
  roofline     for the launch with the largest share of the step, timed with
               events around it inside the timed region (the other launches
               of a timed step run back to back, each overlapping its
               predecessor's end through programmatic dependent launch)
  e2e          the same metric with dY uploaded from pinned host memory and
               dX read back every step, through the same C-ABI calls
  cpu_baseline the CPU oracle on a bounded sample (first images of each layer)
  other_configs  after the timed region: the tiny 8x8 layer, the three batch-8
               layers with warm and cold L2, the two x-gated batch-256 layers of
               the fused ReLU-backward config, and each layer's weight prepack

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--gate none|x|bits] [--autotune 1] [--layers L01,...] [--op dgrad|wgrad|fused|hbm]

--gate x|bits runs every layer with the fused ReLU-backward gate, reading the
saved activation or its 1-bit packed mask; algorithmic bytes, the roofline and
the end-to-end uploads then include that input.

--op wgrad times the weight gradient of the same 22 layers instead (per layer
one split-K GEMM launch and one ordered-reduction launch; dY and the forward
input resident), with per-layer tensor fractions; it prints its own JSON line
(metric "wgrad TFLOP/s ...").  --op hbm measures the DRAM bandwidth of a
write-only fill, a read-only sum and a copy (no dgrad), the ceilings the
write-heavy layers run against.

N > 1 (torchrun, one rank per GPU): every rank runs the full workload on its
own GPU (replicas; dgrad has no exchange step), barrier + max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from implicit_gemm_dgrad_gb300 import synth  # noqa: E402
from implicit_gemm_dgrad_gb300.workloads import RESNET50_B256  # noqa: E402

METRIC = "dgrad TFLOP/s per ResNet-50 layer (1 GB300) and % of slower-of roofline"
WORKLOAD = "resnet50_v1.5_bottleneck_dgrad_b256_bf16_22_layers"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return dict(FALLBACK_PEAKS, source="fallback")


DGRAD_SOURCES = ("cdg_api.cu", "cdg_params.h", "dgrad_sm103.cu", "dgrad_plain_sm103.cu", "dgrad_ext_sm103.cu",
                 "dgrad_act_sm103.cu", "dgrad_device.cuh", "dgrad_variant.cuh", "ptx.cuh", "wait.cuh")


def kernel_sources_sha256() -> str:
    """Hash of the files the dgrad kernel and its planner are built from."""
    import hashlib
    h = hashlib.sha256()
    for name in DGRAD_SOURCES:
        h.update(name.encode())
        with open(os.path.join(ROOT, "implicit_gemm_dgrad_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic(layer_name: str):
    """DRAM bytes (read + write) of one launch of `layer_name` from the
    committed ncu capture, or None when the capture has no such layer or was
    taken of other kernel sources."""
    path = os.path.join(ROOT, "profiles", "dgrad_kernel_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get("layers", {}).get(layer_name)
    if rec is None or d.get("sources_sha256") != kernel_sources_sha256():
        return None
    return int(rec["dram_read_bytes"]) + int(rec["dram_write_bytes"])


def tap_pixels(layer) -> int:
    """dX pixels that some (p, r) and (q, s) reach, h = p*stride - pad + r*dil
    and w = q*stride - pad + s*dil: reachable rows x reachable columns.
    Elsewhere dX is +0.0 whatever the gate holds, so an algorithm need read
    the gate input only here."""
    L = layer
    rows = {p * L.stride - L.pad + r * L.dil for p in range(L.P) for r in range(L.R)}
    cols = {q * L.stride - L.pad + s * L.dil for q in range(L.Q) for s in range(L.S)}
    return L.N * sum(0 <= h < L.H for h in rows) * sum(0 <= w < L.W for w in cols)


def toolchain() -> dict:
    """nvcc and driver versions (read-only queries; None where unavailable)."""
    out = {"nvcc": None, "driver": None, "torch": None}
    try:
        import torch
        out["torch"] = torch.__version__
    except Exception:  # noqa: BLE001 - a missing version must not fail the bench
        pass
    try:
        r = subprocess.run(["nvcc", "--version"], capture_output=True, text=True, timeout=20)
        line = [x for x in r.stdout.splitlines() if "release" in x]
        out["nvcc"] = line[-1].strip() if line else None
    except Exception:  # noqa: BLE001
        pass
    try:
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() == 0:
            buf = ctypes.create_string_buffer(96)
            if lib.nvmlSystemGetDriverVersion(buf, ctypes.c_uint(96)) == 0:
                out["driver"] = buf.value.decode()
            lib.nvmlShutdown()
    except Exception:  # noqa: BLE001
        pass
    return out


def gate_bytes(layer, gate: str) -> int:
    """Algorithmic HBM bytes of one launch: dY + W + dX, plus the gate input
    read once where dX can be non-zero (tap_pixels): the saved activation
    (2 B per element) or the packed mask (each pixel's C bits padded to
    16-byte units)."""
    el = layer.N * layer.H * layer.W * layer.C
    base = layer.bytes - (2 * el if layer.relu else 0)
    px = tap_pixels(layer)
    return base + {"none": 0, "x": 2 * px * layer.C, "bits": px * 16 * ((layer.C + 127) // 128)}[gate]


def wgrad_bytes(layer) -> int:
    """Algorithmic HBM bytes of one wgrad: dY read once, the forward input x
    read once where some filter tap reaches it (tap_pixels: a 1x1 stride-2
    layer uses one pixel in four), dW written once (2-byte elements)."""
    L = layer
    return 2 * (L.N * L.P * L.Q * L.K + tap_pixels(L) * L.C + L.K * L.R * L.S * L.C)


def tensor_peak(peaks, basis: str) -> float:
    """bf16 tensor peak in TFLOP/s: the burst figure (a GEMM timed alone, at
    full clock) or the sustained one (seconds under the power cap)."""
    return peaks["bf16_tflops"] if basis == "burst" else peaks["bf16_tflops_sustained"]


def peak_basis(clocks: dict) -> str:
    """Which tensor peak the timed region ran under: "burst" when the SM
    clock sampled during it held (median within 5 % of the maximum), else
    "sustained" (also when no clock could be read)."""
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    if sm and smax and sm >= 0.95 * smax:
        return "burst"
    return "sustained"


def roofline_time_s(layer, peaks, gate="none", basis="burst"):
    t_tc = layer.flops / (tensor_peak(peaks, basis) * 1e12)
    t_hbm = gate_bytes(layer, gate) / (peaks["hbm_gbs"] * 1e9)
    return max(t_tc, t_hbm), ("tensor" if t_tc >= t_hbm else "hbm")


def layer_record(L, ms, peaks, basis, gate="none"):
    """TFLOP/s, GB/s and the slower-of roofline fraction of one launch of
    layer L that took `ms`, on the chosen tensor-peak basis (and on both)."""
    t = ms * 1e-3
    t_roof, bound = roofline_time_s(L, peaks, gate, basis)
    other = "sustained" if basis == "burst" else "burst"
    return {"ms": round(float(ms), 5), "tflops": round(L.flops / t / 1e12, 2),
            "gbs": round(gate_bytes(L, gate) / t / 1e9, 1), "bound": bound, "roofline_frac": round(t_roof / t, 4),
            f"roofline_frac_{other}": round(roofline_time_s(L, peaks, gate, other)[0] / t, 4),
            "tensor_peak_frac": round(L.flops / t / 1e12 / tensor_peak(peaks, basis), 4)}


class _NvmlClocks:
    """SM clock, power and clock-event reasons read through NVML (ctypes,
    read-only queries), or None when the library is missing."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int):
        import ctypes
        self.c = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.dev = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.dev)) != 0:
            raise OSError("no NVML device")
        v = ctypes.c_uint()
        self.max_sm = float(v.value) if lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(v)) == 0 else None
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")

    def sample(self):
        c = self.c
        v, r, pw = c.c_uint(), c.c_ulonglong(), c.c_uint()
        sm = float(v.value) if self.lib.nvmlDeviceGetClockInfo(self.dev, 1, c.byref(v)) == 0 else None
        reasons = r.value if self.reasons_fn(self.dev, c.byref(r)) == 0 else 0
        power = pw.value / 1000.0 if self.lib.nvmlDeviceGetPowerUsage(self.dev, c.byref(pw)) == 0 else None
        return sm, reasons, power

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clocks, power and clock-event (throttle) reasons sampled during the
    timed region: every 2 ms on a thread through NVML (read-only
    queries), or, where NVML cannot be loaded, every 50 ms by nvidia-smi (the
    sampler then waits for its first sample before the region starts and
    reports the samples taken after it)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.nvml = None
        self.samples = []
        self.path = os.path.join("/tmp", f"cdg_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.nvml = _NvmlClocks(self.gpu)
        except Exception:  # noqa: BLE001 - fall back to nvidia-smi
            self.nvml = None
        if self.nvml is not None:
            import threading
            self.stop = threading.Event()

            def loop():
                while not self.stop.is_set():
                    self.samples.append(self.nvml.sample())
                    time.sleep(0.002)
            self.samples.append(self.nvml.sample())
            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
            return self
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.skip = 0
        if self.proc is not None:
            t0 = time.perf_counter()
            while time.perf_counter() - t0 < 5.0 and self.proc.poll() is None:
                with open(self.path) as f:
                    n = sum(1 for _ in f)
                if n >= 1:
                    self.skip = n
                    break
                time.sleep(0.01)
        return self

    def __exit__(self, *exc):
        if self.nvml is not None:
            self.stop.set()
            self.thread.join(timeout=5)
            self.samples.append(self.nvml.sample())
            return
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.nvml is not None:
            sm = [x[0] for x in self.samples if x[0] is not None]
            reasons = set()
            for _, bits, _ in self.samples:
                for bit, name in _NvmlClocks.REASONS.items():
                    if bits & bit:
                        reasons.add(name)
            power = [x[2] for x in self.samples if x[2] is not None]
            out = {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": self.nvml.max_sm,
                   "sm_min_mhz": min(sm) if sm else None, "reasons": sorted(reasons), "samples": len(self.samples),
                   "power_w_max": max(power) if power else None, "source": "nvml, 2 ms"}
            self.nvml.close()
            return out
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            lines = f.readlines()
        # samples from the timed region; if it was shorter than one period, the last one before it
        lines = lines[self.skip:] or lines[-1:]
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi, 50 ms"}


def cpu_oracle_sample(layers, arrays, images: int):
    """Time the CPU oracle on the first `images` images of every layer (gated
    by the saved activation where the arrays carry one)."""
    import oracle
    t0 = time.perf_counter()
    flops = 0
    for L, (dY, W, x) in zip(layers, arrays):
        oracle.dgrad(dY[:images], W, L.H, L.W, L.stride, L.pad, L.dil,
                     x=None if x is None else x[:images], dtype=L.dtype)
        flops += L.flops * images // L.N
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"first {images} image(s) of each of the {len(layers)} layers "
                      f"({flops / 1e9:.1f} GFLOP, {dt:.1f} s, double precision)",
            "seconds": dt}


def hold_stream(torch, stream, ms: float = 2.0) -> None:
    """Queue a ~ms busy-wait kernel on `stream` (no memory traffic), so that
    the host enqueues the launches and events that follow before the GPU
    reaches them: otherwise a launch shorter than the host's cost of issuing
    it would be timed together with the idle gap before it."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(ms * 2.0e6))


def time_launches(torch, stream, fn, reps: int, flush=None) -> list:
    """Device time (ms) of each of `reps` calls of fn, one CUDA event pair
    around each on `stream`.  With `flush` (a byte buffer larger than L2), the
    buffer is overwritten before every call, outside the events, so each call
    starts with a cold L2; without it, consecutive calls find their data in L2
    (a busy-wait kernel queued first keeps the host's issue cost out of the
    events)."""
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
    torch.cuda.synchronize()
    if flush is None:
        hold_stream(torch, stream)
    for k in range(reps):
        if flush is not None:
            with torch.cuda.stream(stream):
                flush.fill_(k & 0xFF)
        e0[k].record(stream)
        fn()
        e1[k].record(stream)
    torch.cuda.synchronize()
    return [e0[k].elapsed_time(e1[k]) for k in range(reps)]


def other_configs(torch, cdg, dev, stream, peaks, basis, host, state, reps=20):
    """The workloads besides the batch-256 step, each timed on its own
    (outside the timed region): the tiny 8x8 layer (launch-latency bound),
    the three batch-8 layers with warm and with cold L2 (a buffer of twice the
    L2 size written between calls), the two x-gated batch-256 layers of the
    fused ReLU-backward config, the back-to-back fused stage-1 pair against
    its two separate launches, the cost of the fused per-channel sums, GELU
    and SiLU backward on the F1 shape, and the weight prepack of every layer."""
    from implicit_gemm_dgrad_gb300.workloads import BATCH8, FUSED_RELU, TINY
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (128 << 20)
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    out = {"l2_flush_bytes": 2 * l2, "reps": reps}

    def setup(L):
        dY, W, x = synth.make_inputs(L.shape(), L.dtype, L.dist, L.workload, L.index, with_x=L.relu)
        p = cdg.plan(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype, relu=L.relu,
                     out_f32=(L.out == "f32"))
        d_dY = torch.from_numpy(dY.view(np.int16)).to(dev)
        d_W = torch.from_numpy(W.view(np.int16)).to(dev)
        d_x = torch.from_numpy(x.reshape(-1).view(np.int16)).to(dev) if L.relu else None
        d_Wp = torch.empty(p.packed_weight_bytes // 2, dtype=torch.int16, device=dev)
        d_dX = torch.empty(L.N * L.H * L.W * L.C * (2 if L.out == "f32" else 1), dtype=torch.int16, device=dev)
        p.prepack_weights(d_W, d_Wp, stream)
        return p, (lambda: p.dgrad(d_dY, d_Wp, d_dX, d_x, stream))

    def record(L, ms_list, gate="none"):
        ms = float(np.median(ms_list))
        rec = {"layer": L.name, "dtype": L.dtype, "out": L.out}
        rec.update(layer_record(L, ms, peaks, basis, gate))
        rec["ms_min"] = round(float(np.min(ms_list)), 5)
        return rec

    # tiny: 8x8x16, 3x3, fp16 in, fp32 out
    p, run = setup(TINY)
    for _ in range(5):
        run()
    ms = time_launches(torch, stream, run, reps)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(200):
        run()
    t1 = time.perf_counter()
    torch.cuda.synchronize()
    rec = record(TINY, ms)
    rec["host_us_per_call"] = round((t1 - t0) / 200 * 1e6, 2)
    rec["note"] = "launch-latency bound: the whole problem is 11 KB and 0.3 MFLOP"
    if p.device_status(stream) != 0:
        raise RuntimeError("device status after the tiny config")
    out["tiny"] = rec

    out["batch8"] = []
    for L in BATCH8:
        p, run = setup(L)
        for _ in range(5):
            run()
        warm = time_launches(torch, stream, run, reps)
        cold = time_launches(torch, stream, run, reps, flush)
        if p.device_status(stream) != 0:
            raise RuntimeError(f"device status after {L.name}")
        rec = {"layer": L.name, "cold_l2": record(L, cold), "warm_l2": record(L, warm)}
        out["batch8"].append(rec)

    out["fused_relu_x"] = []
    for L in FUSED_RELU:
        p, run = setup(L)
        for _ in range(5):
            run()
        ms = time_launches(torch, stream, run, reps, flush)
        if p.device_status(stream) != 0:
            raise RuntimeError(f"device status after {L.name}")
        rec = record(L, ms, "x")
        rec["gate"] = "saved bf16 activation x, read once where dX can be non-zero; cold L2"
        out["fused_relu_x"].append(rec)

    # back-to-back fusion: ResNet-50 stage 1's 3x3 64->64 dgrad at 56x56, gated
    # by ReLU, feeding the 1x1 64->256 dgrad, one fused launch (g stays on
    # chip) against the same two layers as two launches (g through HBM)
    from implicit_gemm_dgrad_gb300.workloads import by_name
    L4, L3 = by_name("L04_3x3_64_56"), by_name("L03_1x1_256-64_56")
    dY2, W2, x2 = synth.make_inputs(L4.shape(), L4.dtype, L4.dist, L4.workload, L4.index, with_x=True)
    _, W1, _ = synth.make_inputs(L3.shape(), L3.dtype, L3.dist, L3.workload, L3.index)
    up = lambda a: torch.from_numpy(a.reshape(-1).view(np.int16)).to(dev)  # noqa: E731
    d_dY2, d_W2, d_x2, d_W1 = up(dY2), up(W2), up(x2), up(W1)
    f = cdg.FusedPlan(L4.N, L4.H, L4.W, L3.C, L4.C, L4.K, 3, 3, 1, 1, "bf16", act="relu")
    b2, b1 = f.packed_weight_bytes
    d_W2p = torch.empty(b2 // 2, dtype=torch.int16, device=dev)
    d_W1p = torch.empty(b1 // 2, dtype=torch.int16, device=dev)
    f.prepack_weights(d_W2, d_W1, d_W2p, d_W1p, stream)
    d_dX1 = torch.empty(L3.N * L3.H * L3.W * L3.C, dtype=torch.int16, device=dev)
    d_g = torch.empty(L4.N * L4.H * L4.W * L4.C, dtype=torch.int16, device=dev)
    p4 = cdg.plan(L4.N, L4.H, L4.W, L4.C, L4.K, 3, 3, 1, 1, 1, "bf16", relu=True)
    p3 = cdg.plan(L3.N, L3.H, L3.W, L3.C, L3.K, 1, 1, 1, 0, 1, "bf16")
    d_W3p = torch.empty(p3.packed_weight_bytes // 2, dtype=torch.int16, device=dev)
    p3.prepack_weights(d_W1, d_W3p, stream)
    fused = lambda: f.dgrad(d_dY2, d_W2p, d_x2, d_W1p, d_dX1, None, stream)  # noqa: E731

    def unfused():
        p4.dgrad(d_dY2, d_W2p, d_g, d_x2, stream)
        p3.dgrad(d_g, d_W3p, d_dX1, None, stream)
    for _ in range(3):
        fused()
        unfused()
    ms_f = float(np.median(time_launches(torch, stream, fused, reps, flush)))
    ms_u = float(np.median(time_launches(torch, stream, unfused, reps, flush)))
    if f.device_status(stream) != 0 or p4.device_status(stream) != 0 or p3.device_status(stream) != 0:
        raise RuntimeError("device status after the fused pair")
    flops = L4.flops + L3.flops
    fbytes = 2 * (dY2.size + x2.size + W2.size + W1.size) + 2 * d_dX1.numel()
    t_roof = max(flops / (tensor_peak(peaks, basis) * 1e12), fbytes / (peaks["hbm_gbs"] * 1e9))
    out["fused_bottleneck_stage1"] = {
        "what": "dX1 = dgrad_1x1(relu_bwd(dgrad_3x3(dY2, W2), x2), W1): L04 shape gated by ReLU, then L03 shape; "
                "batch 256, bf16, cold L2",
        "fused_ms": round(ms_f, 5), "two_launch_ms": round(ms_u, 5), "speedup": round(ms_u / ms_f, 3),
        "tflops": round(flops / (ms_f * 1e-3) / 1e12, 2), "gbs": round(fbytes / (ms_f * 1e-3) / 1e9, 1),
        "algorithmic_bytes": fbytes, "bound": "hbm" if fbytes / (peaks["hbm_gbs"] * 1e9) > flops /
        (tensor_peak(peaks, basis) * 1e12) else "tensor", "roofline_frac": round(t_roof / (ms_f * 1e-3), 4),
        "plan": {k: f.info()[k] for k in ("box_w", "box_h", "stages", "work_items", "grid", "smem_bytes")}}
    del d_dY2, d_x2, d_g, d_dX1

    # per-channel output sums fused into the epilogue: cost against the same layer without them
    sums = []
    for L, nsum in ((by_name("L03_1x1_256-64_56"), 1), (FUSED_RELU[0], 2)):
        dY, W, x = synth.make_inputs(L.shape(), L.dtype, L.dist, L.workload, L.index, with_x=L.relu)
        d_dY, d_W, d_x = up(dY), up(W), (up(x) if L.relu else None)
        pl = cdg.plan(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype, relu=L.relu)
        ps = cdg.plan(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype, relu=L.relu, sums=nsum)
        d_Wp = torch.empty(pl.packed_weight_bytes // 2, dtype=torch.int16, device=dev)
        pl.prepack_weights(d_W, d_Wp, stream)
        d_dX = torch.empty(L.N * L.H * L.W * L.C, dtype=torch.int16, device=dev)
        d_s = torch.empty(nsum * L.C, dtype=torch.float32, device=dev)
        d_ws = torch.empty(ps.sums_workspace_bytes // 4, dtype=torch.float32, device=dev)
        plain = lambda: pl.dgrad(d_dY, d_Wp, d_dX, d_x, stream)  # noqa: E731
        with_sums = lambda: ps.dgrad_sums(d_dY, d_Wp, d_dX, d_s, d_ws, d_x, stream)  # noqa: E731
        for _ in range(3):
            plain()
            with_sums()
        m0 = float(np.median(time_launches(torch, stream, plain, reps, flush)))
        m1 = float(np.median(time_launches(torch, stream, with_sums, reps, flush)))
        if ps.device_status(stream) != 0:
            raise RuntimeError(f"device status after the sums of {L.name}")
        sums.append({"layer": L.name, "sums": ["sum dX"] + (["sum dX*x"] if nsum == 2 else []),
                     "plain_ms": round(m0, 5), "with_sums_ms": round(m1, 5), "overhead": round(m1 / m0 - 1, 4)})
    out["channel_sums"] = sums

    # activation backward other than ReLU, on the F1 shape (x = the activation's saved input)
    L = FUSED_RELU[0]
    dY, W, _ = synth.make_inputs(L.shape(), L.dtype, L.dist, L.workload, L.index)
    z = synth.to_bits((2.0 * np.random.default_rng(77).standard_normal((L.N, L.H, L.W, L.C))).astype(np.float32),
                      L.dtype)
    d_dY, d_W, d_z = up(dY), up(W), up(z)
    d_dX = torch.empty(L.N * L.H * L.W * L.C, dtype=torch.int16, device=dev)
    acts = []
    for act in ("relu", "gelu", "silu"):
        pa = cdg.plan(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype, relu=True, act=act)
        d_Wp = torch.empty(pa.packed_weight_bytes // 2, dtype=torch.int16, device=dev)
        pa.prepack_weights(d_W, d_Wp, stream)
        run = lambda: pa.dgrad(d_dY, d_Wp, d_dX, d_z, stream)  # noqa: E731
        for _ in range(3):
            run()
        ms = float(np.median(time_launches(torch, stream, run, reps, flush)))
        if pa.device_status(stream) != 0:
            raise RuntimeError(f"device status after {act}")
        rec = {"act": act}
        rec.update(layer_record(L, ms, peaks, basis, "x"))
        acts.append(rec)
    out["activation_bwd_F1"] = acts

    # weight prepack (KRSC -> packed B operand), once per weight update; not part of the metric
    prep = {}
    for (L, p, _d_dY, d_Wp, _d_dX), (_dY, W, _x) in zip(state, host):
        d_W = torch.from_numpy(W.view(np.int16)).to(dev)
        ms = time_launches(torch, stream, lambda: p.prepack_weights(d_W, d_Wp, stream), 5, flush)
        prep[L.name] = round(float(np.median(ms)), 5)
    out["prepack_ms"] = prep
    del flush
    return out


def max_over_ranks(x: float, world: int) -> float:
    """The largest of every rank's x (the slowest replica's time), reduced over
    the gloo control group; x itself when there is one rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def select_layers(names: str):
    layers = RESNET50_B256
    if names:
        keep = set(names.split(","))
        layers = [L for L in layers if L.name in keep]
    return layers


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, as it stands, on a bounded sample.
    Under torchrun only rank 0 runs it; the other ranks return at once."""
    if rank != 0:
        return
    layers = select_layers(args.layers)
    n = args.ref_images
    arrays = [synth.make_inputs(L.shape(), L.dtype, L.dist, L.workload, L.index, batch=n) for L in layers]
    for _ in range(args.warmup):
        cpu_oracle_sample(layers[:1], arrays[:1], 1)
    times, res = [], None
    for _ in range(args.steps):
        res = cpu_oracle_sample(layers, arrays, n)
        times.append(res["seconds"])
    value = res["value"]
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(times)),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "images_per_layer_per_step": n, "layers": len(layers)},
            "cpu_baseline": {k: res[k] for k in ("value", "unit", "cores", "kind", "sample")},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_wgrad(args, rank, world, local_rank):
    """The weight gradient of the same 22 layers: per layer one split-K GEMM
    launch and one ordered-reduction launch; inputs resident; per-layer event
    times from a separate pass, then K timed steps."""
    import torch
    import implicit_gemm_dgrad_gb300 as cdg
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.Stream(device=dev)
    peaks = load_peaks()
    layers = select_layers(args.layers)
    state = []
    with torch.cuda.stream(stream):
        for L in layers:
            dY, W, x = synth.make_inputs(L.shape(), L.dtype, L.dist, L.workload, L.index, with_x=True)
            p = cdg.wgrad_plan(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype)
            d_dY = torch.from_numpy(dY.view(np.int16)).to(dev)
            d_x = torch.from_numpy(x.reshape(-1).view(np.int16)).to(dev)
            d_dW = torch.empty(L.K * L.R * L.S * L.C, dtype=torch.int16, device=dev)
            ws = torch.empty(p.workspace_bytes // 4, dtype=torch.float32, device=dev)
            state.append((L, p, d_dY, d_x, d_dW, ws))
    torch.cuda.synchronize()

    def step():
        for (_, p, d_dY, d_x, d_dW, ws) in state:
            p.wgrad(d_dY, d_x, d_dW, ws, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for (L, p, *_r) in state:
        if p.device_status(stream) != 0:
            raise RuntimeError(f"wgrad device status after warm-up ({L.name})")
    nL = len(state)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nL + 1)] for _ in range(args.steps)]
    hold_stream(torch, stream)
    for k in range(args.steps):
        evs[k][0].record(stream)
        for i, (_, p, d_dY, d_x, d_dW, ws) in enumerate(state):
            p.wgrad(d_dY, d_x, d_dW, ws, stream)
            evs[k][i + 1].record(stream)
    torch.cuda.synchronize()
    per_ms = np.mean([[evs[k][i].elapsed_time(evs[k][i + 1]) for i in range(nL)] for k in range(args.steps)], axis=0)
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        hold_stream(torch, stream)
        for k in range(args.steps):
            e0[k].record(stream)
            step()
            e1[k].record(stream)
        torch.cuda.synchronize()
    total_ms = max_over_ranks(float(sum(e0[k].elapsed_time(e1[k]) for k in range(args.steps))), world)
    ms_per_step = total_ms / args.steps
    flops_step = sum(L.flops for (L, *_r) in state)
    clk = clocks.summary()
    basis = peak_basis(clk)

    def roof(L, b=basis):
        t_tc = L.flops / (tensor_peak(peaks, b) * 1e12)
        t_hbm = wgrad_bytes(L) / (peaks["hbm_gbs"] * 1e9)
        return max(t_tc, t_hbm), ("tensor" if t_tc >= t_hbm else "hbm")

    per_layer = []
    for i, (L, p, *_r) in enumerate(state):
        t = per_ms[i] * 1e-3
        inf = p.info()
        t_roof, bound = roof(L)
        per_layer.append({"layer": L.name, "ms": round(float(per_ms[i]), 5), "tflops": round(L.flops / t / 1e12, 2),
                          "gbs": round(wgrad_bytes(L) / t / 1e9, 1), "bound": bound,
                          "roofline_frac": round(t_roof / t, 4),
                          "roofline_frac_sustained" if basis == "burst" else "roofline_frac_burst":
                              round(roof(L, "sustained" if basis == "burst" else "burst")[0] / t, 4),
                          "tensor_peak_frac": round(L.flops / t / 1e12 / tensor_peak(peaks, basis), 4),
                          "plan": {"splits": inf["splits"], "tile_n": inf["tile_n"], "pos_box": inf["pos_box"],
                                   "stages": inf["stages"], "work_items": inf["work_items"]}})
    if rank != 0:
        return
    dom = int(np.argmax(per_ms))
    Ld = state[dom][0]
    td = per_ms[dom] * 1e-3
    _, dbound = roof(Ld)
    if dbound == "tensor":
        achieved, dpeak, dunit = Ld.flops / td / 1e12, tensor_peak(peaks, basis), "TFLOP/s"
    else:
        achieved, dpeak, dunit = wgrad_bytes(Ld) / td / 1e9, peaks["hbm_gbs"], "GB/s"
    line = {"metric": "wgrad TFLOP/s per ResNet-50 layer (1 GB300)", "op": "wgrad",
            "value": round(world * flops_step * args.steps / (total_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD.replace("dgrad", "wgrad"), "global_batch": 256 * world, "layers": nL,
                       "flops_per_step": flops_step, "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2"},
            "roofline": {"bound": dbound, "achieved": round(achieved, 2), "peak": dpeak, "unit": dunit,
                         "frac": round(achieved / dpeak, 4), "traffic": None,
                         "algorithmic_bytes": wgrad_bytes(Ld), "kernel": f"wgrad_kernel + reduce ({Ld.name})",
                         "launch_ms": round(float(per_ms[dom]), 5),
                         "peak_source": peaks["source"] + (f" {basis} bf16" if dbound == "tensor" else " copy bandwidth"),
                         "peak_basis": basis,
                         "step_roofline_frac": round(sum(roof(L)[0] for (L, *_r) in state) / (ms_per_step * 1e-3), 4)},
            "gpu_launches": 2 * nL * args.steps, "clocks": clk, "per_layer": per_layer,
            "per_layer_timing": "separate pass, one CUDA event pair around each layer's two launches"}
    print(json.dumps(line), flush=True)


def run_fused(args, rank, world, local_rank):
    """The back-to-back fused dgrad of ResNet-50 stage 1 alone (the 3x3 64->64
    layer at 56x56 gated by ReLU, feeding the 1x1 64->256 layer, g kept on
    chip): K timed launches, inputs resident (larger than L2)."""
    import torch
    import implicit_gemm_dgrad_gb300 as cdg
    from implicit_gemm_dgrad_gb300.workloads import by_name
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.Stream(device=dev)
    peaks = load_peaks()
    L4, L3 = by_name("L04_3x3_64_56"), by_name("L03_1x1_256-64_56")
    dY2, W2, x2 = synth.make_inputs(L4.shape(), L4.dtype, L4.dist, L4.workload, L4.index, with_x=True)
    _, W1, _ = synth.make_inputs(L3.shape(), L3.dtype, L3.dist, L3.workload, L3.index)
    up = lambda a: torch.from_numpy(a.reshape(-1).view(np.int16)).to(dev)  # noqa: E731
    with torch.cuda.stream(stream):
        d_dY2, d_W2, d_x2, d_W1 = up(dY2), up(W2), up(x2), up(W1)
        f = cdg.FusedPlan(L4.N, L4.H, L4.W, L3.C, L4.C, L4.K, 3, 3, 1, 1, "bf16", act="relu")
        b2, b1 = f.packed_weight_bytes
        d_W2p = torch.empty(b2 // 2, dtype=torch.int16, device=dev)
        d_W1p = torch.empty(b1 // 2, dtype=torch.int16, device=dev)
        f.prepack_weights(d_W2, d_W1, d_W2p, d_W1p, stream)
        d_dX1 = torch.empty(L3.N * L3.H * L3.W * L3.C, dtype=torch.int16, device=dev)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        f.dgrad(d_dY2, d_W2p, d_x2, d_W1p, d_dX1, None, stream)
    torch.cuda.synchronize()
    if f.device_status(stream) != 0:
        raise RuntimeError("fused device status after warm-up")
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clocks:
        hold_stream(torch, stream)
        for k in range(args.steps):
            e0[k].record(stream)
            f.dgrad(d_dY2, d_W2p, d_x2, d_W1p, d_dX1, None, stream)
            e1[k].record(stream)
        torch.cuda.synchronize()
    total_ms = max_over_ranks(float(sum(e0[k].elapsed_time(e1[k]) for k in range(args.steps))), world)
    if rank != 0:
        return
    clk = clocks.summary()
    basis = peak_basis(clk)
    ms = total_ms / args.steps
    flops = L4.flops + L3.flops
    fbytes = 2 * (dY2.size + x2.size + W2.size + W1.size) + 2 * d_dX1.numel()
    t_tc, t_hbm = flops / (tensor_peak(peaks, basis) * 1e12), fbytes / (peaks["hbm_gbs"] * 1e9)
    bound = "tensor" if t_tc >= t_hbm else "hbm"
    achieved = fbytes / (ms * 1e-3) / 1e9 if bound == "hbm" else flops / (ms * 1e-3) / 1e12
    peak = peaks["hbm_gbs"] if bound == "hbm" else tensor_peak(peaks, basis)
    line = {"metric": "fused back-to-back dgrad TFLOP/s (ResNet-50 stage 1: 3x3 64->64 + ReLU bwd + 1x1 64->256)",
            "op": "fused", "value": round(world * flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "resnet50_stage1_fused_3x3_relu_1x1_b256_bf16", "global_batch": 256 * world,
                       "l2": "inputs larger than L2", "parallelism": f"replicas x{world}"},
            "roofline": {"bound": bound, "achieved": round(achieved, 2), "peak": peak,
                         "unit": "GB/s" if bound == "hbm" else "TFLOP/s", "frac": round(achieved / peak, 4),
                         "traffic": None, "algorithmic_bytes": fbytes, "kernel": "fused_kernel",
                         "peak_basis": basis},
            "gpu_launches": args.steps, "clocks": clk, "plan": f.info()}
    print(json.dumps(line), flush=True)


def run_hbm(args, rank, world, local_rank):
    """DRAM bandwidth that the dgrad layers' byte mix can draw on: a
    write-only fill, a read-only reduction and a 1:1 copy of 4 GiB buffers
    (PyTorch's own kernels, no dgrad), each timed with CUDA events over
    --steps launches after --warmup.  Layers whose bytes are mostly dX writes
    are bounded by the fill's rate, not by the copy's."""
    import torch
    dev = torch.device("cuda", local_rank)
    n = 4 << 30
    a = torch.empty(n, dtype=torch.uint8, device=dev)
    b = torch.empty(n, dtype=torch.uint8, device=dev)
    a.fill_(1)
    out = torch.empty((), dtype=torch.int64, device=dev)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    av = a.view(torch.int64)
    fill_ms = timed(lambda: b.fill_(7))
    read_ms = timed(lambda: torch.sum(av, 0, dtype=torch.int64, out=out))
    copy_ms = timed(lambda: b.copy_(a))
    peaks = load_peaks()
    rec = {"metric": "DRAM bandwidth: write-only fill, read-only sum, 1:1 copy (4 GiB each)", "unit": "GB/s",
           "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "data": "synthetic",
           "write_only_gbs": round(n / fill_ms / 1e6, 1), "read_only_gbs": round(n / read_ms / 1e6, 1),
           "copy_gbs": round(2 * n / copy_ms / 1e6, 1), "measured_copy_peak_gbs": peaks["hbm_gbs"]}
    if rank == 0:
        print(json.dumps(rec), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-images", type=int, default=256,
                    help="images per layer in the CPU-oracle baseline (256 = the whole batch, ~13 s on 16 cores)")
    ap.add_argument("--ref-images", type=int, default=8, help="images per layer per reference-arm step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the tiny, batch-8, x-gated and prepack measurements after the timed region")
    ap.add_argument("--layers", default="", help="comma-separated layer names (default: all 22)")
    ap.add_argument("--autotune", type=int, default=0,
                    help="1: tune every layer's plan with cdg_autotune during set-up (untimed)")
    ap.add_argument("--op", default="dgrad", choices=["dgrad", "wgrad", "fused", "hbm"],
                    help="wgrad: time the weight gradient (split-K GEMM + ordered reduction) of the same layers; "
                         "fused: time the back-to-back fused dgrad of ResNet-50 stage 1 alone; "
                         "hbm: DRAM bandwidth of a write-only fill, a read-only sum and a copy (no dgrad)")
    ap.add_argument("--gate", default="none", choices=["none", "x", "bits"],
                    help="fused ReLU-backward gate on every layer: none; x = the saved bf16 activation; "
                         "bits = its 1-bit packed mask (packed once at set-up, as a forward pass would store it)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import torch.distributed as dist

    import implicit_gemm_dgrad_gb300 as cdg

    if world > 1:
        dist.init_process_group("gloo")  # control path only: barrier and max-over-ranks
    torch.cuda.set_device(local_rank)
    if args.op == "wgrad":
        run_wgrad(args, rank, world, local_rank)
        return
    if args.op == "fused":
        run_fused(args, rank, world, local_rank)
        return
    if args.op == "hbm":
        run_hbm(args, rank, world, local_rank)
        return
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.Stream(device=dev)
    peaks = load_peaks()

    layers = select_layers(args.layers)

    # ---- inputs (seeded, host), upload, plan, prepack
    gate = args.gate
    host, state, gates, h_gate = [], [], [], []
    with torch.cuda.stream(stream):
        for L in layers:
            dY, W, x = synth.make_inputs(L.shape(), L.dtype, L.dist, L.workload, L.index, with_x=(gate != "none"))
            host.append((dY, W, x))
            p = cdg.plan(L.N, L.H, L.W, L.C, L.K, L.R, L.S, L.stride, L.pad, L.dil, L.dtype,
                         relu=(gate == "x"), relu_bits=(gate == "bits"))
            d_dY = torch.from_numpy(dY.view(np.int16)).to(dev)
            d_W = torch.from_numpy(W.view(np.int16)).to(dev)
            d_Wp = torch.empty(p.packed_weight_bytes // 2, dtype=torch.int16, device=dev)
            d_dX = torch.empty(L.N * L.H * L.W * L.C, dtype=torch.int16, device=dev)
            p.prepack_weights(d_W, d_Wp, stream)
            state.append((L, p, d_dY, d_Wp, d_dX))
            if gate == "none":
                gates.append(None)
                continue
            d_x = torch.from_numpy(x.reshape(-1).view(np.int16)).to(dev)
            if gate == "x":
                gates.append(d_x)
            else:
                pixels = L.N * L.H * L.W
                d_bits = torch.empty(cdg.relu_mask_bytes(pixels, L.C), dtype=torch.uint8, device=dev)
                cdg.pack_relu_mask(d_x, d_bits, pixels, L.C, L.dtype, stream)
                gates.append(d_bits)
                del d_x
            h_gate.append(gates[-1].cpu().pin_memory())  # the gate input the end-to-end leg uploads
    torch.cuda.synchronize()
    tuned_ms = {}
    if args.autotune:
        # plan-time tuning (cuDNN-Find style), before and outside every timed region
        for (L, p, d_dY, d_Wp, d_dX) in state:
            tuned_ms[L.name] = p.autotune(d_dY, d_Wp, d_dX, gates[len(tuned_ms)], stream, reps=5)
        torch.cuda.synchronize()

    def step():
        for i, (_, p, d_dY, d_Wp, d_dX) in enumerate(state):
            p.dgrad(d_dY, d_Wp, d_dX, gates[i], stream)

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- warm-up, then the timed region with per-launch events
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for (_, p, *_rest) in state:
        st = p.device_status(stream)
        if st != 0:
            raise RuntimeError(f"device status {st} after warm-up")

    nL = len(state)

    def per_launch_pass(steps):
        """Mean device time of every launch, one event pair around each (the
        events sit between the kernels, so this pass forgoes the overlap of
        consecutive launches that the timed steps get)."""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nL + 1)] for _ in range(steps)]
        torch.cuda.synchronize()
        hold_stream(torch, stream)
        for k in range(steps):
            evs[k][0].record(stream)
            for i, (_, p, d_dY, d_Wp, d_dX) in enumerate(state):
                p.dgrad(d_dY, d_Wp, d_dX, gates[i], stream)
                evs[k][i + 1].record(stream)
        torch.cuda.synchronize()
        ms = np.zeros(nL)
        for k in range(steps):
            for i in range(nL):
                ms[i] += evs[k][i].elapsed_time(evs[k][i + 1])
        return ms / steps

    l2_bytes = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (128 << 20)

    def back_to_back_pass(min_launches):
        """Mean device time of each layer's launch in a stream of launches:
        the layer launched back to back (each launch may overlap the previous
        one's tail, as consecutive layers do in the step) with events only
        around the run, so that the ~3 us an event pair adds to a launch is
        left out.  The launches rotate over copies of dY, dX, the gate input
        and the packed weights, enough that the run's working set is at least
        twice the L2 size: no launch finds its operands in L2."""
        ms = np.zeros(nL)
        for i, (L, p, d_dY, d_Wp, d_dX) in enumerate(state):
            g = gates[i]
            nbytes = (d_dY.numel() + d_dX.numel() + d_Wp.numel()) * 2 + (0 if g is None else g.numel() * g.element_size())
            copies = int(min(8, max(1, -(-2 * l2_bytes // nbytes))))
            bufs = [(d_dY, d_Wp, d_dX, g)]
            for _ in range(copies - 1):
                bufs.append((d_dY.clone(), d_Wp.clone(), torch.empty_like(d_dX), None if g is None else g.clone()))
            reps = copies * max(1, -(-min_launches // copies))
            for (a, w, b, gg) in bufs:
                p.dgrad(a, w, b, gg, stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            hold_stream(torch, stream)
            e0.record(stream)
            for r in range(reps):
                a, w, b, gg = bufs[r % copies]
                p.dgrad(a, w, b, gg, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            ms[i] = e0.elapsed_time(e1) / reps
            del bufs
        torch.cuda.empty_cache()
        return ms

    # per-layer breakdown (passes of their own, before the timed region) and
    # the launch with the largest share of the step
    per_layer_ms_events = per_launch_pass(args.steps)
    per_layer_ms = back_to_back_pass(max(10, args.steps))
    dom = int(np.argmax(per_layer_ms))

    # ---- the timed region: K steps; events at the step boundaries and around
    # the dominant launch only, so that consecutive launches overlap as in use
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    dv0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    dv1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        t_host0 = time.perf_counter()
        hold_stream(torch, stream)  # before the first event: the timed region starts at ev0[0]
        for k in range(args.steps):
            ev0[k].record(stream)
            for i, (_, p, d_dY, d_Wp, d_dX) in enumerate(state):
                if i == dom:
                    dv0[k].record(stream)
                p.dgrad(d_dY, d_Wp, d_dX, gates[i], stream)
                if i == dom:
                    dv1[k].record(stream)
            ev1[k].record(stream)
        torch.cuda.synchronize()
        t_host1 = time.perf_counter()
    barrier()
    step_ms = [ev0[k].elapsed_time(ev1[k]) for k in range(args.steps)]
    dom_ms = float(np.mean([dv0[k].elapsed_time(dv1[k]) for k in range(args.steps)]))
    total_ms = max_over_ranks(float(np.sum(step_ms)), world)
    ms_per_step = total_ms / args.steps
    flops_step = sum(L.flops for (L, *_r) in state)
    value = world * flops_step * args.steps / (total_ms * 1e-3) / 1e12

    clk = clocks.summary()
    basis = peak_basis(clk)
    per_layer = []
    for i, (L, p, *_r) in enumerate(state):
        inf = p.info()
        rec = {"layer": L.name}
        rec.update(layer_record(L, per_layer_ms[i], peaks, basis, gate))
        rec["ms_event_pair"] = round(float(per_layer_ms_events[i]), 5)
        rec["roofline_frac_event_pair"] = layer_record(L, per_layer_ms_events[i], peaks, basis, gate)["roofline_frac"]
        rec["plan"] = {"a_mode": inf["a_mode"], "cta_pair": inf["cta_pair"], "mma_warps": inf["mma_warps"],
                       "tile_n": inf["tile_n"], "stages": inf["stages"], "tuned": inf["tuned"]}
        per_layer.append(rec)

    # dominant launch: the layer with the largest share of the step, timed inside the timed region
    Ld = state[dom][0]
    td = dom_ms * 1e-3
    _, bound = roofline_time_s(Ld, peaks, gate, basis)
    if bound == "tensor":
        achieved, peak, unit = Ld.flops / td / 1e12, tensor_peak(peaks, basis), "TFLOP/s"
    else:
        achieved, peak, unit = gate_bytes(Ld, gate) / td / 1e9, peaks["hbm_gbs"], "GB/s"
    step_roof = {b: sum(roofline_time_s(L, peaks, gate, b)[0] for (L, *_r) in state) / (ms_per_step * 1e-3)
                 for b in ("burst", "sustained")}
    roofline = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4),
                "traffic": profiled_traffic(Ld.name) if gate == "none" else None,
                "algorithmic_bytes": gate_bytes(Ld, gate), "kernel": f"dgrad_kernel ({Ld.name})",
                "peak_source": peaks["source"] + (f" {basis} bf16" if bound == "tensor" else " copy bandwidth"),
                "peak_basis": basis,
                "launch_ms": round(dom_ms, 5),
                "share_of_step": round(dom_ms / ms_per_step, 4),
                "step_roofline_frac": round(step_roof[basis], 4),
                "step_roofline_frac_burst": round(step_roof["burst"], 4),
                "step_roofline_frac_sustained": round(step_roof["sustained"], 4)}

    # ---- end to end: dY from pinned host memory, dX back to pinned host memory, every step
    h_dY = [torch.from_numpy(h[0].view(np.int16)).pin_memory() for h in host]
    h_dX = [torch.empty(L.N * L.H * L.W * L.C, dtype=torch.int16).pin_memory() for (L, *_r) in state]
    h2d = sum(t.numel() * 2 for t in h_dY) + sum(t.numel() * t.element_size() for t in h_gate)
    d2h = sum(t.numel() * 2 for t in h_dX)

    # uploads, kernels and read-backs run on three streams: layer i's upload
    # overlaps layer i-1's kernel and layer i-2's read-back.  Events keep each
    # layer's order (upload -> kernel -> read-back) and, across steps, keep an
    # upload from overwriting a dY the previous step's kernel still reads and a
    # kernel from overwriting a dX not yet read back.
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in state]
    ev_done = [torch.cuda.Event() for _ in state]
    ev_out = [torch.cuda.Event() for _ in state]

    def e2e_step():
        for i, (_, p, d_dY, d_Wp, d_dX) in enumerate(state):
            s_in.wait_event(ev_done[i])  # no-op before the event's first record
            with torch.cuda.stream(s_in):
                d_dY.copy_(h_dY[i], non_blocking=True)
                if h_gate:
                    gates[i].copy_(h_gate[i], non_blocking=True)
            ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            stream.wait_event(ev_out[i])
            p.dgrad(d_dY, d_Wp, d_dX, gates[i], stream)
            ev_done[i].record(stream)
            s_out.wait_event(ev_done[i])
            with torch.cuda.stream(s_out):
                h_dX[i].copy_(d_dX, non_blocking=True)
            ev_out[i].record(s_out)

    e2e_step()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for _ in range(args.e2e_steps):
        e2e_step()
    stream.wait_event(ev_out[-1])  # the last read-back (s_out runs in order)
    e1.record(stream)
    torch.cuda.synchronize()
    for i, (L, p, d_dY, d_Wp, d_dX) in enumerate(state):  # the read-backs hold the kernels' results
        if not torch.equal(h_dX[i][::4099], d_dX[::4099].cpu()):
            raise RuntimeError(f"end-to-end read-back of {L.name} differs from the device result")
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = world * flops_step * args.e2e_steps / (e2e_ms * 1e-3) / 1e12
    for (_, p, *_rest) in state:
        st = p.device_status(stream)
        if st != 0:
            raise RuntimeError(f"device status {st} after timed runs")

    if rank != 0:
        return
    configs = None if args.no_other_configs else other_configs(torch, cdg, dev, stream, peaks, basis, host, state)
    cpu = None
    if not args.no_cpu_baseline:
        c = cpu_oracle_sample([s[0] for s in state], host, args.cpu_images)
        cpu = {k: c[k] for k in ("value", "unit", "cores", "kind", "sample")}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD + {"none": "", "x": "_relu_bwd_x", "bits": "_relu_bwd_bits"}[gate],
                   "global_batch": 256 * world, "layers": nL,
                   "l2": "inputs larger than L2: the step cycles ~5 GB of operands, so each layer's data is "
                         "evicted before its next use",
                   "flops_per_step": flops_step, "parallelism": f"replicas x{world}", "gate": gate,
                   "plans": "autotuned at set-up (cdg_autotune, 5 cold-cache launches per candidate)" if args.autotune
                   else "planner defaults"},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                "copies": "pinned host buffers; uploads, kernels and read-backs on three streams"},
        "gpu_launches": nL * args.steps,
        "clocks": clk,
        "host_wall_s_timed": round(t_host1 - t_host0, 4),
        "per_layer": per_layer,
        "per_layer_timing": "passes of their own before the timed region: ms = each layer launched back to back "
                            "(10 or more launches rotating over enough copies of its buffers that none finds its "
                            "operands in L2), events around the run only; ms_event_pair = one CUDA event pair "
                            "around every launch of the 22-layer sequence (adds ~3 us of event overhead a launch)",
        "per_layer_sum_ms": round(float(np.sum(per_layer_ms)), 4),
        "per_layer_sum_ms_event_pair": round(float(np.sum(per_layer_ms_events)), 4),
        "other_configs": configs,
        "peaks": peaks,
        "toolchain": toolchain(),
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
