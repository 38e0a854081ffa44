"""Benchmark of the one-row decode MLP on GB300.

Default workload: the Qwen3-8B-shaped decode stack (d=4096, f=12288, one row,
36 layers with distinct weights, affine INT8 group 128, ~5.6 GB streamed per
step -- larger than L2, so no flush is needed between steps).  A step is one
pass over the whole stack: per layer add+RMSNorm, gate/up GEMV + SwiGLU, down
GEMV + residual.  Default path: the warmed executor (mt_mlp_plan_run: one
persistent cooperative kernel for the whole stack).  --path calls times the
three single-call C-ABI kernels per layer instead (captured into one CUDA
graph, programmatic dependent launch between them); its time is also
reported beside the executor's as ``calls_path``.

Printed JSON line (one per run, rank 0):
  value       effective HBM GB/s = algorithmic bytes of the step / step time
  e2e         the same metric with the step's inputs copied host->device from
              pinned memory and the output read back, inside the timed region
  roofline    the dominant kernel (the stack kernel; with --path calls the
              gate/up + SwiGLU kernel timed alone over the 36 layers) with CUDA
              events, against the measured HBM peak
  cpu_baseline the float64 CPU oracle timed on one layer of the same workload
  clocks      SM clocks / throttle reasons sampled during the timed region

``--impl reference`` times the CPU oracle (the only reference this method
has: the pages describe Apple-GPU Metal kernels that cannot run here).
Multi-GPU (torchrun): independent replicas, one stack per GPU, no collective
on the data path; value = total bytes of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per decode MLP layer and effective HBM GB/s (fraction of ~8 TB/s peak)"
# ncu summaries under profiles/ and the sources of the kernel each covers (the
# traffic figure is used only while the kernel is unchanged)
PROFILES = {
    "gateup": (os.path.join(ROOT, "profiles", "gateup_affine8_qwen3-8b.txt"),
               ["k_gemv.cuh", "k_phase.cuh", "k_gemv_warp.cuh", "k_gemv_run.cuh", "k_gemv_a8.cu",
                "mt_device.cuh"]),
    "stack": (os.path.join(ROOT, "profiles", "stack_affine8_qwen3-8b.txt"),
              ["k_gemv.cuh", "k_phase.cuh", "k_stack.cu", "mt_device.cuh"]),
}


def kernel_hash(kind: str) -> str:
    h = hashlib.sha256()
    for f in PROFILES[kind][1]:
        with open(os.path.join(ROOT, "quantized_gemv_epilogues_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def profiled_traffic(kind: str):
    """Per-launch DRAM bytes of a kernel from its committed ncu summary, or
    None when the summary is missing or the kernel changed since."""
    path = PROFILES[kind][0]
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as fh:
        for line in fh:
            if ":" in line:
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    if kv.get("kernel_sources_sha256_16") != kernel_hash(kind):
        return None
    try:
        return int(kv["dram_bytes_per_launch_full"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ clocks
# NVML clock event reason bits (nvml.h): software power cap, hardware
# slowdown, software / hardware thermal slowdown.
_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown"}


class ClockSampler:
    """SM clock and clock-event reasons sampled DURING the timed region.

    Reads NVML in-process every ~2 ms from a thread (libnvidia-ml through
    ctypes; reading clocks changes no setting), so a region of a few tens of
    milliseconds gets several samples; falls back to nvidia-smi every 20 ms
    when NVML cannot be loaded.  The GPU is found by its PCI bus id."""

    def __init__(self, gpu_index: int, torch=None):
        self.gpu = gpu_index
        self.torch = torch
        self.samples = []  # (sm_mhz, reasons_mask)
        self.sm_max = None
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None

    # -- NVML
    def _nvml_handle(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        ok = False
        if self.torch is not None:
            try:
                pr = self.torch.cuda.get_device_properties(self.gpu)
                bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0".encode()
                ok = lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(h)) == 0
            except Exception:
                ok = False
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(self.gpu, ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # NVML_CLOCK_SM
            self.sm_max = float(mx.value)
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, reasons

    def _nvml_loop(self, lib, h, reasons):
        import ctypes
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                r = rs.value if reasons(h, ctypes.byref(rs)) == 0 else 0
                self.samples.append((float(clk.value), int(r)))
            time.sleep(0.002)

    # -- nvidia-smi
    def _smi_loop(self):
        fields = "clocks.sm,clocks.max.sm,clocks_event_reasons.active"
        self._proc = subprocess.Popen(
            ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={fields}", "--format=csv,noheader,nounits",
             "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        for line in self._proc.stdout:
            parts = [t.strip() for t in line.split(",")]
            try:
                self.sm_max = float(parts[1])
                self.samples.append((float(parts[0]), int(parts[2], 16)))
            except (ValueError, IndexError):
                pass

    def __enter__(self):
        try:
            lib, h, reasons = self._nvml_handle()
            self.source = "nvml"
            self._thread = threading.Thread(target=self._nvml_loop, args=(lib, h, reasons), daemon=True)
        except (OSError, AttributeError):
            self.source = "nvidia-smi"
            self._thread = threading.Thread(target=self._smi_loop, daemon=True)
        self._thread.start()
        time.sleep(0.005)
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.sm_max, "reasons": ["no samples"], "samples": 0,
                    "source": self.source}
        mask = 0
        for _, r in self.samples:
            mask |= r
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.sm_max,
                "reasons": sorted(n for bit, n in _REASONS.items() if mask & bit),
                "samples": len(self.samples), "source": self.source}


# ------------------------------------------------------------------ stack
class Stack:
    """Device-resident packed weights and activation buffers of a decode stack."""

    def __init__(self, wl, device, layers=None):
        import torch
        import synth
        import quantized_gemv_epilogues_gb300 as mt
        self.mt, self.torch = mt, torch
        self.wl = wl
        self.L = layers or wl.layers
        d, f, M, g = wl.d, wl.f, wl.M, wl.group
        self.dev = device
        bf = torch.bfloat16
        tmp = torch.empty(max(d * f, 1), dtype=torch.float32, device=device)
        self.values = torch.empty(self.L, M, d, dtype=bf, device=device)  # per-layer addends
        self.layers = []
        for l in range(self.L):
            sd = lambda t: synth.seed_for(wl.wid, l, t)
            w_norm = torch.empty(d, dtype=bf, device=device)
            synth.device_bf16(w_norm, sd(synth.T_NORM_W), synth.NORM_W)
            if wl.fmt == synth.FMT_BF16:
                Wg = torch.empty(f, d, dtype=bf, device=device)
                Wu = torch.empty(f, d, dtype=bf, device=device)
                Wd = torch.empty(d, f, dtype=bf, device=device)
                synth.device_bf16(Wg, sd(synth.T_WG), wl.weight_dist)
                synth.device_bf16(Wu, sd(synth.T_WU), wl.weight_dist)
                synth.device_bf16(Wd, sd(synth.T_WD), wl.weight_dist)
                sgu = bgu = sdn = bdn = None
            else:
                bits = wl.bits
                mx = synth.is_mx(wl.fmt)
                sdt = torch.uint8 if mx else bf
                Wg = torch.empty(f, d * bits // 8, dtype=torch.uint8, device=device)
                Wu = torch.empty_like(Wg)
                Wd = torch.empty(d, f * bits // 8, dtype=torch.uint8, device=device)
                sgu = torch.empty(2, f, d // g, dtype=sdt, device=device)
                sdn = torch.empty(d, f // g, dtype=sdt, device=device)
                bgu = None if mx else torch.empty_like(sgu)
                bdn = None if mx else torch.empty_like(sdn)
                for (dst, s_, b_, N, K, t) in ((Wg, sgu[0], None if mx else bgu[0], f, d, synth.T_WG),
                                               (Wu, sgu[1], None if mx else bgu[1], f, d, synth.T_WU),
                                               (Wd, sdn, bdn, d, f, synth.T_WD)):
                    W32 = tmp[:N * K].view(N, K)
                    synth.device_f32(W32, sd(t), wl.weight_dist)
                    if mx:
                        mt.mt_pack_mx(W32, N, K, bits, dst, s_)
                    else:
                        mt.mt_pack_affine(W32, N, K, g, bits, dst, s_, b_)
            values = self.values[l]
            synth.device_bf16(values, sd(synth.T_VALUES), synth.ACT)
            self.layers.append(dict(w=w_norm, Wg=Wg, Wu=Wu, Wd=Wd, sgu=sgu, bgu=bgu, sd=sdn,
                                    bd=bdn, values=values))
        del tmp
        self.r0 = torch.empty(M, d, dtype=bf, device=device)
        synth.device_bf16(self.r0, synth.seed_for(wl.wid, 0, synth.T_RESIDUAL), synth.ACT)
        self.resid = torch.empty(M, d, dtype=bf, device=device)
        self.norm = torch.empty(M, d, dtype=bf, device=device)
        self.h = torch.empty(M, wl.f, dtype=bf, device=device)
        self.out_y = torch.empty(M, d, dtype=bf, device=device)
        self.plan = None
        if M == 1 and not synth.is_mx(wl.fmt):
            self.plan = mt.mt_mlp_plan_create(
                [dict(norm_weight=L["w"], Wg=L["Wg"], Wu=L["Wu"], gu_scales=L["sgu"],
                      gu_biases=L["bgu"], Wd=L["Wd"], d_scales=L["sd"], d_biases=L["bd"])
                 for L in self.layers], d, f, g, wl.fmt, wl.eps)
        torch.cuda.synchronize()

    def close(self):
        if self.plan is not None:
            self.mt.mt_mlp_plan_destroy(self.plan)
            self.plan = None

    def step_executor(self):
        """One pass over the stack: one mt_mlp_plan_run (one kernel)."""
        self.mt.mt_mlp_plan_run(self.plan, self.values, self.r0, self.out_y)

    def step_calls(self):
        """One pass over the stack (3 C-ABI calls per layer)."""
        mt, wl = self.mt, self.wl
        self.resid.copy_(self.r0)
        for L in self.layers:
            mt.mt_add_rmsnorm(L["values"], self.resid, L["w"], wl.eps, self.resid, self.norm)
            mt.mt_swiglu_gateup(self.norm, L["Wg"], L["Wu"], L["sgu"], L["bgu"], wl.group, self.h,
                                fmt=wl.fmt)
            mt.mt_down_residual(self.h, L["Wd"], L["sd"], L["bd"], wl.group, self.resid, self.resid,
                                fmt=wl.fmt)

    def gateup_only(self):
        mt, wl = self.mt, self.wl
        for L in self.layers:
            mt.mt_swiglu_gateup(self.norm, L["Wg"], L["Wu"], L["sgu"], L["bgu"], wl.group, self.h,
                                fmt=wl.fmt)

    def down_only(self):
        mt, wl = self.mt, self.wl
        for L in self.layers:
            mt.mt_down_residual(self.h, L["Wd"], L["sd"], L["bd"], wl.group, self.resid, self.resid,
                                fmt=wl.fmt)

    def run_layers(self, seq, kernels=("norm", "gateup", "down")):
        """The chosen single-call kernels of layers seq[0], seq[1], ... back to
        back (the residual carries over from layer to layer)."""
        mt, wl = self.mt, self.wl
        for l in seq:
            L = self.layers[l]
            if "norm" in kernels:
                mt.mt_add_rmsnorm(L["values"], self.resid, L["w"], wl.eps, self.resid, self.norm)
            if "gateup" in kernels:
                mt.mt_swiglu_gateup(self.norm, L["Wg"], L["Wu"], L["sgu"], L["bgu"], wl.group, self.h,
                                    fmt=wl.fmt)
            if "down" in kernels:
                mt.mt_down_residual(self.h, L["Wd"], L["sd"], L["bd"], wl.group, self.resid,
                                    self.resid, fmt=wl.fmt)

    def rmsnorm_only(self):
        mt, wl = self.mt, self.wl
        for L in self.layers:
            mt.mt_add_rmsnorm(L["values"], self.resid, L["w"], wl.eps, self.resid, self.norm)

    def down_bytes(self):
        import synth
        wl = self.wl
        n = wl.f * wl.d
        w = n * wl.bits // 8 + synth.scale_bytes(wl.fmt, n, wl.group)
        return w + 2 * wl.M * wl.f + 4 * wl.M * wl.d

    def gateup_bytes(self):
        import synth
        wl = self.wl
        n = 2 * wl.f * wl.d
        w = n * wl.bits // 8 + synth.scale_bytes(wl.fmt, n, wl.group)
        return w + 2 * wl.M * wl.d + 2 * wl.M * wl.f


class DirectLaunch:
    """Stands in for a captured graph: replay() calls the launches directly."""

    def __init__(self, fn):
        self.fn = fn

    def replay(self):
        self.fn()


def capture(fn, torch, direct=False):
    if direct:
        fn()
        torch.cuda.synchronize()
        return DirectLaunch(fn)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm (plans, attributes) outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    try:
        with torch.cuda.graph(g):
            fn()
    except RuntimeError as e:  # a launch kind the graph cannot hold: launch directly
        print(f"bench: graph capture failed ({e}); launching directly", file=sys.stderr)
        torch.cuda.synchronize()
        return DirectLaunch(fn)
    torch.cuda.synchronize()
    return g


def time_graph(g, n, torch):
    """Mean ms per replay of g over n back-to-back replays (CUDA events on
    the launching stream)."""
    return time_steps(g, n, torch)[0] / n


def time_steps(g, n, torch):
    """n replays of g on one stream, each bracketed by CUDA events recorded
    on that stream: (total ms from the first start to the last end, per-step
    ms)."""
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        torch.cuda.synchronize()
        ev[0].record(st)
        for i in range(n):
            g.replay()
            ev[i + 1].record(st)
        ev[-1].synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]
    return ev[0].elapsed_time(ev[-1]), per


def step_stats(per_ms):
    """Median, 10th and 90th percentile (nearest rank) of per-step times."""
    v = sorted(per_ms)
    q = lambda f: v[min(len(v) - 1, max(0, int(math.ceil(f * len(v))) - 1))]
    return {"median": round(statistics.median(v), 4), "p10": round(q(0.10), 4), "p90": round(q(0.90), 4),
            "n": len(v)}


# ------------------------------------------------------------------ CPU oracle
class OracleLayer:
    """One layer of `wl` for the float64 CPU oracle: weights generated and
    quantised once (outside any timed region); run() is one oracle pass."""

    def __init__(self, wl):
        import oracle
        import synth
        self.oracle, self.wl = oracle, wl
        d, f, M, g = wl.d, wl.f, wl.M, wl.group
        sd = lambda t: synth.seed_for(wl.wid, 0, t)
        gen = lambda N, K, t: synth.host_f32(N * K, sd(t), wl.weight_dist).reshape(N, K)
        self.Wg = oracle.Weight.from_f32(gen(f, d, synth.T_WG), wl.bits, g)
        self.Wu = oracle.Weight.from_f32(gen(f, d, synth.T_WU), wl.bits, g)
        self.Wd = oracle.Weight.from_f32(gen(d, f, synth.T_WD), wl.bits, g)
        self.v = synth.host_bf16(M * d, sd(synth.T_VALUES), synth.ACT).reshape(M, d)
        self.r = synth.host_bf16(M * d, sd(synth.T_RESIDUAL), synth.ACT).reshape(M, d)
        self.w = synth.host_bf16(d, sd(synth.T_NORM_W), synth.NORM_W)

    def run(self):
        return self.oracle.mlp_layer(self.v, self.r, self.w, self.wl.eps, self.Wg, self.Wu, self.Wd)


def oracle_layer_timing(wl, budget_s: float = 12.0, max_reps: int = 64):
    """Times the CPU oracle on one layer of `wl` for about `budget_s` seconds
    in this process (one thread).  Returns (us_per_layer, reps)."""
    lay = OracleLayer(wl)
    reps, t0 = 0, time.perf_counter()
    while True:
        lay.run()
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= max_reps:
            break
    return el / reps * 1e6, reps


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.TimeoutExpired):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


# Worker state of OraclePool (one layer per process, built once).
_POOL_LAYER = None
_POOL_BARRIER = None


def _pool_init(wl_args, barrier):
    global _POOL_LAYER, _POOL_BARRIER
    sys.path.insert(0, ROOT)
    import synth
    _POOL_LAYER = OracleLayer(synth.QWEN8B.with_(**wl_args))
    _POOL_BARRIER = barrier


def _pool_run(_):
    # every worker waits for all the others, so each takes exactly one pass
    _POOL_BARRIER.wait(timeout=600)
    t0 = time.perf_counter()
    _POOL_LAYER.run()
    return time.perf_counter() - t0


class OraclePool:
    """The CPU oracle on all host cores: `procs` processes (started with
    spawn, so no CUDA state is inherited), each holding one layer of the
    workload quantised by the oracle; step() runs the layer once in every
    process at the same time, i.e. `procs` layers per step."""

    def __init__(self, wl, procs):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.procs = procs
        self.barrier = ctx.Barrier(procs)
        args = dict(d=wl.d, f=wl.f, M=wl.M, group=wl.group, fmt=wl.fmt, eps=wl.eps, wid=wl.wid)
        self.pool = ctx.Pool(procs, initializer=_pool_init, initargs=(args, self.barrier))

    def step(self):
        t0 = time.perf_counter()
        per = self.pool.map(_pool_run, range(self.procs), chunksize=1)
        return time.perf_counter() - t0, per

    def close(self):
        self.pool.terminate()
        self.pool.join()


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_pool_timing(wl, steps: int = 3):
    """Layers per second of the oracle over every host core (one process
    per core, one layer each per step); the first step warms up."""
    procs = host_cores()
    pool = OraclePool(wl, procs)
    try:
        pool.step()
        walls = [pool.step()[0] for _ in range(steps)]
    finally:
        pool.close()
    return procs * steps / sum(walls), procs


def workload_config(wl):
    """The workload only (shared by the GPU arm and the reference arm)."""
    return {"workload": wl.name, "d": wl.d, "f": wl.f, "rows_M": wl.M, "layers": wl.layers,
            "weights": {0: "bf16", 1: "affine8", 2: "affine4"}[wl.fmt], "group": wl.group,
            "eps": wl.eps, "bytes_per_layer": wl.layer_bytes()}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, ws: int, torch, device=None):
    """Max over ranks (gloo on CPU or nccl on GPU)."""
    if ws == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args):
    """The reference arm: the float64 CPU oracle over every host core (one
    process per core), each step one layer of the Qwen3-8B stack in every
    process at once -- a bounded sample of the workload; value = layers per
    step / step time, in the GPU arm's unit.  Under torchrun only rank 0 runs."""
    import synth
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    wl = synth.QWEN8B
    pool = OraclePool(wl, host_cores())
    try:
        for _ in range(max(0, args.warmup)):
            pool.step()
        walls = [pool.step()[0] for _ in range(max(1, args.steps))]
    finally:
        pool.close()
    per_layer_s = sum(walls) / (len(walls) * pool.procs)  # wall time per layer over all cores
    us = per_layer_s * 1e6
    gbs = wl.layer_bytes() / per_layer_s / 1e9
    sample = (f"{pool.procs} processes (one per host core), each one {wl.d}x{wl.f} affine8 g128 "
              f"layer per step, of the {wl.layers}-layer stack; single-threaded binary64 C oracle")
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
            "us_per_layer": round(us, 1), "n_gpus": args.gpus, "steps": len(walls),
            "warmup": args.warmup, "ms_per_step": round(sum(walls) / len(walls) * 1e3, 3),
            "step_ms": step_stats([w * 1e3 for w in walls]), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl),
            "path": "float64 CPU oracle, one layer per process per step, host cores",
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": pool.procs,
                             "threads": pool.procs, "nproc": os.cpu_count(), "cpu_model": cpu_model(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


SWEEP_REPS = 24  # layers per timed graph in the sweep


def measure_layer(wl, args, torch, mt, dev, reps=None):
    """One layer shape, hot and cold: us per layer of the three single calls
    (and of each GEMV alone) and, for one row, of the warmed executor.  Hot:
    the same layer `reps` times in one CUDA graph (weights resident in L2 when
    they fit).  Cold: the graph cycles through enough distinct copies of the
    layer (different seeds) to exceed twice the L2 size, so each layer's
    weights come from HBM."""
    import math
    reps = reps or SWEEP_REPS
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def timed(fn, n_layers, steps):
        gk = capture(fn, torch, direct=args.no_graph)
        for _ in range(max(3, args.warmup)):
            gk.replay()
        us = time_graph(gk, steps, torch) * 1e3 / n_layers
        del gk
        return us

    n_cold = int(math.ceil(2 * l2 / wl.layer_bytes())) + 1
    st = Stack(wl, dev, layers=n_cold)
    hot = [0] * reps
    cold = list(range(n_cold)) * max(1, reps // n_cold)
    pt = {"bytes_per_layer": wl.layer_bytes(), "cold_copies": n_cold}
    for tag, seq in (("", hot), ("_cold", cold)):
        us = timed(lambda: st.run_layers(seq), len(seq), args.steps)
        gu = timed(lambda: st.run_layers(seq, ("gateup",)), len(seq), max(5, args.steps // 2))
        dn = timed(lambda: st.run_layers(seq, ("down",)), len(seq), max(5, args.steps // 2))
        pt.update({"us_per_layer" + tag: round(us, 3),
                   "gbs" + tag: round(wl.layer_bytes() / (us * 1e-6) / 1e9, 1),
                   "gateup_us" + tag: round(gu, 3),
                   "gateup_gbs" + tag: round(st.gateup_bytes() / (gu * 1e-6) / 1e9, 1),
                   "down_us" + tag: round(dn, 3),
                   "down_gbs" + tag: round(st.down_bytes() / (dn * 1e-6) / 1e9, 1)})
    if wl.M == 1 and st.plan is not None:
        # executor: a plan of the same layer `reps` times (hot) and the stack
        # plan over the distinct copies (cold)
        lay = st.layers[0]
        hot_plan = mt.mt_mlp_plan_create(
            [dict(norm_weight=lay["w"], Wg=lay["Wg"], Wu=lay["Wu"], gu_scales=lay["sgu"],
                  gu_biases=lay["bgu"], Wd=lay["Wd"], d_scales=lay["sd"], d_biases=lay["bd"])] * reps,
            wl.d, wl.f, wl.group, wl.fmt, wl.eps)
        vals = torch.zeros(reps, 1, wl.d, dtype=torch.bfloat16, device=dev)
        vals.copy_(st.values[:1].expand(reps, 1, wl.d))
        try:
            us_h = timed(lambda: mt.mt_mlp_plan_run(hot_plan, vals, st.r0, st.out_y), reps, args.steps)
        finally:
            mt.mt_mlp_plan_destroy(hot_plan)
        us_c = timed(st.step_executor, n_cold, args.steps)
        pt.update({"executor_us": round(us_h, 3),
                   "executor_gbs": round(wl.layer_bytes() / (us_h * 1e-6) / 1e9, 1),
                   "executor_us_cold": round(us_c, 3),
                   "executor_gbs_cold": round(wl.layer_bytes() / (us_c * 1e-6) / 1e9, 1)})
    st.close()
    del st
    torch.cuda.empty_cache()
    return pt


def run_sweep(args, torch, synth, mt, dev):
    """Config 5: one d=2048, f=8192 affine INT8 layer (1 % x20 outliers) per
    point, group in {32, 64, 128} x rows M in {1, 2, 4, 8}: us per layer
    (add+RMSNorm, gate/up+SwiGLU, down+residual as single calls) and effective
    GB/s per point, hot and cold (measure_layer; one-row points also time the
    warmed executor).  The JSON line's value is the geometric mean of the cold
    GB/s."""
    import math
    reps = SWEEP_REPS
    points = []
    peak, peak_kind = measured_peaks()
    for g in ((args.sweep_group,) if args.sweep_group else (32, 64, 128)):
        for M in ((args.sweep_rows,) if args.sweep_rows else (1, 2, 4, 8)):
            pt = {"group": g, "M": M}
            pt.update(measure_layer(synth.sweep_point(g, M), args, torch, mt, dev, reps))
            points.append(pt)
    gm = math.exp(sum(math.log(p["gbs_cold"]) for p in points) / len(points))
    gm_hot = math.exp(sum(math.log(p["gbs"]) for p in points) / len(points))
    line = {"metric": METRIC, "value": round(gm, 2), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u8-weights/f32-acc",
            "data": "synthetic",
            "config": {"workload": "sweep d2048 f8192 affine8 (1 % x20 outliers), "
                                   "group {32,64,128} x M {1,2,4,8}, one layer per point",
                       "l2": "value: cold (distinct layer copies > 2x L2 cycled); "
                             f"hot: one layer x {reps} in one graph (geomean {round(gm_hot, 1)} GB/s)"},
            "peak": peak, "peak_kind": peak_kind, "points": points,
            "device_error": mt.mt_device_error()}
    print(json.dumps(line), flush=True)
    return 0


def run_configs(args, torch, synth, mt, dev):
    """Configs 1-3 (tiny, Llama-3.2-1B-shaped affine INT4, Qwen2.5-1.5B-shaped
    bf16): each layer hot and cold through the single calls and the warmed
    executor (measure_layer).  The JSON line's value is the geometric mean of
    the cold GB/s of the single calls."""
    import math
    peak, peak_kind = measured_peaks()
    points = []
    for wl in (synth.TINY, synth.LLAMA1B, synth.QWEN15):
        pt = {"workload": wl.name}
        pt.update(measure_layer(wl, args, torch, mt, dev))
        points.append(pt)
    gm = math.exp(sum(math.log(p["gbs_cold"]) for p in points) / len(points))
    line = {"metric": METRIC, "value": round(gm, 2), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "per-config weights/f32-acc",
            "data": "synthetic",
            "config": {"workload": "configs 1-3: tiny d256 f768 affine8 g64; llama3.2-1b layer d2048 "
                                   "f8192 affine4 g64; qwen2.5-1.5b layer d1536 f8960 bf16; one row",
                       "l2": "value: cold (distinct layer copies > 2x L2 cycled); hot: one layer x "
                             f"{SWEEP_REPS} in one graph"},
            "peak": peak, "peak_kind": peak_kind, "points": points,
            "device_error": mt.mt_device_error()}
    print(json.dumps(line), flush=True)
    return 0


class ProjStack:
    """Device-resident projection weights of one decode step: per layer the
    stacked q/k/v weight (and bias) and the o weight, and one vocabulary
    weight, generated by the seeded generator and packed by the library."""

    def __init__(self, pw, device, M=None):
        import torch
        import synth
        import quantized_gemv_epilogues_gb300 as mt
        self.mt, self.pw = mt, pw
        self.M = M or pw.M
        bf = torch.bfloat16
        biggest = max(p.N * p.K for p in pw.projs)
        tmp = torch.empty(biggest if pw.fmt != synth.FMT_BF16 else 1, dtype=torch.float32, device=device)
        self.items = []   # (projection, layer, W, s, b, bias, x, y)
        self.x = {}
        for p in pw.projs:
            x = torch.empty(self.M, p.K, dtype=bf, device=device)
            synth.device_bf16(x, synth.seed_for(pw.wid, 0, synth.T_X) + p.tensor, synth.ACT)
            y = torch.empty(self.M, p.N, dtype=bf, device=device)
            for l in range(pw.layers if p.per_layer else 1):
                sd = lambda t: synth.seed_for(pw.wid, l, t)
                if pw.fmt == synth.FMT_BF16:
                    W = torch.empty(p.N, p.K, dtype=bf, device=device)
                    synth.device_bf16(W, sd(p.tensor), pw.weight_dist)
                    s = b = None
                else:
                    W = torch.empty(p.N, p.K * pw.bits // 8, dtype=torch.uint8, device=device)
                    s = torch.empty(p.N, p.K // pw.group, dtype=bf, device=device)
                    b = torch.empty_like(s)
                    W32 = tmp[:p.N * p.K].view(p.N, p.K)
                    synth.device_f32(W32, sd(p.tensor), pw.weight_dist)
                    mt.mt_pack_affine(W32, p.N, p.K, pw.group, pw.bits, W, s, b)
                bias = None
                if p.bias is not None:
                    bias = torch.empty(p.N, dtype=bf, device=device)
                    synth.device_bf16(bias, sd(p.bias), synth.PROJ_BIAS)
                self.items.append((p, l, W, s, b, bias, x, y))
        del tmp
        torch.cuda.synchronize()

    def run(self, names=None):
        mt, pw = self.mt, self.pw
        for (p, l, W, s, b, bias, x, y) in self.items:
            if names is None or p.name in names:
                mt.mt_linear_bias(x, W, s, b, pw.group, bias, y, fmt=pw.fmt)

    def launches(self, names=None):
        return sum(1 for it in self.items if names is None or it[0].name in names)

    def bytes(self, names=None):
        pw = self.pw
        tot = 0
        for (p, l, *_rest) in self.items:
            if names is None or p.name in names:
                tot += pw.proj_weight_bytes(p) + 2 * self.M * (p.K + p.N)
        return tot


def run_projections(args, torch, synth, mt, dev):
    """The projection GEMV (mt_linear_bias) over one decode step of each model:
    per layer the stacked q/k/v projection (with its bias where the model has
    one) and the o projection, then the vocabulary projection once.  Every
    weight is distinct and the step's weights exceed the L2, so each launch
    reads its weights from HBM.  Per model: us per step, effective GB/s of the
    step and of each projection kind alone.  The JSON line's value is the
    Qwen3-8B step's GB/s."""
    peak, peak_kind = measured_peaks()
    points = []
    for pw in synth.PROJ_ALL:
        M = args.rows or pw.M
        ps = ProjStack(pw, dev, M)
        pt = {"workload": pw.name, "M": M, "step_bytes": ps.bytes(), "launches": ps.launches()}
        g = capture(ps.run, torch, direct=args.no_graph)
        for _ in range(max(3, args.warmup)):
            g.replay()
        steps = max(5, args.steps // 10)
        with ClockSampler(dev.index or 0, torch) as clk:
            ms = time_graph(g, steps, torch)
        del g
        pt.update({"us_per_step": round(ms * 1e3, 2),
                   "gbs": round(ps.bytes() / (ms * 1e-3) / 1e9, 1),
                   "frac_of_measured_hbm": round(ps.bytes() / (ms * 1e-3) / 1e9 / peak, 4),
                   "clocks": clk.summary()})
        for p in pw.projs:
            gk = capture(lambda: ps.run((p.name,)), torch, direct=args.no_graph)
            for _ in range(3):
                gk.replay()
            us = time_graph(gk, steps, torch) * 1e3 / ps.launches((p.name,))
            del gk
            nb = ps.bytes((p.name,)) / ps.launches((p.name,))
            pt[p.name] = {"K": p.K, "N": p.N, "bias": p.bias is not None, "us_per_launch": round(us, 3),
                          "gbs": round(nb / (us * 1e-6) / 1e9, 1)}
        points.append(pt)
        del ps
        torch.cuda.empty_cache()
    head = points[0]
    lm = head["lm_head"]
    line = {"metric": "µs per decode step of the attention and vocabulary projections and effective HBM GB/s",
            "value": head["gbs"], "unit": "GB/s", "n_gpus": 1,
            "steps": max(5, args.steps // 10), "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "per-model weights/f32-acc",
            "data": "synthetic",
            "config": {"workload": "; ".join(pw.name for pw in synth.PROJ_ALL),
                       "l2": "every weight distinct, step weights > L2"},
            "roofline": {"bound": "hbm", "kernel": "gemv_warp_kernel lm_head 4096x151936 affine8 g128",
                         "achieved": lm["gbs"], "peak": peak, "unit": "GB/s",
                         "frac": round(lm["gbs"] / peak, 4), "peak_kind": peak_kind},
            "points": points, "device_error": mt.mt_device_error()}
    print(json.dumps(line), flush=True)
    return 0


def bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return float(d["bf16_tflops"]), "measured (bf16 dense burst; fp16 runs at the same rate)"
    return 1900.0, "fallback"


def run_prefill(args, torch, synth, mt, dev):
    """Multi-row prefill of the Qwen3-8B layer (d=4096, f=12288, affine INT8
    g128) on the tcgen05 GEMMs: gate/up + SwiGLU and down + residual for M
    activation rows, three distinct layers cycled (455 MB of weights, past the
    L2).  Per M: us per layer, TFLOP/s (6 M d f flops per layer) and effective
    GB/s.  The JSON line's value is the TFLOP/s at the largest M."""
    hbm, hbm_kind = measured_peaks()
    tpk, tpk_kind = bf16_peak()
    points = []
    n_layers = 3
    runs = [(synth.QWEN8B, M) for M in ((args.rows,) if args.rows else (16, 64, 256, 1024, 4096))]
    if not args.rows:  # the dense bf16 layer (Qwen2.5-1.5B shape) at one size
        runs.append((synth.QWEN15, 1024))
    for base, M in runs:
        wl = base.with_(M=M, layers=n_layers)
        st = Stack(wl, dev)
        d, f, g = wl.d, wl.f, wl.group
        bf = torch.bfloat16
        x = torch.empty(M, d, dtype=bf, device=dev)
        hin = torch.empty(M, f, dtype=bf, device=dev)
        res = torch.empty(M, d, dtype=bf, device=dev)
        synth.device_bf16(x, synth.seed_for(wl.wid, M, synth.T_X), synth.ACT)
        synth.device_bf16(hin, synth.seed_for(wl.wid, M, synth.T_H), synth.ACT)
        synth.device_bf16(res, synth.seed_for(wl.wid, M, synth.T_RES3), synth.ACT)
        h = torch.empty(M, f, dtype=bf, device=dev)
        y = torch.empty(M, d, dtype=bf, device=dev)
        ws = torch.empty(max(mt.mt_prefill_workspace_bytes(M, d, f, g), mt.mt_prefill_workspace_bytes(M, f, d, g)),
                         dtype=torch.uint8, device=dev)

        def gateup():
            for L in st.layers:
                mt.mt_prefill_swiglu_gateup(x, L["Wg"], L["Wu"], L["sgu"], L["bgu"], g, h, ws, fmt=wl.fmt)

        def down():
            for L in st.layers:
                mt.mt_prefill_down_residual(hin, L["Wd"], L["sd"], L["bd"], g, res, y, ws, fmt=wl.fmt)

        def both():
            gateup()
            down()

        reps = max(3, min(args.steps // 10, 20))
        res_us = {}
        clk = None
        for name, fn in (("layer", both), ("gateup", gateup), ("down", down)):
            gk = capture(fn, torch, direct=args.no_graph)
            for _ in range(max(3, args.warmup)):
                gk.replay()
            if name == "layer":
                with ClockSampler(dev.index or 0, torch) as clk:
                    res_us[name] = time_graph(gk, reps, torch) * 1e3 / n_layers
            else:
                res_us[name] = time_graph(gk, reps, torch) * 1e3 / n_layers
            del gk
        fl_gu, fl_dn = 2.0 * M * d * (2 * f), 2.0 * M * f * d
        by_gu = st.gateup_bytes()
        by_dn = st.down_bytes()
        pt = {"workload": base.name.split(" stack")[0], "M": M, "us_per_layer": round(res_us["layer"], 2),
              "tflops": round((fl_gu + fl_dn) / (res_us["layer"] * 1e-6) / 1e12, 1),
              "gbs": round((by_gu + by_dn) / (res_us["layer"] * 1e-6) / 1e9, 1),
              "gateup_us": round(res_us["gateup"], 2),
              "gateup_tflops": round(fl_gu / (res_us["gateup"] * 1e-6) / 1e12, 1),
              "down_us": round(res_us["down"], 2),
              "down_tflops": round(fl_dn / (res_us["down"] * 1e-6) / 1e12, 1),
              "clocks": clk.summary() if clk else None}
        pt["frac_of_tensor_peak"] = round(pt["tflops"] / tpk, 4)
        pt["frac_of_hbm_peak"] = round(pt["gbs"] / hbm, 4)
        points.append(pt)
        st.close()
        del st, ws, x, hin, res, h, y
        torch.cuda.empty_cache()
    top = max((p for p in points if p["workload"].startswith("qwen3-8b")), key=lambda p: p["M"])
    line = {"metric": "prefill TFLOP/s of the decode MLP layer's GEMMs (gate/up + SwiGLU, down + residual)",
            "value": top["tflops"], "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8-weights/fp16-mma/f32-acc",
            "data": "synthetic",
            "config": {"workload": "qwen3-8b layer d4096 f12288 affine8 g128, M activation rows, 3 distinct layers cycled",
                       "l2": "weights of 3 layers (467 MB) exceed the L2"},
            "roofline": {"bound": "tensor",
                         "kernel": f"prefill_dq_kernel (bf16 outputs: fp16-dequantised weight tiles; M = {top['M']})",
                         "achieved": top["tflops"], "peak": tpk, "unit": "TFLOP/s",
                         "frac": top["frac_of_tensor_peak"], "peak_kind": tpk_kind},
            "hbm_peak": hbm, "hbm_peak_kind": hbm_kind, "points": points, "device_error": mt.mt_device_error()}
    print(json.dumps(line), flush=True)
    return 0


def run_mx(args, torch, synth, mt, dev):
    """The Qwen3-8B-shaped layer (d=4096, f=12288) with MX block-scaled
    weights (MXFP8, MXFP4), M = 1 and 4: us per layer of the single calls and
    of each GEMV, hot and cold (measure_layer).  The JSON line's value is the
    geometric mean of the cold GB/s."""
    import math
    peak, peak_kind = measured_peaks()
    points = []
    for wl in (synth.QWEN8B_MXFP8, synth.QWEN8B_MXFP4):
        for M in ((args.rows,) if args.rows else (1, 4)):
            w = wl.with_(M=M)
            pt = {"workload": w.name, "M": M}
            pt.update(measure_layer(w, args, torch, mt, dev))
            points.append(pt)
    gm = math.exp(sum(math.log(p["gbs_cold"]) for p in points) / len(points))
    line = {"metric": METRIC, "value": round(gm, 2), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8/mxfp4-weights/f32-acc",
            "data": "synthetic",
            "config": {"workload": "qwen3-8b layer d4096 f12288 with MXFP8 and MXFP4 weights (E8M0 "
                                   "scales per 32), M 1 and 4, single calls",
                       "l2": "value: cold (distinct layer copies > 2x L2 cycled); hot: one layer x "
                             f"{SWEEP_REPS} in one graph"},
            "peak": peak, "peak_kind": peak_kind, "points": points,
            "device_error": mt.mt_device_error()}
    print(json.dumps(line), flush=True)
    return 0


def run_only(args, torch, synth, mt, dev):
    """Profiling aid: the chosen kernels over the workload's layers, warm-up +
    steps times, launched directly (no graph, no timing, no JSON line), so a
    profiler sees plain launches in a known order."""
    if args.workload == "sweep":
        wl = synth.sweep_point(args.sweep_group or 128, args.sweep_rows or 1)
    elif args.workload == "mx":
        wl = {"fp8": synth.QWEN8B_MXFP8, "fp4": synth.QWEN8B_MXFP4}[args.mx].with_(M=args.rows or 1)
    elif args.workload == "projections":
        # one model's vocabulary projection (--proj), launched warm-up + steps times
        pw = {"qwen3-8b": synth.QWEN8B_PROJ, "qwen15": synth.QWEN15_PROJ,
              "llama1b": synth.LLAMA1B_PROJ}[args.proj]
        ps = ProjStack(pw, dev, args.rows or pw.M)
        vocab = [p.name for p in pw.projs if not p.per_layer]
        for _ in range(max(3, args.warmup) + args.steps):
            ps.run(vocab)
        torch.cuda.synchronize()
        return 0
    elif args.workload in ("qwen3-8b", "tiny", "llama1b", "qwen15"):
        wl = {"qwen3-8b": synth.QWEN8B, "tiny": synth.TINY, "llama1b": synth.LLAMA1B,
              "qwen15": synth.QWEN15}[args.workload]
    else:
        raise SystemExit(f"--only does not take --workload {args.workload}")
    if args.layers:
        wl = wl.with_(layers=args.layers)
    stack = Stack(wl, dev)
    fn = {"gateup": stack.gateup_only, "down": stack.down_only,
          "executor": stack.step_executor}[args.only]
    if args.only == "executor" and stack.plan is None:
        raise SystemExit("the executor does not take this workload")
    for _ in range(max(3, args.warmup) + args.steps):
        fn()
    torch.cuda.synchronize()
    stack.close()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="mt", choices=["mt", "reference"])
    ap.add_argument("--workload", default="qwen3-8b",
                    choices=["qwen3-8b", "tiny", "llama1b", "qwen15", "sweep", "configs", "projections", "mx",
                             "prefill"],
                    help="sweep: every group x M point of the d=2048, f=8192 sweep, one line; "
                         "configs: the tiny, Llama-3.2-1B and Qwen2.5-1.5B layers hot and cold, one line; "
                         "projections: attention and vocabulary projections of a decode step per model")
    ap.add_argument("--rows", type=int, default=None,
                    help="projections / mx: rows M (1..8); prefill: one M instead of the list")
    ap.add_argument("--layers", type=int, default=None, help="override the layer count")
    ap.add_argument("--sweep-group", type=int, default=None, choices=[32, 64, 128],
                    help="sweep: only this group size")
    ap.add_argument("--sweep-rows", type=int, default=None, choices=[1, 2, 4, 8],
                    help="sweep: only this row count M")
    ap.add_argument("--path", default="executor", choices=["executor", "calls"],
                    help="timed step: the warmed executor (one kernel per step, default) or "
                         "three single-call kernels per layer")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-pdl", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the step's kernels directly instead of replaying a CUDA graph")
    ap.add_argument("--gemv", default="default", choices=["default", "team", "mma"],
                    help="single-call GEMV kernels: default (warp-task kernel for one row, "
                         "tensor-core kernel for M > 1), team kernel, or tensor-core kernel for every M")
    ap.add_argument("--only", default=None, choices=["gateup", "down", "executor"],
                    help="profiling aid: run only these kernels over the workload's layers "
                         "(no timing, no JSON line); sweep takes one point (--sweep-group, "
                         "--sweep-rows), mx one format (--mx) and --rows, projections one "
                         "model's vocabulary projection (--proj; --only takes any value there)")
    ap.add_argument("--mx", default="fp8", choices=["fp8", "fp4"],
                    help="mx with --only: the MX format")
    ap.add_argument("--proj", default="llama1b", choices=["qwen3-8b", "qwen15", "llama1b"],
                    help="projections with --only: the model whose vocabulary projection runs")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import synth
    import quantized_gemv_epilogues_gb300 as mt

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.no_pdl:
        mt.mt_set_option(mt.MT_OPT_PDL, 0)
    mt.mt_set_option(mt.MT_OPT_GEMV, {"default": 0, "team": 1, "mma": 2}[args.gemv])

    if args.only:
        return run_only(args, torch, synth, mt, dev)
    if args.workload == "sweep":
        return run_sweep(args, torch, synth, mt, dev)
    if args.workload == "configs":
        return run_configs(args, torch, synth, mt, dev)
    if args.workload == "projections":
        return run_projections(args, torch, synth, mt, dev)
    if args.workload == "mx":
        return run_mx(args, torch, synth, mt, dev)
    if args.workload == "prefill":
        return run_prefill(args, torch, synth, mt, dev)
    wl = {"qwen3-8b": synth.QWEN8B, "tiny": synth.TINY, "llama1b": synth.LLAMA1B,
          "qwen15": synth.QWEN15}[args.workload]
    if args.layers:
        wl = wl.with_(layers=args.layers)
    stack = Stack(wl, dev)
    use_exec = args.path == "executor" and stack.plan is not None

    step_fn = stack.step_executor if use_exec else stack.step_calls
    g_step = capture(step_fn, torch, direct=args.no_graph)
    for _ in range(max(3, args.warmup)):
        g_step.replay()
    torch.cuda.synchronize()

    # ---- timed region: K graph replays, each between its own CUDA events
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local, torch) as clk:
        total_ms, per_step = time_steps(g_step, args.steps, torch)
    torch.cuda.synchronize()
    ms = reduce_max(total_ms / args.steps, ws, torch, dev)
    step_bytes = wl.layer_bytes() * wl.layers
    value = ws * step_bytes / (ms * 1e-3) / 1e9
    us_layer = ms * 1e3 / wl.layers
    peak, peak_kind = measured_peaks()

    # ---- the single-call path, and each of its kernels alone over the layers
    per_kernel = {}
    kernel_reps = max(5, args.steps // 4)
    g_calls = g_step if not use_exec else capture(stack.step_calls, torch, direct=args.no_graph)
    for _ in range(3):
        g_calls.replay()
    calls_us = time_graph(g_calls, kernel_reps, torch) * 1e3 / wl.layers
    del g_calls
    for name, fn in (("gateup", stack.gateup_only), ("down", stack.down_only),
                     ("add_rmsnorm", stack.rmsnorm_only)):
        g_k = capture(fn, torch, direct=args.no_graph)
        for _ in range(3):
            g_k.replay()
        per_kernel[name] = time_graph(g_k, kernel_reps, torch) * 1e3 / wl.layers
        del g_k

    if use_exec:
        # the stack kernel is the whole step (plus a 128-byte memset node)
        roof = {"bound": "hbm", "kernel": f"mlp_stack_kernel ({wl.layers} layers, one row)",
                "achieved": round(step_bytes / (ms * 1e-3) / 1e9, 1), "peak": peak, "unit": "GB/s",
                "frac": round(step_bytes / (ms * 1e-3) / 1e9 / peak, 4), "peak_kind": peak_kind,
                "bytes_per_launch": step_bytes, "us_per_launch": round(ms * 1e3, 3),
                "traffic": profiled_traffic("stack")}
    else:
        gu_launch_s = per_kernel["gateup"] * 1e-6
        gu_bytes = stack.gateup_bytes()
        achieved = gu_bytes / gu_launch_s / 1e9
        roof = {"bound": "hbm",
                "kernel": {"default": "gemv_warp_kernel", "team": "gemv_kernel",
                           "mma": "gemv_mma_kernel"}[args.gemv]
                          + " gate/up+SwiGLU (one row)",
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                "bytes_per_launch": gu_bytes, "us_per_launch": round(gu_launch_s * 1e6, 3),
                "traffic": profiled_traffic("gateup")}

    # ---- end to end: pinned host inputs -> device, step, result -> host
    h_vals = stack.values.cpu().pin_memory()
    h_r0 = stack.r0.cpu().pin_memory()
    out_dev = stack.out_y if use_exec else stack.resid
    h_out = torch.empty_like(out_dev, device="cpu").pin_memory()

    def e2e_step():
        stack.values.copy_(h_vals, non_blocking=True)
        stack.r0.copy_(h_r0, non_blocking=True)
        g_step.replay()
        h_out.copy_(out_dev, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = reduce_max((time.perf_counter() - t0) / args.steps, ws, torch, dev)
    h2d = h_vals.numel() * 2 + h_r0.numel() * 2
    d2h = h_out.numel() * 2

    line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s",
            "us_per_layer": round(us_layer, 3), "frac_of_8TBs": round(value / ws / 8000.0, 4),
            "frac_of_measured_hbm": round(value / ws / peak, 4),
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "step_ms": step_stats(per_step),
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": {0: "bf16", 1: "u8", 2: "u4"}[wl.fmt] + "-weights/f32-acc",
            "data": "synthetic", "config": workload_config(wl),
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
            "l2": "inputs larger than L2: each step streams all layers' weights once "
                  f"({wl.layer_bytes() * wl.layers / 1e9:.2f} GB per step vs 129 MB L2)",
            "gpu_launches": (1 if use_exec else 3 * wl.layers) * args.steps,
            "device_error": mt.mt_device_error(),
            "roofline": roof,
            "calls_path": {"us_per_layer": round(calls_us, 3),
                           "gbs": round(wl.layer_bytes() / (calls_us * 1e-6) / 1e9, 1)},
            "kernels_us_per_layer": {k: round(v, 3) for k, v in per_kernel.items()},
            "down_gbs_alone": round(stack.down_bytes() / (per_kernel["down"] * 1e-6) / 1e9, 1),
            "gateup_gbs_alone": round(stack.gateup_bytes() / (per_kernel["gateup"] * 1e-6) / 1e9, 1),
            "e2e": {"value": round(ws * step_bytes / e2e_s / 1e9, 2), "unit": "GB/s",
                    "us_per_layer": round(e2e_s * 1e6 / wl.layers, 3),
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "clocks": clk.summary()}
    if use_exec:
        line["path"] = "warmed executor: mt_mlp_plan_run, one cooperative kernel per step"
    else:
        line["path"] = "single calls: mt_add_rmsnorm + mt_swiglu_gateup + mt_down_residual " \
                       "per layer" + (", no PDL" if args.no_pdl else ", PDL between kernels")
    line["graph"] = "direct launches" if isinstance(g_step, DirectLaunch) else "one CUDA graph per step"
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and wl.name == synth.QWEN8B.name:
        # one thread, then one process per host core (spawned: no CUDA state)
        us_cpu, reps = oracle_layer_timing(wl)
        lps, procs = oracle_pool_timing(wl)
        line["cpu_baseline"] = {"value": round(wl.layer_bytes() * lps / 1e9, 4), "unit": "GB/s",
                                "us_per_layer": round(1e6 / lps, 1), "cores": procs, "threads": procs,
                                "nproc": os.cpu_count(), "cpu_model": cpu_model(), "kind": "oracle",
                                "single_thread": {"value": round(wl.layer_bytes() / (us_cpu * 1e-6) / 1e9, 4),
                                                  "us_per_layer": round(us_cpu, 1), "passes": reps},
                                "sample": f"one {wl.d}x{wl.f} affine8 g128 layer of the same workload per "
                                          f"process, {procs} processes at once (one per host core) for "
                                          "3 rounds after one warm-up round; single-threaded binary64 C "
                                          "oracle; single_thread: one process alone"}
    stack.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
