#!/usr/bin/env python
"""Throughput of the anchor-attention forward H = A Delta^{-1} A^T V on GB300.

One step = one forward over the whole workload (every (batch, head) slice) through the C
ABI.  Prints ONE JSON line on rank 0: the headline workload (long_16k by default) and, timed
in the same run, every other workload ("workloads"), the backward of each ("backward"), the
masked variant ("causal"), the approximation-error diagnostic ("approx_error") and the block
front end with its projections ("block"); --only keeps the headline alone.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

N > 1 runs under torchrun, one rank per GPU; every rank runs the full workload on its own
GPU (slices are independent: weak scaling, no collective on the data path); the timed
region is bracketed by barriers and the max over ranks is reported.

--impl reference times the CPU oracle (plain C, double, one thread) on a bounded sample
of the same workload per step, on rank 0 only.

Timing: W untimed calls, then K calls bracketed by a barrier and a device synchronisation,
CUDA events around each call on the launching stream, input/output sets rotated so that
each step's working set is larger than L2.  Clocks and throttle reasons are sampled through
NVML (about every 0.5 ms) while the timed calls run.  A nonzero device error word after the
timed calls marks the line invalid.
"""
from __future__ import annotations

import argparse
import ctypes
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gen  # noqa: E402

METRIC = "anchor-attn tokens·heads/s at 1 GB300; achieved HBM GB/s vs peak"
UNIT = "tokens*heads/s"
DEFAULT_WORKLOAD = "long_16k"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_L2_BYTES = 126 * 1024 * 1024
FMA_LANES_PER_SM = 128          # fp32 FMA lanes per SM (4 sub-partitions x 32)
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
CSRC = os.path.join(ROOT, "linear_complexity_anchor_gb300", "csrc")
# the files whose code makes each kernel (a recorded ncu capture stays valid while they hold)
KERNEL_SOURCES = {"anchor_umma_kernel": ("umma.cu", "ptx.cuh", "common.cuh"),
                  "anchor_stream_kernel": ("stream.cu", "ptx.cuh", "rowops.cuh"),
                  "anchor_split_kernel": ("split.cu", "ptx.cuh", "rowops.cuh"),
                  "anchor_block_kernel": ("block.cu", "ptx.cuh", "rowops.cuh"),
                  "simt_full_kernel": ("simt.cu", "simt_ops.cuh"),
                  "simt_chunk_kernel": ("simt.cu", "simt_ops.cuh")}
KERNEL_OF_VARIANT = {"umma": "anchor_umma_kernel", "simt_split": "simt_chunk_kernel",
                     "simt_slice": "simt_full_kernel", "stream": "anchor_stream_kernel",
                     "split_tc": "anchor_split_kernel", "short_tc": "anchor_block_kernel"}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(gen.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU-baseline sample time")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch count (a smaller case for profiling)")
    ap.add_argument("--only", action="store_true", help="time the headline workload only (no sub-records)")
    return ap.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(values, device, world: int):
    """Element-wise max of per-rank floats (the timed region's length is the slowest rank's)."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def check_shapes(w: gen.Workload, hQ, hU, hV):
    """The C ABI takes pointers and sizes only: buffers that do not match the sizes passed
    would be read out of bounds, so a mismatch stops here."""
    want = (w.B, w.heads, w.n, w.d)
    if tuple(hQ.shape) != want or tuple(hV.shape) != want or tuple(hU.shape) != (w.heads, w.m, w.d):
        raise ValueError(f"{w.name}: inputs {tuple(hQ.shape)}, {tuple(hU.shape)}, {tuple(hV.shape)} do not match "
                         f"B={w.B} heads={w.heads} n={w.n} m={w.m} d={w.d}")


def kernel_source_hash(kernel: str) -> str:
    """Hash of a kernel's source files' code: line comments and spacing are left out, so that
    an edit to comments alone keeps a recorded ncu capture valid (the sources hold no string
    literal with "//" in it)."""
    h = hashlib.sha256()
    for p in (os.path.join(CSRC, f) for f in KERNEL_SOURCES.get(kernel, ())):
        if os.path.exists(p):
            with open(p) as f:
                for line in f:
                    code = line.split("//", 1)[0].split()
                    if code:
                        h.update(" ".join(code).encode() + b"\n")
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    kernel sources as they are now."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        e = t["entries"][f"{kernel}@{workload}"]
        if e.get("source_hash") != kernel_source_hash(kernel):
            return None
        return int(e["dram_bytes_per_launch"])
    except Exception:
        return None


class NvmlClockSampler:
    """SM clock and throttle reasons read through NVML (ctypes, no Python package needed)
    every ~0.5 ms on a background thread while the timed region runs."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, pci_bus_id: str):
        import threading
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.h)) != 0:
            count = ctypes.c_uint()
            # one visible device: it is the one being timed
            if (self.lib.nvmlDeviceGetCount_v2(ctypes.byref(count)) != 0 or count.value != 1 or
                    self.lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h)) != 0):
                raise RuntimeError(f"no NVML device at {pci_bus_id}")
        mx = ctypes.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
        self.max_mhz = float(mx.value)
        self.samples, self.reasons = [], 0
        self.stop_ev = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)
        self._reason_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def _run(self):
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_ev.is_set():
            if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0:
                self.samples.append(float(mhz.value))
            if self._reason_fn(self.h, ctypes.byref(rs)) == 0:
                self.reasons |= int(rs.value)
            time.sleep(0.0005)

    def start(self):
        self.thread.start()

    def stop(self) -> dict:
        self.stop_ev.set()
        self.thread.join(timeout=5)
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for b, n in self.REASONS.items() if self.reasons & b),
                "samples": len(self.samples), "source": "nvml"}


def clock_sampler(dev_index: int):
    try:
        import torch
        pr = torch.cuda.get_device_properties(dev_index)
        bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        return NvmlClockSampler(bus)
    except Exception:
        return ClockSampler(dev_index)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms during the timed region
    (the fallback where NVML cannot be loaded directly)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r for r in csv.reader(io.StringIO(self.file.read())) if len(r) >= 9]
        self.file.close()
        os.unlink(self.file.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def cpu_baseline(w: gen.Workload, x: dict, budget_s: float, threads: int = 1) -> dict:
    """The oracle as it stands (plain C, double, one thread per slice) on whole slices of the
    same inputs until the time budget is spent (at least one slice per thread).  threads > 1
    runs that many slices at once on a thread pool: the oracle is called through ctypes,
    which releases the GIL, so each call runs on its own host core."""
    import threading
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    oracle.build()
    U = gen.to_float64(x["U"], w.dtype)
    lock = threading.Lock()
    state = {"next": 0, "done": 0}
    t0 = time.perf_counter()

    def worker():
        while True:
            with lock:
                if time.perf_counter() - t0 >= budget_s and state["done"] > 0 or state["next"] >= w.slices:
                    return
                s = state["next"]
                state["next"] += 1
            b, h = divmod(s, w.heads)
            oracle.slice_forward(gen.to_float64(x["Q"][b, h], w.dtype), U[h], gen.to_float64(x["V"][b, h], w.dtype),
                                 w.scale)
            with lock:
                state["done"] += 1

    with ThreadPoolExecutor(max_workers=threads) as ex:
        for f in [ex.submit(worker) for _ in range(threads)]:
            f.result()
    el = time.perf_counter() - t0
    done = state["done"]
    return {"value": done * w.n / el, "unit": UNIT, "cores": threads, "kind": "oracle",
            "cpu": cpu_model(),
            "sample": f"{done} of {w.slices} slices (n={w.n}, m={w.m}, d={w.d}) in {el:.2f} s, "
                      f"C double-precision oracle, {'one slice per thread on ' + str(threads) + ' threads' if threads > 1 else 'single-threaded'}"}


def run_reference(args) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = gen.WORKLOADS[args.workload]
    U = gen.to_float64(gen.make_inputs(w.with_(B=1), seed=0)["U"], w.dtype)

    def step(i: int) -> None:
        b, h = divmod(i % w.slices, w.heads)
        s = gen.slice_inputs(w, b, h, seed=0)
        oracle.slice_forward(gen.to_float64(s["Q"], w.dtype), U[h], gen.to_float64(s["V"], w.dtype), w.scale)

    for i in range(args.warmup):
        step(i)
    el = 0.0
    for i in range(args.steps):
        t0 = time.perf_counter()
        step(args.warmup + i)
        el += time.perf_counter() - t0
    value = args.steps * w.n / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generator, value distributions of the workload)",
        "config": {"workload": w.name, "B": w.B, "heads": w.heads, "n": w.n, "m": w.m, "d": w.d,
                   "input_dtype": w.dtype, "step_sample": "one (batch, head) slice per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "cpu": cpu_model(),
                         "sample": f"one slice of {w.n} tokens per step, {args.steps} steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def l2_bytes(dev) -> int:
    import torch
    try:
        n = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0))
        return n if n > 0 else FALLBACK_L2_BYTES
    except Exception:
        return FALLBACK_L2_BYTES


def host_inputs(w: gen.Workload, seed: int) -> tuple:
    import torch
    x = gen.make_inputs(w, seed=seed)

    def host_tensor(a):
        t = torch.from_numpy(a if w.dtype == "f32" else a.view("int16"))
        return t if w.dtype == "f32" else t.view(torch.bfloat16)

    return x, tuple(host_tensor(x[k]).pin_memory() for k in "QUV")


def time_workload(pkg, w: gen.Workload, hQUV: tuple, K: int, W: int, dev, world: int, sample_clocks: bool):
    """W untimed calls, then K timed calls (CUDA events on the launching stream around each,
    and around all), with input/output sets rotated so that each step's working set exceeds
    L2.  Returns a dict of the timings (max over ranks), the device error word and clocks."""
    import torch
    import torch.distributed as dist
    tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    hQ, hU, hV = hQUV
    check_shapes(w, hQ, hU, hV)
    nsets = max(1, min(8, math.ceil(3 * l2_bytes(dev) / w.algorithmic_bytes)))
    sets = [{"Q": hQ.to(dev), "U": hU.to(dev), "V": hV.to(dev), "H": torch.empty(hQ.shape, dtype=tdt, device=dev)}
            for _ in range(nsets)]
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    fwd = pkg.anchor_attn_forward_f32_ptr if w.dtype == "f32" else pkg.anchor_attn_forward_ptr
    ptrs = [(st["Q"].data_ptr(), st["U"].data_ptr(), st["V"].data_ptr(), st["H"].data_ptr()) for st in sets]

    def call(st):
        pkg.forward(st["Q"], st["U"], st["V"], H=st["H"], scale=w.scale, stream=stream)

    def call_raw(i):  # the C ABI with the same pointers and stream, minus the Python tensor checks
        st_ = fwd(*ptrs[i % nsets], w.B, w.heads, w.n, w.m, w.d, w.scale, stream.cuda_stream)
        if st_ != 0:
            raise RuntimeError(f"anchor_attn call failed: {pkg.status_string(st_)}")

    for i in range(W):
        call(sets[i % nsets])
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = clock_sampler(torch.cuda.current_device()) if sample_clocks else None
    if clocks:
        clocks.start()
        time.sleep(0.01)
    # Queue the timed calls behind a short GPU sleep, so that the host enqueues them faster
    # than the GPU runs them: the events then time the GPU work back to back, not the host's
    # launch overhead (the sleep itself is before t_start).
    with torch.cuda.stream(stream):
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(int(2e6))  # about a millisecond of clock cycles
    # no event between the calls: an event recorded between two launches adds a few
    # microseconds of its own to each gap, so the calls are timed as one batch
    t_start.record(stream)
    for i in range(K):
        call_raw(i)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None
    if world > 1:
        dist.barrier()
    derr = pkg.device_error()
    elapsed_ms = t_start.elapsed_time(t_end)
    call_ms = elapsed_ms / K  # one launch per call: the average launch duration, gaps included
    elapsed_ms, call_ms, derr_max = max_over_ranks([elapsed_ms, call_ms, float(derr)], dev, world)
    return {"elapsed_ms": elapsed_ms, "call_ms": call_ms, "nsets": nsets, "sets": sets, "stream": stream,
            "call": call, "device_error": int(derr_max), "clocks": clk}


def batch_ms(stream, fn, k: int) -> float:
    """Average milliseconds of k calls of fn(i) queued back to back on `stream` behind a short
    GPU sleep (so that the host enqueues them faster than the GPU runs them), timed by two CUDA
    events around the whole batch (an event between two launches adds to the gap)."""
    import torch
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(int(2e6))
        t0.record(stream)
        for i in range(k):
            fn(i)
        t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / k


def time_backward(pkg, w: gen.Workload, hQUV: tuple, K: int, W: int, dev) -> dict:
    """The backward (dQ, dU, dV for an upstream gradient dH) of one workload, timed like the
    forward (CUDA events on the launching stream, W untimed calls first).  Algorithmic work per
    slice: 18 n m d flops (three contractions to recompute A and the summaries, six in the
    gradient pass) and 5 n d elements of traffic (Q, V, dH read, dQ and dV written; U read and
    dU written once per head).  bf16 with d = 64 or 128 and m <= 128 runs on the tensor cores
    (roofline: the measured bf16 peak, and HBM), the rest on CUDA cores (roofline: the fp32 FMA
    peak)."""
    import torch
    hQ, hU, hV = hQUV
    check_shapes(w, hQ, hU, hV)
    Q, U, V = hQ.to(dev), hU.to(dev), hV.to(dev)
    dH = torch.randn(Q.shape, device=dev, generator=torch.Generator(device=dev).manual_seed(1)).to(Q.dtype)
    dQ, dU, dV = torch.empty_like(Q), torch.empty_like(U), torch.empty_like(V)
    stream = torch.cuda.Stream(device=dev)
    fn = pkg.anchor_attn_backward_f32_ptr if w.dtype == "f32" else pkg.anchor_attn_backward_ptr
    ptrs = (Q.data_ptr(), U.data_ptr(), V.data_ptr(), dH.data_ptr(), dQ.data_ptr(), dU.data_ptr(), dV.data_ptr())

    def call():
        st = fn(*ptrs, w.B, w.heads, w.n, w.m, w.d, w.scale, stream.cuda_stream)
        if st != 0:
            raise RuntimeError(f"anchor_attn_backward failed: {pkg.status_string(st)}")

    torch.cuda.synchronize()
    for _ in range(W):
        call()
    torch.cuda.synchronize()
    call_ms = batch_ms(stream, lambda i: call(), K)
    derr = pkg.device_error()
    flops = 18 * w.slices * w.n * w.m * w.d
    hbm = (5 * w.slices * w.n * w.d + 2 * w.heads * w.m * w.d) * w.elem_bytes
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fma_peak = sms * FMA_LANES_PER_SM * 2 * 2070e6 / 1e12
    peak, peak_src = peaks()
    tensor = w.dtype == "bf16" and w.d in (64, 128) and w.m <= 128
    # the library's choice: four launches (two passes, the reduce, the dU sum) at d = 128 and at
    # d = 64 with m > 64; two (one CTA per slice, the dU sum) at d = 64 with m <= 64
    wide = tensor and (w.d == 128 or w.m > 64)
    rec = {"ms_per_call": call_ms, "value": w.slices * w.n / (call_ms / 1e3), "unit": UNIT, "steps": K,
           "kernels_per_call": 4 if wide else 2, "device_error": derr, "path": "tensor" if tensor else "cuda_core",
           "hbm": {"achieved": hbm / (call_ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                   "frac": hbm / (call_ms / 1e3) / 1e9 / peak, "algorithmic_bytes_per_call": hbm,
                   "peak_source": f"{peak_src} hbm_gbs"}}
    if tensor:
        tpeak, tsrc = bf16_peak()
        rec["tensor_roofline"] = {"bound": "tensor", "achieved": flops / (call_ms / 1e3) / 1e12, "peak": tpeak,
                                  "unit": "TFLOP/s", "frac": flops / (call_ms / 1e3) / 1e12 / tpeak,
                                  "peak_source": f"{tsrc} bf16_tflops (burst)", "flops_per_call": flops}
    else:
        rec["fma_roofline"] = {"bound": "alu", "achieved": flops / (call_ms / 1e3) / 1e12, "peak": fma_peak,
                               "unit": "TFLOP/s", "frac": flops / (call_ms / 1e3) / 1e12 / fma_peak,
                               "peak_source": f"{sms} SMs x {FMA_LANES_PER_SM} fp32 FMA lanes x 2 flop x 2070 MHz",
                               "flops_per_call": flops}
    if derr:
        rec["invalid"] = f"device error word {derr:#x} after the timed calls"
    return rec


def time_causal(pkg, w: gen.Workload, hQUV: tuple, K: int, W: int, dev) -> dict:
    """The masked (causal) variant of one workload, timed like the forward.  Algorithmic
    traffic as the forward's (Q, V and H once, U once), the roofline of the tensor-core path
    (bf16, d = 64 or 128, m <= 128); the CUDA-core path also reports its FMA rate, counting the work as
    the forward's 6 n m d."""
    import torch
    hQ, hU, hV = hQUV
    check_shapes(w, hQ, hU, hV)
    Q, U, V = hQ.to(dev), hU.to(dev), hV.to(dev)
    H = torch.empty_like(Q)
    stream = torch.cuda.Stream(device=dev)
    lib = pkg.load()
    fn = lib.anchor_attn_causal_forward_f32 if w.dtype == "f32" else lib.anchor_attn_causal_forward
    args = (Q.data_ptr(), U.data_ptr(), V.data_ptr(), H.data_ptr(), w.B, w.heads, w.n, w.m, w.d, float(w.scale))

    def call():
        st = fn(*args, stream.cuda_stream)
        if st != 0:
            raise RuntimeError(f"anchor_attn_causal_forward failed: {pkg.status_string(st)}")

    torch.cuda.synchronize()
    for _ in range(W):
        call()
    torch.cuda.synchronize()
    call_ms = batch_ms(stream, lambda i: call(), K)
    derr = pkg.device_error()
    peak, peak_src = peaks()
    # the tensor-core kernels: 64 anchors at d = 64, 128 anchors at d = 128 (and d = 64, m > 64)
    tensor = w.dtype == "bf16" and w.d in (64, 128) and w.m <= 128
    rec = {"ms_per_call": call_ms, "value": w.slices * w.n / (call_ms / 1e3), "unit": UNIT, "steps": K,
           "kernels_per_call": 1, "device_error": derr, "path": "tensor" if tensor else "cuda_core",
           "hbm": {"achieved": w.algorithmic_bytes / (call_ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                   "frac": w.algorithmic_bytes / (call_ms / 1e3) / 1e9 / peak,
                   "algorithmic_bytes_per_call": w.algorithmic_bytes, "peak_source": f"{peak_src} hbm_gbs"}}
    if not tensor:
        rec["fma_roofline"] = fma_roofline(w, call_ms, None, dev)
    if derr:
        rec["invalid"] = f"device error word {derr:#x} after the timed calls"
    return rec


def bf16_peak():
    """Dense bf16 tensor peak (TFLOP/s): the burst figure of MEASURED_PEAKS.json, for a kernel
    timed alone."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def time_block(pkg, bw: gen.BlockWorkload, K: int, W: int, dev) -> dict:
    """The block front end (projections + forward in one kernel) on one ViT block workload,
    timed like the forward (GPU sleep, CUDA events on the launching stream, two rotating
    input/output sets so that every call reads its X from HBM).  Its work is dominated by the
    projections (4 n dm d flops per slice against the forward's 6 n m d), so the roofline is
    the bf16 tensor peak.  For context, the same block unfused: one library GEMM for both
    projections, the head-major layout copy of Q and V, and anchor_attn_forward."""
    import numpy as np
    import torch
    w = bw.w
    x = gen.make_block_inputs(bw, seed=0)

    def dev_t(a):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

    base = {k: dev_t(v) for k, v in x.items()}
    sets = [base, {k: v.clone() for k, v in base.items()}]
    for st in sets:
        st["H"] = torch.empty((w.B, w.heads, w.n, w.d), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    lib = pkg.load()

    def call(i):
        st = sets[i % len(sets)]
        rc = lib.anchor_attn_block_forward(st["X"].data_ptr(), st["Wq"].data_ptr(), st["Wv"].data_ptr(),
                                           st["U"].data_ptr(), st["H"].data_ptr(), w.B, w.heads, w.n, w.m, w.d,
                                           bw.dm, float(w.scale), stream.cuda_stream)
        if rc != 0:
            raise RuntimeError(f"anchor_attn_block_forward failed: {pkg.status_string(rc)}")

    Wqv = torch.cat([base["Wq"].reshape(-1, bw.dm), base["Wv"].reshape(-1, bw.dm)], 0)
    hd = w.heads * w.d

    def unfused(i):
        st = sets[i % len(sets)]
        P = st["X"] @ Wqv.t()
        Q = P[..., :hd].reshape(w.B, w.n, w.heads, w.d).permute(0, 2, 1, 3).contiguous()
        V = P[..., hd:].reshape(w.B, w.n, w.heads, w.d).permute(0, 2, 1, 3).contiguous()
        pkg.forward(Q, st["U"], V, H=st["H"], scale=w.scale, stream=stream)

    def timed(fn, k):
        torch.cuda.synchronize()
        for i in range(W):
            with torch.cuda.stream(stream):
                fn(i)
        return batch_ms(stream, fn, k)

    call_ms = timed(call, K)
    derr = pkg.device_error()
    unfused_ms = timed(unfused, min(K, 10))
    tpeak, tsrc = bf16_peak()
    hpeak, hsrc = peaks()
    tflops = bw.flops / (call_ms / 1e3) / 1e12
    rec = {"ms_per_call": call_ms, "value": w.slices * w.n / (call_ms / 1e3), "unit": UNIT, "steps": K,
           "kernels_per_call": 1, "device_error": derr,
           "config": {"B": w.B, "heads": w.heads, "n": w.n, "m": w.m, "d": w.d, "dm": bw.dm},
           "roofline": {"bound": "tensor", "achieved": tflops, "peak": tpeak, "unit": "TFLOP/s",
                        "frac": tflops / tpeak, "kernel": "anchor_block_kernel",
                        "flops_per_launch": bw.flops, "peak_source": f"{tsrc} bf16_tflops (burst)"},
           "hbm": {"achieved": bw.algorithmic_bytes / (call_ms / 1e3) / 1e9, "peak": hpeak, "unit": "GB/s",
                   "frac": bw.algorithmic_bytes / (call_ms / 1e3) / 1e9 / hpeak,
                   "algorithmic_bytes_per_call": bw.algorithmic_bytes},
           "unfused_ms_per_call": unfused_ms,
           "unfused": "torch GEMM of X with [Wq; Wv], head-major copies of Q and V, anchor_attn_forward"}
    if derr:
        rec["invalid"] = f"device error word {derr:#x} after the timed calls"
    return rec


def approx_error(pkg, w: gen.Workload, dev, K: int) -> dict:
    """The approximation-error diagnostic on a workload whose anchors are rows of the keys:
    ||H_full - H_anchor||_F / ||H_full||_F per slice (mean and max), with the time of the
    full-attention reference and of the anchor forward on the same inputs."""
    import torch
    x = gen.make_inputs(w, seed=0)
    x["K"] = gen.make_keys(w, seed=0)

    def dev_t(a):
        t = torch.from_numpy(a if w.dtype == "f32" else a.view("int16"))
        return (t if w.dtype == "f32" else t.view(torch.bfloat16)).to(dev)

    t = {k: dev_t(x[k]) for k in "QUVK"}
    Hf, Ha = torch.empty_like(t["Q"]), torch.empty_like(t["Q"])

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(K):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / K

    ms_full = timed(lambda: pkg.full_forward(t["Q"], t["K"], t["V"], H=Hf, scale=w.scale))
    ms_anchor = timed(lambda: pkg.forward(t["Q"], t["U"], t["V"], H=Ha, scale=w.scale))
    err = pkg.relative_error(Hf, Ha).double().cpu()
    return {"workload": w.name, "rel_frobenius_mean": float(err.mean()), "rel_frobenius_max": float(err.max()),
            "slices": w.slices, "full_attention_ms": ms_full, "anchor_ms": ms_anchor,
            "note": "anchors are rows of the keys plus N(0, 0.1^2) noise; full attention is the CUDA-core "
                    "reference of the diagnostic, not a tuned attention"}


def roofline(w: gen.Workload, plan: dict, call_ms: float) -> dict:
    peak, peak_src = peaks()
    achieved = w.algorithmic_bytes / (call_ms / 1e3) / 1e9
    kernel = KERNEL_OF_VARIANT.get(plan["variant"], plan["variant"])
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": recorded_traffic(w.name, kernel), "peak_source": f"{peak_src} hbm_gbs", "kernel": kernel,
            "algorithmic_bytes_per_launch": w.algorithmic_bytes, "call_ms": call_ms,
            "kernels_per_call": plan["kernels_per_call"]}


def fma_roofline(w: gen.Workload, call_ms: float, sm_mhz, dev) -> dict:
    """The CUDA-core variants against the fp32 FMA peak: 2 flops per FMA lane per clock."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = float(sm_mhz) if sm_mhz else 2070.0
    peak = sms * FMA_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
    achieved = w.flops / (call_ms / 1e3) / 1e12
    return {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "peak_source": f"{sms} SMs x {FMA_LANES_PER_SM} fp32 FMA lanes x 2 flop x {mhz:.0f} MHz",
            "flops_per_launch": w.flops}


def run_ours(args) -> None:
    import torch
    import torch.distributed as dist
    import linear_complexity_anchor_gb300 as pkg

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkg.load()
    if pkg.device_error() != 0:
        raise RuntimeError("device error word set before the bench started")
    w = gen.WORKLOADS[args.workload]
    if args.batch is not None:
        w = w.with_(B=args.batch)
    plan = pkg.query_plan(w.dtype, w.B, w.heads, w.n, w.m, w.d)
    x, hQUV = host_inputs(w, seed=rank)
    K = args.steps
    t = time_workload(pkg, w, hQUV, K, args.warmup, dev, world, sample_clocks=True)
    units = world * w.slices * w.n * K
    value = units / (t["elapsed_ms"] / 1e3)

    # end to end through the C ABI with host buffers (anchor_attn_forward_host): every step
    # copies the pinned inputs to the device and H back, chunk by chunk, overlapped with the
    # forward of the neighbouring chunks
    hQ, hU, hV = hQUV
    tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    E = max(1, args.e2e_steps)
    hH = torch.empty(hQ.shape, dtype=tdt).pin_memory()
    stream = t["stream"]
    host_fn = pkg.anchor_attn_forward_host_f32_ptr if w.dtype == "f32" else pkg.anchor_attn_forward_host_ptr
    hptrs = (hQ.data_ptr(), hU.data_ptr(), hV.data_ptr(), hH.data_ptr())

    def host_call():
        st_ = host_fn(*hptrs, w.B, w.heads, w.n, w.m, w.d, w.scale, stream.cuda_stream)
        if st_ != 0:
            raise RuntimeError(f"anchor_attn_forward_host failed: {pkg.status_string(st_)}")

    host_call()  # warm-up: the library's copy streams and events are made on the first call
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(E):
        host_call()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_err = pkg.device_error()
    e2e_ms = e0.elapsed_time(e1)
    (e2e_ms,) = max_over_ranks([e2e_ms], dev, world)
    e2e_value = world * w.slices * w.n * E / (e2e_ms / 1e3)
    elem = 4 if w.dtype == "f32" else 2
    h2d = (hQ.numel() + hU.numel() + hV.numel()) * elem
    d2h = hH.numel() * elem
    del t["sets"]
    torch.cuda.empty_cache()

    # every other workload, timed the same way in the same run
    subs = {}
    if not args.only:
        for name in sorted(gen.WORKLOADS):
            if name == w.name:
                continue
            ws = gen.WORKLOADS[name]
            wplan = pkg.query_plan(ws.dtype, ws.B, ws.heads, ws.n, ws.m, ws.d)
            _, hq = host_inputs(ws, seed=rank)
            ts = time_workload(pkg, ws, hq, K, args.warmup, dev, world, sample_clocks=True)
            rec = {"ms_per_step": ts["elapsed_ms"] / K,
                   "value": world * ws.slices * ws.n * K / (ts["elapsed_ms"] / 1e3), "unit": UNIT,
                   "dtype": ws.dtype, "variant": wplan["variant"],
                   "config": {"B": ws.B, "heads": ws.heads, "n": ws.n, "m": ws.m, "d": ws.d},
                   "l2": f"{ws.algorithmic_bytes / 1e6:.1f} MB per step, {ts['nsets']} rotating set(s)",
                   "roofline": roofline(ws, wplan, ts["call_ms"]), "device_error": ts["device_error"],
                   "clocks": ts["clocks"]}
            if wplan["variant"].startswith("simt"):
                rec["fma_roofline"] = fma_roofline(ws, ts["call_ms"], (ts["clocks"] or {}).get("sm_mhz"), dev)
            if ts["device_error"]:
                rec["invalid"] = f"device error word {ts['device_error']:#x} after the timed calls"
            subs[name] = rec
            del ts
            torch.cuda.empty_cache()

    # the backward of every workload (fewer steps)
    bwd = {}
    if not args.only and world == 1:
        for name in sorted(gen.WORKLOADS):
            ws = gen.WORKLOADS[name] if name != w.name else w  # the headline's own (--batch) shape
            _, hq = host_inputs(ws, seed=rank) if name != w.name else (None, hQUV)
            bwd[name] = time_backward(pkg, ws, hq, min(K, 10), min(args.warmup, 3), dev)
            torch.cuda.empty_cache()

    diag = approx_error(pkg, gen.WORKLOADS["deit_base"], dev, min(K, 10)) if not args.only and world == 1 else None
    causal = {}
    if not args.only and world == 1:
        for name in sorted(gen.WORKLOADS):
            ws = gen.WORKLOADS[name] if name != w.name else w  # the headline's own (--batch) shape
            _, hq = host_inputs(ws, seed=rank) if name != w.name else (None, hQUV)
            causal[name] = time_causal(pkg, ws, hq, min(K, 10), min(args.warmup, 3), dev)
            torch.cuda.empty_cache()

    block = {}
    if not args.only and world == 1:
        for name in sorted(gen.BLOCK_WORKLOADS):
            block[name] = time_block(pkg, gen.BLOCK_WORKLOADS[name], K, min(args.warmup, 3), dev)
            torch.cuda.empty_cache()

    cpu = cpu_par = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, x, args.cpu_seconds)
        cpu_par = cpu_baseline(w, x, max(4.0, args.cpu_seconds / 2), threads=os.cpu_count() or 1)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": t["elapsed_ms"] / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded counter-based generator; value distributions of the workload)",
            "config": {"workload": w.name, "B": w.B, "heads": w.heads, "n": w.n, "m": w.m, "d": w.d,
                       "scale": w.scale, "variant": plan["variant"],
                       "l2": (f"inputs larger than L2: {w.algorithmic_bytes / 1e6:.0f} MB per step, "
                              f"{t['nsets']} rotating input/output set(s)")},
            "roofline": roofline(w, plan, t["call_ms"]),
            "cpu_baseline": cpu,
            "cpu_baseline_parallel": cpu_par,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": E},
            "gpu_launches": plan["kernels_per_call"] * K,
            "clocks": t["clocks"],
            "device_error": t["device_error"],
            "workloads": subs,
            "backward": bwd,
            "approx_error": diag,
            "causal": causal,
            "block": block,
        }
        if t["device_error"] or e2e_err:
            line["invalid"] = f"device error word {t['device_error'] | e2e_err:#x} after the timed calls"
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
