#!/usr/bin/env python
"""Throughput of the anchor-attention forward H = A Delta^{-1} A^T V on GB300.

One step = one forward over the whole workload (every (batch, head) slice) through the C
ABI.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

N > 1 runs under torchrun, one rank per GPU; every rank runs the full workload on its own
GPU (slices are independent: weak scaling, no collective on the data path); the timed
region is bracketed by barriers and the max over ranks is reported.

--impl reference times the CPU oracle (plain C, double, one thread) on a bounded sample
of the same workload per step, on rank 0 only.
"""
from __future__ import annotations

import argparse
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
L2_BYTES = 129 * 1024 * 1024
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
KERNEL_SOURCES = [os.path.join(ROOT, "linear_complexity_anchor_gb300", "csrc", f)
                  for f in ("umma.cu", "simt.cu", "api.cu", "common.cuh", "ptx.cuh")]


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


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code: line comments and spacing are left out, so that an
    edit to comments alone keeps a recorded ncu capture valid (the sources hold no string
    literal with "//" in it)."""
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
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
        if e.get("source_hash") != kernel_source_hash():
            return None
        return int(e["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms during the timed region."""
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
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline(w: gen.Workload, x: dict, budget_s: float) -> dict:
    """The oracle as it stands (one thread, double) on whole slices of the same inputs until
    the time budget is spent (at least one slice)."""
    import oracle
    oracle.build()
    U = gen.to_float64(x["U"], w.dtype)
    done, t0 = 0, time.perf_counter()
    while True:
        b, h = divmod(done % w.slices, w.heads)
        oracle.slice_forward(gen.to_float64(x["Q"][b, h], w.dtype), U[h], gen.to_float64(x["V"][b, h], w.dtype),
                             w.scale)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or done >= w.slices:
            break
    return {"value": done * w.n / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{done} of {w.slices} slices (n={w.n}, m={w.m}, d={w.d}) in {el:.2f} s, "
                      f"single-threaded C double-precision oracle"}


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
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"one slice of {w.n} tokens per step, {args.steps} steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


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
    w = gen.WORKLOADS[args.workload]
    if args.batch is not None:
        w = w.with_(B=args.batch)
    tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    plan = pkg.query_plan(w.dtype, w.B, w.heads, w.n, w.m, w.d)

    x = gen.make_inputs(w, seed=rank)

    def host_tensor(a):
        t = torch.from_numpy(a if w.dtype == "f32" else a.view("int16"))
        return t if w.dtype == "f32" else t.view(torch.bfloat16)

    hQ, hU, hV = (host_tensor(x[k]).pin_memory() for k in "QUV")
    step_bytes = w.algorithmic_bytes
    nsets = max(1, min(8, math.ceil(3 * L2_BYTES / step_bytes)))
    sets = []
    for _ in range(nsets):
        sets.append({"Q": hQ.to(dev), "U": hU.to(dev), "V": hV.to(dev),
                     "H": torch.empty(hQ.shape, dtype=tdt, device=dev)})
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    def call(s):
        pkg.forward(s["Q"], s["U"], s["V"], H=s["H"], scale=w.scale, stream=stream)

    for i in range(args.warmup):
        call(sets[i % nsets])
    torch.cuda.synchronize()

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.15)
    t_start.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        call(sets[i % nsets])
        ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    call_ms = sum(a.elapsed_time(b) for a, b in ev) / K
    elapsed_ms, call_ms = max_over_ranks([elapsed_ms, call_ms], dev, world)

    units = world * w.slices * w.n * K
    value = units / (elapsed_ms / 1e3)

    # end to end through the public API: pinned host inputs -> device, forward, H -> host
    E = max(1, args.e2e_steps)
    hH = torch.empty(hQ.shape, dtype=tdt).pin_memory()
    s0 = sets[0]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(E):
        with torch.cuda.stream(stream):
            s0["Q"].copy_(hQ, non_blocking=True)
            s0["U"].copy_(hU, non_blocking=True)
            s0["V"].copy_(hV, non_blocking=True)
            call(s0)
            hH.copy_(s0["H"], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    (e2e_ms,) = max_over_ranks([e2e_ms], dev, world)
    e2e_value = world * w.slices * w.n * E / (e2e_ms / 1e3)
    elem = 4 if w.dtype == "f32" else 2
    h2d = (hQ.numel() + hU.numel() + hV.numel()) * elem
    d2h = hH.numel() * elem

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, x, args.cpu_seconds)

    if rank == 0:
        peak, peak_src = peaks()
        achieved = w.algorithmic_bytes / (call_ms / 1e3) / 1e9
        kernel = {"umma": "anchor_umma_kernel", "simt_split": "simt_partial_kernel",
                  "simt_slice": "simt_slice_kernel"}.get(plan["variant"], plan["variant"])
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded counter-based generator; value distributions of the workload)",
            "config": {"workload": w.name, "B": w.B, "heads": w.heads, "n": w.n, "m": w.m, "d": w.d,
                       "scale": w.scale, "variant": plan["variant"],
                       "l2": (f"inputs larger than L2: {step_bytes / 1e6:.0f} MB per step, "
                              f"{nsets} rotating input/output set(s)")},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": recorded_traffic(w.name, kernel),
                         "peak_source": f"{peak_src} hbm_gbs", "kernel": kernel,
                         "algorithmic_bytes_per_launch": w.algorithmic_bytes,
                         "call_ms": call_ms, "kernels_per_call": plan["kernels_per_call"]},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": E},
            "gpu_launches": plan["kernels_per_call"] * K,
            "clocks": clk,
        }
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
