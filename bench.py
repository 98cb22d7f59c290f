"""Benchmark: simulated ring AllReduce on one GB300.

Workload (the configuration the headline is quoted on): 8 ranks x 67,108,864
bf16 elements (128 MiB per rank, 2 GiB moved per step), values normal(0, 1)
with 1% of entries scaled by 100, ring order, SUM.  A step is one
``ar_allreduce`` call through the C ABI (one fused kernel launch).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  ``value`` is effective HBM GB/s (2*N*D*b bytes per
step / time, summed over replicas for N GPUs; each GPU runs an independent
replica, there is no cross-GPU data path).  ``--impl reference`` times the CPU
oracle on this host's cores on a bounded sample of the same workload.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "simulated-AllReduce algbw & effective HBM GB/s (frac of GB300 peak), 1 GPU"
WORKLOAD = "ring AllReduce SUM, 8 ranks x 67,108,864 bf16 (128 MiB per rank)"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ("ar_fused.cuh", "ar_device.cuh", "ar_fused_bf16_sum.cu")
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "fused_ring_bf16_8x128MiB.md")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--algo", default="ring", help="ring | tree | ring_stepwise | tree_stepwise")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg (profiling runs)")
    p.add_argument("--count", type=int, default=0,
                   help="elements per rank (default: the full workload); smaller counts are for profiling")
    p.add_argument("--variants", action="store_true", help="also time tree and step-wise orders (extra keys)")
    return p.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only; timing reduction)
# ---------------------------------------------------------------------------

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl"
        import torch
        if not torch.cuda.is_available():
            backend = "gloo"
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []  # (t, sm, sm_max, reasons)
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, smax = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            reasons = []
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                               parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.append(name)
            self.samples.append((time.time(), sm, smax, reasons))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        sel = [s for s in self.samples if t0 - 0.15 <= s[0] <= t1 + 0.15]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({r for s in sel for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in sel), "sm_max_mhz": max(s[2] for s in sel),
                "reasons": reasons, "samples": len(sel)}


# ---------------------------------------------------------------------------
# roofline inputs
# ---------------------------------------------------------------------------

def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "allreduce_gradient_reduction_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the kernel source as it is now."""
    try:
        text = open(PROFILE_SUMMARY, encoding="utf-8").read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash():
        return None
    return int(m_bytes.group(1))


# ---------------------------------------------------------------------------
# the CPU oracle as the baseline
# ---------------------------------------------------------------------------

def oracle_sample_time(n: int, count: int, steps: int = 1):
    """Time the oracle's ring AllReduce (single thread) on n x count bf16 of
    the same input recipe.  Returns (seconds per pass, GB/s in the metric)."""
    import oracle
    from allreduce_gradient_reduction_gb300 import workloads as W
    oracle.build()
    x = W.large_inputs(n, count)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.allreduce(x, algo="ring", op="sum", dtype="bf16")
    dt = (time.perf_counter() - t0) / steps
    return dt, 2 * n * count * 2 / dt / 1e9


def run_reference(args, ws, rank):
    """Reference arm: the CPU oracle, as it stands, on this host's cores."""
    if rank != 0:
        return 0
    from allreduce_gradient_reduction_gb300 import workloads as W
    n = W.LARGE["nranks"]
    sample = 1 << 21  # elements per rank per step: a bounded slice of the workload
    import oracle
    oracle.build()
    x = W.large_inputs(n, sample)
    for _ in range(args.warmup):
        oracle.allreduce(x, algo="ring", op="sum", dtype="bf16")
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.allreduce(x, algo="ring", op="sum", dtype="bf16")
    dt = (time.perf_counter() - t0) / args.steps
    value = 2 * n * sample * 2 / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "nranks": n, "count_per_rank": W.LARGE["count"],
                   "sample_count_per_rank": sample, "algo": "ring", "op": "sum"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n} ranks x {sample} bf16 per step (1/{W.LARGE['count'] // sample} of the "
                                   "workload), literal message simulation, one thread"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def main():
    args = parse()
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        rc = run_reference(args, ws, rank)
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return rc

    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from allreduce_gradient_reduction_gb300 import binding as ar
    from allreduce_gradient_reduction_gb300 import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    n, count = W.LARGE["nranks"], (args.count or W.LARGE["count"])
    nbytes_step = 2 * n * count * 2  # every rank element read once, the result written once per rank

    # inputs: generated on the host (seeded), pinned, uploaded once
    host = torch.empty((n, count), dtype=torch.int16, pin_memory=True)
    for r in range(n):
        host[r].copy_(torch.from_numpy(W.large_rank(r, count).view(np.int16)))
    bufs = [torch.empty(count, dtype=torch.int16, device=dev) for _ in range(n)]
    for r in range(n):
        bufs[r].copy_(host[r], non_blocking=True)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    sid = int(stream.cuda_stream)

    def step(algo=args.algo):
        rc = ar.ar_allreduce(bufs, count=count, dtype="bf16", op="sum", algo=algo, stream=sid)
        if rc:
            raise ar.ArError(rc, "ar_allreduce")

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(ws)
    ms_local = e0.elapsed_time(e1) / args.steps
    clocks.stop()
    ms = max_over_ranks(ms_local, ws)
    rc, status = ar.ar_device_status(sid)
    if rc or status:
        raise ar.ArError(rc or status, "device status")

    value = ws * nbytes_step / (ms / 1e3) / 1e9
    algbw = count * 2 / (ms / 1e3) / 1e9
    peak, peak_kind = hbm_peak()
    achieved = nbytes_step / (ms_local / 1e3) / 1e9

    # end to end through the public call: pinned host -> device, AllReduce, device -> host
    e2e = None
    if not args.no_e2e:
        e2e_steps = max(3, min(args.steps, 20))
        out_host = torch.empty((n, count), dtype=torch.int16, pin_memory=True)
        for r in range(n):  # warm the copy path once
            bufs[r].copy_(host[r], non_blocking=True)
        step()
        for r in range(n):
            out_host[r].copy_(bufs[r], non_blocking=True)
        torch.cuda.synchronize()
        barrier(ws)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(e2e_steps):
            for r in range(n):
                bufs[r].copy_(host[r], non_blocking=True)
            step()
            for r in range(n):
                out_host[r].copy_(bufs[r], non_blocking=True)
        f1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        ms_e2e = max_over_ranks(f0.elapsed_time(f1) / e2e_steps, ws)
        e2e = {"value": ws * nbytes_step / (ms_e2e / 1e3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": n * count * 2, "d2h_bytes_per_step": n * count * 2, "steps": e2e_steps,
               "ms_per_step": ms_e2e, "result_ranks_identical": bool(torch.equal(out_host[0], out_host[n - 1]))}

    variants = {}
    if args.variants:
        for algo in ("tree", "ring_stepwise", "tree_stepwise"):
            for _ in range(3):
                step(algo)
            torch.cuda.synchronize()
            v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            k = max(10, args.steps // 10)
            v0.record(stream)
            for _ in range(k):
                step(algo)
            v1.record(stream)
            torch.cuda.synchronize()
            vms = v0.elapsed_time(v1) / k
            variants[algo] = {"ms_per_step": vms, "effective_gbs": nbytes_step / (vms / 1e3) / 1e9}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        sample = count // 4
        dt, gbs = oracle_sample_time(n, sample)
        cpu = {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} ranks x {sample} bf16 (1/4 of the workload), one literal ring pass, "
                         f"{dt:.2f} s, one thread"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "nranks": n, "count_per_rank": count, "algo": args.algo,
                       "op": "sum", "l2": "inputs larger than L2 (2 GiB touched per step vs 129 MB L2)",
                       "parallelism": "replicas" if ws > 1 else "single GPU"},
            "algbw_gbs": algbw * ws,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind, "traffic": profiled_traffic(),
                         "algorithmic_bytes_per_launch": nbytes_step},
            "e2e": e2e,
            "gpu_launches": args.steps,
            "clocks": clocks.summary(t_wall0, t_wall1),
            "cpu_baseline": cpu,
        }
        if variants:
            line["variants"] = variants
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
