"""Benchmark: simulated ring AllReduce on one GB300.

Workload (the configuration the headline is quoted on): 8 ranks x 67,108,864
bf16 elements (128 MiB per rank, 2 GiB moved per step), values normal(0, 1)
with 1% of entries scaled by 100, ring order, SUM.  A step is one
``ar_allreduce`` call through the C ABI (one fused kernel launch).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  ``value`` is effective HBM GB/s (2*N*D*b bytes per
step / time, summed over replicas for N GPUs; each GPU runs an independent
replica, there is no cross-GPU data path).  ``e2e`` is the same metric for
``ar_allreduce_host`` on page-locked host buffers (every step's inputs come
from host memory and its result goes back there).  ``--impl reference`` times
the CPU oracle on this host's cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
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
# DRAM bytes per launch of the headline kernel from one ncu capture, with the
# hash of the kernel sources it was taken on (machine-readable; the summary
# beside it gives the command)
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "headline_traffic.json")

def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)  # about 0.6 s timed: several clock samples
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--algo", default="ring", help="ring | tree | ring_stepwise | tree_stepwise")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-procs", type=int, default=0,
                   help="processes for the CPU oracle baseline (default: every host core)")
    p.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg (profiling runs)")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip timing the small, bucket and GPT-2 configurations beside the headline")
    p.add_argument("--rank-offsets", choices=["aligned", "mixed"], default="aligned",
                   help="large and bucket workloads: 'mixed' starts rank r's buffer (3r+1) mod (16/element size) "
                        "elements into its allocation, so the ranks sit at different addresses modulo 16")
    p.add_argument("--count", type=int, default=0,
                   help="elements per rank (default: the full workload); smaller counts are for profiling")
    p.add_argument("--nranks", type=int, default=0,
                   help="ranks of the large workload (default: 8); other counts are for profiling")
    p.add_argument("--variants", action="store_true", help="also time tree and step-wise orders (extra keys)")
    p.add_argument("--workload", choices=["large", "bucket", "gpt2"], default="large",
                   help="large: the headline (default); bucket: 8 x 25 MiB f32 AVG; gpt2: DDP buckets of GPT-2 small")
    p.add_argument("--sweep", action="store_true",
                   help="latency/bandwidth sweep (sizes x ranks x dtypes x ops x orders); points go to --sweep-out")
    p.add_argument("--sweep-out", default="sweep.jsonl")
    p.add_argument("--sweep-ranks", default="2,4,8,16,64")
    p.add_argument("--overlap", action="store_true",
                   help="gpt2 workload: also time a synthetic backward with and without overlapped bucket reduction")
    p.add_argument("--overlap-tokens", type=int, default=256)
    p.add_argument("--overlap-eager", action="store_true",
                   help="time the overlap variants with direct launches instead of CUDA-graph replays")
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
    """DRAM bytes per launch from the committed ncu capture, if it was taken
    on the kernel source as it is now."""
    try:
        with open(TRAFFIC_FILE, encoding="utf-8") as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    v = rec.get("dram_bytes_per_launch")
    return int(v) if isinstance(v, int) else None


# ---------------------------------------------------------------------------
# the CPU oracle as the baseline
# ---------------------------------------------------------------------------

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the
    machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=20).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def oracle_pass_time(x, procs: int, passes: int, gpu_result=None):
    """Time the oracle's ring AllReduce over the bf16 bit patterns x (n x count)
    on `procs` processes (each holding one element range): one untimed pass,
    then `passes` timed ones.  Returns (seconds per pass, GB/s in the metric,
    median GB/s of one process on its own range, parity) -- parity compares
    the oracle's result with `gpu_result` (rank 0's result of the same inputs
    on the GPU, or None) range by range."""
    import oracle
    from oracle import parallel as oracle_parallel
    oracle.build()
    n, count = x.shape
    parity = None
    with oracle_parallel.Pool(procs) as pool:
        widths = pool.load(x, algo="ring", op="sum", dtype="bf16")
        pool.run()
        total, per = 0.0, [0.0] * procs
        for _ in range(passes):
            dt, p = pool.run()
            total += dt
            per = [a + b for a, b in zip(per, p)]
        if gpu_result is not None:
            parity = pool.compare(gpu_result)
            parity.pop("differing_ranges", None)
    per_gbs = sorted(2 * n * w * 2 * passes / max(t, 1e-9) / 1e9 for w, t in zip(widths, per))
    dt = total / passes
    return dt, 2 * n * count * 2 / dt / 1e9, per_gbs[len(per_gbs) // 2], parity


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
    procs = args.cpu_procs or host_cores()
    from oracle import parallel as oracle_parallel
    with oracle_parallel.Pool(procs) as pool:
        pool.load(x, algo="ring", op="sum", dtype="bf16")
        for _ in range(args.warmup):
            pool.run()
        total = 0.0
        for _ in range(args.steps):
            total += pool.run()[0]
    dt = total / max(args.steps, 1)
    value = 2 * n * sample * 2 / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "nranks": n, "count_per_rank": W.LARGE["count"],
                   "sample_count_per_rank": sample, "algo": "ring", "op": "sum"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": procs, "kind": "oracle", "cpu_model": cpu_model(),
                         "sample": f"{n} ranks x {sample} bf16 per step (1/{W.LARGE['count'] // sample} of the "
                                   f"workload), literal message simulation, element ranges split over {procs} "
                                   "processes"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# latency / bandwidth sweep
# ---------------------------------------------------------------------------

def fit_alpha_beta(points, phases, bw_factor):
    """Least-squares fit of t = A + B * D over (D bytes per rank, t seconds),
    relative error weighting; returns alpha = A / phases (seconds per step)
    and beta = B / bw_factor (seconds per byte), the page's alpha-beta model
    T = phases * alpha + bw_factor * D * beta."""
    import numpy as np
    d = np.array([p[0] for p in points], dtype=np.float64)
    t = np.array([p[1] for p in points], dtype=np.float64)
    w = 1.0 / t
    A = np.stack([np.ones_like(d), d], axis=1) * w[:, None]
    (a, b), *_ = np.linalg.lstsq(A, t * w, rcond=None)
    return a / phases, b / bw_factor


def graph_time(call, torch, stream, reps=20):
    """Per-call device time of `call` replayed from a CUDA graph, or None if
    the call cannot be captured."""
    try:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for _ in range(reps):
                if call(int(side.cuda_stream)):
                    raise RuntimeError("call failed during capture")
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(5):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (5 * reps)
    except Exception:
        torch.cuda.synchronize()
        return None


def run_sweep(args, ws, rank, dev, torch, ar):
    """Per-rank message 4 KiB .. 1 GiB x N in --sweep-ranks (N x size <= 64 GiB)
    x {f32, bf16} x {SUM, MAX} x {ring, tree, ring_stepwise, tree_stepwise,
    binomial_stepwise}, uniform(-1, 1) values.  Writes one JSON line per point
    to --sweep-out and prints one summary line: the alpha-beta fit of every
    order per (N, dtype), and the ring/tree crossover measured between the
    step-wise ring and the step-wise binomial (and halving/doubling) trees,
    beside where the pages' alpha-beta model puts it."""
    import math
    from allreduce_gradient_reduction_gb300 import workloads as W
    stream = torch.cuda.current_stream()
    sid = int(stream.cuda_stream)
    ranks = [int(x) for x in args.sweep_ranks.split(",")]
    gen = torch.Generator(device=dev)
    gen.manual_seed(W.BASE_SEED + 1000 * W.CONFIG_SWEEP)
    fits, crossover, npoints = {}, {}, 0
    with open(args.sweep_out, "w") as out:
        for n in ranks:
            max_bytes = min(W.SWEEP_BYTES[-1], W.SWEEP_CAP_BYTES // n)
            bufs = [torch.empty(max_bytes, dtype=torch.uint8, device=dev) for _ in range(n)]
            for dt in ("f32", "bf16"):
                es = 4 if dt == "f32" else 2
                tdt = torch.float32 if dt == "f32" else torch.bfloat16
                for b in bufs:
                    b.view(tdt).uniform_(-1.0, 1.0, generator=gen)
                curves = {}
                for op in ("sum", "max"):
                    for algo in ("ring", "tree", "ring_stepwise", "tree_stepwise", "binomial_stepwise"):
                        if (algo.startswith("tree") or algo.startswith("binomial")) and n & (n - 1):
                            continue
                        for nbytes in W.SWEEP_BYTES:
                            if nbytes > max_bytes:
                                break
                            count = nbytes // es
                            views = [b[:nbytes] for b in bufs]
                            call = lambda s=None: ar.ar_allreduce(views, count=count, dtype=dt, op=op, algo=algo,
                                                                  stream=sid if s is None else s)
                            for _ in range(3):
                                ar.check(call(), "sweep")
                            torch.cuda.synchronize()
                            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                            e0.record(stream)
                            ar.check(call(), "sweep")
                            e1.record(stream)
                            torch.cuda.synchronize()
                            est = e0.elapsed_time(e1)
                            k = int(min(200, max(5, 30.0 / max(est, 1e-3))))
                            e0.record(stream)
                            for _ in range(k):
                                call()
                            e1.record(stream)
                            torch.cuda.synchronize()
                            t = e0.elapsed_time(e1) / k / 1e3
                            rc, st = ar.ar_device_status(sid)
                            ar.check(rc or st, "sweep status")
                            rec = {"nranks": n, "bytes_per_rank": nbytes, "dtype": dt, "op": op, "algo": algo,
                                   "us": t * 1e6, "effective_gbs": 2 * n * nbytes / t / 1e9,
                                   "algbw_gbs": nbytes / t / 1e9, "l2_resident": 2 * n * nbytes <= 129e6}
                            if nbytes <= (1 << 20):
                                # device time without the host's per-call cost: 20 calls replayed from a graph
                                rec["graph_us"] = graph_time(call, torch, stream)
                                # host cost of a prepared call (checks and tables done once)
                                plan = ar.Plan("allreduce", views, count=count, dtype=dt, op=op, algo=algo)
                                for _ in range(3):
                                    ar.check(plan.run(sid), "plan")
                                torch.cuda.synchronize()
                                e0.record(stream)
                                for _ in range(k):
                                    plan.run(sid)
                                e1.record(stream)
                                torch.cuda.synchronize()
                                rec["plan_us"] = e0.elapsed_time(e1) * 1e3 / k
                                plan.close()
                            out.write(json.dumps(rec) + "\n")
                            npoints += 1
                            if op == "sum":
                                curves.setdefault(algo, []).append((nbytes, t))
                L = math.log2(n)
                for algo, pts in curves.items():
                    stepwise = algo.endswith("stepwise")
                    steps = (2 * (n - 1) if algo.startswith("ring") else 2 * int(L)) if stepwise else 1
                    # per-rank traffic factor of the pages' model: 2(N-1)/N D for ring and
                    # halving/doubling; the binomial tree's root moves 2 log2(N) D
                    factor = 2 * L if algo.startswith("binomial") else 2 * (n - 1) / n
                    alpha, beta = fit_alpha_beta(pts, steps, factor)
                    fits[f"N{n}_{dt}_{algo}"] = {"alpha_us": alpha * 1e6, "beta_ps_per_byte": beta * 1e12,
                                                 "steps": steps}
                if "ring_stepwise" in curves and "binomial_stepwise" in curves:
                    rs = dict(curves["ring_stepwise"])

                    def first_ring_win(other):
                        # the smallest size from which the ring is faster by 2% or more at that size
                        # and at every larger one measured (None: the ring never pulls ahead)
                        os_ = dict(curves[other])
                        sizes = sorted(d for d in rs if d in os_)
                        win = None
                        for d in reversed(sizes):
                            if rs[d] < 0.98 * os_[d]:
                                win = d
                            else:
                                break
                        return win

                    def ratios(other):
                        os_ = dict(curves[other])
                        return {str(d): round(rs[d] / os_[d], 3) for d in sorted(rs) if d in os_}
                    f = fits[f"N{n}_{dt}_ring_stepwise"]
                    a_, b_ = f["alpha_us"] * 1e-6, f["beta_ps_per_byte"] * 1e-12
                    # where the pages' alpha-beta model puts the ring/tree crossover, with the
                    # fitted ring alpha and beta: against a binomial tree whose root moves
                    # 2 log2(N) D, and against a pipelined tree moving 2 D
                    model_binom = ((n - 1 - L) * a_ / ((L - (n - 1) / n) * b_)) if n > 2 else None
                    model_pipe = (n - 1 - L) * n * a_ / b_
                    crossover[f"N{n}_{dt}"] = {
                        "crossover_measured_ring_vs_binomial_bytes": first_ring_win("binomial_stepwise"),
                        "crossover_measured_ring_vs_halving_doubling_bytes": first_ring_win("tree_stepwise"),
                        "model_ring_vs_binomial_bytes": model_binom,
                        "model_ring_vs_pipelined_tree_bytes": model_pipe,
                        "ring_over_binomial_time_by_bytes": ratios("binomial_stepwise")}
            del bufs
            torch.cuda.empty_cache()
    line = {"metric": METRIC + " (sweep)", "points": npoints, "points_file": args.sweep_out, "unit": "us",
            "alpha_beta": fits, "ring_tree_crossover": crossover, "data": "synthetic uniform(-1,1)"}
    if rank == 0:
        print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# workloads of our arm: host inputs (pinned), device buffers, one step
# ---------------------------------------------------------------------------

def rank_offsets(n: int, esize: int, kind: str) -> list:
    """Element offset of each rank's buffer inside its allocation."""
    vec = 16 // esize
    return [0] * n if kind == "aligned" else [(3 * r + 1) % vec for r in range(n)]


def rank_buffers(n, count, dtype, dev, esize, kind):
    """One device allocation per rank (16 elements of slack), each rank's
    buffer a view at its offset (all 0 unless kind == 'mixed')."""
    import torch
    return [torch.empty(count + 16, dtype=dtype, device=dev)[o:o + count] for o in rank_offsets(n, esize, kind)]


class LargeWorkload:
    """8 ranks x 67,108,864 bf16, ring SUM: the headline configuration."""
    dtype, op = "bf16", "sum"

    def __init__(self, args, dev, torch, np, W, ar):
        self.ar, self.args = ar, args
        self.n, self.count = (args.nranks or W.LARGE["nranks"]), (args.count or W.LARGE["count"])
        self.bytes_step = 2 * self.n * self.count * 2
        self.host = torch.empty((self.n, self.count), dtype=torch.int16, pin_memory=True)
        for r in range(self.n):
            self.host[r].copy_(torch.from_numpy(W.large_rank(r, self.count).view(np.int16)))
        self.out = torch.empty_like(self.host, pin_memory=True)
        self.bufs = rank_buffers(self.n, self.count, torch.int16, dev, 2, args.rank_offsets)
        self.h2d = [(self.host[r], self.bufs[r]) for r in range(self.n)]
        self.d2h = [(self.bufs[r], self.out[r]) for r in range(self.n)]
        headline = self.count == W.LARGE["count"] and self.n == W.LARGE["nranks"] and args.algo == "ring"
        self.workload = WORKLOAD if headline else (
            f"{args.algo} AllReduce SUM, {self.n} ranks x {self.count:,} bf16 ({self.count * 2 / 2**20:g} MiB per rank)")
        if args.rank_offsets == "mixed":
            self.workload += ", rank buffers at different addresses modulo 16"
        self.config = {"nranks": self.n, "count_per_rank": self.count, "algo": args.algo, "op": self.op,
                       "l2": ("inputs larger than L2" if self.n * self.count * 2 > 129e6 else "inputs partly L2-resident")
                       + f" ({2 * self.n * self.count * 2 / 2**30:g} GiB touched per step vs 129 MB L2)",
                       "rank_offset_elements": rank_offsets(self.n, 2, args.rank_offsets)}

    def step(self, sid, algo):
        rc = self.ar.ar_allreduce(self.bufs, count=self.count, dtype=self.dtype, op=self.op, algo=algo, stream=sid)
        if rc:
            raise self.ar.ArError(rc, "ar_allreduce")

    def device_set(self):
        return self.bufs, lambda sid: self.step(sid, self.args.algo)

    def second_set(self):
        import torch
        bufs = rank_buffers(self.n, self.count, self.bufs[0].dtype, self.bufs[0].device, 2, self.args.rank_offsets)

        def step(sid):
            rc = self.ar.ar_allreduce(bufs, count=self.count, dtype=self.dtype, op=self.op, algo=self.args.algo,
                                      stream=sid)
            if rc:
                raise self.ar.ArError(rc, "ar_allreduce")
        return bufs, step

    def cpu_baseline(self, gpu_result=None):
        import numpy as np
        procs = self.args.cpu_procs or host_cores()
        passes = 3
        res = gpu_result.view(np.uint16) if gpu_result is not None else None
        dt, gbs, one, parity = oracle_pass_time(self.host.numpy().view(np.uint16), procs, passes, res)
        return {"value": gbs, "unit": "GB/s", "cores": procs, "kind": "oracle", "cpu_model": cpu_model(),
                "one_process_gbs": one,
                "sample": f"the whole workload ({self.n} ranks x {self.count} bf16), literal ring passes: "
                          f"1 untimed + {passes} timed at {dt:.3f} s each, element ranges split over "
                          f"{procs} processes",
                "parity": parity}


class BucketWorkload:
    """8 ranks x 6,553,600 f32 (one 25 MiB DDP bucket), ring AVG."""
    dtype, op = "f32", "avg"

    def __init__(self, args, dev, torch, np, W, ar):
        self.ar, self.args = ar, args
        self.n, self.count = W.BUCKET["nranks"], (args.count or W.BUCKET["count"])
        self.bytes_step = 2 * self.n * self.count * 4
        x = W.bucket_inputs(self.n, self.count)
        self.host = torch.from_numpy(x).pin_memory()
        self.out = torch.empty_like(self.host, pin_memory=True)
        self.bufs = rank_buffers(self.n, self.count, torch.float32, dev, 4, args.rank_offsets)
        self.h2d = [(self.host[r], self.bufs[r]) for r in range(self.n)]
        self.d2h = [(self.bufs[r], self.out[r]) for r in range(self.n)]
        self.workload = "ring AllReduce AVG, 8 ranks x 6,553,600 f32 (one 25 MiB DDP bucket)"
        if args.rank_offsets == "mixed":
            self.workload += ", rank buffers at different addresses modulo 16"
        self.config = {"nranks": self.n, "count_per_rank": self.count, "algo": args.algo, "op": self.op,
                       "l2": "inputs larger than L2 (409.6 MiB touched per step vs 129 MB L2)",
                       "rank_offset_elements": rank_offsets(self.n, 4, args.rank_offsets)}

    def step(self, sid, algo, int8=False, op=None):
        if int8:
            import torch
            if getattr(self, "resid", None) is None:
                self.resid = [torch.zeros_like(b) for b in self.bufs]
            rc = self.ar.ar_allreduce_int8_ef(self.bufs, self.resid, count=self.count, op=self.op, stream=sid)
        else:
            rc = self.ar.ar_allreduce(self.bufs, count=self.count, dtype=self.dtype, op=op or self.op, algo=algo,
                                      stream=sid)
        if rc:
            raise self.ar.ArError(rc, "ar_allreduce")

    def device_set(self):
        return self.bufs, lambda sid: self.step(sid, self.args.algo)

    def second_set(self):
        bufs = rank_buffers(self.n, self.count, self.bufs[0].dtype, self.bufs[0].device, 4, self.args.rank_offsets)

        def step(sid):
            rc = self.ar.ar_allreduce(bufs, count=self.count, dtype=self.dtype, op=self.op, algo=self.args.algo,
                                      stream=sid)
            if rc:
                raise self.ar.ArError(rc, "ar_allreduce")
        return bufs, step

    def cpu_baseline(self, gpu_result=None):
        import numpy as np
        import oracle
        from allreduce_gradient_reduction_gb300 import workloads as W
        oracle.build()
        x = W.bucket_inputs(self.n, self.count)
        t0 = time.perf_counter()
        out, _ = oracle.allreduce(x, algo="ring", op="avg", dtype="f32")
        dt = time.perf_counter() - t0
        parity = None
        if gpu_result is not None:
            same = all(np.array_equal(out[r].view(np.uint32), gpu_result.view(np.uint32)) for r in range(self.n))
            parity = {"vs": "oracle", "elements": int(self.count), "bit_identical": bool(same)}
        return {"value": self.bytes_step / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                "cpu_model": cpu_model(),
                "sample": f"the whole workload, one literal ring pass, {dt:.2f} s, one thread", "parity": parity}


class Gpt2Workload:
    """GPT-2 small gradients (148 tensors, 124,439,808 f32 per rank), 8 ranks,
    DDP buckets of 25 MiB in reverse order, AVG; each rank's gradients are
    views into one flat allocation."""
    dtype, op = "f32", "avg"

    def __init__(self, args, dev, torch, np, W, ar):
        self.ar, self.args = ar, args
        self.n = W.GPT2["nranks"]
        self.counts = W.gpt2_small_counts()
        self.total = int(self.counts.sum())
        self.bytes_step = 2 * self.n * self.total * 4
        offs = np.concatenate([[0], np.cumsum(self.counts)])
        self.host = torch.empty((self.n, self.total), dtype=torch.float32, pin_memory=True)
        for r in range(self.n):
            self.host[r].copy_(torch.from_numpy(np.concatenate(W.gpt2_rank_grads(r, self.counts))))
        self.out = torch.empty_like(self.host, pin_memory=True)
        self.flats = [torch.empty(self.total, dtype=torch.float32, device=dev) for _ in range(self.n)]
        self.grads = [[f[offs[t]:offs[t + 1]] for t in range(len(self.counts))] for f in self.flats]
        self.h2d = [(self.host[r], self.flats[r]) for r in range(self.n)]
        self.d2h = [(self.flats[r], self.out[r]) for r in range(self.n)]
        self.ws = None
        self.workload = "DDP bucketed AllReduce AVG, 8 ranks x GPT-2 small gradients (124,439,808 f32, 25 MiB buckets)"
        self.config = {"nranks": self.n, "params_per_rank": self.total, "tensors": len(self.counts),
                       "bucket_cap_bytes": 25 << 20, "algo": args.algo, "op": self.op, "path": "fused",
                       "l2": "inputs larger than L2 (8 GB touched per step)"}

    def step(self, sid, algo, literal=False):
        ws, wbytes = None, 0
        if literal:
            import torch
            if self.ws is None:
                self.ws = [torch.empty(self.total, dtype=torch.float32, device=self.flats[0].device)
                           for _ in range(self.n)]
            ws, wbytes = self.ws, self.total * 4
        rc = self.ar.ar_bucketed_allreduce(self.grads, counts=self.counts, dtype=self.dtype, op=self.op, algo=algo,
                                           workspace=ws, workspace_bytes=wbytes, stream=sid)
        if rc:
            raise self.ar.ArError(rc, "ar_bucketed_allreduce")

    def device_set(self):
        return self.flats, lambda sid: self.step(sid, self.args.algo)

    def second_set(self):
        import numpy as np
        import torch
        flats = [torch.empty_like(f) for f in self.flats]
        offs = np.concatenate([[0], np.cumsum(self.counts)])
        grads = [[f[offs[t]:offs[t + 1]] for t in range(len(self.counts))] for f in flats]

        def step(sid):
            rc = self.ar.ar_bucketed_allreduce(grads, counts=self.counts, dtype=self.dtype, op=self.op,
                                               algo=self.args.algo, stream=sid)
            if rc:
                raise self.ar.ArError(rc, "ar_bucketed_allreduce")
        return flats, step

    def overlap(self, sid, tokens, iters=5, eager=False):
        """Synthetic backward: for every tensor in reverse registration order and
        every rank, a GEMM of the shape of its weight gradient (dW = X^T dY over
        `tokens` tokens; a column sum for vectors) writes the gradient on the
        compute stream.  Times the backward alone, backward then the bucketed
        AllReduce, and backward with the reducer starting each bucket as soon
        as its gradients exist (DDP's overlap)."""
        import torch
        shapes = [s for _, s in __import__("allreduce_gradient_reduction_gb300.workloads",
                                           fromlist=["x"]).gpt2_small_shapes()]
        dev = self.flats[0].device
        gen = torch.Generator(device=dev)
        gen.manual_seed(7)
        amax = max(s[0] for s in shapes if len(s) == 2)
        bmax = max(s[-1] for s in shapes)
        X = [torch.randn(tokens, amax, device=dev, generator=gen) * 1e-2 for _ in range(self.n)]
        Y = [torch.randn(tokens, bmax, device=dev, generator=gen) * 1e-2 for _ in range(self.n)]
        compute = torch.cuda.current_stream()
        # the reducer's stream at normal priority and at the highest (as a
        # collective library's would be), so its blocks go first as GEMM blocks retire
        reducers = {}
        for prio in (0, -1):
            comm = torch.cuda.Stream(priority=prio)
            reducers[prio] = (comm, self.ar.Reducer(self.grads, counts=self.counts, dtype=self.dtype, op=self.op,
                                                    algo="ring", comm_stream=comm))
        red = reducers[0][1]

        def backward(mark=None):
            for t in range(len(shapes) - 1, -1, -1):
                shp = shapes[t]
                for r in range(self.n):
                    g = self.grads[r][t]
                    if len(shp) == 2:
                        torch.mm(X[r][:, :shp[0]].t(), Y[r][:, :shp[1]], out=g.view(shp))
                    else:
                        torch.sum(Y[r][:, :shp[0]], 0, out=g)
                if mark:
                    mark(t)

        def seq():
            backward()
            self.step(int(torch.cuda.current_stream().cuda_stream), "ring")

        def ovl_with(rd):
            def ovl():
                s = torch.cuda.current_stream()
                backward(lambda t: self.ar.check(rd.mark_ready(t, s), "mark_ready"))
                self.ar.check(rd.finish(s), "finish")
            return ovl

        # each variant is captured once into a CUDA graph and replayed, so the
        # numbers are GPU time, not the host's launch rate (1184 GEMM launches);
        # eager=True launches them directly (graphs drop stream priorities), for
        # token counts whose GEMMs outlast their launches
        def timed(fn):
            fn()
            torch.cuda.synchronize()
            if eager:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(compute)
                for _ in range(iters):
                    fn()
                e1.record(compute)
                torch.cuda.synchronize()
                return e0.elapsed_time(e1) / iters
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(compute)
            for _ in range(iters):
                g.replay()
            e1.record(compute)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / iters

        tf32 = torch.backends.cuda.matmul.allow_tf32
        torch.backends.cuda.matmul.allow_tf32 = True  # mixed-precision-like backward on the tensor cores
        by_blocks = {}
        try:
            t_bwd, t_seq = timed(backward), timed(seq)
            # block caps for the overlapped reductions: none (one block per
            # tile), then a few "channels" of the GPU's 152 SMs
            for prio, (_, rd) in reducers.items():
                for cap in (0, 304, 152, 76, 38):
                    self.ar.check(rd.set_max_blocks(cap), "set_max_blocks")
                    by_blocks[f"prio{prio}_blocks{cap}"] = timed(ovl_with(rd))
        finally:
            torch.backends.cuda.matmul.allow_tf32 = tf32
        nbuckets = red.buckets
        for _, rd in reducers.values():
            rd.close()
        best = min(by_blocks, key=by_blocks.get)
        t_ovl = by_blocks[best]
        t_ar = t_seq - t_bwd
        return {"tokens": tokens, "backward_ms": t_bwd, "sequential_ms": t_seq, "overlapped_ms": t_ovl,
                "overlapped_ms_by_stream_priority_and_max_blocks": by_blocks, "best": best,
                "allreduce_ms_in_sequence": t_ar, "exposed_comm_ms": t_ovl - t_bwd,
                "hidden_fraction": (t_seq - t_ovl) / t_ar if t_ar > 0 else None, "buckets": nbuckets,
                "launch": "eager" if eager else "cuda graph",
                "note": "backward = per-rank TF32 GEMMs (dW = X^T dY) on the compute stream; both streams share "
                        "one GPU"}

    def cpu_baseline(self, gpu_result=None):
        """The oracle's literal bucketed AllReduce (pack, ring, unpack) over the
        whole workload, one bucket per process at a time on every host core;
        its per-tensor digests check the GPU's result of the same inputs."""
        import numpy as np
        import oracle
        from oracle import parallel as oracle_parallel
        oracle.build()
        host = self.host.numpy()
        offs = np.concatenate([[0], np.cumsum(self.counts)])
        grads = [[host[r, offs[t]:offs[t + 1]] for t in range(len(self.counts))] for r in range(self.n)]
        procs = self.args.cpu_procs or host_cores()
        t0 = time.perf_counter()
        with oracle_parallel.Pool(procs) as pool:
            want, slowest = pool.bucketed_digests(grads, op="avg", dtype="f32", cap_bytes=25 << 20)
        dt = time.perf_counter() - t0
        parity = None
        if gpu_result is not None:
            same = all(oracle_parallel.digest(gpu_result[offs[t]:offs[t + 1]]) == want[0][t]
                       for t in range(len(self.counts)))
            parity = {"vs": "oracle", "elements": int(self.total), "tensors": len(self.counts),
                      "bit_identical": bool(same)}
        return {"value": self.bytes_step / dt / 1e9, "unit": "GB/s", "cores": procs, "kind": "oracle",
                "cpu_model": cpu_model(),
                "sample": f"the whole workload (8 ranks x {self.total} f32, 17 buckets), literal pack, ring, unpack, "
                          f"buckets spread over {procs} processes: {dt:.2f} s wall (includes sending the inputs), "
                          f"slowest process {slowest:.2f} s",
                "parity": parity}


# ---------------------------------------------------------------------------
# end to end: host inputs in, host results out
# ---------------------------------------------------------------------------

# The pages' own figures, other hardware: quoted as context, never as a target.
PAGES_CONTEXT = {
    "nvlink_h100_gbs_bidirectional": 900, "nvlink_a100_gbs_per_gpu": 600, "infiniband_hdr_gbs": 25,
    "ddp_bucket_mb": 25, "note": "figures printed on the pages for other hardware; context only",
}


def accuracy(wl, step, torch, np, dev):
    """Fresh inputs, one step, then sampled positions against the order-free
    float64 reduction: the largest |error| / sum|x|, the tolerance stated for
    the dtype (1e-5 f32, 2^-7 bf16) and the fraction of positions above it,
    and the recursive-summation bound gamma_{N-1} of the ring's N-1 rounded
    additions."""
    for src, dst in wl.h2d:
        dst.copy_(src)
    torch.cuda.synchronize()
    step()
    torch.cuda.synchronize()
    count = wl.h2d[0][0].numel()
    pos = np.unique(np.random.default_rng(12345).integers(0, count, 1 << 16))
    idx = torch.from_numpy(pos).to(dev)
    x = np.stack([src.numpy()[pos] for src, _ in wl.h2d])
    got = np.stack([dst[idx].cpu().numpy() for _, dst in wl.h2d])
    if wl.dtype == "bf16":
        def f64(a):
            return (a.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        u, tol = 2.0 ** -8, 2.0 ** -7
    else:
        def f64(a):
            return a.astype(np.float64)
        u, tol = 2.0 ** -24, 1e-5
    xs = f64(x)
    scale = 1.0 / wl.n if wl.op == "avg" else 1.0
    ref, absum = xs.sum(axis=0) * scale, np.abs(xs).sum(axis=0) * scale
    err = np.abs(f64(got) - ref).max(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(absum > 0, err / absum, 0.0)
    k = wl.n - 1
    gamma = k * u / (1 - k * u)
    return {"vs": "float64 order-free reduction", "positions": int(pos.size),
            "max_err_over_abs_sum": float(ratio.max()), "tolerance": tol,
            "frac_above_tolerance": float((ratio > tol).mean()), "gamma_bound": gamma,
            "within_gamma_bound": bool((ratio <= gamma * (1 + 1e-9)).all()),
            "ranks_identical": bool(all(np.array_equal(got[r], got[0]) for r in range(wl.n)))}


def end_to_end_host_call(wl, args, ws, stream, torch):
    """The same metric through the library's host-buffer call: every step,
    one ar_allreduce_host takes the N rank buffers in page-locked host memory
    and leaves the result in them, so every element crosses the CPU-GPU link
    once each way.  Reported: the zero-copy form (the fused kernel reads and
    writes the host buffers directly); beside it the staged form (pieces
    copied in and out around the kernel).  Successive steps do not overlap:
    each reads what the previous one wrote."""
    ar = wl.ar
    steps = max(3, min(args.steps, 20))
    sid = int(stream.cuda_stream)
    host = wl.host.clone().pin_memory()  # the inputs stay untouched for the other legs
    rows = list(host)
    work = [torch.empty_like(b) for b in wl.bufs]
    io_bytes = sum(r.numel() * r.element_size() for r in rows)

    def call(dev_bufs):
        ar.check(ar.ar_allreduce_host(rows, dev_bufs, count=wl.count, dtype=wl.dtype, op=wl.op, algo=args.algo,
                                      stream=sid), "ar_allreduce_host")

    def timed(dev_bufs):
        call(dev_bufs)
        call(dev_bufs)
        torch.cuda.synchronize()
        barrier(ws)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(steps):
            call(dev_bufs)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        return max_over_ranks(t0.elapsed_time(t1) / steps, ws)

    ms_staged = timed(work)
    ms = timed(None)  # zero-copy: the reported figure
    identical = bool(all(torch.equal(rows[0], r) for r in rows[1:]))
    # one zero-copy call on the original inputs against the device-buffer call
    host.copy_(wl.host)
    call(None)
    for b, src in zip(work, wl.host):
        b.copy_(src, non_blocking=True)
    ar.check(ar.ar_allreduce(work, count=wl.count, dtype=wl.dtype, op=wl.op, algo=args.algo, stream=sid),
             "ar_allreduce")
    torch.cuda.synchronize()
    matches = bool(torch.equal(host[0], work[0].cpu()))
    del work, host, rows
    torch.cuda.empty_cache()
    return {"value": ws * wl.bytes_step / (ms / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": io_bytes,
            "d2h_bytes_per_step": io_bytes, "steps": steps, "ms_per_step": ms,
            "call": "ar_allreduce_host, zero-copy: one fused launch reads every rank's elements from the "
                    "page-locked host buffers and writes the result back to them across the CPU-GPU link",
            "staged_ms_per_step": ms_staged,
            "staged": "the same call with device working buffers: pieces of up to 16 MiB per rank overlap "
                      "upload, reduction and download on three streams",
            "result_ranks_identical": identical, "matches_device_call": matches}


def end_to_end(wl, args, ws, stream, torch):
    """The same metric through the public call with the step's inputs copied
    from pinned host memory and its results copied back inside the timed
    region, every step.  Two device buffer sets alternate between steps, so
    the upload of step k+1, the reduction of step k and the download of step
    k-1 run on three streams at once (the host link is full duplex); the
    strictly sequential form is reported beside it."""
    steps = max(3, min(args.steps, 20))
    io_bytes = sum(src.numel() * src.element_size() for src, _ in wl.h2d)
    sets = [wl.device_set(), wl.second_set()]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    uploaded, reduced, downloaded = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def run(k):
        b = k % 2
        targets, step_fn = sets[b]
        with torch.cuda.stream(up):
            if k >= 2:
                up.wait_event(downloaded[b])  # the set's previous results are out
            for (src, _), dst in zip(wl.h2d, targets):
                dst.copy_(src, non_blocking=True)
            uploaded[b].record(up)
        stream.wait_event(uploaded[b])
        step_fn(int(stream.cuda_stream))
        reduced[b].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(reduced[b])
            for src, (_, dst) in zip(targets, wl.d2h):
                dst.copy_(src, non_blocking=True)
            downloaded[b].record(down)

    def timed(pipelined):
        torch.cuda.synchronize()
        barrier(ws)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        up.wait_stream(stream)
        for k in range(steps):
            run(k)
            if not pipelined:
                stream.wait_stream(down)
                up.wait_stream(down)
        stream.wait_stream(down)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        return max_over_ranks(t0.elapsed_time(t1) / steps, ws)

    run(0)
    run(1)  # warm both sets and the copy paths
    ms_seq = timed(False)
    ms = timed(True)
    return {"value": ws * wl.bytes_step / (ms / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": io_bytes,
            "d2h_bytes_per_step": io_bytes, "steps": steps, "ms_per_step": ms,
            "ms_per_step_sequential": ms_seq, "pipelining": "two buffer sets, upload/reduce/download streams",
            "result_ranks_identical": bool(torch.equal(wl.out[0], wl.out[wl.n - 1]))}


# ---------------------------------------------------------------------------
# the other configurations, timed beside the headline
# ---------------------------------------------------------------------------

def timed_calls(call, k, stream, torch, warm=3):
    """Milliseconds per call over k back-to-back calls (CUDA events on the
    launching stream, after `warm` untimed calls), and the wall window."""
    for _ in range(warm):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record(stream)
    for _ in range(k):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / k, (t0, time.time())


def other_workloads(dev, torch, np, W, ar, stream, clocks, peak):
    """The small, bucket and GPT-2 configurations, each timed the way the
    headline is (CUDA events over back-to-back calls on the launching stream),
    with the clocks sampled during each window."""
    sid = int(stream.cuda_stream)
    out = {}

    def chk(rc, what):
        if rc:
            raise ar.ArError(rc, what)

    # small: 4 ranks x 4096 f32 integers, ring SUM -- latency bound (L2 resident)
    n, count = W.SMALL["nranks"], W.SMALL["count"]
    x = W.small_inputs(n, count)
    bufs = [torch.from_numpy(x[r]).to(dev) for r in range(n)]
    call = lambda s=sid: chk(ar.ar_allreduce(bufs, count=count, dtype="f32", op="sum", algo="ring", stream=s), "small")
    eager_ms, win = timed_calls(call, 2000, stream, torch)
    plan = ar.Plan("allreduce", bufs, count=count, dtype="f32", op="sum", algo="ring")
    plan_ms, _ = timed_calls(lambda: chk(plan.run(sid), "small plan"), 2000, stream, torch)
    plan.close()
    graph_us = graph_time(lambda s: ar.ar_allreduce(bufs, count=count, dtype="f32", op="sum", algo="ring", stream=s),
                          torch, stream, reps=50)
    nbytes = 2 * n * count * 4
    out["small"] = {"workload": "ring AllReduce SUM, 4 ranks x 4096 f32 (integers in [-8, 8])",
                    "us_per_call_eager": eager_ms * 1e3, "us_per_call_prepared": plan_ms * 1e3,
                    "us_per_call_graph": graph_us, "algorithmic_bytes": nbytes,
                    "note": "latency bound and L2 resident: eager = one ar_allreduce through the binding per call "
                            "(host-bound), prepared = ar_plan_run, graph = 50 calls replayed from a CUDA graph "
                            "(device time)", "clocks": clocks.summary(*win)}
    del bufs

    # bucket: 8 ranks x 6,553,600 f32 (one 25 MiB DDP bucket), ring AVG, then MAX on the same data
    n, count = W.BUCKET["nranks"], W.BUCKET["count"]
    x = W.bucket_inputs(n, count)
    bufs = [torch.from_numpy(x[r]).to(dev) for r in range(n)]
    nbytes = 2 * n * count * 4
    for op in ("avg", "max"):
        ms, win = timed_calls(lambda: chk(ar.ar_allreduce(bufs, count=count, dtype="f32", op=op, algo="ring",
                                                          stream=sid), "bucket"), 200, stream, torch)
        gbs = nbytes / (ms / 1e3) / 1e9
        out[f"bucket_{op}"] = {"workload": f"ring AllReduce {op.upper()}, 8 ranks x 6,553,600 f32 (one 25 MiB bucket)",
                               "ms_per_step": ms, "effective_gbs": gbs, "frac": gbs / peak,
                               "algorithmic_bytes": nbytes, "clocks": clocks.summary(*win)}
    del bufs

    # the headline configuration with every rank buffer at a different address
    # modulo 16 (rank r starts (3r + 1) mod 8 elements into its allocation):
    # the staged kernel
    n, count = W.LARGE["nranks"], W.LARGE["count"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(W.BASE_SEED + 1000 * W.CONFIG_LARGE + 7)
    bufs = rank_buffers(n, count, torch.bfloat16, dev, 2, "mixed")
    for b in bufs:
        b.copy_(torch.randn(count, device=dev, generator=gen).to(torch.bfloat16))
    nbytes = 2 * n * count * 2
    ms, win = timed_calls(lambda: chk(ar.ar_allreduce(bufs, count=count, dtype="bf16", op="sum", algo="ring",
                                                      stream=sid), "large mixed"), 200, stream, torch)
    gbs = nbytes / (ms / 1e3) / 1e9
    out["large_mixed_offsets"] = {
        "workload": "ring AllReduce SUM, 8 ranks x 67,108,864 bf16, rank buffers at eight different addresses "
                    "modulo 16 (element offsets " + ", ".join(str(o) for o in rank_offsets(n, 2, "mixed")) + ")",
        "ms_per_step": ms, "effective_gbs": gbs, "frac": gbs / peak, "algorithmic_bytes": nbytes,
        "clocks": clocks.summary(*win)}
    del bufs
    torch.cuda.empty_cache()

    # GPT-2 small gradients in 25 MiB reverse-order buckets, AVG: fused and literal
    counts = W.gpt2_small_counts()
    total = int(counts.sum())
    n = W.GPT2["nranks"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(W.BASE_SEED + 1000 * W.CONFIG_GPT2)
    flats = [torch.randn(total, device=dev, generator=gen).mul_(1e-4) for _ in range(n)]
    offs = np.concatenate([[0], np.cumsum(counts)])
    grads = [[f[offs[t]:offs[t + 1]] for t in range(len(counts))] for f in flats]
    ws = [torch.empty(total, device=dev) for _ in range(n)]
    nbytes = 2 * n * total * 4
    for mode in ("fused", "literal"):
        w, wb = (ws, total * 4) if mode == "literal" else (None, 0)
        launches0 = ar.ar_kernel_launches()
        chk(ar.ar_bucketed_allreduce(grads, counts=counts, dtype="f32", op="avg", algo="ring", workspace=w,
                                     workspace_bytes=wb, stream=sid), "gpt2")
        per_step = ar.ar_kernel_launches() - launches0
        ms, win = timed_calls(lambda: chk(ar.ar_bucketed_allreduce(grads, counts=counts, dtype="f32", op="avg",
                                                                   algo="ring", workspace=w, workspace_bytes=wb,
                                                                   stream=sid), "gpt2"),
                              40 if mode == "fused" else 20, stream, torch)
        gbs = nbytes / (ms / 1e3) / 1e9
        rec = {"workload": "DDP bucketed AllReduce AVG, 8 ranks x GPT-2 small gradients (148 tensors, "
                           f"{total:,} f32, 17 buckets of <= 25 MiB), {mode}",
               "ms_per_step": ms, "effective_gbs": gbs, "frac": gbs / peak, "algorithmic_bytes": nbytes,
               "launches_per_step": per_step, "clocks": clocks.summary(*win)}
        if mode == "literal":
            rec["moved_bytes"] = 3 * nbytes  # pack, AllReduce, unpack: each 2 N P b
            rec["moved_gbs"] = 3 * gbs
        out[f"gpt2_{mode}"] = rec
    del flats, grads, ws
    torch.cuda.empty_cache()
    out["note"] = ("each timed like the headline (CUDA events over back-to-back calls); bucket and small inputs "
                   "from the seeded host recipe, GPT-2 gradients and the mixed-offset rows drawn on the device "
                   "(normal(0, 1e-4); normal(0, 1)); frac is of the measured copy bandwidth")
    return out


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
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    # one process per node compiles (a no-op when the library is up to date);
    # the others wait, then only load it
    if local == 0:
        __graft_entry__.build()
    barrier(ws)
    if local != 0:
        __graft_entry__.build()
    from allreduce_gradient_reduction_gb300 import binding as ar
    from allreduce_gradient_reduction_gb300 import workloads as W

    if args.sweep:
        return run_sweep(args, ws, rank, dev, torch, ar)
    wl = {"large": LargeWorkload, "bucket": BucketWorkload, "gpt2": Gpt2Workload}[args.workload](
        args, dev, torch, np, W, ar)
    for src, dst in wl.h2d:
        dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    sid = int(stream.cuda_stream)
    nbytes_step = wl.bytes_step

    def step(algo=args.algo, **kw):
        wl.step(sid, algo, **kw)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = ar.ar_kernel_launches()
    t_wall0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    launches = ar.ar_kernel_launches() - launches0
    barrier(ws)
    ms_local = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms_local, ws)
    rc, status = ar.ar_device_status(sid)
    if rc or status:
        raise ar.ArError(rc or status, "device status")

    # the spread of single steps (outside the timed region): each one bracketed
    # by its own events, so launch gaps count against it
    singles = []
    for _ in range(20):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        singles.append((a, b))
    torch.cuda.synchronize()
    single_ms = sorted(a.elapsed_time(b) for a, b in singles)

    value = ws * nbytes_step / (ms / 1e3) / 1e9
    algbw = nbytes_step / (2 * wl.n) / (ms / 1e3) / 1e9
    # one step is `launches / steps` kernels; the roofline is per step of the hot path
    achieved = nbytes_step / (ms_local / 1e3) / 1e9

    # end to end through the public call: pinned host -> device, AllReduce, device -> host
    e2e = None
    if not args.no_e2e:
        if hasattr(wl, "host") and hasattr(wl, "count") and args.algo in ("ring", "tree", "naive", "dbtree"):
            e2e = end_to_end_host_call(wl, args, ws, stream, torch)
        else:  # bucketed and step-wise calls: device-buffer calls with the copies around them
            e2e = end_to_end(wl, args, ws, stream, torch)

    peak, peak_kind = hbm_peak()
    others = None
    if (isinstance(wl, LargeWorkload) and not args.count and not args.no_workloads and rank == 0
            and args.algo == "ring"):
        others = other_workloads(dev, torch, np, W, ar, stream, clocks, peak)
    clocks.stop()

    variants = {}
    if args.variants:
        orders = ("ring", "tree", "ring_stepwise", "tree_stepwise")
        if not isinstance(wl, Gpt2Workload):
            orders += ("dbtree", "naive")
        # (name, one call, algorithmic bytes of that call)
        todo = [(a, (lambda a=a: step(a)), nbytes_step) for a in orders if a != args.algo]
        if isinstance(wl, Gpt2Workload):
            todo += [("ring_literal", lambda: step("ring", literal=True), nbytes_step)]
        if isinstance(wl, BucketWorkload):
            # the residuals are read and written too: 4 N D floats
            todo += [("int8_ef", lambda: step("ring", int8=True), 2 * nbytes_step),
                     ("ring_max", lambda: step("ring", op="max"), nbytes_step)]  # MAX on the same data
        if not isinstance(wl, Gpt2Workload):
            # the other collectives on the same buffers, each against its own bytes:
            # ReduceScatter and Reduce read N D and write D, AllGather and
            # Broadcast read D and write (N - 1) D
            per = nbytes_step // (2 * wl.n)  # D * b
            c = dict(count=wl.count, dtype=wl.dtype, stream=sid)

            def chk(rc):
                if rc:
                    raise ar.ArError(rc, "collective variant")

            todo += [
                ("reduce_scatter", lambda: chk(ar.ar_reduce_scatter(wl.bufs, op=wl.op, **c)), (wl.n + 1) * per),
                ("all_gather", lambda: chk(ar.ar_all_gather(wl.bufs, **c)), wl.n * per),
                ("reduce", lambda: chk(ar.ar_reduce(wl.bufs, op=wl.op, root=0, **c)), (wl.n + 1) * per),
                ("broadcast", lambda: chk(ar.ar_broadcast(wl.bufs, root=0, **c)), wl.n * per),
            ]
        for name, call, nbytes in todo:
            for _ in range(3):
                call()
            torch.cuda.synchronize()
            v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            k = max(10, args.steps // 10)
            v0.record(stream)
            for _ in range(k):
                call()
            v1.record(stream)
            torch.cuda.synchronize()
            vms = v0.elapsed_time(v1) / k
            variants[name] = {"ms_per_step": vms, "effective_gbs": nbytes / (vms / 1e3) / 1e9}
            if nbytes != nbytes_step:
                variants[name]["algorithmic_bytes"] = nbytes

    overlap = None
    if args.overlap and isinstance(wl, Gpt2Workload):
        try:
            overlap = wl.overlap(sid, args.overlap_tokens, eager=args.overlap_eager)
        except Exception as exc:  # reported in the line; the headline numbers above stand
            overlap = {"error": f"{type(exc).__name__}: {exc}"}

    acc = accuracy(wl, step, torch, np, dev) if rank == 0 else None

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        # the accuracy step left the result of fresh inputs on the device:
        # the oracle's own pass over the same inputs checks it bit for bit
        rows = [dst for _, dst in wl.h2d]
        gpu_result = rows[0].cpu().numpy() if all(torch.equal(r, rows[0]) for r in rows[1:]) else None
        cpu = wl.cpu_baseline(gpu_result)
        if gpu_result is None and cpu is not None:
            cpu["parity"] = {"vs": "oracle", "bit_identical": False, "note": "ranks differ on the device"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
            "config": {"workload": wl.workload, **wl.config,
                       "parallelism": "replicas" if ws > 1 else "single GPU"},
            "algbw_gbs": algbw * ws,
            "single_step_ms": {"median": statistics.median(single_ms), "best": single_ms[0],
                               "worst": single_ms[-1], "samples": len(single_ms)},
            "accuracy": acc, "context": PAGES_CONTEXT,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         # the capture is of the headline kernel: aligned ring, full size
                         "traffic": profiled_traffic() if (isinstance(wl, LargeWorkload) and wl.workload == WORKLOAD
                                                           and args.rank_offsets == "aligned") else None,
                         "algorithmic_bytes_per_launch": nbytes_step},
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks.summary(t_wall0, t_wall1),
            "cpu_baseline": cpu,
        }
        if others:
            line["workloads"] = others
        if variants:
            line["variants"] = variants
        if overlap:
            line["overlap"] = overlap
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        barrier(ws)  # rank 0's accuracy and printing come last: leave together
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
