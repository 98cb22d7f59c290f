"""The oracle on many host cores (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may use this module.  It adds no arithmetic: each worker
process runs the oracle's own functions (``oracle.allreduce``,
``oracle.bucketed_allreduce``) on its share of a workload, as they stand.

Two ways of splitting the work, both exact:

* Element ranges of a plain collective.  In every schedule the oracle
  simulates, an element's value depends only on its own column of the N
  rank buffers and on the chunk that holds it, so a worker that carries the
  positions [lo, hi) of a buffer of ``count`` elements through the oracle's
  sampled-positions mode computes exactly those positions of the full run.
* Whole buckets of a bucketed AllReduce.  Buckets are reduced independently
  (each is packed, AllReduced and unpacked on its own).  A worker runs the
  oracle's bucketed AllReduce on one bucket's tensors alone, in registration
  order; planned again, they form exactly that bucket (the worker checks
  this), so its result equals the full run's on those tensors.

Workers are started with ``spawn`` (never ``fork``: a child forked after the
parent touched the GPU can hang).  Results come back as SHA-256 digests, so
nothing large crosses the pipes on the way back.
"""
from __future__ import annotations

import hashlib
import os
import time

import numpy as np


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def digest(a) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def _worker(conn):
    import oracle
    oracle.lib()
    x = pos = count = out = None
    kw = {}
    while True:
        msg = conn.recv()
        kind = msg[0]
        if kind == "load":
            _, x, lo, count, kw = msg
            pos = np.arange(lo, lo + x.shape[1], dtype=np.int64)
            conn.send(0.0)
        elif kind == "run":
            t0 = time.perf_counter()
            out, _ = oracle.collective(x, count=count, positions=pos, **{**kw, **msg[1]})
            conn.send(time.perf_counter() - t0)
        elif kind == "digest":
            # rank 0's values on this range, and whether every rank holds them
            conn.send((digest(out[0]), bool(all(np.array_equal(out[r], out[0]) for r in range(out.shape[0])))))
        elif kind == "bucketed":
            # one oracle run per bucket, on that bucket's tensors alone
            _, buckets, kw = msg
            t0 = time.perf_counter()
            res = []
            for grads, counts, expect in buckets:
                _, _, bcount = oracle.bucket_plan(counts, dtype=kw["dtype"], cap_bytes=kw["cap_bytes"])
                if list(bcount) != [expect]:
                    res = ("plan differs", list(bcount), expect)
                    break
                r_out, _ = oracle.bucketed_allreduce(grads, **kw)
                res.append([[digest(t) for t in row] for row in r_out])
            if isinstance(res, tuple):
                conn.send(res)
            else:
                conn.send(("ok", time.perf_counter() - t0, res))
        else:
            return


class Pool:
    """``procs`` spawned oracle processes, each holding one share of the input
    (loaded before any timing, so a timed pass moves no data)."""

    def __init__(self, procs: int | None = None):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.conns, self.procs = [], []
        for _ in range(procs or host_cores()):
            a, b = ctx.Pipe()
            p = ctx.Process(target=_worker, args=(b,), daemon=True)
            p.start()
            self.conns.append(a)
            self.procs.append(p)
        self.widths = []

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # ---- element ranges of one collective ------------------------------------

    def load(self, x, **kw):
        """Split the (N, count) rank buffers x into contiguous element ranges,
        one per process; ``kw`` are the oracle.collective arguments (algo, op,
        dtype, phases).  Returns the range widths."""
        count = x.shape[1]
        b = np.linspace(0, count, len(self.conns) + 1).astype(np.int64)
        for i, c in enumerate(self.conns):
            c.send(("load", np.ascontiguousarray(x[:, b[i]:b[i + 1]]), int(b[i]), count, kw))
        for c in self.conns:
            c.recv()
        self.widths = [int(b[i + 1] - b[i]) for i in range(len(self.conns))]
        return self.widths

    def run(self, **kw):
        """One pass over the loaded input (``kw`` overrides the collective's
        arguments given to load); returns (wall seconds, per-process seconds)."""
        t0 = time.perf_counter()
        for c in self.conns:
            c.send(("run", kw))
        per = [c.recv() for c in self.conns]
        return time.perf_counter() - t0, per

    def digests(self):
        """Per process: (sha256 of rank 0's result on its range, ranks identical)."""
        for c in self.conns:
            c.send(("digest",))
        return [c.recv() for c in self.conns]

    def compare(self, result) -> dict:
        """Compare `result` (count elements: one rank's result of the same
        collective, from elsewhere) with the last pass, range by range."""
        got = self.digests()
        lo, same, bad = 0, True, []
        for i, (w, (d, ranks_equal)) in enumerate(zip(self.widths, got)):
            ok = ranks_equal and digest(result[lo:lo + w]) == d
            if not ok:
                bad.append((lo, lo + w))
            same = same and ok
            lo += w
        return {"vs": "oracle", "elements": int(lo), "ranges": len(self.widths), "bit_identical": bool(same),
                "differing_ranges": bad}

    # ---- whole buckets of a bucketed AllReduce -----------------------------------

    def bucketed_digests(self, grads, *, op="avg", dtype="f32", algo="ring", cap_bytes=25 << 20):
        """oracle.bucketed_allreduce(grads, ...) split by bucket over the
        processes; returns (digests[r][t] of every result tensor, seconds of
        the slowest process)."""
        import oracle
        n, nt = len(grads), len(grads[0])
        counts = np.array([np.asarray(grads[0][t]).size for t in range(nt)], dtype=np.int64)
        bucket_of, _, bcount = oracle.bucket_plan(counts, dtype=dtype, cap_bytes=cap_bytes)
        # largest buckets first, each to the least-loaded process
        load = [0] * len(self.conns)
        share = [[] for _ in self.conns]
        for b in np.argsort(-bcount, kind="stable"):
            i = int(np.argmin(load))
            share[i].append(int(b))
            load[i] += int(bcount[b])
        kw = {"op": op, "dtype": dtype, "algo": algo, "cap_bytes": cap_bytes}
        sent = []
        for c, bs in zip(self.conns, share):
            if not bs:
                continue
            # each bucket's tensors alone, in registration order: planned
            # again they form exactly that bucket
            items, tids = [], []
            for b in bs:
                ts = [t for t in range(nt) if bucket_of[t] == b]
                items.append(([[grads[r][t] for t in ts] for r in range(n)], counts[ts], int(bcount[b])))
                tids.append(ts)
            c.send(("bucketed", items, kw))
            sent.append((c, tids))
        out = [[None] * nt for _ in range(n)]
        slowest = 0.0
        for c, tids in sent:
            res = c.recv()
            if res[0] != "ok":
                raise RuntimeError(f"oracle worker: {res}")
            slowest = max(slowest, res[1])
            for ts, dig in zip(tids, res[2]):
                for r in range(n):
                    for k, t in enumerate(ts):
                        out[r][t] = dig[r][k]
        return out, slowest

    def close(self):
        for c in self.conns:
            try:
                c.send(("stop",))
            except (BrokenPipeError, OSError):
                pass
        for p in self.procs:
            p.join(timeout=60)
        self.conns, self.procs = [], []
