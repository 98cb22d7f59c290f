"""CPU oracle for the simulated AllReduce (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The CUDA library never loads it
and shares no code with it.

The arithmetic and the message schedules live in ``ar_oracle.c`` (a literal
simulation of ranks exchanging messages, see the header of that file for the
passages each part follows).  This module compiles it with the system C
compiler and wraps it with numpy: bf16 values travel as ``uint16`` bit
patterns.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
against values and invariants fixed by the pages or by arithmetic (worked
examples, exact integer sums, library float32/bf16 additions in the stated
order, error bounds, step and volume counts).  The one convention the pages do
not pin is the ring's chunk rotation (which chunk each rank sends first):
every printed example is integer-valued, so order-free.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ar_oracle.c")
_LIB = os.path.join(_HERE, "libar_oracle.so")

MAX_RANKS = 256
DTYPES = {"f32": 0, "bf16": 1, "i32": 2, "f16": 3}
OPS = {"sum": 0, "max": 1, "avg": 2}
ALGOS = {"ring": 0, "tree": 1, "binomial": 2, "naive": 3, "dbtree": 4}
PHASE_RS, PHASE_AG = 1, 2
NP_STORAGE = {"f32": np.float32, "bf16": np.uint16, "i32": np.int32, "f16": np.uint16}

ERR_MISSING = -4


class Stats(ctypes.Structure):
    _fields_ = [
        ("steps", ctypes.c_int32),
        ("fail_step", ctypes.c_int32),
        ("fail_rank", ctypes.c_int32),
        ("pad", ctypes.c_int32),
        ("sent", ctypes.c_int64 * MAX_RANKS),
        ("recv", ctypes.c_int64 * MAX_RANKS),
    ]


class Fault(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("rank", ctypes.c_int32), ("step", ctypes.c_int32)]


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"oracle {what} failed with code {code}")
        self.code = code


def build(force: bool = False) -> str:
    """Compile ar_oracle.c into libar_oracle.so (plain C11, IEEE arithmetic:
    no fast-math, no floating-point contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
           "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        vp = ctypes.c_void_p
        L.oracle_collective.argtypes = [ctypes.c_int, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.c_int,
                                        ctypes.c_int64, ctypes.POINTER(ctypes.c_int64), ctypes.c_int64,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(Stats),
                                        ctypes.POINTER(Fault)]
        L.oracle_rooted.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.c_int,
                                    ctypes.c_int64, ctypes.POINTER(ctypes.c_int64), ctypes.c_int64, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.POINTER(Stats)]
        L.oracle_int8_ef_allreduce.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.c_int, ctypes.c_int64,
                                               ctypes.c_int, ctypes.POINTER(Stats)]
        L.oracle_step.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp, ctypes.c_int64]
        L.oracle_f32_to_bf16.argtypes = [vp, vp, ctypes.c_int64]
        L.oracle_f32_to_f16.argtypes = [vp, vp, ctypes.c_int64]
        L.oracle_f16_to_f32.argtypes = [vp, vp, ctypes.c_int64]
        L.oracle_chunk_range.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]
        L.oracle_bucket_plan.argtypes = [ctypes.POINTER(ctypes.c_int64), ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                         ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64),
                                         ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)]
        L.oracle_bucketed_allreduce.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(ctypes.c_int64),
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int64, ctypes.POINTER(ctypes.c_int32),
                                                ctypes.POINTER(ctypes.c_int64), ctypes.c_int64, vp,
                                                ctypes.POINTER(Stats)]
        _lib = L
    return _lib


def _ptrs(arrays):
    return (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])


def _check(x: np.ndarray, dtype: str) -> np.ndarray:
    want = NP_STORAGE[dtype]
    if x.dtype != want:
        raise TypeError(f"{dtype} values travel as {np.dtype(want).name}, got {x.dtype}")
    return np.ascontiguousarray(x)


def collective(x, *, algo="ring", op="sum", dtype="f32", phases=PHASE_RS | PHASE_AG, count=None,
               positions=None, fault=None, raise_on_error=True):
    """Run one simulated collective.

    ``x`` is an (N, m) array (or a list of N equal-length 1-D arrays): rank r's
    values.  Without ``positions`` m is the element count; with ``positions``
    (strictly increasing indices into a buffer of ``count`` elements) the ranks
    carry only those elements.  Returns ``(out, stats)`` with ``out`` shaped
    like ``x`` and ``stats`` a dict: ``steps``, ``sent``/``recv`` (elements per
    rank), ``fail_step``/``fail_rank`` and ``rc``.
    """
    xs = [_check(np.asarray(a), dtype) for a in x]
    n = len(xs)
    m = xs[0].shape[0] if n else 0
    if any(a.shape != (m,) for a in xs):
        raise ValueError("ranks must hold equal-length 1-D buffers")
    outs = [np.empty_like(a) for a in xs]
    pos_arr = None
    if positions is not None:
        pos_arr = np.ascontiguousarray(positions, dtype=np.int64)
        if pos_arr.shape != (m,):
            raise ValueError("one position per carried value")
        if count is None:
            raise ValueError("positions need the full element count")
    total = m if count is None else int(count)
    st = Stats()
    f = None
    if fault is not None:
        f = Fault(*fault)
    rc = lib().oracle_collective(
        ALGOS[algo], _ptrs(xs), _ptrs(outs), n, total,
        pos_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if pos_arr is not None else None,
        m, DTYPES[dtype], OPS[op], phases, ctypes.byref(st), ctypes.byref(f) if f is not None else None)
    stats = {"rc": rc, "steps": st.steps, "fail_step": st.fail_step, "fail_rank": st.fail_rank,
             "sent": np.array(st.sent[:n], dtype=np.int64), "recv": np.array(st.recv[:n], dtype=np.int64)}
    if rc != 0 and raise_on_error:
        raise OracleError(rc, "collective")
    return (np.stack(outs) if n else np.empty((0, 0), dtype=NP_STORAGE[dtype])), stats


def allreduce(x, **kw):
    return collective(x, phases=PHASE_RS | PHASE_AG, **kw)


def reduce_scatter(x, **kw):
    return collective(x, phases=PHASE_RS, **kw)


def all_gather(x, **kw):
    return collective(x, phases=PHASE_AG, **kw)


def _rooted(kind, x, *, algo="ring", op="sum", dtype="f32", root=0, count=None, positions=None,
            raise_on_error=True):
    xs = [_check(np.asarray(a), dtype) for a in x]
    n = len(xs)
    m = xs[0].shape[0] if n else 0
    outs = [np.empty_like(a) for a in xs]
    pos_arr = None
    if positions is not None:
        pos_arr = np.ascontiguousarray(positions, dtype=np.int64)
    total = m if count is None else int(count)
    st = Stats()
    rc = lib().oracle_rooted(kind, ALGOS[algo], _ptrs(xs), _ptrs(outs), n, total,
                             pos_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if pos_arr is not None else None,
                             m, DTYPES[dtype], OPS[op], root, ctypes.byref(st))
    stats = {"rc": rc, "steps": st.steps, "sent": np.array(st.sent[:n], dtype=np.int64),
             "recv": np.array(st.recv[:n], dtype=np.int64)}
    if rc != 0 and raise_on_error:
        raise OracleError(rc, "rooted collective")
    return np.stack(outs), stats


def reduce(x, *, root=0, **kw):
    """Reduce to `root` (ring, tree or naive order); only out[root] is the result."""
    return _rooted(0, x, root=root, **kw)


def broadcast(x, *, root=0, dtype="f32", **kw):
    """Copy the root's buffer to every rank."""
    return _rooted(1, x, root=root, dtype=dtype, **kw)


def int8_ef_allreduce(x, e, *, op="sum"):
    """8-bit quantised AllReduce with error feedback (see ar_oracle.c).
    ``x`` and ``e`` are (N, D) float32: gradients and residuals.  Returns
    (reduced x, new residuals, stats)."""
    xs = [np.array(a, dtype=np.float32, copy=True) for a in x]
    es = [np.array(a, dtype=np.float32, copy=True) for a in e]
    n = len(xs)
    st = Stats()
    rc = lib().oracle_int8_ef_allreduce(_ptrs(xs), _ptrs(es), n, xs[0].size if n else 0, OPS[op], ctypes.byref(st))
    if rc:
        raise OracleError(rc, "int8_ef_allreduce")
    stats = {"steps": st.steps, "sent": np.array(st.sent[:n], dtype=np.int64)}
    return np.stack(xs), np.stack(es), stats


def step(a, b, *, op="sum", dtype="f32"):
    """out[i] = step(a[i], b[i]) as a ring receiver applies it (a = received)."""
    a = _check(np.asarray(a), dtype)
    b = _check(np.asarray(b), dtype)
    out = np.empty_like(a)
    rc = lib().oracle_step(DTYPES[dtype], OPS[op], a.ctypes.data, b.ctypes.data, out.ctypes.data, a.size)
    if rc:
        raise OracleError(rc, "step")
    return out


def f32_to_bf16(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_f32_to_bf16(x.ctypes.data, out.ctypes.data, x.size)
    return out


def f32_to_f16(x):
    """binary32 -> binary16 bit patterns, round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_f32_to_f16(x.ctypes.data, out.ctypes.data, x.size)
    return out


def f16_to_f32(h):
    """binary16 bit patterns -> binary32 values (exact)."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    lib().oracle_f16_to_f32(h.ctypes.data, out.ctypes.data, h.size)
    return out


def chunk_range(count: int, nranks: int, c: int):
    lo, hi = ctypes.c_int64(), ctypes.c_int64()
    rc = lib().oracle_chunk_range(count, nranks, c, ctypes.byref(lo), ctypes.byref(hi))
    if rc:
        raise OracleError(rc, "chunk_range")
    return lo.value, hi.value


def bucket_plan(counts, *, dtype="f32", cap_bytes=25 << 20):
    counts = np.ascontiguousarray(counts, dtype=np.int64)
    t = counts.size
    bucket_of = np.zeros(max(t, 1), dtype=np.int32)
    offset = np.zeros(max(t, 1), dtype=np.int64)
    bcount = np.zeros(max(t, 1), dtype=np.int64)
    nb = ctypes.c_int32()
    rc = lib().oracle_bucket_plan(counts.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), t, DTYPES[dtype], cap_bytes,
                                  bucket_of.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                  offset.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                  bcount.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), ctypes.byref(nb))
    if rc:
        raise OracleError(rc, "bucket_plan")
    return bucket_of[:t], offset[:t], bcount[:nb.value]


def bucketed_allreduce(grads, *, op="avg", dtype="f32", algo="ring", cap_bytes=25 << 20, samples=None):
    """``grads[r][t]`` is rank r's tensor t (1-D).  Without ``samples`` returns
    the full result in the same nesting; with ``samples`` = (tensor_ids,
    indices) (distinct pairs) returns an (N, nsamp) array of results there."""
    n = len(grads)
    t = len(grads[0]) if n else 0
    flat = [_check(np.asarray(g).reshape(-1), dtype) for row in grads for g in row]
    counts = np.array([flat[i].size for i in range(t)], dtype=np.int64)
    st = Stats()
    vp = ctypes.c_void_p
    ins = (vp * len(flat))(*[a.ctypes.data for a in flat])
    if samples is None:
        outs_np = [np.empty_like(a) for a in flat]
        outs = (vp * len(flat))(*[a.ctypes.data for a in outs_np])
        rc = lib().oracle_bucketed_allreduce(ins, outs, counts.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), t, n,
                                             DTYPES[dtype], OPS[op], ALGOS[algo], cap_bytes, None, None, 0, None,
                                             ctypes.byref(st))
        if rc:
            raise OracleError(rc, "bucketed_allreduce")
        return [[outs_np[r * t + i] for i in range(t)] for r in range(n)], st
    tid = np.ascontiguousarray(samples[0], dtype=np.int32)
    idx = np.ascontiguousarray(samples[1], dtype=np.int64)
    out = np.empty((n, tid.size), dtype=NP_STORAGE[dtype])
    rc = lib().oracle_bucketed_allreduce(ins, (vp * max(len(flat), 1))(), counts.ctypes.data_as(
        ctypes.POINTER(ctypes.c_int64)), t, n, DTYPES[dtype], OPS[op], ALGOS[algo], cap_bytes,
        tid.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        tid.size, out.ctypes.data, ctypes.byref(st))
    if rc:
        raise OracleError(rc, "bucketed_allreduce")
    return out, st
