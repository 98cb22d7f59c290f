"""Python binding of libar_gb300.so (include/ar.h): argument marshalling only.

Every function takes the same arguments as its C counterpart.  Where the C
function takes an array of device pointers, this binding accepts a sequence of
torch CUDA tensors (their data pointers are passed) or plain integers.  Enum
arguments accept the C value or its lower-case name ("f32", "sum", "ring",
...).  A stream is a torch.cuda.Stream, an integer cudaStream_t, or None (the
current torch stream).  Each call returns the C status; ``check()`` raises
ArError on a non-zero one.

Loading fails loudly: without the compiled library there is no fallback.
"""
from __future__ import annotations

import array
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libar_gb300.so")

DTYPE = {"f32": 0, "bf16": 1, "i32": 2, "f16": 3}
OP = {"sum": 0, "max": 1, "avg": 2}
ALGO = {"ring": 0, "ring_stepwise": 1, "tree": 2, "tree_stepwise": 3, "naive": 4, "dbtree": 5,
        "binomial_stepwise": 6}
STATUS = {0: "AR_OK", -1: "AR_ERR_INVALID_ARG", -2: "AR_ERR_UNSUPPORTED", -3: "AR_ERR_CUDA",
          -4: "AR_ERR_TIMEOUT", -5: "AR_ERR_NO_DEVICE", -6: "AR_ERR_TOO_LARGE", -7: "AR_ERR_HOST"}
AR_OK, AR_ERR_INVALID_ARG, AR_ERR_UNSUPPORTED, AR_ERR_CUDA, AR_ERR_TIMEOUT = 0, -1, -2, -3, -4
MAX_RANKS = 64
MAX_COUNT = 1 << 56  # AR_MAX_COUNT
DEFAULT_BUCKET_CAP_BYTES = 25 << 20

EXPORTS = ("ar_allreduce", "ar_reduce_scatter", "ar_all_gather", "ar_reduce", "ar_broadcast", "ar_allreduce_int8_ef",
           "ar_allreduce_host",
           "ar_bucket_plan",
           "ar_bucketed_allreduce",
           "ar_bucketed_allreduce_noalloc", "ar_chunk_range", "ar_device_status", "ar_set_barrier_timeout_ns", "ar_debug_skip_barrier",
           "ar_last_cuda_error", "ar_strerror", "ar_version", "ar_kernel_launches", "ar_reducer_create",
           "ar_reducer_mark_ready", "ar_reducer_finish", "ar_reducer_destroy", "ar_reducer_buckets",
           "ar_reducer_set_max_blocks", "ar_plan_create", "ar_plan_run", "ar_plan_destroy")


class ArError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        super().__init__(f"{what}: {STATUS.get(code, code)} ({code})")
        self.code = code


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(the CUDA library is required; there is no CPU fallback)")
    L = ctypes.CDLL(LIB_PATH)
    i64, i32, vp, cint = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int
    pp = ctypes.POINTER(vp)
    L.ar_allreduce.argtypes = [pp, cint, i64, cint, cint, cint, vp]
    L.ar_reduce_scatter.argtypes = [pp, cint, i64, cint, cint, cint, vp]
    L.ar_all_gather.argtypes = [pp, cint, i64, cint, cint, vp]
    L.ar_reduce.argtypes = [pp, cint, i64, cint, cint, cint, cint, vp]
    L.ar_broadcast.argtypes = [pp, cint, i64, cint, cint, vp]
    L.ar_allreduce_int8_ef.argtypes = [pp, pp, cint, i64, cint, vp]
    L.ar_allreduce_host.argtypes = [pp, pp, cint, i64, cint, cint, cint, i64, vp]
    L.ar_bucket_plan.argtypes = [ctypes.POINTER(i64), cint, cint, i64, ctypes.POINTER(i32), ctypes.POINTER(i64),
                                 ctypes.POINTER(i64), ctypes.POINTER(i32)]
    L.ar_bucketed_allreduce.argtypes = [pp, ctypes.POINTER(i64), cint, cint, cint, cint, cint, i64, pp, i64, vp]
    L.ar_bucketed_allreduce_noalloc.argtypes = [pp, ctypes.POINTER(i64), cint, cint, cint, cint, cint, i64, vp]
    L.ar_chunk_range.argtypes = [i64, cint, cint, ctypes.POINTER(i64), ctypes.POINTER(i64)]
    L.ar_device_status.argtypes = [vp, ctypes.POINTER(cint)]
    L.ar_set_barrier_timeout_ns.argtypes = [i64]
    L.ar_debug_skip_barrier.argtypes = [cint]
    L.ar_last_cuda_error.argtypes = []
    L.ar_strerror.argtypes = [cint]
    L.ar_strerror.restype = ctypes.c_char_p
    L.ar_version.argtypes = []
    L.ar_kernel_launches.argtypes = []
    L.ar_reducer_create.argtypes = [pp, ctypes.POINTER(i64), cint, cint, cint, cint, cint, i64, vp,
                                    ctypes.POINTER(vp)]
    L.ar_reducer_mark_ready.argtypes = [vp, cint, vp]
    L.ar_reducer_finish.argtypes = [vp, vp]
    L.ar_reducer_destroy.argtypes = [vp]
    L.ar_reducer_buckets.argtypes = [vp]
    L.ar_reducer_set_max_blocks.argtypes = [vp, cint]
    L.ar_plan_create.argtypes = [cint, pp, cint, i64, cint, cint, cint, cint, ctypes.POINTER(vp)]
    L.ar_plan_run.argtypes = [vp, vp]
    L.ar_plan_destroy.argtypes = [vp]
    for name in EXPORTS:
        if name != "ar_strerror":
            getattr(L, name).restype = cint
    L.ar_kernel_launches.restype = i64
    return L


lib = _load()


def _enum(table, v):
    return table[v] if isinstance(v, str) else int(v)


def _ptr(x) -> int:
    if isinstance(x, int):
        return x
    if x is None:
        return 0
    return int(x.data_ptr())


_ARRAY_TYPES = {}


def _ptr_array(xs):
    """A C array of the addresses of xs (tensors, addresses or None), built
    over an array of 64-bit words: at 64 ranks about half the cost of ctypes'
    element-by-element constructor."""
    n = max(len(xs), 1)
    t = _ARRAY_TYPES.get(n)
    if t is None:
        t = _ARRAY_TYPES[n] = ctypes.c_void_p * n
    try:
        addrs = [x.data_ptr() for x in xs]
    except AttributeError:
        addrs = [_ptr(x) for x in xs]
    return t.from_buffer(array.array("Q", addrs or [0]))


def _stream(s) -> int:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _count(bufs, count):
    if count is not None:
        return int(count)
    return int(bufs[0].numel()) if len(bufs) and not isinstance(bufs[0], int) else 0


def check(rc: int, what: str = "ar") -> int:
    if rc != AR_OK:
        raise ArError(rc, what)
    return rc


def ar_allreduce(bufs, nranks=None, count=None, dtype="f32", op="sum", algo="ring", stream=None) -> int:
    n = len(bufs) if nranks is None else int(nranks)
    return lib.ar_allreduce(_ptr_array(bufs), n, _count(bufs, count), _enum(DTYPE, dtype), _enum(OP, op),
                            _enum(ALGO, algo), _stream(stream))


def ar_reduce_scatter(bufs, nranks=None, count=None, dtype="f32", op="sum", algo="ring", stream=None) -> int:
    n = len(bufs) if nranks is None else int(nranks)
    return lib.ar_reduce_scatter(_ptr_array(bufs), n, _count(bufs, count), _enum(DTYPE, dtype), _enum(OP, op),
                                 _enum(ALGO, algo), _stream(stream))


def ar_all_gather(bufs, nranks=None, count=None, dtype="f32", algo="ring", stream=None) -> int:
    n = len(bufs) if nranks is None else int(nranks)
    return lib.ar_all_gather(_ptr_array(bufs), n, _count(bufs, count), _enum(DTYPE, dtype), _enum(ALGO, algo),
                             _stream(stream))


def ar_reduce(bufs, nranks=None, count=None, dtype="f32", op="sum", algo="ring", root=0, stream=None) -> int:
    n = len(bufs) if nranks is None else int(nranks)
    return lib.ar_reduce(_ptr_array(bufs), n, _count(bufs, count), _enum(DTYPE, dtype), _enum(OP, op),
                         _enum(ALGO, algo), int(root), _stream(stream))


def ar_broadcast(bufs, nranks=None, count=None, dtype="f32", root=0, stream=None) -> int:
    n = len(bufs) if nranks is None else int(nranks)
    return lib.ar_broadcast(_ptr_array(bufs), n, _count(bufs, count), _enum(DTYPE, dtype), int(root),
                            _stream(stream))


def ar_allreduce_host(host_bufs, dev_bufs=None, nranks=None, count=None, dtype="f32", op="sum", algo="ring",
                      piece_elems=0, stream=None) -> int:
    """host_bufs: CPU tensors or host addresses.  dev_bufs None: zero-copy on
    page-locked host buffers; else device working buffers (staged pieces)."""
    n = len(host_bufs) if nranks is None else int(nranks)
    return lib.ar_allreduce_host(_ptr_array(host_bufs), None if dev_bufs is None else _ptr_array(dev_bufs), n,
                                 _count(host_bufs, count),
                                 _enum(DTYPE, dtype), _enum(OP, op), _enum(ALGO, algo), int(piece_elems),
                                 _stream(stream))


def ar_allreduce_int8_ef(grads, residuals, nranks=None, count=None, op="sum", stream=None) -> int:
    n = len(grads) if nranks is None else int(nranks)
    return lib.ar_allreduce_int8_ef(_ptr_array(grads), _ptr_array(residuals), n, _count(grads, count),
                                    _enum(OP, op), _stream(stream))


def ar_bucket_plan(counts, dtype="f32", cap_bytes=DEFAULT_BUCKET_CAP_BYTES):
    """Returns (status, bucket_of_tensor, offset_in_bucket, bucket_count) as lists."""
    t = len(counts)
    c = (ctypes.c_int64 * max(t, 1))(*[int(x) for x in counts])
    bo = (ctypes.c_int32 * max(t, 1))()
    off = (ctypes.c_int64 * max(t, 1))()
    bc = (ctypes.c_int64 * max(t, 1))()
    nb = ctypes.c_int32()
    rc = lib.ar_bucket_plan(c, t, _enum(DTYPE, dtype), int(cap_bytes), bo, off, bc, ctypes.byref(nb))
    return rc, list(bo[:t]), list(off[:t]), list(bc[:nb.value])


def ar_bucketed_allreduce(grads, counts=None, ntensors=None, nranks=None, dtype="f32", op="avg", algo="ring",
                          bucket_cap_bytes=DEFAULT_BUCKET_CAP_BYTES, workspace=None, workspace_bytes=0,
                          stream=None) -> int:
    """``grads`` is a list over ranks of lists over tensors (or a flat
    row-major list with ``ntensors``/``nranks`` given)."""
    if len(grads) and isinstance(grads[0], (list, tuple)):
        nr, nt = len(grads), len(grads[0])
        flat = [g for row in grads for g in row]
        if counts is None:
            counts = [int(g.numel()) for g in grads[0]]
    else:
        nr, nt, flat = int(nranks), int(ntensors), list(grads)
    c = (ctypes.c_int64 * max(nt, 1))(*[int(x) for x in counts])
    ws = _ptr_array(workspace) if workspace is not None else None
    if workspace is not None and workspace_bytes == 0 and not isinstance(workspace[0], int):
        workspace_bytes = int(workspace[0].numel() * workspace[0].element_size())
    return lib.ar_bucketed_allreduce(_ptr_array(flat), c, nt, nr, _enum(DTYPE, dtype), _enum(OP, op),
                                     _enum(ALGO, algo), int(bucket_cap_bytes), ws, int(workspace_bytes),
                                     _stream(stream))


def ar_bucketed_allreduce_noalloc(grads, counts=None, ntensors=None, nranks=None, dtype="f32", op="avg",
                                  algo="ring", bucket_cap_bytes=DEFAULT_BUCKET_CAP_BYTES, stream=None) -> int:
    """Same arguments as ar_bucketed_allreduce without the workspace: the
    library's fixed scratch array stands in for it (see include/ar.h)."""
    if len(grads) and isinstance(grads[0], (list, tuple)):
        nr, nt = len(grads), len(grads[0])
        flat = [g for row in grads for g in row]
        if counts is None:
            counts = [int(g.numel()) for g in grads[0]]
    else:
        nr, nt, flat = int(nranks), int(ntensors), list(grads)
    c = (ctypes.c_int64 * max(nt, 1))(*[int(x) for x in counts])
    return lib.ar_bucketed_allreduce_noalloc(_ptr_array(flat), c, nt, nr, _enum(DTYPE, dtype), _enum(OP, op),
                                             _enum(ALGO, algo), int(bucket_cap_bytes), _stream(stream))


NOALLOC_SCRATCH_BYTES = 32 << 20
NOALLOC_MAX_TENSORS = 1024


class Reducer:
    """Overlapped bucket reduction (ar_reducer_*): create once over the
    gradient tensors, then per iteration ``mark_ready(t, stream)`` for every
    tensor as its gradients are produced and ``finish(stream)``."""

    def __init__(self, grads, counts=None, dtype="f32", op="avg", algo="ring",
                 bucket_cap_bytes=DEFAULT_BUCKET_CAP_BYTES, comm_stream=None):
        nr, nt = len(grads), len(grads[0])
        flat = [g for row in grads for g in row]
        if counts is None:
            counts = [int(g.numel()) for g in grads[0]]
        c = (ctypes.c_int64 * max(nt, 1))(*[int(x) for x in counts])
        h = ctypes.c_void_p()
        check(lib.ar_reducer_create(_ptr_array(flat), c, nt, nr, _enum(DTYPE, dtype), _enum(OP, op),
                                    _enum(ALGO, algo), int(bucket_cap_bytes), _stream(comm_stream), ctypes.byref(h)),
              "ar_reducer_create")
        self.handle = h
        self.ntensors = nt

    @property
    def buckets(self) -> int:
        return lib.ar_reducer_buckets(self.handle)

    def set_max_blocks(self, max_blocks: int) -> int:
        return lib.ar_reducer_set_max_blocks(self.handle, int(max_blocks))

    def mark_ready(self, tensor: int, stream=None) -> int:
        return lib.ar_reducer_mark_ready(self.handle, int(tensor), _stream(stream))

    def finish(self, stream=None) -> int:
        return lib.ar_reducer_finish(self.handle, _stream(stream))

    def close(self):
        if self.handle:
            lib.ar_reducer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


PLAN_KIND = {"allreduce": 0, "reduce_scatter": 1, "all_gather": 2, "reduce": 3}


class Plan:
    """A prepared collective (ar_plan_*): arguments checked and launch tables
    built once; ``run(stream)`` only enqueues the kernels."""

    def __init__(self, kind, bufs, count=None, dtype="f32", op="sum", algo="ring", root=0):
        h = ctypes.c_void_p()
        check(lib.ar_plan_create(PLAN_KIND[kind] if isinstance(kind, str) else int(kind), _ptr_array(bufs),
                                 len(bufs), _count(bufs, count), _enum(DTYPE, dtype), _enum(OP, op), _enum(ALGO, algo),
                                 int(root), ctypes.byref(h)), "ar_plan_create")
        self.handle = h

    def run(self, stream=None) -> int:
        return lib.ar_plan_run(self.handle, _stream(stream))

    def close(self):
        if self.handle:
            lib.ar_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def ar_chunk_range(count, nranks, c):
    lo, hi = ctypes.c_int64(), ctypes.c_int64()
    rc = lib.ar_chunk_range(int(count), int(nranks), int(c), ctypes.byref(lo), ctypes.byref(hi))
    return rc, lo.value, hi.value


def ar_device_status(stream=None):
    """Returns (status of the call, asynchronous device status)."""
    st = ctypes.c_int()
    rc = lib.ar_device_status(_stream(stream), ctypes.byref(st))
    return rc, st.value


def ar_set_barrier_timeout_ns(ns: int) -> int:
    return lib.ar_set_barrier_timeout_ns(int(ns))


def ar_debug_skip_barrier(barrier: int) -> int:
    return lib.ar_debug_skip_barrier(int(barrier))


def ar_last_cuda_error() -> int:
    return lib.ar_last_cuda_error()


def ar_strerror(code: int) -> str:
    return lib.ar_strerror(int(code)).decode()


def ar_version() -> int:
    return lib.ar_version()


def ar_kernel_launches() -> int:
    return lib.ar_kernel_launches()
