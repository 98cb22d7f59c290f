"""ar_allreduce_host: rank buffers in host memory, AllReduced through the GPU
in pieces whose upload, reduction and download overlap.  The result must be
the oracle's bit for bit, for any piece size, page-locked or pageable host
memory, and must be complete when the caller's stream is."""
import numpy as np
import pytest

import oracle
from allreduce_gradient_reduction_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ar():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from allreduce_gradient_reduction_gb300 import build as b
    b.build()
    from allreduce_gradient_reduction_gb300 import binding
    torch.cuda.set_device(0)
    return binding


TORCH_DT = {"f32": torch.float32, "bf16": torch.int16, "i32": torch.int32, "f16": torch.int16}
HALF = ("bf16", "f16")


def host_rows(x, dtype, pinned):
    a = np.ascontiguousarray(x)
    if dtype in HALF:
        a = a.view(np.int16)
    t = torch.from_numpy(a.copy())
    return t.pin_memory() if pinned else t


def as_np(t, dtype):
    a = t.numpy()
    return a.view(np.uint16) if dtype in HALF else a


def inputs(n, count, dtype, seed):
    if dtype == "i32":
        return W.uniform_inputs(n, count, "i32", config=seed)
    if dtype == "bf16":
        return W.large_inputs(n, count, config=seed)
    if dtype == "f16":
        return W.uniform_inputs(n, count, "f16", config=seed)
    return W.normal_inputs(n, count, 1.0, seed)


def same_bits(got, want, dtype):
    bits = {"bf16": np.uint16, "f16": np.uint16, "f32": np.uint32, "i32": np.uint32}[dtype]
    return np.array_equal(np.asarray(got).view(bits), np.asarray(want).view(bits))


@pytest.mark.parametrize("mode", ["staged", "zero_copy"])
@pytest.mark.parametrize("algo", ["ring", "tree", "naive", "dbtree"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
def test_host_allreduce_matches_oracle(ar, algo, dtype, mode):
    for n in (2, 3, 8, 16):
        if algo == "tree" and n & (n - 1):
            continue
        for count, piece in ((1, 0), (n * 64 + 5, 64), (4099, 100), (3 * 2048 * n + 13, 1000), (70_001, 0)):
            for op in ["sum", "max"] + ([] if dtype == "i32" else ["avg"]):
                x = inputs(n, count, dtype, seed=40 + n + count)
                with np.errstate(all="ignore"):
                    want, _ = oracle.allreduce(x, algo=algo, op=op, dtype=dtype)
                hb = host_rows(x, dtype, pinned=True)
                dv = None if mode == "zero_copy" else [torch.empty(count, dtype=TORCH_DT[dtype], device="cuda")
                                                       for _ in range(n)]
                ar.check(ar.ar_allreduce_host(list(hb), dv, count=count, dtype=dtype, op=op, algo=algo,
                                              piece_elems=piece), "host allreduce")
                torch.cuda.synchronize()
                got = as_np(hb, dtype)
                assert same_bits(got, want, dtype), (algo, dtype, op, n, count, piece)


@pytest.mark.parametrize("pinned", [True, False])
def test_host_allreduce_equals_device_call_for_every_piece_size(ar, pinned):
    n, count, dtype = 8, 8 * 4096 + 77, "bf16"
    x = inputs(n, count, dtype, seed=7)
    dv = [torch.from_numpy(np.ascontiguousarray(x[r]).view(np.int16)).cuda() for r in range(n)]
    ar.check(ar.ar_allreduce(dv, count=count, dtype=dtype, op="sum", algo="ring"), "device call")
    torch.cuda.synchronize()
    want = np.stack([t.cpu().numpy() for t in dv]).view(np.uint16)
    for piece in (0, 64, 128, 4096, 4095, count, 10 * count):
        hb = host_rows(x, dtype, pinned)
        work = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(n)]
        ar.check(ar.ar_allreduce_host(list(hb), work, count=count, dtype=dtype, op="sum", algo="ring",
                                      piece_elems=piece), "host allreduce")
        torch.cuda.synchronize()
        assert same_bits(as_np(hb, dtype), want, dtype), (pinned, piece)


@pytest.mark.parametrize("dtype,count", [("bf16", 5_000_001), ("f32", 3_000_000 + 17)])
def test_host_allreduce_default_pieces_on_large_rows(ar, dtype, count):
    """Large enough for the default schedule's small first and last pieces
    (the last three cut at an element count that is not a multiple of 64)."""
    n = 8
    x = inputs(n, count, dtype, seed=11)
    dv = [torch.from_numpy(np.ascontiguousarray(x[r]).view(np.int16 if dtype == "bf16" else np.float32)).cuda()
          for r in range(n)]
    ar.check(ar.ar_allreduce(dv, count=count, dtype=dtype, op="sum", algo="ring"), "device call")
    hb = host_rows(x, dtype, pinned=True)
    work = [torch.empty(count, dtype=TORCH_DT[dtype], device="cuda") for _ in range(n)]
    ar.check(ar.ar_allreduce_host(list(hb), work, count=count, dtype=dtype, op="sum", algo="ring"), "host allreduce")
    torch.cuda.synchronize()
    want = np.stack([t.cpu().numpy() for t in dv])
    assert same_bits(as_np(hb, dtype), want.view(np.uint16) if dtype == "bf16" else want, dtype)
    # sampled positions against the oracle, first and last elements included
    pos = np.unique(np.concatenate([[0, 1, count - 2, count - 1], np.random.default_rng(3).integers(0, count, 2000)]))
    want_s, _ = oracle.allreduce(np.ascontiguousarray(x[:, pos]), algo="ring", op="sum", dtype=dtype, positions=pos,
                                 count=count)
    assert same_bits(np.ascontiguousarray(as_np(hb, dtype)[:, pos]), want_s, dtype)


def test_host_allreduce_completes_with_the_callers_stream(ar):
    """Work already on the stream runs first (here: it writes the device
    buffers, which the uploads then overwrite), and synchronising only that
    stream is enough to read the result."""
    n, count = 4, 1 << 20
    x = W.normal_inputs(n, count, 1.0, 3)
    want, _ = oracle.allreduce(x, algo="ring", op="avg", dtype="f32")
    hb = host_rows(x, "f32", pinned=True)
    work = [torch.empty(count, dtype=torch.float32, device="cuda") for _ in range(n)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for t in work:
            t.fill_(123.0)
        ar.check(ar.ar_allreduce_host(list(hb), work, count=count, dtype="f32", op="avg", algo="ring",
                                      piece_elems=1 << 16, stream=s), "host allreduce")
    s.synchronize()
    assert same_bits(as_np(hb, "f32"), want, "f32")
    # a second call on the same buffers (each rank now holds the average)
    ar.check(ar.ar_allreduce_host(list(hb), work, count=count, dtype="f32", op="avg", algo="ring", stream=s),
             "second call")
    s.synchronize()
    want2, _ = oracle.allreduce(want, algo="ring", op="avg", dtype="f32")
    assert same_bits(as_np(hb, "f32"), want2, "f32")


@pytest.mark.parametrize("mode", ["staged", "zero_copy"])
def test_host_allreduce_stays_inside_its_buffers(ar, mode):
    """Rows carved out of one page-locked block between guard bands, at
    offsets that are element-aligned but not all 16-byte aligned: the bands
    (host and device side) must come back untouched and the rows correct."""
    guard, n = 4096, 3
    for count, shifts in ((1, [0, 1, 2]), (1001, [1, 1, 1]), (3 * 2048 + 7, [0, 3, 1]), (70_001, [2, 2, 2])):
        x = W.normal_inputs(n, count, 1.0, 60 + count)
        want, _ = oracle.allreduce(x, algo="ring", op="sum", dtype="f32")
        span = guard + count + 8 + guard
        block = torch.full((n, span), 7.5, dtype=torch.float32).pin_memory()
        rows = []
        for r in range(n):
            o = guard + shifts[r]
            block[r, o:o + count] = torch.from_numpy(x[r])
            rows.append(block[r, o:o + count])
        devblock = torch.full((n, span), -3.0, device="cuda")
        dv = None if mode == "zero_copy" else [devblock[r, guard + shifts[r]:guard + shifts[r] + count]
                                               for r in range(n)]
        ar.check(ar.ar_allreduce_host(rows, dv, count=count, dtype="f32", op="sum", algo="ring", piece_elems=640),
                 "host allreduce")
        torch.cuda.synchronize()
        for r in range(n):
            o = guard + shifts[r]
            assert same_bits(rows[r].numpy(), want[r], "f32"), (mode, count, shifts, r)
            assert bool((block[r, :o] == 7.5).all()) and bool((block[r, o + count:] == 7.5).all()), (mode, count, r)
            if dv is not None:
                d = devblock[r].cpu()
                assert bool((d[:o] == -3.0).all()) and bool((d[o + count:] == -3.0).all()), (mode, count, r)


def test_zero_copy_needs_mapped_page_locked_memory(ar):
    n, count = 4, 1000
    x = W.normal_inputs(n, count, 1.0, 21)
    want, _ = oracle.allreduce(x, algo="tree", op="sum", dtype="f32")
    pageable = host_rows(x, "f32", pinned=False)
    assert ar.ar_allreduce_host(list(pageable), None, count=count, algo="tree") == ar.AR_ERR_INVALID_ARG
    assert same_bits(as_np(pageable, "f32"), x, "f32")  # refused before any work
    on_device = [torch.zeros(count, device="cuda") for _ in range(n)]
    assert ar.ar_allreduce_host(on_device, None, count=count, algo="tree") == ar.AR_ERR_INVALID_ARG
    pinned = host_rows(x, "f32", pinned=True)
    assert ar.ar_allreduce_host([pinned[0], pinned[0], pinned[1], pinned[2]], None, count=count,
                                algo="tree") == ar.AR_ERR_INVALID_ARG  # duplicate
    # rows ending far past their page-locked allocation
    assert ar.ar_allreduce_host(list(pinned), None, count=count + 1_000_000, algo="tree") == ar.AR_ERR_INVALID_ARG
    ar.check(ar.ar_allreduce_host(list(pinned), None, count=count, algo="tree"), "zero copy")
    torch.cuda.synchronize()
    assert same_bits(as_np(pinned, "f32"), want, "f32")


def test_host_allreduce_argument_checks(ar):
    n, count = 2, 256
    hb = [torch.zeros(count).pin_memory() for _ in range(n)]
    work = [torch.empty(count, device="cuda") for _ in range(n)]
    assert ar.ar_allreduce_host(hb, work, count=count, algo="ring_stepwise") == ar.AR_ERR_UNSUPPORTED
    assert ar.ar_allreduce_host(hb, work, count=count, algo="tree_stepwise") == ar.AR_ERR_UNSUPPORTED
    assert ar.ar_allreduce_host(hb, [work[0], work[0]], count=count) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_allreduce_host([hb[0], hb[0]], work, count=count) == ar.AR_ERR_INVALID_ARG
    pinned_ws = [torch.zeros(count).pin_memory() for _ in range(n)]
    assert ar.ar_allreduce_host(hb, pinned_ws, count=count) == ar.AR_ERR_INVALID_ARG  # working space not on the device
    assert ar.ar_allreduce_host(hb, work, count=count, piece_elems=-1) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_allreduce_host(hb, work, count=0) == ar.AR_OK
