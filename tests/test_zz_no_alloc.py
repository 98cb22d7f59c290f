"""GPU test of ar_bucketed_allreduce_noalloc, the entry point for callers
that are not allowed to allocate memory (a process whose device memory is
handed out by another allocator or a fixed pool, an engine that bans
allocation on its hot path because cudaMalloc can synchronise the device).

On two calls in a row (the second one finds the scratch array holding the
first call's data) it must give, bit for bit, what the CPU oracle's bucketed
AllReduce gives, and what ar_bucketed_allreduce gives on the same inputs,
without taking any device memory during the call.  The cases cover the
compiled and the runtime-N ring (N = 8, 3, 5), the tree, every dtype, SUM,
AVG and MAX, and buckets just inside and just past the per-rank slice of the
scratch at a rank count that does not divide it.  This file is named so that
pytest collects it last."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SCRATCH = 32 << 20  # AR_NOALLOC_SCRATCH_BYTES
# A narrowed transformer block (width 256, GPT-2's 768 bias/norm vectors)
# plus ragged small tensors; every tensor fits the per-rank slice of the
# scratch (32 MiB / 8 ranks = 4 MiB), the two largest exceed the bucket cap
COUNTS = [768, 768, 256 * 2304, 2304, 256 * 768, 768, 768, 768, 256 * 3072, 3072, 5, 1001, 3, 4096 + 7]
CAP = 2 << 20
ES = {"f32": 4, "i32": 4, "bf16": 2, "f16": 2}


@pytest.fixture(scope="module")
def ar():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from allreduce_gradient_reduction_gb300 import build as b
    b.build()
    from allreduce_gradient_reduction_gb300 import binding
    torch.cuda.set_device(0)
    return binding


def host_grads(n, counts, seed, dtype):
    """Rank r's tensors as numpy arrays in the oracle's storage types."""
    g = np.random.Generator(np.random.PCG64(seed))
    out = []
    for _ in range(n):
        row = []
        for c in counts:
            if dtype == "i32":
                row.append(g.integers(-(1 << 20), 1 << 20, size=c, dtype=np.int32))
                continue
            x = g.standard_normal(c).astype(np.float32) * np.float32(1e-3)
            if dtype == "bf16":
                x = (x.view(np.uint32) >> 16).astype(np.uint16)
            elif dtype == "f16":
                x = x.astype(np.float16).view(np.uint16)
            row.append(x)
        out.append(row)
    return out


def to_dev(a):
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()


def bits(a):
    return a.view(np.uint16) if a.dtype in (np.int16, np.uint16) else a.view(np.uint32)


def run_twice(ar, n, counts, dtype, op, algo, cap):
    for call in range(2):
        host = host_grads(n, counts, 100 + 7 * call + n, dtype)
        want, _ = oracle.bucketed_allreduce(host, op=op, dtype=dtype, algo=algo, cap_bytes=cap)
        grads = [[to_dev(t) for t in row] for row in host]
        ref = [[to_dev(t) for t in row] for row in host]
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        ar.check(ar.ar_bucketed_allreduce_noalloc(grads, counts=counts, dtype=dtype, op=op, algo=algo,
                                                  bucket_cap_bytes=cap), "noalloc")
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        if call == 1:
            assert free_after == free_before  # nothing was allocated on the device
        ar.check(ar.ar_bucketed_allreduce(ref, counts=counts, dtype=dtype, op=op, algo=algo,
                                          bucket_cap_bytes=cap), "ar_bucketed_allreduce")
        torch.cuda.synchronize()
        for r in range(n):
            for t in range(len(counts)):
                got = bits(grads[r][t].cpu().numpy())
                assert np.array_equal(got, bits(want[r][t])), ("oracle", call, r, t)
                assert np.array_equal(got, bits(ref[r][t].cpu().numpy())), ("entry point", call, r, t)


@pytest.mark.parametrize("n,dtype,op,algo", [(8, "f32", "avg", "ring"), (8, "bf16", "sum", "tree"),
                                             (8, "f16", "avg", "ring"), (3, "f32", "max", "ring"),
                                             (2, "i32", "sum", "ring"), (5, "bf16", "avg", "ring")])
def test_noalloc_matches_oracle_and_bucketed_allreduce_twice(ar, n, dtype, op, algo):
    run_twice(ar, n, COUNTS, dtype, op, algo, CAP)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_noalloc_slice_boundary_at_three_ranks(ar, dtype):
    """32 MiB / 3 ranks = 11,184,640 bytes (a multiple of 256): a bucket of
    exactly that many bytes still fits the rank's slice, one element more
    does not."""
    n = 3
    slice_bytes = (SCRATCH // n) & ~255
    fit = slice_bytes // ES[dtype]
    counts = [fit - 1001, 1001]  # one bucket of exactly the slice
    run_twice(ar, n, counts, dtype, "avg", "ring", slice_bytes)
    over = [torch.zeros(fit + 1, dtype=torch.float32 if dtype == "f32" else torch.int16, device="cuda")
            for _ in range(n)]
    rc = ar.ar_bucketed_allreduce_noalloc([[b] for b in over], counts=[fit + 1], dtype=dtype, op="avg",
                                          bucket_cap_bytes=slice_bytes + 64)
    assert rc == -6  # AR_ERR_TOO_LARGE


def test_noalloc_rejects_what_does_not_fit(ar):
    n = 8
    big = [torch.zeros(2 << 20, dtype=torch.float32, device="cuda") for _ in range(n)]  # 8 MiB each > 4 MiB slice
    rc = ar.ar_bucketed_allreduce_noalloc([[b] for b in big], counts=[2 << 20], dtype="f32", op="avg")
    assert rc == -6  # AR_ERR_TOO_LARGE
    small = [[torch.zeros(16, device="cuda")] for _ in range(n)]
    for algo in ("ring_stepwise", "tree_stepwise", "naive", "dbtree"):
        assert ar.ar_bucketed_allreduce_noalloc(small, counts=[16], algo=algo) == ar.AR_ERR_UNSUPPORTED, algo
    # the same answers as ar_bucketed_allreduce for the orders it does not take
    for algo in ("naive", "dbtree"):
        assert ar.ar_bucketed_allreduce(small, counts=[16], algo=algo) == ar.AR_ERR_UNSUPPORTED, algo
    assert ar.ar_bucketed_allreduce_noalloc(small, counts=[16], algo=99) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_bucketed_allreduce_noalloc(small, counts=[16], dtype="i32", op="avg") == ar.AR_ERR_UNSUPPORTED
    three = [[torch.zeros(16, device="cuda")] for _ in range(3)]
    assert ar.ar_bucketed_allreduce_noalloc(three, counts=[16], algo="tree") == ar.AR_ERR_UNSUPPORTED
    many = [[torch.zeros(1, device="cuda") for _ in range(1025)] for _ in range(2)]
    assert ar.ar_bucketed_allreduce_noalloc(many, counts=[1] * 1025) == -6
