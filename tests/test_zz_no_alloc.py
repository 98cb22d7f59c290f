"""GPU test of ar_bucketed_allreduce_noalloc, the entry point for callers
that are not allowed to allocate memory (a process whose device memory is
handed out by another allocator or a fixed pool, an engine that bans
allocation on its hot path because cudaMalloc can synchronise the device).

It must give exactly what ar_bucketed_allreduce gives on the same inputs, on
two calls in a row (the second one finds the scratch array holding the first
call's data), without taking any device memory during the call.  This file is
named so that pytest collects it last."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

N = 8
# A narrowed transformer block (width 256, GPT-2's 768 bias/norm vectors)
# plus ragged small tensors; every tensor fits the per-rank slice of the
# scratch (32 MiB / 8 ranks = 4 MiB), the two largest exceed the bucket cap
COUNTS = [768, 768, 256 * 2304, 2304, 256 * 768, 768, 768, 768, 256 * 3072, 3072, 5, 1001, 3, 4096 + 7]
CAP = 2 << 20


@pytest.fixture(scope="module")
def ar():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from allreduce_gradient_reduction_gb300 import build as b
    b.build()
    from allreduce_gradient_reduction_gb300 import binding
    torch.cuda.set_device(0)
    return binding


def make_grads(seed, dtype):
    g = np.random.Generator(np.random.PCG64(seed))
    out = []
    for _ in range(N):
        row = []
        for c in COUNTS:
            x = g.standard_normal(c).astype(np.float32) * np.float32(1e-3)
            if dtype == "bf16":
                x = (x.view(np.uint32) >> 16).astype(np.uint16).view(np.int16)
            elif dtype == "f16":
                x = x.astype(np.float16).view(np.int16)
            row.append(torch.from_numpy(x).cuda())
        out.append(row)
    return out


def bits(t):
    a = t.cpu().numpy()
    return a.view(np.uint16) if a.dtype == np.int16 else a.view(np.uint32)


@pytest.mark.parametrize("dtype,op,algo", [("f32", "avg", "ring"), ("bf16", "sum", "tree"), ("f16", "avg", "ring")])
def test_noalloc_matches_bucketed_allreduce_twice(ar, dtype, op, algo):
    for call in range(2):
        grads = make_grads(100 + call, dtype)
        ref = [[t.clone() for t in row] for row in grads]
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        rc = ar.ar_bucketed_allreduce_noalloc(grads, counts=COUNTS, dtype=dtype, op=op, algo=algo,
                                              bucket_cap_bytes=CAP)
        ar.check(rc, "noalloc")
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        if call == 1:
            assert free_after == free_before  # nothing was allocated on the device
        ar.check(ar.ar_bucketed_allreduce(ref, counts=COUNTS, dtype=dtype, op=op, algo=algo,
                                          bucket_cap_bytes=CAP), "reference entry point")
        torch.cuda.synchronize()
        for r in range(N):
            for t in range(len(COUNTS)):
                got, want = bits(grads[r][t]), bits(ref[r][t])
                nan_g = np.isnan(got.view(np.float32)) if dtype == "f32" else np.zeros(got.shape, bool)
                assert np.array_equal(got[~nan_g], want[~nan_g]), (call, r, t)


def test_noalloc_rejects_what_does_not_fit(ar):
    big = [torch.zeros(2 << 20, dtype=torch.float32, device="cuda") for _ in range(N)]  # 8 MiB each > 4 MiB slice
    rc = ar.ar_bucketed_allreduce_noalloc([[b] for b in big], counts=[2 << 20], dtype="f32", op="avg")
    assert rc == -6  # AR_ERR_TOO_LARGE
    small = [[torch.zeros(16, device="cuda")] for _ in range(N)]
    assert ar.ar_bucketed_allreduce_noalloc(small, counts=[16], algo="ring_stepwise") == ar.AR_ERR_UNSUPPORTED
    many = [[torch.zeros(1, device="cuda") for _ in range(1025)] for _ in range(2)]
    assert ar.ar_bucketed_allreduce_noalloc(many, counts=[1] * 1025) == -6
