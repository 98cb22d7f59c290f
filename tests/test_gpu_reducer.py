"""The overlapped bucket reducer (ar_reducer_*): buckets start on a
communication stream while later gradients are still being produced on the
compute stream; the result must equal ar_bucketed_allreduce bit for bit,
whatever order the gradients become ready in."""
import numpy as np
import pytest

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


COUNTS = [5, 300, 17, 1024, 3, 999, 64, 4096 + 3, 1, 2048, 0, 777, 65536, 12]


def make(n, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    return [[torch.from_numpy(g.standard_normal(c).astype(np.float32)).cuda() for c in COUNTS] for _ in range(n)]


@pytest.mark.parametrize("algo", ["ring", "tree", "ring_stepwise"])
@pytest.mark.parametrize("order", ["reverse", "random", "forward"])
def test_reducer_matches_bucketed_allreduce(ar, algo, order):
    n, cap = 8, 4 * 3000
    compute, comm = torch.cuda.Stream(), torch.cuda.Stream()
    grads = make(n, 1)
    red = ar.Reducer(grads, counts=COUNTS, op="avg", algo=algo, bucket_cap_bytes=cap, comm_stream=comm)
    assert red.buckets == len(ar.ar_bucket_plan(COUNTS, "f32", cap)[3])
    if algo != "ring_stepwise":
        ar.check(red.set_max_blocks(3), "max blocks")  # few blocks striding: same results
    g = np.random.Generator(np.random.PCG64(2))
    for it in range(3):  # the handle is reused across iterations
        fresh = make(n, 10 + it)
        ref = [[t.clone() for t in row] for row in fresh]
        torch.cuda.synchronize()
        idx = list(range(len(COUNTS)))[::-1] if order == "reverse" else (
            list(g.permutation(len(COUNTS))) if order == "random" else list(range(len(COUNTS))))
        with torch.cuda.stream(compute):
            for t in idx:
                for r in range(n):  # "backward" writes rank r's gradient t on the compute stream
                    grads[r][t].copy_(fresh[r][t])
                ar.check(red.mark_ready(t, compute), "mark_ready")
            ar.check(red.finish(compute), "finish")
        compute.synchronize()
        ar.check(ar.ar_bucketed_allreduce(ref, counts=COUNTS, op="avg", algo=algo, bucket_cap_bytes=cap), "ref")
        torch.cuda.synchronize()
        for r in range(n):
            for t in range(len(COUNTS)):
                assert torch.equal(grads[r][t], ref[r][t]), (it, r, t)
    red.close()


def test_reducer_rejects_misuse(ar):
    n = 2
    grads = make(n, 3)
    red = ar.Reducer(grads, counts=COUNTS, bucket_cap_bytes=4 * 3000)
    s = torch.cuda.current_stream()
    assert red.mark_ready(0, s) == 0
    assert red.mark_ready(0, s) == ar.AR_ERR_INVALID_ARG  # marked twice
    assert red.finish(s) == ar.AR_ERR_INVALID_ARG         # others never marked
    assert red.mark_ready(len(COUNTS), s) == ar.AR_ERR_INVALID_ARG
    for t in range(1, len(COUNTS)):
        assert red.mark_ready(t, s) == 0
    assert red.finish(s) == 0
    torch.cuda.synchronize()
    red.close()
