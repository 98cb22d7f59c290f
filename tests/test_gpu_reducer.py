"""The overlapped bucket reducer (ar_reducer_*): buckets start on a
communication stream while later gradients are still being produced on the
compute stream.  Its result must equal the CPU oracle's bucketed AllReduce
bit for bit, whatever order the gradients become ready in, and a bucket's
reduction must be enqueued exactly when its last gradient is marked ready and
every earlier bucket has started (DDP starts buckets in bucket order as soon
as they fill: "Allreduce：大模型分布式训练的核心通信算法与优化实践" §4.1
通信与计算重叠)."""
import numpy as np
import pytest

import oracle

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
ORACLE_ALGO = {"ring": "ring", "ring_stepwise": "ring", "tree": "tree"}


def host(n, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    return [[g.standard_normal(c).astype(np.float32) for c in COUNTS] for _ in range(n)]


def make(n, seed):
    return [[torch.from_numpy(t).cuda() for t in row] for row in host(n, seed)]


def started_after_each_mark(order, cap):
    """For marks in `order`: how many buckets may have started after each one
    -- the longest prefix of buckets (the oracle's plan) whose tensors are all
    marked."""
    bucket_of, _, bcount = oracle.bucket_plan(COUNTS, dtype="f32", cap_bytes=cap)
    left = np.bincount(bucket_of, minlength=bcount.size).tolist()
    started, out = 0, []
    for t in order:
        left[bucket_of[t]] -= 1
        while started < len(left) and left[started] == 0:
            started += 1
        out.append(started)
    return out


@pytest.mark.parametrize("algo", ["ring", "tree", "ring_stepwise"])
@pytest.mark.parametrize("order", ["reverse", "random", "forward"])
def test_reducer_matches_oracle(ar, algo, order):
    n, cap = 8, 4 * 3000
    compute, comm = torch.cuda.Stream(), torch.cuda.Stream()
    grads = make(n, 1)
    red = ar.Reducer(grads, counts=COUNTS, op="avg", algo=algo, bucket_cap_bytes=cap, comm_stream=comm)
    assert red.buckets == len(oracle.bucket_plan(COUNTS, dtype="f32", cap_bytes=cap)[2])
    if algo != "ring_stepwise":
        ar.check(red.set_max_blocks(3), "max blocks")  # few blocks striding: same results
    g = np.random.Generator(np.random.PCG64(2))
    for it in range(3):  # the handle is reused across iterations
        fresh_host = host(n, 10 + it)
        want, _ = oracle.bucketed_allreduce(fresh_host, op="avg", dtype="f32", algo=ORACLE_ALGO[algo],
                                            cap_bytes=cap)
        fresh = [[torch.from_numpy(t).cuda() for t in row] for row in fresh_host]
        torch.cuda.synchronize()
        idx = list(range(len(COUNTS)))[::-1] if order == "reverse" else (
            [int(i) for i in g.permutation(len(COUNTS))] if order == "random" else list(range(len(COUNTS))))
        expect_started = started_after_each_mark(idx, cap)
        started_launches = []
        with torch.cuda.stream(compute):
            l0 = ar.ar_kernel_launches()
            for t in idx:
                for r in range(n):  # "backward" writes rank r's gradient t on the compute stream
                    grads[r][t].copy_(fresh[r][t])
                ar.check(red.mark_ready(t, compute), "mark_ready")
                started_launches.append(ar.ar_kernel_launches() - l0)
            ar.check(red.finish(compute), "finish")
        compute.synchronize()
        # a bucket's kernels are enqueued at the mark that completes it (and
        # its predecessors), never before: launches grow exactly when the
        # count of startable buckets does
        prev_b, prev_l = 0, 0
        for k, (b, l) in enumerate(zip(expect_started, started_launches)):
            if b == prev_b:
                assert l == prev_l, (it, k, idx[k], b, l)
            else:
                assert l >= prev_l + (b - prev_b), (it, k, idx[k], b, l)
            prev_b, prev_l = b, l
        assert prev_b == red.buckets
        for r in range(n):
            for t in range(len(COUNTS)):
                got = grads[r][t].cpu().numpy().view(np.uint32)
                assert np.array_equal(got, want[r][t].view(np.uint32)), (it, r, t)
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
