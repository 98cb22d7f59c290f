"""Prepared collectives (ar_plan_*) and CUDA-graph capture: both must give
exactly what the direct call gives."""
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


def dev(x):
    a = np.ascontiguousarray(x)
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()


def host(bufs, dtype):
    out = np.stack([b.cpu().numpy() for b in bufs])
    return out.view(np.uint16) if dtype == "bf16" else out


@pytest.mark.parametrize("kind,algo", [("allreduce", "ring"), ("allreduce", "tree"), ("allreduce", "ring_stepwise"),
                                       ("allreduce", "dbtree"), ("reduce_scatter", "ring"),
                                       ("all_gather", "tree"), ("reduce", "naive")])
def test_plan_matches_oracle_over_repeated_runs(ar, kind, algo):
    n, count, dtype = 8, 3 * 4096 * 8 + 5, "bf16"
    bufs = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(n)]
    plan = ar.Plan(kind, bufs, count=count, dtype=dtype, op="sum", algo=algo, root=3)
    ref_algo = {"ring_stepwise": "ring"}.get(algo, algo)
    for it in range(3):  # same buffers, new data each run
        x = W.large_inputs(n, count, config=3000 + it)
        for r in range(n):
            bufs[r].copy_(dev(x[r]))
        ar.check(plan.run(), "plan run")
        got = host(bufs, dtype)
        if kind == "allreduce":
            want, _ = oracle.allreduce(x, algo=ref_algo, dtype=dtype)
            assert np.array_equal(got, want)
        elif kind == "reduce_scatter":
            want, _ = oracle.reduce_scatter(x, algo=ref_algo, dtype=dtype)
            for r in range(n):
                lo, hi = oracle.chunk_range(count, n, r)
                assert np.array_equal(got[r, lo:hi], want[r, lo:hi])
        elif kind == "all_gather":
            want, _ = oracle.all_gather(x, algo=ref_algo, dtype=dtype)
            assert np.array_equal(got, want)
        else:
            want, _ = oracle.reduce(x, algo=ref_algo, dtype=dtype, root=3)
            assert np.array_equal(got[3], want[3])
    plan.close()


def test_plan_rejects_bad_arguments(ar):
    bufs = [torch.zeros(16, device="cuda") for _ in range(3)]
    with pytest.raises(ar.ArError):
        ar.Plan("allreduce", bufs, algo="tree")  # three ranks: no tree
    with pytest.raises(ar.ArError):
        ar.Plan("reduce", bufs, root=5)
    with pytest.raises(ar.ArError):
        ar.Plan("allreduce", [bufs[0], bufs[0], bufs[1]])  # duplicate buffer


@pytest.mark.parametrize("algo", ["ring", "tree", "ring_stepwise", "tree_stepwise"])
def test_allreduce_replayed_from_a_cuda_graph(ar, algo):
    n, count = 8, 1 << 18
    x = W.normal_inputs(n, count, 1.0, 44)
    bufs = [dev(x[r]) for r in range(n)]
    plan = ar.Plan("allreduce", bufs, count=count, algo=algo)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    # warm-up outside the capture: any one-time set-up (the barrier block) happens here
    ar.check(ar.ar_allreduce(bufs, count=count, algo=algo, stream=side), "warm-up call")
    ar.check(plan.run(side), "warm-up plan")
    side.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        ar.check(ar.ar_allreduce(bufs, count=count, algo=algo, stream=side), "captured call")
        ar.check(plan.run(side), "captured plan")
    for it in range(2):
        x = W.normal_inputs(n, count, 1.0, 45 + it)
        for r in range(n):
            bufs[r].copy_(dev(x[r]))
        g.replay()
        torch.cuda.synchronize()
        once, _ = oracle.allreduce(x, algo=algo.replace("_stepwise", ""), dtype="f32")
        twice, _ = oracle.allreduce(once, algo=algo.replace("_stepwise", ""), dtype="f32")  # two calls in the graph
        assert np.array_equal(host(bufs, "f32"), twice)
    rc, st = ar.ar_device_status()
    assert rc == 0 and st == 0
    plan.close()
