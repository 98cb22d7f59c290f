"""Parity of the CUDA path (called through the C ABI) with the CPU oracle.

Integers, MAX and the fixed-order f32/bf16 folds must match bit for bit (NaN
compared as NaN, payload-free); AllGather must copy bits exactly.  Sizes span
several tiles and ragged tails.  The full-size workloads (8 x 128 MiB bf16 in
ring and tree order, GPT-2 small's gradients in 25 MiB buckets) are compared
with the oracle on every element (the oracle's runs split over host
processes), and element by element on sampled positions plus every chunk
boundary."""
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
from allreduce_gradient_reduction_gb300 import workloads as W
from oracle import parallel as oracle_parallel

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

NP_TO_TORCH = {np.dtype(np.float32): torch.float32, np.dtype(np.uint16): torch.int16,
               np.dtype(np.int32): torch.int32}


@pytest.fixture(scope="module")
def ar():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from allreduce_gradient_reduction_gb300 import build as b
    b.build()
    from allreduce_gradient_reduction_gb300 import binding
    torch.cuda.set_device(0)
    return binding


def to_dev(row: np.ndarray) -> "torch.Tensor":
    a = np.ascontiguousarray(row)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def from_dev(bufs, dtype):
    out = np.stack([b.cpu().numpy() for b in bufs]) if bufs else np.zeros((0, 0))
    return out.view(np.uint16) if dtype in HALF else out


HALF = ("bf16", "f16")  # dtypes stored as 16-bit patterns


def f64(x, dtype):
    if dtype == "f16":
        return np.ascontiguousarray(x, dtype=np.uint16).view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (np.asarray(x).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(x).astype(np.float64)


def assert_same(got, want, dtype, what=""):
    """Bit equality with NaN == NaN."""
    got, want = np.asarray(got), np.asarray(want)
    assert got.shape == want.shape, what
    if dtype == "i32":
        bad = got != want
    else:
        gv, wv = f64(got, dtype), f64(want, dtype)
        gn, wn = np.isnan(gv), np.isnan(wv)
        bits = np.uint16 if dtype in HALF else np.uint32
        bad = (gn != wn) | (~gn & ~wn & (got.view(bits) != want.view(bits)))
    if bad.any():
        idx = np.argwhere(bad)
        i = tuple(idx[0])
        raise AssertionError(f"{what}: {len(idx)} elements differ; first at {i}: got {got[i]!r} want {want[i]!r}")


def run_collective(ar, fn_name, x, dtype, count=None, check_status=True, **kw):
    bufs = [to_dev(x[r]) for r in range(x.shape[0])]
    rc = getattr(ar, fn_name)(bufs, count=x.shape[1] if count is None else count, dtype=dtype, **kw)
    ar.check(rc, fn_name)
    torch.cuda.synchronize()
    if check_status:
        rc, st = ar.ar_device_status()
        assert rc == 0 and st == 0, (rc, st)
    return from_dev(bufs, dtype), bufs


def inputs(n, count, dtype, kind, seed):
    if kind == "bits":
        return W.random_bits(n, count, dtype, seed)
    if dtype == "i32":
        return W.uniform_inputs(n, count, "i32", config=seed)
    if dtype == "bf16":
        return W.large_inputs(n, count, config=seed)
    if dtype == "f16":
        return W.normal_inputs(n, count, 1.0, seed).astype(np.float16).view(np.uint16)
    return W.normal_inputs(n, count, 1.0, seed)


ALGOS = ["ring", "tree", "ring_stepwise", "tree_stepwise"]
ORACLE_ALGO = {"ring": "ring", "ring_stepwise": "ring", "tree": "tree", "tree_stepwise": "tree",
               "binomial_stepwise": "binomial"}


def counts_for(n):
    base = [1, n - 1, n + 1, 1000, 4099, 3 * 2048 * n + 13]
    if n >= 64:
        base = [1, n + 1, 4099, 70_001]
    return [c for c in base if c > 0]


# --------------------------------------------------------------------------
# AllReduce / ReduceScatter / AllGather against the oracle, many shapes
# --------------------------------------------------------------------------

@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
@pytest.mark.parametrize("n", [2, 3, 4, 5, 8, 16, 32, 64])
def test_allreduce_matches_oracle(ar, algo, dtype, n):
    if algo.startswith("tree") and n & (n - 1):
        pytest.skip("tree order needs a power of two")
    ops = ["sum", "max"] + ([] if dtype == "i32" else ["avg"])
    for count in counts_for(n):
        for op in ops:
            kind = "bits" if (count % 2 and op != "sum") else "values"
            x = inputs(n, count, dtype, kind, seed=n * 7919 + count)
            with np.errstate(all="ignore"):
                want, _ = oracle.allreduce(x, algo=ORACLE_ALGO[algo], op=op, dtype=dtype)
            got, _ = run_collective(ar, "ar_allreduce", x, dtype, op=op, algo=algo)
            assert_same(got, want, dtype, f"{algo} {dtype} {op} n={n} count={count}")


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
def test_allreduce_special_values(ar, algo, dtype):
    # NaN, infinities, subnormals, signed zeros in every position
    for n in (2, 4, 8):
        for count in (37, 8 * 1024 + 3):
            x = W.random_bits(n, count, dtype, seed=1000 + n + count)
            for op in ["sum", "max"] + ([] if dtype == "i32" else ["avg"]):
                with np.errstate(all="ignore"):
                    want, _ = oracle.allreduce(x, algo=ORACLE_ALGO[algo], op=op, dtype=dtype)
                got, _ = run_collective(ar, "ar_allreduce", x, dtype, op=op, algo=algo)
                assert_same(got, want, dtype, f"{algo} {dtype} {op} n={n} count={count}")


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
def test_reduce_scatter_matches_oracle(ar, algo, dtype):
    for n in (2, 3, 4, 8, 16):
        if algo.startswith("tree") and n & (n - 1):
            continue
        for count in (n, 4099, 2 * 2048 * n + 5):
            x = inputs(n, count, dtype, "values", seed=50 + n + count)
            for op in ["sum", "max"] + ([] if dtype == "i32" else ["avg"]):
                want, _ = oracle.reduce_scatter(x, algo=ORACLE_ALGO[algo], op=op, dtype=dtype)
                got, _ = run_collective(ar, "ar_reduce_scatter", x, dtype, op=op, algo=algo)
                for r in range(n):
                    lo, hi = oracle.chunk_range(count, n, r)
                    assert_same(got[r, lo:hi], want[r, lo:hi], dtype, f"{algo} {op} n={n} count={count} rank {r}")


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
def test_all_gather_copies_bits(ar, algo, dtype):
    for n in (2, 3, 4, 8, 16):
        if algo.startswith("tree") and n & (n - 1):
            continue
        for count in (1, n + 1, 4099, 3 * 2048 * n + 7):
            x = W.random_bits(n, count, dtype, seed=77 + n + count)  # NaN payloads must survive
            want, _ = oracle.all_gather(x, algo=ORACLE_ALGO[algo], dtype=dtype)
            bufs = [to_dev(x[r]) for r in range(n)]
            ar.check(ar.ar_all_gather(bufs, count=count, dtype=dtype, algo=algo), "all_gather")
            got = from_dev(bufs, dtype)
            bits = {"bf16": np.uint16, "f16": np.uint16, "f32": np.uint32, "i32": np.uint32}[dtype]
            assert np.array_equal(got.view(bits), want.view(bits)), (algo, n, count)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
@pytest.mark.parametrize("n", [2, 4, 8, 16, 32, 64])
def test_binomial_stepwise_matches_oracle(ar, n, dtype):
    """The literal binomial reduce-to-root-then-broadcast schedule against the
    oracle's message simulation of the same schedule, bit for bit, in the
    one-block form (small rows) and the grid-barrier form; its values must
    equal the tree order's (the same pairwise fold)."""
    for count in counts_for(n):
        x = inputs(n, count, dtype, "bits" if count % 2 else "values", seed=700 + n + count)
        for op in ["sum", "max"] + ([] if dtype == "i32" else ["avg"]):
            with np.errstate(all="ignore"):
                want, st = oracle.allreduce(x, algo="binomial", op=op, dtype=dtype)
                tree, _ = oracle.allreduce(x, algo="tree", op=op, dtype=dtype)
            assert st["steps"] == 2 * int(math.log2(n))
            got, _ = run_collective(ar, "ar_allreduce", x, dtype, op=op, algo="binomial_stepwise")
            assert_same(got, want, dtype, f"binomial n={n} count={count} {op}")
            assert_same(got, tree, dtype, f"binomial = tree n={n} count={count} {op}")


def cluster_form_counts(n, algo, es):
    """Counts whose plain step-wise call takes the cluster form: more than
    3072 element updates in a step or more than 160 KiB in all (so not one
    block), the busiest block folding at most 1024 elements in an average
    step (6144 when every chunk is cut on a 16-byte boundary and the steps
    move 16-byte vectors), the ranks spread over the largest power-of-two
    cluster of at most 16 blocks.  Both kinds of count are returned."""
    c = 2
    while c * 2 <= 16 and c * 2 <= n:
        c *= 2
    if c > n:
        return []
    nloc = -(-n // c)
    vec = 16 // es
    out, out_vec = [], []
    for count in list(range(1, 40000, 7)) + list(range(n * vec, 200000, n * vec)):
        stride = -(-count * es // 16) * 16
        step = count * (1 if algo.startswith("ring") else n // 2)
        one_block = step <= 3072 and n * stride <= 160 * 1024
        if algo.startswith("ring"):
            work = nloc * -(-count // n)
        elif algo.startswith("tree"):
            work = nloc * (count - count // n) // (n.bit_length() - 1)
        else:
            work = nloc * count
        aligned = count % (n * vec) == 0
        limit = 6144 if aligned else 1024
        if not one_block and nloc * stride <= 160 * 1024 and work <= limit:
            (out_vec if aligned else out).append(count)
    pick = lambda v: sorted({v[0], v[len(v) // 2], v[-1]}) if v else []
    return pick(out) + pick(out_vec)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n", [4, 8, 16, 32, 64])
def test_stepwise_cluster_form(ar, n, dtype):
    """Rows too large for one block's shared memory (or with more than 3072
    element updates in a step) whose steps are small run the literal
    schedule in one thread-block cluster, ranks spread over its blocks'
    shared memory, each step reading the senders' values from the other
    blocks' shared memory: ring, tree and binomial, AllReduce, ReduceScatter
    and AllGather, against the oracle bit for bit."""
    es = 4 if dtype == "f32" else 2
    tested = 0
    for algo in ("ring_stepwise", "tree_stepwise", "binomial_stepwise"):
        for count in cluster_form_counts(n, algo, es):
            tested += 1
            x = inputs(n, count, dtype, "values", seed=1300 + n + count)
            for op in ("sum", "avg"):
                want, _ = oracle.allreduce(x, algo=ORACLE_ALGO[algo], op=op, dtype=dtype)
                got, _ = run_collective(ar, "ar_allreduce", x, dtype, op=op, algo=algo)
                assert_same(got, want, dtype, f"cluster {algo} n={n} count={count} {op}")
            if algo == "binomial_stepwise":
                continue
            want, _ = oracle.reduce_scatter(x, algo=ORACLE_ALGO[algo], op="max", dtype=dtype)
            got, _ = run_collective(ar, "ar_reduce_scatter", x, dtype, op="max", algo=algo)
            for r in range(n):
                lo, hi = oracle.chunk_range(count, n, r)
                assert_same(got[r, lo:hi], want[r, lo:hi], dtype, f"cluster RS {algo} n={n} count={count}")
            want, _ = oracle.all_gather(x, algo=ORACLE_ALGO[algo], dtype=dtype)
            got, _ = run_collective(ar, "ar_all_gather", x, dtype, algo=algo)
            assert_same(got, want, dtype, f"cluster AG {algo} n={n} count={count}")
    assert tested > 0


def test_binomial_stepwise_takes_allreduce_only(ar):
    bufs = [torch.zeros(64, device="cuda") for _ in range(4)]
    assert ar.ar_allreduce(bufs[:3], count=64, algo="binomial_stepwise") == ar.AR_ERR_UNSUPPORTED
    assert ar.ar_reduce_scatter(bufs, count=64, algo="binomial_stepwise") == ar.AR_ERR_UNSUPPORTED
    assert ar.ar_all_gather(bufs, count=64, algo="binomial_stepwise") == ar.AR_ERR_UNSUPPORTED
    assert ar.ar_reduce(bufs, count=64, algo="binomial_stepwise", root=0) == ar.AR_ERR_UNSUPPORTED
    grads = [[b] for b in bufs]
    assert ar.ar_bucketed_allreduce(grads, counts=[64], algo="binomial_stepwise") == ar.AR_ERR_UNSUPPORTED
    assert ar.ar_bucketed_allreduce_noalloc(grads, counts=[64], algo="binomial_stepwise") == ar.AR_ERR_UNSUPPORTED
    host = [torch.zeros(64).pin_memory() for _ in range(4)]
    assert ar.ar_allreduce_host(host, None, count=64, algo="binomial_stepwise") == ar.AR_ERR_UNSUPPORTED
    plan = ar.Plan("allreduce", bufs, count=64, algo="binomial_stepwise")  # prepared AllReduce is fine
    ar.check(plan.run(), "plan")
    torch.cuda.synchronize()
    plan.close()


# --------------------------------------------------------------------------
# Alignment, degenerate sizes, streams
# --------------------------------------------------------------------------

@pytest.mark.parametrize("algo", ALGOS + ["dbtree", "naive"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
def test_unaligned_buffers(ar, algo, dtype):
    """Element-aligned but not 16-byte aligned buffers.  The same offset in
    every rank takes the vector path cut at that offset; different offsets
    per rank take the one-element-per-thread path.  Both must give the same
    bits, and nothing before a buffer is touched."""
    n, count = 8, 5000 + 2048 * 8 + 3
    x = inputs(n, count, dtype, "values", seed=9)
    want, _ = oracle.allreduce(x, algo=ORACLE_ALGO.get(algo, algo), op="sum", dtype=dtype)
    vec = 8 if dtype in HALF else 4
    layouts = [[s] * n for s in range(1, vec)] + [[r % vec for r in range(n)], [(3 * r + 1) % vec for r in range(n)]]
    for shifts in layouts:
        big = [to_dev(np.concatenate([x[r][:shifts[r]], x[r]])) for r in range(n)]
        views = [b[s:] for b, s in zip(big, shifts)]
        ar.check(ar.ar_allreduce(views, count=count, dtype=dtype, op="sum", algo=algo), "unaligned")
        torch.cuda.synchronize()
        got = from_dev(views, dtype)
        assert_same(got, want, dtype, f"{algo} shifts {shifts}")
        for r in range(n):
            assert np.array_equal(from_dev([big[r][:shifts[r]]], dtype)[0], x[r, :shifts[r]])


@pytest.mark.parametrize("n", [2, 3, 4, 5, 6, 7, 8, 16, 24, 32, 64])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
def test_mixed_phase_rows(ar, n, dtype):
    """Rank buffers at different addresses modulo 16 (the staged kernel:
    aligned words of every rank copied to shared memory, through eight slots
    beyond eight ranks, folded in the first buffer's frame, stored back at
    each rank's phase), in every order the rank count allows, for AllReduce,
    ReduceScatter (owner store) and Reduce (root store), over a size whose
    chunks span several tiles and end ragged.  Every rank count the kernel
    is compiled for (2-8, 16, 32, 64) and the runtime-rank ring and double
    binary tree (24).
    Nothing outside the buffers may change."""
    vec = 8 if dtype in HALF else 4
    count = 3 * 512 * vec * min(n, 8) + 2048 * n + 13
    x = inputs(n, count, dtype, "values", seed=41 + n)
    shifts = [(5 * r + 1) % vec for r in range(n)]
    algos = ["ring", "naive", "dbtree"] + (["tree"] if n & (n - 1) == 0 else [])
    ops = ["sum", "max"] + ([] if dtype == "i32" else ["avg"])
    for algo in algos:
        for op in ops:
            kinds = ("allreduce", "reduce_scatter", "reduce") if algo in ("ring", "tree") else ("allreduce",)
            for kind in kinds:
                big = [to_dev(np.concatenate([x[r][:shifts[r]], x[r], x[r][:7]])) for r in range(n)]
                views = [b[s:s + count] for b, s in zip(big, shifts)]
                oa = ORACLE_ALGO.get(algo, algo)
                what = f"{kind} {algo} {op} n={n} shifts={shifts}"
                if kind == "allreduce":
                    want, _ = oracle.allreduce(x, algo=oa, op=op, dtype=dtype)
                    ar.check(ar.ar_allreduce(views, count=count, dtype=dtype, op=op, algo=algo), what)
                elif kind == "reduce_scatter":
                    want, _ = oracle.reduce_scatter(x, algo=oa, op=op, dtype=dtype)
                    ar.check(ar.ar_reduce_scatter(views, count=count, dtype=dtype, op=op, algo=algo), what)
                else:
                    want, _ = oracle.reduce(x, algo=oa, op=op, dtype=dtype, root=n - 1)
                    ar.check(ar.ar_reduce(views, count=count, dtype=dtype, op=op, algo=algo, root=n - 1), what)
                torch.cuda.synchronize()
                got = from_dev(views, dtype)
                for r in range(n):
                    if kind == "reduce_scatter":
                        lo, hi = oracle.chunk_range(count, n, r)
                        assert_same(got[r, lo:hi], want[r, lo:hi], dtype, f"{what} rank {r}")
                    elif kind == "reduce" and r != n - 1:
                        assert_same(got[r], x[r], dtype, f"{what} non-root {r}")
                    else:
                        assert_same(got[r], want[r], dtype, f"{what} rank {r}")
                    edge = from_dev([big[r]], dtype)[0]
                    assert np.array_equal(edge[:shifts[r]], x[r, :shifts[r]]), f"{what} before rank {r}"
                    assert np.array_equal(edge[shifts[r] + count:], x[r, :7]), f"{what} after rank {r}"


@pytest.mark.parametrize("n", [16, 32, 64])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
def test_unaligned_wide_rings(ar, n, dtype):
    """The 16-, 32- and 64-rank ring kernels with every buffer at the same
    offset from 16 bytes (vectors cut at that offset, scalar head and tail),
    and the ReduceScatter form that stores to the chunk owner only."""
    count = 2048 * n + 4099
    x = inputs(n, count, dtype, "values", seed=31 + n)
    want, _ = oracle.allreduce(x, algo="ring", op="sum", dtype=dtype)
    want_rs, _ = oracle.reduce_scatter(x, algo="ring", op="sum", dtype=dtype)
    shift = 3 if dtype in HALF else 1
    for fn in ("ar_allreduce", "ar_reduce_scatter"):
        big = [to_dev(np.concatenate([x[r][:shift], x[r]])) for r in range(n)]
        views = [b[shift:] for b in big]
        ar.check(getattr(ar, fn)(views, count=count, dtype=dtype, op="sum", algo="ring"), fn)
        torch.cuda.synchronize()
        got = from_dev(views, dtype)
        if fn == "ar_allreduce":
            assert_same(got, want, dtype, f"wide ring n={n}")
        else:
            for r in range(n):
                lo, hi = oracle.chunk_range(count, n, r)
                assert_same(got[r, lo:hi], want_rs[r, lo:hi], dtype, f"wide ring RS n={n} rank {r}")
        for r in range(n):
            assert np.array_equal(from_dev([big[r][:shift]], dtype)[0], x[r, :shift])


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_unaligned_reduce_scatter_all_gather_broadcast(ar, dtype):
    n, count = 4, 3 * 2048 * 4 + 77
    x = inputs(n, count, dtype, "values", seed=19)
    vec = 8 if dtype in HALF else 4
    for shifts in ([3] * n, [r % vec for r in range(n)]):
        def views_of(data):
            big = [to_dev(np.concatenate([data[r][:shifts[r]], data[r]])) for r in range(n)]
            return [b[s:] for b, s in zip(big, shifts)]
        for algo in ("ring", "tree", "ring_stepwise"):
            want, _ = oracle.reduce_scatter(x, algo=ORACLE_ALGO[algo], op="sum", dtype=dtype)
            v = views_of(x)
            ar.check(ar.ar_reduce_scatter(v, count=count, dtype=dtype, op="sum", algo=algo), "rs")
            got = from_dev(v, dtype)
            for r in range(n):
                lo, hi = oracle.chunk_range(count, n, r)
                assert_same(got[r, lo:hi], want[r, lo:hi], dtype, f"rs {algo} {shifts}")
            want, _ = oracle.all_gather(x, algo=ORACLE_ALGO[algo], dtype=dtype)
            v = views_of(x)
            ar.check(ar.ar_all_gather(v, count=count, dtype=dtype, algo=algo), "ag")
            assert_same(from_dev(v, dtype), want, dtype, f"ag {algo} {shifts}")
        want, _ = oracle.broadcast(x, root=2, dtype=dtype)
        v = views_of(x)
        ar.check(ar.ar_broadcast(v, count=count, dtype=dtype, root=2), "broadcast")
        assert_same(from_dev(v, dtype), want, dtype, f"broadcast {shifts}")


def test_degenerate_sizes(ar):
    x = W.normal_inputs(4, 10, 1.0, 3)
    bufs = [to_dev(x[r]) for r in range(4)]
    ar.check(ar.ar_allreduce(bufs, count=0), "count 0")
    torch.cuda.synchronize()
    assert np.array_equal(from_dev(bufs, "f32"), x)  # nothing moved
    one = [to_dev(x[0])]
    for algo in ALGOS:
        ar.check(ar.ar_allreduce(one, count=10, op="avg", algo=algo), "one rank")
    torch.cuda.synchronize()
    assert np.array_equal(one[0].cpu().numpy(), x[0])


def test_runs_on_the_given_stream(ar):
    n, count = 8, 1 << 20
    x = W.normal_inputs(n, count, 1.0, 4)
    want, _ = oracle.allreduce(x, op="sum", dtype="f32")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        bufs = [to_dev(x[r]) for r in range(n)]
        ar.check(ar.ar_allreduce(bufs, dtype="f32", op="sum", stream=s), "stream")
    s.synchronize()
    assert_same(from_dev(bufs, "f32"), want, "f32")


def test_rejects_memory_it_cannot_use(ar):
    x = torch.zeros(1024, device="cuda")
    y = torch.zeros(1024, device="cuda")
    host = np.zeros(1024, dtype=np.float32)
    assert ar.ar_allreduce([x, host.ctypes.data], count=1024) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_allreduce([x, y], count=1 << 30) == ar.AR_ERR_INVALID_ARG  # past the allocation
    assert ar.ar_allreduce([x, x[512:]], count=1024) == ar.AR_ERR_INVALID_ARG  # overlap


# --------------------------------------------------------------------------
# The printed examples and the configured workloads
# --------------------------------------------------------------------------

def test_three_rank_example(ar):
    x = W.three_rank_example()
    got, _ = run_collective(ar, "ar_allreduce", x, "f32", op="sum", algo="ring")
    assert np.all(got == 6.0)
    got, _ = run_collective(ar, "ar_allreduce", x, "f32", op="sum", algo="ring_stepwise")
    assert np.all(got == 6.0)


def test_printed_examples_on_gpu(ar):
    x = np.stack([np.full(6, r + 1, dtype=np.float32) for r in range(4)])  # ones(2,3)*(rank+1)
    for algo in ALGOS:
        got, _ = run_collective(ar, "ar_allreduce", x, "f32", op="sum", algo=algo)
        assert np.all(got == 10.0), algo
    x = np.stack([np.full(4, r, dtype=np.float32) for r in range(4)])   # ones(4)*rank, then / world size
    for algo in ALGOS:
        got, _ = run_collective(ar, "ar_allreduce", x, "f32", op="avg", algo=algo)
        assert np.all(got == 1.5), algo


def test_small_workload(ar):
    x = W.small_inputs()
    exact = x.astype(np.float64).sum(axis=0)
    for algo in ALGOS:
        got, _ = run_collective(ar, "ar_allreduce", x, "f32", op="sum", algo=algo)
        assert np.array_equal(got, np.broadcast_to(exact, got.shape)), algo


def test_bucket_workload_full_compare(ar):
    x = W.bucket_inputs()
    for op in ("avg", "max"):
        want, _ = oracle.allreduce(x, algo="ring", op=op, dtype="f32")
        for algo in ("ring", "ring_stepwise"):
            got, _ = run_collective(ar, "ar_allreduce", x, "f32", op=op, algo=algo)
            assert_same(got, want, "f32", f"{algo} {op}")
    # f32 stays inside the stated tolerance against the order-free sum
    s, _ = run_collective(ar, "ar_allreduce", x, "f32", op="sum", algo="ring")
    xv = x.astype(np.float64)
    assert np.all(np.abs(s[0] - xv.sum(axis=0)) <= 1e-5 * np.abs(xv).sum(axis=0))


def sample_positions(count, n, k, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    pos = [g.integers(0, count, size=k)]
    for c in range(n + 1):
        lo = oracle.chunk_range(count, n, c)[0] if c < n else count
        pos.append(np.arange(lo - 2, lo + 3))
    p = np.unique(np.concatenate(pos))
    return p[(p >= 0) & (p < count)]


@pytest.mark.slow
def test_large_workload_full_compare(ar):
    """8 ranks x 67,108,864 bf16, the configuration the benchmark times, in
    ring and in tree order: every element of the result compared with the
    oracle (oracle processes on every host core, each carrying one element
    range through the full simulation, compared by digests of the ranges),
    every rank identical, and on sampled positions plus every chunk boundary
    +-2 the values one by one and the bf16 error bound."""
    n, count = W.LARGE["nranks"], W.LARGE["count"]
    x = W.large_inputs(n, count)
    pos = sample_positions(count, n, 1 << 16, 5)
    xs = np.ascontiguousarray(x[:, pos])
    with oracle_parallel.Pool() as pool:
        pool.load(x, op="sum", dtype="bf16")
        for algo in ("ring", "tree"):
            want, _ = oracle.allreduce(xs, algo=algo, op="sum", dtype="bf16", count=count, positions=pos)
            bufs = [to_dev(x[r]) for r in range(n)]
            ar.check(ar.ar_allreduce(bufs, count=count, dtype="bf16", op="sum", algo=algo), algo)
            torch.cuda.synchronize()
            for r in range(1, n):
                assert torch.equal(bufs[r], bufs[0]), (algo, r)  # every rank identical
            got = bufs[0][torch.from_numpy(pos).cuda()].cpu().numpy().view(np.uint16)
            assert_same(got, want[0], "bf16", algo)
            # bf16 error stays within the recursive-summation bound gamma_k * sum|x|
            xv = f64(xs, "bf16")
            depth = n - 1 if algo == "ring" else int(math.log2(n))
            u = 2.0 ** -8
            err = np.abs(f64(got, "bf16") - xv.sum(axis=0))
            assert np.all(err <= depth * u / (1 - depth * u) * np.abs(xv).sum(axis=0))
            # every element against the oracle's full run
            res0 = bufs[0].cpu().numpy().view(np.uint16)
            del bufs
            pool.run(algo=algo)
            cmp = pool.compare(res0)
            assert cmp["bit_identical"] and cmp["elements"] == count, (algo, cmp)


def bucket_boundary_samples(counts, n, cap=25 << 20, dtype="f32"):
    """(tensor, index) of every bucket chunk boundary +-2 and every tensor's
    first and last two elements, from the oracle's bucket plan: the places
    where the fused bucketed kernel switches segments and rank order."""
    bucket_of, offset, bcount = oracle.bucket_plan(counts, dtype=dtype, cap_bytes=cap)
    tid, idx = [], []
    for t, c in enumerate(counts):
        if c == 0:
            continue
        B, o = int(bcount[bucket_of[t]]), int(offset[t])
        cand = [0, 1, c - 2, c - 1]
        for k in range(n + 1):
            lo = oracle.chunk_range(B, n, k)[0] if k < n else B
            cand += list(range(lo - o - 2, lo - o + 3))
        for i in sorted(set(cand)):
            if 0 <= i < c:
                tid.append(t)
                idx.append(i)
    return np.array(tid, dtype=np.int32), np.array(idx, dtype=np.int64)


@pytest.mark.slow
def test_gpt2_bucketed_full_compare(ar):
    """GPT-2 small gradients, 8 ranks, 25 MiB buckets, AVG: the fused,
    literal (whole and per-bucket workspace) and step-wise paths, each compared
    with the oracle's bucketed AllReduce on every element of every tensor of
    every rank (the oracle split by bucket over host processes, compared by
    digests), and element by element on every bucket chunk boundary +-2."""
    n = W.GPT2["nranks"]
    counts = W.gpt2_small_counts()
    host = [W.gpt2_rank_grads(r, counts) for r in range(n)]
    with oracle_parallel.Pool() as pool:
        want_digest, _ = pool.bucketed_digests(host, op="avg", dtype="f32", cap_bytes=25 << 20)
    tid, idx = bucket_boundary_samples(counts, n)
    g = np.random.Generator(np.random.PCG64(8))
    rt = g.integers(0, counts.size, size=4000).astype(np.int32)
    ri = (g.random(rt.size) * counts[rt]).astype(np.int64)
    pairs = np.unique(np.stack([np.concatenate([tid, rt]), np.concatenate([idx, ri])], axis=1), axis=0)
    tid, idx = pairs[:, 0].astype(np.int32), pairs[:, 1].astype(np.int64)
    want, _ = oracle.bucketed_allreduce(host, op="avg", dtype="f32", samples=(tid, idx))

    flat_len = int(counts.sum())
    offs = np.concatenate([[0], np.cumsum(counts)])
    for mode in ("fused", "whole", "per_bucket", "stepwise"):
        # one flat allocation per rank with the tensors as views into it
        flats = [torch.from_numpy(np.concatenate(host[r])).cuda() for r in range(n)]
        grads = [[flats[r][offs[t]:offs[t + 1]] for t in range(counts.size)] for r in range(n)]
        ws, wbytes = None, 0
        if mode in ("whole", "per_bucket"):
            per = flat_len if mode == "whole" else int(max(oracle.bucket_plan(counts, dtype="f32")[2]))
            ws = [torch.empty(per, dtype=torch.float32, device="cuda") for _ in range(n)]
            wbytes = per * 4
        algo = "ring_stepwise" if mode == "stepwise" else "ring"
        rc = ar.ar_bucketed_allreduce(grads, counts=counts, dtype="f32", op="avg", algo=algo, workspace=ws,
                                      workspace_bytes=wbytes)
        ar.check(rc, mode)
        torch.cuda.synchronize()
        sel = torch.from_numpy(offs[tid] + idx).cuda()
        got = np.stack([flats[r][sel].cpu().numpy() for r in range(n)])
        assert_same(got, want, "f32", mode)
        host_res = [f.cpu().numpy() for f in flats]
        del flats, grads, ws

        def rank_digests(r):
            return [oracle_parallel.digest(host_res[r][offs[t]:offs[t + 1]]) for t in range(counts.size)]
        with ThreadPoolExecutor(max_workers=n) as ex:
            got_digest = list(ex.map(rank_digests, range(n)))
        bad = [(r, t) for r in range(n) for t in range(counts.size) if got_digest[r][t] != want_digest[r][t]]
        assert not bad, (mode, f"{len(bad)} (rank, tensor) results differ from the oracle, first {bad[:5]}")
        del host_res


def test_bucketed_small_full_compare(ar):
    g = np.random.Generator(np.random.PCG64(21))
    counts = [5, 300, 17, 1024, 3, 999, 64, 4096 + 3, 1, 2048]
    for n in (2, 3, 8):
        for dtype in ("f32", "bf16", "f16"):
            if dtype == "f32":
                host = [[g.standard_normal(c).astype(np.float32) for c in counts] for _ in range(n)]
            elif dtype == "f16":
                host = [[g.standard_normal(c).astype(np.float16).view(np.uint16) for c in counts] for _ in range(n)]
            else:
                host = [[W.f32_to_bf16_bits_truncate(g.standard_normal(c).astype(np.float32)) for c in counts]
                        for _ in range(n)]
            es = 4 if dtype == "f32" else 2
            cap = es * 1500
            for algo in ("ring", "tree", "ring_stepwise", "tree_stepwise"):
                if algo.startswith("tree") and n & (n - 1):
                    continue
                want, _ = oracle.bucketed_allreduce(host, op="avg", dtype=dtype, algo=ORACLE_ALGO[algo],
                                                    cap_bytes=cap)
                for literal in (False, True):
                    grads = [[to_dev(t) for t in row] for row in host]
                    ws = None
                    if literal:
                        ws = [torch.empty(sum(counts) + 8, dtype=torch.float32, device="cuda") for _ in range(n)]
                    rc = ar.ar_bucketed_allreduce(grads, counts=counts, dtype=dtype, op="avg", algo=algo,
                                                  bucket_cap_bytes=cap, workspace=ws,
                                                  workspace_bytes=(sum(counts) + 8) * 4 if literal else 0)
                    ar.check(rc, f"bucketed {algo}")
                    torch.cuda.synchronize()
                    for r in range(n):
                        for t in range(len(counts)):
                            got = grads[r][t].cpu().numpy()
                            if dtype in HALF:
                                got = got.view(np.uint16)
                            assert_same(got, want[r][t], dtype, f"{algo} literal={literal} n={n} r={r} t={t}")


# --------------------------------------------------------------------------
# Exhaustive bf16 step: every pair of bf16 values through a 2-rank ring
# --------------------------------------------------------------------------

@pytest.mark.slow
def test_f16_step_exhaustive(ar):
    all16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    block = 1 << 12  # values of `a` per block: 2^28 pairs
    a_dev = torch.empty(block << 16, dtype=torch.int16, device="cuda")
    b_dev = torch.empty(block << 16, dtype=torch.int16, device="cuda")
    b_row = torch.from_numpy(all16.view(np.int16)).cuda().repeat(block)
    for a0 in range(0, 1 << 16, block):
        a_vals = np.repeat(all16[a0:a0 + block], 1 << 16)
        a_dev.copy_(torch.from_numpy(a_vals.view(np.int16)))
        b_dev.copy_(b_row)
        ar.check(ar.ar_allreduce([a_dev, b_dev], count=a_vals.size, dtype="f16", op="sum", algo="ring"), "pairs")
        torch.cuda.synchronize()
        got = a_dev.cpu().numpy().view(np.uint16)
        want = oracle.step(a_vals, np.tile(all16, block), op="sum", dtype="f16")
        assert_same(got, want, "f16", f"a block {a0}")


def test_bf16_step_exhaustive(ar):
    all16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    block = 1 << 12  # values of `a` per block: 2^28 pairs
    a_dev = torch.empty(block << 16, dtype=torch.int16, device="cuda")
    b_dev = torch.empty(block << 16, dtype=torch.int16, device="cuda")
    b_row = torch.from_numpy(all16.view(np.int16)).cuda().repeat(block)
    for a0 in range(0, 1 << 16, block):
        a_vals = np.repeat(all16[a0:a0 + block], 1 << 16)
        a_dev.copy_(torch.from_numpy(a_vals.view(np.int16)))
        b_dev.copy_(b_row)
        ar.check(ar.ar_allreduce([a_dev, b_dev], count=a_vals.size, dtype="bf16", op="sum", algo="ring"), "pairs")
        torch.cuda.synchronize()
        got = a_dev.cpu().numpy().view(np.uint16)
        want = oracle.step(a_vals, np.tile(all16, block), op="sum", dtype="bf16")
        assert_same(got, want, "bf16", f"a block {a0}")


# --------------------------------------------------------------------------
# Failure detection without a fault: a barrier nobody completes times out
# --------------------------------------------------------------------------

@pytest.mark.parametrize("count", [1 << 16, 1 << 22])  # grids of at most 128 blocks (one counter) and more (groups)
@pytest.mark.parametrize("algo", ["ring_stepwise", "tree_stepwise", "binomial_stepwise"])
def test_barrier_timeout_is_reported(ar, algo, count):
    n = 8
    x = W.normal_inputs(n, count, 1.0, 12)
    ar.ar_set_barrier_timeout_ns(50_000_000)  # 50 ms
    try:
        bufs = [to_dev(x[r]) for r in range(n)]
        ar.ar_debug_skip_barrier(1)
        ar.check(ar.ar_allreduce(bufs, count=count, dtype="f32", op="sum", algo=algo), "launch")
        rc, st = ar.ar_device_status()
        assert rc == 0 and st == ar.AR_ERR_TIMEOUT
        rc, st = ar.ar_device_status()
        assert rc == 0 and st == 0  # read once, then cleared
        # the context is still usable and the next call is correct
        want, _ = oracle.allreduce(x, algo=ORACLE_ALGO[algo], op="sum", dtype="f32")
        got, _ = run_collective(ar, "ar_allreduce", x, "f32", op="sum", algo=algo)
        assert_same(got, want, "f32", algo)
    finally:
        ar.ar_debug_skip_barrier(-1)
        ar.ar_set_barrier_timeout_ns(0)


# --------------------------------------------------------------------------
# Reduce, Broadcast and the naive (index) order
# --------------------------------------------------------------------------

@pytest.mark.parametrize("algo", ["ring", "tree", "naive"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
def test_reduce_matches_oracle(ar, algo, dtype):
    for n in (2, 3, 5, 8, 16):
        if algo == "tree" and n & (n - 1):
            continue
        for count in (1, n + 1, 4099, 2 * 2048 * n + 9):
            x = inputs(n, count, dtype, "bits" if count % 2 else "values", seed=900 + n + count)
            for op in ["sum", "max"] + ([] if dtype == "i32" else ["avg"]):
                for root in sorted({0, n - 1, n // 2}):
                    with np.errstate(all="ignore"):
                        want, _ = oracle.reduce(x, algo=algo, op=op, dtype=dtype, root=root)
                    bufs = [to_dev(x[r]) for r in range(n)]
                    ar.check(ar.ar_reduce(bufs, count=count, dtype=dtype, op=op, algo=algo, root=root), "reduce")
                    got = from_dev(bufs, dtype)
                    assert_same(got[root], want[root], dtype, f"{algo} {op} n={n} count={count} root={root}")
                    others = [r for r in range(n) if r != root]
                    assert np.array_equal(got[others].view(np.uint8), x[others].view(np.uint8))  # untouched


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
def test_naive_allreduce_matches_oracle(ar, dtype):
    for n in (2, 3, 8, 64):
        for count in (1, 4099, 70_001):
            x = inputs(n, count, dtype, "values", seed=1300 + n + count)
            for op in ["sum", "max"] + ([] if dtype == "i32" else ["avg"]):
                want, _ = oracle.allreduce(x, algo="naive", op=op, dtype=dtype)
                got, _ = run_collective(ar, "ar_allreduce", x, dtype, op=op, algo="naive")
                assert_same(got, want, dtype, f"naive {op} n={n} count={count}")
    x = inputs(4, 100, dtype, "values", seed=5)
    bufs = [to_dev(x[r]) for r in range(4)]
    assert ar.ar_reduce_scatter(bufs, count=100, dtype=dtype, algo="naive") == ar.AR_ERR_UNSUPPORTED


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
def test_broadcast_copies_bits(ar, dtype):
    for n in (2, 3, 8, 16):
        for count in (1, 4099, 3 * 2048 + 7):
            x = W.random_bits(n, count, dtype, seed=1700 + n + count)
            for root in sorted({0, n - 1, 1}):
                want, _ = oracle.broadcast(x, root=root, dtype=dtype)
                bufs = [to_dev(x[r]) for r in range(n)]
                ar.check(ar.ar_broadcast(bufs, count=count, dtype=dtype, root=root), "broadcast")
                got = from_dev(bufs, dtype)
                assert np.array_equal(got.view(np.uint8), want.view(np.uint8)), (n, count, root)
    bufs = [to_dev(np.zeros(4, np.float32)) for _ in range(2)]
    assert ar.ar_broadcast(bufs, count=4, root=2) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_reduce(bufs, count=4, root=-1) == ar.AR_ERR_INVALID_ARG


# --------------------------------------------------------------------------
# Double binary tree
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
@pytest.mark.parametrize("n", [2, 3, 4, 5, 6, 7, 8, 12, 16, 64])
def test_dbtree_matches_oracle(ar, dtype, n):
    """Aligned rows: the register-resident kernel (2, 4, 8, 16, 64 ranks)
    and the staged kernel, compiled for the rank count (3, 5, 6, 7) or
    taking it at run time (12)."""
    for count in [c for c in (1, 2, n + 1, 4099, 2 * 2048 * n + 11) if c > 0]:
        for op in ["sum", "max"] + ([] if dtype == "i32" else ["avg"]):
            x = inputs(n, count, dtype, "bits" if (count % 2 and op != "sum") else "values", seed=2100 + n + count)
            with np.errstate(all="ignore"):
                want, _ = oracle.allreduce(x, algo="dbtree", op=op, dtype=dtype)
            got, _ = run_collective(ar, "ar_allreduce", x, dtype, op=op, algo="dbtree")
            assert_same(got, want, dtype, f"dbtree {op} n={n} count={count}")


def test_dbtree_only_for_allreduce(ar):
    x = W.normal_inputs(4, 64, 1.0, 1)
    bufs = [to_dev(x[r]) for r in range(4)]
    assert ar.ar_reduce_scatter(bufs, count=64, algo="dbtree") == ar.AR_ERR_UNSUPPORTED
    assert ar.ar_all_gather(bufs, count=64, algo="dbtree") == ar.AR_ERR_UNSUPPORTED
    assert ar.ar_reduce(bufs, count=64, algo="dbtree", root=1) == ar.AR_ERR_UNSUPPORTED


# --------------------------------------------------------------------------
# 8-bit quantised AllReduce with error feedback
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 3, 8, 16, 64])
def test_int8_ef_matches_oracle(ar, n):
    for count in (1, 127, 128 * n, 128 * 3 * n + 77, 70_001):
        for op in ("sum", "avg"):
            x = W.normal_inputs(n, count, 1e-3, 2500 + n + count)
            e = W.normal_inputs(n, count, 1e-6, 2600 + n + count)
            for it in range(2):  # the residuals carry over to the next call
                want_x, want_e, _ = oracle.int8_ef_allreduce(x, e, op=op)
                xd = [to_dev(x[r]) for r in range(n)]
                ed = [to_dev(e[r]) for r in range(n)]
                ar.check(ar.ar_allreduce_int8_ef(xd, ed, count=count, op=op), "int8_ef")
                got_x, got_e = from_dev(xd, "f32"), from_dev(ed, "f32")
                assert_same(got_x, want_x, "f32", f"x n={n} count={count} {op} it={it}")
                assert_same(got_e, want_e, "f32", f"e n={n} count={count} {op} it={it}")
                x, e = W.normal_inputs(n, count, 1e-3, 2700 + it + n + count), got_e


def int8_tie_inputs(n, count, seed):
    """Per 128-block: one element at the block maximum m, the others at, or a
    hair beside, the quantisation ties (j + 1/2) * s with s = m / 127 -- some
    within two ulps, some a relative 2^-24 .. 2^-12 away -- so that the code
    rounding meets ties and near-ties of every kind."""
    g = np.random.default_rng(seed)
    x = np.zeros((n, count), np.float32)
    for r in range(n):
        for b0 in range(0, count, 128):
            w = min(128, count - b0)
            m = np.float32(g.uniform(0.5, 2.0) * 2.0 ** int(g.integers(-30, 30)))
            s = np.float32(m / np.float32(127.0))
            j = g.integers(-127, 127, size=w).astype(np.float64)
            rel = np.where(g.random(w) < 0.5, 0.0, g.choice([-1, 1], w) * 2.0 ** g.uniform(-24, -12, w))
            y = ((j + 0.5) * (1.0 + rel) * np.float64(s)).astype(np.float32)
            ulps = g.integers(-2, 3, size=w)
            for k in range(2):
                y = np.where(ulps > k, np.nextafter(y, np.float32(np.inf)), y)
                y = np.where(ulps < -k, np.nextafter(y, np.float32(-np.inf)), y)
            y = np.clip(y, -m, m)
            y[int(g.integers(0, w))] = m if g.random() < 0.5 else -m
            x[r, b0:b0 + w] = y
    return x


@pytest.mark.parametrize("n", [2, 4, 8])
def test_int8_ef_rounding_ties(ar, n):
    for count in (128 * 8 * n, 128 * 5 * n + 45):
        x = int8_tie_inputs(n, count, 90 + n + count)
        e = np.zeros_like(x)
        for op in ("sum", "avg"):
            want_x, want_e, _ = oracle.int8_ef_allreduce(x, e, op=op)
            xd = [to_dev(x[r]) for r in range(n)]
            ed = [to_dev(e[r]) for r in range(n)]
            ar.check(ar.ar_allreduce_int8_ef(xd, ed, count=count, op=op), "int8_ef ties")
            assert_same(from_dev(xd, "f32"), want_x, "f32", f"x ties n={n} count={count} {op}")
            assert_same(from_dev(ed, "f32"), want_e, "f32", f"e ties n={n} count={count} {op}")


def test_int8_ef_unaligned_and_rejects(ar):
    n, count = 4, 1000
    x = W.normal_inputs(n, count, 1.0, 31)
    e = np.zeros_like(x)
    want_x, want_e, _ = oracle.int8_ef_allreduce(x, e, op="avg")
    bx = [to_dev(np.concatenate([[0.0], x[r]]).astype(np.float32)) for r in range(n)]
    be = [to_dev(np.concatenate([[0.0], e[r]]).astype(np.float32)) for r in range(n)]
    xd, ed = [b[1:] for b in bx], [b[1:] for b in be]
    ar.check(ar.ar_allreduce_int8_ef(xd, ed, count=count, op="avg"), "unaligned int8")
    assert_same(from_dev(xd, "f32"), want_x, "f32", "x unaligned")
    assert_same(from_dev(ed, "f32"), want_e, "f32", "e unaligned")
    assert ar.ar_allreduce_int8_ef(xd, ed, count=count, op="max") == ar.AR_ERR_UNSUPPORTED
    assert ar.ar_allreduce_int8_ef(xd, xd, count=count) == ar.AR_ERR_INVALID_ARG  # grads overlap residuals


# --------------------------------------------------------------------------
# Large sweep points, sampled: the full-size buffers are generated rank by
# rank; the oracle carries the sampled positions (and every chunk boundary)
# through its messages
# --------------------------------------------------------------------------

@pytest.fixture(scope="module")
def pool():
    with oracle_parallel.Pool() as p:
        yield p


@pytest.mark.slow
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n", [2, 4, 8, 16, 64])
def test_sweep_points_full_compare(ar, pool, n, dtype):
    """The latency/bandwidth sweep's points with N x size <= 2 GiB are
    compared with the oracle on every element: 1 MiB per rank and the
    largest such size (2 GiB / N), uniform(-1, 1) inputs as the sweep draws
    them, SUM and MAX in the fused and step-wise orders, every rank identical
    and rank 0 against the oracle's full run (element ranges over host
    processes, compared by digests)."""
    es = 2 if dtype == "bf16" else 4
    orders = ["ring", "ring_stepwise"] + (["tree", "tree_stepwise", "binomial_stepwise"] if n & (n - 1) == 0 else [])
    for nbytes in (1 << 20, (2 << 30) // n):
        count = nbytes // es
        x = np.stack([W.uniform_rank(r, count, dtype) for r in range(n)])
        pool.load(x, dtype=dtype)
        for i, algo in enumerate(orders):
            op = "sum" if i % 2 == 0 else "max"
            bufs = [to_dev(x[r]) for r in range(n)]
            ar.check(ar.ar_allreduce(bufs, count=count, dtype=dtype, op=op, algo=algo), "sweep point")
            torch.cuda.synchronize()
            for r in range(1, n):
                assert torch.equal(bufs[r], bufs[0]), (algo, r)
            res0 = bufs[0].cpu().numpy()
            if dtype == "bf16":
                res0 = res0.view(np.uint16)
            del bufs
            pool.run(algo=ORACLE_ALGO.get(algo, algo), op=op)
            cmp = pool.compare(res0)
            assert cmp["bit_identical"], (n, nbytes, algo, op, cmp["differing_ranges"][:3])
        del x


@pytest.mark.slow
@pytest.mark.parametrize("n,nbytes,dtype,op,algo", [
    (16, 256 << 20, "bf16", "sum", "ring"),
    (64, 64 << 20, "f32", "max", "tree"),
    (2, 1 << 30, "f32", "sum", "ring"),
    (8, 512 << 20, "bf16", "sum", "dbtree"),
])
def test_large_sweep_points_sampled(ar, n, nbytes, dtype, op, algo):
    """Sweep points beyond 2 GiB in all: 2^20 seeded sample positions and
    every chunk boundary +-2 carried through the oracle's messages."""
    es = 2 if dtype == "bf16" else 4
    count = nbytes // es
    pos = sample_positions(count, n, 1 << 20, 11)
    if algo == "dbtree":
        pos = np.unique(np.concatenate([pos, [count // 2 - 1, count // 2]]))
    bufs, xs = [], []
    for r in range(n):
        row = W.uniform_rank(r, count, dtype)
        xs.append(row[pos])
        bufs.append(to_dev(row))
        del row
    xs = np.stack(xs)
    with np.errstate(all="ignore"):
        want, _ = oracle.allreduce(xs, algo=algo, op=op, dtype=dtype, count=count, positions=pos)
    ar.check(ar.ar_allreduce(bufs, count=count, dtype=dtype, op=op, algo=algo), "large sweep point")
    torch.cuda.synchronize()
    idx = torch.from_numpy(pos).cuda()
    for r in (0, n // 2, n - 1):
        got = bufs[r][idx].cpu().numpy()
        if dtype == "bf16":
            got = got.view(np.uint16)
        assert_same(got, want[r], dtype, f"rank {r}")
    for r in range(1, n):
        assert torch.equal(bufs[r], bufs[0]), r


@pytest.mark.slow
@pytest.mark.parametrize("dtype,op,algo", [("f32", "sum", "ring"), ("bf16", "max", "tree")])
def test_largest_sweep_point_sampled(ar, dtype, op, algo):
    """The sweep's largest point: 64 ranks x 1 GiB (64 GiB of rank buffers),
    drawn on the device; sampled positions and every chunk boundary go
    through the oracle."""
    n, nbytes = 64, 1 << 30
    free, _ = torch.cuda.mem_get_info()
    if free < n * nbytes + (8 << 30):
        pytest.skip("needs about 72 GiB of free device memory")
    es = 2 if dtype == "bf16" else 4
    count = nbytes // es
    pos = sample_positions(count, n, 1 << 20, 12)
    idx = torch.from_numpy(pos).cuda()
    bufs = [W.uniform_rank_device(r, count, dtype, torch) for r in range(n)]
    xs = np.stack([b[idx].cpu().numpy() for b in bufs])
    if dtype == "bf16":
        xs = xs.view(np.uint16)
    with np.errstate(all="ignore"):
        want, _ = oracle.allreduce(xs, algo=algo, op=op, dtype=dtype, count=count, positions=pos)
    ar.check(ar.ar_allreduce(bufs, count=count, dtype=dtype, op=op, algo=algo), "largest sweep point")
    torch.cuda.synchronize()
    for r in (0, 1, n // 2, n - 1):
        got = bufs[r][idx].cpu().numpy()
        if dtype == "bf16":
            got = got.view(np.uint16)
        assert_same(got, want[r], dtype, f"rank {r}")
    for r in range(1, n):
        assert torch.equal(bufs[r], bufs[0]), r
    del bufs
    torch.cuda.empty_cache()


@pytest.mark.slow
@pytest.mark.parametrize("algo", ["ring", "tree", "dbtree"])
def test_more_than_2g_elements_sampled(ar, algo):
    """2 ranks x (2^31 + 12,345) bf16 (4.3 GB each): element indices and byte
    offsets past 32 bits, on sampled positions, chunk boundaries and the
    double binary tree's half boundary."""
    n, count = 2, (1 << 31) + 12_345
    free, _ = torch.cuda.mem_get_info()
    if free < 3 * n * count * 2:
        pytest.skip("needs about 26 GB of free device memory")
    pos = sample_positions(count, n, 1 << 14, 13)
    pos = np.unique(np.concatenate([pos, count // 2 + np.arange(-2, 3), [(1 << 31) - 1, 1 << 31, count - 1]]))
    pos = pos[(pos >= 0) & (pos < count)]
    idx = torch.from_numpy(pos).cuda()
    bufs = [W.uniform_rank_device(r, count, "bf16", torch, config=21) for r in range(n)]
    xs = np.stack([b[idx].cpu().numpy() for b in bufs]).view(np.uint16)
    want, _ = oracle.allreduce(xs, algo=algo, op="sum", dtype="bf16", count=count, positions=pos)
    ar.check(ar.ar_allreduce(bufs, count=count, dtype="bf16", op="sum", algo=algo), "2G elements")
    torch.cuda.synchronize()
    for r in range(n):
        assert_same(bufs[r][idx].cpu().numpy().view(np.uint16), want[r], "bf16", f"rank {r}")
    assert torch.equal(bufs[0], bufs[1])
    del bufs
    torch.cuda.empty_cache()


@pytest.mark.slow
def test_int8_ef_more_than_2g_elements_sampled(ar):
    """8-bit path on 2 ranks x (2^31 + 300) f32: quantisation blocks and
    chunks past 32-bit indices.  A block that lies in one chunk depends only
    on its own elements and that chunk, so the oracle checks it on a small
    buffer that puts the same block, in the same chunk, at a block boundary
    (the other block of that buffer is zero filler)."""
    n, count = 2, (1 << 31) + 300
    free, _ = torch.cuda.mem_get_info()
    if free < 2 * n * count * 4 + (8 << 30):
        pytest.skip("needs about 44 GB of free device memory")
    x = [W.uniform_rank_device(r, count, "f32", torch, config=22) for r in range(n)]
    e = [torch.zeros(count, dtype=torch.float32, device="cuda") for _ in range(n)]
    starts = [0, 128 * 1000, (1 << 31) - 128, 1 << 31, (count - 1) // 128 * 128]
    blocks = [np.arange(b, min(b + 128, count), dtype=np.int64) for b in starts]
    before = [np.stack([t[torch.from_numpy(b).cuda()].cpu().numpy() for t in x]) for b in blocks]
    ar.check(ar.ar_allreduce_int8_ef(x, e, count=count, op="avg"), "int8 2G")
    torch.cuda.synchronize()
    for b, x0 in zip(blocks, before):
        chunks = {((int(el) + 1) * n - 1) // count for el in b}
        assert len(chunks) == 1
        c, m = chunks.pop(), len(b)
        off = 0 if c == 0 else 128  # chunk 0 = [0, 128) of 256; chunk 1 starts at or before 128 of 128 + m
        small = np.zeros((n, 256 if c == 0 else 128 + m), np.float32)
        small[:, off:off + m] = x0
        wx, we, _ = oracle.int8_ef_allreduce(small, np.zeros_like(small), op="avg")
        idx = torch.from_numpy(b).cuda()
        got_x = np.stack([t[idx].cpu().numpy() for t in x])
        got_e = np.stack([t[idx].cpu().numpy() for t in e])
        assert_same(got_x, wx[:, off:off + m], "f32", f"x block at {b[0]}")
        assert_same(got_e, we[:, off:off + m], "f32", f"e block at {b[0]}")
    del x, e
    torch.cuda.empty_cache()
