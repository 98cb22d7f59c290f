"""Seeded random cases against the oracle: rank counts, sizes, dtypes, ops,
orders, and per-rank buffer offsets (aligned, one shared offset, or offsets
that differ by rank), for the collectives and for bucketed tensor lists."""
import numpy as np
import pytest

import oracle
from allreduce_gradient_reduction_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ES = {"f32": 4, "bf16": 2, "i32": 4, "f16": 2}
TORCH = {"f32": torch.float32, "bf16": torch.int16, "i32": torch.int32, "f16": torch.int16}
HALF = ("bf16", "f16")


@pytest.fixture(scope="module")
def ar():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from allreduce_gradient_reduction_gb300 import build as b
    b.build()
    from allreduce_gradient_reduction_gb300 import binding
    torch.cuda.set_device(0)
    return binding


def place(row, dtype, shift):
    """A device buffer holding `row`, starting `shift` elements into its allocation."""
    a = np.ascontiguousarray(row)
    if dtype in HALF:
        a = a.view(np.int16)
    big = torch.zeros(a.size + shift + 8, dtype=TORCH[dtype], device="cuda")
    v = big[shift:shift + a.size]
    v.copy_(torch.from_numpy(a))
    return v


def host(v, dtype):
    out = v.cpu().numpy()
    return out.view(np.uint16) if dtype in HALF else out


def same_bits(got, want, dtype):
    if dtype == "i32":
        return np.array_equal(got, want)
    bits = np.uint16 if dtype in HALF else np.uint32

    def val(x):
        if dtype == "bf16":
            return (x.astype(np.uint32) << 16).view(np.float32)
        if dtype == "f16":
            return np.ascontiguousarray(x, dtype=np.uint16).view(np.float16)
        return x
    f, g = val(got), val(want)
    nan = np.isnan(f) & np.isnan(g)
    return bool(np.all(nan | (got.view(bits) == want.view(bits))))


def shifts_for(rng, n, dtype):
    vec = 16 // ES[dtype]
    kind = rng.integers(0, 3)
    if kind == 0:
        return [0] * n
    if kind == 1:
        return [int(rng.integers(1, vec))] * n
    return [int(rng.integers(0, vec)) for _ in range(n)]


@pytest.mark.parametrize("block", range(12))
def test_random_collectives(ar, block):
    rng = np.random.default_rng(7000 + block)
    for case in range(50):
        n = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 16, 32, 64]))
        count = int(rng.choice([0, 1, n - 1, n, n + 1, int(rng.integers(1, 300)), int(rng.integers(300, 20000))]))
        count = max(count, 0)
        dtype = str(rng.choice(["f32", "bf16", "i32", "f16"]))
        kind = str(rng.choice(["allreduce", "reduce_scatter", "all_gather", "reduce", "broadcast"]))
        algos = ["ring", "ring_stepwise", "naive", "dbtree"] + (
            ["tree", "tree_stepwise", "binomial_stepwise"] if n & (n - 1) == 0 else [])
        if kind in ("reduce_scatter", "all_gather"):
            algos = [a for a in algos if a not in ("naive", "dbtree", "binomial_stepwise")]
        if kind == "reduce":
            algos = [a for a in algos if a in ("ring", "tree", "naive")]
        algo = str(rng.choice(algos))
        ops = ["sum", "max"] + ([] if dtype == "i32" else ["avg"])
        op = str(rng.choice(ops))
        root = int(rng.integers(0, n))
        x = W.random_bits(n, count, dtype, seed=int(rng.integers(1 << 30))) if rng.random() < 0.3 else (
            W.uniform_inputs(n, count, dtype, config=int(rng.integers(1 << 20))) if count else
            np.zeros((n, 0), dtype=np.uint16 if dtype in HALF else (np.int32 if dtype == "i32" else np.float32)))
        shifts = shifts_for(rng, n, dtype)
        bufs = [place(x[r], dtype, shifts[r]) for r in range(n)]
        oa = {"ring_stepwise": "ring", "tree_stepwise": "tree", "binomial_stepwise": "binomial"}.get(algo, algo)
        what = f"case {block}/{case}: {kind} {algo} {dtype} {op} n={n} count={count} shifts={shifts}"
        with np.errstate(all="ignore"):
            if kind == "allreduce":
                want, _ = oracle.allreduce(x, algo=oa, op=op, dtype=dtype)
                ar.check(ar.ar_allreduce(bufs, count=count, dtype=dtype, op=op, algo=algo), what)
            elif kind == "reduce_scatter":
                want, _ = oracle.reduce_scatter(x, algo=oa, op=op, dtype=dtype)
                ar.check(ar.ar_reduce_scatter(bufs, count=count, dtype=dtype, op=op, algo=algo), what)
            elif kind == "all_gather":
                want, _ = oracle.all_gather(x, algo=oa, dtype=dtype)
                ar.check(ar.ar_all_gather(bufs, count=count, dtype=dtype, algo=algo), what)
            elif kind == "reduce":
                want, _ = oracle.reduce(x, algo=oa, op=op, dtype=dtype, root=root)
                ar.check(ar.ar_reduce(bufs, count=count, dtype=dtype, op=op, algo=algo, root=root), what)
            else:
                want, _ = oracle.broadcast(x, root=root, dtype=dtype)
                ar.check(ar.ar_broadcast(bufs, count=count, dtype=dtype, root=root), what)
        torch.cuda.synchronize()
        for r in range(n):
            got = host(bufs[r], dtype)
            if kind == "reduce_scatter":
                lo, hi = oracle.chunk_range(count, n, r)
                assert same_bits(got[lo:hi], want[r][lo:hi], dtype), f"{what} rank {r}"
            elif kind == "reduce":
                if r == root:
                    assert same_bits(got, want[r], dtype), f"{what} root"
                else:
                    assert same_bits(got, x[r], dtype), f"{what} non-root rank {r} changed"
            else:
                assert same_bits(got, want[r], dtype), f"{what} rank {r}"
        rc, st = ar.ar_device_status()
        assert rc == 0 and st == 0, what


@pytest.mark.parametrize("block", range(6))
def test_random_bucketed(ar, block):
    rng = np.random.default_rng(8000 + block)
    for case in range(12):
        n = int(rng.choice([2, 3, 4, 8, 16, 32, 64]))  # 16-64: several launch tables per bucketed call
        t = int(rng.integers(1, 12))
        counts = [int(rng.choice([0, 1, 7, int(rng.integers(1, 5000))])) for _ in range(t)]
        if sum(counts) == 0:
            counts[0] = 5
        cap = int(rng.choice([64, 4096, 16384, 25 << 20]))
        algo = str(rng.choice(["ring", "tree", "ring_stepwise"] if n & (n - 1) == 0 else ["ring", "ring_stepwise"]))
        path = str(rng.choice(["fused", "literal"]))
        grads = [[W.normal_inputs(1, c, 1.0, int(rng.integers(1 << 20)))[0] for c in counts] for _ in range(n)]
        want, _ = oracle.bucketed_allreduce(grads, op="avg", dtype="f32", algo=algo.replace("_stepwise", ""),
                                            cap_bytes=cap)
        shifts = [shifts_for(rng, n, "f32") for _ in range(t)]  # per tensor, per rank
        dg = [[place(grads[r][i], "f32", shifts[i][r]) for i in range(t)] for r in range(n)]
        ws = None
        if path == "literal":
            ws = [torch.empty(max(sum(counts), 1), dtype=torch.float32, device="cuda") for _ in range(n)]
        what = f"bucketed case {block}/{case}: n={n} counts={counts} cap={cap} {algo} {path}"
        ar.check(ar.ar_bucketed_allreduce(dg, counts=counts, dtype="f32", op="avg", algo=algo, bucket_cap_bytes=cap,
                                          workspace=ws), what)
        torch.cuda.synchronize()
        for r in range(n):
            for i in range(t):
                assert same_bits(host(dg[r][i], "f32"), want[r][i], "f32"), f"{what} rank {r} tensor {i}"


@pytest.mark.parametrize("block", range(4))
def test_random_int8_ef(ar, block):
    rng = np.random.default_rng(9000 + block)
    for case in range(15):
        n = int(rng.choice([1, 2, 3, 4, 5, 8, 13, 16]))
        count = int(rng.choice([0, 1, 127, 128, 129, int(rng.integers(1, 3000)), int(rng.integers(3000, 40000))]))
        op = str(rng.choice(["sum", "avg"]))
        shift = int(rng.choice([0, 0, 1, 3]))  # elements, the same for every buffer
        x = W.normal_inputs(n, count, float(rng.choice([1e-3, 1.0, 50.0])), int(rng.integers(1 << 20)))
        e = W.normal_inputs(n, count, 1e-5, int(rng.integers(1 << 20)))
        what = f"int8 case {block}/{case}: n={n} count={count} {op} shift={shift}"
        for it in range(2):  # the residuals carry over
            want_x, want_e, _ = oracle.int8_ef_allreduce(x, e, op=op)
            xd = [place(x[r], "f32", shift) for r in range(n)]
            ed = [place(e[r], "f32", shift) for r in range(n)]
            ar.check(ar.ar_allreduce_int8_ef(xd, ed, count=count, op=op), what)
            torch.cuda.synchronize()
            for r in range(n):
                assert same_bits(host(xd[r], "f32"), want_x[r], "f32"), f"{what} it={it} x rank {r}"
                assert same_bits(host(ed[r], "f32"), want_e[r], "f32"), f"{what} it={it} e rank {r}"
            e = np.stack([host(t, "f32") for t in ed]) if count else e
            x = W.normal_inputs(n, count, 1e-3, int(rng.integers(1 << 20)))


@pytest.mark.parametrize("block", range(2))
def test_random_plans(ar, block):
    """Prepared calls, each run three times on new data, against the oracle."""
    rng = np.random.default_rng(9500 + block)
    for case in range(10):
        n = int(rng.choice([2, 3, 4, 8, 16]))
        count = int(rng.integers(1, 20000))
        dtype = str(rng.choice(["f32", "bf16", "i32", "f16"]))
        kind = str(rng.choice(["allreduce", "reduce_scatter", "all_gather", "reduce"]))
        algos = ["ring", "ring_stepwise"] + (["tree", "tree_stepwise"] if n & (n - 1) == 0 else [])
        if kind == "allreduce":
            algos += ["naive", "dbtree"]
        if kind == "reduce":
            algos = [a for a in algos if not a.endswith("stepwise")] + ["naive"]
        algo = str(rng.choice(algos))
        op = str(rng.choice(["sum", "max"] + ([] if dtype == "i32" else ["avg"])))
        root = int(rng.integers(0, n))
        shifts = shifts_for(rng, n, dtype)
        bufs = [place(np.zeros(count, dtype={"f32": np.float32, "bf16": np.uint16, "i32": np.int32, "f16": np.uint16}[dtype]),
                      dtype, shifts[r]) for r in range(n)]
        plan = ar.Plan(kind, bufs, count=count, dtype=dtype, op=op, algo=algo, root=root)
        oa = {"ring_stepwise": "ring", "tree_stepwise": "tree", "binomial_stepwise": "binomial"}.get(algo, algo)
        what = f"plan case {block}/{case}: {kind} {algo} {dtype} {op} n={n} count={count}"
        for it in range(3):
            x = W.uniform_inputs(n, count, dtype, config=int(rng.integers(1 << 20)))
            for r in range(n):
                src = np.ascontiguousarray(x[r])
                bufs[r].copy_(torch.from_numpy(src.view(np.int16) if dtype in HALF else src))
            ar.check(plan.run(), what)
            torch.cuda.synchronize()
            with np.errstate(all="ignore"):
                if kind == "allreduce":
                    want, _ = oracle.allreduce(x, algo=oa, op=op, dtype=dtype)
                elif kind == "reduce_scatter":
                    want, _ = oracle.reduce_scatter(x, algo=oa, op=op, dtype=dtype)
                elif kind == "all_gather":
                    want, _ = oracle.all_gather(x, algo=oa, dtype=dtype)
                else:
                    want, _ = oracle.reduce(x, algo=oa, op=op, dtype=dtype, root=root)
            for r in range(n):
                got = host(bufs[r], dtype)
                if kind == "reduce_scatter":
                    lo, hi = oracle.chunk_range(count, n, r)
                    assert same_bits(got[lo:hi], want[r][lo:hi], dtype), f"{what} it={it} rank {r}"
                elif kind == "reduce":
                    if r == root:
                        assert same_bits(got, want[r], dtype), f"{what} it={it} root"
                else:
                    assert same_bits(got, want[r], dtype), f"{what} it={it} rank {r}"
        plan.close()


@pytest.mark.parametrize("block", range(4))
def test_random_host_buffer_calls(ar, block):
    """ar_allreduce_host with random shapes, orders, piece sizes, host-row
    offsets, page-locked or pageable rows, zero-copy or staged."""
    rng = np.random.default_rng(9500 + block)
    for case in range(10):
        n = int(rng.choice([1, 2, 3, 4, 8, 16, 64]))
        count = int(rng.choice([1, n + 1, int(rng.integers(1, 3000)), int(rng.integers(3000, 60000))]))
        dtype = str(rng.choice(["f32", "bf16", "i32", "f16"]))
        algos = ["ring", "naive", "dbtree"] + (["tree"] if n & (n - 1) == 0 else [])
        algo = str(rng.choice(algos))
        op = str(rng.choice(["sum", "max"] + ([] if dtype == "i32" else ["avg"])))
        pinned = bool(rng.integers(0, 2))
        mode = str(rng.choice(["zero_copy", "staged"])) if pinned else "staged"
        piece = int(rng.choice([0, 64, int(rng.integers(1, 5000))]))
        x = (W.random_bits(n, count, dtype, int(rng.integers(1 << 20))) if op != "sum" or dtype == "i32"
             else W.normal_inputs(n, count, 1.0, int(rng.integers(1 << 20))) if dtype == "f32"
             else W.large_inputs(n, count, config=int(rng.integers(1 << 20))) if dtype == "bf16"
             else W.uniform_inputs(n, count, "f16", config=int(rng.integers(1 << 20))))
        with np.errstate(all="ignore"):
            want, _ = oracle.allreduce(x, algo=algo, op=op, dtype=dtype)
        shifts = shifts_for(rng, n, dtype)
        a = np.ascontiguousarray(x).view(np.int16) if dtype in HALF else np.ascontiguousarray(x)
        block_t = torch.zeros((n, count + 8), dtype=TORCH[dtype])
        if pinned:
            block_t = block_t.pin_memory()
        rows = []
        for r in range(n):
            block_t[r, shifts[r]:shifts[r] + count] = torch.from_numpy(a[r])
            rows.append(block_t[r, shifts[r]:shifts[r] + count])
        dv = None if mode == "zero_copy" else [place(np.zeros(count, dtype=a.dtype), dtype, s) for s in shifts]
        what = f"host case {block}/{case}: n={n} count={count} {dtype} {op} {algo} {mode} pinned={pinned} piece={piece}"
        ar.check(ar.ar_allreduce_host(rows, dv, count=count, dtype=dtype, op=op, algo=algo, piece_elems=piece), what)
        torch.cuda.synchronize()
        for r in range(n):
            got = rows[r].numpy()
            assert same_bits(got.view(np.uint16) if dtype in HALF else got, want[r], dtype), f"{what} rank {r}"
