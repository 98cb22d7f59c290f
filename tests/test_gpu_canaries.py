"""Out-of-bounds writes, caught with guard bands instead of a memory
sanitizer.  Every rank buffer sits inside a larger allocation
between guard bands filled with a byte pattern; after each call the bands
must be untouched.  Sizes are odd, ragged and unaligned (element-aligned but
not 16-byte aligned), so every tail and scalar path runs."""
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

GUARD = 4096
PATTERN = 0xA5
ES = {"f32": 4, "bf16": 2, "i32": 4, "f16": 2}
TORCH = {"f32": torch.float32, "bf16": torch.int16, "i32": torch.int32, "f16": torch.int16}


@pytest.fixture(scope="module")
def ar():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from allreduce_gradient_reduction_gb300 import build as b
    b.build()
    from allreduce_gradient_reduction_gb300 import binding
    torch.cuda.set_device(0)
    return binding


class Guarded:
    """`n` buffers of `count` elements, each at byte offset GUARD + shift of
    its own allocation of GUARD + shift + count * es + GUARD bytes."""

    def __init__(self, n, count, dtype, shift, seed):
        es = ES[dtype]
        shifts = shift if isinstance(shift, (list, tuple)) else [shift] * n  # bytes, per rank
        self.span = [(GUARD + sh, GUARD + sh + count * es) for sh in shifts]
        self.raw = [torch.full((hi + GUARD,), PATTERN, dtype=torch.uint8, device="cuda") for _, hi in self.span]
        g = torch.Generator(device="cuda")
        g.manual_seed(seed)
        self.bufs = []
        for r, (lo, hi) in zip(self.raw, self.span):
            v = r[lo:hi].view(TORCH[dtype])
            if dtype == "f32":
                v.copy_(torch.randn(count, device="cuda", generator=g))
            else:
                v.copy_(torch.randint(-1000, 1000, (count,), device="cuda", generator=g).to(TORCH[dtype]))
            self.bufs.append(v)

    def check(self, what):
        torch.cuda.synchronize()
        for i, (r, (lo, hi)) in enumerate(zip(self.raw, self.span)):
            head, tail = r[:lo].cpu().numpy(), r[hi:].cpu().numpy()
            assert (head == PATTERN).all(), f"{what}: rank {i} wrote before its buffer"
            assert (tail == PATTERN).all(), f"{what}: rank {i} wrote past its buffer"


def sizes(n):
    return [1, n - 1, n + 1, 127, 1000, 4099, 3 * 2048 * n + 13]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
@pytest.mark.parametrize("n", [2, 3, 8, 12, 16])
def test_collectives_stay_inside_their_buffers(ar, n, dtype):
    algos = ["ring", "ring_stepwise", "naive", "dbtree"] + (
        ["tree", "tree_stepwise", "binomial_stepwise"] if n & (n - 1) == 0 else [])
    for count in [c for c in sizes(n) if c > 0]:
        # aligned; the same offset in every rank (vectors cut at it); offsets
        # differing by rank (the staged kernel, or one element per thread)
        for shift in (0, ES[dtype], [(r * ES[dtype]) % 16 for r in range(n)]):
            G = Guarded(n, count, dtype, shift, seed=count + n)
            for algo in algos:
                ar.check(ar.ar_allreduce(G.bufs, count=count, dtype=dtype, op="max", algo=algo), "allreduce")
                G.check(f"allreduce {algo} n={n} count={count} shift={shift}")
                if algo in ("naive", "dbtree", "binomial_stepwise"):
                    continue
                ar.check(ar.ar_reduce_scatter(G.bufs, count=count, dtype=dtype, op="max", algo=algo), "rs")
                G.check(f"reduce_scatter {algo} n={n} count={count} shift={shift}")
                ar.check(ar.ar_all_gather(G.bufs, count=count, dtype=dtype, algo=algo), "ag")
                G.check(f"all_gather {algo} n={n} count={count} shift={shift}")
                if not algo.endswith("stepwise"):
                    ar.check(ar.ar_reduce(G.bufs, count=count, dtype=dtype, op="max", algo=algo, root=n - 1), "reduce")
                    G.check(f"reduce {algo} n={n} count={count} shift={shift}")
            ar.check(ar.ar_broadcast(G.bufs, count=count, dtype=dtype, root=n // 2), "broadcast")
            G.check(f"broadcast n={n} count={count} shift={shift}")


@pytest.mark.parametrize("n", [2, 3, 8])
def test_int8_ef_stays_inside_its_buffers(ar, n):
    for count in (1, 127, 129, 1000, 128 * 3 * n + 77):
        for shift in (0, 4, [(4 * r) % 16 for r in range(n)]):
            X = Guarded(n, count, "f32", shift, seed=5 + count)
            E = Guarded(n, count, "f32", shift, seed=6 + count)
            ar.check(ar.ar_allreduce_int8_ef(X.bufs, E.bufs, count=count, op="avg"), "int8_ef")
            X.check(f"int8 grads n={n} count={count} shift={shift}")
            E.check(f"int8 residuals n={n} count={count} shift={shift}")


@pytest.mark.parametrize("path", ["fused", "literal_per_bucket", "literal_all_buckets"])
def test_bucketed_stays_inside_its_tensors(ar, path):
    n = 4
    counts = [1, 7, 4099, 129, 33_000, 5, 2048 * 3 + 1]
    cap = 64 * 1024  # several buckets, one tensor larger than a bucket
    tensors = [[Guarded(1, c, "f32", 4 * (t % 2), seed=100 * r + t) for t, c in enumerate(counts)] for r in range(n)]
    grads = [[g.bufs[0] for g in row] for row in tensors]
    ws = None
    if path != "fused":
        _, bo, off, bc = ar.ar_bucket_plan(counts, "f32", cap)
        wsg = Guarded(n, max(bc) if path == "literal_per_bucket" else sum(bc), "f32", 0, seed=9)
        ws = wsg.bufs
    ar.check(ar.ar_bucketed_allreduce(grads, counts=counts, dtype="f32", op="avg", bucket_cap_bytes=cap,
                                      workspace=ws), "bucketed")
    for r, row in enumerate(tensors):
        for t, g in enumerate(row):
            g.check(f"{path} bucketed rank {r} tensor {t}")
    if ws is not None:
        wsg.check("literal workspace")
