"""Pins for the CPU oracle: values and invariants fixed by the pages or by
arithmetic, each chosen so that a plausible mistake in the oracle (a wrong
chunk rotation, a dropped step, a wrong rounding, a transposed operand, a
miscounted message) fails at least one of them.  No GPU needed."""
from fractions import Fraction
import math
import os

import numpy as np
import pytest

import oracle
from allreduce_gradient_reduction_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ALL_DTYPES = ("f32", "bf16", "i32", "f16")


def read_golden(name):
    spec = {"ranks": {}}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "rank":
                spec["ranks"][int(vals[0])] = [float(v) for v in vals[1:]]
            elif key in ("nranks", "count"):
                spec[key] = int(vals[0])
            elif key == "op":
                spec[key] = vals[0]
            else:
                spec[key] = [float(v) for v in vals]
    return spec


def to_storage(vals, dtype):
    a = np.asarray(vals, dtype=np.float32)
    if dtype == "f32":
        return a
    if dtype == "i32":
        return a.astype(np.int32)
    if dtype == "f16":
        return a.astype(np.float16).view(np.uint16)  # the golden values are exact in binary16
    return (a.view(np.uint32) >> 16).astype(np.uint16)  # the golden values are exact in bf16


def to_f64(x, dtype):
    x = np.asarray(x)
    if dtype == "bf16":
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype == "f16":
        return np.ascontiguousarray(x, dtype=np.uint16).view(np.float16).astype(np.float64)
    return x.astype(np.float64)


def algos_for(n):
    out = ["ring", "naive", "dbtree"]
    if n & (n - 1) == 0:
        out += ["tree", "binomial"]
    return out


# --------------------------------------------------------------------------
# Worked examples printed on the pages
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ALL_DTYPES)
@pytest.mark.parametrize("name", ["three_rank_sum.txt", "four_rank_ones.txt"])
def test_printed_sum_examples(oracle_lib, name, dtype):
    g = read_golden(name)
    x = np.stack([to_storage(g["ranks"][r], dtype) for r in range(g["nranks"])])
    for algo in algos_for(g["nranks"]):
        out, st = oracle.allreduce(x, algo=algo, op="sum", dtype=dtype)
        assert np.all(to_f64(out, dtype) == np.asarray(g["expect"])[None, :]), algo


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_printed_ddp_average(oracle_lib, dtype):
    g = read_golden("ddp_average.txt")
    x = np.stack([to_storage(g["ranks"][r], dtype) for r in range(g["nranks"])])
    for algo in algos_for(g["nranks"]):
        s, _ = oracle.allreduce(x, algo=algo, op="sum", dtype=dtype)
        a, _ = oracle.allreduce(x, algo=algo, op="avg", dtype=dtype)
        assert np.all(to_f64(s, dtype) == g["expect_sum"]), algo
        assert np.all(to_f64(a, dtype) == g["expect_avg"]), algo


@pytest.mark.parametrize("n", [2, 3, 5, 8, 16])
def test_ddp_average_general_n(oracle_lib, n):
    # ones * rank summed over N ranks is N(N-1)/2; divided by N it is (N-1)/2
    x = np.stack([np.full(7, r, dtype=np.float32) for r in range(n)])
    out, _ = oracle.allreduce(x, op="avg", dtype="f32")
    assert np.all(out == np.float32((n - 1) / 2))


# --------------------------------------------------------------------------
# Chunk partition
# --------------------------------------------------------------------------

@pytest.mark.parametrize("count,n", [(0, 1), (0, 5), (1, 3), (7, 8), (8, 8), (9, 8), (4096, 4), (1001, 7),
                                     (67_108_864, 8), ((1 << 40) + 3, 64)])
def test_chunk_partition(oracle_lib, count, n):
    rngs = [oracle.chunk_range(count, n, c) for c in range(n)]
    assert rngs[0][0] == 0 and rngs[-1][1] == count
    for (lo, hi), (lo2, _) in zip(rngs, rngs[1:]):
        assert hi == lo2  # contiguous, in order
    sizes = [hi - lo for lo, hi in rngs]
    assert min(sizes) >= 0 and max(sizes) - min(sizes) <= 1
    if count % n == 0:
        assert all(s == count // n for s in sizes)


def test_chunk_partition_three_rank_scalar(oracle_lib):
    # one element split three ways: the element lies in the last chunk
    assert [oracle.chunk_range(1, 3, c) for c in range(3)] == [(0, 0), (0, 0), (0, 1)]


# --------------------------------------------------------------------------
# Elementwise arithmetic
# --------------------------------------------------------------------------

def bf16_round_by_value(v):
    """Round finite float64 values to bf16 by value: find the bf16 grid
    spacing of the binade, take the two neighbours, pick the nearer, ties to
    the even multiple; magnitudes at 2^128 and beyond become infinity."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, e = np.frexp(a)
    ulp = np.ldexp(1.0, np.maximum(e - 8, -133))
    q = a / ulp
    fl = np.floor(q)
    rem = q - fl
    up = (rem > 0.5) | ((rem == 0.5) & (np.fmod(fl, 2.0) == 1.0))
    r = (fl + up) * ulp
    r = np.where(r >= 2.0 ** 128, np.inf, r)
    return np.copysign(r, v)


def test_bf16_rounding_edges(oracle_lib):
    hi = np.arange(1 << 16, dtype=np.uint32)
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x4000, 0xC000], dtype=np.uint32)
    bits = (hi[:, None] << 16 | lows[None, :]).reshape(-1)
    f = bits.view(np.float32)
    finite = np.isfinite(f)
    got = oracle.f32_to_bf16(f)
    gv = to_f64(got, "bf16")
    want = bf16_round_by_value(f[finite].astype(np.float64))
    assert np.array_equal(gv[finite], want)
    assert np.array_equal(np.signbit(gv[finite]), np.signbit(want))
    # infinities stay, NaNs stay NaN
    inf = np.isinf(f)
    assert np.array_equal(gv[inf], f[inf].astype(np.float64))
    assert np.all(np.isnan(gv[np.isnan(f)]))


def test_bf16_rounding_random(oracle_lib):
    g = np.random.Generator(np.random.PCG64(7))
    bits = g.integers(0, 1 << 32, size=2_000_000, dtype=np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    gv = to_f64(oracle.f32_to_bf16(f), "bf16")
    assert np.array_equal(gv, bf16_round_by_value(f.astype(np.float64)))


def _frac_round_bf16(x: Fraction):
    """Correctly rounded bf16 value of an exact rational (nearest, ties even);
    returns a float (inf on overflow)."""
    if x == 0:
        return 0.0
    s = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** max(e - 7, -133)
    q = a / ulp
    fl = q.numerator // q.denominator
    rem = q - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * ulp
    if r >= Fraction(2) ** 128:
        return s * math.inf
    return s * float(r)


def _bf16_pairs(n, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    a = g.integers(0, 1 << 16, size=n, dtype=np.uint16)
    # b near a in exponent half the time, so rounding is non-trivial
    b_near = (a.astype(np.int32) + g.integers(-2000, 2000, size=n)).clip(0, 0xFFFF).astype(np.uint16)
    b_near ^= (g.integers(0, 2, size=n, dtype=np.uint16) << 15)
    b_far = g.integers(0, 1 << 16, size=n, dtype=np.uint16)
    b = np.where(g.random(n) < 0.5, b_near, b_far).astype(np.uint16)
    fa, fb = to_f64(a, "bf16"), to_f64(b, "bf16")
    keep = np.isfinite(fa) & np.isfinite(fb)
    return a[keep], b[keep]


def test_bf16_add_is_correctly_rounded(oracle_lib):
    a, b = _bf16_pairs(30000, 11)
    got = to_f64(oracle.step(a, b, op="sum", dtype="bf16"), "bf16")
    fa, fb = to_f64(a, "bf16"), to_f64(b, "bf16")
    for i in range(a.size):
        exact = Fraction(float(fa[i])) + Fraction(float(fb[i]))
        want = _frac_round_bf16(exact)
        if exact == 0:
            want = -0.0 if (math.copysign(1, fa[i]) < 0 and math.copysign(1, fb[i]) < 0) else 0.0
        assert got[i] == want and math.copysign(1, got[i]) == math.copysign(1, want), (hex(a[i]), hex(b[i]))


def test_bf16_add_matches_torch_cpu(oracle_lib):
    torch = pytest.importorskip("torch")
    a, b = _bf16_pairs(1_000_000, 12)
    got = oracle.step(a, b, op="sum", dtype="bf16")
    ta = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    tb = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)
    want = (ta + tb).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(to_f64(want, "bf16"))
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all(np.isnan(to_f64(got[nan], "bf16")))


def test_f32_add_matches_numpy(oracle_lib):
    a = W.random_bits(1, 500_000, "f32", 3)[0]
    b = W.random_bits(1, 500_000, "f32", 4)[0]
    b[::3] = a[::3] * np.float32(-0.75)  # cancellation
    with np.errstate(all="ignore"):
        want = a + b
    got = oracle.step(a, b, op="sum", dtype="f32")
    nan = np.isnan(want)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))
    assert np.all(np.isnan(got[nan]))


def test_i32_add_wraps(oracle_lib):
    a = np.array([2**31 - 1, -2**31, 5, -7, 0], dtype=np.int32)
    b = np.array([1, -1, -5, 7, 0], dtype=np.int32)
    want = [((int(x) + int(y) + 2**31) % 2**32) - 2**31 for x, y in zip(a, b)]
    assert oracle.step(a, b, op="sum", dtype="i32").tolist() == want


def test_max_special_values(oracle_lib):
    nan, inf = np.float32("nan"), np.float32("inf")
    a = np.array([0.0, -0.0, -0.0, nan, 1.0, -inf, 3.0, -2.0], dtype=np.float32)
    b = np.array([-0.0, 0.0, -0.0, 1.0, nan, 5.0, 2.0, -1.0], dtype=np.float32)
    got = oracle.step(a, b, op="max", dtype="f32")
    assert got[0] == 0 and not np.signbit(got[0])
    assert got[1] == 0 and not np.signbit(got[1])
    assert got[2] == 0 and np.signbit(got[2])
    assert np.isnan(got[3]) and np.isnan(got[4])
    assert got[5:].tolist() == [5.0, 3.0, -1.0]
    ab, bb = to_storage(a, "f32"), to_storage(b, "f32")
    ab = (a.view(np.uint32) >> 16).astype(np.uint16)
    bb = (b.view(np.uint32) >> 16).astype(np.uint16)
    gb = to_f64(oracle.step(ab, bb, op="max", dtype="bf16"), "bf16")
    assert gb[0] == 0 and not np.signbit(gb[0])
    assert gb[2] == 0 and np.signbit(gb[2])
    assert np.isnan(gb[3]) and np.isnan(gb[4])
    assert gb[5:].tolist() == [5.0, 3.0, -1.0]
    ia = np.array([-5, 7, -2**31], dtype=np.int32)
    ib = np.array([3, -9, 2**31 - 1], dtype=np.int32)
    assert oracle.step(ia, ib, op="max", dtype="i32").tolist() == [3, 7, 2**31 - 1]


# --------------------------------------------------------------------------
# binary16 (f16): conversions and the SUM / AVG / MAX steps
# --------------------------------------------------------------------------

def _frac_round_f16(x: Fraction):
    """Correctly rounded binary16 value of an exact rational (nearest, ties to
    even; 10 fraction bits, unit 2^-24 below the normal range); a float, inf
    when the rounded magnitude reaches 2^16."""
    if x == 0:
        return 0.0
    s = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** max(e - 10, -24)
    q = a / ulp
    fl = q.numerator // q.denominator
    rem = q - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * ulp
    if r >= 2 ** 16:
        return s * math.inf
    return s * float(r)


def test_f16_decodes_every_pattern(oracle_lib):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f32(h)
    want = h.view(np.float16).astype(np.float32)  # numpy's binary16 widening
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))
    # and every non-NaN pattern survives the trip back
    assert np.array_equal(oracle.f32_to_f16(got[~nan]), h[~nan])


def test_f16_rounding_by_value(oracle_lib):
    # ties and near-ties at the subnormal unit, the normal/subnormal boundary,
    # the top binade and the overflow threshold, plus their neighbours
    base = [2.0 ** -25, 3 * 2.0 ** -25, 2.0 ** -24, 1.5 * 2.0 ** -24, 2.0 ** -14 - 2.0 ** -25,
            2.0 ** -14 - 2.0 ** -26, 2.0 ** -14, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 2049.0, 2051.0,
            65504.0, 65505.0, 65519.0, 65520.0, 65536.0, 1e-9, 0.1, 1.0 / 3.0, 1e5]
    f = np.array(base, dtype=np.float32)
    f = np.concatenate([f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(0))])
    f = np.concatenate([f, -f])
    got = to_f64(oracle.f32_to_f16(f), "f16")
    for v, g in zip(f.tolist(), got.tolist()):
        want = _frac_round_f16(Fraction(v))
        assert g == want and math.copysign(1, g) == math.copysign(1, v if want == 0 else want), (v, g, want)


def test_f16_rounding_matches_numpy(oracle_lib):
    g = np.random.Generator(np.random.PCG64(16))
    # magnitudes from far below the smallest subnormal to past the overflow threshold
    f = (g.standard_normal(2_000_000) * np.exp2(g.uniform(-30, 18, 2_000_000))).astype(np.float32)
    with np.errstate(over="ignore"):
        want = f.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.f32_to_f16(f), want)


def _f16_pairs(n, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    a = g.integers(0, 1 << 16, size=n, dtype=np.uint16)
    b_near = (a.astype(np.int32) + g.integers(-1500, 1500, size=n)).clip(0, 0xFFFF).astype(np.uint16)
    b_near ^= (g.integers(0, 2, size=n, dtype=np.uint16) << 15)
    b_far = g.integers(0, 1 << 16, size=n, dtype=np.uint16)
    b = np.where(g.random(n) < 0.5, b_near, b_far).astype(np.uint16)
    fa, fb = to_f64(a, "f16"), to_f64(b, "f16")
    keep = np.isfinite(fa) & np.isfinite(fb)
    return a[keep], b[keep]


def test_f16_add_is_correctly_rounded(oracle_lib):
    a, b = _f16_pairs(30000, 21)
    got = to_f64(oracle.step(a, b, op="sum", dtype="f16"), "f16")
    fa, fb = to_f64(a, "f16"), to_f64(b, "f16")
    for i in range(a.size):
        exact = Fraction(float(fa[i])) + Fraction(float(fb[i]))
        want = _frac_round_f16(exact)
        if exact == 0:
            want = -0.0 if (math.copysign(1, fa[i]) < 0 and math.copysign(1, fb[i]) < 0) else 0.0
        assert got[i] == want and math.copysign(1, got[i]) == math.copysign(1, want), (hex(a[i]), hex(b[i]))


def test_f16_add_matches_numpy(oracle_lib):
    a, b = _f16_pairs(1_000_000, 22)
    got = oracle.step(a, b, op="sum", dtype="f16")
    with np.errstate(over="ignore"):
        want = (a.view(np.float16) + b.view(np.float16)).view(np.uint16)
    assert np.array_equal(got, want)


def test_f16_avg_is_the_correctly_rounded_quotient(oracle_lib):
    for n in (2, 3, 5, 8, 13, 64):
        x = W.uniform_inputs(n, 3000, "f16", config=40 + n)
        s, _ = oracle.allreduce(x, algo="ring", op="sum", dtype="f16")
        a, _ = oracle.allreduce(x, algo="ring", op="avg", dtype="f16")
        sv, av = to_f64(s[0], "f16"), to_f64(a[0], "f16")
        for i in range(sv.size):
            want = _frac_round_f16(Fraction(float(sv[i])) / n)
            if want == 0:
                want = math.copysign(0.0, sv[i])
            assert av[i] == want and math.copysign(1, av[i]) == math.copysign(1, want), (n, i, sv[i])


def test_f16_max_special_values(oracle_lib):
    nan, inf = np.float16("nan"), np.float16("inf")
    a = np.array([0.0, -0.0, -0.0, nan, 1.0, -inf, 3.0, -2.0, 6e-8], dtype=np.float16)
    b = np.array([-0.0, 0.0, -0.0, 1.0, nan, 5.0, 2.0, -1.0, -6e-8], dtype=np.float16)
    got = to_f64(oracle.step(a.view(np.uint16), b.view(np.uint16), op="max", dtype="f16"), "f16")
    assert got[0] == 0 and not np.signbit(got[0])
    assert got[1] == 0 and not np.signbit(got[1])
    assert got[2] == 0 and np.signbit(got[2])
    assert np.isnan(got[3]) and np.isnan(got[4])
    assert got[5:].tolist() == [5.0, 3.0, -1.0, float(np.float16(6e-8))]


# --------------------------------------------------------------------------
# Brute force on tiny inputs: order-free results must be exact
# --------------------------------------------------------------------------

SIZES = [0, 1, 2, 3, 5, 7, 8, 9, 31, 257, 1000]


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8])
def test_bruteforce_integers_and_max(oracle_lib, n):
    g = np.random.Generator(np.random.PCG64(100 + n))
    for count in SIZES + [n - 1, n, n + 1]:
        if count < 0:
            continue
        xi = g.integers(-2**31, 2**31, size=(n, count), dtype=np.int64).astype(np.int32)
        exact = ((xi.astype(object).sum(axis=0) + 2**31) % 2**32) - 2**31 if count else np.zeros(0)
        xf = g.integers(-8, 9, size=(n, count)).astype(np.float32)
        xb = to_storage(xf.reshape(-1), "bf16").reshape(n, count)
        xr = g.standard_normal((n, count)).astype(np.float32)
        for algo in algos_for(n):
            out, _ = oracle.allreduce(xi, algo=algo, op="sum", dtype="i32")
            assert [list(map(int, row)) for row in out] == [list(map(int, exact))] * n, (algo, count)
            out, _ = oracle.allreduce(xi, algo=algo, op="max", dtype="i32")
            assert np.array_equal(out, np.broadcast_to(xi.max(axis=0), out.shape))
            out, _ = oracle.allreduce(xf, algo=algo, op="sum", dtype="f32")
            assert np.array_equal(out, np.broadcast_to(xf.astype(np.float64).sum(axis=0), out.shape))
            out, _ = oracle.allreduce(xb, algo=algo, op="sum", dtype="bf16")  # |sum| <= 64: exact in bf16
            assert np.array_equal(to_f64(out, "bf16"), np.broadcast_to(xf.astype(np.float64).sum(axis=0), out.shape))
            out, _ = oracle.allreduce(to_storage(xf.reshape(-1), "f16").reshape(n, count), algo=algo, op="sum",
                                      dtype="f16")  # exact in binary16 too
            assert np.array_equal(to_f64(out, "f16"), np.broadcast_to(xf.astype(np.float64).sum(axis=0), out.shape))
            out, _ = oracle.allreduce(xr, algo=algo, op="max", dtype="f32")
            assert np.array_equal(out, np.broadcast_to(xr.max(axis=0), out.shape))


# --------------------------------------------------------------------------
# Fold order: the message simulation equals the closed-form per-element fold
# --------------------------------------------------------------------------

def _lib_add(dtype):
    """Addition by a library routine in the storage type: numpy float32 /
    int32, torch's CPU bf16 addition."""
    if dtype == "bf16":
        import torch

        def add(a, b):
            ta = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
            tb = torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)
            return (ta + tb).view(torch.int16).numpy().view(np.uint16)
        return add
    if dtype == "f16":
        return lambda a, b: (np.ascontiguousarray(a).view(np.float16) +
                             np.ascontiguousarray(b).view(np.float16)).view(np.uint16)
    return lambda a, b: a + b


def ring_closed_form(x, dtype):
    """Chunk c (balanced floor split) folds x_{c+1}, x_{c+2}, ..., x_c."""
    n, count = x.shape
    add = _lib_add(dtype)
    out = np.empty(count, dtype=x.dtype)
    for c in range(n):
        lo, hi = oracle.chunk_range(count, n, c)
        acc = x[(c + 1) % n, lo:hi].copy()
        for k in range(2, n + 1):
            acc = add(acc, x[(c + k) % n, lo:hi])
        out[lo:hi] = acc
    return out


def tree_closed_form(x, dtype):
    """Balanced pairwise tree over ranks: (x0+x1), (x2+x3), ... then pairs of
    pairs, the lower-rank partial first."""
    add = _lib_add(dtype)
    level = [x[r] for r in range(x.shape[0])]
    while len(level) > 1:
        level = [add(level[2 * i], level[2 * i + 1]) for i in range(len(level) // 2)]
    return level[0]


@pytest.mark.parametrize("dtype", ALL_DTYPES)
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8, 16])
def test_ring_order_closed_form(oracle_lib, dtype, n):
    with np.errstate(over="ignore"):
        for count in [1, n - 1, n, n + 3, 97, 1024 + 5]:
            if count <= 0:
                continue
            x = W.uniform_inputs(n, count, dtype, config=900 + count) if dtype != "f32" else \
                W.normal_inputs(n, count, 1.0, 900 + count)
            out, _ = oracle.allreduce(x, algo="ring", op="sum", dtype=dtype)
            want = ring_closed_form(x, dtype)
            assert np.array_equal(out, np.broadcast_to(want, out.shape)), count


@pytest.mark.parametrize("dtype", ALL_DTYPES)
@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32])
def test_tree_order_closed_form(oracle_lib, dtype, n):
    with np.errstate(over="ignore"):
        for count in [1, n + 3, 257]:
            x = W.uniform_inputs(n, count, dtype, config=700 + count) if dtype != "f32" else \
                W.normal_inputs(n, count, 1.0, 700 + count)
            want = tree_closed_form(x, dtype)
            for algo in ("tree", "binomial"):
                out, _ = oracle.allreduce(x, algo=algo, op="sum", dtype=dtype)
                assert np.array_equal(out, np.broadcast_to(want, out.shape)), (algo, count)


def test_ring_order_differs_from_other_rotations(oracle_lib):
    # the fold order is observable in f32: a rotation one rank off gives other bits
    n, count = 8, 4096
    x = W.large_inputs(n, count, config=42)
    out, _ = oracle.allreduce(x, algo="ring", op="sum", dtype="bf16")
    add = _lib_add("bf16")
    wrong = np.empty(count, dtype=np.uint16)
    for c in range(n):
        lo, hi = oracle.chunk_range(count, n, c)
        acc = x[c % n, lo:hi].copy()  # starts at x_c instead of x_{c+1}
        for k in range(1, n):
            acc = add(acc, x[(c + k) % n, lo:hi])
        wrong[lo:hi] = acc
    assert not np.array_equal(out[0], wrong)


# --------------------------------------------------------------------------
# AVG
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 3, 8])
def test_avg_f32_is_sum_then_divide(oracle_lib, n):
    x = W.normal_inputs(n, 999, 1e-3, 55)
    s, _ = oracle.allreduce(x, op="sum", dtype="f32")
    a, _ = oracle.allreduce(x, op="avg", dtype="f32")
    assert np.array_equal(a, s / np.float32(n))


@pytest.mark.parametrize("n", [3, 8])
def test_avg_bf16_correctly_rounded_quotient(oracle_lib, n):
    x = W.uniform_inputs(n, 3000, "bf16", config=66)
    s, _ = oracle.allreduce(x, op="sum", dtype="bf16")
    a, _ = oracle.allreduce(x, op="avg", dtype="bf16")
    sv, av = to_f64(s[0], "bf16"), to_f64(a[0], "bf16")
    for i in range(sv.size):
        want = _frac_round_bf16(Fraction(float(sv[i])) / n)
        assert av[i] == want, i


def test_avg_rejects_integers(oracle_lib):
    x = np.zeros((2, 4), dtype=np.int32)
    _, st = oracle.allreduce(x, op="avg", dtype="i32", raise_on_error=False)
    assert st["rc"] == -2


# --------------------------------------------------------------------------
# Invariants of the collective
# --------------------------------------------------------------------------

@pytest.mark.parametrize("algo", ["ring", "tree"])
@pytest.mark.parametrize("dtype", ALL_DTYPES)
def test_rs_plus_ag_equals_allreduce(oracle_lib, algo, dtype):
    for n in ([2, 4, 8, 16] if algo == "tree" else [2, 3, 5, 8]):
        for count in [1, n, 3 * n + 1, 1000]:
            x = W.random_bits(n, count, dtype, seed=n * 1000 + count)
            ops = ["sum", "max"] + (["avg"] if dtype != "i32" else [])
            for op in ops:
                with np.errstate(all="ignore"):
                    ar, _ = oracle.allreduce(x, algo=algo, op=op, dtype=dtype)
                    rs, _ = oracle.reduce_scatter(x, algo=algo, op=op, dtype=dtype)
                    # AllGather of the owned shards only: fill everything else with junk first
                    shards = W.random_bits(n, count, dtype, seed=5)
                    for r in range(n):
                        lo, hi = oracle.chunk_range(count, n, r)
                        shards[r, lo:hi] = rs[r, lo:hi]
                        # after ReduceScatter the owner holds the finished chunk
                        assert _same(rs[r, lo:hi], ar[r, lo:hi], dtype)
                    ag, _ = oracle.all_gather(shards, algo=algo, dtype=dtype)
                assert _same(ag, ar, dtype), (n, count, op)
                # every rank ends identical
                assert all(_same(ar[r], ar[0], dtype) for r in range(n))


def _same(a, b, dtype):
    """Bit equality, with all NaNs equal to each other."""
    a, b = np.asarray(a), np.asarray(b)
    if dtype == "i32":
        return np.array_equal(a, b)
    fa, fb = to_f64(a, dtype), to_f64(b, dtype)
    na, nb = np.isnan(fa), np.isnan(fb)
    if not np.array_equal(na, nb):
        return False
    ua = a.view(np.uint16 if dtype in ("bf16", "f16") else np.uint32)
    ub = b.view(np.uint16 if dtype in ("bf16", "f16") else np.uint32)
    return np.array_equal(ua[~na], ub[~nb])


@pytest.mark.parametrize("algo", ["ring", "tree"])
def test_all_gather_copies_bits(oracle_lib, algo):
    # AllGather forwards finished chunks without arithmetic: NaN payloads,
    # signed zeros and subnormals arrive bit for bit
    n, count = 8, 64
    x = np.zeros((n, count), dtype=np.uint32)
    special = np.array([0x7FC00001, 0xFFC12345, 0x80000000, 0x00000001, 0x7F800000, 0x807FFFFF], dtype=np.uint32)
    for r in range(n):
        lo, hi = oracle.chunk_range(count, n, r)
        x[r, lo:hi] = np.resize(special + r, hi - lo)
    out, _ = oracle.all_gather(x.view(np.float32), algo=algo, dtype="f32")
    want = np.zeros(count, dtype=np.uint32)
    for r in range(n):
        lo, hi = oracle.chunk_range(count, n, r)
        want[lo:hi] = x[r, lo:hi]
    assert np.array_equal(out.view(np.uint32), np.broadcast_to(want, out.shape))


@pytest.mark.parametrize("n", [2, 3, 4, 8, 16])
def test_ring_volume_and_steps(oracle_lib, n):
    count = 64 * n  # N divides D
    x = np.ones((n, count), dtype=np.float32)
    _, st = oracle.allreduce(x, algo="ring", dtype="f32")
    assert st["steps"] == 2 * (n - 1)
    assert np.all(st["sent"] == 2 * (n - 1) * count // n)
    assert np.all(st["recv"] == 2 * (n - 1) * count // n)
    _, st = oracle.reduce_scatter(x, algo="ring", dtype="f32")
    assert st["steps"] == n - 1 and np.all(st["sent"] == (n - 1) * count // n)
    # uneven split: each rank sends every chunk but its own in ReduceScatter
    # and every chunk but its successor's in AllGather
    count = 10 * n + 3
    x = np.ones((n, count), dtype=np.float32)
    _, st = oracle.allreduce(x, algo="ring", dtype="f32")
    size = [oracle.chunk_range(count, n, c)[1] - oracle.chunk_range(count, n, c)[0] for c in range(n)]
    for r in range(n):
        assert st["sent"][r] == (count - size[r]) + (count - size[(r + 1) % n])
    assert st["sent"].sum() == 2 * (n - 1) * count


@pytest.mark.parametrize("n", [2, 4, 8, 16, 64])
def test_tree_volume_and_steps(oracle_lib, n):
    count = 8 * n
    x = np.ones((n, count), dtype=np.float32)
    _, st = oracle.allreduce(x, algo="tree", dtype="f32")
    L = int(math.log2(n))
    assert st["steps"] == 2 * L
    # halving then doubling moves the bandwidth-optimal 2(N-1)/N * D per rank
    assert np.all(st["sent"] == 2 * (n - 1) * count // n)
    _, st = oracle.allreduce(x, algo="binomial", dtype="f32")
    assert st["steps"] == 2 * L
    # the root receives log2 N full buffers and sends log2 N full buffers
    assert st["sent"][0] + st["recv"][0] == 2 * count * L


@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_naive_root_volume(oracle_lib, n):
    count = 12
    x = np.ones((n, count), dtype=np.float32)
    _, st = oracle.allreduce(x, algo="naive", dtype="f32")
    assert st["recv"][0] == (n - 1) * count and st["sent"][0] == (n - 1) * count
    assert st["sent"][0] + st["recv"][0] == 2 * (n - 1) * count


def test_tree_needs_power_of_two(oracle_lib):
    x = np.ones((3, 4), dtype=np.float32)
    for algo in ("tree", "binomial"):
        _, st = oracle.allreduce(x, algo=algo, dtype="f32", raise_on_error=False)
        assert st["rc"] == -2


# --------------------------------------------------------------------------
# Error bound against the order-free sum
# --------------------------------------------------------------------------

def gamma(k, u):
    return k * u / (1 - k * u)


@pytest.mark.parametrize("dtype,u", [("f32", 2.0 ** -24), ("bf16", 2.0 ** -8), ("f16", 2.0 ** -11)])
@pytest.mark.parametrize("n", [2, 8, 64])
def test_error_bound(oracle_lib, dtype, u, n):
    count = 20000 if n < 64 else 2000
    x = W.uniform_inputs(n, count, dtype, config=300 + n)
    xv = to_f64(x, dtype)
    exact = xv.sum(axis=0)  # exact enough: float64 has 29+ spare bits here
    absum = np.abs(xv).sum(axis=0)
    for algo, depth in (("ring", n - 1), ("tree", int(math.log2(n)))):
        out, _ = oracle.allreduce(x, algo=algo, op="sum", dtype=dtype)
        err = np.abs(to_f64(out[0], dtype) - exact)
        assert np.all(err <= gamma(depth, u) * absum), algo
    if dtype == "f32":
        out, _ = oracle.allreduce(x, algo="ring", op="sum", dtype=dtype)
        assert np.all(np.abs(out[0] - exact) <= 1e-5 * absum)


# --------------------------------------------------------------------------
# Sampled positions carry the same values as the full run
# --------------------------------------------------------------------------

@pytest.mark.parametrize("algo,n", [("ring", 8), ("ring", 5), ("tree", 8)])
@pytest.mark.parametrize("dtype", ALL_DTYPES)
def test_sampled_positions_match_full(oracle_lib, algo, n, dtype):
    count = 10_007
    x = W.random_bits(n, count, dtype, seed=31)
    g = np.random.Generator(np.random.PCG64(9))
    pos = np.unique(np.concatenate([g.integers(0, count, 300), [0, count - 1],
                                    [oracle.chunk_range(count, n, c)[0] for c in range(n)]]))
    pos = pos[(pos >= 0) & (pos < count)]
    for op in ["sum", "max"] + (["avg"] if dtype != "i32" else []):
        with np.errstate(all="ignore"):
            full, _ = oracle.allreduce(x, algo=algo, op=op, dtype=dtype)
            part, _ = oracle.allreduce(x[:, pos], algo=algo, op=op, dtype=dtype, count=count, positions=pos)
        assert _same(part, full[:, pos], dtype)


# --------------------------------------------------------------------------
# DDP buckets
# --------------------------------------------------------------------------

def greedy_buckets_by_prefix(counts, esize, cap):
    """Independent formulation of the fill rule: from the current start in the
    reversed list, a bucket takes the longest run of tensors whose bytes sum
    to at most the cap (at least one tensor)."""
    rev = list(range(len(counts)))[::-1]
    buckets, i = [], 0
    while i < len(rev):
        csum = np.cumsum([counts[t] * esize for t in rev[i:]])
        k = int(np.searchsorted(csum, cap, side="right"))
        k = max(k, 1)
        buckets.append(rev[i:i + k])
        i += k
    return buckets


def test_bucket_plan_gpt2(oracle_lib):
    counts = W.gpt2_small_counts()
    assert counts.size == 148 and counts.sum() == 124_439_808
    bucket_of, offset, bcount = oracle.bucket_plan(counts, dtype="f32", cap_bytes=25 << 20)
    want = greedy_buckets_by_prefix(counts, 4, 25 << 20)
    assert len(bcount) == len(want)
    for b, members in enumerate(want):
        assert [int(bucket_of[t]) for t in members] == [b] * len(members)
        off = 0
        for t in members:  # laid out in reverse registration order
            assert offset[t] == off
            off += counts[t]
        assert bcount[b] == off
    # by hand: the last block's tail ln_f, then layer 11 from mlp.c_proj.bias back
    # to attn.c_attn.bias fits (5,318,400 floats); attn.c_attn.weight would overflow
    assert bcount[0] == 2 * 768 + 768 + 2359296 + 3072 + 2359296 + 2 * 768 + 768 + 589824 + 2304
    # the embedding table (50257 x 768 floats = 147.2 MiB) sits alone in the last bucket
    assert bcount[-1] == 50257 * 768 and list(bucket_of).count(len(bcount) - 1) == 1
    assert np.all(bcount[:-1] * 4 <= 25 << 20)


def test_bucket_plan_one_full_bucket(oracle_lib):
    # 6,553,600 floats are exactly 25 MiB: one bucket, filled to the cap
    _, _, bcount = oracle.bucket_plan([6_553_600], dtype="f32", cap_bytes=25 << 20)
    assert bcount.tolist() == [6_553_600]
    _, _, bcount = oracle.bucket_plan([6_553_600, 1], dtype="f32", cap_bytes=25 << 20)
    assert bcount.tolist() == [1, 6_553_600]
    # the same 25 MiB as two tensors still make one full bucket
    _, _, bcount = oracle.bucket_plan([3_276_800, 3_276_800], dtype="f32", cap_bytes=25 << 20)
    assert bcount.tolist() == [6_553_600]


@pytest.mark.parametrize("seed", range(5))
def test_bucket_plan_random(oracle_lib, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    counts = g.integers(0, 5000, size=int(g.integers(1, 60)))
    counts[g.random(counts.size) < 0.1] = 40000  # oversized
    cap = 4 * 10000
    bucket_of, offset, bcount = oracle.bucket_plan(counts, dtype="f32", cap_bytes=cap)
    want = greedy_buckets_by_prefix(counts, 4, cap)
    got = [[t for t in range(counts.size)[::-1] if bucket_of[t] == b] for b in range(len(bcount))]
    assert got == want


def test_bucketed_allreduce_equals_per_bucket_collective(oracle_lib):
    g = np.random.Generator(np.random.PCG64(77))
    counts = [5, 300, 17, 1024, 3, 999, 64]
    n = 4
    grads = [[g.standard_normal(c).astype(np.float32) for c in counts] for _ in range(n)]
    cap = 4 * 1100
    out, _ = oracle.bucketed_allreduce(grads, op="avg", dtype="f32", cap_bytes=cap)
    bucket_of, offset, bcount = oracle.bucket_plan(counts, dtype="f32", cap_bytes=cap)
    for b in range(len(bcount)):
        packed = np.zeros((n, bcount[b]), dtype=np.float32)
        for r in range(n):
            for t, c in enumerate(counts):
                if bucket_of[t] == b:
                    packed[r, offset[t]:offset[t] + c] = grads[r][t]
        red, _ = oracle.allreduce(packed, op="avg", dtype="f32")
        for r in range(n):
            for t, c in enumerate(counts):
                if bucket_of[t] == b:
                    assert np.array_equal(out[r][t], red[r, offset[t]:offset[t] + c])
    # samples carry the same values
    tid = np.array([0, 1, 1, 3, 6, 5, 2], dtype=np.int32)
    idx = np.array([4, 0, 299, 512, 63, 0, 16], dtype=np.int64)
    samp, _ = oracle.bucketed_allreduce(grads, op="avg", dtype="f32", cap_bytes=cap, samples=(tid, idx))
    for r in range(n):
        assert np.array_equal(samp[r], [out[r][t][i] for t, i in zip(tid, idx)])


def test_bucketed_ddp_average_values(oracle_lib):
    # every tensor of rank r holds r: the averaged gradients are (N-1)/2 everywhere
    n = 8
    counts = [7, 1, 33, 4096]
    grads = [[np.full(c, r, dtype=np.float32) for c in counts] for r in range(n)]
    out, _ = oracle.bucketed_allreduce(grads, op="avg", dtype="f32", cap_bytes=4 * 40)
    for r in range(n):
        for t in range(len(counts)):
            assert np.all(out[r][t] == np.float32(3.5))


# --------------------------------------------------------------------------
# Failure detection on the host: a lost message or a departed rank is
# reported, never waited for
# --------------------------------------------------------------------------

def test_lost_message_is_detected(oracle_lib):
    n, count = 4, 16
    x = np.ones((n, count), dtype=np.float32)
    _, st = oracle.allreduce(x, algo="ring", dtype="f32", fault=(1, 2, 1), raise_on_error=False)
    assert st["rc"] == oracle.ERR_MISSING
    assert st["fail_step"] == 1 and st["fail_rank"] == 3  # rank 2's successor notices


def test_departed_rank_is_detected(oracle_lib):
    n, count = 8, 64
    x = np.ones((n, count), dtype=np.float32)
    for algo in ("ring", "tree"):
        _, st = oracle.allreduce(x, algo=algo, dtype="f32", fault=(2, 5, 3), raise_on_error=False)
        assert st["rc"] == oracle.ERR_MISSING and st["fail_step"] == 3, algo
    _, st = oracle.allreduce(x, algo="ring", dtype="f32", fault=(2, 5, 100), raise_on_error=False)
    assert st["rc"] == 0  # leaving after the last step harms nobody


# --------------------------------------------------------------------------
# Reduce and Broadcast: AllReduce = Reduce + Broadcast ("AllReduce 集合通信", §语义)
# --------------------------------------------------------------------------

def naive_closed_form(x, dtype):
    """Index order x_0, x_1, ..., x_{N-1}, folded with library additions."""
    add = _lib_add(dtype)
    acc = x[0].copy()
    for r in range(1, x.shape[0]):
        acc = add(acc, x[r])
    return acc


@pytest.mark.parametrize("dtype", ALL_DTYPES)
@pytest.mark.parametrize("n", [2, 3, 4, 8])
def test_reduce_then_broadcast_is_allreduce(oracle_lib, dtype, n):
    for count in (1, n + 1, 517):
        x = W.random_bits(n, count, dtype, seed=400 + n + count)
        for algo in ["ring", "naive"] + (["tree"] if n & (n - 1) == 0 else []):
            for op in ["sum", "max"] + ([] if dtype == "i32" else ["avg"]):
                for root in {0, n - 1, n // 2}:
                    with np.errstate(all="ignore"):
                        ar, _ = oracle.allreduce(x, algo=algo, op=op, dtype=dtype)
                        red, _ = oracle.reduce(x, algo=algo, op=op, dtype=dtype, root=root)
                        bc, _ = oracle.broadcast(red, root=root, dtype=dtype)
                    assert _same(red[root], ar[0], dtype), (algo, op, root)
                    assert _same(bc, ar, dtype), (algo, op, root)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_naive_order_closed_form(oracle_lib, dtype):
    n, count = 5, 300
    x = W.uniform_inputs(n, count, dtype, config=77) if dtype == "bf16" else W.normal_inputs(n, count, 1.0, 77)
    for root in (0, 3):
        red, _ = oracle.reduce(x, algo="naive", op="sum", dtype=dtype, root=root)
        assert np.array_equal(red[root], naive_closed_form(x, dtype))
    ar, _ = oracle.allreduce(x, algo="naive", op="sum", dtype=dtype)
    assert np.array_equal(ar[1], naive_closed_form(x, dtype))


def test_broadcast_copies_bits_and_volume(oracle_lib):
    n, count = 6, 33
    x = W.random_bits(n, count, "f32", seed=3)
    out, st = oracle.broadcast(x, root=2, dtype="f32")
    assert np.array_equal(out.view(np.uint32), np.broadcast_to(x[2].view(np.uint32), out.shape))
    assert st["sent"][2] == (n - 1) * count and st["steps"] == n - 1


def test_reduce_root_volume(oracle_lib):
    n, count = 8, 64 * 8
    x = np.ones((n, count), dtype=np.float32)
    _, st = oracle.reduce(x, algo="naive", root=3)
    assert st["recv"][3] == (n - 1) * count
    _, st = oracle.reduce(x, algo="ring", root=3)
    # ReduceScatter (N-1)/N D per rank, then the N-1 foreign chunks to the root
    assert st["recv"][3] == (n - 1) * count // n + (n - 1) * count // n


# --------------------------------------------------------------------------
# Double binary tree
# --------------------------------------------------------------------------

def inorder_fold(vals, lo, hi, add):
    """In-order binary tree over positions lo..hi (1-based): the root is the
    position with the most trailing zero bits; ((left) + own) + (right)."""
    if lo > hi:
        return None
    root = max(range(lo, hi + 1), key=lambda p: (p & -p))
    acc = vals[root]
    left = inorder_fold(vals, lo, root - 1, add)
    right = inorder_fold(vals, root + 1, hi, add)
    if left is not None:
        acc = add(left, acc)
    if right is not None:
        acc = add(acc, right)
    return acc


def dbtree_closed_form(x, dtype):
    n, count = x.shape
    add = _lib_add(dtype)
    half = count // 2
    out = np.empty(count, dtype=x.dtype)
    a = {p: x[p - 1, :half] for p in range(1, n + 1)}        # tree A: rank p-1 at position p
    b = {p: x[p % n, half:] for p in range(1, n + 1)}        # tree B: rank p mod N at position p
    out[:half] = inorder_fold(a, 1, n, add)
    out[half:] = inorder_fold(b, 1, n, add)
    return out


@pytest.mark.parametrize("dtype", ALL_DTYPES)
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 8, 13, 16])
def test_dbtree_closed_form(oracle_lib, dtype, n):
    with np.errstate(over="ignore"):
        for count in (2, 2 * n + 1, 513):
            x = W.uniform_inputs(n, count, dtype, config=800 + count) if dtype != "f32" else \
                W.normal_inputs(n, count, 1.0, 800 + count)
            out, _ = oracle.allreduce(x, algo="dbtree", op="sum", dtype=dtype)
            assert np.array_equal(out, np.broadcast_to(dbtree_closed_form(x, dtype), out.shape)), count


def test_dbtree_worked_shapes(oracle_lib):
    # by hand from the stated shape, N = 4: tree A reduces ((x0 + x1) + x2) + x3,
    # tree B (ranks shifted by one) ((x1 + x2) + x3) + x0; distinct f32 values
    # whose sums round differently in the two orders tell the shapes apart
    x = np.array([[1e8], [1.0], [-1e8], [1.0]], dtype=np.float32)
    x = np.repeat(x, 2, axis=1)  # element 0 in half A, element 1 in half B
    out, _ = oracle.allreduce(x, algo="dbtree", op="sum", dtype="f32")
    f = np.float32
    a = ((f(1e8) + f(1.0)) + f(-1e8)) + f(1.0)
    b = ((f(1.0) + f(-1e8)) + f(1.0)) + f(1e8)
    assert out[0, 0] == a and out[0, 1] == b and a != b


@pytest.mark.parametrize("n", [2, 4, 7, 8, 16])
def test_dbtree_volume_and_steps(oracle_lib, n):
    count = 64 * n
    x = np.ones((n, count), dtype=np.float32)
    _, st = oracle.allreduce(x, algo="dbtree", dtype="f32")
    # each tree moves its half up (N-1 messages) and down (N-1 messages)
    assert st["sent"].sum() == 2 * (n - 1) * count
    # logarithmic depth: up and down one tree of height floor(log2 N)
    h = int(math.floor(math.log2(n)))
    assert st["steps"] <= 2 * (h + 1)
    if n % 2 == 0:
        # every rank is a leaf in one of the two trees: no rank relays more
        # than one half's worth of partials up and down
        assert st["sent"].max() <= count // 2 * 3 + count // 2


# --------------------------------------------------------------------------
# 8-bit quantised AllReduce with error feedback.  The pages give only the idea
# (8-bit payloads dequantised by the receiver, the compression error fed into
# the next round); the block scheme is this library's own, pinned by exact
# cases and error bounds rather than by printed values.
# --------------------------------------------------------------------------

def test_int8_exact_when_values_sit_on_the_grid(oracle_lib):
    # every block of both ranks has max |value| = 127, so the scale is exactly 1
    # and integers quantise without error; the sums stay within 127 as well
    g = np.random.Generator(np.random.PCG64(5))
    d = 128 * 6
    a = g.integers(-63, 64, size=d).astype(np.float32)
    b = g.integers(-63, 64, size=d).astype(np.float32)
    a[::128], b[::128] = 127, 0
    a[1::128], b[1::128] = 0, -127
    x = np.stack([a, b])
    e = np.zeros_like(x)
    out, e_new, _ = oracle.int8_ef_allreduce(x, e, op="sum")
    assert np.array_equal(out, np.broadcast_to(a + b, out.shape))
    assert np.all(e_new == 0)
    out, _, _ = oracle.int8_ef_allreduce(x, e, op="avg")
    assert np.array_equal(out, np.broadcast_to((a + b) / np.float32(2), out.shape))


@pytest.mark.parametrize("n", [2, 3, 8])
def test_int8_error_bounds(oracle_lib, n):
    d = 128 * 5 + 37
    x = W.normal_inputs(n, d, 1e-3, 60 + n)
    e = W.normal_inputs(n, d, 1e-5, 70 + n)
    out, e_new, st = oracle.int8_ef_allreduce(x, e, op="sum")
    y = x.astype(np.float64) + e.astype(np.float64)
    blocks = [(lo, min(lo + 128, d)) for lo in range(0, d, 128)]
    scale = np.zeros((n, d))
    for lo, hi in blocks:
        scale[:, lo:hi] = np.abs(y[:, lo:hi]).max(axis=1, keepdims=True) / 127
    # the residual is the rounding error of one 8-bit code: at most half a step
    assert np.all(np.abs(e_new) <= scale / 2 * (1 + 1e-5) + 1e-12)
    # every rank gets the same values, within the quantisation errors of the
    # contributions and of the requantised result of the exact sum
    exact = y.sum(axis=0)
    bound = (scale / 2).sum(axis=0) + np.abs(exact).max() / 127 / 2 + 1e-6 * np.abs(y).sum(axis=0)
    for r in range(n):
        assert np.all(np.abs(out[r] - exact) <= bound * 1.01 + 1e-9)
        assert np.array_equal(out[r], out[0])


def test_int8_feedback_telescopes(oracle_lib):
    # one rank, a constant gradient: what the quantiser lets through over K
    # rounds adds up to K * x minus the residual left at the end
    d, k = 256, 20
    x = W.normal_inputs(1, d, 1.0, 9)
    e = np.zeros_like(x)
    total = np.zeros(d)
    for _ in range(k):
        xe = x[0].astype(np.float64) + e[0]
        out, e, _ = oracle.int8_ef_allreduce(x, e, op="sum")
        total += xe - e[0]   # = y^ of this round
    assert np.allclose(total, k * x[0].astype(np.float64) - e[0], rtol=0, atol=1e-4)


def test_int8_codes_round_half_to_even(oracle_lib):
    # one rank, one block whose maximum is 127: the scale is exactly 1, so the
    # codes are the values rounded to integers, ties to even, and the
    # residual is what rounding dropped
    y = np.zeros(128, dtype=np.float32)
    ties = np.array([0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 126.5, -126.5, 0.25, 0.75, -0.75], dtype=np.float32)
    y[:ties.size] = ties
    y[-1] = 127.0
    _, e_new, _ = oracle.int8_ef_allreduce(y[None, :], np.zeros((1, 128), np.float32), op="sum")
    codes = y - e_new[0]
    want = np.array([0, 2, 2, 4, 0, -2, -2, 126, -126, 0, 1, -1], dtype=np.float32)
    assert np.array_equal(codes[:ties.size], want)
    assert codes[-1] == 127.0


def test_int8_feedback_is_unbiased(oracle_lib):
    # one rank, the same gradient every round: with the compression error fed
    # back, the results of K rounds average to the gradient within one code
    # step over K; without feedback every round would return the same rounded
    # value, off by up to half a step
    d, k = 256, 64
    x = W.normal_inputs(1, d, 1.0, 19)
    e = np.zeros_like(x)
    outs = []
    for _ in range(k):
        out, e, _ = oracle.int8_ef_allreduce(x, e, op="sum")
        outs.append(out[0].astype(np.float64))
    mean = np.mean(outs, axis=0)
    step = np.repeat([np.abs(x[0, lo:lo + 128]).max() / 127 for lo in range(0, d, 128)], 128)
    assert np.all(np.abs(mean - x[0]) <= 1.5 * step / k)
    # and the plain rounding error it removes is far larger somewhere
    assert np.abs(outs[0] - x[0]).max() > 10 * (1.5 * step / k).max()


def int8_by_definition(x, e, op):
    """The 8-bit scheme written out per chunk in numpy binary32 (each step one
    IEEE operation): codes per 128-block, the owner's fold in ring order,
    requantisation per block cut at the chunk's ends."""
    n, d = x.shape
    f = np.float32
    y = (x.astype(f) + e.astype(f)).astype(f)
    yh = np.zeros_like(y)
    for lo in range(0, d, 128):
        blk = y[:, lo:lo + 128]
        s = (np.abs(blk).max(axis=1) / f(127)).astype(f)
        with np.errstate(divide="ignore", invalid="ignore"):
            q = np.where(s[:, None] > 0, np.clip(np.rint(blk / s[:, None]), -127, 127), f(0))
        q = q.astype(np.int8).astype(f)  # an 8-bit integer code: a zero code is +0
        yh[:, lo:lo + 128] = (q * s[:, None]).astype(f)
    e_new = (y - yh).astype(f)
    out = np.zeros_like(y)
    for c in range(n):
        lo, hi = c * d // n, (c + 1) * d // n
        if hi == lo:
            continue
        a = yh[(c + 1) % n, lo:hi].copy()
        for p in range(1, n):
            a = (a + yh[(c + 1 + p) % n, lo:hi]).astype(f)
        if op == "avg":
            a = (a / f(n)).astype(f)
        res = np.zeros_like(a)
        b = lo // 128 * 128
        while b < hi:
            plo, phi = max(b, lo), min(b + 128, hi)
            piece = a[plo - lo:phi - lo]
            s = f(np.abs(piece).max() / f(127))
            q = np.clip(np.rint(piece / s), -127, 127).astype(np.int8).astype(f) if s > 0 else np.zeros_like(piece)
            res[plo - lo:phi - lo] = (q * s).astype(f)
            b += 128
        out[:, lo:hi] = res
    return out, e_new


@pytest.mark.parametrize("n,d", [(1, 300), (2, 128 * 3 + 5), (3, 1000), (5, 128 * 5 + 77), (8, 128 * 24 + 3)])
def test_int8_messages_realise_the_definition(oracle_lib, n, d):
    # the literal simulation (codes and scales routed to chunk owners, then
    # requantised chunks broadcast) equals the scheme written out per chunk
    x = W.normal_inputs(n, d, 1e-2, 40 + n)
    e = W.normal_inputs(n, d, 1e-4, 50 + n)
    for op in ("sum", "avg"):
        got_x, got_e, _ = oracle.int8_ef_allreduce(x, e, op=op)
        want_x, want_e = int8_by_definition(x, e, op)
        assert np.array_equal(got_x.view(np.uint32), want_x.view(np.uint32)), (n, d, op)
        assert np.array_equal(got_e.view(np.uint32), want_e.view(np.uint32)), (n, d, op)


@pytest.mark.parametrize("n", [2, 4, 8])
def test_int8_payload_volume(oracle_lib, n):
    d = 128 * n * 3
    x = np.ones((n, d), dtype=np.float32)
    _, _, st = oracle.int8_ef_allreduce(x, np.zeros_like(x))
    assert np.all(st["sent"] == 2 * (n - 1) * d // n) and st["steps"] == 2 * (n - 1)
