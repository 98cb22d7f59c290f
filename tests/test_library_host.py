"""CPU checks of the CUDA library: it loads, exports every symbol the header
declares, and its host-only logic (chunk partition, bucket plan, argument
checks, error strings) agrees with the oracle.  No GPU is touched: no compute
entry point is called with valid device memory here."""
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
from allreduce_gradient_reduction_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ar.h")


@pytest.fixture(scope="module")
def ar():
    from allreduce_gradient_reduction_gb300 import build as b
    b.build()
    from allreduce_gradient_reduction_gb300 import binding
    return binding


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ar_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ar_allreduce", "ar_reduce_scatter", "ar_all_gather", "ar_bucketed_allreduce",
                     "ar_bucket_plan", "ar_chunk_range", "ar_device_status", "ar_strerror"):
        assert required in names


def test_library_exports_every_declared_symbol(ar):
    for name in declared_functions():
        assert hasattr(ar.lib, name), name
    assert set(declared_functions()) <= set(ar.EXPORTS) | {"ar_version"}
    nm = subprocess.run(["nm", "-D", "--defined-only", ar.LIB_PATH], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\bT (ar_[a-z_]+)\b", nm.stdout))
    assert set(declared_functions()) <= exported


def test_library_does_not_link_the_oracle(ar):
    nm = subprocess.run(["nm", "-D", ar.LIB_PATH], capture_output=True, text=True, check=True)
    assert "oracle_" not in nm.stdout
    ldd = subprocess.run(["ldd", ar.LIB_PATH], capture_output=True, text=True)
    assert "oracle" not in ldd.stdout


@pytest.mark.parametrize("count,n", [(0, 1), (1, 3), (7, 8), (9, 8), (4096, 4), (1001, 7), (67_108_864, 8),
                                     ((1 << 40) + 3, 64)])
def test_chunk_range_matches_oracle(ar, count, n):
    for c in range(n):
        rc, lo, hi = ar.ar_chunk_range(count, n, c)
        assert rc == 0 and (lo, hi) == oracle.chunk_range(count, n, c)
    assert ar.ar_chunk_range(count, n, n)[0] == ar.AR_ERR_INVALID_ARG
    assert ar.ar_chunk_range(-1, n, 0)[0] == ar.AR_ERR_INVALID_ARG


def test_bucket_plan_matches_oracle_gpt2(ar):
    counts = W.gpt2_small_counts()
    rc, bo, off, bc = ar.ar_bucket_plan(counts, "f32", 25 << 20)
    ob, oo, oc = oracle.bucket_plan(counts, dtype="f32", cap_bytes=25 << 20)
    assert rc == 0
    assert bo == ob.tolist() and off == oo.tolist() and bc == oc.tolist()
    assert len(bc) == 17 and sum(bc) == 124_439_808


@pytest.mark.parametrize("seed", range(10))
def test_bucket_plan_matches_oracle_random(ar, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    counts = g.integers(0, 3000, size=int(g.integers(1, 80)))
    counts[g.random(counts.size) < 0.1] = 20000
    for dt in ("f32", "bf16", "i32"):
        cap = int(g.integers(1, 50000))
        rc, bo, off, bc = ar.ar_bucket_plan(counts, dt, cap)
        ob, oo, oc = oracle.bucket_plan(counts, dtype=dt, cap_bytes=cap)
        assert rc == 0 and bo == ob.tolist() and off == oo.tolist() and bc == oc.tolist()


def test_argument_checks_without_device(ar):
    # rejected before any device work
    assert ar.lib.ar_allreduce(None, 2, 10, 0, 0, 0, None) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_allreduce([1 << 20, 1 << 21], count=-1, stream=0) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_allreduce([1 << 20] * 65, count=4, stream=0) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_allreduce([1 << 20, 1 << 21], count=4, dtype="i32", op="avg", stream=0) == ar.AR_ERR_UNSUPPORTED
    assert ar.ar_allreduce([1 << 20, 1 << 21, 1 << 22], count=4, algo="tree", stream=0) == ar.AR_ERR_UNSUPPORTED
    assert ar.ar_allreduce([1 << 20, 1 << 20], count=4, stream=0) == ar.AR_ERR_INVALID_ARG  # duplicate
    assert ar.ar_allreduce([1 << 20, (1 << 20) + 8], count=4, stream=0) == ar.AR_ERR_INVALID_ARG  # overlap
    assert ar.ar_allreduce([(1 << 20) + 2, 1 << 21], count=4, stream=0) == ar.AR_ERR_INVALID_ARG  # misaligned f32
    assert ar.ar_allreduce([0, 1 << 21], count=4, stream=0) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_allreduce([1 << 20, 1 << 21], count=4, dtype=7, stream=0) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_allreduce([1 << 20, 1 << 21], count=4, algo=9, stream=0) == ar.AR_ERR_INVALID_ARG
    assert ar.lib.ar_device_status(None, None) == ar.AR_ERR_INVALID_ARG
    rc = ar.ar_bucket_plan([5, 6], "f32", 0)[0]
    assert rc == ar.AR_ERR_INVALID_ARG


def test_no_device_is_reported_not_faked(ar):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # plausible but unbacked pointers: the library must refuse, never compute on the host
    rc = ar.ar_allreduce([1 << 20, 1 << 24], count=16, stream=0)
    assert rc in (ar.AR_ERR_INVALID_ARG, -5, ar.AR_ERR_CUDA)


def test_strerror_and_version(ar):
    for code, name in ar.STATUS.items():
        assert ar.ar_strerror(code).startswith(name)
    assert ar.ar_version() >= 100
