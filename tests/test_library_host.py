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
    assert ar.ar_allreduce([1 << 20, 1 << 21], count=4, dtype=4, stream=0) == ar.AR_ERR_INVALID_ARG
    assert ar.DTYPE["f16"] == 3 and "AR_F16 = 3" in open(HEADER).read()
    assert ar.ar_allreduce([1 << 20, (1 << 20) + 4], count=4, dtype="f16", stream=0) == ar.AR_ERR_INVALID_ARG  # overlap
    assert ar.ar_allreduce([1 << 20, 1 << 21], count=4, algo=9, stream=0) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_allreduce([1 << 20, 1 << 21], count=4, algo=7, stream=0) == ar.AR_ERR_INVALID_ARG
    assert ar.ALGO["binomial_stepwise"] == 6 and "AR_BINOMIAL_STEPWISE = 6" in open(HEADER).read()
    assert ar.ar_allreduce([1 << 20, 1 << 21, 1 << 22], count=4, algo="binomial_stepwise",
                           stream=0) == ar.AR_ERR_UNSUPPORTED  # not a power of two
    assert ar.lib.ar_device_status(None, None) == ar.AR_ERR_INVALID_ARG
    rc = ar.ar_bucket_plan([5, 6], "f32", 0)[0]
    assert rc == ar.AR_ERR_INVALID_ARG


def test_counts_that_overflow_byte_ranges_are_refused(ar):
    """Element counts whose byte size would wrap past 2^64 (or past the
    documented ceiling, 2^56 elements) and buffers whose end passes the top
    of the address space are argument errors, found before any device work:
    a wrapped end could otherwise pass the range checks."""
    limit = 1 << 56
    assert ar.MAX_COUNT == limit
    ptrs = [1 << 20, 1 << 40]
    assert ar.ar_allreduce(ptrs, count=limit + 1, stream=0) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_allreduce(ptrs, count=1 << 62, stream=0) == ar.AR_ERR_INVALID_ARG  # 4 * 2^62 = 2^64
    assert ar.ar_reduce_scatter(ptrs, count=(1 << 63) - 1, stream=0) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_all_gather(ptrs, count=1 << 62, dtype="bf16", stream=0) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_allreduce_int8_ef(ptrs, [1 << 44, 1 << 45], count=1 << 62, stream=0) == ar.AR_ERR_INVALID_ARG
    top = (1 << 64) - 64  # 16 f32 from here would end past 2^64
    assert ar.ar_allreduce([top, 1 << 20], count=32, stream=0) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_bucket_plan([1 << 62], "f32", 25 << 20)[0] == ar.AR_ERR_INVALID_ARG
    assert ar.ar_bucket_plan([1 << 55] * 3, "f32", 25 << 20)[0] == ar.AR_ERR_INVALID_ARG  # sum > 2^56
    rc, bo, off, bc = ar.ar_bucket_plan([1 << 55] * 2, "f32", 25 << 20)  # sum = 2^56: accepted
    assert rc == ar.AR_OK and list(bc) == [1 << 55, 1 << 55]
    header = open(os.path.join(ROOT, "include", "ar.h")).read()
    assert "#define AR_MAX_COUNT (1LL << 56)" in header


def test_host_buffer_allreduce_checks_without_device(ar):
    h, d = [1 << 20, 1 << 21], [1 << 40, 1 << 41]
    assert ar.ar_allreduce_host(h, d, count=4, algo="ring_stepwise", stream=0) == ar.AR_ERR_UNSUPPORTED
    assert ar.ar_allreduce_host(h, d, count=4, dtype="i32", op="avg", stream=0) == ar.AR_ERR_UNSUPPORTED
    assert ar.ar_allreduce_host([1 << 20, 1 << 20], d, count=4, stream=0) == ar.AR_ERR_INVALID_ARG  # duplicate
    assert ar.ar_allreduce_host(h, [1 << 20, 1 << 41], count=4, stream=0) == ar.AR_ERR_INVALID_ARG  # host = device
    assert ar.ar_allreduce_host(h, d, count=4, piece_elems=-1, stream=0) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_allreduce_host(h, d, count=1 << 62, stream=0) == ar.AR_ERR_INVALID_ARG
    assert ar.lib.ar_allreduce_host(None, None, 2, 4, 0, 0, 0, 0, None) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_allreduce_host([0, 0], [0, 0], count=0, stream=0) == ar.AR_OK  # nothing to move
    # zero-copy needs mapped page-locked memory: unbacked addresses are refused, never computed on the host
    assert ar.ar_allreduce_host(h, None, count=4, stream=0) in (ar.AR_ERR_INVALID_ARG, ar.AR_ERR_CUDA, -5)


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


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "ar.h"

int main(void) {
  int64_t lo = -1, hi = -1;
  int64_t counts[4] = {10, 300, 7, 2000};
  int32_t bucket_of[4];
  int64_t offset[4], bcount[4];
  int32_t nb = 0;
  int rc;
  void* none[2] = {0, 0};
  if (ar_version() <= 0) return 1;
  if (ar_chunk_range(10, 3, 2, &lo, &hi) != AR_OK || lo != 6 || hi != 10) return 2;
  rc = ar_bucket_plan(counts, 4, AR_F32, 4096, bucket_of, offset, bcount, &nb);
  if (rc != AR_OK) return 3;
  printf("%d", nb);
  for (int i = 0; i < nb; ++i) printf(" %lld", (long long)bcount[i]);
  printf("\n");
  /* argument checks run on the host, before any CUDA call */
  if (ar_allreduce(none, 0, 16, AR_F32, AR_SUM, AR_RING, 0) != AR_ERR_INVALID_ARG) return 4;
  if (ar_allreduce(none, 2, 16, AR_I32, AR_AVG, AR_RING, 0) != AR_ERR_UNSUPPORTED) return 5;
  if (strncmp(ar_strerror(AR_ERR_TIMEOUT), "AR_ERR_TIMEOUT", 14) != 0) return 6;
  return 0;
}
"""


def test_c_program_compiles_links_and_runs_against_the_header(ar, tmp_path):
    """The boundary is plain C: a C11 program includes include/ar.h, links
    libar_gb300.so and calls the host-side entry points (no GPU needed)."""
    src = tmp_path / "use_ar.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_ar"
    libdir = os.path.dirname(ar.LIB_PATH) if hasattr(ar, "LIB_PATH") else os.path.join(
        ROOT, "allreduce_gradient_reduction_gb300")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-L", libdir, "-lar_gb300", "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=dict(os.environ, LD_LIBRARY_PATH=libdir))
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    want = oracle.bucket_plan([10, 300, 7, 2000], dtype="f32", cap_bytes=4096)
    fields = r.stdout.split()
    assert int(fields[0]) == len(want[2])
    assert [int(v) for v in fields[1:]] == [int(v) for v in want[2]]


def test_count_zero_is_a_no_op_with_any_pointers(ar):
    # an empty tensor's data pointer is NULL; with nothing to move the calls
    # succeed without looking at the pointers (and without touching CUDA)
    nulls = [0, 0, 0, 0]
    assert ar.ar_allreduce(nulls, count=0, dtype="bf16", algo="ring", stream=0) == ar.AR_OK
    assert ar.ar_reduce_scatter(nulls, count=0, algo="tree", stream=0) == ar.AR_OK
    assert ar.ar_all_gather(nulls, count=0, stream=0) == ar.AR_OK
    assert ar.ar_reduce(nulls, count=0, root=2, stream=0) == ar.AR_OK
    assert ar.ar_broadcast(nulls, count=0, root=1, stream=0) == ar.AR_OK
    assert ar.ar_allreduce_int8_ef(nulls, nulls, count=0, op="avg", stream=0) == ar.AR_OK
    # argument checks still apply
    assert ar.ar_reduce(nulls, count=0, root=7, stream=0) == ar.AR_ERR_INVALID_ARG
    assert ar.ar_allreduce(nulls, count=0, dtype="i32", op="avg", stream=0) == ar.AR_ERR_UNSUPPORTED
