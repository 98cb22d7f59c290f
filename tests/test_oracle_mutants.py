"""The pins must catch plausible mistakes in the oracle.  Each case plants one
mistake in a copy of the oracle's C source (on the CPU, in a temporary
directory), loads the mutant in place of the real library and checks that at
least one pin fails.  No GPU needed."""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "ar_oracle.c")

# (name, [(original text, replacement)], pins to run)
MUTANTS = [
    ("ring rotation one rank off",
     [("int j = mod(r - 1 - t, s->n);\n      if ((rc = post(s, r, (r + 1) % s->n, &j, 1))) return rc;",
       "int j = mod(r - t, s->n);\n      if ((rc = post(s, r, (r + 1) % s->n, &j, 1))) return rc;"),
      ("int j = mod(r - 2 - t, s->n);", "int j = mod(r - 1 - t, s->n);"),
      ("int j = mod(r - t, s->n);\n      if ((rc = post(s, r, (r + 1) % s->n, &j, 1))) return rc;\n    }\n    for (r = 0; r < s->n; ++r) {\n      int j = mod(r - 1 - t, s->n);\n      message* mb;\n      if ((rc = take(s, r, mod(r - 1, s->n), &j, 1, &mb))) return rc;\n      memcpy",
       "int j = mod(r + 1 - t, s->n);\n      if ((rc = post(s, r, (r + 1) % s->n, &j, 1))) return rc;\n    }\n    for (r = 0; r < s->n; ++r) {\n      int j = mod(r - t, s->n);\n      message* mb;\n      if ((rc = take(s, r, mod(r - 1, s->n), &j, 1, &mb))) return rc;\n      memcpy")],
     ["ring_order"]),
    ("ring drops its last ReduceScatter step",
     [("for (t = 0; t < s->n - 1; ++t) {\n    for (r = 0; r < s->n; ++r) {\n      int j = mod(r - 1 - t",
       "for (t = 0; t < s->n - 2; ++t) {\n    for (r = 0; r < s->n; ++r) {\n      int j = mod(r - 1 - t")],
     ["bruteforce", "printed"]),
    ("bf16 ties round away from zero",
     [("if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;", "if (lo >= 0x8000u) hi += 1u;")],
     ["bf16_round"]),
    ("bf16 truncates",
     [("if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;", "(void)lo;")],
     ["bf16_round"]),
    ("f16 ties round away from zero",
     [("if (rem > half || (rem == half && (q & 1u))) q += 1u;", "if (rem >= half) q += 1u;")],
     ["f16_round"]),
    ("f16 subnormals flushed to zero",
     [("return (uint16_t)(sign | q); /* subnormal; q == 1024 is the smallest normal */",
       "return (uint16_t)(q == 1024u ? (sign | q) : sign);")],
     ["f16_round"]),
    ("tree pairs the farthest ranks first",
     [("for (k = 0; k < L; ++k) {\n    int h = 1 << k;\n    for (r = 0; r < s->n; ++r) {\n      int p = r ^ h;\n      int c = kept_set(s->n, p, h, set);",
       "for (k = 0; k < L; ++k) {\n    int h = s->n >> (k + 1);\n    for (r = 0; r < s->n; ++r) {\n      int p = r ^ h;\n      int c = kept_set(s->n, p, h, set);"),
      ("for (r = 0; r < s->n; ++r) {\n      int p = r ^ h, i;\n      int c = kept_set(s->n, r, h, set);\n      int64_t off = 0;\n      message* mb;\n      if ((rc = take(s, r, p, set, c, &mb))) return rc;\n      for (i = 0; i < c; ++i) {\n        unsigned char* own",
       "for (r = 0; r < s->n; ++r) {\n      int p = r ^ h, i;\n      int c = kept_set(s->n, r, h, set);\n      int64_t off = 0;\n      message* mb;\n      if ((rc = take(s, r, p, set, c, &mb))) return rc;\n      for (i = 0; i < c; ++i) {\n        unsigned char* own")],
     ["tree_order"]),
    ("AVG divides twice",
     [("for (r = 0; r < nranks; ++r) divide_by(dtype, chunk_ptr(s, r, r), chunk_len(s, r), nranks);",
       "for (r = 0; r < nranks; ++r) { divide_by(dtype, chunk_ptr(s, r, r), chunk_len(s, r), nranks);"
       " divide_by(dtype, chunk_ptr(s, r, r), chunk_len(s, r), nranks); }")],
     ["avg"]),
    ("MAX prefers -0",
     [("r = ua & ub;", "r = ua | ub;")],
     ["max"]),
    ("f32 SUM flushes subnormal results to zero",
     [("d[i] = (op == OR_MAX) ? f32_max(a[i], b[i]) : a[i] + b[i];",
       "d[i] = (op == OR_MAX) ? f32_max(a[i], b[i]) : ((a[i] + b[i] > -1.17549435e-38f && "
       "a[i] + b[i] < 1.17549435e-38f) ? 0.0f : a[i] + b[i]);")],
     ["f32_add"]),
    ("bucket closes at the cap instead of after it",
     [("if (b < 0 || (fill > 0 && fill + bytes > cap_bytes)) {", "if (b < 0 || (fill > 0 && fill + bytes >= cap_bytes)) {")],
     ["bucket"]),
    ("buckets filled in registration order",
     [("for (t = ntensors - 1; t >= 0; --t) {\n    int64_t bytes;", "for (t = 0; t < ntensors; ++t) {\n    int64_t bytes;")],
     ["bucket"]),
    ("double binary tree: both halves on the same tree",
     [("sb = dbtree_half(s, &t, 1 % s->n, s->khalf, s->m, avg);", "sb = dbtree_half(s, &t, 0, s->khalf, s->m, avg);")],
     ["dbtree"]),
    ("double binary tree: a node folds its own value last",
     [("if (held[p][0]) combine(s->dtype, s->op, held[p][0], SLICE(p), SLICE(p), len);\n      if (held[p][1]) combine(s->dtype, s->op, SLICE(p), held[p][1], SLICE(p), len);",
       "if (held[p][1]) combine(s->dtype, s->op, SLICE(p), held[p][1], SLICE(p), len);\n      if (held[p][0]) combine(s->dtype, s->op, held[p][0], SLICE(p), SLICE(p), len);")],
     ["dbtree"]),
    ("int8 codes round half away from zero",
     [("q = nearbyintf(y / s); /* default rounding mode: to nearest, ties to even */", "q = roundf(y / s);")],
     ["int8"]),
    ("int8 compression error not fed back",
     [("e[lo + i] = y[i] - (float)q[lo + i] * scale[b];", "e[lo + i] = 0.0f;")],
     ["int8"]),
    ("int8 scale over 128 steps",
     [("  return m / 127.0f;\n}", "  return m / 128.0f;\n}")],
     ["int8"]),
    ("int8 owner folds in index order",
     [("int rr = (c + 1 + p) % nranks;", "int rr = p;")],
     ["int8"]),
    ("naive Reduce folds the root's own value first",
     [("memcpy(s->rank[root], got[0], (size_t)s->m * (size_t)s->es);\n      for (r = 1; r < s->n; ++r) combine(s->dtype, s->op, s->rank[root], got[r], s->rank[root], s->m);",
       "memcpy(s->rank[root], got[root], (size_t)s->m * (size_t)s->es);\n      for (r = 0; r < s->n; ++r) if (r != root) combine(s->dtype, s->op, s->rank[root], got[r], s->rank[root], s->m);")],
     ["rooted"]),
    ("Broadcast skips the last rank",
     [("    if (r == root) continue;\n    if ((rc = post(s, root, r, all, s->n))) return rc;",
       "    if (r == root || r == s->n - 1) continue;\n    if ((rc = post(s, root, r, all, s->n))) return rc;")],
     ["rooted"]),
    ("Reduce files gathered chunks one slot off",
     [("memcpy(chunk_ptr(s, root, r), mb->data, (size_t)mb->n * (size_t)s->es);",
       "memcpy(chunk_ptr(s, root, (r + 1) % s->n), mb->data, (size_t)mb->n * (size_t)s->es);")],
     ["rooted"]),
    ("ring counts only received volume",
     [("s->st->sent[src] += total;", "(void)total;")],
     ["volume"]),
]


def run_pins(which):
    o = oracle
    if "ring_order" in which:
        for dt in P.ALL_DTYPES:
            for n in (3, 8):
                P.test_ring_order_closed_form(o, dt, n)
    if "tree_order" in which:
        for dt in ("f32", "bf16"):
            P.test_tree_order_closed_form(o, dt, 8)
    if "bruteforce" in which:
        for n in (2, 3, 8):
            P.test_bruteforce_integers_and_max(o, n)
    if "printed" in which:
        for dt in P.ALL_DTYPES:
            P.test_printed_sum_examples(o, "four_rank_ones.txt", dt)
    if "bf16_round" in which:
        P.test_bf16_rounding_edges(o)
        P.test_bf16_add_is_correctly_rounded(o)
    if "f16_round" in which:
        P.test_f16_rounding_by_value(o)
        P.test_f16_add_is_correctly_rounded(o)
    if "avg" in which:
        P.test_printed_ddp_average(o, "f32")
        P.test_avg_f32_is_sum_then_divide(o, 8)
    if "max" in which:
        P.test_max_special_values(o)
    if "f32_add" in which:
        P.test_f32_add_matches_numpy(o)
    if "bucket" in which:
        P.test_bucket_plan_one_full_bucket(o)
        P.test_bucket_plan_gpt2(o)
    if "volume" in which:
        P.test_ring_volume_and_steps(o, 4)
    if "rooted" in which:
        for dt in ("f32", "bf16"):
            P.test_naive_order_closed_form(o, dt)
        for n in (3, 4):
            P.test_reduce_then_broadcast_is_allreduce(o, "f32", n)
        P.test_broadcast_copies_bits_and_volume(o)
    if "int8" in which:
        P.test_int8_exact_when_values_sit_on_the_grid(o)
        P.test_int8_codes_round_half_to_even(o)
        P.test_int8_feedback_is_unbiased(o)
        for n, d in ((2, 128 * 3 + 5), (3, 1000), (5, 128 * 5 + 77)):
            P.test_int8_messages_realise_the_definition(o, n, d)
        for n in (2, 3):
            P.test_int8_error_bounds(o, n)
    if "dbtree" in which:
        for dt in ("f32", "bf16"):
            for n in (4, 5, 8):
                P.test_dbtree_closed_form(o, dt, n)
        P.test_dbtree_worked_shapes(o)


@pytest.mark.parametrize("name,edits,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, monkeypatch, name, edits, pins):
    src = open(SRC, encoding="utf-8").read()
    for old, new in edits:
        assert old in src, f"mutation site not found for {name!r}"
        src = src.replace(old, new, 1)
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src, encoding="utf-8")
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
                    "-w", "-o", str(so), str(mpath)], check=True)
    real = oracle.lib()
    mutant = ctypes.CDLL(str(so))
    for fname in ("oracle_collective", "oracle_step", "oracle_f32_to_bf16", "oracle_chunk_range",
                  "oracle_bucket_plan", "oracle_bucketed_allreduce", "oracle_int8_ef_allreduce", "oracle_rooted"):
        getattr(mutant, fname).argtypes = getattr(real, fname).argtypes
    monkeypatch.setattr(oracle, "_lib", mutant)
    with pytest.raises((AssertionError, oracle.OracleError)):
        run_pins(pins)


def test_real_oracle_passes_the_same_pins():
    run_pins({"ring_order", "tree_order", "bruteforce", "printed", "bf16_round", "f16_round", "avg", "max", "f32_add",
              "bucket", "volume", "dbtree", "int8", "rooted"})
