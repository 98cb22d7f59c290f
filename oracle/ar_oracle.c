/*
 * CPU oracle for the simulated AllReduce.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * What it is: a plain, deliberately slow, literal simulation of N ranks that
 * exchange messages.  Every rank owns a private copy of its buffer; in every
 * communication step each rank first *posts* a message (a copy of the values it
 * sends, tagged with the chunk ids it covers), then every rank *receives* the
 * message addressed to it and applies the elementwise step.  Sent and received
 * element counts and the number of steps are recorded per rank.
 *
 * Sources (page title, section):
 *  - AllReduce semantics: N processes hold equal-length data, all end with the
 *    same reduction.  "AllReduce" concept page, §3 技术原理; "AllReduce 集合通信",
 *    §语义：Reduce 与 Broadcast 的合一.
 *  - Ring = ReduceScatter (N-1 steps, send one chunk to the next rank, receive
 *    one from the previous rank, accumulate in place) + AllGather (N-1 steps,
 *    forward finished chunks, no accumulation).  "Allreduce：大模型分布式训练的
 *    核心通信算法与优化实践" §2.2; "AllReduce 集合通信" §两阶段流程.
 *    Reading of the chunk rotation: rank r ends ReduceScatter owning chunk r
 *    (P0 holds the sum of chunk 0, P1 of chunk 1, ... in §2.2 of the tutorial),
 *    so in step s rank r sends chunk (r-1-s) mod N and chunk c is folded in the
 *    order x_{c+1}, x_{c+2}, ..., x_{c+N-1}, x_c.
 *  - Average: SUM, then divide by the world size once.  Tutorial §3.1;
 *    "AllReduce 集合通信" §DDP 梯度同步中的地位.
 *  - Tree / recursive halving: step 1 pairs ranks (0,1), (2,3), ...; step 2
 *    combines (0/1) with (2/3); log2 N steps.  "【AI Infra小白入门⑩】集合通信
 *    基础：AllReduce、Ring算法与NCCL全解析" §四 4.1.  Message schedule used here:
 *    recursive halving (partner r XOR 2^k, k = 0 first) for ReduceScatter, then
 *    recursive doubling in reverse order for AllGather.
 *  - Binomial reduce-to-root then broadcast (leaves to root, root to leaves):
 *    "AllReduce算法详解" §4.3.1-4.3.2 (a second tree schedule; same pairing).
 *  - Naive central reduce + broadcast: "AllReduce 集合通信" §朴素实现与主节点瓶颈;
 *    tutorial §2.1.
 *  - DDP bucketing: buckets of at most bucket_cap (25 MB by default) filled
 *    with parameters in reverse order.  Tutorial §4.1; "AllReduce 集合通信"
 *    §DDP 梯度同步中的地位.
 *  - Double binary tree (two complementary trees, half the data each) and
 *    the 8-bit quantised AllReduce with error feedback: see their functions.
 *
 * PARITY UNPINNED by the pages, for three choices: the ring's chunk rotation
 * (every example the pages print is integer-valued, hence order-free), the
 * double binary tree's shape, and the 8-bit scheme.  Each is pinned here
 * only by the reading stated at its function and by closed forms and worked
 * cases of that reading, never by a value the pages print.
 *
 * Elementwise step (the pages fix only "sum" / "max"; the arithmetic is IEEE):
 *  - f32 SUM: IEEE binary32 addition, round to nearest even (C float `+`,
 *    compiled without contraction or fast-math).
 *  - bf16 SUM: convert both to binary32 (exact), add, round to bf16 by round-
 *    to-nearest-even on the dropped 16 bits.  NaN results become 0x7FC0.
 *  - f16 SUM (IEEE binary16; the tutorial §4.2 names FP16 beside BF16 as the
 *    half-size gradient type): convert both to binary32 (exact), add, round
 *    to binary16 nearest-even.  Both roundings together equal one correct
 *    rounding of the exact sum, because binary32 carries 24 >= 2*11 + 2
 *    significand bits.  NaN results become 0x7E00.
 *  - i32 SUM: two's-complement wrap-around.
 *  - MAX: IEEE 754-2019 maximum: NaN if either operand is NaN, +0 > -0.
 *  - AVG: SUM, then the owner of each reduced chunk divides once by N
 *    (binary32 IEEE division; for bf16 and f16 the binary32 quotient is
 *    rounded to the storage type).  AVG on i32 is rejected.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_MAX_RANKS 256

enum { OR_F32 = 0, OR_BF16 = 1, OR_I32 = 2, OR_F16 = 3 };
enum { OR_SUM = 0, OR_MAX = 1, OR_AVG = 2 };
enum { OR_RING = 0, OR_TREE = 1, OR_BINOMIAL = 2, OR_NAIVE = 3, OR_DBTREE = 4 };
enum { OR_PHASE_RS = 1, OR_PHASE_AG = 2 };
enum {
  OR_OK = 0,
  OR_EINVAL = -1,
  OR_EUNSUPPORTED = -2,
  OR_ENOMEM = -3,
  OR_EMISSING = -4, /* a receiver found no message: a rank dropped out or a message was lost */
  OR_ESCHEDULE = -5 /* a message arrived with chunks the schedule did not expect */
};

typedef struct {
  int32_t steps;     /* communication steps executed */
  int32_t fail_step; /* step at which a receiver found no message, else -1 */
  int32_t fail_rank; /* that receiver, else -1 */
  int32_t pad;
  int64_t sent[OR_MAX_RANKS]; /* elements each rank sent */
  int64_t recv[OR_MAX_RANKS]; /* elements each rank received */
} oracle_stats;

/* Host-side failure injection: kind 1 loses the message that `rank` posts at
 * global step `step`; kind 2 makes `rank` stop sending from global step `step`
 * on (it has left the job). */
typedef struct {
  int32_t kind;
  int32_t rank;
  int32_t step;
} oracle_fault;

/* ------------------------------------------------------------------------ */
/* Elementwise arithmetic                                                   */
/* ------------------------------------------------------------------------ */

static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static int f32_is_nan(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return (u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0;
}

/* Round a binary32 value to bfloat16 (8-bit significand), nearest-even:
 * keep the upper 16 bits, add one unit if the dropped 16 bits are above half,
 * or exactly half with the kept part odd.  A carry out of the significand
 * moves into the exponent, which is what rounding up to the next binade (or to
 * infinity) means. */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u, hi, lo;
  if (f32_is_nan(f)) return 0x7FC0u;
  memcpy(&u, &f, 4);
  hi = u >> 16;
  lo = u & 0xFFFFu;
  if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;
  return (uint16_t)hi;
}

/* IEEE binary16: sign, 5 exponent bits (bias 15), 10 fraction bits.  Every
 * binary16 value is exactly a binary32 value. */
static float f16_to_f32(uint16_t h) {
  const int e = (h >> 10) & 0x1F, m = h & 0x3FF;
  float v;
  if (e == 0x1F) {
    uint32_t u = (h & 0x8000u) ? 0xFF800000u : 0x7F800000u;
    if (m) u = 0x7FC00000u;
    memcpy(&v, &u, 4);
    return v;
  }
  v = e ? ldexpf((float)(1024 + m), e - 25) : ldexpf((float)m, -24);
  return (h & 0x8000u) ? -v : v;
}

/* Round a binary32 value to binary16, nearest-even.  The significand with its
 * hidden bit is shifted right to the binary16 unit of the value's exponent
 * (2^-24 below the normal range), rounding on the bits shifted out; a carry
 * into the next binade, or past the largest finite value, is what rounding up
 * there means. */
static uint16_t f32_to_f16_rne(float f) {
  uint32_t u, sign, e, m, shift, q, rem, half;
  uint64_t sig;
  int E;
  if (f32_is_nan(f)) return 0x7E00u;
  memcpy(&u, &f, 4);
  sign = (u >> 16) & 0x8000u;
  e = (u >> 23) & 0xFFu;
  m = u & 0x7FFFFFu;
  if (e == 0xFFu) return (uint16_t)(sign | 0x7C00u); /* infinity */
  if (e == 0 && m == 0) return (uint16_t)sign;       /* zero */
  sig = e ? (uint64_t)(m | 0x800000u) : (uint64_t)m;  /* value = sig * 2^(E - 23) */
  E = e ? (int)e - 127 : -126;
  /* binary16 unit at exponent E: 2^(E-10) for E >= -14, else 2^-24 */
  shift = (uint32_t)(E >= -14 ? 13 : (-E - 1)); /* 23 - 10, or 23 - (E + 24) */
  if (shift > 24) return (uint16_t)sign; /* sig < 2^24: less than half a unit, and never a tie */
  q = (uint32_t)(sig >> shift);
  rem = (uint32_t)(sig & ((1ull << shift) - 1));
  half = 1u << (shift - 1);
  if (rem > half || (rem == half && (q & 1u))) q += 1u;
  if (E >= -14) {
    /* q holds the significand with its hidden bit: 1024..2048 */
    if (q == 2048u) {
      q = 1024u;
      E += 1;
    }
    if (E > 15) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | ((uint32_t)(E + 15) << 10) | (q - 1024u));
  }
  return (uint16_t)(sign | q); /* subnormal; q == 1024 is the smallest normal */
}

static float f32_max(float a, float b) {
  uint32_t ua, ub, r;
  float out;
  if (f32_is_nan(a) || f32_is_nan(b)) {
    r = 0x7FC00000u;
    memcpy(&out, &r, 4);
    return out;
  }
  if (a > b) return a;
  if (b > a) return b;
  /* equal: only +0 / -0 can differ in bits; +0 wins unless both are -0 */
  memcpy(&ua, &a, 4);
  memcpy(&ub, &b, 4);
  r = ua & ub;
  memcpy(&out, &r, 4);
  return out;
}

/* dst[i] = step(first[i], second[i]) */
static void combine(int dtype, int op, const void* first, const void* second, void* dst, int64_t n) {
  int64_t i;
  if (dtype == OR_F32) {
    const float* a = (const float*)first;
    const float* b = (const float*)second;
    float* d = (float*)dst;
    for (i = 0; i < n; ++i) d[i] = (op == OR_MAX) ? f32_max(a[i], b[i]) : a[i] + b[i];
  } else if (dtype == OR_BF16) {
    const uint16_t* a = (const uint16_t*)first;
    const uint16_t* b = (const uint16_t*)second;
    uint16_t* d = (uint16_t*)dst;
    for (i = 0; i < n; ++i) {
      float fa = bf16_to_f32(a[i]), fb = bf16_to_f32(b[i]);
      if (op == OR_MAX) {
        if (f32_is_nan(fa) || f32_is_nan(fb)) d[i] = 0x7FC0u;
        else if (fa > fb) d[i] = a[i];
        else if (fb > fa) d[i] = b[i];
        else d[i] = (uint16_t)(a[i] & b[i]);
      } else {
        d[i] = f32_to_bf16_rne(fa + fb);
      }
    }
  } else if (dtype == OR_F16) {
    const uint16_t* a = (const uint16_t*)first;
    const uint16_t* b = (const uint16_t*)second;
    uint16_t* d = (uint16_t*)dst;
    for (i = 0; i < n; ++i) {
      float fa = f16_to_f32(a[i]), fb = f16_to_f32(b[i]);
      if (op == OR_MAX) {
        if (f32_is_nan(fa) || f32_is_nan(fb)) d[i] = 0x7E00u;
        else if (fa > fb) d[i] = a[i];
        else if (fb > fa) d[i] = b[i];
        else d[i] = (uint16_t)(a[i] & b[i]);
      } else {
        d[i] = f32_to_f16_rne(fa + fb);
      }
    }
  } else {
    const int32_t* a = (const int32_t*)first;
    const int32_t* b = (const int32_t*)second;
    int32_t* d = (int32_t*)dst;
    for (i = 0; i < n; ++i) {
      if (op == OR_MAX) d[i] = a[i] > b[i] ? a[i] : b[i];
      else d[i] = (int32_t)((uint32_t)a[i] + (uint32_t)b[i]);
    }
  }
}

static void divide_by(int dtype, void* data, int64_t n, int nranks) {
  int64_t i;
  float fn = (float)nranks;
  if (dtype == OR_F32) {
    float* d = (float*)data;
    for (i = 0; i < n; ++i) d[i] = d[i] / fn;
  } else if (dtype == OR_BF16) {
    uint16_t* d = (uint16_t*)data;
    for (i = 0; i < n; ++i) d[i] = f32_to_bf16_rne(bf16_to_f32(d[i]) / fn);
  } else if (dtype == OR_F16) {
    uint16_t* d = (uint16_t*)data;
    for (i = 0; i < n; ++i) d[i] = f32_to_f16_rne(f16_to_f32(d[i]) / fn);
  }
}

static int esize_of(int dtype) { return (dtype == OR_BF16 || dtype == OR_F16) ? 2 : 4; }

/* Exported single step, for table checks: out[i] = step(recv[i], local[i]). */
int oracle_step(int dtype, int op, const void* recv, const void* local, void* out, int64_t n) {
  if (dtype < 0 || dtype > 3 || op < 0 || op > 1 || n < 0) return OR_EINVAL;
  combine(dtype, op, recv, local, out, n);
  return OR_OK;
}

/* Exported binary32 -> bf16 rounding, for tests of the rounding itself. */
int oracle_f32_to_bf16(const float* in, uint16_t* out, int64_t n) {
  int64_t i;
  for (i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(in[i]);
  return OR_OK;
}

/* Exported binary32 <-> binary16 conversions, for tests of them. */
int oracle_f32_to_f16(const float* in, uint16_t* out, int64_t n) {
  int64_t i;
  for (i = 0; i < n; ++i) out[i] = f32_to_f16_rne(in[i]);
  return OR_OK;
}

int oracle_f16_to_f32(const uint16_t* in, float* out, int64_t n) {
  int64_t i;
  for (i = 0; i < n; ++i) out[i] = f16_to_f32(in[i]);
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Chunk partition                                                          */
/* ------------------------------------------------------------------------ */

/* Each rank buffer of `count` elements is split into N contiguous chunks,
 * chunk c = [floor(c*count/N), floor((c+1)*count/N)).  The pages split the data
 * "evenly into N blocks" without saying what happens when N does not divide
 * the length; this balanced floor split is the reading used throughout. */
int oracle_chunk_range(int64_t count, int nranks, int c, int64_t* lo, int64_t* hi) {
  if (count < 0 || nranks < 1 || c < 0 || c >= nranks || !lo || !hi) return OR_EINVAL;
  *lo = (int64_t)(((__int128)c * count) / nranks);
  *hi = (int64_t)(((__int128)(c + 1) * count) / nranks);
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Ranks and messages                                                       */
/* ------------------------------------------------------------------------ */

typedef struct {
  int present;
  int src;
  int nchunks;
  int chunks[OR_MAX_RANKS];
  int64_t n;
  unsigned char* data;
} message;

typedef struct {
  int n, dtype, op, es;
  int64_t m;                      /* positions held per rank */
  int64_t klo[OR_MAX_RANKS + 1];  /* chunk j = local positions [klo[j], klo[j+1]) */
  unsigned char* rank[OR_MAX_RANKS];
  message box[OR_MAX_RANKS];      /* one inbox per rank, emptied every step */
  oracle_stats* st;
  const oracle_fault* fault;
  int step;
  int64_t khalf; /* first local position of the second half (double binary tree) */
} sim;

static int64_t chunk_len(const sim* s, int j) { return s->klo[j + 1] - s->klo[j]; }

static unsigned char* chunk_ptr(const sim* s, int r, int j) {
  return s->rank[r] + (size_t)s->klo[j] * (size_t)s->es;
}

/* Rank `src` posts the listed chunks of its current buffer to `dst`. */
static int post(sim* s, int src, int dst, const int* chunks, int nchunks) {
  message* mb = &s->box[dst];
  int64_t total = 0, off = 0;
  int i;
  if (s->fault && s->fault->kind == 2 && s->fault->rank == src && s->step >= s->fault->step)
    return OR_OK; /* the rank has left: it sends nothing */
  for (i = 0; i < nchunks; ++i) total += chunk_len(s, chunks[i]);
  s->st->sent[src] += total;
  if (s->fault && s->fault->kind == 1 && s->fault->rank == src && s->fault->step == s->step)
    return OR_OK; /* lost on the wire */
  if (mb->present) return OR_ESCHEDULE; /* two messages for one receiver in one step */
  mb->data = (unsigned char*)malloc((size_t)(total > 0 ? total : 1) * (size_t)s->es);
  if (!mb->data) return OR_ENOMEM;
  for (i = 0; i < nchunks; ++i) {
    int64_t len = chunk_len(s, chunks[i]);
    memcpy(mb->data + (size_t)off * (size_t)s->es, chunk_ptr(s, src, chunks[i]), (size_t)len * (size_t)s->es);
    off += len;
    mb->chunks[i] = chunks[i];
  }
  mb->present = 1;
  mb->src = src;
  mb->nchunks = nchunks;
  mb->n = total;
  return OR_OK;
}

/* Rank `dst` takes the message from `src`, which must cover exactly `chunks`. */
static int take(sim* s, int dst, int src, const int* chunks, int nchunks, message** out) {
  message* mb = &s->box[dst];
  int i;
  if (!mb->present || mb->src != src) {
    if (s->st->fail_step < 0) {
      s->st->fail_step = s->step;
      s->st->fail_rank = dst;
    }
    return OR_EMISSING;
  }
  if (mb->nchunks != nchunks) return OR_ESCHEDULE;
  for (i = 0; i < nchunks; ++i)
    if (mb->chunks[i] != chunks[i]) return OR_ESCHEDULE;
  s->st->recv[dst] += mb->n;
  *out = mb;
  return OR_OK;
}

static void drop_box(sim* s, int dst) {
  if (s->box[dst].present) free(s->box[dst].data);
  s->box[dst].present = 0;
  s->box[dst].data = NULL;
}

static void clear_boxes(sim* s) {
  int r;
  for (r = 0; r < s->n; ++r) drop_box(s, r);
}

static int mod(int a, int n) { return ((a % n) + n) % n; }

/* ------------------------------------------------------------------------ */
/* Ring                                                                     */
/* ------------------------------------------------------------------------ */

/* ReduceScatter: N-1 steps; in step t rank r sends chunk (r-1-t) mod N to
 * rank r+1, which folds it into its own copy of that chunk: own = step(recv,
 * own).  Afterwards rank r holds the reduced chunk r. */
static int ring_reduce_scatter(sim* s) {
  int t, r, rc;
  for (t = 0; t < s->n - 1; ++t) {
    for (r = 0; r < s->n; ++r) {
      int j = mod(r - 1 - t, s->n);
      if ((rc = post(s, r, (r + 1) % s->n, &j, 1))) return rc;
    }
    for (r = 0; r < s->n; ++r) {
      int j = mod(r - 2 - t, s->n);
      message* mb;
      if ((rc = take(s, r, mod(r - 1, s->n), &j, 1, &mb))) return rc;
      combine(s->dtype, s->op, mb->data, chunk_ptr(s, r, j), chunk_ptr(s, r, j), mb->n);
    }
    clear_boxes(s);
    s->step++;
    s->st->steps++;
  }
  return OR_OK;
}

/* AllGather: N-1 steps; in step t rank r sends chunk (r-t) mod N to rank r+1,
 * which stores it unchanged. */
static int ring_all_gather(sim* s) {
  int t, r, rc;
  for (t = 0; t < s->n - 1; ++t) {
    for (r = 0; r < s->n; ++r) {
      int j = mod(r - t, s->n);
      if ((rc = post(s, r, (r + 1) % s->n, &j, 1))) return rc;
    }
    for (r = 0; r < s->n; ++r) {
      int j = mod(r - 1 - t, s->n);
      message* mb;
      if ((rc = take(s, r, mod(r - 1, s->n), &j, 1, &mb))) return rc;
      memcpy(chunk_ptr(s, r, j), mb->data, (size_t)mb->n * (size_t)s->es);
    }
    clear_boxes(s);
    s->step++;
    s->st->steps++;
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Tree: recursive halving / recursive doubling                             */
/* ------------------------------------------------------------------------ */

static int log2_exact(int n) {
  int k = 0;
  while ((1 << k) < n) ++k;
  return (1 << k) == n ? k : -1;
}

/* Chunks j with j = r (mod 2h): the set rank r keeps after the halving step
 * of distance h. */
static int kept_set(int n, int r, int h, int* out) {
  int j, c = 0;
  for (j = 0; j < n; ++j)
    if (j % (2 * h) == r % (2 * h)) out[c++] = j;
  return c;
}

/* Step k = 0, 1, ..., log2 N - 1 with distance h = 2^k: rank r and partner
 * p = r XOR h exchange; each sends the partial values of the chunks the other
 * keeps, and the receiver folds lower-rank value first: own = step(lower,
 * upper).  After step k rank r holds, for the chunks j = r (mod 2h), the
 * reduction over the 2h ranks that agree with r above bit k, combined as a
 * balanced pairwise tree (ranks 0&1, 2&3, ... then pairs of pairs). */
static int tree_reduce_scatter(sim* s) {
  int L = log2_exact(s->n), k, r, rc;
  int set[OR_MAX_RANKS];
  for (k = 0; k < L; ++k) {
    int h = 1 << k;
    for (r = 0; r < s->n; ++r) {
      int p = r ^ h;
      int c = kept_set(s->n, p, h, set);
      if ((rc = post(s, r, p, set, c))) return rc;
    }
    for (r = 0; r < s->n; ++r) {
      int p = r ^ h, i;
      int c = kept_set(s->n, r, h, set);
      int64_t off = 0;
      message* mb;
      if ((rc = take(s, r, p, set, c, &mb))) return rc;
      for (i = 0; i < c; ++i) {
        unsigned char* own = chunk_ptr(s, r, set[i]);
        unsigned char* got = mb->data + (size_t)off * (size_t)s->es;
        int64_t len = chunk_len(s, set[i]);
        if (r < p) combine(s->dtype, s->op, own, got, own, len);
        else combine(s->dtype, s->op, got, own, own, len);
        off += len;
      }
    }
    clear_boxes(s);
    s->step++;
    s->st->steps++;
  }
  return OR_OK;
}

/* Reverse of the halving: k = log2 N - 1 down to 0; rank r sends the chunks
 * it holds (j = r mod 2h) to r XOR h, which copies them. */
static int tree_all_gather(sim* s) {
  int L = log2_exact(s->n), k, r, rc;
  int set[OR_MAX_RANKS];
  for (k = L - 1; k >= 0; --k) {
    int h = 1 << k;
    for (r = 0; r < s->n; ++r) {
      int c = kept_set(s->n, r, h, set);
      if ((rc = post(s, r, r ^ h, set, c))) return rc;
    }
    for (r = 0; r < s->n; ++r) {
      int p = r ^ h, i;
      int c = kept_set(s->n, p, h, set);
      int64_t off = 0;
      message* mb;
      if ((rc = take(s, r, p, set, c, &mb))) return rc;
      for (i = 0; i < c; ++i) {
        int64_t len = chunk_len(s, set[i]);
        memcpy(chunk_ptr(s, r, set[i]), mb->data + (size_t)off * (size_t)s->es, (size_t)len * (size_t)s->es);
        off += len;
      }
    }
    clear_boxes(s);
    s->step++;
    s->st->steps++;
  }
  return OR_OK;
}

/* Binomial tree: leaves to root, then root to leaves.  Reduce step k
 * (distance h = 2^k): every rank r = h (mod 2h) sends its whole partial to
 * r - h, which folds own (lower) first.  Broadcast in reverse: every rank
 * r = 0 (mod 2h) sends the whole result to r + h. */
static int binomial_allreduce(sim* s, int avg) {
  int L = log2_exact(s->n), k, r, rc, j;
  int all[OR_MAX_RANKS];
  for (j = 0; j < s->n; ++j) all[j] = j;
  for (k = 0; k < L; ++k) {
    int h = 1 << k;
    for (r = 0; r < s->n; ++r)
      if (r % (2 * h) == h)
        if ((rc = post(s, r, r - h, all, s->n))) return rc;
    for (r = 0; r < s->n; ++r)
      if (r % (2 * h) == 0) {
        message* mb;
        if ((rc = take(s, r, r + h, all, s->n, &mb))) return rc;
        combine(s->dtype, s->op, s->rank[r], mb->data, s->rank[r], s->m);
      }
    clear_boxes(s);
    s->step++;
    s->st->steps++;
  }
  if (avg) divide_by(s->dtype, s->rank[0], s->m, s->n);
  for (k = L - 1; k >= 0; --k) {
    int h = 1 << k;
    for (r = 0; r < s->n; ++r)
      if (r % (2 * h) == 0)
        if ((rc = post(s, r, r + h, all, s->n))) return rc;
    for (r = 0; r < s->n; ++r)
      if (r % (2 * h) == h) {
        message* mb;
        if ((rc = take(s, r, r - h, all, s->n, &mb))) return rc;
        memcpy(s->rank[r], mb->data, (size_t)s->m * (size_t)s->es);
      }
    clear_boxes(s);
    s->step++;
    s->st->steps++;
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Naive: rank 0 gathers, reduces, broadcasts                              */
/* ------------------------------------------------------------------------ */

/* Root-side fold order is x_0, x_1, ..., x_{N-1} (own value first).  The
 * pages give this schedule only as the bottleneck example; it is compared
 * only where the result does not depend on order (integers, MAX). */
static int naive_allreduce(sim* s, int avg) {
  int r, j, rc;
  int all[OR_MAX_RANKS];
  for (j = 0; j < s->n; ++j) all[j] = j;
  /* gather: one message per non-root rank, received one after another */
  for (r = 1; r < s->n; ++r) {
    message* mb;
    if ((rc = post(s, r, 0, all, s->n))) return rc;
    if ((rc = take(s, 0, r, all, s->n, &mb))) return rc;
    combine(s->dtype, s->op, s->rank[0], mb->data, s->rank[0], s->m);
    clear_boxes(s);
  }
  s->step++;
  s->st->steps++;
  if (avg) divide_by(s->dtype, s->rank[0], s->m, s->n);
  for (r = 1; r < s->n; ++r) {
    message* mb;
    if ((rc = post(s, 0, r, all, s->n))) return rc;
    if ((rc = take(s, r, 0, all, s->n, &mb))) return rc;
    memcpy(s->rank[r], mb->data, (size_t)s->m * (size_t)s->es);
    clear_boxes(s);
  }
  s->step++;
  s->st->steps++;
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Double binary tree                                                       */
/* ------------------------------------------------------------------------ */

/* Two binary trees that run at the same time, each reducing and then
 * broadcasting half of the data ("AllReduce" concept page §3 技术原理: two
 * disjoint binary trees; "AllReduce 集合通信" §带宽最优与延迟的取舍).  The pages
 * give no tree shape; the one used here: positions 1..N form an in-order
 * binary tree (the root of a range is its position with the most trailing
 * zero bits; left subtree below it, right subtree above it); tree A puts rank
 * p-1 at position p, tree B rank p mod N (shifted by one, so for even N every
 * rank that is a leaf of one tree is inner in the other).  Tree A reduces the
 * first half of the elements, [0, floor(D/2)), tree B the second.  A node
 * folds its left child's partial, its own value, then its right child's
 * partial: ((L (+) own) (+) R). */

typedef struct {
  int parent[OR_MAX_RANKS + 2], left[OR_MAX_RANKS + 2], right[OR_MAX_RANKS + 2];
  int sub_h[OR_MAX_RANKS + 2]; /* 0 for a leaf */
  int depth[OR_MAX_RANKS + 2]; /* 0 for the root */
  int root;
} inorder_tree;

static int trailing_zeros(int p) {
  int k = 0;
  while (!(p & 1)) {
    p >>= 1;
    ++k;
  }
  return k;
}

/* the position with the most trailing zero bits in [lo, hi] */
static int inorder_root_of(int lo, int hi) {
  int p, best = lo, bt = -1;
  for (p = lo; p <= hi; ++p)
    if (trailing_zeros(p) > bt) {
      bt = trailing_zeros(p);
      best = p;
    }
  return best;
}

static int inorder_build(inorder_tree* t, int lo, int hi, int parent, int depth) {
  int best, hl, hr;
  if (lo > hi) return -1;
  best = inorder_root_of(lo, hi);
  t->parent[best] = parent;
  t->depth[best] = depth;
  hl = inorder_build(t, lo, best - 1, best, depth + 1);
  hr = inorder_build(t, best + 1, hi, best, depth + 1);
  t->left[best] = lo <= best - 1 ? inorder_root_of(lo, best - 1) : 0;
  t->right[best] = best + 1 <= hi ? inorder_root_of(best + 1, hi) : 0;
  t->sub_h[best] = 1 + (hl > hr ? hl : hr);
  return t->sub_h[best];
}

/* Reduce then broadcast elements [a, b) of every rank over tree `t`, where
 * position p holds rank (p - 1 + shift) mod N.  Returns the number of
 * communication steps (reduce plus broadcast). */
static int dbtree_half(sim* s, const inorder_tree* t, int shift, int64_t a, int64_t b, int avg) {
  int n = s->n, p, k, maxh = t->sub_h[t->root], maxd = 0;
  int64_t len = b - a;
  size_t bytes = (size_t)(len > 0 ? len : 1) * (size_t)s->es;
  unsigned char* held[OR_MAX_RANKS + 2][2];
  memset(held, 0, sizeof(held));
#define RANK_AT(pos) (((pos) - 1 + shift) % n)
#define SLICE(pos) (s->rank[RANK_AT(pos)] + (size_t)a * (size_t)s->es)
  for (k = 0; k <= maxh; ++k) {
    /* nodes whose subtrees are complete fold what their children sent */
    for (p = 1; p <= n; ++p) {
      if (t->sub_h[p] != k) continue;
      if (held[p][0]) combine(s->dtype, s->op, held[p][0], SLICE(p), SLICE(p), len);
      if (held[p][1]) combine(s->dtype, s->op, SLICE(p), held[p][1], SLICE(p), len);
      free(held[p][0]);
      free(held[p][1]);
      held[p][0] = held[p][1] = NULL;
    }
    /* and send the partial to their parent (copied: the message) */
    for (p = 1; p <= n; ++p) {
      int q, side;
      if (t->sub_h[p] != k || !t->parent[p]) continue;
      q = t->parent[p];
      side = t->left[q] == p ? 0 : 1;
      held[q][side] = (unsigned char*)malloc(bytes);
      if (!held[q][side]) return OR_ENOMEM;
      memcpy(held[q][side], SLICE(p), (size_t)len * (size_t)s->es);
      s->st->sent[RANK_AT(p)] += len;
      s->st->recv[RANK_AT(q)] += len;
    }
  }
  if (avg) divide_by(s->dtype, SLICE(t->root), len, n);
  for (p = 1; p <= n; ++p)
    if (t->depth[p] > maxd) maxd = t->depth[p];
  for (k = 0; k < maxd; ++k)
    for (p = 1; p <= n; ++p) {
      int c;
      if (t->depth[p] != k) continue;
      for (c = 0; c < 2; ++c) {
        int ch = c ? t->right[p] : t->left[p];
        if (!ch) continue;
        memcpy(SLICE(ch), SLICE(p), (size_t)len * (size_t)s->es);
        s->st->sent[RANK_AT(p)] += len;
        s->st->recv[RANK_AT(ch)] += len;
      }
    }
#undef RANK_AT
#undef SLICE
  return maxh + maxd;
}

static int dbtree_allreduce(sim* s, int avg) {
  inorder_tree t;
  int sa, sb;
  memset(&t, 0, sizeof(t));
  inorder_build(&t, 1, s->n, 0, 0);
  t.root = inorder_root_of(1, s->n);
  sa = dbtree_half(s, &t, 0, 0, s->khalf, avg);
  if (sa < 0) return sa;
  sb = dbtree_half(s, &t, 1 % s->n, s->khalf, s->m, avg);
  if (sb < 0) return sb;
  s->st->steps += sa > sb ? sa : sb; /* the two trees run at the same time */
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Entry point                                                              */
/* ------------------------------------------------------------------------ */

/*
 * Simulate one collective over N ranks.
 *
 *  algo     OR_RING, OR_TREE (recursive halving/doubling), OR_BINOMIAL, OR_NAIVE
 *  in[r]    rank r's values, out[r] its result (may alias in[r]); npos values
 *           each when `positions` is given, else `count` values
 *  positions  NULL, or a strictly increasing list of npos element indices in
 *           [0, count): the simulation then carries only those positions in
 *           its messages (elements are independent, and the chunk of each
 *           position follows from `count`)
 *  phases   OR_PHASE_RS (ReduceScatter; AVG divides here), OR_PHASE_AG
 *           (AllGather of the shard each rank owns), or both (AllReduce)
 *  st       filled with step and volume counts
 *  fault    NULL or a host-side failure to inject
 */
int oracle_collective(int algo, const void* const* in, void* const* out, int nranks, int64_t count,
                      const int64_t* positions, int64_t npos, int dtype, int op, int phases,
                      oracle_stats* st, const oracle_fault* fault) {
  sim* s;
  int r, j, rc = OR_OK;
  int64_t i, m;
  oracle_stats local_st;
  if (!st) st = &local_st;
  memset(st, 0, sizeof(*st));
  st->fail_step = -1;
  st->fail_rank = -1;
  if (nranks < 1 || nranks > OR_MAX_RANKS || count < 0 || !in || !out) return OR_EINVAL;
  if (dtype < 0 || dtype > 3 || op < 0 || op > 2 || phases < 1 || phases > 3) return OR_EINVAL;
  if (op == OR_AVG && dtype == OR_I32) return OR_EUNSUPPORTED;
  if (algo < 0 || algo > 4) return OR_EINVAL;
  if ((algo == OR_TREE || algo == OR_BINOMIAL) && log2_exact(nranks) < 0) return OR_EUNSUPPORTED;
  if ((algo == OR_BINOMIAL || algo == OR_NAIVE || algo == OR_DBTREE) && phases != 3) return OR_EUNSUPPORTED;
  m = positions ? npos : count;
  if (positions) {
    for (i = 0; i < npos; ++i)
      if (positions[i] < 0 || positions[i] >= count || (i > 0 && positions[i] <= positions[i - 1])) return OR_EINVAL;
  }
  s = (sim*)calloc(1, sizeof(sim));
  if (!s) return OR_ENOMEM;
  s->n = nranks;
  s->dtype = dtype;
  s->op = op;
  s->es = esize_of(dtype);
  s->m = m;
  s->st = st;
  s->fault = fault;
  /* chunk j covers the local positions whose element index lies in chunk j */
  for (j = 0; j <= nranks; ++j) {
    int64_t lo = (int64_t)(((__int128)j * count) / nranks);
    if (!positions) {
      s->klo[j] = lo;
    } else {
      int64_t k = 0;
      while (k < npos && positions[k] < lo) ++k;
      s->klo[j] = k;
    }
  }
  s->khalf = count / 2;
  if (positions) {
    int64_t k = 0;
    while (k < npos && positions[k] < count / 2) ++k;
    s->khalf = k;
  }
  for (r = 0; r < nranks; ++r) {
    s->rank[r] = (unsigned char*)malloc((size_t)(m > 0 ? m : 1) * (size_t)s->es);
    if (!s->rank[r]) {
      rc = OR_ENOMEM;
      goto done;
    }
    memcpy(s->rank[r], in[r], (size_t)m * (size_t)s->es);
  }
  if (algo == OR_DBTREE) {
    rc = dbtree_allreduce(s, op == OR_AVG);
  } else if (algo == OR_RING || algo == OR_TREE) {
    if (phases & OR_PHASE_RS) {
      rc = algo == OR_RING ? ring_reduce_scatter(s) : tree_reduce_scatter(s);
      if (rc) goto done;
      if (op == OR_AVG)
        for (r = 0; r < nranks; ++r) divide_by(dtype, chunk_ptr(s, r, r), chunk_len(s, r), nranks);
    }
    if (phases & OR_PHASE_AG) {
      rc = algo == OR_RING ? ring_all_gather(s) : tree_all_gather(s);
      if (rc) goto done;
    }
  } else if (algo == OR_BINOMIAL) {
    rc = binomial_allreduce(s, op == OR_AVG);
  } else {
    rc = naive_allreduce(s, op == OR_AVG);
  }
  if (rc) goto done;
  for (r = 0; r < nranks; ++r) memcpy(out[r], s->rank[r], (size_t)m * (size_t)s->es);
done:
  clear_boxes(s);
  for (r = 0; r < nranks; ++r) free(s->rank[r]);
  free(s);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Reduce and Broadcast (the rest of the collectives table)                 */
/* ------------------------------------------------------------------------ */

/* Reduce: the reduction lands at `root` only ("AllReduce 集合通信" §语义:
 * Reduce = reduce to the root; the other ranks' buffers are left as the
 * schedule leaves them).  Ring / tree: ReduceScatter as in the AllReduce
 * (AVG at the owners), then every owner r != root sends its finished chunk
 * to the root, one message per step.  Naive: the root receives every other
 * buffer and folds x_0, x_1, ..., x_{N-1} in index order. */
static int reduce_to_root(sim* s, int algo, int root, int avg) {
  int r, j, rc;
  int all[OR_MAX_RANKS];
  if (algo == OR_NAIVE) {
    unsigned char* got[OR_MAX_RANKS] = {0};
    for (j = 0; j < s->n; ++j) all[j] = j;
    for (r = 0; r < s->n; ++r) {
      message* mb;
      if (r == root) continue;
      if ((rc = post(s, r, root, all, s->n))) return rc;
      if ((rc = take(s, root, r, all, s->n, &mb))) return rc;
      got[r] = mb->data; /* keep the received copy; the box is emptied by hand */
      s->box[root].data = NULL;
      s->box[root].present = 0;
      s->step++;
      s->st->steps++;
    }
    got[root] = (unsigned char*)malloc((size_t)(s->m > 0 ? s->m : 1) * (size_t)s->es);
    if (!got[root]) rc = OR_ENOMEM;
    else {
      memcpy(got[root], s->rank[root], (size_t)s->m * (size_t)s->es);
      memcpy(s->rank[root], got[0], (size_t)s->m * (size_t)s->es);
      for (r = 1; r < s->n; ++r) combine(s->dtype, s->op, s->rank[root], got[r], s->rank[root], s->m);
      if (avg) divide_by(s->dtype, s->rank[root], s->m, s->n);
      rc = OR_OK;
    }
    for (r = 0; r < s->n; ++r) free(got[r]);
    return rc;
  }
  rc = algo == OR_RING ? ring_reduce_scatter(s) : tree_reduce_scatter(s);
  if (rc) return rc;
  if (avg)
    for (r = 0; r < s->n; ++r) divide_by(s->dtype, chunk_ptr(s, r, r), chunk_len(s, r), s->n);
  for (r = 0; r < s->n; ++r) {
    message* mb;
    if (r == root) continue;
    if ((rc = post(s, r, root, &r, 1))) return rc;
    if ((rc = take(s, root, r, &r, 1, &mb))) return rc;
    memcpy(chunk_ptr(s, root, r), mb->data, (size_t)mb->n * (size_t)s->es);
    clear_boxes(s);
    s->step++;
    s->st->steps++;
  }
  return OR_OK;
}

/* Broadcast: the root's buffer is copied to every rank, one message per
 * receiving rank ("AllReduce 集合通信" §语义; "【AI Infra小白入门⑩】" §二). */
static int broadcast_from_root(sim* s, int root) {
  int r, j, rc;
  int all[OR_MAX_RANKS];
  for (j = 0; j < s->n; ++j) all[j] = j;
  for (r = 0; r < s->n; ++r) {
    message* mb;
    if (r == root) continue;
    if ((rc = post(s, root, r, all, s->n))) return rc;
    if ((rc = take(s, r, root, all, s->n, &mb))) return rc;
    memcpy(s->rank[r], mb->data, (size_t)s->m * (size_t)s->es);
    clear_boxes(s);
    s->step++;
    s->st->steps++;
  }
  return OR_OK;
}

enum { OR_KIND_REDUCE = 0, OR_KIND_BROADCAST = 1 };

/*
 * Rooted collectives.  kind OR_KIND_REDUCE (algo ring, tree or naive; op as
 * for AllReduce) or OR_KIND_BROADCAST (algo and op ignored).  Other
 * arguments as oracle_collective.  After a Reduce only out[root] is defined
 * by the operation; the other outputs hold what the schedule left there.
 */
int oracle_rooted(int kind, int algo, const void* const* in, void* const* out, int nranks, int64_t count,
                  const int64_t* positions, int64_t npos, int dtype, int op, int root, oracle_stats* st) {
  sim* s;
  int r, j, rc = OR_OK;
  int64_t i, m;
  oracle_stats local_st;
  if (!st) st = &local_st;
  memset(st, 0, sizeof(*st));
  st->fail_step = -1;
  st->fail_rank = -1;
  if (nranks < 1 || nranks > OR_MAX_RANKS || count < 0 || !in || !out || root < 0 || root >= nranks) return OR_EINVAL;
  if (dtype < 0 || dtype > 3 || kind < 0 || kind > 1) return OR_EINVAL;
  if (kind == OR_KIND_REDUCE) {
    if (op < 0 || op > 2 || (algo != OR_RING && algo != OR_TREE && algo != OR_NAIVE)) return OR_EINVAL;
    if (op == OR_AVG && dtype == OR_I32) return OR_EUNSUPPORTED;
    if (algo == OR_TREE && log2_exact(nranks) < 0) return OR_EUNSUPPORTED;
  }
  m = positions ? npos : count;
  if (positions)
    for (i = 0; i < npos; ++i)
      if (positions[i] < 0 || positions[i] >= count || (i > 0 && positions[i] <= positions[i - 1])) return OR_EINVAL;
  s = (sim*)calloc(1, sizeof(sim));
  if (!s) return OR_ENOMEM;
  s->n = nranks;
  s->dtype = dtype;
  s->op = op == OR_MAX ? OR_MAX : OR_SUM;
  s->es = esize_of(dtype);
  s->m = m;
  s->st = st;
  for (j = 0; j <= nranks; ++j) {
    int64_t lo = (int64_t)(((__int128)j * count) / nranks);
    if (!positions) {
      s->klo[j] = lo;
    } else {
      int64_t k = 0;
      while (k < npos && positions[k] < lo) ++k;
      s->klo[j] = k;
    }
  }
  for (r = 0; r < nranks; ++r) {
    s->rank[r] = (unsigned char*)malloc((size_t)(m > 0 ? m : 1) * (size_t)s->es);
    if (!s->rank[r]) {
      rc = OR_ENOMEM;
      goto done;
    }
    memcpy(s->rank[r], in[r], (size_t)m * (size_t)s->es);
  }
  rc = kind == OR_KIND_REDUCE ? reduce_to_root(s, algo, root, op == OR_AVG) : broadcast_from_root(s, root);
  if (rc) goto done;
  for (r = 0; r < nranks; ++r) memcpy(out[r], s->rank[r], (size_t)m * (size_t)s->es);
done:
  clear_boxes(s);
  for (r = 0; r < nranks; ++r) free(s->rank[r]);
  free(s);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* 8-bit quantised AllReduce with error feedback                            */
/* ------------------------------------------------------------------------ */

/* "Allreduce：大模型分布式训练的核心通信算法与优化实践" §4.2: gradients are
 * quantised to 8-bit integers for transmission and dequantised by the
 * receiver; error feedback carries this round's compression error into the
 * next round.  The pages fix nothing more; the scheme here (PARITY UNPINNED
 * by the pages: pinned only by its own exact cases and error bounds):
 *
 *  - blocks of OR_Q8 = 128 consecutive elements from the start of the buffer;
 *  - every rank r: y = x + e (its residual), per block s = max|y| / 127,
 *    q = round-half-even(y / s) clamped to [-127, 127] (q = 0 when s = 0),
 *    y^ = q * s, new residual e = y - y^  (binary32, round to nearest);
 *  - ReduceScatter with 8-bit payloads: every rank sends each chunk's q
 *    (and the scales of the blocks it touches) to the chunk's owner; the
 *    owner folds the dequantised contributions in ring order x[c+1], ...,
 *    x[c] in binary32 (AVG: then divides by N);
 *  - AllGather with 8-bit payloads: the owner requantises its chunk (blocks
 *    cut at the chunk's ends, same rule, no feedback) and sends (q, s) to
 *    every rank; every rank, the owner included, keeps q * s.
 * Inputs must be finite. */

#define OR_Q8 128

static float q8_scale(const float* y, int64_t n) {
  float m = 0.0f;
  int64_t i;
  for (i = 0; i < n; ++i)
    if (fabsf(y[i]) > m) m = fabsf(y[i]);
  return m / 127.0f;
}

static signed char q8_code(float y, float s) {
  float q;
  if (s == 0.0f) return 0;
  q = nearbyintf(y / s); /* default rounding mode: to nearest, ties to even */
  if (q > 127.0f) q = 127.0f;
  if (q < -127.0f) q = -127.0f;
  return (signed char)q;
}

/* one rank: quantise x + e block by block; returns codes and scales, updates e */
static void q8_encode(const float* x, float* e, int64_t count, signed char* q, float* scale) {
  int64_t b, i, nb = (count + OR_Q8 - 1) / OR_Q8;
  float y[OR_Q8];
  for (b = 0; b < nb; ++b) {
    int64_t lo = b * OR_Q8, n = (count - lo < OR_Q8) ? count - lo : OR_Q8;
    for (i = 0; i < n; ++i) y[i] = x[lo + i] + e[lo + i];
    scale[b] = q8_scale(y, n);
    for (i = 0; i < n; ++i) {
      q[lo + i] = q8_code(y[i], scale[b]);
      e[lo + i] = y[i] - (float)q[lo + i] * scale[b];
    }
  }
}

/*
 * x[r], e[r]: rank r's gradient and residual (count binary32 each), updated
 * in place: x gets the reduced result, e the new residual.  op OR_SUM or
 * OR_AVG.  st counts the 8-bit payload elements sent and received.
 */
/* An 8-bit message: the codes of one chunk and the scales of the blocks it
 * touches (block b0 first). */
typedef struct {
  signed char* q;
  float* s;
  int64_t b0;
} q8_msg;

static int64_t chunk_bound(int64_t count, int n, int c) { return (int64_t)(((__int128)c * count) / n); }

int oracle_int8_ef_allreduce(float* const* x, float* const* e, int nranks, int64_t count, int op,
                             oracle_stats* st) {
  int r, c, t, rc = OR_OK;
  int64_t nb, i;
  signed char* q[OR_MAX_RANKS] = {0};
  float* sc[OR_MAX_RANKS] = {0};
  q8_msg* inbox = NULL;  /* inbox[c * N + r]: rank r's payload for owner c */
  q8_msg* outbox = NULL; /* outbox[c]: owner c's requantised chunk */
  float* acc = NULL;
  oracle_stats local_st;
  if (!st) st = &local_st;
  memset(st, 0, sizeof(*st));
  st->fail_step = -1;
  st->fail_rank = -1;
  if (nranks < 1 || nranks > OR_MAX_RANKS || count < 0 || (op != OR_SUM && op != OR_AVG)) return OR_EINVAL;
  nb = (count + OR_Q8 - 1) / OR_Q8;
  inbox = (q8_msg*)calloc((size_t)nranks * nranks, sizeof(q8_msg));
  outbox = (q8_msg*)calloc((size_t)nranks, sizeof(q8_msg));
  acc = (float*)malloc((size_t)(count > 0 ? count : 1) * sizeof(float));
  if (!inbox || !outbox || !acc) {
    rc = OR_ENOMEM;
    goto done;
  }
  for (r = 0; r < nranks; ++r) {
    q[r] = (signed char*)malloc((size_t)(count > 0 ? count : 1));
    sc[r] = (float*)malloc((size_t)(nb > 0 ? nb : 1) * sizeof(float));
    if (!q[r] || !sc[r]) {
      rc = OR_ENOMEM;
      goto done;
    }
    q8_encode(x[r], e[r], count, q[r], sc[r]);
  }
  /* ReduceScatter: in step t rank r posts chunk (r + t + 1) mod N of its codes
   * to that chunk's owner */
  for (t = 0; t < nranks - 1; ++t) {
    for (r = 0; r < nranks; ++r) {
      int j = (r + t + 1) % nranks;
      int64_t lo = chunk_bound(count, nranks, j), hi = chunk_bound(count, nranks, j + 1);
      int64_t b0 = lo / OR_Q8, b1 = hi > lo ? (hi - 1) / OR_Q8 + 1 : b0;
      q8_msg* m = &inbox[(size_t)j * nranks + r];
      m->q = (signed char*)malloc((size_t)(hi - lo > 0 ? hi - lo : 1));
      m->s = (float*)malloc((size_t)(b1 - b0 > 0 ? b1 - b0 : 1) * sizeof(float));
      if (!m->q || !m->s) {
        rc = OR_ENOMEM;
        goto done;
      }
      memcpy(m->q, q[r] + lo, (size_t)(hi - lo));
      memcpy(m->s, sc[r] + b0, (size_t)(b1 - b0) * sizeof(float));
      m->b0 = b0;
      st->sent[r] += hi - lo;
      st->recv[j] += hi - lo;
    }
    st->steps++;
  }
  /* every owner folds the dequantised contributions of its chunk in ring
   * order x[c+1], ..., x[c] (its own from its own codes), then requantises
   * the chunk, blocks cut at the chunk's ends */
  for (c = 0; c < nranks; ++c) {
    int64_t lo = chunk_bound(count, nranks, c), hi = chunk_bound(count, nranks, c + 1), b;
    for (i = lo; i < hi; ++i) {
      int p;
      float a = 0.0f;
      for (p = 0; p < nranks; ++p) {
        int rr = (c + 1 + p) % nranks;
        float v;
        if (rr == c) {
          v = (float)q[c][i] * sc[c][i / OR_Q8];
        } else {
          const q8_msg* m = &inbox[(size_t)c * nranks + rr];
          v = (float)m->q[i - lo] * m->s[i / OR_Q8 - m->b0];
        }
        a = p == 0 ? v : a + v;
      }
      if (op == OR_AVG) a = a / (float)nranks;
      acc[i] = a;
    }
    outbox[c].q = (signed char*)malloc((size_t)(hi - lo > 0 ? hi - lo : 1));
    outbox[c].s = (float*)malloc((size_t)((hi - lo) / OR_Q8 + 2) * sizeof(float));
    if (!outbox[c].q || !outbox[c].s) {
      rc = OR_ENOMEM;
      goto done;
    }
    outbox[c].b0 = lo / OR_Q8;
    for (b = lo / OR_Q8; b * OR_Q8 < hi; ++b) {
      int64_t blo = b * OR_Q8 > lo ? b * OR_Q8 : lo;
      int64_t bhi = (b + 1) * OR_Q8 < hi ? (b + 1) * OR_Q8 : hi;
      float s = q8_scale(acc + blo, bhi - blo);
      outbox[c].s[b - outbox[c].b0] = s;
      for (i = blo; i < bhi; ++i) outbox[c].q[i - lo] = q8_code(acc[i], s);
    }
  }
  /* AllGather: in step t owner r posts its requantised chunk to rank
   * (r + t + 1) mod N; every rank, the owner included, keeps codes x scales */
  for (t = 0; t < nranks - 1; ++t) {
    for (r = 0; r < nranks; ++r) {
      int j = (r + t + 1) % nranks;
      int64_t lo = chunk_bound(count, nranks, r), hi = chunk_bound(count, nranks, r + 1);
      st->sent[r] += hi - lo;
      st->recv[j] += hi - lo;
    }
    st->steps++;
  }
  for (c = 0; c < nranks; ++c) {
    int64_t lo = chunk_bound(count, nranks, c), hi = chunk_bound(count, nranks, c + 1);
    for (r = 0; r < nranks; ++r)
      for (i = lo; i < hi; ++i) x[r][i] = (float)outbox[c].q[i - lo] * outbox[c].s[i / OR_Q8 - outbox[c].b0];
  }
done:
  for (r = 0; r < nranks; ++r) {
    free(q[r]);
    free(sc[r]);
  }
  if (inbox)
    for (i = 0; i < (int64_t)nranks * nranks; ++i) {
      free(inbox[i].q);
      free(inbox[i].s);
    }
  if (outbox)
    for (c = 0; c < nranks; ++c) {
      free(outbox[c].q);
      free(outbox[c].s);
    }
  free(inbox);
  free(outbox);
  free(acc);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* DDP buckets                                                              */
/* ------------------------------------------------------------------------ */

/*
 * Bucket plan.  Walk the tensors in reverse registration order and add each
 * to the current bucket while the bucket stays within cap_bytes; a tensor that
 * does not fit closes the bucket and opens the next one; a tensor larger than
 * the cap therefore sits alone.  Inside a bucket tensors are laid out in the
 * order they were added (reverse registration order).  Bucket 0 holds the
 * last-registered tensors.
 */
int oracle_bucket_plan(const int64_t* counts, int ntensors, int dtype, int64_t cap_bytes,
                       int32_t* bucket_of, int64_t* offset_in_bucket, int64_t* bucket_count, int32_t* nbuckets) {
  int t, b = -1;
  int64_t fill = 0;
  int es;
  if (ntensors < 0 || cap_bytes <= 0 || dtype < 0 || dtype > 3 || !nbuckets) return OR_EINVAL;
  es = esize_of(dtype);
  for (t = ntensors - 1; t >= 0; --t) {
    int64_t bytes;
    if (counts[t] < 0) return OR_EINVAL;
    bytes = counts[t] * es;
    if (b < 0 || (fill > 0 && fill + bytes > cap_bytes)) {
      ++b;
      bucket_count[b] = 0;
      fill = 0;
    }
    bucket_of[t] = b;
    offset_in_bucket[t] = bucket_count[b];
    bucket_count[b] += counts[t];
    fill += bytes;
  }
  *nbuckets = b + 1;
  return OR_OK;
}

typedef struct {
  int64_t pos;
  int64_t id;
} pair;

static int cmp_pair(const void* a, const void* b) {
  int64_t x = ((const pair*)a)->pos, y = ((const pair*)b)->pos;
  return x < y ? -1 : (x > y ? 1 : 0);
}

/*
 * Bucketed AllReduce, literally: for each bucket, every rank packs its
 * tensors into a flat bucket buffer, the ranks run one collective over the
 * bucket buffers, and every rank copies the result back into its tensors.
 *
 *  grads_in / grads_out  [nranks * ntensors] pointers, row-major by rank
 *  samp_tensor / samp_index / nsamp   when nsamp > 0 only these elements are
 *           carried (tensor id, element index; all distinct), and results go
 *           to samp_out[r * nsamp + i]; grads_out is then unused
 */
int oracle_bucketed_allreduce(const void* const* grads_in, void* const* grads_out, const int64_t* counts,
                              int ntensors, int nranks, int dtype, int op, int algo, int64_t cap_bytes,
                              const int32_t* samp_tensor, const int64_t* samp_index, int64_t nsamp,
                              void* samp_out, oracle_stats* st_total) {
  int32_t *bucket_of = NULL, nb = 0;
  int64_t *off = NULL, *bcount = NULL;
  int es, b, r, t, rc = OR_OK;
  oracle_stats st;
  if (ntensors < 0 || nranks < 1 || nranks > OR_MAX_RANKS || dtype < 0 || dtype > 3) return OR_EINVAL;
  es = esize_of(dtype);
  bucket_of = (int32_t*)calloc((size_t)(ntensors + 1), sizeof(int32_t));
  off = (int64_t*)calloc((size_t)(ntensors + 1), sizeof(int64_t));
  bcount = (int64_t*)calloc((size_t)(ntensors + 1), sizeof(int64_t));
  if (!bucket_of || !off || !bcount) {
    rc = OR_ENOMEM;
    goto out;
  }
  if ((rc = oracle_bucket_plan(counts, ntensors, dtype, cap_bytes, bucket_of, off, bcount, &nb))) goto out;
  if (st_total) {
    memset(st_total, 0, sizeof(*st_total));
    st_total->fail_step = -1;
    st_total->fail_rank = -1;
  }
  for (b = 0; b < nb; ++b) {
    void* bufs[OR_MAX_RANKS];
    int64_t* pos = NULL;
    int64_t* which = NULL; /* sample id of each carried position */
    int64_t m = 0, i;
    if (nsamp > 0) {
      /* this bucket's samples as (bucket offset, sample id), ascending */
      pair* ps = (pair*)malloc((size_t)(nsamp + 1) * sizeof(pair));
      pos = (int64_t*)malloc((size_t)(nsamp + 1) * sizeof(int64_t));
      which = (int64_t*)malloc((size_t)(nsamp + 1) * sizeof(int64_t));
      if (!ps || !pos || !which) {
        free(ps);
        free(pos);
        free(which);
        rc = OR_ENOMEM;
        goto out;
      }
      for (i = 0; i < nsamp; ++i) {
        int32_t ts = samp_tensor[i];
        if (ts < 0 || ts >= ntensors || samp_index[i] < 0 || samp_index[i] >= counts[ts]) {
          rc = OR_EINVAL;
          break;
        }
        if (bucket_of[ts] == b) {
          ps[m].pos = off[ts] + samp_index[i];
          ps[m].id = i;
          ++m;
        }
      }
      if (!rc) {
        qsort(ps, (size_t)m, sizeof(pair), cmp_pair);
        for (i = 0; i < m; ++i) {
          if (i > 0 && ps[i].pos == ps[i - 1].pos) rc = OR_EINVAL; /* samples must be distinct */
          pos[i] = ps[i].pos;
          which[i] = ps[i].id;
        }
      }
      free(ps);
      if (rc) {
        free(pos);
        free(which);
        goto out;
      }
    } else {
      m = bcount[b];
    }
    for (r = 0; r < nranks; ++r) {
      bufs[r] = malloc((size_t)(m > 0 ? m : 1) * (size_t)es);
      if (!bufs[r]) {
        int q;
        for (q = 0; q < r; ++q) free(bufs[q]);
        free(pos);
        free(which);
        rc = OR_ENOMEM;
        goto out;
      }
    }
    /* pack */
    for (r = 0; r < nranks; ++r) {
      if (nsamp > 0) {
        for (i = 0; i < m; ++i) {
          /* find the tensor holding bucket offset pos[i] */
          for (t = 0; t < ntensors; ++t)
            if (bucket_of[t] == b && pos[i] >= off[t] && pos[i] < off[t] + counts[t]) break;
          memcpy((unsigned char*)bufs[r] + (size_t)i * es,
                 (const unsigned char*)grads_in[(size_t)r * ntensors + t] + (size_t)(pos[i] - off[t]) * es, (size_t)es);
        }
      } else {
        for (t = 0; t < ntensors; ++t)
          if (bucket_of[t] == b)
            memcpy((unsigned char*)bufs[r] + (size_t)off[t] * es, grads_in[(size_t)r * ntensors + t],
                   (size_t)counts[t] * es);
      }
    }
    rc = oracle_collective(algo, (const void* const*)bufs, bufs, nranks, bcount[b], nsamp > 0 ? pos : NULL, m, dtype, op, 3,
                           &st, NULL);
    if (!rc) {
      if (st_total) {
        st_total->steps += st.steps;
        for (r = 0; r < nranks; ++r) {
          st_total->sent[r] += st.sent[r];
          st_total->recv[r] += st.recv[r];
        }
      }
      /* unpack */
      for (r = 0; r < nranks; ++r) {
        if (nsamp > 0) {
          for (i = 0; i < m; ++i)
            memcpy((unsigned char*)samp_out + ((size_t)r * nsamp + which[i]) * es, (unsigned char*)bufs[r] + (size_t)i * es,
                   (size_t)es);
        } else {
          for (t = 0; t < ntensors; ++t)
            if (bucket_of[t] == b)
              memcpy(grads_out[(size_t)r * ntensors + t], (unsigned char*)bufs[r] + (size_t)off[t] * es,
                     (size_t)counts[t] * es);
        }
      }
    }
    for (r = 0; r < nranks; ++r) free(bufs[r]);
    free(pos);
    free(which);
    if (rc) goto out;
  }
out:
  free(bucket_of);
  free(off);
  free(bcount);
  return rc;
}

int oracle_max_ranks(void) { return OR_MAX_RANKS; }
