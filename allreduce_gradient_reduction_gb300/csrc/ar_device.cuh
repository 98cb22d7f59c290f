// Device-side building blocks shared by the kernels: the element step for
// each (dtype, op), 16-byte vector forms of it, streaming loads and stores,
// and the segment/tile bookkeeping.
//
// Element step (the pages ask for sum / max / average; the arithmetic is
// IEEE): f32 SUM is one binary32 addition rounded to nearest even (compiled
// without fast-math, so subnormals are kept); bf16 and f16 SUM give the sum
// correctly rounded to the storage type, nearest-even (the same value as
// widening both operands to binary32, adding, and rounding back -- the
// rounding a step-wise ring applies after every received chunk), computed
// by the packed half-precision addition; i32 SUM wraps;
// MAX is the IEEE 754-2019 maximum (NaN propagates, +0 > -0).  AVG divides
// once by N with IEEE binary32 division.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ar_internal.h"

namespace ar {

// ---- programmatic dependent launch ------------------------------------------
// The fused, gather and copy kernels are launched so that the next kernel on
// the stream may start while this one drains: every block first allows its
// dependents to launch, then waits until the kernels it depends on have
// completed and their writes are visible.  Nothing touches global memory
// before that wait, so a kernel never sees a predecessor's data half
// written; what overlaps is the next launch and its blocks' start-up with
// the last blocks of this one.  (The launch attribute is what makes the
// dependency programmatic; launched without it, both instructions do
// nothing.)
__device__ __forceinline__ void pdl_prologue() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int DT>
struct ElemSize {
  static constexpr int value = (DT == BF16 || DT == F16) ? 2 : 4;
};

// ---- one 32-bit word: 1 f32, 2 bf16, 2 f16 or 1 i32 ------------------------

// IEEE maximum of two binary32 values: the NaN-propagating maximum
// instruction (+0 > -0).  On the bucket workload (8 x 25 MiB f32 MAX) 64.1 us
// against 65.1 us for compares of the two values.
__device__ __forceinline__ uint32_t f32_max_bits(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.f32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);  // .x (low 16 bits) = lo
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ float f16_to_float(uint32_t h) { return __half2float(__ushort_as_half((unsigned short)h)); }

__device__ __forceinline__ uint32_t pack_f16x2_rn(float lo, float hi) {
  __half2 r = __floats2half2_rn(lo, hi);  // .x (low 16 bits) = lo
  return *reinterpret_cast<uint32_t*>(&r);
}

// IEEE maximum of two pairs of 16-bit floats at once: the packed
// NaN-propagating maximum instruction (a NaN operand gives a NaN; +0 > -0).
// Measured on 8 x 128 MiB: bf16 312.5 us, f16 314.5 us, against 341.7 and
// 337.3 us for a per-half compare of the widened values, and 368-370 us for
// an integer-SIMD form (order-preserving keys and a per-halfword maximum).
__device__ __forceinline__ uint32_t bf16x2_max_hw(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmax2_nan(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t f16x2_max_hw(uint32_t a, uint32_t b) {
  __half2 r = __hmax2_nan(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

template <int DT, int OP>
__device__ __forceinline__ uint32_t step_word(uint32_t a, uint32_t b) {
  if constexpr (DT == F32) {
    if constexpr (OP == SUM) return __float_as_uint(__fadd_rn(__uint_as_float(a), __uint_as_float(b)));
    else return f32_max_bits(a, b);
  } else if constexpr (DT == BF16) {
    if constexpr (OP == SUM) {
      // the packed bf16 addition, rounded to nearest even, subnormals kept:
      // one correct rounding of the exact sum per half, which is what
      // widening to binary32, adding and rounding back gives (24 >= 2*8+2,
      // so that double rounding is innocuous); checked over all 2^32 pairs
      uint32_t r;
      asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
      return r;
    } else {
      return bf16x2_max_hw(a, b);
    }
  } else if constexpr (DT == F16) {
    if constexpr (OP == SUM) {
      // the packed binary16 addition, rounded to nearest even, subnormals
      // kept (no .ftz): the correctly rounded sum, as widening, adding in
      // binary32 and rounding back gives (24 >= 2*11+2); checked over all
      // 2^32 pairs
      uint32_t r;
      asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
      return r;
    } else {
      return f16x2_max_hw(a, b);
    }
  } else {
    if constexpr (OP == SUM) {
      // two's-complement wrap-around, as one opaque instruction: the
      // compiler must not reassociate a long fold of them (that would keep
      // every loaded value live at once and spill)
      uint32_t r;
      asm("add.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
      return r;
    }
    else return (uint32_t)max((int32_t)a, (int32_t)b);
  }
}

template <int DT>
__device__ __forceinline__ uint32_t div_word(uint32_t a, float fn) {
  if constexpr (DT == F32) {
    return __float_as_uint(__fdiv_rn(__uint_as_float(a), fn));
  } else if constexpr (DT == BF16) {
    return pack_bf16x2_rn(__fdiv_rn(__uint_as_float(a << 16), fn), __fdiv_rn(__uint_as_float(a & 0xFFFF0000u), fn));
  } else if constexpr (DT == F16) {
    return pack_f16x2_rn(__fdiv_rn(f16_to_float(a & 0xFFFFu), fn), __fdiv_rn(f16_to_float(a >> 16), fn));
  } else {
    return a;
  }
}

// ---- 16-byte vectors --------------------------------------------------------

template <int DT, int OP>
__device__ __forceinline__ uint4 step_vec(const uint4& a, const uint4& b) {
  return make_uint4(step_word<DT, OP>(a.x, b.x), step_word<DT, OP>(a.y, b.y), step_word<DT, OP>(a.z, b.z),
                    step_word<DT, OP>(a.w, b.w));
}

template <int DT>
__device__ __forceinline__ uint4 div_vec(const uint4& a, float fn) {
  return make_uint4(div_word<DT>(a.x, fn), div_word<DT>(a.y, fn), div_word<DT>(a.z, fn), div_word<DT>(a.w, fn));
}

// Streaming accesses: every byte is touched once, so keep it out of L1 and
// mark it first in line for L2 eviction.
__device__ __forceinline__ uint4 ld_stream(const void* p) { return __ldcs(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ void st_stream(void* p, const uint4& v) { __stcs(reinterpret_cast<uint4*>(p), v); }
// L2-coherent accesses for kernels whose phases read what other blocks wrote.
__device__ __forceinline__ uint4 ld_l2(const void* p) { return __ldcg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ void st_l2(void* p, const uint4& v) { __stcg(reinterpret_cast<uint4*>(p), v); }

// 16-byte global -> shared copy that bypasses L1; both addresses 16-byte
// aligned.  cp_async_wait_all waits for all of this thread's copies.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned sa = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// waits until at most K of this thread's committed groups are still in flight
template <int K>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(K) : "memory");
}
// the same for a count known only after unrolling (0..7)
__device__ __forceinline__ void cp_async_wait_pending(int k) {
  switch (k) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    case 6: cp_async_wait<6>(); break;
    default: cp_async_wait<7>(); break;
  }
}

// Bulk shared -> global copy (the tensor-memory-access engine, no tensor
// map): both addresses 16-byte aligned, a size that is a multiple of 16.
// The shared data must be made visible to the async proxy first
// (fence_proxy_async_shared by the threads that wrote it, then a block
// barrier).  bulk_commit closes this thread's group of bulk copies;
// bulk_wait_read waits until they have read their shared memory,
// bulk_wait_all until their writes are done.
__device__ __forceinline__ void bulk_store(void* gmem, const void* smem, uint32_t bytes) {
  const unsigned sa = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem), "r"(sa), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... all but this thread's most recent group
__device__ __forceinline__ void bulk_wait_read_but_one() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---- single elements --------------------------------------------------------

template <int ES>
__device__ __forceinline__ uint32_t ld_elem(const void* base, int64_t e) {
  if constexpr (ES == 2) return __ldcg(reinterpret_cast<const unsigned short*>(base) + e);
  else return __ldcg(reinterpret_cast<const unsigned int*>(base) + e);
}

template <int ES>
__device__ __forceinline__ void st_elem(void* base, int64_t e, uint32_t v) {
  if constexpr (ES == 2) __stcg(reinterpret_cast<unsigned short*>(base) + e, (unsigned short)v);
  else __stcg(reinterpret_cast<unsigned int*>(base) + e, v);
}

// ---- segments and tiles -----------------------------------------------------

// Index of the segment holding `tile`: the last segment whose tile_begin is <= tile.
template <class TABLE>
__device__ __forceinline__ int find_seg(const TABLE& t, int64_t tile) {
  int lo = 0, hi = t.nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (t.seg[mid].tile_begin <= tile) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Full 16-byte vectors of a segment: [vb, ve) in units of VEC elements.
// Elements outside them (at most VEC-1 on each side) are "scalars": with
// ve > vb they are [begin, vb*VEC - shift) and [ve*VEC - shift, end);
// otherwise all of [begin, end).
struct SegShape {
  int64_t vb, ve;
  int head, tail;  // scalar counts before / after the vectors
};

// Rows whose N buffers share the same address modulo 16 (not necessarily 0)
// still move in 16-byte vectors: with `shift` = (address mod 16) / element
// size, vector v of the row covers elements [v*VEC - shift, (v+1)*VEC -
// shift), at byte offset v*16 - shift*ES from every buffer of the row, which
// is 16-byte aligned in all of them.  shift = 0 for aligned rows.
__host__ __device__ __forceinline__ int row_shift(const void* p0, int es) {
  return (int)(((uintptr_t)p0 & 15) / (uintptr_t)es);
}

template <int VEC>
__device__ __forceinline__ SegShape seg_shape(const Seg& s, int shift = 0) {
  SegShape r;
  r.vb = (s.begin + shift + VEC - 1) / VEC;
  r.ve = (s.end + shift) / VEC;
  if (r.ve > r.vb) {
    r.head = (int)(r.vb * VEC - shift - s.begin);
    r.tail = (int)(s.end - (r.ve * VEC - shift));
  } else {
    r.ve = r.vb;
    r.head = (int)(s.end - s.begin);
    r.tail = 0;
  }
  return r;
}

// Element index of scalar k (0 <= k < head + tail) of a segment.
template <int VEC>
__device__ __forceinline__ int64_t scalar_elem(const Seg& s, const SegShape& sh, int k, int shift = 0) {
  return k < sh.head ? s.begin + k : sh.ve * VEC - shift + (k - sh.head);
}

__device__ __forceinline__ int rot(int k, int n) { return k >= n ? k - n : k; }

// ---- scalar folds (runtime N) -----------------------------------------------

// Ring order for element e of chunk c: x[c+1], x[c+2], ..., x[c].
template <int DT, int OP>
__device__ uint32_t fold_ring_scalar(const void* const* P, int n, int c, int64_t e) {
  constexpr int ES = ElemSize<DT>::value;
  uint32_t acc = ld_elem<ES>(P[rot(c + 1, n)], e);
  for (int p = 1; p < n; ++p) acc = step_word<DT, OP>(acc, ld_elem<ES>(P[rot(c + 1 + p, n)], e));
  return acc;
}

// Balanced pairwise tree over ranks 0..n-1 (n a power of two), lower first.
template <int DT, int OP>
__device__ uint32_t fold_tree_scalar(const void* const* P, int n, int64_t e) {
  constexpr int ES = ElemSize<DT>::value;
  uint32_t stack[8];
  int top = 0;
  for (int r = 0; r < n; ++r) {
    uint32_t v = ld_elem<ES>(P[r], e);
    for (int k = r; k & 1; k >>= 1) v = step_word<DT, OP>(stack[--top], v);
    stack[top++] = v;
  }
  return stack[0];
}

// Double binary tree: positions 1..N form an in-order binary tree whose root
// over [lo, hi] is the position with the most trailing zero bits -- hi with
// every bit below the highest bit in which lo and hi differ cleared; position
// p holds rank (p - 1 + shift) mod N (tree A: shift 0, tree B: shift 1).  A
// node folds ((left subtree) (+) own) (+) (right subtree).
__host__ __device__ constexpr int highest_bit(unsigned v) {
  int b = -1;
  while (v) {
    v >>= 1;
    ++b;
  }
  return b;
}

__host__ __device__ constexpr int inorder_root(int lo, int hi) {
  return lo == hi ? lo : (hi & ~((1 << highest_bit((unsigned)(lo ^ hi))) - 1));
}

// The fold over positions 1..n, without recursion (a device stack whose
// depth the compiler cannot bound could overflow the per-thread stack): an
// explicit frame stack of at most log2(n) + 2 entries emulates it.
template <int DT, int OP>
__device__ uint32_t fold_dbtree_scalar(const void* const* P, int n, int shift, int64_t e) {
  constexpr int ES = ElemSize<DT>::value;
  struct Frame {
    int lo, hi, r, stage;  // stage 0: new, 1: left subtree folded, 2: right subtree folded
    uint32_t acc;
  };
  Frame f[10];  // n <= 64: ranges at least halve on each push
  int sp = 0;
  f[0] = {1, n, inorder_root(1, n), 0, 0u};
  uint32_t ret = 0u;  // value of the subtree that finished last
  for (;;) {
    Frame& t = f[sp];
    const uint32_t own = t.stage == 2 ? 0u : ld_elem<ES>(P[(t.r - 1 + shift) % n], e);
    if (t.stage == 0 && t.lo < t.r) {
      t.stage = 1;
      f[sp + 1] = {t.lo, t.r - 1, inorder_root(t.lo, t.r - 1), 0, 0u};
      ++sp;
      continue;
    }
    if (t.stage == 0) t.acc = own;
    else if (t.stage == 1) t.acc = step_word<DT, OP>(ret, own);
    else t.acc = step_word<DT, OP>(t.acc, ret);
    if (t.stage != 2 && t.r < t.hi) {
      t.stage = 2;
      f[sp + 1] = {t.r + 1, t.hi, inorder_root(t.r + 1, t.hi), 0, 0u};
      ++sp;
      continue;
    }
    ret = t.acc;
    if (sp == 0) return ret;
    --sp;
  }
}

// One element in the order of `order` (chunk c selects the ring rotation,
// and for the double binary tree the tree: 0 = A, 1 = B).
template <int DT, int OP, int ORDER>
__device__ __forceinline__ uint32_t fold_scalar(const void* const* P, int n, int c, int64_t e) {
  if constexpr (ORDER == RING) return fold_ring_scalar<DT, OP>(P, n, c, e);
  else if constexpr (ORDER == TREE) return fold_tree_scalar<DT, OP>(P, n, e);
  else return fold_dbtree_scalar<DT, OP>(P, n, c, e);
}

}  // namespace ar
