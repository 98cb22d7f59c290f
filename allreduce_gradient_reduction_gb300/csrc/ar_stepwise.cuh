// Step-wise kernels: the literal communication schedule, one grid-wide phase
// per step, in one persistent cooperative kernel.
//
// Ring ("Allreduce：大模型分布式训练的核心通信算法与优化实践" §2.2; "AllReduce 集合
// 通信" §两阶段流程): ReduceScatter step s (s = 0..N-2): rank r sends chunk
// (r-1-s) mod N to rank r+1, which folds it into its own copy,
// own = step(received, own) -- so chunk j moves from rank j+1+s to j+2+s.
// AllGather step s: rank r forwards chunk (r-s) mod N to r+1 unchanged.
// Tree ("【AI Infra小白入门⑩】集合通信基础" §四 4.1): recursive halving, step k
// (distance h = 2^k, k = 0 first) pairs rank r with r XOR h; rank r keeps the
// chunks j = r (mod 2h) and folds lower rank first; then recursive doubling in
// reverse order copies the halves back.  AVG divides at the owner after the
// last ReduceScatter step.
// Binomial ("4、AllReduce算法详解" §4.3, reduce to a root then broadcast; nearest
// ranks first as in the primer's §四 4.1): reduce step k (h = 2^k, k = 0
// first) has rank r = h (mod 2h) send its whole buffer to r - h, which folds
// it in (lower rank first); broadcast step k (k = log2 N - 1 first) has rank
// r = 0 (mod 2h) send its whole buffer to r + h.  AVG divides at rank 0 after
// the last reduce step.  Whole buffers move, so the table has one segment.
//
// "Sending" chunk j from rank a to rank b is rank b's threads reading rank
// a's buffer in HBM: one GPU holds all ranks.  Within a phase no location is
// both read as a source and written, so a phase needs no intra-phase ordering;
// between phases a bounded grid barrier orders everything.  Loads and stores
// go through L2 (.cg), the coherence point for data other blocks wrote.
#pragma once

#include <cooperative_groups.h>

#include "ar_device.cuh"

namespace ar {

constexpr int kStepBlock = 256;
constexpr int kStepUnroll = 2;
constexpr unsigned kMaxSpin = 1u << 23;  // backstop if the global timer misbehaves
constexpr int kTimeoutStatus = -4;       // AR_ERR_TIMEOUT

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int ld_relaxed_s32(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid-wide barrier with a bounded wait.  Returns false when the kernel must
// stop: this block timed out (it then raises `abort` for the others and
// records AR_ERR_TIMEOUT in the sticky status) or another block already did.
// The abort flag and the clock are read every 32 polls, and the poll backs
// off only after 1024 (measured: 64 ranks x 64 KiB bf16 ring 279.6 -> 260.9
// us, 2.2 -> 2.1 us a step; never backing off made no further difference).
// The block's stores are ordered before its arrival by the CTA barrier and
// the gpu-scope release of the arrival (release is cumulative); the acquire
// load that sees the last arrival orders every later load after all of them.
__device__ bool grid_barrier(SyncBlock* sb, unsigned target, bool arrive, int64_t timeout_ns) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    if (arrive) red_release_add(&sb->counter, 1u);
    const uint64_t t0 = global_ns();
    unsigned spins = 0;
    while (ld_acquire_u32(&sb->counter) < target) {
      if ((++spins & 31) == 0) {
        if (ld_relaxed_s32(&sb->abort)) {
          ok = 0;
          break;
        }
        if (spins > kMaxSpin || global_ns() - t0 > (uint64_t)timeout_ns) {
          atomicExch(&sb->abort, 1);
          atomicCAS(&sb->status, 0, kTimeoutStatus);
          ok = 0;
          break;
        }
      }
      if (spins > 1024) __nanosleep(64);
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

__device__ __forceinline__ int ilog2(int n) { return 31 - __clz(n); }

template <int DT, int OP, bool VECTOR>
__global__ void __launch_bounds__(kStepBlock) stepwise_kernel(const __grid_constant__ StepArgs a) {
  constexpr int ES = ElemSize<DT>::value;
  constexpr int VEC = VECTOR ? 16 / ES : 1;
  constexpr int TILE = kStepBlock * kStepUnroll;
  const SegTable& T = a.tab;
  const int n = T.nranks;
  const bool ring = a.order == RING;
  const bool binom = a.order == BINOMIAL;
  const int L = ring ? 0 : ilog2(n);
  const int n_rs = (a.phases & 1) ? (ring ? n - 1 : L) : 0;
  const int n_ag = (a.phases & 2) ? (ring ? n - 1 : L) : 0;
  const int Q = n_rs + n_ag;

  for (int q = 0; q < Q; ++q) {
    const bool rs = q < n_rs;
    const int s = rs ? q : q - n_rs;     // step within its half
    const int k = rs ? s : L - 1 - s;    // tree distance exponent
    const int h = 1 << k;
    const int inst = ring ? 1 : (n >> (k + 1));  // rank pairs per chunk in a tree or binomial step
    const bool avg = a.avg && rs && s == n_rs - 1;
    const int64_t total = (int64_t)inst * T.ntiles;

    for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
      const int m = (int)(w / T.ntiles);
      const int64_t tile = w - (int64_t)m * T.ntiles;
      const Seg& sg = T.seg[find_seg(T, tile)];
      const int j = sg.chunk;
      int src, dst;
      if (ring) {
        src = rs ? (j + 1 + s) % n : (j + s) % n;
        dst = src + 1 == n ? 0 : src + 1;
      } else if (binom) {
        dst = m * 2 * h + (rs ? 0 : h);
        src = dst ^ h;
      } else {
        dst = rs ? ((j & (2 * h - 1)) + m * 2 * h) : (((j ^ h) & (2 * h - 1)) + m * 2 * h);
        src = dst ^ h;
      }
      const bool src_first = ring || src < dst;  // ring: received first; trees: lower rank first
      const void* const* P = T.ptr + (size_t)sg.tensor * n;
      const char* ps = static_cast<const char*>(P[src]);
      char* pd = static_cast<char*>(const_cast<void*>(P[dst]));
      const int64_t ti = tile - sg.tile_begin;

      if constexpr (VECTOR) {
        const int shift = row_shift(P[0], ES);  // the row's buffers share it
        const SegShape sh = seg_shape<VEC>(sg, shift);
        uint4 xs[kStepUnroll], xd[kStepUnroll];
        int64_t off[kStepUnroll];
        bool ok[kStepUnroll];
#pragma unroll
        for (int u = 0; u < kStepUnroll; ++u) {
          const int64_t v = sh.vb + ti * TILE + u * kStepBlock + threadIdx.x;
          ok[u] = v < sh.ve;
          off[u] = v * 16 - shift * ES;
          if (ok[u]) {
            xs[u] = ld_l2(ps + off[u]);
            if (rs) xd[u] = ld_l2(pd + off[u]);
          }
        }
#pragma unroll
        for (int u = 0; u < kStepUnroll; ++u) {
          if (!ok[u]) continue;
          uint4 r = xs[u];
          if (rs) {
            r = src_first ? step_vec<DT, OP>(xs[u], xd[u]) : step_vec<DT, OP>(xd[u], xs[u]);
            if (avg) r = div_vec<DT>(r, a.fn);
          }
          st_l2(pd + off[u], r);
        }
        if (ti == 0 && (int)threadIdx.x < sh.head + sh.tail) {
          const int64_t e = scalar_elem<VEC>(sg, sh, threadIdx.x, shift);
          uint32_t r = ld_elem<ES>(ps, e);
          if (rs) {
            const uint32_t d = ld_elem<ES>(pd, e);
            r = src_first ? step_word<DT, OP>(r, d) : step_word<DT, OP>(d, r);
            if (avg) r = div_word<DT>(r, a.fn);
          }
          st_elem<ES>(pd, e, r);
        }
      } else {
#pragma unroll
        for (int u = 0; u < kStepUnroll; ++u) {
          const int64_t e = sg.begin + ti * TILE + u * kStepBlock + threadIdx.x;
          if (e >= sg.end) continue;
          uint32_t r = ld_elem<ES>(ps, e);
          if (rs) {
            const uint32_t d = ld_elem<ES>(pd, e);
            r = src_first ? step_word<DT, OP>(r, d) : step_word<DT, OP>(d, r);
            if (avg) r = div_word<DT>(r, a.fn);
          }
          st_elem<ES>(pd, e, r);
        }
      }
    }
    if (q + 1 < Q) {
      const bool arrive = !(blockIdx.x == 0 && q == a.skip_barrier);
      if (!grid_barrier(a.sync, (unsigned)(q + 1) * gridDim.x, arrive, a.timeout_ns)) return;
    }
  }
}

// The same schedule for a small buffer row, in one block: every rank's
// buffer is staged in shared memory (elements at their own size, each rank's
// region padded to 16 bytes), the phases run there with a block barrier
// between them, and the final state is written back.  Same per-element
// operations in the same order as stepwise_kernel, so the same bits; a phase
// costs a block barrier instead of a grid barrier and an L2 round trip.
// Sizes here are small enough for 32-bit index arithmetic.
constexpr int kSmemStepBlock = 1024;
constexpr int kSmemStepUnroll = 4;  // 16-byte copies in flight per thread while staging

template <int ES>
struct SmemWord;
template <>
struct SmemWord<2> {
  using type = unsigned short;
};
template <>
struct SmemWord<4> {
  using type = unsigned int;
};

// Moves every rank's buffer between global memory and its shared-memory
// region (to_smem: global -> shared).  16-byte pieces when the buffers are
// 16-byte aligned, then the last count * ES % 16 bytes element by element.
template <int ES, bool TO_SMEM>
__device__ __forceinline__ void smem_stage(const SmemStepArgs& a, unsigned char* S, int stride, int n, int count) {
  using Wd = typename SmemWord<ES>::type;
  const int nvec = a.vec ? count * ES / 16 : 0;
  const int total = n * nvec;
  for (int i0 = threadIdx.x; i0 < total; i0 += kSmemStepUnroll * kSmemStepBlock) {
    uint4 v[kSmemStepUnroll];
#pragma unroll
    for (int u = 0; u < kSmemStepUnroll; ++u) {
      const int i = i0 + u * kSmemStepBlock;
      if (i < total) {
        const int r = i / nvec, k = i - r * nvec;
        uint4* sp = reinterpret_cast<uint4*>(S + r * stride) + k;
        if constexpr (TO_SMEM) v[u] = ld_l2(static_cast<const uint4*>(a.ptr[r]) + k);
        else v[u] = *sp;
      }
    }
#pragma unroll
    for (int u = 0; u < kSmemStepUnroll; ++u) {
      const int i = i0 + u * kSmemStepBlock;
      if (i < total) {
        const int r = i / nvec, k = i - r * nvec;
        uint4* sp = reinterpret_cast<uint4*>(S + r * stride) + k;
        if constexpr (TO_SMEM) *sp = v[u];
        else st_l2(static_cast<uint4*>(const_cast<void*>(a.ptr[r])) + k, v[u]);
      }
    }
  }
  const int done = nvec * 16 / ES, rest = count - done;  // elements left per rank
  for (int i = threadIdx.x; i < n * rest; i += kSmemStepBlock) {
    const int r = i / rest, e = done + (i - r * rest);
    Wd* sp = reinterpret_cast<Wd*>(S + r * stride) + e;
    if constexpr (TO_SMEM) *sp = (Wd)ld_elem<ES>(a.ptr[r], e);
    else st_elem<ES>(const_cast<void*>(a.ptr[r]), e, *sp);
  }
}

template <int DT, int OP>
__global__ void __launch_bounds__(kSmemStepBlock) stepwise_smem_kernel(const __grid_constant__ SmemStepArgs a) {
  constexpr int ES = ElemSize<DT>::value;
  using Wd = typename SmemWord<ES>::type;
  extern __shared__ __align__(16) unsigned char S[];  // rank r's elements at S + r * stride
  const int n = a.nranks;
  const int count = (int)a.count;
  const int stride = (count * ES + 15) / 16 * 16;
  smem_stage<ES, true>(a, S, stride, n, count);
  __syncthreads();
  const bool ring = a.order == RING;
  const bool binom = a.order == BINOMIAL;
  const int L = ring ? 0 : ilog2(n);
  const int n_rs = (a.phases & 1) ? (ring ? n - 1 : L) : 0;
  const int n_ag = (a.phases & 2) ? (ring ? n - 1 : L) : 0;
  for (int q = 0; q < n_rs + n_ag; ++q) {
    const bool rs = q < n_rs;
    const int s = rs ? q : q - n_rs;
    const int k = rs ? s : L - 1 - s;
    const int h = 1 << k;
    const int inst = ring ? 1 : (n >> (k + 1));
    const bool avg = a.avg && rs && s == n_rs - 1;
    for (int w = threadIdx.x; w < inst * count; w += kSmemStepBlock) {
      const int m = w / count;
      const int e = w - m * count;
      const int j = ((e + 1) * n - 1) / count;  // chunk [floor(jD/N), floor((j+1)D/N)) holding e
      int src, dst;
      if (ring) {
        src = rs ? (j + 1 + s) % n : (j + s) % n;
        dst = src + 1 == n ? 0 : src + 1;
      } else if (binom) {
        dst = m * 2 * h + (rs ? 0 : h);
        src = dst ^ h;
      } else {
        dst = rs ? ((j & (2 * h - 1)) + m * 2 * h) : (((j ^ h) & (2 * h - 1)) + m * 2 * h);
        src = dst ^ h;
      }
      Wd* ps = reinterpret_cast<Wd*>(S + src * stride) + e;
      Wd* pd = reinterpret_cast<Wd*>(S + dst * stride) + e;
      uint32_t r = *ps;
      if (rs) {
        const uint32_t d = *pd;
        r = (ring || src < dst) ? step_word<DT, OP>(r, d) : step_word<DT, OP>(d, r);
        if (avg) r = div_word<DT>(r, a.fn);
      }
      *pd = (Wd)r;
    }
    __syncthreads();
  }
  smem_stage<ES, false>(a, S, stride, n, count);
}

// ---- the same schedule in one thread-block cluster ---------------------------
//
// For rows too large for one block's shared memory but small enough that a
// grid-wide barrier per step would dominate: the C blocks of one cluster
// hold the N rank buffers between them (rank r in block r mod C, at
// (r / C) * stride of its shared memory).  In a step each block folds the
// elements its own ranks receive, reading the sender's values straight from
// the sender block's shared memory (distributed shared memory), and the
// steps are separated by the cluster's hardware barrier, whose release /
// acquire order the writes of one step before the reads of the next.  Same
// per-element operations in the same order as stepwise_kernel, so the same
// bits.  Each block moves only its own ranks in and out of global memory.
constexpr int kClusterStepBlock = 512;

// What rank r receives in step s of its half (rs: the reduce half), k the
// tree distance exponent: `nch` chunks j0, j0 + jstep, ... from rank `src`
// (binomial: the whole buffer as one range), or nothing (nch = 0).
struct StepRecv {
  int src, j0, jstep, nch;
  bool whole;
};

__device__ __forceinline__ StepRecv step_recv(int order, bool rs, int s, int k, int n, int r) {
  StepRecv v{0, 0, 1, 0, false};
  const int h = order == RING ? 1 : 1 << k;  // (the ring has no distance)
  if (order == RING) {
    v.src = r == 0 ? n - 1 : r - 1;
    v.j0 = ((r - (rs ? 2 : 1) - s) % n + n) % n;
    v.nch = 1;
  } else if (order == BINOMIAL) {
    const bool recv = rs ? (r & (2 * h - 1)) == 0 : (r & (2 * h - 1)) == h;
    if (recv) {
      v.src = r ^ h;
      v.nch = 1;
      v.whole = true;
    }
  } else {
    v.src = r ^ h;
    v.j0 = (rs ? r : (r ^ h)) & (2 * h - 1);
    v.jstep = 2 * h;
    v.nch = n / (2 * h);
  }
  return v;
}

template <int DT, int OP>
__global__ void __launch_bounds__(kClusterStepBlock) stepwise_cluster_kernel(const __grid_constant__ SmemStepArgs a) {
  namespace cg = cooperative_groups;
  constexpr int ES = ElemSize<DT>::value;
  using Wd = typename SmemWord<ES>::type;
  extern __shared__ __align__(16) unsigned char S[];
  cg::cluster_group cl = cg::this_cluster();
  const int C = (int)cl.num_blocks();
  const int me = (int)cl.block_rank();
  const int n = a.nranks;
  const int count = (int)a.count;
  const int stride = (count * ES + 15) / 16 * 16;
  const int nloc = (n - me + C - 1) / C;  // ranks me, me + C, ...
  const int maxch = (count + n - 1) / n;  // elements of the largest chunk
  constexpr int VEC = 16 / ES;
  // chunks (and whole buffers) cut on 16-byte boundaries of the staged rows
  const bool vmode = count % (n * VEC) == 0;

  // stage this block's ranks in (16-byte pieces when aligned, then the tail)
  const int nvec = a.vec ? count * ES / 16 : 0;
  for (int i = threadIdx.x; i < nloc * nvec; i += kClusterStepBlock) {
    const int l = i / nvec, kk = i - l * nvec;
    reinterpret_cast<uint4*>(S + l * stride)[kk] = ld_l2(static_cast<const uint4*>(a.ptr[me + l * C]) + kk);
  }
  const int done = nvec * 16 / ES, rest = count - done;
  for (int i = threadIdx.x; i < nloc * rest; i += kClusterStepBlock) {
    const int l = i / rest, e = done + (i - l * rest);
    reinterpret_cast<Wd*>(S + l * stride)[e] = (Wd)ld_elem<ES>(a.ptr[me + l * C], e);
  }
  cl.sync();

  const bool ring = a.order == RING;
  const int L = ring ? 0 : ilog2(n);
  const int n_rs = (a.phases & 1) ? (ring ? n - 1 : L) : 0;
  const int n_ag = (a.phases & 2) ? (ring ? n - 1 : L) : 0;
  for (int q = 0; q < n_rs + n_ag; ++q) {
    const bool rs = q < n_rs;
    const int s = rs ? q : q - n_rs;
    const int k = rs ? s : L - 1 - s;
    const bool avg = a.avg && rs && s == n_rs - 1;
    // items: (local rank, chunk of its list, offset in the chunk), four
    // per thread at a time so their remote loads are in flight together;
    // index arithmetic in 32 bits (count * nranks < 2^31 for rows this size)
    const bool whole = a.order == BINOMIAL;
    const int nch_max = ring || whole ? 1 : n / (2 << k);
    constexpr int CU = 4;
    if (vmode) {
      // every chunk starts and ends on a 16-byte boundary: 16-byte items
      const int per_ch = (whole ? count : maxch) / VEC;
      const int span = nch_max * per_ch;
      const int items = nloc * span;
      for (int w0 = threadIdx.x; w0 < items; w0 += CU * kClusterStepBlock) {
        uint4* pd[CU];
        const uint4* ps[CU];
        bool go[CU], src_first[CU];
#pragma unroll
        for (int u = 0; u < CU; ++u) {
          const int w = w0 + u * kClusterStepBlock;
          go[u] = false;
          pd[u] = nullptr;
          ps[u] = nullptr;
          src_first[u] = true;
          if (w < items) {
            const int l = w / span;
            const int rem = w - l * span;
            const int ci = rem / per_ch, offv = rem - ci * per_ch;
            const int r = me + l * C;
            const StepRecv v = step_recv(a.order, rs, s, k, n, r);
            if (ci < v.nch) {
              const int e = (v.whole ? 0 : (v.j0 + ci * v.jstep) * (count / n)) + offv * VEC;
              go[u] = true;
              pd[u] = reinterpret_cast<uint4*>(S + l * stride + e * ES);
              ps[u] = cl.map_shared_rank(reinterpret_cast<uint4*>(S + (v.src / C) * stride + e * ES), v.src % C);
              src_first[u] = ring || v.src < r;
            }
          }
        }
        uint4 x[CU], d[CU];
#pragma unroll
        for (int u = 0; u < CU; ++u) {
          if (go[u]) {
            x[u] = *ps[u];
            if (rs) d[u] = *pd[u];
          }
        }
#pragma unroll
        for (int u = 0; u < CU; ++u) {
          if (!go[u]) continue;
          uint4 y = x[u];
          if (rs) {
            y = src_first[u] ? step_vec<DT, OP>(x[u], d[u]) : step_vec<DT, OP>(d[u], x[u]);
            if (avg) y = div_vec<DT>(y, a.fn);
          }
          *pd[u] = y;
        }
      }
      cl.sync();
      continue;
    }
    const int per_ch = whole ? count : maxch;
    const int span = nch_max * per_ch;
    const int items = nloc * span;
    for (int w0 = threadIdx.x; w0 < items; w0 += CU * kClusterStepBlock) {
      Wd* pd[CU];
      const Wd* ps[CU];
      bool go[CU], src_first[CU];
#pragma unroll
      for (int u = 0; u < CU; ++u) {
        const int w = w0 + u * kClusterStepBlock;
        go[u] = false;
        pd[u] = nullptr;
        ps[u] = nullptr;
        src_first[u] = true;
        if (w < items) {
          const int l = w / span;
          const int rem = w - l * span;
          const int ci = rem / per_ch, off = rem - ci * per_ch;
          const int r = me + l * C;
          const StepRecv v = step_recv(a.order, rs, s, k, n, r);
          int e = off;
          bool in = ci < v.nch;
          if (in && !v.whole) {
            const int j = v.j0 + ci * v.jstep;
            const int lo = j * count / n, hi = (j + 1) * count / n;
            e = lo + off;
            in = e < hi;
          }
          if (in) {
            go[u] = true;
            pd[u] = reinterpret_cast<Wd*>(S + l * stride) + e;
            ps[u] = cl.map_shared_rank(reinterpret_cast<Wd*>(S + (v.src / C) * stride) + e, v.src % C);
            src_first[u] = ring || v.src < r;
          }
        }
      }
      uint32_t x[CU], d[CU];
#pragma unroll
      for (int u = 0; u < CU; ++u) {
        if (go[u]) {
          x[u] = *ps[u];
          d[u] = rs ? (uint32_t)*pd[u] : 0u;
        }
      }
#pragma unroll
      for (int u = 0; u < CU; ++u) {
        if (!go[u]) continue;
        uint32_t y = x[u];
        if (rs) {
          y = src_first[u] ? step_word<DT, OP>(x[u], d[u]) : step_word<DT, OP>(d[u], x[u]);
          if (avg) y = div_word<DT>(y, a.fn);
        }
        *pd[u] = (Wd)y;
      }
    }
    cl.sync();
  }

  // stage this block's ranks out
  for (int i = threadIdx.x; i < nloc * nvec; i += kClusterStepBlock) {
    const int l = i / nvec, kk = i - l * nvec;
    st_l2(static_cast<uint4*>(const_cast<void*>(a.ptr[me + l * C])) + kk, reinterpret_cast<const uint4*>(S + l * stride)[kk]);
  }
  for (int i = threadIdx.x; i < nloc * rest; i += kClusterStepBlock) {
    const int l = i / rest, e = done + (i - l * rest);
    st_elem<ES>(const_cast<void*>(a.ptr[me + l * C]), e, reinterpret_cast<const Wd*>(S + l * stride)[e]);
  }
}

}  // namespace ar
