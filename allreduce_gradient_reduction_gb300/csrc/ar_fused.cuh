// Fused single-pass AllReduce / ReduceScatter kernels.
//
// One pass over HBM: each thread owns 16-byte vectors of one segment (a run
// of elements inside one chunk c), loads the N rank vectors at that position,
// folds them in the order the schedule would -- ring: x[c+1], x[c+2], ...,
// x[c] around the ring ("Allreduce：大模型分布式训练的核心通信算法与优化实践"
// §2.2, "AllReduce 集合通信" §两阶段流程); tree: the balanced pairwise tree
// (0,1), (2,3), ... ("【AI Infra小白入门⑩】集合通信基础" §四 4.1) -- rounding
// to the storage type after every step, optionally divides by N (DDP's
// average, same tutorial §3.1), and stores the finished vector to every rank
// (AllReduce) or to the chunk owner only (ReduceScatter).  Every element is
// read once per rank and written once per destination: 2*N*D*b bytes for an
// AllReduce of D elements of b bytes, the minimum.
//
// The fold is per element, so the result is bit-identical to the step-wise
// schedule (ReduceScatter's N-1 accumulate steps then AllGather's N-1 copies)
// regardless of how elements are spread over threads.  A thread reads all N
// values of a vector before it writes any, so working in place is safe.
#pragma once

#include "ar_device.cuh"

namespace ar {

constexpr int kFusedBlock = 256;

// 16-byte vector positions per thread per tile (U), chosen so that each
// thread keeps about 8 rank loads of 16 bytes in flight (U x min(N, 8)) and
// stays within 64 registers: 4 blocks of 256 threads per SM.  Measured on
// GB300 (8 x 128 MiB bf16 ring): U=1 at 4 blocks/SM 309.8 us, U=2 310.7 us,
// U=3 at 2 blocks/SM 311.3 us, U=4 at 1 block/SM 343.5 us -- occupancy
// matters more than loads per thread once the grid is one tile per block.
// Resident blocks per SM the register budget is cut for: 4 (64 registers) for
// up to 8 ranks; the in-order double-binary-tree fold of 8 ranks keeps more
// partial sums live and gets 3 (80 registers), without spills.  Beyond 8
// ranks every order keeps two groups of 8 rank loads in flight.  The ring
// then gets 3 (at 2 it was 1.9% slower on 64 x 64 MiB; at 3 as fast as one
// group at a time at 4 blocks per SM, and twice as fast for calls of
// 4-64 KiB).  The trees, which also hold finished subtrees, get 2 (128
// registers), without spills.
__host__ __device__ constexpr int fused_min_blocks(int order, int nr) {
  return nr > 8 ? (order == RING ? 3 : 2) : (order == DBTREE && nr == 8 ? 3 : 4);
}
__host__ __device__ constexpr int fused_unroll(int order, int nr) {
  return (nr == 2) ? 2 : 1;
}

// Grids are sized one tile per block, not persistent: blocks start in index
// order, so the blocks in flight at any moment cover a compact window of
// consecutive tiles in all 2N streams, which keeps HBM rows open; on GB300
// this measured 5-10% faster than a grid of resident blocks striding over
// the tiles.  The loop in the kernels still strides, for grids at the cap.
constexpr int64_t kMaxGrid = 1 << 30;

template <int DT, int OP, int NR>
__device__ __forceinline__ uint4 tree_fold_regs(uint4 (&x)[NR]) {
#pragma unroll
  for (int w = 1; w < NR; w <<= 1)
#pragma unroll
    for (int i = 0; i < NR; i += 2 * w) x[i] = step_vec<DT, OP>(x[i], x[i + w]);
  return x[0];
}

// Double binary tree over register-resident rank vectors x[rank] (see
// inorder_root): ((left) (+) own) (+) (right), positions LO..HI, shift SH.
template <int DT, int OP, int NR, int SH, int LO, int HI>
__device__ __forceinline__ uint4 inorder_fold_regs(const uint4 (&x)[NR]) {
  constexpr int R = inorder_root(LO, HI);
  uint4 acc = x[(R - 1 + SH) % NR];
  if constexpr (LO < R) acc = step_vec<DT, OP>(inorder_fold_regs<DT, OP, NR, SH, LO, R - 1>(x), acc);
  if constexpr (R < HI) acc = step_vec<DT, OP>(acc, inorder_fold_regs<DT, OP, NR, SH, R + 1, HI>(x));
  return acc;
}

// Double binary tree over many ranks.  The in-order fold of positions LO..HI
// visits them in increasing order (left subtree, own, right subtree), so the
// rank vectors can be streamed eight positions at a time: the loads of a
// group go out together when its first position is needed, and only that
// group and the pending partial sums live in registers.  Position p holds
// rank p - 1 + rank_shift (mod NR).
template <int NR>
struct DbtStream {
  const void* const* P;
  int64_t base;
  int rank_shift;
  bool ok;
  uint4 g[8];
  template <int POS>
  __device__ __forceinline__ uint4 at() {
    if constexpr ((POS - 1) % 8 == 0) {
      // keep each group's loads here: hoisting all of them (integer adds may
      // be reassociated freely) would need NR vectors of registers at once
      asm volatile("" ::: "memory");
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (ok) g[q] = ld_stream(static_cast<const char*>(P[rot(POS - 1 + q + rank_shift, NR)]) + base);
    }
    return g[(POS - 1) % 8];
  }
};

template <int DT, int OP, int NR, int LO, int HI>
__device__ __forceinline__ uint4 inorder_fold_stream(DbtStream<NR>& st) {
  constexpr int R = inorder_root(LO, HI);
  uint4 acc;
  if constexpr (LO < R) {
    const uint4 left = inorder_fold_stream<DT, OP, NR, LO, R - 1>(st);
    acc = step_vec<DT, OP>(left, st.template at<R>());
  } else {
    acc = st.template at<R>();
  }
  if constexpr (R < HI) acc = step_vec<DT, OP>(acc, inorder_fold_stream<DT, OP, NR, R + 1, HI>(st));
  return acc;
}

// The row's buffers share their address modulo 16: every rank is read and
// written in aligned 16-byte vectors at the same offset.
template <class ARGS, int DT, int OP, int ORDER, int NR>
__global__ void __launch_bounds__(kFusedBlock, fused_min_blocks(ORDER, NR))
    fused_vec_kernel(const __grid_constant__ ARGS a) {
  constexpr int ES = ElemSize<DT>::value;
  constexpr int VEC = 16 / ES;
  constexpr int U = fused_unroll(ORDER, NR);
  pdl_prologue();
  const auto& T = a.tab;
  const int n = NR > 0 ? NR : T.nranks;

  for (int64_t tile = blockIdx.x; tile < T.ntiles; tile += gridDim.x) {
    const Seg& s = T.seg[find_seg(T, tile)];
    const void* const* P = T.ptr + (size_t)s.tensor * n;
    const int shift = row_shift(P[0], ES);  // all the row's buffers share it
    const SegShape sh = seg_shape<VEC>(s, shift);
    const int64_t ti = tile - s.tile_begin;
    const int c = s.chunk;

    // position u of this thread is byte offset base + u * kStride in every
    // rank, 16-byte aligned in all of them
    const int64_t v0 = sh.vb + ti * (kFusedBlock * U) + threadIdx.x;
    const int64_t base = v0 * 16 - shift * ES;
    constexpr int64_t kStride = (int64_t)kFusedBlock * 16;
    bool ok[U];  // this thread folds position u
#pragma unroll
    for (int u = 0; u < U; ++u) ok[u] = v0 + u * kFusedBlock < sh.ve;
    auto ld = [&](int rk, int u) -> uint4 { return ld_stream(static_cast<const char*>(P[rk]) + base + u * kStride); };

    uint4 acc[U];
    if constexpr (ORDER == RING && NR > 8) {
      // 16, 32 or 64 ranks: groups of 8 in ring order, the loads of group
      // g + 1 in flight while group g is folded (16 vectors of registers)
      static_assert(U == 1, "one vector position per thread for wide rings");
      constexpr int G = 8;
      uint4 cur[G], nxt[G];
#pragma unroll
      for (int q = 0; q < G; ++q)
        if (ok[0]) cur[q] = ld_stream(static_cast<const char*>(P[rot(c + 1 + q, NR)]) + base);
#pragma unroll
      for (int g = 0; g < NR; g += G) {
        // keep group g + 2's loads behind group g's fold (integer adds may
        // be reassociated, which would let every load hoist)
        asm volatile("" ::: "memory");
        if (g + G < NR) {
#pragma unroll
          for (int q = 0; q < G; ++q)
            if (ok[0]) nxt[q] = ld_stream(static_cast<const char*>(P[rot(c + 1 + g + G + q, NR)]) + base);
        }
#pragma unroll
        for (int q = 0; q < G; ++q) acc[0] = (g + q == 0) ? cur[q] : step_vec<DT, OP>(acc[0], cur[q]);
        if (g + G < NR) {
#pragma unroll
          for (int q = 0; q < G; ++q) cur[q] = nxt[q];
        }
      }
    } else if constexpr (ORDER == RING && NR > 0) {
      uint4 x[U][NR];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int p = 0; p < NR; ++p)
          if (ok[u]) x[u][p] = ld(rot(c + 1 + p, NR), u);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        acc[u] = x[u][0];
#pragma unroll
        for (int p = 1; p < NR; ++p) acc[u] = step_vec<DT, OP>(acc[u], x[u][p]);
      }
    } else if constexpr (ORDER == RING) {
      // any N: groups of 8 ranks in ring order, folded as they arrive
      for (int g = 0; g < n; g += 8) {
        uint4 x[U][8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (g + q < n) {
            const int rk = rot(c + 1 + g + q, n);
#pragma unroll
            for (int u = 0; u < U; ++u)
              if (ok[u]) x[u][q] = ld(rk, u);
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (g + q < n) {
            const int rk = rot(c + 1 + g + q, n);
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const uint4 v = x[u][q];
              acc[u] = (g + q == 0) ? v : step_vec<DT, OP>(acc[u], v);
            }
          }
        }
      }
    } else if constexpr (ORDER == DBTREE) {
      // chunk 0: tree A over the first half of the elements, chunk 1: tree B.
      // Tree B is tree A over the ranks shifted by one, so the shift goes
      // into which buffer lands at each position, and one tree is compiled.
      const int rank_shift = c == 0 ? 0 : 1;
      if constexpr (NR <= 8) {
        uint4 x[U][NR];
#pragma unroll
        for (int p = 0; p < NR; ++p) {
          const int rk = rot(p + rank_shift, NR);
#pragma unroll
          for (int u = 0; u < U; ++u)
            if (ok[u]) x[u][p] = ld(rk, u);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          acc[u] = inorder_fold_regs<DT, OP, NR, 0, 1, NR>(x[u]);
        }
      } else {
        static_assert(U == 1, "one vector position per thread for wide trees");
        DbtStream<NR> st{P, base, rank_shift, ok[0], {}};
        acc[0] = inorder_fold_stream<DT, OP, NR, 1, NR>(st);
      }
    } else if constexpr (NR <= 8) {
      uint4 x[U][NR];
#pragma unroll
      for (int p = 0; p < NR; ++p) {
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (ok[u]) x[u][p] = ld(p, u);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        acc[u] = tree_fold_regs<DT, OP, NR>(x[u]);
      }
    } else {
      // N = 16, 32, 64: aligned subtrees of 8 ranks, each folded as it
      // arrives and merged with its finished siblings (a binary counter over
      // the subtree index), which is the same balanced tree.  The loads of
      // subtree g + 1 are in flight while subtree g is folded.
      static_assert(U == 1, "one vector position per thread for wide trees");
      constexpr int G = 8;
      uint4 cur[G], nxt[G], stk[4];
      int top = 0;
#pragma unroll
      for (int q = 0; q < G; ++q)
        if (ok[0]) cur[q] = ld_stream(static_cast<const char*>(P[q]) + base);
#pragma unroll
      for (int g = 0; g < NR / G; ++g) {
        asm volatile("" ::: "memory");  // subtree g + 2's loads stay behind this fold
        if (g + 1 < NR / G) {
#pragma unroll
          for (int q = 0; q < G; ++q)
            if (ok[0]) nxt[q] = ld_stream(static_cast<const char*>(P[(g + 1) * G + q]) + base);
        }
        uint4 v = tree_fold_regs<DT, OP, G>(cur);
#pragma unroll
        for (int k = g; k & 1; k >>= 1) v = step_vec<DT, OP>(stk[--top], v);
        stk[top++] = v;
        if (g + 1 < NR / G) {
#pragma unroll
          for (int q = 0; q < G; ++q) cur[q] = nxt[q];
        }
      }
      acc[0] = stk[0];
    }

    if (a.avg) {
#pragma unroll
      for (int u = 0; u < U; ++u) acc[u] = div_vec<DT>(acc[u], a.fn);
    }
    if (a.owner_only || a.to_root) {
      char* dst = static_cast<char*>(const_cast<void*>(P[a.owner_only ? c : a.root])) + base;
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (ok[u]) st_stream(dst + u * kStride, acc[u]);
    } else if constexpr (NR > 0) {
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        char* dst = static_cast<char*>(const_cast<void*>(P[r])) + base;
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (ok[u]) st_stream(dst + u * kStride, acc[u]);
      }
    } else {
      for (int r = 0; r < n; ++r) {
        char* dst = static_cast<char*>(const_cast<void*>(P[r])) + base;
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (ok[u]) st_stream(dst + u * kStride, acc[u]);
      }
    }

    // elements of the segment outside its full vectors
    if (ti == 0 && (int)threadIdx.x < sh.head + sh.tail) {
      const int64_t e = scalar_elem<VEC>(s, sh, threadIdx.x, shift);
      // beyond 8 ranks the fold runs over the table's runtime rank count: a
      // loop unrolled over 32 or 64 ranks would hoist every load and spill
      uint32_t r = fold_scalar<DT, OP, ORDER>(P, NR > 8 ? T.nranks : n, c, e);
      if (a.avg) r = div_word<DT>(r, a.fn);
      if (a.owner_only || a.to_root) {
        st_elem<ES>(const_cast<void*>(P[a.owner_only ? c : a.root]), e, r);
      } else {
        for (int q = 0; q < n; ++q) st_elem<ES>(const_cast<void*>(P[q]), e, r);
      }
    }
  }
}

// ---- host side ---------------------------------------------------------------

// Tiles of `tile_elems` vectors (or elements) per segment; a segment with
// leftover scalars but no full vector still gets one tile.  `shifted`: the
// kernel cuts vectors at the row's shift (row_shift of its first pointer),
// as the fused, gather and step-wise kernels do; the copy kernels do not.
template <class TABLE>
inline int64_t fill_tiles(TABLE& t, int vec, int64_t tile_units, bool shifted = false) {
  int64_t acc = 0;
  for (int i = 0; i < t.nseg; ++i) {
    Seg& s = t.seg[i];
    s.tile_begin = acc;
    int64_t units, extra;
    if (vec > 1) {
      const int sh = shifted ? row_shift(t.ptr[(size_t)s.tensor * t.nranks], 16 / vec) : 0;
      int64_t vb = (s.begin + sh + vec - 1) / vec, ve = (s.end + sh) / vec;
      if (ve < vb) ve = vb;
      units = ve - vb;
      extra = (s.end - s.begin) - units * vec;
    } else {
      units = s.end - s.begin;
      extra = 0;
    }
    int64_t tiles = (units + tile_units - 1) / tile_units;
    if (tiles == 0 && extra > 0) tiles = 1;
    acc += tiles;
  }
  t.ntiles = acc;
  return acc;
}

// Launch with programmatic stream serialization (see pdl_prologue): the
// kernel may begin launching while the one before it on the stream drains.
// Measured back to back on GB300 (bit-identical results): 8 x 128 MiB bf16
// ring 309.3 -> 306.8 us, 8 x 25 MiB f32 AVG 64.6 -> 62.3 us, its AllGather
// 34.9 -> 32.7 us and Broadcast 34.8 -> 32.5 us; a 4 x 16 KiB call replayed
// from a CUDA graph 1.65 -> 1.78 us.
template <typename K, typename ARGS>
inline cudaError_t launch_pdl(K kernel, unsigned grid, unsigned block, cudaStream_t stream, const ARGS& a,
                              size_t smem = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <typename K>
inline int blocks_per_sm(K kernel, int block) {
  int b = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, block, 0) != cudaSuccess || b < 1) b = 1;
  return b;
}

inline unsigned grid_for(int64_t ntiles, int64_t cap = 0) {
  int64_t g = ntiles < kMaxGrid ? ntiles : kMaxGrid;
  if (cap > 0 && g > cap) g = cap;
  return (unsigned)g;
}

template <int DT, int OP, int ORDER, int NR, class ARGS>
cudaError_t launch_fused_vec(ARGS& a, cudaStream_t stream) {
  constexpr int64_t kTile = (int64_t)kFusedBlock * fused_unroll(ORDER, NR);
  if (fill_tiles(a.tab, 16 / ElemSize<DT>::value, kTile, true) == 0) return cudaSuccess;
  count_launch();
  return launch_pdl(fused_vec_kernel<ARGS, DT, OP, ORDER, NR>, grid_for(a.tab.ntiles, a.max_grid), kFusedBlock,
                    stream, a);
}

// Dispatch on order and rank count for one (dtype, op), rows whose buffers
// share their address modulo 16.  Double binary trees of other rank counts
// than these, and rows whose buffers do not, take the staged kernel.
template <int DT, int OP, class ARGS>
cudaError_t launch_fused_typed(int order, ARGS& a, cudaStream_t stream) {
  const int n = a.tab.nranks;
  if (order == DBTREE) {
    switch (n) {
      case 2: return launch_fused_vec<DT, OP, DBTREE, 2>(a, stream);
      case 4: return launch_fused_vec<DT, OP, DBTREE, 4>(a, stream);
      case 8: return launch_fused_vec<DT, OP, DBTREE, 8>(a, stream);
      case 16: return launch_fused_vec<DT, OP, DBTREE, 16>(a, stream);
      case 32: return launch_fused_vec<DT, OP, DBTREE, 32>(a, stream);
      case 64: return launch_fused_vec<DT, OP, DBTREE, 64>(a, stream);
      default: return cudaErrorNotSupported;
    }
  }
  if (order == RING) {
    switch (n) {
      case 2: return launch_fused_vec<DT, OP, RING, 2>(a, stream);
      case 4: return launch_fused_vec<DT, OP, RING, 4>(a, stream);
      case 8: return launch_fused_vec<DT, OP, RING, 8>(a, stream);
      case 16: return launch_fused_vec<DT, OP, RING, 16>(a, stream);
      case 32: return launch_fused_vec<DT, OP, RING, 32>(a, stream);
      case 64: return launch_fused_vec<DT, OP, RING, 64>(a, stream);
      default: return launch_fused_vec<DT, OP, RING, 0>(a, stream);
    }
  }
  switch (n) {
    case 2: return launch_fused_vec<DT, OP, TREE, 2>(a, stream);
    case 4: return launch_fused_vec<DT, OP, TREE, 4>(a, stream);
    case 8: return launch_fused_vec<DT, OP, TREE, 8>(a, stream);
    case 16: return launch_fused_vec<DT, OP, TREE, 16>(a, stream);
    case 32: return launch_fused_vec<DT, OP, TREE, 32>(a, stream);
    case 64: return launch_fused_vec<DT, OP, TREE, 64>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ar

#define AR_DEFINE_FUSED(NAME, DT, OP)                                                              \
  namespace ar {                                                                                  \
  cudaError_t NAME(int order, FusedArgs& a, cudaStream_t s) { return launch_fused_typed<DT, OP>(order, a, s); }      \
  cudaError_t NAME(int order, SmallFusedArgs& a, cudaStream_t s) { return launch_fused_typed<DT, OP>(order, a, s); } \
  }
