// Fused AllReduce / ReduceScatter / Reduce for rows whose rank buffers sit
// at different addresses modulo 16, and double binary trees of the rank
// counts the kernels in ar_fused.cuh are not compiled for: the same fold, in
// the same order, as those kernels, with every rank's words staged in shared
// memory and realigned there.
#pragma once

#include <atomic>

#include "ar_fused.cuh"

namespace ar {

// ---- helpers for rows whose buffers sit at different addresses modulo 16 ------

// Offset of buffer p from the row's first buffer within a 16-byte word.
__device__ __forceinline__ int byte_phase(const void* p, const void* p0) {
  return (int)(((uintptr_t)p - (uintptr_t)p0) & 15);
}

__device__ __forceinline__ uint32_t pick4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, int k) {
  return k < 2 ? (k == 0 ? a0 : a1) : (k == 2 ? a2 : a3);
}

// Bytes [lo, hi) of the aligned 16-byte word at `w` get bytes [lo, hi) of v
// (lo, hi multiples of 2), as naturally aligned 8-, 4- and 2-byte stores.
__device__ __forceinline__ void st_stream_part(char* w, const uint4& v, int lo, int hi) {
  int pos = lo;
  while (pos < hi) {
    const int k = pos >> 2;
    if ((pos & 7) == 0 && pos + 8 <= hi) {
      __stcs(reinterpret_cast<uint2*>(w + pos), make_uint2(pick4(v.x, v.y, v.z, v.w, k), pick4(v.y, v.z, v.w, v.w, k)));
      pos += 8;
    } else if ((pos & 3) == 0 && pos + 4 <= hi) {
      __stcs(reinterpret_cast<unsigned int*>(w + pos), pick4(v.x, v.y, v.z, v.w, k));
      pos += 4;
    } else {
      __stcs(reinterpret_cast<unsigned short*>(w + pos),
             (unsigned short)(pick4(v.x, v.y, v.z, v.w, k) >> ((pos & 2) * 8)));
      pos += 2;
    }
  }
}

// ---- rows whose buffers sit at different addresses modulo 16: staged form ----
//
// The fold of the fused kernel with the realignment done in shared memory.
// A block takes a tile of kStageTileVecs vectors of the row's frame (the
// first buffer's 16-byte grid).  (1) Every thread copies aligned 16-byte
// words of the ranks straight into shared memory (cp.async, no registers),
// rank r's words from the one holding the tile's first byte in buffer r:
// the tile's bytes then sit off_r = (P[r] - P[0]) mod 16 bytes into its
// slot.  One commit group per rank, in the order the fold takes them; up to
// eight ranks each have a slot (4-byte elements: up to five ranks), more
// stream through the slots, a slot refilled as soon as its rank is folded.
// (2) Each thread folds 4-byte words of the frame, kStageBlock apart
// (consecutive threads, consecutive words: no bank conflicts), a rank as
// soon as its copies have landed: word w of rank r is bytes [4w + off_r,
// 4w + off_r + 4) of its slot, two word loads and a funnel shift when off_r
// is 2 mod 4, one load otherwise.
// (3) The results go to shared memory four times, the k-th copy shifted by
// k words, and for 2-byte elements (with eight slots) four more times moved
// by one element, so that the 16-byte words a destination at off = 4k + h
// bytes needs are consecutive entries of one copy.  (4) One bulk copy
// (cp.async.bulk, the tensor-memory-access engine) per destination writes
// its whole words; its first and last word also hold bytes of the
// neighbouring tiles and are written in part by plain stores.  (Rows of 2
// or 4 ranks of 2-byte elements keep four copies, for occupancy, and store
// their 2 mod 4 byte destinations word by word, shifted in registers.)  A
// block reads all its inputs before its first store and writes only its
// tile's bytes, so working in place is safe: bytes of a staged word outside
// the tile are never used.
constexpr int kStageBlock = 256;
constexpr int kStageSlots = 8;
// Rank slots a block holds: one per rank up to eight ranks (but see
// kStageSlotsF32); NR = 0 (a runtime rank count) and more ranks stream
// through eight.  The gather forms
// (AllGather, Broadcast: one owner's words copied to the other ranks; GATHER
// 1 for up to eight ranks, 2 beyond) hold one.
// Rows of 4-byte elements and 6 to 8 ranks stream through five slots: they
// keep four result copies, so the slots set the block's shared memory, and
// five blocks of 41 KB per SM beat three of 66 KB (f32 at four offsets, bit
// for bit the same: 8 x 25 MiB AVG 66.0 -> 63.8 us, 8 x 64 MiB ring 159.2 ->
// 156.2, tree 161.6 -> 155.9; four slots 64.1, 156.3 and 156.8).
constexpr int kStageSlotsF32 = 5;
__host__ __device__ constexpr int stage_slots(int nr, int gather, int es) {
  return gather                                                 ? 1
         : es == 4 && nr > kStageSlotsF32 && nr <= kStageSlots ? kStageSlotsF32
         : nr > 0 && nr < kStageSlots                          ? nr
                                                                : kStageSlots;
}
constexpr int kStageTileVecs = 512;
constexpr int kStageSlotBytes = kStageTileVecs * 16 + 16;          // one rank's staged words
constexpr int kStageCopyBytes = (kStageTileVecs + 2) * 16;         // one shifted copy of the result
__host__ __device__ constexpr int stage_copies(int es, int nr, int gather) {
  return gather == 1 ? 2 : es == 2 && (gather == 2 || stage_slots(nr, gather, es) == kStageSlots) ? 8 : 4;
}
// Gather form 1 keeps its slot and two copy buffers apart (it builds one
// destination's copy while the bulk copy of the previous one reads the
// other); the other forms reuse the slots for the copies.
__host__ __device__ constexpr int stage_smem_bytes(int nr, int es, int gather) {
  return gather == 1 ? kStageSlotBytes + 2 * kStageCopyBytes
         : stage_slots(nr, gather, es) * kStageSlotBytes > stage_copies(es, nr, gather) * kStageCopyBytes
             ? stage_slots(nr, gather, es) * kStageSlotBytes
             : stage_copies(es, nr, gather) * kStageCopyBytes;
}
// Resident blocks per SM: as many as shared memory allows, since the tiles
// in flight are what keeps HBM busy (three at 66 KB, six at 33 KB with 40
// registers and no spills; the gather form eight at 25 KB; 5-, 6- and 7-rank
// rings of 2-byte elements five, four and three; 4-byte elements of 6 to 8
// ranks five).  Measured, 2-byte elements at eight offsets:
// 4 x 128 MiB 162.8 / 158.5 / 157.5 us and 2 x 128 MiB 98.1 / 89.3 / 83.9 us
// at four / five / six blocks; 8 x 128 MiB 446.7 us at two, 351.4 at three
// (before the bulk stores).
__host__ __device__ constexpr int stage_min_blocks(int nr, int es, int gather) {
  // what an SM's 228 KB of shared memory (1 KB reserved per block) holds,
  // at most 8 for the gather form and 6 for the folds
  return (gather == 1 ? 8 : 6) < 233472 / (stage_smem_bytes(nr, es, gather) + 1024)
             ? (gather == 1 ? 8 : 6)
             : 233472 / (stage_smem_bytes(nr, es, gather) + 1024);
}

// The double binary tree's in-order fold (see inorder_root) over G groups
// of words at once: positions LO..HI in increasing order, `take(p, v)`
// handing over position p + 1's words when they have landed.
template <int DT, int OP, int G, int LO, int HI, class TAKE>
__device__ __forceinline__ void stage_inorder(uint4 (&acc)[G], TAKE& take) {
  constexpr int R = inorder_root(LO, HI);
  if constexpr (LO < R) {
    stage_inorder<DT, OP, G, LO, R - 1>(acc, take);
    uint4 own[G];
    take(R - 1, own);
#pragma unroll
    for (int j = 0; j < G; ++j) acc[j] = step_vec<DT, OP>(acc[j], own[j]);
  } else {
    take(R - 1, acc);
  }
  if constexpr (R < HI) {
    uint4 right[G];
    stage_inorder<DT, OP, G, R + 1, HI>(right, take);
#pragma unroll
    for (int j = 0; j < G; ++j) acc[j] = step_vec<DT, OP>(acc[j], right[j]);
  }
}

// NR: 2, 4, 8, 16, 32 or 64 ranks (rings and trees), 2 to 8, 16 or 32
// (double binary trees), 3, 5, 6 or 7 (rings), 0 = the table's rank count
// (rings and double binary trees).  The double binary tree's unrolled fold
// beats the run-time one up to 32 ranks and loses at 64 (bf16 at eight
// offsets: 16 x 32 MiB 161.5 against 216.8 us, 32 x 16 MiB f32 164.9
// against 186.3, 64 x 8 MiB 262.7 against 223.1).  Every order folds the ranks in increasing position order, so
// each is folded as soon as its copies have landed.  GATHER: no fold, the
// segment's owner (its chunk id) is copied to every other rank, a copy built
// per destination in turn (1: up to eight ranks, whose phases seldom
// repeat) or all eight phases at once (2: more ranks).
template <class ARGS, int DT, int OP, int ORDER, int NR, int GATHER>
__global__ void __launch_bounds__(kStageBlock, stage_min_blocks(NR, ElemSize<DT>::value, GATHER))
    fused_stage_kernel(const __grid_constant__ ARGS a) {
  constexpr int ES = ElemSize<DT>::value;
  constexpr int VEC = 16 / ES;
  constexpr int TV = kStageTileVecs;
  constexpr int G = TV * 4 / kStageBlock / 4;  // groups of 4 frame words per thread
  static_assert(G * 4 * kStageBlock == TV * 4, "tile is a whole number of word groups");
  constexpr int NS = stage_slots(NR, GATHER, ES);
  constexpr bool kStream = !GATHER && (NR == 0 || NR > NS);  // ranks stream through the slots
  static_assert(NR == 0 ? ORDER == RING || ORDER == DBTREE
                        : NR <= 64 && ((NR & (NR - 1)) == 0 || ORDER == RING || (ORDER == DBTREE && NR < kStageSlots)),
                "no staged form");
  constexpr bool kHalfCopies = stage_copies(ES, NR, GATHER) == 8;
  extern __shared__ __align__(16) unsigned char S[];
  pdl_prologue();
  const auto& T = a.tab;
  const int n = NR > 0 ? NR : T.nranks;
  const int tid = threadIdx.x;
  const int lane = tid & 31;

  for (int64_t tile = blockIdx.x; tile < T.ntiles; tile += gridDim.x) {
    const Seg& s = T.seg[find_seg(T, tile)];
    const void* const* P = T.ptr + (size_t)s.tensor * n;
    const int shift = row_shift(P[0], ES);
    const SegShape sh = seg_shape<VEC>(s, shift);
    const int64_t ti = tile - s.tile_begin;
    const int c = s.chunk;
    const int64_t t0 = sh.vb + ti * TV;
    const int nv = (int)(sh.ve - t0 < TV ? sh.ve - t0 : TV);  // vectors in this tile (<= 0: scalars only)
    const int64_t base = t0 * 16 - shift * ES;                 // vector t0 in every buffer, aligned in P[0]

    if (nv > 0) {
      // (1) the rank at fold position p, its aligned words [0, nv + (off != 0))
      // into slot p (mod the slot count), one commit group each
      const int rank_shift = ORDER == DBTREE && c != 0 ? 1 : 0;
      auto rank_at = [&](int p) -> int {
        if constexpr (GATHER) return c;
        else if constexpr (ORDER == RING) return rot(c + 1 + p, n);
        else if constexpr (ORDER == DBTREE) return rot(p + rank_shift, n);
        else return p;
      };
      auto slot = [&](int p) -> unsigned char* { return S + (p % NS) * kStageSlotBytes; };
      auto issue = [&](int p) {
        const int r = rank_at(p);
        const int off = byte_phase(P[r], P[0]);
        const char* g = static_cast<const char*>(P[r]) + base - off;
        const int nw = nv + (off != 0);
        unsigned char* d = slot(p);
        for (int i = tid; i < nw; i += kStageBlock) cp_async16(d + i * 16, g + i * 16);
        cp_async_commit();
      };
      if constexpr (GATHER) {
        issue(0);
      } else if constexpr (kStream) {
        const int first = n < NS ? n : NS;
        for (int p = 0; p < first; ++p) issue(p);
      } else {
#pragma unroll
        for (int p = 0; p < NR; ++p) issue(p);
      }

      // (2) fold frame words w = tid + (4j + k) * kStageBlock, k = 0..3, of group j
      auto group = [&](int p, int j) -> uint4 {
        const int off = byte_phase(P[rank_at(p)], P[0]);
        const uint32_t* sl = reinterpret_cast<const uint32_t*>(slot(p)) + (off >> 2) + tid + 4 * j * kStageBlock;
        auto word = [&](int q) -> uint32_t {
          if constexpr (ES == 4) return sl[q * kStageBlock];
          else return __funnelshift_r(sl[q * kStageBlock], sl[q * kStageBlock + 1], (uint32_t)(off & 2) * 8);
        };
        return make_uint4(word(0), word(1), word(2), word(3));
      };
      uint4 res[G];
      // copies allowed in flight when position p is needed: those issued
      // after it (streaming: up to p + NS - 2, a slot being refilled one
      // step late, after the next position's barrier)
      auto later_than = [&](int p) -> int {
        int later = n - 1 - p;
        if (kStream && p > 0 && later > NS - 2) later = NS - 2;
        if (kStream && p == 0 && later > NS - 1) later = NS - 1;
        return later;
      };
      if constexpr (GATHER) {
        cp_async_wait_all();
        __syncthreads();
#pragma unroll
        for (int j = 0; j < G; ++j) res[j] = group(0, j);
      } else if constexpr (ORDER == DBTREE && NR > 0) {
        // the in-order tree visits positions in increasing order too
        auto take = [&](int p, uint4 (&v)[G]) {
          cp_async_wait_pending(later_than(p));
          __syncthreads();  // position p has landed; every thread has folded position p - 1
          if (kStream && p > 0 && p - 1 + NS < n) issue(p - 1 + NS);
#pragma unroll
          for (int j = 0; j < G; ++j) v[j] = group(p, j);
        };
        stage_inorder<DT, OP, G, 1, (NR > 0 ? NR : 1)>(res, take);
      } else {
        // rank p is folded as soon as its copies have landed, while the
        // later ranks' copies are still in flight; the tree keeps finished
        // subtrees on a stack (a binary counter over the rank index), which
        // is the same balanced pairwise tree
        auto arrive = [&](int p) {
          cp_async_wait_pending(later_than(p));
          __syncthreads();  // rank p has landed; every thread has folded rank p - 1
          // streaming: rank p - 1's slot is free, refill it
          if (kStream && p > 0 && p - 1 + NS < n) issue(p - 1 + NS);
        };
        // 64-rank trees fold subtrees of 8 in a loop (below); measured on
        // bf16 at eight offsets, 64 x 8 MiB 244.9 -> 200.2 us, while 16 x 32
        // MiB (164.6 -> 171.7) and 32 x 16 MiB f32 (168.3 -> 179.6) were
        // faster fully unrolled
        constexpr bool kWideTree = ORDER == TREE && NR == 64;
        // entries the counter holds: log2 of the ranks it counts over
        constexpr int kDepth = ORDER == RING ? 1 : kWideTree || NR <= 16 ? 4 : NR == 32 ? 5 : 6;
        uint4 stk[G][kDepth];
        int top = 0;
        // pos: the rank's place in its subtree (p itself up to 8 ranks)
        auto fold = [&](int p, int pos) {
          arrive(p);
#pragma unroll
          for (int j = 0; j < G; ++j) {
            uint4 v = group(p, j);
            if constexpr (ORDER == RING) {
              stk[j][0] = p == 0 ? v : step_vec<DT, OP>(stk[j][0], v);
            } else {
              int t = top;
#pragma unroll
              for (int k = pos; k & 1; k >>= 1) v = step_vec<DT, OP>(stk[j][--t], v);
              stk[j][t] = v;
            }
          }
          if constexpr (ORDER != RING) {
            for (int k = pos; k & 1; k >>= 1) --top;
            ++top;
          }
        };
        if constexpr (ORDER == DBTREE) {
          // a rank count known at run time.  In the in-order tree over
          // positions 1..n (see inorder_root) position q sits at level
          // tz(q): odd positions are leaves, and node q of level l >= 1 has
          // the 2^l - 1 positions before it as its left subtree.  A leaf
          // completes at once and, while the subtree it completes is a right
          // child (the bits of q above bit 0 are ones), completes its parent
          // too, whose held value takes it in.  Node q of level l >= 1 holds
          // (its left subtree) (+) x_q until then.  Subtrees whose parent
          // would lie past n fold in at the end, right-nested from the
          // lowest open level up.  Every index into `hold` is a constant.
          constexpr int kLevels = 6;  // 64 positions: levels 1..6
          static_assert((1 << kLevels) >= kMaxRanks && (1 << kLevels) < 2 * kMaxRanks, "a level per bit of q");
          uint4 hold[kLevels][G], cur[G];
          unsigned open = 0;  // bit l: node of level l holding
          bool pend = false;  // cur: a finished subtree waiting for its parent
#pragma unroll 1
          for (int p = 0; p < n; ++p) {
            arrive(p);
            const unsigned q = p + 1;
            if (q & 1) {
              const int casc = __ffs(~(q >> 1)) - 1;  // levels of the parents it completes
#pragma unroll
              for (int j = 0; j < G; ++j) cur[j] = group(p, j);
              // a uniform early exit, not predication: 12-64 ranks 2-3% faster
#pragma unroll
              for (int l = 1; l <= kLevels; ++l) {
                if (l > casc) break;
#pragma unroll
                for (int j = 0; j < G; ++j) cur[j] = step_vec<DT, OP>(hold[l - 1][j], cur[j]);
              }
              open &= ~((2u << casc) - 2u);
              pend = true;
            } else {
              const int t = __ffs(q) - 1;
              uint4 v[G];
#pragma unroll
              for (int j = 0; j < G; ++j) v[j] = step_vec<DT, OP>(cur[j], group(p, j));
#pragma unroll
              for (int l = 1; l <= kLevels; ++l)
                if (l == t) {
#pragma unroll
                  for (int j = 0; j < G; ++j) hold[l - 1][j] = v[j];
                }
              open |= 1u << t;
              pend = false;
            }
          }
#pragma unroll
          for (int l = 1; l <= kLevels; ++l)
            if (open & (1u << l)) {
#pragma unroll
              for (int j = 0; j < G; ++j) cur[j] = pend ? step_vec<DT, OP>(hold[l - 1][j], cur[j]) : hold[l - 1][j];
              pend = true;
            }
#pragma unroll
          for (int j = 0; j < G; ++j) res[j] = cur[j];
        } else if constexpr (kWideTree) {
          // subtrees of 8 consecutive ranks, each folded by the unrolled
          // counter above, merged by a counter over the subtree index in a
          // loop that is not unrolled (unrolled over 64 ranks the kernel is
          // much larger and slower)
          uint4 done[G][3];
#pragma unroll 1
          for (int g = 0; g < NR / kStageSlots; ++g) {
            top = 0;
#pragma unroll
            for (int q = 0; q < kStageSlots; ++q) fold(q + kStageSlots * g, q);
            int t = 0;
            for (int k = g; k & 1; k >>= 1) ++t;  // subtrees merged now
            const int base_top = __popc(g) - t;  // finished subtrees below them
#pragma unroll
            for (int j = 0; j < G; ++j) {
              uint4 v = stk[j][0];
              for (int k = 0; k < t; ++k) v = step_vec<DT, OP>(done[j][base_top + t - 1 - k], v);
              done[j][base_top] = v;
            }
          }
#pragma unroll
          for (int j = 0; j < G; ++j) res[j] = done[j][0];
        } else if constexpr (NR > 0) {
#pragma unroll
          for (int p = 0; p < NR; ++p) fold(p, p);
#pragma unroll
          for (int j = 0; j < G; ++j) res[j] = stk[j][0];
        } else {
#pragma unroll 1
          for (int p = 0; p < n; ++p) fold(p, p);
#pragma unroll
          for (int j = 0; j < G; ++j) res[j] = stk[j][0];
        }
      }
      if (a.avg) {
#pragma unroll
        for (int j = 0; j < G; ++j) res[j] = div_vec<DT>(res[j], a.fn);
      }
      __syncthreads();  // every slot has been read

      if constexpr (GATHER == 1) {
        // (3+4) per destination: a copy of the owner's words in its phase
        // (word m at index m + k + 4, for h = 2 the stream one element
        // earlier), built while the bulk copy of the destination before
        // reads the other buffer
        const int offc = byte_phase(P[c], P[0]);
        const uint32_t* own = reinterpret_cast<const uint32_t*>(S) + (offc >> 2);  // the staged slot
        int idx = 0;
#pragma unroll 1
        for (int r = 0; r < n; ++r) {
          if (r == c) continue;
          const int off = byte_phase(P[r], P[0]);
          const int k = off >> 2;
          const bool h = ES == 2 && (off & 2);
          uint32_t* cw = reinterpret_cast<uint32_t*>(S + kStageSlotBytes + (idx & 1) * kStageCopyBytes);
          if (idx >= 2) {
            if (tid == 0) bulk_wait_read_but_one();  // the buffer's previous bulk copy has read it
            __syncthreads();
          }
#pragma unroll
          for (int j = 0; j < G; ++j) {
            const uint32_t f[4] = {res[j].x, res[j].y, res[j].z, res[j].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int m = tid + (4 * j + q) * kStageBlock;
              uint32_t v = f[q];
              if (h) {
                uint32_t below = __shfl_up_sync(0xffffffffu, f[q], 1);
                if (lane == 0 && m > 0) {
                  below = own[m - 1];
                  if constexpr (ES == 2) below = __funnelshift_r(below, own[m], (uint32_t)(offc & 2) * 8);
                }
                v = __funnelshift_l(below, f[q], 16);
              }
              cw[k + 4 + m] = v;
            }
          }
          if (h && tid == kStageBlock - 1) cw[k + 4 + 4 * TV] = __funnelshift_l(res[G - 1].w, 0u, 16);
          fence_proxy_async_shared();
          __syncthreads();
          const uint4* cp = reinterpret_cast<const uint4*>(cw);
          char* g = static_cast<char*>(const_cast<void*>(P[r])) + base - off;
          const int lo = off != 0;
          if (tid == 0 && nv > lo) bulk_store(g + 16 * lo, cp + lo + 1, 16 * (nv - lo));
          if (off != 0 && tid == 32) st_stream_part(g, cp[1], off, 16);
          if (off != 0 && tid == 64) st_stream_part(g + 16 * (int64_t)nv, cp[nv + 1], 0, off);
          if (tid == 0) bulk_commit();
          ++idx;
        }
      } else {
      // (3) copy k holds frame word m at word index m + k + 4
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t* cp = reinterpret_cast<uint32_t*>(S + k * kStageCopyBytes) + k + 4 + tid;
#pragma unroll
        for (int j = 0; j < G; ++j) {
          cp[(4 * j + 0) * kStageBlock] = res[j].x;
          cp[(4 * j + 1) * kStageBlock] = res[j].y;
          cp[(4 * j + 2) * kStageBlock] = res[j].z;
          cp[(4 * j + 3) * kStageBlock] = res[j].w;
        }
      }
      if constexpr (kHalfCopies) {
        // copies 4..7 the same for the stream one element earlier: its word
        // m is the last element of frame word m - 1 and the first of word m
        __syncthreads();  // lane 0 reads the word below from copy 0
        const uint32_t* c0 = reinterpret_cast<const uint32_t*>(S) + 4 + tid;
#pragma unroll
        for (int j = 0; j < G; ++j) {
          uint32_t f[4] = {res[j].x, res[j].y, res[j].z, res[j].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int m_off = (4 * j + q) * kStageBlock;  // this thread's word m = tid + m_off
            uint32_t below = __shfl_up_sync(0xffffffffu, f[q], 1);
            if (lane == 0) below = c0[m_off - 1];
            const uint32_t h = __funnelshift_l(below, f[q], 16);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              reinterpret_cast<uint32_t*>(S + (4 + k) * kStageCopyBytes)[k + 4 + tid + m_off] = h;
          }
        }
        // one word past the tile: a full tile's last destination word starts
        // with the last element of its last frame word
        if (tid == kStageBlock - 1) {
          const uint32_t h = __funnelshift_l(res[G - 1].w, 0u, 16);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            reinterpret_cast<uint32_t*>(S + (4 + k) * kStageCopyBytes)[k + 4 + 4 * TV] = h;
        }
      }
      fence_proxy_async_shared();  // the bulk copies read them through the async proxy
      __syncthreads();

      // (4) destination word i of rank r: bytes [16i, 16i + 16) from the
      // aligned word holding the tile's first byte, i.e. frame bytes
      // [16i - off, 16i + 16 - off): words 4i - k .. 4i - k + 3 (entry i + 1
      // of copy k) and, for h = 2, word 4i - k - 1 (entry i of copy k, .w)
      auto put = [&](int r) {
        const int off = byte_phase(P[r], P[0]);
        const int k = off >> 2;
        const uint32_t hs = (uint32_t)(off & 2) * 8;
        const uint4* cp = reinterpret_cast<const uint4*>(S + ((kHalfCopies && hs ? 4 : 0) + k) * kStageCopyBytes);
        char* g = static_cast<char*>(const_cast<void*>(P[r])) + base - off;
        const int nw = nv + (off != 0);
        if (ES == 4 || hs == 0 || kHalfCopies) {
          // destination word i is entry i + 1 of the copy: its whole words
          // leave in one bulk copy, the two partial words by plain stores
          const int lo = off != 0;
          if (tid == 0 && nv > lo) bulk_store(g + 16 * lo, cp + lo + 1, 16 * (nv - lo));
          if (off != 0 && tid == 32) st_stream_part(g, cp[1], off, 16);
          if (off != 0 && tid == 64) st_stream_part(g + 16 * (int64_t)nv, cp[nv + 1], 0, off);
          return;
        }
        if constexpr (ES == 2 && !kHalfCopies) {  // 2 mod 4 bytes off: each word shifted by one element
          for (int i0 = tid - lane; i0 < nw; i0 += kStageBlock) {  // whole warps: the shuffle needs every lane
            const int i = i0 + lane;
            const int ic = i < TV ? i : TV;  // lanes past the end read an entry that exists and store nothing
            const uint4 cur = cp[ic + 1];
            uint32_t prev = __shfl_up_sync(0xffffffffu, cur.w, 1);
            if (lane == 0) prev = cp[ic].w;
            const uint4 v = make_uint4(__funnelshift_l(prev, cur.x, 16), __funnelshift_l(cur.x, cur.y, 16),
                                       __funnelshift_l(cur.y, cur.z, 16), __funnelshift_l(cur.z, cur.w, 16));
            if (i >= nw) continue;
            if (i == 0) st_stream_part(g, v, off, 16);
            else if (i == nv) st_stream_part(g + 16 * (int64_t)i, v, 0, off);
            else st_stream(g + 16 * (int64_t)i, v);
          }
        }
      };
      if constexpr (GATHER == 2) {
#pragma unroll 1
        for (int r = 0; r < n; ++r)
          if (r != c) put(r);
      } else if (a.owner_only || a.to_root) {
        put(a.owner_only ? c : a.root);
      } else if constexpr (NR > 0 && NR <= kStageSlots) {
#pragma unroll
        for (int r = 0; r < NR; ++r) put(r);
      } else {
#pragma unroll 1
        for (int r = 0; r < n; ++r) put(r);
      }
      if (tid == 0) bulk_commit();
      }
    }

    // elements of the segment outside its full vectors
    if (ti == 0 && tid < sh.head + sh.tail) {
      const int64_t e = scalar_elem<VEC>(s, sh, tid, shift);
      if constexpr (GATHER) {
        const uint32_t v = ld_elem<ES>(P[c], e);
        for (int q = 0; q < n; ++q)
          if (q != c) st_elem<ES>(const_cast<void*>(P[q]), e, v);
      } else {
        uint32_t r = fold_scalar<DT, OP, ORDER>(P, n, c, e);
        if (a.avg) r = div_word<DT>(r, a.fn);
        if (a.owner_only || a.to_root) {
          st_elem<ES>(const_cast<void*>(P[a.owner_only ? c : a.root]), e, r);
        } else {
          for (int q = 0; q < n; ++q) st_elem<ES>(const_cast<void*>(P[q]), e, r);
        }
      }
    }
    // the next tile's copies overwrite shared memory every thread and every
    // bulk copy has finished reading
    if (tile + gridDim.x < T.ntiles) {
      if (tid == 0) bulk_wait_read();
      __syncthreads();
    }
  }
  if (tid == 0) bulk_wait_all();
}

template <int DT, int OP, int ORDER, int NR, int GATHER = 0, class ARGS>
cudaError_t launch_fused_stage(ARGS& a, cudaStream_t stream) {
  constexpr int kSmem = stage_smem_bytes(NR, ElemSize<DT>::value, GATHER);
  auto kernel = fused_stage_kernel<ARGS, DT, OP, ORDER, NR, GATHER>;
  // opened once per context to the shared memory the kernel uses
  static std::atomic<unsigned long long> opened[256];
  cudaError_t e = open_kernel(reinterpret_cast<const void*>(kernel), kSmem, false, opened);
  if (e != cudaSuccess) return e;
  if (fill_tiles(a.tab, 16 / ElemSize<DT>::value, kStageTileVecs, true) == 0) return cudaSuccess;
  count_launch();
  return launch_pdl(kernel, grid_for(a.tab.ntiles, a.max_grid), kStageBlock, stream, a, (size_t)kSmem);
}

// The staged kernel for one (dtype, op): every order and rank count the
// order takes (trees: powers of two up to 64).  cudaErrorNotSupported for
// any other.
template <int DT, int OP, class ARGS>
cudaError_t launch_stage_typed(int order, ARGS& a, cudaStream_t stream) {
  const int n = a.tab.nranks;
  switch (order * 100 + n) {
    case RING * 100 + 2: return launch_fused_stage<DT, OP, RING, 2>(a, stream);
    case RING * 100 + 3: return launch_fused_stage<DT, OP, RING, 3>(a, stream);
    case RING * 100 + 4: return launch_fused_stage<DT, OP, RING, 4>(a, stream);
    case RING * 100 + 5: return launch_fused_stage<DT, OP, RING, 5>(a, stream);
    case RING * 100 + 6: return launch_fused_stage<DT, OP, RING, 6>(a, stream);
    case RING * 100 + 7: return launch_fused_stage<DT, OP, RING, 7>(a, stream);
    case RING * 100 + 8: return launch_fused_stage<DT, OP, RING, 8>(a, stream);
    case TREE * 100 + 2: return launch_fused_stage<DT, OP, TREE, 2>(a, stream);
    case TREE * 100 + 4: return launch_fused_stage<DT, OP, TREE, 4>(a, stream);
    case TREE * 100 + 8: return launch_fused_stage<DT, OP, TREE, 8>(a, stream);
    case TREE * 100 + 16: return launch_fused_stage<DT, OP, TREE, 16>(a, stream);
    case TREE * 100 + 32: return launch_fused_stage<DT, OP, TREE, 32>(a, stream);
    case TREE * 100 + 64: return launch_fused_stage<DT, OP, TREE, 64>(a, stream);
    case DBTREE * 100 + 2: return launch_fused_stage<DT, OP, DBTREE, 2>(a, stream);
    case DBTREE * 100 + 3: return launch_fused_stage<DT, OP, DBTREE, 3>(a, stream);
    case DBTREE * 100 + 4: return launch_fused_stage<DT, OP, DBTREE, 4>(a, stream);
    case DBTREE * 100 + 5: return launch_fused_stage<DT, OP, DBTREE, 5>(a, stream);
    case DBTREE * 100 + 6: return launch_fused_stage<DT, OP, DBTREE, 6>(a, stream);
    case DBTREE * 100 + 7: return launch_fused_stage<DT, OP, DBTREE, 7>(a, stream);
    case DBTREE * 100 + 8: return launch_fused_stage<DT, OP, DBTREE, 8>(a, stream);
    case DBTREE * 100 + 16: return launch_fused_stage<DT, OP, DBTREE, 16>(a, stream);
    case DBTREE * 100 + 32: return launch_fused_stage<DT, OP, DBTREE, 32>(a, stream);
    default: break;
  }
  if (order == RING) return launch_fused_stage<DT, OP, RING, 0>(a, stream);
  if (order == DBTREE) return launch_fused_stage<DT, OP, DBTREE, 0>(a, stream);
  return cudaErrorNotSupported;
}

}  // namespace ar

// AllGather / Broadcast of rows whose buffers sit at different addresses
// modulo 16 (element size of DT; the table's chunk ids name the owners).
#define AR_DEFINE_STAGE_GATHER(NAME, DT)                                                            \
  namespace ar {                                                                                      \
  cudaError_t NAME(FusedArgs& a, cudaStream_t s) {                                                    \
    return a.tab.nranks <= kStageSlots ? launch_fused_stage<DT, SUM, RING, 0, 1>(a, s)                \
                                       : launch_fused_stage<DT, SUM, RING, 0, 2>(a, s);               \
  }                                                                                                   \
  }

#define AR_DEFINE_STAGE(NAME, DT, OP)                                                                \
  namespace ar {                                                                                      \
  cudaError_t NAME(int order, FusedArgs& a, cudaStream_t s) { return launch_stage_typed<DT, OP>(order, a, s); } \
  cudaError_t NAME(int order, SmallFusedArgs& a, cudaStream_t s) { return launch_stage_typed<DT, OP>(order, a, s); } \
  }
