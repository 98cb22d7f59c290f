// Copy kernels (fused AllGather, bucket pack/unpack) and the fused-kernel
// dispatcher.
#include "ar_stage.cuh"

namespace ar {

// ---- fused AllGather ---------------------------------------------------------
// AllGather forwards finished chunks with no arithmetic ("AllReduce" concept
// page §3; "Allreduce：大模型分布式训练的核心通信算法与优化实践" §2.2 第二阶段):
// after N-1 forwarding steps every rank holds every owner's chunk bit for bit.
// One pass: read chunk c of its owner c once, write it to the N-1 others.

// Two 16-byte positions per thread and 4 resident blocks per SM (64
// registers): 1-4% faster alone than four positions without the cap.
constexpr int kGatherUnroll = 2;

// Rows whose buffers share their address modulo 16: 16-byte vectors cut at
// that offset, the segment's scalar ends one element per thread.
template <int ES>
__global__ void __launch_bounds__(kFusedBlock, 4) gather_kernel(const __grid_constant__ SegTable T) {
  constexpr int VEC = 16 / ES;
  constexpr int TILE = kFusedBlock * kGatherUnroll;
  pdl_prologue();
  const int n = T.nranks;
  for (int64_t tile = blockIdx.x; tile < T.ntiles; tile += gridDim.x) {
    const Seg& s = T.seg[find_seg(T, tile)];
    const int c = s.chunk;
    const void* const* P = T.ptr + (size_t)s.tensor * n;
    const char* src = static_cast<const char*>(P[c]);
    const int64_t ti = tile - s.tile_begin;
    const int shift = row_shift(P[0], ES);  // the row's buffers share it
    const SegShape sh = seg_shape<VEC>(s, shift);
    uint4 x[kGatherUnroll];
    int64_t off[kGatherUnroll];
    bool ok[kGatherUnroll];
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {
      const int64_t v = sh.vb + ti * TILE + u * kFusedBlock + threadIdx.x;
      ok[u] = v < sh.ve;
      off[u] = v * 16 - shift * ES;
      if (ok[u]) x[u] = ld_stream(src + off[u]);
    }
    for (int r = 0; r < n; ++r) {
      if (r == c) continue;
      char* dst = static_cast<char*>(const_cast<void*>(P[r]));
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u)
        if (ok[u]) st_stream(dst + off[u], x[u]);
    }
    if (ti == 0 && (int)threadIdx.x < sh.head + sh.tail) {
      const int64_t e = scalar_elem<VEC>(s, sh, threadIdx.x, shift);
      const uint32_t v = ld_elem<ES>(src, e);
      for (int r = 0; r < n; ++r)
        if (r != c) st_elem<ES>(const_cast<void*>(P[r]), e, v);
    }
  }
}

template <int ES>
static cudaError_t launch_gather_typed(SegTable& t, cudaStream_t stream) {
  if (fill_tiles(t, 16 / ES, (int64_t)kFusedBlock * kGatherUnroll, true) == 0) return cudaSuccess;
  count_launch();
  return launch_pdl(gather_kernel<ES>, grid_for(t.ntiles), kFusedBlock, stream, t);
}

cudaError_t launch_stage_gather4(FusedArgs&, cudaStream_t);
cudaError_t launch_stage_gather2(FusedArgs&, cudaStream_t);

// Rows whose buffers share their address modulo 16 take the vector copy
// kernel; the others the staged kernel's gather form (the owner's words
// staged in shared memory, each destination written by bulk copies at its
// own offset).
cudaError_t launch_gather(int esize, bool vec, SegTable& t, cudaStream_t s) {
  if (vec) return esize == 2 ? launch_gather_typed<2>(t, s) : launch_gather_typed<4>(t, s);
  FusedArgs a;
  a.tab = t;
  a.avg = 0;
  a.owner_only = 0;
  a.to_root = 0;
  a.root = 0;
  a.max_grid = 0;
  a.fn = 1.0f;
  return esize == 2 ? launch_stage_gather2(a, s) : launch_stage_gather4(a, s);
}

// ---- bucket pack / unpack ----------------------------------------------------
// The literal DDP path copies every rank's gradients into one flat bucket
// buffer per rank before the AllReduce and back afterwards ("Allreduce：..."
// §4.1; "AllReduce 集合通信" §DDP 梯度同步中的地位).  One segment per tensor;
// seg.aux is the tensor's element offset in the packed buffer; seg.chunk = 1
// marks a segment whose both sides are 16-byte aligned for every rank.

constexpr int kCopyUnroll = 2;

template <int ES>
__device__ __forceinline__ void copy_elems(char* dst, const char* src, int64_t e0, int cnt) {
  for (int i = 0; i < cnt; ++i) st_elem<ES>(dst, e0 + i, ld_elem<ES>(src, e0 + i));
}

template <int ES>
__global__ void __launch_bounds__(kFusedBlock) copy_kernel(const __grid_constant__ CopyArgs a) {
  constexpr int VEC = 16 / ES;
  constexpr int TILE = kFusedBlock * kCopyUnroll;
  pdl_prologue();
  const SegTable& T = a.tab;
  const int n = T.nranks;
  for (int64_t tile = blockIdx.x; tile < T.ntiles; tile += gridDim.x) {
    const Seg& s = T.seg[find_seg(T, tile)];
    const SegShape sh = seg_shape<VEC>(s);
    const int64_t ti = tile - s.tile_begin;
    const bool vec = s.chunk != 0;
    for (int r = 0; r < n; ++r) {
      // element e of the tensor sits at element (aux + e) of the packed side
      const char* tens = static_cast<const char*>(T.ptr[(size_t)s.tensor * n + r]);
      const char* pack = static_cast<const char*>(a.packed[r]) + s.aux * ES;
      const char* src = a.to_packed ? tens : pack;
      char* dst = const_cast<char*>(a.to_packed ? pack : tens);
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t v = sh.vb + ti * TILE + u * kFusedBlock + threadIdx.x;
        if (v >= sh.ve) continue;
        if (vec) st_stream(dst + v * 16, ld_stream(src + v * 16));
        else copy_elems<ES>(dst, src, v * VEC, VEC);
      }
      if (ti == 0 && (int)threadIdx.x < sh.head + sh.tail) {
        const int64_t e = scalar_elem<VEC>(s, sh, threadIdx.x);
        copy_elems<ES>(dst, src, e, 1);
      }
    }
  }
}

cudaError_t launch_copy(CopyArgs& a, cudaStream_t stream) {
  const int es = a.esize;
  if (fill_tiles(a.tab, 16 / es, (int64_t)kFusedBlock * kCopyUnroll) == 0) return cudaSuccess;
  count_launch();
  if (es == 2) return launch_pdl(copy_kernel<2>, grid_for(a.tab.ntiles), kFusedBlock, stream, a);
  return launch_pdl(copy_kernel<4>, grid_for(a.tab.ntiles), kFusedBlock, stream, a);
}

// ---- fused dispatch ----------------------------------------------------------

cudaError_t launch_fused_f32_sum(int, FusedArgs&, cudaStream_t);
cudaError_t launch_fused_f32_max(int, FusedArgs&, cudaStream_t);
cudaError_t launch_fused_bf16_sum(int, FusedArgs&, cudaStream_t);
cudaError_t launch_fused_bf16_max(int, FusedArgs&, cudaStream_t);
cudaError_t launch_fused_i32_sum(int, FusedArgs&, cudaStream_t);
cudaError_t launch_fused_i32_max(int, FusedArgs&, cudaStream_t);
cudaError_t launch_fused_f32_sum(int, SmallFusedArgs&, cudaStream_t);
cudaError_t launch_fused_f32_max(int, SmallFusedArgs&, cudaStream_t);
cudaError_t launch_fused_bf16_sum(int, SmallFusedArgs&, cudaStream_t);
cudaError_t launch_fused_bf16_max(int, SmallFusedArgs&, cudaStream_t);
cudaError_t launch_fused_i32_sum(int, SmallFusedArgs&, cudaStream_t);
cudaError_t launch_fused_i32_max(int, SmallFusedArgs&, cudaStream_t);
cudaError_t launch_fused_f16_sum(int, FusedArgs&, cudaStream_t);
cudaError_t launch_fused_f16_max(int, FusedArgs&, cudaStream_t);
cudaError_t launch_fused_f16_sum(int, SmallFusedArgs&, cudaStream_t);
cudaError_t launch_fused_f16_max(int, SmallFusedArgs&, cudaStream_t);

#define AR_DECLARE_STAGE(NAME)                           \
  cudaError_t NAME(int, FusedArgs&, cudaStream_t);       \
  cudaError_t NAME(int, SmallFusedArgs&, cudaStream_t);
AR_DECLARE_STAGE(launch_stage_f32_sum)
AR_DECLARE_STAGE(launch_stage_f32_max)
AR_DECLARE_STAGE(launch_stage_bf16_sum)
AR_DECLARE_STAGE(launch_stage_bf16_max)
AR_DECLARE_STAGE(launch_stage_f16_sum)
AR_DECLARE_STAGE(launch_stage_f16_max)
AR_DECLARE_STAGE(launch_stage_i32_sum)
AR_DECLARE_STAGE(launch_stage_i32_max)

template <class ARGS>
static cudaError_t launch_stage_any(int dtype, int op, int order, ARGS& a, cudaStream_t s) {
  switch (dtype * 2 + op) {
    case F32 * 2 + SUM: return launch_stage_f32_sum(order, a, s);
    case F32 * 2 + MAX: return launch_stage_f32_max(order, a, s);
    case BF16 * 2 + SUM: return launch_stage_bf16_sum(order, a, s);
    case BF16 * 2 + MAX: return launch_stage_bf16_max(order, a, s);
    case I32 * 2 + SUM: return launch_stage_i32_sum(order, a, s);
    case I32 * 2 + MAX: return launch_stage_i32_max(order, a, s);
    case F16 * 2 + SUM: return launch_stage_f16_sum(order, a, s);
    case F16 * 2 + MAX: return launch_stage_f16_max(order, a, s);
    default: return cudaErrorInvalidValue;
  }
}

// `vec`: every row's buffers share their address modulo 16.  Rows that do
// not take the staged kernel, and so do double binary trees of rank counts
// the register-resident kernel is not compiled for (other than 2, 4, 8, 16,
// 32 and 64), aligned or not: measured on 5 x 64 MiB bf16, 665.3 us for the
// element-wise kernel that took them before, 97.8 staged.
template <class ARGS>
static cudaError_t launch_fused_any(int dtype, int op, int order, bool vec, ARGS& a, cudaStream_t s) {
  const int n = a.tab.nranks;
  const bool dbtree_regs = n == 2 || n == 4 || n == 8 || n == 16 || n == 32 || n == 64;
  if (!vec || (order == DBTREE && !dbtree_regs)) return launch_stage_any(dtype, op, order, a, s);
  switch (dtype * 2 + op) {
    case F32 * 2 + SUM: return launch_fused_f32_sum(order, a, s);
    case F32 * 2 + MAX: return launch_fused_f32_max(order, a, s);
    case BF16 * 2 + SUM: return launch_fused_bf16_sum(order, a, s);
    case BF16 * 2 + MAX: return launch_fused_bf16_max(order, a, s);
    case I32 * 2 + SUM: return launch_fused_i32_sum(order, a, s);
    case I32 * 2 + MAX: return launch_fused_i32_max(order, a, s);
    case F16 * 2 + SUM: return launch_fused_f16_sum(order, a, s);
    case F16 * 2 + MAX: return launch_fused_f16_max(order, a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fused(int dtype, int op, int order, bool vec, FusedArgs& a, cudaStream_t s) {
  return launch_fused_any(dtype, op, order, vec, a, s);
}

cudaError_t launch_fused(int dtype, int op, int order, bool vec, SmallFusedArgs& a, cudaStream_t s) {
  return launch_fused_any(dtype, op, order, vec, a, s);
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 1;
  return n;
}

}  // namespace ar
