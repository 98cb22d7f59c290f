// Internal interface between the C-ABI layer (ar_api.cpp) and the kernel
// translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace ar {

enum Dtype { F32 = 0, BF16 = 1, I32 = 2, F16 = 3 };
enum Op { SUM = 0, MAX = 1 };  // AVG = SUM plus the `avg` flag
enum Order { RING = 0, TREE = 1, DBTREE = 2, BINOMIAL = 3 };  // BINOMIAL: step-wise kernels only

constexpr int kMaxRanks = 64;
constexpr int kPtrCap = 512;  // pointers one launch can describe
constexpr int kSegCap = 256;  // segments one launch can describe

// A run of elements of one "tensor" (a row of nranks buffers) that lies in a
// single chunk, so every element of it is reduced in the same rank order.
struct Seg {
  int64_t begin;       // first element, relative to the tensor's base pointers
  int64_t end;         // one past the last element
  int64_t tile_begin;  // first tile of this segment (filled by the launcher)
  int64_t aux;         // copy kernels: element offset on the packed side
  int32_t tensor;      // row in the pointer table: ptr[tensor * nranks + rank]
  int32_t chunk;       // chunk id c (ring order starts at rank c+1); copy kernels: 1 = vectorisable
};

template <int PTRS, int SEGS>
struct SegTableT {
  const void* ptr[PTRS];
  Seg seg[SEGS];
  int32_t nranks;
  int32_t nseg;
  int64_t ntiles;
};
// Launch tables travel as kernel parameters, and a launch costs more the
// larger they are (16 KB: about 0.9 us more per call than 3 KB).  Calls
// whose rows fit use the small form.
using SegTable = SegTableT<kPtrCap, kSegCap>;
constexpr int kSmallSegCap = 72;
using SmallSegTable = SegTableT<kMaxRanks, kSmallSegCap>;

// Per-device block used by the step-wise kernels' grid barrier.
struct SyncBlock {
  unsigned int counter;  // arrivals; reset before each launch
  int abort;             // set by the first block that gives up; reset before each launch
  int status;            // sticky: AR_ERR_TIMEOUT until read by ar_device_status
  int pad;
};

template <class TABLE>
struct FusedArgsT {
  TABLE tab;
  int32_t avg;         // divide reduced values by nranks
  int32_t owner_only;  // ReduceScatter: store to the chunk owner only
  int32_t to_root;     // Reduce: store to rank `root` only
  int32_t root;
  int32_t max_grid;    // > 0: at most this many blocks (they stride over the tiles)
  float fn;            // (float)nranks
};
using FusedArgs = FusedArgsT<SegTable>;
using SmallFusedArgs = FusedArgsT<SmallSegTable>;

struct StepArgs {
  SegTable tab;
  SyncBlock* sync;
  int64_t timeout_ns;
  int32_t order;      // RING, TREE or BINOMIAL
  int32_t phases;     // bit 0 ReduceScatter (BINOMIAL: reduce to rank 0), bit 1 AllGather (BINOMIAL: broadcast)
  int32_t avg;
  int32_t skip_barrier;  // test hook, -1 = off
  float fn;
};

// The step-wise schedule of one buffer row small enough to live in one
// block's shared memory (each rank's count elements, padded to 16 bytes).
struct SmemStepArgs {
  const void* ptr[kMaxRanks];
  int64_t count;
  int32_t nranks;
  int32_t order;   // RING, TREE or BINOMIAL
  int32_t phases;  // bit 0 ReduceScatter (BINOMIAL: reduce to rank 0), bit 1 AllGather (BINOMIAL: broadcast)
  int32_t avg;
  int32_t vec;     // every pointer 16-byte aligned
  float fn;
};
constexpr int64_t kSmemStepBytes = 160 * 1024;  // shared memory the small step-wise kernel may use
// One block does a phase's element updates at about 0.45 ns each, a grid
// barrier plus phase of the multi-block kernel costs about 2.2 us: the block
// path is taken while a phase has at most this many element updates.
constexpr int64_t kSmemStepMaxPhaseElems = 3072;
inline int64_t smem_step_bytes(int nranks, int64_t count, int esize) {
  return (int64_t)nranks * ((count * esize + 15) / 16 * 16);
}
// The cluster form spreads the ranks over the blocks of one thread-block
// cluster (at most kSmemStepBytes of each block's shared memory).  A step
// there costs a cluster barrier (about 1 us) plus the busiest block's folds
// (about 0.22 ns per element with 16-byte vectors); a step of the
// grid-barrier form costs 2-5.5 us whatever its size.  So the cluster form
// pays while the busiest block folds few elements in an average step of the
// schedule.  Measured on GB300 against the grid-barrier form (bf16,
// CUDA-graph replay of 20 calls): with chunks cut on 16-byte boundaries
// (count a multiple of nranks * 16 / element size) it won up to about 6144
// elements per block per step (64 ranks x 16 KiB tree 66.0 -> 28.2 us,
// 16 x 128 KiB ring 67.6 -> 51.2 us, 8 x 16 KiB tree 14.4 -> 11.2 us) and
// lost from 7680 on (16 x 64 KiB tree 19.2 -> 23.8 us, 4 x 64 KiB ring
// 14.4 -> 18.3 us, 8 x 128 KiB ring 32.8 -> 38.8 us).  Otherwise a step
// moves one element at a time and the limit is the lower one.
constexpr int64_t kClusterStepMaxBlockElems = 1024;
constexpr int64_t kClusterStepMaxBlockElemsVec = 6144;
// Elements the busiest of the cluster's blocks folds in an average step,
// each block holding nloc ranks: ring, one chunk per rank in every step;
// tree, count * (1 - 1/N) per rank over the log2(N) halving steps (and the
// same over the doubling steps); binomial, up to a whole buffer per rank
// in every step.
inline int64_t cluster_step_mean_elems(int nranks, int64_t count, int order, int64_t nloc) {
  if (order == RING) return nloc * ((count + nranks - 1) / nranks);
  if (order == TREE) {
    int levels = 0;
    while ((2 << levels) <= nranks) ++levels;
    return nloc * (count - count / nranks) / levels;
  }
  return nloc * count;
}
// Blocks in the cluster for a row: the largest power of two that is at
// least 2 and at most max_size and nranks, if its blocks hold the row and
// the busiest block folds at most the limit above in an average step; 0
// otherwise.
inline int cluster_step_size(int nranks, int64_t count, int esize, int order, int max_size) {
  const int64_t stride = (count * esize + 15) / 16 * 16;
  int c = 2;
  while (c * 2 <= max_size && c * 2 <= nranks) c *= 2;
  if (c > nranks || c > max_size) return 0;
  const int64_t nloc = (nranks + c - 1) / c;
  if (nloc * stride > kSmemStepBytes) return 0;
  const bool vec = count % ((int64_t)nranks * (16 / esize)) == 0;
  const int64_t limit = vec ? kClusterStepMaxBlockElemsVec : kClusterStepMaxBlockElems;
  return cluster_step_mean_elems(nranks, count, order, nloc) <= limit ? c : 0;
}

struct CopyArgs {
  SegTable tab;                  // ptr[tensor * nranks + r] = tensor side
  const void* packed[kMaxRanks]; // packed side base per rank; seg.aux = element offset there
  int32_t to_packed;             // 1 = pack (tensor -> packed), 0 = unpack
  int32_t esize;
};

struct Int8Args {
  float* x[kMaxRanks];  // gradients, reduced in place
  float* e[kMaxRanks];  // error-feedback residuals, updated in place
  int64_t count;
  int32_t nranks;
  int32_t avg;
  int32_t vec;          // every pointer 16-byte aligned
  float fn;
};

// Launchers.  Each fills tab.seg[*].tile_begin and tab.ntiles for its own
// tile shape, then enqueues on `stream`.  `vec`: every row's buffers share
// their address modulo 16, so 16-byte vectors line up across ranks; rows
// that do not take the staged kernel (launch_fused, launch_gather) or one
// element per thread (launch_stepwise).
cudaError_t launch_fused(int dtype, int op, int order, bool vec, FusedArgs& args, cudaStream_t stream);
cudaError_t launch_fused(int dtype, int op, int order, bool vec, SmallFusedArgs& args, cudaStream_t stream);
cudaError_t launch_gather(int esize, bool vec, SegTable& tab, cudaStream_t stream);
cudaError_t launch_copy(CopyArgs& args, cudaStream_t stream);
cudaError_t launch_stepwise(int dtype, int op, bool vec, StepArgs& args, cudaStream_t stream);
cudaError_t launch_stepwise_smem(int dtype, int op, SmemStepArgs& args, cudaStream_t stream);
cudaError_t launch_stepwise_cluster(int dtype, int op, SmemStepArgs& args, int cluster_size, cudaStream_t stream);
int cluster_step_max_size();
cudaError_t launch_int8_ef(Int8Args& args, cudaStream_t stream);

int sm_count();

// ar_api.cpp helpers that other translation units share.
// The argument rules every collective entry point applies (ranges of nranks,
// count, dtype, op and algo; AVG on i32 and trees of other than 2^k ranks are
// AR_ERR_UNSUPPORTED).
int check_common(int nranks, int64_t count, int dtype, int op, int algo);
// Records a CUDA failure for ar_last_cuda_error and maps it to a status.
int note_cuda_failure(cudaError_t e);
// Unique id of the context current on this thread (0 if none is current).
// Device addresses the library caches per device are keyed by it, so a
// context that was torn down (cudaDeviceReset) and replaced is noticed.
int current_context_id(unsigned long long* id);
// Applies a kernel's per-function settings -- the opt-in to `smem_bytes` of
// dynamic shared memory and, with `big_clusters`, to clusters past the
// portable eight blocks -- once per context.  `tag` has one entry per device
// ordinal holding the id of the context they were last applied in: function
// attributes belong to the module as loaded in one context, and a context
// torn down and replaced (cudaDeviceReset) loads the module anew with the
// defaults.
cudaError_t open_kernel(const void* kernel, int smem_bytes, bool big_clusters,
                        std::atomic<unsigned long long>* tag);

// Counts every kernel launch the library enqueues (ar_kernel_launches).
void count_launch();

}  // namespace ar
