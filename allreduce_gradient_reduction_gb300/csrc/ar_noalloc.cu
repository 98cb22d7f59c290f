// Bucketed gradient AllReduce that allocates no memory.
//
// Who needs it: callers that are not allowed to call cudaMalloc -- a process
// whose device memory is handed out by another allocator or a fixed pool that
// must account for every byte, an engine that bans allocation on its hot path
// because cudaMalloc can synchronise the device and stall every stream, or a
// runtime that must not fail for lack of memory once it has started.
// ar_bucketed_allreduce's literal path needs a pack workspace from the caller;
// this entry point takes that workspace from a fixed-size array compiled into
// the library instead, and keeps its host bookkeeping in fixed-size static
// tables, so the call allocates nothing on the device or on the host heap.
//
// The price: the array is held on every GPU where the library's device code
// is loaded, until the process exits; its size caps the buckets it can take;
// and all calls share it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "../../include/ar.h"
#include "ar_internal.h"

// The scratch: per rank, one slice of AR_NOALLOC_SCRATCH_BYTES / nranks
// (rounded down to 256 bytes) that holds the packed buckets of that rank.
static __device__ __align__(256) unsigned char g_noalloc_scratch[AR_NOALLOC_SCRATCH_BYTES];

namespace {

using ar::Seg;

constexpr int kMaxTensors = AR_NOALLOC_MAX_TENSORS;
constexpr int kMaxRanges = AR_MAX_RANKS * kMaxTensors;

struct Range {
  uintptr_t lo, hi;
};

// Host-side tables, shared by every call (calls are serialised on the host
// by g_mu; the device scratch is shared as well, see the header).
std::mutex g_mu;
Range g_ranges[kMaxRanges];
int32_t g_bucket_of[kMaxTensors];
int64_t g_offset[kMaxTensors];
int64_t g_bcount[kMaxTensors];
int64_t g_base[kMaxTensors];
// Device address of the scratch, per device ordinal, and the context it was
// looked up in (the address belongs to that context's copy of the module).
unsigned char* g_scratch_addr[256];
unsigned long long g_scratch_ctx[256];

typedef CUresult (*PointerGetAttributeFn)(void*, CUpointer_attribute, CUdeviceptr);

PointerGetAttributeFn attr_fn() {
  static PointerGetAttributeFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PointerGetAttributeFn>(p);
  }();
  return fn;
}

// Same rules as the other entry points: element-aligned, pairwise disjoint,
// device memory of the current device.  Sorts g_ranges[0..n) in place.
int check_ranges(int n, int esize, int dev) {
  for (int i = 0; i < n; ++i)
    if (g_ranges[i].lo == 0 || g_ranges[i].hi < g_ranges[i].lo || g_ranges[i].lo % (uintptr_t)esize)
      return AR_ERR_INVALID_ARG;
  std::sort(g_ranges, g_ranges + n, [](const Range& a, const Range& b) { return a.lo < b.lo; });
  for (int i = 1; i < n; ++i)
    if (g_ranges[i].lo < g_ranges[i - 1].hi || g_ranges[i].lo == g_ranges[i - 1].lo) return AR_ERR_INVALID_ARG;
  PointerGetAttributeFn attr = attr_fn();
  if (!attr) return ar::note_cuda_failure(cudaErrorNotSupported);
  uintptr_t alloc_lo = 0, alloc_hi = 0;
  for (int i = 0; i < n; ++i) {
    const Range& r = g_ranges[i];
    if (alloc_hi > alloc_lo && r.lo >= alloc_lo && r.hi <= alloc_hi) continue;
    unsigned int mtype = 0;
    int ordinal = -1;
    CUdeviceptr start = 0;
    size_t size = 0;
    if (attr(&mtype, CU_POINTER_ATTRIBUTE_MEMORY_TYPE, (CUdeviceptr)r.lo) != CUDA_SUCCESS ||
        mtype != CU_MEMORYTYPE_DEVICE)
      return AR_ERR_INVALID_ARG;
    if (attr(&ordinal, CU_POINTER_ATTRIBUTE_DEVICE_ORDINAL, (CUdeviceptr)r.lo) != CUDA_SUCCESS || ordinal != dev)
      return AR_ERR_INVALID_ARG;
    if (attr(&start, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, (CUdeviceptr)r.lo) != CUDA_SUCCESS ||
        attr(&size, CU_POINTER_ATTRIBUTE_RANGE_SIZE, (CUdeviceptr)r.lo) != CUDA_SUCCESS)
      return AR_ERR_INVALID_ARG;
    alloc_lo = (uintptr_t)start;
    alloc_hi = (uintptr_t)start + size;
    if (r.hi > alloc_hi) return AR_ERR_INVALID_ARG;
  }
  return AR_OK;
}

// Set-up, once per device, with that device current: the device address of
// the scratch array.  (In host code the array's name is only a host-side
// stand-in, not a device address.)  The address is cached per device together
// with the id of the context it was looked up in; if that context has since
// been torn down and replaced (cudaDeviceReset), the module was loaded again,
// possibly elsewhere, and the address is looked up anew.
int scratch_address(int dev, unsigned char** out) {
  if (dev < 0 || dev >= 256) return AR_ERR_NO_DEVICE;
  unsigned long long ctx = 0;
  int rc = ar::current_context_id(&ctx);
  if (rc) return rc;
  if (ctx == 0 || !g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // binds the device's context if none is current
    if (e != cudaSuccess) return ar::note_cuda_failure(e);
    if ((rc = ar::current_context_id(&ctx))) return rc;
    g_scratch_addr[dev] = static_cast<unsigned char*>(p);
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_addr[dev];
  return AR_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

int64_t chunk_lo(int64_t count, int n, int c) { return (int64_t)(((__int128)c * count) / n); }

int noalloc_body(void* const* grads, const int64_t* counts, int ntensors, int nranks, ar_dtype dtype, ar_op op,
                 ar_algo algo, int64_t bucket_cap_bytes, cudaStream_t stream) {
  // the argument rules of ar_bucketed_allreduce: out-of-range values are
  // AR_ERR_INVALID_ARG; AVG on i32, trees of other than 2^k ranks, and the
  // orders the bucketed call does not take (naive, double binary tree) are
  // AR_ERR_UNSUPPORTED
  int rc = ar::check_common(nranks, 0, dtype, op, algo);
  if (rc) return rc;
  if (algo == AR_NAIVE || algo == AR_DBTREE) return AR_ERR_UNSUPPORTED;
  // the step-wise kernels need a barrier block the library would allocate
  if (algo == AR_RING_STEPWISE || algo == AR_TREE_STEPWISE || algo == AR_BINOMIAL_STEPWISE) return AR_ERR_UNSUPPORTED;
  if (ntensors < 0 || bucket_cap_bytes <= 0) return AR_ERR_INVALID_ARG;
  if (ntensors == 0) return AR_OK;
  if (!grads || !counts) return AR_ERR_INVALID_ARG;
  if (ntensors > kMaxTensors) return AR_ERR_TOO_LARGE;
  const int es = (dtype == AR_BF16 || dtype == AR_F16) ? 2 : 4;

  std::lock_guard<std::mutex> lk(g_mu);
  int32_t nb = 0;
  rc = ar_bucket_plan(counts, ntensors, dtype, bucket_cap_bytes, g_bucket_of, g_offset, g_bcount, &nb);
  if (rc) return rc;
  // per-rank slice of the scratch, and whether the largest bucket fits in it
  const int64_t slice = ((int64_t)AR_NOALLOC_SCRATCH_BYTES / nranks) & ~(int64_t)255;
  int64_t total = 0;
  for (int b = 0; b < nb; ++b) {
    if (g_bcount[b] * es > slice) return AR_ERR_TOO_LARGE;
    g_base[b] = total;
    total += g_bcount[b];
  }
  int n = 0;
  for (int r = 0; r < nranks; ++r)
    for (int t = 0; t < ntensors; ++t) {
      if (counts[t] == 0) continue;
      const uintptr_t p = (uintptr_t)grads[(size_t)r * ntensors + t];
      g_ranges[n++] = {p, p + (uintptr_t)counts[t] * es};
    }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return ar::note_cuda_failure(e);
  if ((rc = check_ranges(n, es, dev))) return rc;
  if (nranks == 1) return AR_OK;
  unsigned char* scratch = nullptr;
  if ((rc = scratch_address(dev, &scratch))) return rc;
  const int order = algo == AR_TREE ? ar::TREE : ar::RING;
  const int dop = op == AR_MAX ? ar::MAX : ar::SUM;
  const int rows_cap = ar::kPtrCap / nranks;

  // Buckets [b0, b1) whose packed sizes fit one slice go through together:
  // pack every tensor of them, AllReduce each bucket as a flat buffer, unpack.
  int b0 = 0;
  while (b0 < nb) {
    int b1 = b0;
    int64_t used = 0;
    while (b1 < nb && (used + g_bcount[b1]) * es <= slice) used += g_bcount[b1++];
    const int64_t shift = g_base[b0];

    // copy the group's tensors into (to_packed = 1) or out of (0) the scratch
    auto copy = [&](int to_packed) -> int {
      ar::CopyArgs ca;
      memset(&ca, 0, sizeof(ca));
      for (int r = 0; r < nranks; ++r) ca.packed[r] = scratch + (size_t)r * slice;
      ca.esize = es;
      ca.to_packed = to_packed;
      int rows = 0;
      for (int t = 0; t <= ntensors; ++t) {
        const bool last = t == ntensors;
        if (last || rows == rows_cap || ca.tab.nseg == ar::kSegCap) {
          if (ca.tab.nseg > 0) {
            ca.tab.nranks = nranks;
            cudaError_t le = ar::launch_copy(ca, stream);
            if (le != cudaSuccess) return ar::note_cuda_failure(le);
          }
          ca.tab.nseg = 0;
          rows = 0;
        }
        if (last) break;
        if (counts[t] == 0 || g_bucket_of[t] < b0 || g_bucket_of[t] >= b1) continue;
        const int64_t aux = g_base[g_bucket_of[t]] - shift + g_offset[t];
        bool v = (aux * es) % 16 == 0;
        for (int r = 0; r < nranks; ++r) {
          const void* p = grads[(size_t)r * ntensors + t];
          ca.tab.ptr[rows * nranks + r] = p;
          v = v && aligned16(p);
        }
        Seg& s = ca.tab.seg[ca.tab.nseg++];
        s = Seg{};
        s.begin = 0;
        s.end = counts[t];
        s.aux = aux;
        s.tensor = rows;
        s.chunk = v ? 1 : 0;
        ++rows;
      }
      return AR_OK;
    };

    // AllReduce of every bucket of the group as a flat buffer, N chunks each
    auto reduce = [&]() -> int {
      ar::FusedArgs fa;
      memset(&fa, 0, sizeof(fa));
      fa.avg = op == AR_AVG;
      fa.owner_only = 0;
      fa.fn = (float)nranks;
      bool vec = true;
      int rows = 0;
      auto flush = [&]() -> int {
        if (fa.tab.nseg == 0) return AR_OK;
        fa.tab.nranks = nranks;
        cudaError_t le = ar::launch_fused(dtype, dop, order, vec, fa, stream);
        fa.tab.nseg = 0;
        rows = 0;
        vec = true;
        return le == cudaSuccess ? AR_OK : ar::note_cuda_failure(le);
      };
      for (int b = b0; b < b1; ++b) {
        if (rows == rows_cap || fa.tab.nseg + nranks > ar::kSegCap) {
          if (int r2 = flush()) return r2;
        }
        for (int r = 0; r < nranks; ++r) {
          const void* p = scratch + (size_t)r * slice + (size_t)(g_base[b] - shift) * es;
          fa.tab.ptr[rows * nranks + r] = p;
          vec = vec && aligned16(p);
        }
        for (int c = 0; c < nranks; ++c) {
          const int64_t lo = chunk_lo(g_bcount[b], nranks, c), hi = chunk_lo(g_bcount[b], nranks, c + 1);
          if (hi <= lo) continue;
          Seg& s = fa.tab.seg[fa.tab.nseg++];
          s = Seg{};
          s.begin = lo;
          s.end = hi;
          s.tensor = rows;
          s.chunk = c;
        }
        ++rows;
      }
      return flush();
    };

    if ((rc = copy(1))) return rc;
    if ((rc = reduce())) return rc;
    if ((rc = copy(0))) return rc;
    b0 = b1;
  }
  return AR_OK;
}

}  // namespace

// Nothing may unwind through the C ABI: an exception (the lock can throw)
// becomes AR_ERR_HOST, as in every other entry point.
extern "C" int ar_bucketed_allreduce_noalloc(void* const* grads, const int64_t* counts, int ntensors, int nranks,
                                             ar_dtype dtype, ar_op op, ar_algo algo, int64_t bucket_cap_bytes,
                                             ar_stream_t stream) {
  try {
    return noalloc_body(grads, counts, ntensors, nranks, dtype, op, algo, bucket_cap_bytes, (cudaStream_t)stream);
  } catch (...) {
    return AR_ERR_HOST;
  }
}
