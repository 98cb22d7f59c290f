// C ABI of the simulated-AllReduce library: argument checks, chunk and bucket
// planning, descriptor tables, and kernel launches.  Declarations and the
// contract of every entry point are in include/ar.h.
#include "../../include/ar.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "ar_internal.h"

namespace {

using ar::Seg;
using ar::SegTable;

thread_local cudaError_t g_last_cuda = cudaSuccess;
std::atomic<int64_t> g_timeout_ns{1000000000LL};
std::atomic<int> g_skip_barrier{-1};

int cuda_fail(cudaError_t e) {
  g_last_cuda = e;
  return e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver ? AR_ERR_NO_DEVICE : AR_ERR_CUDA;
}

int esize_of(int dtype) { return (dtype == AR_BF16 || dtype == AR_F16) ? 2 : 4; }

bool is_pow2(int n) { return n > 0 && (n & (n - 1)) == 0; }

bool is_stepwise(int algo) {
  return algo == AR_RING_STEPWISE || algo == AR_TREE_STEPWISE || algo == AR_BINOMIAL_STEPWISE;
}

// Chunk c of `count` elements split n ways: [floor(c*count/n), floor((c+1)*count/n)).
int64_t chunk_lo(int64_t count, int n, int c) { return (int64_t)(((__int128)c * count) / n); }

// ---- pointer checks -----------------------------------------------------------

typedef CUresult (*PointerGetAttributesFn)(unsigned int, CUpointer_attribute*, void**, CUdeviceptr);

PointerGetAttributesFn pointer_attrs_fn() {
  static PointerGetAttributesFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttributes", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PointerGetAttributesFn>(p);
  }();
  return fn;
}

struct Range {
  uintptr_t lo, hi;
};

// Every range must be non-null, element aligned and pairwise disjoint (sorts rs).
int check_disjoint(std::vector<Range>& rs, int esize) {
  for (const Range& r : rs) {
    if (r.lo == 0 || r.hi < r.lo) return AR_ERR_INVALID_ARG;  // NULL, or an end past the address space
    if (r.lo % (uintptr_t)esize) return AR_ERR_INVALID_ARG;
  }
  std::sort(rs.begin(), rs.end(), [](const Range& a, const Range& b) { return a.lo < b.lo; });
  for (size_t i = 1; i < rs.size(); ++i)
    if (rs[i].lo < rs[i - 1].hi || rs[i].lo == rs[i - 1].lo) return AR_ERR_INVALID_ARG;
  return AR_OK;
}

// ... and lie inside device memory of the current device.
int check_ranges(std::vector<Range>& rs, int esize) {
  int rc = check_disjoint(rs, esize);
  if (rc) return rc;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  PointerGetAttributesFn attrs = pointer_attrs_fn();
  if (!attrs) return cuda_fail(cudaErrorNotSupported);
  // ranges are sorted: one driver query (four attributes) per allocation they fall into
  uintptr_t alloc_lo = 0, alloc_hi = 0;
  for (const Range& r : rs) {
    if (r.lo >= alloc_lo && r.hi <= alloc_hi && alloc_hi > alloc_lo) continue;
    unsigned int mtype = 0;
    int ordinal = -1;
    CUdeviceptr start = 0;
    size_t size = 0;
    CUpointer_attribute which[4] = {CU_POINTER_ATTRIBUTE_MEMORY_TYPE, CU_POINTER_ATTRIBUTE_DEVICE_ORDINAL,
                                    CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, CU_POINTER_ATTRIBUTE_RANGE_SIZE};
    void* out[4] = {&mtype, &ordinal, &start, &size};
    if (attrs(4, which, out, (CUdeviceptr)r.lo) != CUDA_SUCCESS) return AR_ERR_INVALID_ARG;
    if (mtype != CU_MEMORYTYPE_DEVICE || ordinal != dev || size == 0) return AR_ERR_INVALID_ARG;
    alloc_lo = (uintptr_t)start;
    alloc_hi = (uintptr_t)start + size;
    if (r.lo < alloc_lo || r.hi > alloc_hi) return AR_ERR_INVALID_ARG;
  }
  return AR_OK;
}

// Every range must be non-null, element aligned, pairwise disjoint, and lie
// inside page-locked host memory that kernels on the current device reach at
// the same address (a mapped allocation under unified addressing).
int check_mapped_host(std::vector<Range>& rs, int esize) {
  int rc = check_disjoint(rs, esize);
  if (rc) return rc;
  PointerGetAttributesFn attrs = pointer_attrs_fn();
  if (!attrs) return cuda_fail(cudaErrorNotSupported);
  for (const Range& r : rs) {
    unsigned int mtype = 0;
    CUdeviceptr devptr = 0, start = 0;
    size_t size = 0;
    CUpointer_attribute which[4] = {CU_POINTER_ATTRIBUTE_MEMORY_TYPE, CU_POINTER_ATTRIBUTE_DEVICE_POINTER,
                                    CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, CU_POINTER_ATTRIBUTE_RANGE_SIZE};
    void* out[4] = {&mtype, &devptr, &start, &size};
    if (attrs(4, which, out, (CUdeviceptr)r.lo) != CUDA_SUCCESS) return AR_ERR_INVALID_ARG;
    if (mtype != CU_MEMORYTYPE_HOST || devptr != (CUdeviceptr)r.lo || size == 0) return AR_ERR_INVALID_ARG;
    if (r.lo < (uintptr_t)start || r.hi > (uintptr_t)start + size) return AR_ERR_INVALID_ARG;
  }
  return AR_OK;
}

int check_common(int nranks, int64_t count, int dtype, int op, int algo) {
  if (nranks < 1 || nranks > AR_MAX_RANKS || count < 0 || count > AR_MAX_COUNT) return AR_ERR_INVALID_ARG;
  if (dtype < AR_F32 || dtype > AR_F16 || op < AR_SUM || op > AR_AVG) return AR_ERR_INVALID_ARG;
  if (algo < AR_RING || algo > AR_BINOMIAL_STEPWISE) return AR_ERR_INVALID_ARG;
  if (op == AR_AVG && dtype == AR_I32) return AR_ERR_UNSUPPORTED;
  if ((algo == AR_TREE || algo == AR_TREE_STEPWISE || algo == AR_BINOMIAL_STEPWISE) && !is_pow2(nranks))
    return AR_ERR_UNSUPPORTED;
  return AR_OK;
}

int check_bufs(void* const* bufs, int nranks, int64_t count, int dtype) {
  if (!bufs) return AR_ERR_INVALID_ARG;
  if (count == 0) return AR_OK;  // nothing is accessed: any pointers (NULL included) will do
  std::vector<Range> rs;
  for (int r = 0; r < nranks; ++r) {
    uintptr_t p = (uintptr_t)bufs[r];
    rs.push_back({p, p + (uintptr_t)count * esize_of(dtype)});
  }
  return check_ranges(rs, esize_of(dtype));
}

// The fused, gather and step-wise kernels move a row in 16-byte vectors
// when all its buffers have the same address modulo 16 (they cut the
// vectors at that offset); true 16-byte alignment is needed only where
// shared or packed staging assumes it.
bool same_phase16(void* const* p, int n) {
  for (int i = 1; i < n; ++i)
    if (((uintptr_t)p[i] & 15) != ((uintptr_t)p[0] & 15)) return false;
  return true;
}

bool all_aligned16(void* const* p, int n) {
  for (int i = 0; i < n; ++i)
    if ((uintptr_t)p[i] % 16) return false;
  return true;
}

// ---- the current context's identity --------------------------------------------

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <class FN>
FN driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    p = nullptr;
  return reinterpret_cast<FN>(p);
}

int context_id(unsigned long long* id) {
  static CtxGetCurrentFn cur = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn getid = driver_fn<CtxGetIdFn>("cuCtxGetId");
  *id = 0;
  if (!cur || !getid) return cuda_fail(cudaErrorNotSupported);
  CUcontext c = nullptr;
  if (cur(&c) != CUDA_SUCCESS) return cuda_fail(cudaErrorDeviceUninitialized);
  if (c && getid(c, id) != CUDA_SUCCESS) return cuda_fail(cudaErrorDeviceUninitialized);
  return AR_OK;
}

// ---- per-device barrier block for the step-wise kernels ------------------------

// One block per device, allocated on first use and tagged with the context it
// was allocated in: a context that was torn down (cudaDeviceReset) took the
// block with it, so a new context gets a new one.
std::mutex g_sync_mu;
ar::SyncBlock* g_sync[256] = {};
unsigned long long g_sync_ctx[256] = {};

int sync_block(ar::SyncBlock** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 256) return AR_ERR_NO_DEVICE;
  unsigned long long ctx = 0;
  int rc = context_id(&ctx);
  if (rc) return rc;
  if (ctx == 0) {
    // no context current on this thread yet: let the runtime bind its own
    // (cudaFree of NULL frees nothing), then ask again
    if ((e = cudaFree(nullptr)) != cudaSuccess) return cuda_fail(e);
    if ((rc = context_id(&ctx))) return rc;
  }
  std::lock_guard<std::mutex> lk(g_sync_mu);
  if (!g_sync[dev] || g_sync_ctx[dev] != ctx) {
    void* p = nullptr;
    if ((e = cudaMalloc(&p, sizeof(ar::SyncBlock))) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMemset(p, 0, sizeof(ar::SyncBlock))) != cudaSuccess) {
      cudaFree(p);
      return cuda_fail(e);
    }
    g_sync[dev] = static_cast<ar::SyncBlock*>(p);
    g_sync_ctx[dev] = ctx;
  }
  *out = g_sync[dev];
  return AR_OK;
}

// ---- per-device copy streams of the host-buffer AllReduce ------------------------

struct HostPipe {
  std::mutex mu;  // one call at a time enqueues on this device's streams and events
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t start = nullptr, uploaded = nullptr, reduced = nullptr, done = nullptr;
};
std::mutex g_pipe_mu;
HostPipe g_pipe[256];

int host_pipe(HostPipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 256) return AR_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_pipe_mu);
  HostPipe& p = g_pipe[dev];
  if (!p.done) {
    cudaStream_t st[2] = {nullptr, nullptr};
    cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaStreamCreateWithFlags(&st[i], cudaStreamNonBlocking);
    for (int i = 0; i < 4 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
    if (e != cudaSuccess) {
      for (cudaEvent_t x : ev)
        if (x) cudaEventDestroy(x);
      for (cudaStream_t x : st)
        if (x) cudaStreamDestroy(x);
      return cuda_fail(e);
    }
    p.up = st[0], p.down = st[1];
    p.start = ev[0], p.uploaded = ev[1], p.reduced = ev[2], p.done = ev[3];
  }
  *out = &p;
  return AR_OK;
}

// First element of every piece of the host-buffer AllReduce.  An explicit
// piece size is used as given (rounded up to 64 elements).  By default the
// pieces hold count / 8 elements, between 1 MiB and 16 MiB per rank, and the
// first and last three are 1/8, 1/4 and 1/2 of that: the time when only the
// first upload or only the last download is running is what the overlap
// cannot hide, so those pieces are small, and the rest are large, which the
// copy engines move most efficiently.
std::vector<int64_t> host_pieces(int64_t count, int es, int64_t piece_elems) {
  auto round64 = [](int64_t v) { return std::max<int64_t>(64, (v + 63) / 64 * 64); };
  std::vector<int64_t> starts;
  if (piece_elems > 0) {
    const int64_t p = round64(piece_elems);
    for (int64_t a = 0; a < count; a += p) starts.push_back(a);
    return starts;
  }
  const int64_t lo = ((int64_t)1 << 20) / es, hi = ((int64_t)16 << 20) / es;
  const int64_t p = round64(std::min(hi, std::max(lo, count / 8)));
  const int64_t ramp[3] = {round64(p / 8), round64(p / 4), round64(p / 2)};
  const int64_t ramp_total = 2 * (ramp[0] + ramp[1] + ramp[2]);
  int64_t a = 0;
  if (count >= ramp_total + p) {
    const int64_t tail = (count - ramp_total / 2) / 64 * 64;  // first of the last three pieces
    for (int i = 0; i < 3; ++i) starts.push_back(a), a += ramp[i];
    const int64_t mid = tail - a;
    const int64_t nmid = (mid + p - 1) / p, step = round64((mid + nmid - 1) / nmid);
    for (; a < tail; a += step) starts.push_back(a);
    a = tail;
    for (int i = 2; i >= 0; --i) starts.push_back(a), a += ramp[i];
  } else {
    for (; a < count; a += p) starts.push_back(a);
  }
  return starts;
}

// ---- one launch over a descriptor table ----------------------------------------

struct Job {
  int dtype, op, algo, phases;  // phases: 1 RS, 2 AG, 3 both
  bool avg;
  bool vec;
  int root = -1;  // Reduce: the rank that receives the result
  int max_grid = 0;  // fused kernels: cap on the number of blocks (0 = one per tile)
  int64_t row_count = 0;  // plain collectives: elements per rank of their single buffer row (0: several rows)
  bool aligned = false;   // every buffer 16-byte aligned (the single-block step-wise form stages with it)
};

// A table whose rows fit the small launch form (see ar::SmallSegTable).
bool fits_small(const SegTable& tab) {
  if (tab.nseg < 1 || tab.nseg > ar::kSmallSegCap) return false;
  return (int64_t)(tab.seg[tab.nseg - 1].tensor + 1) * tab.nranks <= ar::kMaxRanks;
}

template <class ARGS>
void fill_fused(const Job& j, int nranks, ARGS& a) {
  a.avg = j.avg ? 1 : 0;
  a.owner_only = j.phases == 1 ? 1 : 0;
  a.to_root = j.root >= 0 ? 1 : 0;
  a.root = j.root >= 0 ? j.root : 0;
  a.max_grid = j.max_grid;
  a.fn = (float)nranks;
}

int run_table(const Job& j, SegTable& tab, cudaStream_t s) {
  const int dop = j.op == AR_MAX ? ar::MAX : ar::SUM;
  const bool stepwise = is_stepwise(j.algo);
  const int order = j.algo == AR_DBTREE ? ar::DBTREE
                    : j.algo == AR_BINOMIAL_STEPWISE ? ar::BINOMIAL
                    : (j.algo == AR_TREE || j.algo == AR_TREE_STEPWISE) ? ar::TREE : ar::RING;
  cudaError_t e;
  // element updates in the busiest phase: the chunk's count for the ring,
  // N/2 pairs of it in the first tree or binomial step
  const int64_t phase_elems = j.row_count * (order == ar::TREE || order == ar::BINOMIAL ? tab.nranks / 2 : 1);
  const bool one_block = stepwise && j.row_count > 0 && phase_elems <= ar::kSmemStepMaxPhaseElems &&
                         ar::smem_step_bytes(tab.nranks, j.row_count, esize_of(j.dtype)) <= ar::kSmemStepBytes;
  int csize = 0;
  if (stepwise && !one_block && j.row_count > 0)
    csize = ar::cluster_step_size(tab.nranks, j.row_count, esize_of(j.dtype), order, ar::cluster_step_max_size());
  if (one_block || csize > 0) {
    // a small row: the whole schedule in one block's shared memory, or in
    // one thread-block cluster's (no grid barrier, so the barrier test hook
    // is consumed without effect)
    g_skip_barrier.exchange(-1);
    ar::SmemStepArgs a;
    memset(&a, 0, sizeof(a));
    for (int r = 0; r < tab.nranks; ++r) a.ptr[r] = tab.ptr[r];
    a.count = j.row_count;
    a.nranks = tab.nranks;
    a.order = order;
    a.phases = j.phases;
    a.avg = j.avg ? 1 : 0;
    a.vec = j.aligned ? 1 : 0;
    a.fn = (float)tab.nranks;
    e = one_block ? ar::launch_stepwise_smem(j.dtype, dop, a, s) : ar::launch_stepwise_cluster(j.dtype, dop, a, csize, s);
  } else if (stepwise) {
    ar::SyncBlock* sb = nullptr;
    int rc = sync_block(&sb);
    if (rc) return rc;
    // counter and abort start at zero for every launch; status stays sticky
    if ((e = cudaMemsetAsync(sb, 0, 2 * sizeof(int), s)) != cudaSuccess) return cuda_fail(e);
    ar::StepArgs a;
    a.tab = tab;
    a.sync = sb;
    a.timeout_ns = g_timeout_ns.load();
    a.order = order;
    a.phases = j.phases;
    a.avg = j.avg ? 1 : 0;
    a.skip_barrier = g_skip_barrier.exchange(-1);
    a.fn = (float)tab.nranks;
    e = ar::launch_stepwise(j.dtype, dop, j.vec, a, s);
  } else if (j.phases == 2) {
    e = ar::launch_gather(esize_of(j.dtype), j.vec, tab, s);
  } else if (fits_small(tab)) {
    ar::SmallFusedArgs a;
    const int nptr = (tab.seg[tab.nseg - 1].tensor + 1) * tab.nranks;
    memcpy(a.tab.ptr, tab.ptr, sizeof(void*) * (size_t)nptr);
    memcpy(a.tab.seg, tab.seg, sizeof(Seg) * (size_t)tab.nseg);
    a.tab.nranks = tab.nranks;
    a.tab.nseg = tab.nseg;
    a.tab.ntiles = 0;
    fill_fused(j, tab.nranks, a);
    e = ar::launch_fused(j.dtype, dop, order, j.vec, a, s);
  } else {
    ar::FusedArgs a;
    a.tab = tab;
    fill_fused(j, tab.nranks, a);
    e = ar::launch_fused(j.dtype, dop, order, j.vec, a, s);
  }
  return e == cudaSuccess ? AR_OK : cuda_fail(e);
}

// Rows (one per tensor: nranks pointers) and their segments, packed into as
// few descriptor tables as the launch limits allow.
struct TableBuilder {
  int nranks;
  std::vector<const void*> ptrs;  // row-major
  std::vector<Seg> segs;
  int add_row(void* const* row_ptrs) {
    for (int r = 0; r < nranks; ++r) ptrs.push_back(row_ptrs[r]);
    return (int)(ptrs.size() / nranks) - 1;
  }
  void add_seg(int row, int64_t begin, int64_t end, int chunk, int64_t aux = 0) {
    if (end <= begin) return;
    Seg s{};
    s.begin = begin;
    s.end = end;
    s.aux = aux;
    s.tensor = row;
    s.chunk = chunk;
    segs.push_back(s);
  }
  // Calls fn(table) for consecutive groups of whole rows.
  template <typename F>
  int for_each_table(F fn) {
    const int rows = (int)(ptrs.size() / nranks);
    const int rows_cap = ar::kPtrCap / nranks;
    if (rows_cap < 1) return AR_ERR_TOO_LARGE;
    SegTable t;
    size_t si = 0;
    int row0 = 0;
    while (row0 < rows) {
      memset(&t, 0, sizeof(t));
      t.nranks = nranks;
      int nrow = 0;
      // take rows while both the pointer and the segment tables have room
      size_t sj = si;
      while (row0 + nrow < rows && nrow < rows_cap) {
        size_t sk = sj;
        while (sk < segs.size() && segs[sk].tensor == row0 + nrow) ++sk;
        if ((int)(sk - si) > ar::kSegCap) break;
        ++nrow;
        sj = sk;
      }
      if (nrow == 0) return AR_ERR_TOO_LARGE;  // one row alone has too many segments
      for (int r = 0; r < nrow; ++r)
        for (int k = 0; k < nranks; ++k) t.ptr[r * nranks + k] = ptrs[(size_t)(row0 + r) * nranks + k];
      t.nseg = (int)(sj - si);
      for (int k = 0; k < t.nseg; ++k) {
        t.seg[k] = segs[si + k];
        t.seg[k].tensor -= row0;
      }
      if (t.nseg > 0) {
        int rc = fn(t);
        if (rc) return rc;
      }
      si = sj;
      row0 += nrow;
    }
    return AR_OK;
  }
};

// phases: 1 ReduceScatter, 2 AllGather, 3 AllReduce; root >= 0: Reduce to root
// Checks the arguments and builds the launch of a collective.  *empty is set
// when there is nothing to do (count 0 or one rank).
int build_collective(void* const* bufs, int nranks, int64_t count, int dtype, int op, int algo, int phases, int root,
                     TableBuilder& tb, Job& j, bool* empty, bool bufs_checked = false) {
  *empty = false;
  int rc = check_common(nranks, count, dtype, phases == 2 ? AR_SUM : op, algo);
  if (rc) return rc;
  if ((algo == AR_NAIVE || algo == AR_DBTREE || algo == AR_BINOMIAL_STEPWISE) && phases != 3)
    return AR_ERR_UNSUPPORTED;  // AllReduce / Reduce only
  if ((algo == AR_DBTREE || algo == AR_BINOMIAL_STEPWISE) && root >= 0) return AR_ERR_UNSUPPORTED;  // AllReduce only
  if (!bufs_checked && (rc = check_bufs(bufs, nranks, count, dtype))) return rc;
  if (count == 0 || nranks == 1) {
    *empty = true;
    return AR_OK;
  }
  int row = tb.add_row(bufs);
  if (algo == AR_NAIVE) {
    // index order x[0], x[1], ..., x[N-1] is the ring order of chunk N-1
    tb.add_seg(row, 0, count, nranks - 1);
  } else if (algo == AR_DBTREE) {
    // tree A reduces the first half (chunk id 0), tree B the second (1)
    tb.add_seg(row, 0, count / 2, 0);
    tb.add_seg(row, count / 2, count, 1);
  } else if (algo == AR_BINOMIAL_STEPWISE) {
    // whole buffers move in every step: one segment
    tb.add_seg(row, 0, count, 0);
  } else {
    for (int c = 0; c < nranks; ++c) tb.add_seg(row, chunk_lo(count, nranks, c), chunk_lo(count, nranks, c + 1), c);
  }
  j = Job{dtype, op, algo == AR_NAIVE ? AR_RING : algo, phases, op == AR_AVG, same_phase16(bufs, nranks)};  // naive = ring kernel
  j.root = root;
  j.row_count = count;
  j.aligned = all_aligned16(bufs, nranks);
  return AR_OK;
}

// phases: 1 ReduceScatter, 2 AllGather, 3 AllReduce; root >= 0: Reduce to root
int collective(void* const* bufs, int nranks, int64_t count, int dtype, int op, int algo, int phases,
               cudaStream_t stream, int root = -1) {
  TableBuilder tb{nranks, {}, {}};
  Job j{};
  bool empty = false;
  int rc = build_collective(bufs, nranks, count, dtype, op, algo, phases, root, tb, j, &empty);
  if (rc || empty) return rc;
  return tb.for_each_table([&](SegTable& t) { return run_table(j, t, stream); });
}

// Rows of the fused bucketed AllReduce for the tensors `keep(t)` selects: each
// tensor is cut at its bucket's chunk boundaries, and each piece is folded in
// the order its bucket position implies (as if the bucket had been packed).
// Returns whether every row can move in 16-byte vectors (same_phase16).
template <typename Keep>
bool add_bucket_rows(TableBuilder& tb, void* const* grads, const int64_t* counts, int ntensors, int nranks,
                     const int32_t* bucket_of, const int64_t* offset, const int64_t* bcount, Keep keep) {
  bool vec = true;
  std::vector<void*> row(nranks);
  for (int t = 0; t < ntensors; ++t) {
    if (counts[t] == 0 || !keep(t)) continue;
    for (int r = 0; r < nranks; ++r) row[r] = grads[(size_t)r * ntensors + t];
    vec = vec && same_phase16(row.data(), nranks);
    const int rw = tb.add_row(row.data());
    const int64_t B = bcount[bucket_of[t]], o = offset[t];
    for (int c = 0; c < nranks; ++c) {
      const int64_t lo = std::max(chunk_lo(B, nranks, c), o), hi = std::min(chunk_lo(B, nranks, c + 1), o + counts[t]);
      tb.add_seg(rw, lo - o, hi - o, c);
    }
  }
  return vec;
}

int plan_buckets(const int64_t* counts, int ntensors, int dtype, int64_t cap, int32_t* bucket_of, int64_t* offset,
                 int64_t* bcount, int32_t* nb) {
  const int es = esize_of(dtype);
  int b = -1;
  int64_t fill = 0, total = 0;
  for (int t = ntensors - 1; t >= 0; --t) {
    if (counts[t] < 0 || counts[t] > AR_MAX_COUNT - total) return AR_ERR_INVALID_ARG;
    total += counts[t];
    const int64_t bytes = counts[t] * es;
    if (b < 0 || (fill > 0 && fill + bytes > cap)) {
      ++b;
      bcount[b] = 0;
      fill = 0;
    }
    bucket_of[t] = b;
    offset[t] = bcount[b];
    bcount[b] += counts[t];
    fill += bytes;
  }
  *nb = b + 1;
  return AR_OK;
}

}  // namespace

namespace ar {
// Lets other translation units report a CUDA failure the same way.
int note_cuda_failure(cudaError_t e) { return cuda_fail(e); }
int check_common(int nranks, int64_t count, int dtype, int op, int algo) {
  return ::check_common(nranks, count, dtype, op, algo);
}
int current_context_id(unsigned long long* id) { return context_id(id); }

cudaError_t open_kernel(const void* kernel, int smem_bytes, bool big_clusters,
                        std::atomic<unsigned long long>* tag) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
  unsigned long long ctx = 0;
  if (context_id(&ctx) != AR_OK) return cudaErrorDeviceUninitialized;
  if (ctx != 0 && tag[dev].load() == ctx) return cudaSuccess;
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes)) != cudaSuccess)
    return e;
  if (big_clusters && (e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
    return e;
  // the first runtime call on this thread may have made the device's context current
  if (ctx == 0 && context_id(&ctx) != AR_OK) return cudaErrorDeviceUninitialized;
  tag[dev].store(ctx);
  return cudaSuccess;
}

std::atomic<int64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace ar

// ---- overlapped bucket reduction (DDP's reducer) --------------------------------
//
// DDP does not wait for the whole backward pass: as soon as every gradient of
// a bucket is ready it starts that bucket's AllReduce asynchronously, so the
// communication overlaps the rest of the backward computation, and it starts
// buckets in bucket order ("Allreduce：..." §4.1 通信与计算重叠; "AllReduce 集合
// 通信" §DDP 梯度同步中的地位).  Here the compute work runs on the caller's
// compute stream and the bucket reductions on a communication stream; an event
// recorded when a bucket becomes ready orders the two.

// A collective whose arguments were checked and whose launch tables were
// built once: running it only enqueues the kernels.
struct ar_plan {
  Job job{};
  std::vector<SegTable> tables;
};

struct ar_reducer {
  int nranks = 0, ntensors = 0, nbuckets = 0;
  Job job{};
  cudaStream_t comm = nullptr;
  std::vector<int32_t> bucket_of;
  std::vector<int> left;           // per bucket: tensors not yet marked this iteration
  std::vector<char> ready;         // per tensor
  std::vector<std::vector<SegTable>> tables;  // per bucket: launch tables, built once
  std::vector<cudaEvent_t> ready_ev;          // per bucket
  cudaEvent_t done_ev = nullptr;
  int next = 0;                    // next bucket to start (buckets start in order)
  int64_t ntables = 0;
};

namespace {

void reducer_reset(ar_reducer* red) {
  std::fill(red->ready.begin(), red->ready.end(), 0);
  std::fill(red->left.begin(), red->left.end(), 0);
  for (int t = 0; t < red->ntensors; ++t) red->left[red->bucket_of[t]]++;
  red->next = 0;
}

void reducer_free(ar_reducer* red) {
  for (cudaEvent_t e : red->ready_ev)
    if (e) cudaEventDestroy(e);
  if (red->done_ev) cudaEventDestroy(red->done_ev);
  delete red;
}

}  // namespace

// Nothing may unwind through the C ABI: a host allocation failure (or any
// other exception) in an entry point becomes AR_ERR_HOST.
template <class F>
int guarded(F f) noexcept {
  try {
    return f();
  } catch (...) {
    return AR_ERR_HOST;
  }
}

extern "C" {

int ar_allreduce(void* const* bufs, int nranks, int64_t count, ar_dtype dtype, ar_op op, ar_algo algo,
                 ar_stream_t stream) {
  return guarded([&]() -> int {
    return collective(bufs, nranks, count, dtype, op, algo, 3, (cudaStream_t)stream);
  });
}

int ar_reduce_scatter(void* const* bufs, int nranks, int64_t count, ar_dtype dtype, ar_op op, ar_algo algo,
                      ar_stream_t stream) {
  return guarded([&]() -> int {
    return collective(bufs, nranks, count, dtype, op, algo, 1, (cudaStream_t)stream);
  });
}

int ar_all_gather(void* const* bufs, int nranks, int64_t count, ar_dtype dtype, ar_algo algo, ar_stream_t stream) {
  return guarded([&]() -> int {
    return collective(bufs, nranks, count, dtype, AR_SUM, algo, 2, (cudaStream_t)stream);
  });
}

int ar_reduce(void* const* bufs, int nranks, int64_t count, ar_dtype dtype, ar_op op, ar_algo algo, int root,
              ar_stream_t stream) {
  return guarded([&]() -> int {
    if (root < 0 || root >= nranks) return AR_ERR_INVALID_ARG;
    if (is_stepwise(algo)) return AR_ERR_UNSUPPORTED;
    return collective(bufs, nranks, count, dtype, op, algo, 3, (cudaStream_t)stream, root);
  });
}

int ar_broadcast(void* const* bufs, int nranks, int64_t count, ar_dtype dtype, int root, ar_stream_t stream) {
  return guarded([&]() -> int {
    if (root < 0 || root >= nranks) return AR_ERR_INVALID_ARG;
    int rc = check_common(nranks, count, dtype, AR_SUM, AR_RING);
    if (rc) return rc;
    if ((rc = check_bufs(bufs, nranks, count, dtype))) return rc;
    if (count == 0 || nranks == 1) return AR_OK;
    // one segment owned by the root: the AllGather copy kernel sends it to every other rank
    TableBuilder tb{nranks, {}, {}};
    tb.add_seg(tb.add_row(bufs), 0, count, root);
    Job j{dtype, AR_SUM, AR_RING, 2, false, same_phase16(bufs, nranks)};
    return tb.for_each_table([&](SegTable& t) { return run_table(j, t, (cudaStream_t)stream); });
  });
}

int ar_allreduce_host(void* const* host_bufs, void* const* dev_bufs, int nranks, int64_t count, ar_dtype dtype,
                      ar_op op, ar_algo algo, int64_t piece_elems, ar_stream_t stream_) {
  return guarded([&]() -> int {
    int rc = check_common(nranks, count, dtype, op, algo);
    if (rc) return rc;
    if (is_stepwise(algo)) return AR_ERR_UNSUPPORTED;
    if (!host_bufs || piece_elems < 0) return AR_ERR_INVALID_ARG;
    if (count == 0) return AR_OK;  // nothing is accessed
    const int es = esize_of(dtype);
    if (!dev_bufs) {
      // zero-copy: one fused launch reads and writes the mapped host buffers
      std::vector<Range> rs;
      for (int r = 0; r < nranks; ++r) {
        const uintptr_t h = (uintptr_t)host_bufs[r];
        rs.push_back({h, h + (uintptr_t)count * es});
      }
      if ((rc = check_mapped_host(rs, es))) return rc;
      TableBuilder tb{nranks, {}, {}};
      Job j{};
      bool empty = false;
      if ((rc = build_collective(host_bufs, nranks, count, dtype, op, algo, 3, -1, tb, j, &empty, true)) || empty)
        return rc;
      return tb.for_each_table([&](SegTable& t) { return run_table(j, t, (cudaStream_t)stream_); });
    }
    {
      std::vector<Range> all;
      for (int r = 0; r < nranks; ++r) {
        const uintptr_t h = (uintptr_t)host_bufs[r], d = (uintptr_t)dev_bufs[r];
        all.push_back({h, h + (uintptr_t)count * es});
        all.push_back({d, d + (uintptr_t)count * es});
      }
      if ((rc = check_disjoint(all, es))) return rc;
    }
    if ((rc = check_bufs(dev_bufs, nranks, count, dtype))) return rc;
    if (nranks == 1) return AR_OK;  // a single rank already holds the reduction
    HostPipe* hp = nullptr;
    if ((rc = host_pipe(&hp))) return rc;
    std::lock_guard<std::mutex> lk(hp->mu);
    const std::vector<int64_t> starts = host_pieces(count, es, piece_elems);
    // every piece is folded in the order of its elements' chunks of the whole buffer
    Job j{dtype, op, algo == AR_NAIVE ? AR_RING : algo, 3, op == AR_AVG, same_phase16(dev_bufs, nranks)};
    j.aligned = all_aligned16(dev_bufs, nranks);
    cudaStream_t s = (cudaStream_t)stream_;
    cudaError_t e;
    if ((e = cudaEventRecord(hp->start, s)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaStreamWaitEvent(hp->up, hp->start, 0)) != cudaSuccess) return cuda_fail(e);
    for (size_t k = 0; k < starts.size(); ++k) {
      const int64_t a = starts[k], b = k + 1 < starts.size() ? starts[k + 1] : count;
      const size_t off = (size_t)a * es, bytes = (size_t)(b - a) * es;
      for (int r = 0; r < nranks; ++r)
        if ((e = cudaMemcpyAsync(static_cast<char*>(dev_bufs[r]) + off, static_cast<const char*>(host_bufs[r]) + off,
                                 bytes, cudaMemcpyHostToDevice, hp->up)) != cudaSuccess)
          return cuda_fail(e);
      if ((e = cudaEventRecord(hp->uploaded, hp->up)) != cudaSuccess) return cuda_fail(e);
      if ((e = cudaStreamWaitEvent(s, hp->uploaded, 0)) != cudaSuccess) return cuda_fail(e);
      TableBuilder tb{nranks, {}, {}};
      const int row = tb.add_row(dev_bufs);
      if (algo == AR_NAIVE) {
        tb.add_seg(row, a, b, nranks - 1);
      } else if (algo == AR_DBTREE) {
        tb.add_seg(row, a, std::min(b, count / 2), 0);
        tb.add_seg(row, std::max(a, count / 2), b, 1);
      } else {
        for (int c = 0; c < nranks; ++c)
          tb.add_seg(row, std::max(a, chunk_lo(count, nranks, c)), std::min(b, chunk_lo(count, nranks, c + 1)), c);
      }
      if ((rc = tb.for_each_table([&](SegTable& t) { return run_table(j, t, s); }))) return rc;
      if ((e = cudaEventRecord(hp->reduced, s)) != cudaSuccess) return cuda_fail(e);
      if ((e = cudaStreamWaitEvent(hp->down, hp->reduced, 0)) != cudaSuccess) return cuda_fail(e);
      for (int r = 0; r < nranks; ++r)
        if ((e = cudaMemcpyAsync(static_cast<char*>(host_bufs[r]) + off, static_cast<const char*>(dev_bufs[r]) + off,
                                 bytes, cudaMemcpyDeviceToHost, hp->down)) != cudaSuccess)
          return cuda_fail(e);
    }
    if ((e = cudaEventRecord(hp->done, hp->down)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaStreamWaitEvent(s, hp->done, 0)) != cudaSuccess) return cuda_fail(e);
    return AR_OK;
  });
}

int ar_allreduce_int8_ef(void* const* grads, void* const* residuals, int nranks, int64_t count, ar_op op,
                         ar_stream_t stream) {
  return guarded([&]() -> int {
    int rc = check_common(nranks, count, AR_F32, op, AR_RING);
    if (rc) return rc;
    if (op == AR_MAX) return AR_ERR_UNSUPPORTED;
    if (!grads || !residuals) return AR_ERR_INVALID_ARG;
    if (count == 0) return AR_OK;  // nothing is accessed
    std::vector<Range> rs;
    for (int r = 0; r < nranks; ++r) {
      rs.push_back({(uintptr_t)grads[r], (uintptr_t)grads[r] + (uintptr_t)count * 4});
      rs.push_back({(uintptr_t)residuals[r], (uintptr_t)residuals[r] + (uintptr_t)count * 4});
    }
    if ((rc = check_ranges(rs, 4))) return rc;
    if (count == 0) return AR_OK;
    ar::Int8Args a;
    memset(&a, 0, sizeof(a));
    for (int r = 0; r < nranks; ++r) {
      a.x[r] = static_cast<float*>(grads[r]);
      a.e[r] = static_cast<float*>(residuals[r]);
    }
    a.count = count;
    a.nranks = nranks;
    a.avg = op == AR_AVG ? 1 : 0;
    a.vec = all_aligned16(grads, nranks) && all_aligned16(residuals, nranks) ? 1 : 0;
    a.fn = (float)nranks;
    cudaError_t e = ar::launch_int8_ef(a, (cudaStream_t)stream);
    return e == cudaSuccess ? AR_OK : cuda_fail(e);
  });
}

int ar_chunk_range(int64_t count, int nranks, int c, int64_t* lo, int64_t* hi) {
  if (count < 0 || nranks < 1 || c < 0 || c >= nranks || !lo || !hi) return AR_ERR_INVALID_ARG;
  *lo = chunk_lo(count, nranks, c);
  *hi = chunk_lo(count, nranks, c + 1);
  return AR_OK;
}

int ar_bucket_plan(const int64_t* counts, int ntensors, ar_dtype dtype, int64_t cap_bytes, int32_t* bucket_of_tensor,
                   int64_t* offset_in_bucket, int64_t* bucket_count, int32_t* nbuckets) {
  return guarded([&]() -> int {
    if (ntensors < 0 || cap_bytes <= 0 || dtype < AR_F32 || dtype > AR_F16 || !nbuckets) return AR_ERR_INVALID_ARG;
    if (ntensors > 0 && (!counts || !bucket_of_tensor || !offset_in_bucket || !bucket_count)) return AR_ERR_INVALID_ARG;
    return plan_buckets(counts, ntensors, dtype, cap_bytes, bucket_of_tensor, offset_in_bucket, bucket_count, nbuckets);
  });
}

int ar_bucketed_allreduce(void* const* grads, const int64_t* counts, int ntensors, int nranks, ar_dtype dtype,
                          ar_op op, ar_algo algo, int64_t bucket_cap_bytes, void* const* workspace,
                          int64_t workspace_bytes, ar_stream_t stream_) {
  return guarded([&]() -> int {
    cudaStream_t stream = (cudaStream_t)stream_;
    int rc = check_common(nranks, 0, dtype, op, algo);
    if (rc) return rc;
    if (algo == AR_NAIVE || algo == AR_DBTREE || algo == AR_BINOMIAL_STEPWISE) return AR_ERR_UNSUPPORTED;
    if (ntensors < 0 || bucket_cap_bytes <= 0) return AR_ERR_INVALID_ARG;
    if (ntensors == 0) return AR_OK;
    if (!grads || !counts) return AR_ERR_INVALID_ARG;
    const int es = esize_of(dtype);
    std::vector<int32_t> bucket_of(ntensors);
    std::vector<int64_t> offset(ntensors), bcount(ntensors);
    int32_t nb = 0;
    if ((rc = plan_buckets(counts, ntensors, dtype, bucket_cap_bytes, bucket_of.data(), offset.data(), bcount.data(),
                           &nb)))
      return rc;
    {
      std::vector<Range> rs;
      for (int r = 0; r < nranks; ++r)
        for (int t = 0; t < ntensors; ++t) {
          if (counts[t] == 0) continue;
          uintptr_t p = (uintptr_t)grads[(size_t)r * ntensors + t];
          rs.push_back({p, p + (uintptr_t)counts[t] * es});
        }
      if ((rc = check_ranges(rs, es))) return rc;
    }
    if (nranks == 1) return AR_OK;
    const bool avg = op == AR_AVG;
    // row t of the pointer table: tensor t of every rank
    std::vector<void*> row(nranks);
    auto tensor_row = [&](int t) {
      for (int r = 0; r < nranks; ++r) row[r] = grads[(size_t)r * ntensors + t];
      return row.data();
    };

    if (!workspace) {
      // Fused: no packing; one pass reads and writes every gradient element once.
      TableBuilder tb{nranks, {}, {}};
      const bool vec = add_bucket_rows(tb, grads, counts, ntensors, nranks, bucket_of.data(), offset.data(),
                                       bcount.data(), [](int) { return true; });
      Job j{dtype, op, algo, 3, avg, vec};
      return tb.for_each_table([&](SegTable& t) { return run_table(j, t, stream); });
    }

    // Literal: pack -> AllReduce the flat buckets -> unpack.
    int64_t total = 0, largest = 0;
    std::vector<int64_t> base(nb);
    for (int b = 0; b < nb; ++b) {
      base[b] = total;
      total += bcount[b];
      largest = std::max(largest, bcount[b]);
    }
    if (workspace_bytes < largest * es) return AR_ERR_INVALID_ARG;
    {
      std::vector<Range> rs;
      for (int r = 0; r < nranks; ++r) {
        uintptr_t p = (uintptr_t)workspace[r];
        rs.push_back({p, p + (uintptr_t)workspace_bytes});
      }
      for (int r = 0; r < nranks; ++r)
        for (int t = 0; t < ntensors; ++t) {
          if (counts[t] == 0) continue;
          uintptr_t p = (uintptr_t)grads[(size_t)r * ntensors + t];
          rs.push_back({p, p + (uintptr_t)counts[t] * es});
        }
      if ((rc = check_ranges(rs, es))) return rc;
    }
    const bool whole = workspace_bytes >= total * es;
    const bool ws_aligned = all_aligned16(workspace, nranks);

    // buckets [b0, b1) at once: pack them, reduce them, unpack them
    auto run_buckets = [&](int b0, int b1) -> int {
      const int64_t shift = base[b0];  // packed offset of bucket b0 in the workspace
      auto copy = [&](int to_packed) -> int {
        TableBuilder cb{nranks, {}, {}};
        for (int t = 0; t < ntensors; ++t) {
          if (counts[t] == 0 || bucket_of[t] < b0 || bucket_of[t] >= b1) continue;
          void** rp = tensor_row(t);
          const int64_t aux = base[bucket_of[t]] - shift + offset[t];
          const bool v = all_aligned16(rp, nranks) && ws_aligned && (aux * es) % 16 == 0;
          const int rw = cb.add_row(rp);
          cb.add_seg(rw, 0, counts[t], v ? 1 : 0, aux);
        }
        ar::CopyArgs ca;
        for (int r = 0; r < nranks; ++r) ca.packed[r] = workspace[r];
        ca.to_packed = to_packed;
        ca.esize = es;
        return cb.for_each_table([&](SegTable& t) {
          ca.tab = t;
          cudaError_t e = ar::launch_copy(ca, stream);
          return e == cudaSuccess ? AR_OK : cuda_fail(e);
        });
      };
      auto reduce = [&]() -> int {
        TableBuilder tb{nranks, {}, {}};
        bool vec = ws_aligned;
        std::vector<void*> wrow(nranks);
        for (int b = b0; b < b1; ++b) {
          for (int r = 0; r < nranks; ++r) wrow[r] = static_cast<char*>(workspace[r]) + (base[b] - shift) * es;
          vec = vec && all_aligned16(wrow.data(), nranks);
          const int rw = tb.add_row(wrow.data());
          for (int c = 0; c < nranks; ++c)
            tb.add_seg(rw, chunk_lo(bcount[b], nranks, c), chunk_lo(bcount[b], nranks, c + 1), c);
        }
        Job j{dtype, op, algo, 3, avg, vec};
        return tb.for_each_table([&](SegTable& t) { return run_table(j, t, stream); });
      };
      int r2 = copy(1);
      if (!r2) r2 = reduce();
      if (!r2) r2 = copy(0);
      return r2;
    };

    if (whole) return run_buckets(0, nb);
    for (int b = 0; b < nb; ++b)
      if ((rc = run_buckets(b, b + 1))) return rc;
    return AR_OK;
  });
}

int ar_reducer_create(void* const* grads, const int64_t* counts, int ntensors, int nranks, ar_dtype dtype, ar_op op,
                      ar_algo algo, int64_t bucket_cap_bytes, ar_stream_t comm_stream, ar_reducer** out) {
  return guarded([&]() -> int {
    if (!out) return AR_ERR_INVALID_ARG;
    *out = nullptr;
    int rc = check_common(nranks, 0, dtype, op, algo);
    if (rc) return rc;
    if (algo == AR_NAIVE || algo == AR_DBTREE || algo == AR_BINOMIAL_STEPWISE) return AR_ERR_UNSUPPORTED;
    if (ntensors < 1 || bucket_cap_bytes <= 0 || !grads || !counts) return AR_ERR_INVALID_ARG;
    const int es = esize_of(dtype);
    ar_reducer* red = new ar_reducer;
    red->nranks = nranks;
    red->ntensors = ntensors;
    red->comm = (cudaStream_t)comm_stream;
    red->bucket_of.resize(ntensors);
    std::vector<int64_t> offset(ntensors), bcount(ntensors);
    int32_t nb = 0;
    if ((rc = plan_buckets(counts, ntensors, dtype, bucket_cap_bytes, red->bucket_of.data(), offset.data(),
                           bcount.data(), &nb))) {
      reducer_free(red);
      return rc;
    }
    {
      std::vector<Range> rs;
      for (int r = 0; r < nranks; ++r)
        for (int t = 0; t < ntensors; ++t) {
          if (counts[t] == 0) continue;
          uintptr_t p = (uintptr_t)grads[(size_t)r * ntensors + t];
          rs.push_back({p, p + (uintptr_t)counts[t] * es});
        }
      if ((rc = check_ranges(rs, es))) {
        reducer_free(red);
        return rc;
      }
    }
    red->nbuckets = nb;
    red->left.resize(nb);
    red->ready.resize(ntensors);
    red->tables.resize(nb);
    red->ready_ev.assign(nb, nullptr);
    bool vec = true;
    for (int b = 0; b < nb && nranks > 1; ++b) {
      TableBuilder tb{nranks, {}, {}};
      vec = add_bucket_rows(tb, grads, counts, ntensors, nranks, red->bucket_of.data(), offset.data(), bcount.data(),
                            [&](int t) { return red->bucket_of[t] == b; }) && vec;
      rc = tb.for_each_table([&](SegTable& t) {
        red->tables[b].push_back(t);
        return AR_OK;
      });
      if (rc) {
        reducer_free(red);
        return rc;
      }
      red->ntables += (int64_t)red->tables[b].size();
    }
    red->job = Job{dtype, op, algo, 3, op == AR_AVG, vec};
    cudaError_t e = cudaSuccess;
    for (int b = 0; b < nb && e == cudaSuccess; ++b) e = cudaEventCreateWithFlags(&red->ready_ev[b], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&red->done_ev, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      reducer_free(red);
      return cuda_fail(e);
    }
    reducer_reset(red);
    *out = red;
    return AR_OK;
  });
}

int ar_reducer_mark_ready(ar_reducer* red, int tensor, ar_stream_t compute_stream) {
  return guarded([&]() -> int {
    if (!red || tensor < 0 || tensor >= red->ntensors || red->ready[tensor]) return AR_ERR_INVALID_ARG;
    red->ready[tensor] = 1;
    const int b = red->bucket_of[tensor];
    cudaError_t e;
    if (--red->left[b] == 0 && (e = cudaEventRecord(red->ready_ev[b], (cudaStream_t)compute_stream)) != cudaSuccess)
      return cuda_fail(e);
    // start every bucket whose turn has come
    while (red->next < red->nbuckets && red->left[red->next] == 0) {
      const int nb = red->next++;
      if ((e = cudaStreamWaitEvent(red->comm, red->ready_ev[nb], 0)) != cudaSuccess) return cuda_fail(e);
      for (SegTable& t : red->tables[nb]) {
        int rc = run_table(red->job, t, red->comm);
        if (rc) return rc;
      }
    }
    return AR_OK;
  });
}

int ar_reducer_finish(ar_reducer* red, ar_stream_t compute_stream) {
  return guarded([&]() -> int {
    if (!red) return AR_ERR_INVALID_ARG;
    if (red->next < red->nbuckets) return AR_ERR_INVALID_ARG;  // some gradient was never marked ready
    cudaError_t e;
    if ((e = cudaEventRecord(red->done_ev, red->comm)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaStreamWaitEvent((cudaStream_t)compute_stream, red->done_ev, 0)) != cudaSuccess) return cuda_fail(e);
    reducer_reset(red);
    return AR_OK;
  });
}

int ar_reducer_destroy(ar_reducer* red) {
  return guarded([&]() -> int {
    if (!red) return AR_ERR_INVALID_ARG;
    reducer_free(red);
    return AR_OK;
  });
}

int ar_reducer_buckets(const ar_reducer* red) { return red ? red->nbuckets : AR_ERR_INVALID_ARG; }

int ar_reducer_set_max_blocks(ar_reducer* red, int max_blocks) {
  if (!red || max_blocks < 0) return AR_ERR_INVALID_ARG;
  red->job.max_grid = max_blocks;
  return AR_OK;
}

int ar_plan_create(int kind, void* const* bufs, int nranks, int64_t count, ar_dtype dtype, ar_op op, ar_algo algo,
                   int root, ar_plan** out) {
  return guarded([&]() -> int {
    if (!out) return AR_ERR_INVALID_ARG;
    *out = nullptr;
    int phases = 3;
    switch (kind) {
      case AR_PLAN_ALLREDUCE: root = -1; break;
      case AR_PLAN_REDUCE_SCATTER: phases = 1, root = -1; break;
      case AR_PLAN_ALL_GATHER: phases = 2, root = -1, op = AR_SUM; break;
      case AR_PLAN_REDUCE:
        if (root < 0 || root >= nranks) return AR_ERR_INVALID_ARG;
        if (is_stepwise(algo)) return AR_ERR_UNSUPPORTED;
        break;
      default: return AR_ERR_INVALID_ARG;
    }
    TableBuilder tb{nranks, {}, {}};
    Job j{};
    bool empty = false;
    int rc = build_collective(bufs, nranks, count, dtype, op, algo, phases, root, tb, j, &empty);
    if (rc) return rc;
    ar_plan* plan = new ar_plan;
    plan->job = j;
    if (!empty) {
      rc = tb.for_each_table([&](SegTable& t) {
        plan->tables.push_back(t);
        return AR_OK;
      });
      if (rc) {
        delete plan;
        return rc;
      }
    }
    *out = plan;
    return AR_OK;
  });
}

int ar_plan_run(const ar_plan* plan, ar_stream_t stream) {
  return guarded([&]() -> int {
    if (!plan) return AR_ERR_INVALID_ARG;
    for (const SegTable& t : plan->tables) {
      SegTable copy = t;  // the launchers fill in the tile layout
      int rc = run_table(plan->job, copy, (cudaStream_t)stream);
      if (rc) return rc;
    }
    return AR_OK;
  });
}

int ar_plan_destroy(ar_plan* plan) {
  return guarded([&]() -> int {
    if (!plan) return AR_ERR_INVALID_ARG;
    delete plan;
    return AR_OK;
  });
}

int ar_device_status(ar_stream_t stream, int* status) {
  return guarded([&]() -> int {
    if (!status) return AR_ERR_INVALID_ARG;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e);
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e);
    *status = AR_OK;
    ar::SyncBlock* sb = nullptr;
    unsigned long long ctx = 0;
    int rc = context_id(&ctx);
    if (rc) return rc;
    {
      // a block from a context that no longer exists holds no status
      std::lock_guard<std::mutex> lk(g_sync_mu);
      if (dev >= 0 && dev < 256 && g_sync_ctx[dev] == ctx) sb = g_sync[dev];
    }
    if (!sb) return AR_OK;
    int v = 0;
    if ((e = cudaMemcpy(&v, &sb->status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaMemset(&sb->status, 0, sizeof(int))) != cudaSuccess) return cuda_fail(e);
    *status = v;
    return AR_OK;
  });
}

int ar_set_barrier_timeout_ns(int64_t ns) {
  g_timeout_ns.store(ns > 0 ? ns : 1000000000LL);
  return AR_OK;
}

int ar_debug_skip_barrier(int barrier) {
  g_skip_barrier.store(barrier < 0 ? -1 : barrier);
  return AR_OK;
}

int ar_last_cuda_error(void) { return (int)g_last_cuda; }

const char* ar_strerror(int status) {
  switch (status) {
    case AR_OK: return "AR_OK";
    case AR_ERR_INVALID_ARG: return "AR_ERR_INVALID_ARG: invalid argument";
    case AR_ERR_UNSUPPORTED: return "AR_ERR_UNSUPPORTED: unsupported combination";
    case AR_ERR_CUDA: return "AR_ERR_CUDA: a CUDA call failed";
    case AR_ERR_TIMEOUT: return "AR_ERR_TIMEOUT: a step-wise barrier wait ran out";
    case AR_ERR_NO_DEVICE: return "AR_ERR_NO_DEVICE: no usable CUDA device";
    case AR_ERR_HOST: return "AR_ERR_HOST: host-side failure (out of host memory)";
    case AR_ERR_TOO_LARGE: return "AR_ERR_TOO_LARGE: descriptor tables too large";
    default: return "unknown ar_status";
  }
}

int ar_version(void) { return 100; }

int64_t ar_kernel_launches(void) { return ar::g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
