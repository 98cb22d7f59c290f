// Step-wise kernel instantiations and their cooperative launcher.
#include <atomic>

#include "ar_fused.cuh"
#include "ar_stepwise.cuh"

namespace ar {

template <int DT, int OP, bool VECTOR>
static cudaError_t launch_step_typed(StepArgs& a, cudaStream_t stream) {
  constexpr int VEC = VECTOR ? 16 / ElemSize<DT>::value : 1;
  if (fill_tiles(a.tab, VEC, (int64_t)kStepBlock * kStepUnroll, VECTOR) == 0) return cudaSuccess;
  static const int bps = blocks_per_sm(stepwise_kernel<DT, OP, VECTOR>, kStepBlock);
  // persistent: every block must be resident at once (the launch checks it);
  // more blocks than the widest phase has tiles would only wait at barriers
  int64_t widest = a.tab.ntiles * (a.order == TREE || a.order == BINOMIAL ? a.tab.nranks / 2 : 1);
  int64_t grid = (int64_t)bps * sm_count();
  if (grid > widest) grid = widest;
  if (grid < 1) grid = 1;
  void* params[] = {&a};
  count_launch();
  return cudaLaunchCooperativeKernel((const void*)stepwise_kernel<DT, OP, VECTOR>, dim3((unsigned)grid),
                                     dim3(kStepBlock), params, 0, stream);
}

template <int DT, int OP>
static cudaError_t launch_step_op(bool vec, StepArgs& a, cudaStream_t s) {
  return vec ? launch_step_typed<DT, OP, true>(a, s) : launch_step_typed<DT, OP, false>(a, s);
}

template <int DT, int OP>
static cudaError_t launch_smem_typed(SmemStepArgs& a, cudaStream_t stream) {
  // opened once per context to the largest shared memory the path uses
  static std::atomic<unsigned long long> opened[256];
  cudaError_t e = open_kernel(reinterpret_cast<const void*>(stepwise_smem_kernel<DT, OP>), (int)kSmemStepBytes,
                              false, opened);
  if (e != cudaSuccess) return e;
  const size_t bytes = (size_t)smem_step_bytes(a.nranks, a.count, ElemSize<DT>::value);
  stepwise_smem_kernel<DT, OP><<<1, kSmemStepBlock, bytes, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

// ---- cluster form -----------------------------------------------------------

template <int DT, int OP>
static cudaError_t launch_cluster_typed(SmemStepArgs& a, int csize, cudaStream_t stream) {
  static std::atomic<unsigned long long> opened[256];  // once per context
  auto kernel = stepwise_cluster_kernel<DT, OP>;
  cudaError_t e = open_kernel(reinterpret_cast<const void*>(kernel), (int)kSmemStepBytes, true, opened);
  if (e != cudaSuccess) return e;
  const int es = ElemSize<DT>::value;
  const int64_t stride = (a.count * es + 15) / 16 * 16;
  const size_t bytes = (size_t)(((int64_t)a.nranks + csize - 1) / csize * stride);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)csize);
  cfg.blockDim = dim3(kClusterStepBlock);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)csize;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

// The largest cluster the cluster kernel can be launched with on the current
// device with a full shared-memory budget per block (0 if none).
int cluster_step_max_size() {
  static std::atomic<int> cached[256];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return 0;
  int v = cached[dev].load();
  if (v) return v > 0 ? v : 0;
  auto kernel = stepwise_cluster_kernel<F32, SUM>;
  int best = -1;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemStepBytes) == cudaSuccess &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16);
    cfg.blockDim = dim3(kClusterStepBlock);
    cfg.dynamicSmemBytes = (size_t)kSmemStepBytes;
    int sz = 0;
    if (cudaOccupancyMaxPotentialClusterSize(&sz, (const void*)kernel, &cfg) == cudaSuccess && sz >= 2) best = sz;
  }
  (void)cudaGetLastError();  // a refused query leaves nothing behind
  cached[dev].store(best);
  return best > 0 ? best : 0;
}

cudaError_t launch_stepwise_cluster(int dtype, int op, SmemStepArgs& a, int csize, cudaStream_t s) {
  switch (dtype * 2 + op) {
    case F32 * 2 + SUM: return launch_cluster_typed<F32, SUM>(a, csize, s);
    case F32 * 2 + MAX: return launch_cluster_typed<F32, MAX>(a, csize, s);
    case BF16 * 2 + SUM: return launch_cluster_typed<BF16, SUM>(a, csize, s);
    case BF16 * 2 + MAX: return launch_cluster_typed<BF16, MAX>(a, csize, s);
    case I32 * 2 + SUM: return launch_cluster_typed<I32, SUM>(a, csize, s);
    case I32 * 2 + MAX: return launch_cluster_typed<I32, MAX>(a, csize, s);
    case F16 * 2 + SUM: return launch_cluster_typed<F16, SUM>(a, csize, s);
    case F16 * 2 + MAX: return launch_cluster_typed<F16, MAX>(a, csize, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_stepwise_smem(int dtype, int op, SmemStepArgs& a, cudaStream_t s) {
  if (smem_step_bytes(a.nranks, a.count, (dtype == BF16 || dtype == F16) ? 2 : 4) > kSmemStepBytes)
    return cudaErrorInvalidValue;
  switch (dtype * 2 + op) {
    case F32 * 2 + SUM: return launch_smem_typed<F32, SUM>(a, s);
    case F32 * 2 + MAX: return launch_smem_typed<F32, MAX>(a, s);
    case BF16 * 2 + SUM: return launch_smem_typed<BF16, SUM>(a, s);
    case BF16 * 2 + MAX: return launch_smem_typed<BF16, MAX>(a, s);
    case I32 * 2 + SUM: return launch_smem_typed<I32, SUM>(a, s);
    case I32 * 2 + MAX: return launch_smem_typed<I32, MAX>(a, s);
    case F16 * 2 + SUM: return launch_smem_typed<F16, SUM>(a, s);
    case F16 * 2 + MAX: return launch_smem_typed<F16, MAX>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_stepwise(int dtype, int op, bool vec, StepArgs& a, cudaStream_t s) {
  switch (dtype * 2 + op) {
    case F32 * 2 + SUM: return launch_step_op<F32, SUM>(vec, a, s);
    case F32 * 2 + MAX: return launch_step_op<F32, MAX>(vec, a, s);
    case BF16 * 2 + SUM: return launch_step_op<BF16, SUM>(vec, a, s);
    case BF16 * 2 + MAX: return launch_step_op<BF16, MAX>(vec, a, s);
    case I32 * 2 + SUM: return launch_step_op<I32, SUM>(vec, a, s);
    case I32 * 2 + MAX: return launch_step_op<I32, MAX>(vec, a, s);
    case F16 * 2 + SUM: return launch_step_op<F16, SUM>(vec, a, s);
    case F16 * 2 + MAX: return launch_step_op<F16, MAX>(vec, a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ar
