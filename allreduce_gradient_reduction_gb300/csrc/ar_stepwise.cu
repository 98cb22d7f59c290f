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
  // opened once per device to the largest shared memory the path uses
  static std::atomic<bool> opened[256];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
  if (!opened[dev].load()) {
    e = cudaFuncSetAttribute(stepwise_smem_kernel<DT, OP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemStepBytes);
    if (e != cudaSuccess) return e;
    opened[dev].store(true);
  }
  const size_t bytes = (size_t)smem_step_bytes(a.nranks, a.count, ElemSize<DT>::value);
  stepwise_smem_kernel<DT, OP><<<1, kSmemStepBlock, bytes, stream>>>(a);
  count_launch();
  return cudaGetLastError();
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
