// Fused kernels for f16 max, small launch tables (see ar_fused_f16_max.cu).
#include "ar_fused.cuh"

namespace ar {
cudaError_t launch_fused_f16_max(int order, SmallFusedArgs& a, cudaStream_t s) {
  return launch_fused_typed<F16, MAX>(order, a, s);
}
}  // namespace ar
