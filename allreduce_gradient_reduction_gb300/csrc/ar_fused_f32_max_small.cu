// Fused kernels for f32 max, small launch tables (see ar_fused_f32_max.cu).
#include "ar_fused.cuh"

namespace ar {
cudaError_t launch_fused_f32_max(int order, SmallFusedArgs& a, cudaStream_t s) {
  return launch_fused_typed<F32, MAX>(order, a, s);
}
}  // namespace ar
