// Fused kernels for f16 max, large launch tables.  The maximum's kernels take
// longest to compile, so each table form has its own translation unit and the
// build compiles them in parallel.
#include "ar_fused.cuh"

namespace ar {
cudaError_t launch_fused_f16_max(int order, FusedArgs& a, cudaStream_t s) {
  return launch_fused_typed<F16, MAX>(order, a, s);
}
}  // namespace ar
