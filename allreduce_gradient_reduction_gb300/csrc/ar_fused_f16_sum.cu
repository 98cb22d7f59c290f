// Fused kernels for f16 sum: one translation unit per (dtype, op) so the
// build compiles them in parallel.
#include "ar_fused.cuh"
AR_DEFINE_FUSED(launch_fused_f16_sum, F16, SUM)
