// Fused kernels for i32 sum: one translation unit per (dtype, op) so the
// build compiles them in parallel.
#include "ar_fused.cuh"
AR_DEFINE_FUSED(launch_fused_i32_sum, I32, SUM)
