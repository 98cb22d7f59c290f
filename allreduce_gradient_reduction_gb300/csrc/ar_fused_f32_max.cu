// Fused kernels for f32 max: one translation unit per (dtype, op) so the
// build compiles them in parallel.
#include "ar_fused.cuh"
AR_DEFINE_FUSED(launch_fused_f32_max, F32, MAX)
