// Fused kernels for bf16 max: one translation unit per (dtype, op) so the
// build compiles them in parallel.
#include "ar_fused.cuh"
AR_DEFINE_FUSED(launch_fused_bf16_max, BF16, MAX)
