// Fused kernels for f32 rows whose buffers sit at different addresses modulo
// 16 (sum and max): one translation unit per dtype, compiled in parallel.
#include "ar_fused.cuh"
AR_DEFINE_FUSED_SHIFT(launch_fused_shift_f32_sum, F32, SUM)
AR_DEFINE_FUSED_SHIFT(launch_fused_shift_f32_max, F32, MAX)
