// Fused kernels for bf16 rows whose buffers sit at different addresses modulo
// 16 (sum and max): one translation unit per dtype, compiled in parallel.
#include "ar_fused.cuh"
AR_DEFINE_FUSED_SHIFT(launch_fused_shift_bf16_sum, BF16, SUM)
AR_DEFINE_FUSED_SHIFT(launch_fused_shift_bf16_max, BF16, MAX)
