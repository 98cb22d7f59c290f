// Fused kernels for i32 rows whose buffers sit at different addresses modulo
// 16, sum: one translation unit per dtype and op, compiled in parallel.
#include "ar_stage.cuh"
AR_DEFINE_STAGE(launch_stage_i32_sum, I32, SUM)
