// Fused kernels for f32 rows whose buffers sit at different addresses modulo
// 16 (sum and max): one translation unit per dtype, compiled in parallel.
#include "ar_stage.cuh"
AR_DEFINE_STAGE(launch_stage_f32_sum, F32, SUM)
AR_DEFINE_STAGE(launch_stage_f32_max, F32, MAX)
AR_DEFINE_STAGE_GATHER(launch_stage_gather4, F32)
