// Fused kernels for f16 rows whose buffers sit at different addresses modulo
// 16 (sum and max): one translation unit per dtype, compiled in parallel.
#include "ar_stage.cuh"
AR_DEFINE_STAGE(launch_stage_f16_sum, F16, SUM)
AR_DEFINE_STAGE(launch_stage_f16_max, F16, MAX)
