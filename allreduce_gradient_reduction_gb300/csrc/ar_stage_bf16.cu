// Fused kernels for bf16 rows whose buffers sit at different addresses modulo
// 16 (sum and max): one translation unit per dtype, compiled in parallel.
#include "ar_stage.cuh"
AR_DEFINE_STAGE(launch_stage_bf16_sum, BF16, SUM)
AR_DEFINE_STAGE(launch_stage_bf16_max, BF16, MAX)
AR_DEFINE_STAGE_GATHER(launch_stage_gather2, BF16)
