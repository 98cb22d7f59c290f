// Fused kernels for f16 rows whose buffers sit at different addresses modulo
// 16, max: one translation unit per dtype and op, compiled in parallel.
#include "ar_stage.cuh"
AR_DEFINE_STAGE(launch_stage_f16_max, F16, MAX)
