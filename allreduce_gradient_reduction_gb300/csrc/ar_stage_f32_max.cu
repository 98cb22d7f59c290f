// Fused kernels for f32 rows whose buffers sit at different addresses modulo
// 16, max: one translation unit per dtype and op, compiled in parallel.
#include "ar_stage.cuh"
AR_DEFINE_STAGE(launch_stage_f32_max, F32, MAX)
