// AllGather / Broadcast for rows whose buffers sit at different addresses
// modulo 16 (4- and 2-byte elements).
#include "ar_stage.cuh"
AR_DEFINE_STAGE_GATHER(launch_stage_gather4, F32)
AR_DEFINE_STAGE_GATHER(launch_stage_gather2, BF16)
