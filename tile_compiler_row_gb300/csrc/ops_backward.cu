// Backward row kernels on FP32 rows (FP32 arithmetic): every built plan (see bwd_inst.cuh).
#define TILE_BWD_T float
#define TILE_BWD_NAME 
#include "bwd_inst.cuh"
