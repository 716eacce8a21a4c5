// Backward row kernels on FP16 rows (FP32 arithmetic): every built plan (see bwd_inst.cuh).
#define TILE_BWD_T __half
#define TILE_BWD_NAME _f16
#include "bwd_inst.cuh"
