// Backward row kernels on BF16 rows (FP32 arithmetic): every built plan (see bwd_inst.cuh).
#define TILE_BWD_T __nv_bfloat16
#define TILE_BWD_NAME _bf16
#include "bwd_inst.cuh"
