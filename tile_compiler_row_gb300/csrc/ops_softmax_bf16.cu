// softmax on BF16 rows (FP32 arithmetic): every built plan (see ops_inst.cuh).
#define TILE_INST_OP tile::OP_SOFTMAX
#define TILE_INST_T __nv_bfloat16
#define TILE_INST_NAME softmax_bf16
#include "ops_inst.cuh"
