// layernorm on FP16 rows (FP32 arithmetic): every built plan (see ops_inst.cuh).
#define TILE_INST_OP tile::OP_LN
#define TILE_INST_T __half
#define TILE_INST_NAME layernorm_f16
#include "ops_inst.cuh"
