// row_sum: every built plan (see ops_inst.cuh).
#define TILE_INST_OP tile::OP_SUM
#define TILE_INST_T float
#define TILE_INST_NAME row_sum
#include "ops_inst.cuh"
