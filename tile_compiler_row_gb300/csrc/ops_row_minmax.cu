// row_minmax: every built plan (see ops_inst.cuh).
#define TILE_INST_OP tile::OP_MINMAX
#define TILE_INST_T float
#define TILE_INST_NAME row_minmax
#include "ops_inst.cuh"
