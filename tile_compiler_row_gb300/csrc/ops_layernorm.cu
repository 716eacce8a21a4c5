// layernorm: every built plan (see ops_inst.cuh).
#define TILE_INST_OP tile::OP_LN
#define TILE_INST_T float
#define TILE_INST_NAME layernorm
#include "ops_inst.cuh"
