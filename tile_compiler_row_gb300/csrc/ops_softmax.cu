// softmax: every built plan (see ops_inst.cuh).
#define TILE_INST_OP tile::OP_SOFTMAX
#define TILE_INST_T float
#define TILE_INST_NAME softmax
#include "ops_inst.cuh"
