// rmsnorm: every built plan (see ops_inst.cuh).
#define TILE_INST_OP tile::OP_RMS
#define TILE_INST_T float
#define TILE_INST_NAME rmsnorm
#include "ops_inst.cuh"
