// Host-side launchers, one per operation (defined in ops_<op>.cu).
#pragma once
#include <cuda_runtime.h>

namespace tile {
constexpr int kMaxDevices = 64;

#define TILE_DECLARE_OP(name)                                                          \
    cudaError_t launch_##name(int plan_id, const float *x, const float *r, float *y,   \
                              long long rows, int width, float eps, cudaStream_t stream); \
    cudaError_t status_##name(unsigned int *value, cudaStream_t stream);
TILE_DECLARE_OP(residual_layernorm)
TILE_DECLARE_OP(layernorm)
TILE_DECLARE_OP(rmsnorm)
TILE_DECLARE_OP(softmax)
#undef TILE_DECLARE_OP
}  // namespace tile
