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

// Check arguments, pick a plan and launch `op` on device buffers (the body of
// the four compute entry points).  Returns a TILE_* status.
int run_selected(int op, const float *in, const float *res, float *out, int rows, int width,
                 float eps, cudaStream_t stream);

// The pipeline of tile_run_host_f32 over a given device workspace.
int run_host(int op, const float *h_in, const float *h_res, float *h_out, int rows, int width,
             float eps, void *d_work, size_t work_bytes, cudaStream_t stream);

// The cudaError_t behind the last TILE_ERR_CUDA on this host thread.
void set_last_cuda_error(int err);
int last_cuda_error();
}  // namespace tile
