// Host-side launchers, one per operation (defined in ops_<op>.cu).
#pragma once
#include <cuda_runtime.h>

namespace tile {
constexpr int kMaxDevices = 64;

// Row-kernel operations (template argument OP of the row kernels).
enum { OP_RESLN = 0, OP_LN = 1, OP_RMS = 2, OP_SOFTMAX = 3, OP_SUM = 4, OP_MINMAX = 5 };

// Arguments of one row-kernel launch.  x, r: [rows][width] inputs of the
// launch's element type (FP32, BF16 or FP16; r: residual LayerNorm only).
// gamma, beta: optional FP32 per-column scale and shift applied after
// LayerNorm / RMSNorm (NULL = none).  y: [rows][width] output of the element
// type, or [rows] FP32 row sums / row minima; y2: [rows] FP32 row maxima.
// status: the launching op's device error word (filled by the launcher).
struct RowArgs {
    const void *x;
    const void *r;
    const float *gamma;
    const float *beta;
    void *y;
    float *y2;
    long long rows;
    int width;
    float eps;
    unsigned int *status;
    float inv_n;           // 1 / width rounded to FP32 (the 2-byte kernels multiply by it)
};

// Arguments of one backward-kernel launch (bwd_kernel.cuh).  x: forward
// input (LayerNorm / RMSNorm) or forward output y (softmax); dy: upstream
// gradient; dx: input gradient; all [rows][width] of the launch's element
// type (FP32, BF16 or FP16).  gamma: optional FP32 [width]; stats: optional
// FP32 [rows][2] (mean, rstd) output.
struct BwdArgs {
    const void *x;
    const void *dy;
    const float *gamma;
    void *dx;
    float *stats;
    long long rows;
    int width;
    float eps;
    unsigned int *status;
    float inv_n;           // 1 / width rounded to FP32 (the 2-byte kernels multiply by it)
};

// Shared-memory-staged row kernel (staged.cu): kernel_op is OP_RESLN, OP_LN,
// OP_RMS or OP_SOFTMAX; elem the element type (ELEM_F32, ELEM_BF16,
// ELEM_F16, the values of the ABI's TILE_DTYPE_*); plan_id one of
// TILE_STAGED_LIST.
enum { ELEM_F32 = 0, ELEM_BF16 = 1, ELEM_F16 = 2 };
cudaError_t launch_staged(int kernel_op, int elem, int plan_id, RowArgs args,
                          cudaStream_t stream);
cudaError_t status_staged(unsigned int *value, cudaStream_t stream);
// R-rows-per-CTA kernel (multi.cu): kernel_op as launch_staged; plan_id one
// of TILE_MULTI_LIST.
cudaError_t launch_multi(int kernel_op, int elem, int plan_id, RowArgs args,
                         cudaStream_t stream);
cudaError_t status_multi(unsigned int *value, cudaStream_t stream);
// The staged kernel with each CTA's first copy withheld and the barrier
// waits limited to `spin_limit` polls (tile_test_staged_wait_timeout).
cudaError_t launch_staged_withheld(int kernel_op, int elem, int plan_id, RowArgs args,
                                   unsigned int spin_limit, cudaStream_t stream);

// Backward kernel ops (bwd_kernel.cuh).
enum { BWD_LN_OP = 0, BWD_RMS_OP = 1, BWD_SOFTMAX_OP = 2 };
cudaError_t launch_backward(int op, int plan_id, BwdArgs args, cudaStream_t stream);
cudaError_t status_backward(unsigned int *value, cudaStream_t stream);
cudaError_t launch_backward_bf16(int op, int plan_id, BwdArgs args, cudaStream_t stream);
cudaError_t status_backward_bf16(unsigned int *value, cudaStream_t stream);
cudaError_t launch_backward_f16(int op, int plan_id, BwdArgs args, cudaStream_t stream);
cudaError_t status_backward_f16(unsigned int *value, cudaStream_t stream);

// Parameter gradients (param_grad.cu): column sums of dy * xhat and dy over
// param_blocks(rows) fixed row blocks into ws [nblk][2][width], then summed.
int param_blocks(long long rows);
// x, dy: [rows][width] of element type elem (ELEM_F32, ELEM_BF16, ELEM_F16).
cudaError_t launch_param_grad(int elem, const void *x, const void *dy, const float *stats,
                              float *dgamma, float *dbeta, long long rows, int width, float *ws,
                              cudaStream_t stream);
cudaError_t status_param_grad(unsigned int *value, cudaStream_t stream);

// Largest register stripe per input (floats per thread) of a backward plan:
// two stripes are held, so plans above it (K * elements per vector) are not
// built for backward.
constexpr int kMaxStripeBwd = 32;
// The same budget for the raw-word kernel of 2-byte rows of 16-byte vectors,
// in elements per stripe (two 2-byte elements per register: 64 elements are
// 32 registers per stripe).
constexpr int kMaxStripeBwdRaw = 64;

#define TILE_DECLARE_OP(name)                                                            \
    cudaError_t launch_##name(int plan_id, RowArgs args, cudaStream_t stream);          \
    cudaError_t status_##name(unsigned int *value, cudaStream_t stream);
TILE_DECLARE_OP(residual_layernorm)
TILE_DECLARE_OP(layernorm)
TILE_DECLARE_OP(rmsnorm)
TILE_DECLARE_OP(softmax)
TILE_DECLARE_OP(row_sum)
TILE_DECLARE_OP(row_minmax)
TILE_DECLARE_OP(residual_layernorm_bf16)
TILE_DECLARE_OP(layernorm_bf16)
TILE_DECLARE_OP(rmsnorm_bf16)
TILE_DECLARE_OP(softmax_bf16)
TILE_DECLARE_OP(row_sum_bf16)
TILE_DECLARE_OP(row_minmax_bf16)
TILE_DECLARE_OP(residual_layernorm_f16)
TILE_DECLARE_OP(layernorm_f16)
TILE_DECLARE_OP(rmsnorm_f16)
TILE_DECLARE_OP(softmax_f16)
TILE_DECLARE_OP(row_sum_f16)
TILE_DECLARE_OP(row_minmax_f16)
#undef TILE_DECLARE_OP

// Largest register stripe (floats per thread) a plan on 2-byte elements
// (BF16, FP16) may use: plans with K * 8 above it are not built for them.
constexpr int kMaxStripeBf16 = 64;

// Pointwise value/derivative pairs (pair_kernel.cu): kind 0 = sigmoid,
// 1 = tanh-approximate GELU, over n elements.
enum { PAIR_SIGMOID = 0, PAIR_GELU_TANH = 1 };
cudaError_t launch_pairs(int kind, const float *x, float *y, float *dy, long long n,
                         cudaStream_t stream);
cudaError_t status_pairs(unsigned int *value, cudaStream_t stream);

// Argument checks + launch of a pair kernel (the body of the pair entry points).
int run_pairs(int kind, const float *in, float *value, float *derivative, long long n,
              cudaStream_t stream);

// Check arguments, pick a plan and launch `op` on device buffers (the body of
// the four compute entry points).  select_rows > 0 picks the plan as for a
// call of that many rows (a chunk of a larger matrix takes the whole
// matrix's plan, so its results are bitwise those of a single call).
// Returns a TILE_* status.
int run_selected(int op, const float *in, const float *res, float *out, int rows, int width,
                 float eps, cudaStream_t stream, long long select_rows = 0);

// The argument checks of the host entry points that need no CUDA call (op,
// shape, eps, NULL buffers, output overlapping an input); a TILE_* status.
int check_host_args(int op, const float *h_in, const float *h_res, const float *h_out,
                    int rows, int width, float eps);

// The pipeline of tile_run_host_f32 over a given device workspace.
int run_host(int op, const float *h_in, const float *h_res, float *h_out, int rows, int width,
             float eps, void *d_work, size_t work_bytes, cudaStream_t stream);

// A launch failure injected on the host for tests (tile_inject_launch_failure):
// cudaSuccess, or the error the next launch attempt must report instead of
// launching.
cudaError_t injected_launch_failure();

// Whether 2-byte launches may take the whole-vector kernel forms (false
// while tile_test_force_general_kernels holds them on the general forms).
bool whole_vector_kernels();

// The cudaError_t behind the last TILE_ERR_CUDA on this host thread.
void set_last_cuda_error(int err);
int last_cuda_error();
}  // namespace tile
