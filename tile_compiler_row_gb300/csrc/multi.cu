// Launchers of the R-rows-per-CTA kernel (multi_kernel.cuh) for the
// normalisers and softmax, FP32, BF16 and FP16, over the plans of plans.h
// (TILE_MULTI_LIST), plus their device error word.
#include <atomic>

#include "launch.h"
#include "multi_kernel.cuh"
#include "plans.h"

namespace tile {
namespace {

__device__ unsigned int g_status;   // device error word of the R-row kernels

unsigned int *status_address(cudaError_t *err) {
    static std::atomic<unsigned int *> cache[kMaxDevices];
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    unsigned int *p = cache[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        *err = cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_status);
        if (*err != cudaSuccess) return nullptr;
        cache[dev].store(p, std::memory_order_release);
    }
    return p;
}

template <int OP, class T, int S, int K, int R>
cudaError_t launch_one(RowArgs a, cudaStream_t stream) {
    constexpr int EV = 16 / sizeof(T);
    if constexpr (R * K * EV > 64) {
        (void)a;
        (void)stream;
        return cudaErrorInvalidValue;     // not built: stripe above 64 floats
    } else {
        cudaError_t err = cudaSuccess;
        a.status = status_address(&err);
        if (a.status == nullptr) return err;
        const long long grid = (a.rows + R - 1) / R;
        row_multi_kernel<OP, T, S, K, R>
            <<<static_cast<unsigned int>(grid), 32 * S, 0, stream>>>(a);
        return cudaGetLastError();
    }
}

template <int OP, class T>
cudaError_t launch_op(int plan_id, RowArgs a, cudaStream_t stream) {
    switch (plan_id) {
#define TILE_CASE(id, S, K, R) \
    case id: return launch_one<OP, T, S, K, R>(a, stream);
        TILE_MULTI_LIST(TILE_CASE)
#undef TILE_CASE
        default: return cudaErrorInvalidValue;
    }
}

template <class T>
cudaError_t launch_type(int op, int plan_id, RowArgs a, cudaStream_t stream) {
    switch (op) {
        case OP_RESLN: return launch_op<OP_RESLN, T>(plan_id, a, stream);
        case OP_LN: return launch_op<OP_LN, T>(plan_id, a, stream);
        case OP_RMS: return launch_op<OP_RMS, T>(plan_id, a, stream);
        case OP_SOFTMAX: return launch_op<OP_SOFTMAX, T>(plan_id, a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_multi(int kernel_op, int elem, int plan_id, RowArgs a, cudaStream_t stream) {
    switch (elem) {
        case ELEM_F32: return launch_type<float>(kernel_op, plan_id, a, stream);
        case ELEM_BF16: return launch_type<__nv_bfloat16>(kernel_op, plan_id, a, stream);
        case ELEM_F16: return launch_type<__half>(kernel_op, plan_id, a, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t status_multi(unsigned int *value, cudaStream_t stream) {
    cudaError_t err = cudaMemcpyFromSymbolAsync(value, g_status, sizeof(unsigned int), 0,
                                                cudaMemcpyDeviceToHost, stream);
    if (err != cudaSuccess) return err;
    err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) return err;
    if (*value == 0) return cudaSuccess;
    const unsigned int zero = 0;
    err = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(unsigned int), 0,
                                  cudaMemcpyHostToDevice, stream);
    if (err != cudaSuccess) return err;
    return cudaStreamSynchronize(stream);
}

}  // namespace tile
