// Launchers of the shared-memory-staged row kernel (staged_kernel.cuh) for
// the normalisers and softmax, FP32 and BF16, over the staged plans of
// plans.h (TILE_STAGED_LIST), plus their device error word.
#include <atomic>

#include "launch.h"
#include "plans.h"
#include "staged_kernel.cuh"

namespace tile {
namespace {

__device__ unsigned int g_status;   // device error word of the staged kernels

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

int sm_count(cudaError_t *err) {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        *err = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        if (*err != cudaSuccess) return 0;
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

// Whether a plan keeps gamma/beta in registers across rows: 2-byte rows
// (where reloading them per row costs the most against the row's bytes),
// the normalisers, and a stripe of at most 32 floats (gamma and beta then
// take 64 registers more).
template <int OP, class T, int K>
constexpr bool resident_params() {
    return sizeof(T) == 2 && OP != OP_SOFTMAX && K * (16 / sizeof(T)) <= 32;
}

template <int OP, class T, int S, int K, int KB, bool AFF>
cudaError_t launch_kernel(RowArgs a, StagedHooks hooks, cudaStream_t stream) {
    {
        cudaError_t err = cudaSuccess;
        a.status = status_address(&err);
        if (a.status == nullptr) return err;
        const int sms = sm_count(&err);
        if (sms == 0) return err;
        auto kernel = row_staged_kernel<OP, T, S, K, AFF>;
        const int nin = (OP == OP_RESLN) ? 2 : 1;
        const size_t stage = static_cast<size_t>(a.width) * sizeof(T) * nin;
        // as many stages as fit the plan's budget of KB kilobytes, 1 to 8
        int nst = static_cast<int>((static_cast<size_t>(KB) << 10) / stage);
        if (nst > kMaxStages) nst = kMaxStages;
        if (nst < 1) nst = 1;
        const size_t dyn = stage * nst;
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(dyn));
        if (err != cudaSuccess) return err;
        int per_sm = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 32 * S, dyn);
        if (err != cudaSuccess) return err;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        long long grid = static_cast<long long>(sms) * per_sm;
        if (grid > a.rows) grid = a.rows;
        kernel<<<static_cast<unsigned int>(grid), 32 * S, dyn, stream>>>(a, nst, hooks);
        return cudaGetLastError();
    }
}

template <int OP, class T, int S, int K, int KB>
cudaError_t launch_one(RowArgs a, StagedHooks hooks, cudaStream_t stream) {
    constexpr int EV = 16 / sizeof(T);
    if constexpr (K * EV > 64) {
        (void)a;
        (void)hooks;
        (void)stream;
        return cudaErrorInvalidValue;     // not built: stripe above 64 floats
    } else if constexpr (resident_params<OP, T, K>()) {
        if (a.gamma != nullptr) return launch_kernel<OP, T, S, K, KB, true>(a, hooks, stream);
        return launch_kernel<OP, T, S, K, KB, false>(a, hooks, stream);
    } else {
        return launch_kernel<OP, T, S, K, KB, false>(a, hooks, stream);
    }
}

template <int OP, class T>
cudaError_t launch_op(int staged_id, RowArgs a, StagedHooks h, cudaStream_t stream) {
    switch (staged_id) {
#define TILE_CASE(id, S, K, KB) \
    case id: return launch_one<OP, T, S, K, KB>(a, h, stream);
        TILE_STAGED_LIST(TILE_CASE)
#undef TILE_CASE
        default: return cudaErrorInvalidValue;
    }
}

template <class T>
cudaError_t launch_type(int op, int staged_id, RowArgs a, StagedHooks h, cudaStream_t stream) {
    switch (op) {
        case OP_RESLN: return launch_op<OP_RESLN, T>(staged_id, a, h, stream);
        case OP_LN: return launch_op<OP_LN, T>(staged_id, a, h, stream);
        case OP_RMS: return launch_op<OP_RMS, T>(staged_id, a, h, stream);
        case OP_SOFTMAX: return launch_op<OP_SOFTMAX, T>(staged_id, a, h, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_hooked(int kernel_op, int elem, int plan_id, RowArgs a, StagedHooks h,
                          cudaStream_t stream) {
    switch (elem) {
        case ELEM_F32: return launch_type<float>(kernel_op, plan_id, a, h, stream);
        case ELEM_BF16: return launch_type<__nv_bfloat16>(kernel_op, plan_id, a, h, stream);
        case ELEM_F16: return launch_type<__half>(kernel_op, plan_id, a, h, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_staged(int kernel_op, int elem, int plan_id, RowArgs a, cudaStream_t stream) {
    return launch_hooked(kernel_op, elem, plan_id, a, StagedHooks{kWaitSpins, 0}, stream);
}

cudaError_t launch_staged_withheld(int kernel_op, int elem, int plan_id, RowArgs a,
                                   unsigned int spin_limit, cudaStream_t stream) {
    if (spin_limit < 1) return cudaErrorInvalidValue;
    return launch_hooked(kernel_op, elem, plan_id, a, StagedHooks{spin_limit, 1}, stream);
}

cudaError_t status_staged(unsigned int *value, cudaStream_t stream) {
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
