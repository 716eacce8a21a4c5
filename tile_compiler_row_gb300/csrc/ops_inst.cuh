// Instantiates every built plan for one operation and element type and
// provides its host-side launcher and device error word.  Included once per
// (op, type) by ops_<op>[_bf16|_f16].cu with TILE_INST_OP (tile::OP_*),
// TILE_INST_T (float, __nv_bfloat16 or __half) and TILE_INST_NAME (a C identifier)
// defined, so each compiles as its own translation unit, in parallel.
#include "row_kernel.cuh"
#include "plans.h"
#include "launch.h"

#include <atomic>

#define TILE_CAT2(a, b) a##b
#define TILE_CAT(a, b) TILE_CAT2(a, b)

namespace tile {
namespace {
__device__ unsigned int g_status;   // this op's device error word

// Device address of g_status, looked up once per device.
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

template <int V, int S, int P, int K, int C>
cudaError_t launch_plan(RowArgs args, cudaStream_t stream) {
    constexpr int EV = (V == 4) ? Elem<TILE_INST_T>::kVec : 1;
    if constexpr (sizeof(TILE_INST_T) == 2 && K * EV > kMaxStripeBf16) {
        (void)args;
        (void)stream;
        return cudaErrorInvalidValue;     // not built: stripe too large for BF16
    } else {
        cudaError_t err = cudaSuccess;
        args.status = status_address(&err);
        if (args.status == nullptr) return err;
        const long long rows = args.rows;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned int>(((rows + P - 1) / P) * C), 1, 1);
        cfg.blockDim = dim3(32 * S * P, 1, 1);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        if (C > 1) {
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = C;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
        }
        // 2-byte rows that are 16-byte aligned and hold whole vectors take
        // the kernel without a scalar head and tail (bitwise the same results)
        if constexpr (V == 4 && sizeof(TILE_INST_T) == 2) {
            if ((reinterpret_cast<uintptr_t>(args.x) & 15) == 0 && args.width % EV == 0 &&
                whole_vector_kernels())
                return cudaLaunchKernelEx(
                    &cfg, row_kernel<TILE_INST_OP, TILE_INST_T, V, S, P, K, C, true>, args);
        }
        return cudaLaunchKernelEx(&cfg, row_kernel<TILE_INST_OP, TILE_INST_T, V, S, P, K, C>,
                                  args);
    }
}
}  // namespace

cudaError_t TILE_CAT(launch_, TILE_INST_NAME)(int plan_id, RowArgs args, cudaStream_t stream) {
    switch (plan_id) {
#define TILE_CASE(id, V, S, P, K, C) \
    case id: return launch_plan<V, S, P, K, C>(args, stream);
        TILE_PLAN_LIST(TILE_CASE)
#undef TILE_CASE
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t TILE_CAT(status_, TILE_INST_NAME)(unsigned int *value, cudaStream_t stream) {
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
