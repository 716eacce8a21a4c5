// Backward row kernels (bwd_kernel.cuh) for one element type: every built
// plan whose two stripes fit the register budget, for LayerNorm, RMSNorm and
// softmax, plus the launcher and device error word.  Included once per type
// by ops_backward[_bf16|_f16].cu with TILE_BWD_T (float, __nv_bfloat16 or
// __half) and TILE_BWD_NAME (the launcher's suffix) defined.
#include <atomic>

#include "bwd_kernel.cuh"
#include "launch.h"
#include "plans.h"

#define TILE_BWD_CAT2(a, b) a##b
#define TILE_BWD_CAT(a, b) TILE_BWD_CAT2(a, b)

namespace tile {
namespace {
__device__ unsigned int g_status;   // device error word of the backward kernels

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

template <int OP, int V, int S, int P, int K, int C>
cudaError_t launch_plan(BwdArgs args, cudaStream_t stream) {
    constexpr int EV = (V == 4) ? Elem<TILE_BWD_T>::kVec : 1;
    // 2-byte rows of 16-byte vectors use the raw-word kernel
    constexpr bool kRaw = sizeof(TILE_BWD_T) == 2 && V == 4;
    constexpr int kBudget = kRaw ? kMaxStripeBwdRaw : kMaxStripeBwd;
    if constexpr (K * EV > kBudget) {
        (void)args;
        (void)stream;
        return cudaErrorInvalidValue;     // not built: two stripes too large
    } else {
        cudaError_t err = cudaSuccess;
        args.status = status_address(&err);
        if (args.status == nullptr) return err;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned int>(((args.rows + P - 1) / P) * C), 1, 1);
        cfg.blockDim = dim3(32 * S * P, 1, 1);
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
        if constexpr (kRaw) {
            // G (gamma may be present) is a template argument of the raw
            // kernel.  RMSNorm launches the G = false kernel without gamma,
            // which then does not carry the registers gamma's loads need
            // (measured 0-5 % faster); LayerNorm always launches G = true and
            // tests gamma at run time, because its G = false kernel measured
            // up to 28 % slower at 2048-16384 columns; softmax has no gamma.
            if constexpr (OP == BWD_LN_OP) {
                // Rows 16-byte aligned and of whole vectors (all three
                // pointers share the phase) take the kernel without a
                // scalar head and tail where that measured faster: plan 6's
                // shape (S = 4, P = 1, K = 4), 7 % at 65536 x 4096 BF16 (64
                // registers instead of 70, 8 CTAs per SM instead of 7).  At
                // plans 4 and 7 the same kernel measured 3 % and 33 %
                // slower, at 1024 and 16384 columns within about 1 %.
                if constexpr (S == 4 && P == 1 && K == 4 && C == 1) {
                    if ((reinterpret_cast<uintptr_t>(args.x) & 15) == 0 && args.width % EV == 0 &&
                        whole_vector_kernels())
                        return cudaLaunchKernelEx(
                            &cfg, row_bwd_raw_kernel<OP, TILE_BWD_T, S, P, K, C, true, true>,
                            args);
                }
                return cudaLaunchKernelEx(&cfg, row_bwd_raw_kernel<OP, TILE_BWD_T, S, P, K, C, true>,
                                          args);
            } else if constexpr (OP == BWD_RMS_OP) {
                if (args.gamma != nullptr)
                    return cudaLaunchKernelEx(
                        &cfg, row_bwd_raw_kernel<OP, TILE_BWD_T, S, P, K, C, true>, args);
            }
            return cudaLaunchKernelEx(&cfg, row_bwd_raw_kernel<OP, TILE_BWD_T, S, P, K, C, false>,
                                      args);
        } else
            return cudaLaunchKernelEx(&cfg, row_bwd_kernel<OP, TILE_BWD_T, V, S, P, K, C>, args);
    }
}

template <int OP>
cudaError_t launch_op(int plan_id, BwdArgs args, cudaStream_t stream) {
    switch (plan_id) {
#define TILE_CASE(id, V, S, P, K, C) \
    case id: return launch_plan<OP, V, S, P, K, C>(args, stream);
        TILE_PLAN_LIST(TILE_CASE)
#undef TILE_CASE
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace

cudaError_t TILE_BWD_CAT(launch_backward, TILE_BWD_NAME)(int op, int plan_id, BwdArgs args,
                                                         cudaStream_t stream) {
    switch (op) {
        case BWD_LN: return launch_op<BWD_LN>(plan_id, args, stream);
        case BWD_RMS: return launch_op<BWD_RMS>(plan_id, args, stream);
        case BWD_SOFTMAX: return launch_op<BWD_SOFTMAX>(plan_id, args, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t TILE_BWD_CAT(status_backward, TILE_BWD_NAME)(unsigned int *value,
                                                         cudaStream_t stream) {
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
