// Pointwise value/derivative pairs: one read, two writes per element.
//
// "Multi-output pointwise fusion: evidence and limits" ("Measurement
// definitions and population") evaluates sigmoid and tanh-approximate GELU,
// each returning its value and derivative into separate outputs from one
// fused element grid.  Here one streaming kernel per function reads x once
// and writes both outputs: float4 accesses when the three pointers share a
// 16-byte phase (scalar head and tail around the aligned body), scalar
// accesses otherwise; each thread has four vectors in flight.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "launch.h"

namespace tile {
namespace {

__device__ unsigned int g_status;    // device error word of the pair kernels
enum { STATUS_BAD_LAUNCH = 1u };
constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// sigmoid(x) and sigmoid'(x) = e / (1 + e)^2 with e = exp(-|x|) in (0, 1],
// which neither overflows nor cancels for large |x|.
__device__ __forceinline__ void sigmoid_pair(float x, float &y, float &dy) {
    const float e = expf(-fabsf(x));
    const float inv = 1.0f / (1.0f + e);
    y = x >= 0.0f ? inv : e * inv;
    dy = e * inv * inv;
}

// tanh GELU (Hendrycks and Gimpel 2016), g(x) = x/2 (1 + tanh u),
// u = sqrt(2/pi) (x + 0.044715 x^3), evaluated through the identity
// (1 + tanh u)/2 = sigmoid(2u), which stays accurate where 1 + tanh u
// cancels (large negative x):
//   g(x)  = x sigmoid(2u)
//   g'(x) = sigmoid(2u) + 2 x sigmoid'(2u) u',  u' = sqrt(2/pi) (1 + 3 * 0.044715 x^2).
__device__ __forceinline__ void gelu_tanh_pair(float x, float &y, float &dy) {
    const float c = 0.7978845608028654f;          // sqrt(2/pi)
    const float a = 0.044715f;
    const float x2 = x * x;
    const float u2 = 2.0f * c * fmaf(a * x2, x, x);
    float s, ds;
    sigmoid_pair(u2, s, ds);
    y = x * s;
    const float du = c * fmaf(3.0f * a, x2, 1.0f);
    dy = ds == 0.0f ? s : fmaf(2.0f * x * ds, du, s);
}

template <int KIND>
__device__ __forceinline__ void pair(float x, float &y, float &dy) {
    if constexpr (KIND == PAIR_SIGMOID)
        sigmoid_pair(x, y, dy);
    else
        gelu_tanh_pair(x, y, dy);
}

template <int KIND>
__global__ void __launch_bounds__(kThreads)
    pair_kernel(const float *__restrict__ x, float *__restrict__ y, float *__restrict__ dy,
                long long n, int vec, unsigned int *status) {
    if (blockDim.x != kThreads) {
        if (threadIdx.x == 0) atomicOr(status, STATUS_BAD_LAUNCH);
        return;
    }
    const long long tid = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
    const long long stride = static_cast<long long>(gridDim.x) * kThreads;
    if (!vec) {
        for (long long i = tid; i < n; i += stride) {
            float a, b;
            pair<KIND>(__ldcs(x + i), a, b);
            __stcs(y + i, a);
            __stcs(dy + i, b);
        }
        return;
    }
    // head scalars up to the 16-byte boundary, float4 body, tail scalars
    const int mis = static_cast<int>((reinterpret_cast<uintptr_t>(x) >> 2) & 3);
    long long h = (4 - mis) & 3;
    if (h > n) h = n;
    const long long nb = (n - h) >> 2;
    const long long t0 = h + 4 * nb;
    if (tid < h) {
        float a, b;
        pair<KIND>(__ldcs(x + tid), a, b);
        __stcs(y + tid, a);
        __stcs(dy + tid, b);
    }
    if (tid < n - t0) {
        float a, b;
        pair<KIND>(__ldcs(x + t0 + tid), a, b);
        __stcs(y + t0 + tid, a);
        __stcs(dy + t0 + tid, b);
    }
    const float4 *x4 = reinterpret_cast<const float4 *>(x + h);
    float4 *y4 = reinterpret_cast<float4 *>(y + h);
    float4 *d4 = reinterpret_cast<float4 *>(dy + h);
    for (long long i0 = tid; i0 < nb; i0 += stride * kUnroll) {
        float4 in[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const long long i = i0 + u * stride;
            if (i < nb) in[u] = __ldcs(x4 + i);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const long long i = i0 + u * stride;
            if (i < nb) {
                float4 a, b;
                pair<KIND>(in[u].x, a.x, b.x);
                pair<KIND>(in[u].y, a.y, b.y);
                pair<KIND>(in[u].z, a.z, b.z);
                pair<KIND>(in[u].w, a.w, b.w);
                __stcs(y4 + i, a);
                __stcs(d4 + i, b);
            }
        }
    }
}

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

}  // namespace

cudaError_t launch_pairs(int kind, const float *x, float *y, float *dy, long long n,
                         cudaStream_t stream) {
    cudaError_t err = cudaSuccess;
    unsigned int *status = status_address(&err);
    if (status == nullptr) return err;
    const uintptr_t px = reinterpret_cast<uintptr_t>(x);
    const int vec = ((px ^ reinterpret_cast<uintptr_t>(y)) & 15) == 0 &&
                    ((px ^ reinterpret_cast<uintptr_t>(dy)) & 15) == 0;
    // One pass: every thread handles kUnroll vectors once (a grid over the
    // whole array streamed faster on GB300 than a persistent grid of a few
    // CTAs per SM walking it); the grid-stride loop only covers arrays past
    // the grid-size limit.
    const long long per_block = static_cast<long long>(kThreads) * (vec ? 4 : 1) * kUnroll;
    long long blocks = (n + per_block - 1) / per_block;
    const long long cap = 0x7fffffffLL;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (kind == PAIR_SIGMOID)
        pair_kernel<PAIR_SIGMOID><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
            x, y, dy, n, vec, status);
    else
        pair_kernel<PAIR_GELU_TANH><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
            x, y, dy, n, vec, status);
    return cudaGetLastError();
}

cudaError_t status_pairs(unsigned int *value, cudaStream_t stream) {
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
