// Parameter gradients of LayerNorm / RMSNorm: column sums over all rows,
//   dgamma[j] = sum_i dy[i][j] * (x[i][j] - mean_i) * rstd_i
//   dbeta[j]  = sum_i dy[i][j]
// with (mean_i, rstd_i) the row statistics the backward kernel wrote
// (mean 0 for RMSNorm).
//
// x and dy are FP32, BF16 or FP16 (widened exactly; all sums are FP32).
// Stage 1 splits the rows into nblk fixed blocks; a thread owns 4 adjacent
// columns (one aligned load per row when the rows allow it, else scalars)
// and accumulates compensated (TwoSum) sums over its block's rows: FP32 rows
// four in flight, each added compensated; 2-byte rows eight in flight as raw
// words, added as pairwise trees of four.  Block partials go to the caller's
// workspace [nblk][2][width].
// Stage 2 sums the nblk partials of each column in a fixed order (eight
// interleaved warp slices, then the slices in warp order).  The partition
// depends only on (rows, width) and the device (its SM count and the
// kernel's resident CTAs per SM), so results are bitwise reproducible on a
// device.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <type_traits>

#include "launch.h"
#include "row_kernel.cuh"

namespace tile {
namespace {

__device__ unsigned int g_status;   // device error word of the parameter kernels
constexpr int kThreads = 256;
constexpr int kRowsInFlight = 4;

// Element `hi` (0: lower address) of a 32-bit word of two 2-byte values.
template <class T>
__device__ __forceinline__ float widen_half(unsigned int w, int hi) {
    if constexpr (std::is_same<T, __half>::value) {
        const __half2 h = *reinterpret_cast<const __half2 *>(&w);
        return hi ? __high2float(h) : __low2float(h);
    } else {
        return __uint_as_float(hi ? (w & 0xffff0000u) : (w << 16));
    }
}

// Element `hi` of a 32-bit word of two 2-byte values plus c, one
// mixed-precision add (add.rn.f32.bf16 / .f16): the 2-byte value enters
// exactly, so this is round(x + c) as after an explicit widening.
#define TILE_ADD_HALF(TY, HALF)                                                          \
    "{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tadd.rn.f32." TY " %0, " HALF ", %2;\n\t}"
template <class T>
__device__ __forceinline__ float add_half(unsigned int w, int hi, float c) {
    float r;
    if constexpr (std::is_same<T, __half>::value) {
        if (hi)
            asm(TILE_ADD_HALF("f16", "h") : "=f"(r) : "r"(w), "f"(c));
        else
            asm(TILE_ADD_HALF("f16", "l") : "=f"(r) : "r"(w), "f"(c));
    } else {
        if (hi)
            asm(TILE_ADD_HALF("bf16", "h") : "=f"(r) : "r"(w), "f"(c));
        else
            asm(TILE_ADD_HALF("bf16", "l") : "=f"(r) : "r"(w), "f"(c));
    }
    return r;
}
#undef TILE_ADD_HALF

// Columns a stage-1 thread owns: four (one 16-byte FP32 or 8-byte BF16 /
// FP16 load per row).
constexpr int kCols = 4;

// Two pairwise trees of four rows each go into one compensated add; the
// tree adds at most 2u sum|terms| of error, the compensated running sum and
// the final rounding u each: within 3u sum|terms| (4u is what the tests
// allow).  FP32 rows (bound by DRAM) add every row compensated.
__device__ __forceinline__ float tree4(float a, float b, float c, float d) {
    return (a + b) + (c + d);
}

// FP32 rows, and 2-byte rows that are not whole aligned groups of four:
// four rows in flight, widened at load.
template <class T>
__device__ __forceinline__ void rows_widened(const T *__restrict__ x, const T *__restrict__ dy,
                                             const float *__restrict__ stats, long long r0,
                                             long long r1, int width, int c0, int ncol, int vec,
                                             float (&sg)[kCols], float (&cg)[kCols],
                                             float (&sb)[kCols], float (&cb)[kCols]) {
    for (long long r = r0; r < r1; r += kRowsInFlight) {
        float xv[kRowsInFlight][kCols], dv[kRowsInFlight][kCols], mu[kRowsInFlight],
            rs[kRowsInFlight];
#pragma unroll
        for (int q = 0; q < kRowsInFlight; ++q) {
            const long long rr = r + q;
            if (rr < r1) {
                const T *xr = x + rr * width + c0;
                const T *dr = dy + rr * width + c0;
                if (vec) {
                    if constexpr (sizeof(T) == 4) {
                        const float4 tx = __ldcs(reinterpret_cast<const float4 *>(xr));
                        const float4 td = __ldcs(reinterpret_cast<const float4 *>(dr));
                        xv[q][0] = tx.x; xv[q][1] = tx.y; xv[q][2] = tx.z; xv[q][3] = tx.w;
                        dv[q][0] = td.x; dv[q][1] = td.y; dv[q][2] = td.z; dv[q][3] = td.w;
                    } else {
                        const uint2 tx = __ldcs(reinterpret_cast<const uint2 *>(xr));
                        const uint2 td = __ldcs(reinterpret_cast<const uint2 *>(dr));
                        xv[q][0] = widen_half<T>(tx.x, 0); xv[q][1] = widen_half<T>(tx.x, 1);
                        xv[q][2] = widen_half<T>(tx.y, 0); xv[q][3] = widen_half<T>(tx.y, 1);
                        dv[q][0] = widen_half<T>(td.x, 0); dv[q][1] = widen_half<T>(td.x, 1);
                        dv[q][2] = widen_half<T>(td.y, 0); dv[q][3] = widen_half<T>(td.y, 1);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < kCols; ++j) {
                        xv[q][j] = j < ncol ? Elem<T>::load(xr + j) : 0.0f;
                        dv[q][j] = j < ncol ? Elem<T>::load(dr + j) : 0.0f;
                    }
                }
                mu[q] = __ldg(stats + 2 * rr);
                rs[q] = __ldg(stats + 2 * rr + 1);
            } else {
#pragma unroll
                for (int j = 0; j < kCols; ++j) xv[q][j] = dv[q][j] = 0.0f;
                mu[q] = rs[q] = 0.0f;
            }
        }
        if constexpr (sizeof(T) == 2) {
#pragma unroll
            for (int j = 0; j < kCols; ++j) {
                float t[kRowsInFlight];
#pragma unroll
                for (int q = 0; q < kRowsInFlight; ++q)
                    t[q] = dv[q][j] * ((xv[q][j] - mu[q]) * rs[q]);
                comp_add(sg[j], cg[j], tree4(t[0], t[1], t[2], t[3]));
                comp_add(sb[j], cb[j], tree4(dv[0][j], dv[1][j], dv[2][j], dv[3][j]));
            }
        } else {
#pragma unroll
            for (int q = 0; q < kRowsInFlight; ++q)
#pragma unroll
                for (int j = 0; j < kCols; ++j) {
                    comp_add(sg[j], cg[j], dv[q][j] * ((xv[q][j] - mu[q]) * rs[q]));
                    comp_add(sb[j], cb[j], dv[q][j]);
                }
        }
    }
}

// (a0, a1) -= (b0, b1), one packed instruction (PTX sub.rn.f32x2, sm_100
// and later); each lane is rounded as the scalar subtraction.
__device__ __forceinline__ void sub_x2(float &a0, float &a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb;\n\tmov.b64 ra, {%0, %1};\n\tmov.b64 rb, {%2, %3};\n\t"
        "sub.rn.f32x2 ra, ra, rb;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1) : "f"(b0), "f"(b1));
}

// comp_add on two independent (sum, compensation) pairs at once: the same
// TwoSum steps lane by lane on packed pairs, so each lane's result is
// bitwise that of comp_add.
__device__ __forceinline__ void comp_add_x2(float (&s)[2], float (&c)[2], float v0, float v1) {
    float n0 = s[0], n1 = s[1];
    add_x2(n0, n1, v0, v1);                  // s' = s + v
    float b0 = n0, b1 = n1;
    sub_x2(b0, b1, s[0], s[1]);              // bb = s' - s
    float r0 = n0, r1 = n1;
    sub_x2(r0, r1, b0, b1);                  // s' - bb
    float a0 = s[0], a1 = s[1];
    sub_x2(a0, a1, r0, r1);                  // s - (s' - bb)
    sub_x2(v0, v1, b0, b1);                  // v - bb
    add_x2(a0, a1, v0, v1);                  // e
    add_x2(c[0], c[1], a0, a1);              // c += e
    s[0] = n0;
    s[1] = n1;
}

// 2-byte rows of whole aligned groups of four: eight rows in flight kept as
// raw words (a register carries 4 bytes of DRAM data instead of 2), summed
// as two trees of four.  The two columns of a word go through packed f32x2
// pairs (the products, the trees and the compensated sums), each lane
// rounded as the scalar code rounds it, so the results are bitwise those
// of one column at a time with a third fewer instructions.
template <class T>
__device__ __forceinline__ void rows_raw(const T *__restrict__ x, const T *__restrict__ dy,
                                         const float *__restrict__ stats, long long r0,
                                         long long r1, int width, int c0,
                                         float (&sg)[kCols], float (&cg)[kCols],
                                         float (&sb)[kCols], float (&cb)[kCols]) {
    constexpr int R = 2 * kRowsInFlight;   // a multiple of 4
    for (long long r = r0; r < r1; r += R) {
        unsigned int xw[R][2], dw[R][2];
        float mu[R], rs[R];
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const long long rr = r + q;
            if (rr < r1) {
                const uint2 tx = __ldcs(reinterpret_cast<const uint2 *>(x + rr * width + c0));
                const uint2 td = __ldcs(reinterpret_cast<const uint2 *>(dy + rr * width + c0));
                xw[q][0] = tx.x; xw[q][1] = tx.y;
                dw[q][0] = td.x; dw[q][1] = td.y;
                mu[q] = __ldg(stats + 2 * rr);
                rs[q] = __ldg(stats + 2 * rr + 1);
            } else {
                xw[q][0] = xw[q][1] = dw[q][0] = dw[q][1] = 0u;   // +0.0
                mu[q] = rs[q] = 0.0f;
            }
        }
#pragma unroll
        for (int w = 0; w < kCols / 2; ++w)          // columns 2w and 2w + 1
#pragma unroll
            for (int g = 0; g < R / 4; ++g) {
                float t[4][2], d[4][2];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int q = 4 * g + q4;
                    float x0 = add_half<T>(xw[q][w], 0, -mu[q]);         // x - mu
                    float x1 = add_half<T>(xw[q][w], 1, -mu[q]);
                    mul_x2(x0, x1, rs[q], rs[q]);                        // (x - mu) rstd
                    d[q4][0] = widen_half<T>(dw[q][w], 0);
                    d[q4][1] = widen_half<T>(dw[q][w], 1);
                    t[q4][0] = d[q4][0];
                    t[q4][1] = d[q4][1];
                    mul_x2(t[q4][0], t[q4][1], x0, x1);                  // dy xhat
                }
                // tree4 on pairs: (a + b) + (c + d)
                add_x2(t[0][0], t[0][1], t[1][0], t[1][1]);
                add_x2(t[2][0], t[2][1], t[3][0], t[3][1]);
                add_x2(t[0][0], t[0][1], t[2][0], t[2][1]);
                add_x2(d[0][0], d[0][1], d[1][0], d[1][1]);
                add_x2(d[2][0], d[2][1], d[3][0], d[3][1]);
                add_x2(d[0][0], d[0][1], d[2][0], d[2][1]);
                float sgp[2] = {sg[2 * w], sg[2 * w + 1]}, cgp[2] = {cg[2 * w], cg[2 * w + 1]};
                float sbp[2] = {sb[2 * w], sb[2 * w + 1]}, cbp[2] = {cb[2 * w], cb[2 * w + 1]};
                comp_add_x2(sgp, cgp, t[0][0], t[0][1]);
                comp_add_x2(sbp, cbp, d[0][0], d[0][1]);
                sg[2 * w] = sgp[0]; sg[2 * w + 1] = sgp[1];
                cg[2 * w] = cgp[0]; cg[2 * w + 1] = cgp[1];
                sb[2 * w] = sbp[0]; sb[2 * w + 1] = sbp[1];
                cb[2 * w] = cbp[0]; cb[2 * w + 1] = cbp[1];
            }
    }
}

// Two resident CTAs per SM (at most 128 registers a thread): the 2-byte
// kernel keeps its eight raw rows and two trees without spilling; three
// (85 registers) ran 2 % slower at 65536 x 4096 BF16.
template <class T>
__global__ void __launch_bounds__(kThreads, 2)
    param_partial_kernel(const T *__restrict__ x, const T *__restrict__ dy,
                         const float *__restrict__ stats, float *__restrict__ ws, long long rows,
                         int width, int rows_per_block, int vec, int with_beta,
                         unsigned int *status) {
    if (blockDim.x != kThreads) {
        if (threadIdx.x == 0) atomicOr(status, 1u);
        return;
    }
    const int c0 = (blockIdx.x * kThreads + threadIdx.x) * kCols;   // first owned column
    if (c0 >= width) return;
    const long long r0 = static_cast<long long>(blockIdx.y) * rows_per_block;
    long long r1 = r0 + rows_per_block;
    if (r1 > rows) r1 = rows;
    const int ncol = width - c0 < kCols ? width - c0 : kCols;

    float sg[kCols], cg[kCols], sb[kCols], cb[kCols];
#pragma unroll
    for (int j = 0; j < kCols; ++j) sg[j] = cg[j] = sb[j] = cb[j] = 0.0f;
    if constexpr (sizeof(T) == 2) {
        if (vec)
            rows_raw<T>(x, dy, stats, r0, r1, width, c0, sg, cg, sb, cb);
        else
            rows_widened<T>(x, dy, stats, r0, r1, width, c0, ncol, vec, sg, cg, sb, cb);
    } else {
        rows_widened<T>(x, dy, stats, r0, r1, width, c0, ncol, vec, sg, cg, sb, cb);
    }
    float *wg = ws + static_cast<long long>(blockIdx.y) * 2 * width + c0;
    float *wb = wg + width;
    for (int j = 0; j < ncol; ++j) {
        wg[j] = __fadd_rn(sg[j], cg[j]);
        if (with_beta) wb[j] = __fadd_rn(sb[j], cb[j]);
    }
}

// Stage 2: a CTA owns 32 columns; warp w sums row blocks w, w+8, w+16, ...
// (coalesced 128-byte reads), then warp 0 combines the 8 warp partials in
// warp order.
__global__ void __launch_bounds__(kThreads)
    param_final_kernel(const float *__restrict__ ws, int nblk, int width,
                       float *__restrict__ dgamma, float *__restrict__ dbeta,
                       unsigned int *status) {
    constexpr int kWarps = kThreads / 32;
    __shared__ float part[4][kWarps][32];
    if (blockDim.x != kThreads) {
        if (threadIdx.x == 0) atomicOr(status, 1u);
        return;
    }
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + lane;
    float sg = 0.0f, cg = 0.0f, sb = 0.0f, cb = 0.0f;
    if (c < width) {
        for (int b = warp; b < nblk; b += kWarps) {
            comp_add(sg, cg, ws[static_cast<long long>(b) * 2 * width + c]);
            if (dbeta != nullptr)
                comp_add(sb, cb, ws[static_cast<long long>(b) * 2 * width + width + c]);
        }
    }
    part[0][warp][lane] = sg;
    part[1][warp][lane] = cg;
    part[2][warp][lane] = sb;
    part[3][warp][lane] = cb;
    __syncthreads();
    if (warp == 0 && c < width) {
        float tg = part[0][0][lane], ug = part[1][0][lane];
        float tb = part[2][0][lane], ub = part[3][0][lane];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) {
            comp_merge(tg, ug, part[0][w][lane], part[1][w][lane]);
            comp_merge(tb, ub, part[2][w][lane], part[3][w][lane]);
        }
        dgamma[c] = __fadd_rn(tg, ug);
        if (dbeta != nullptr) dbeta[c] = __fadd_rn(tb, ub);
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

int param_blocks(long long rows) {
    long long nblk = (rows + 31) / 32;
    if (nblk > 512) nblk = 512;
    if (nblk < 1) nblk = 1;
    return static_cast<int>(nblk);
}

namespace {

// CTA slots of stage 1 on this device (SMs x resident CTAs) for the kernel
// of element type elem, cached.
template <class T>
int partial_slots_of(int elem) {
    static std::atomic<int> cache[kMaxDevices][3];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int v = cache[dev][elem].load(std::memory_order_relaxed);
    if (v == 0) {
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, param_partial_kernel<T>,
                                                          kThreads, 0) != cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        v = sms * per_sm;
        cache[dev][elem].store(v, std::memory_order_relaxed);
    }
    return v;
}

// Row blocks for stage 1: at most param_blocks(rows) (what the workspace
// holds), and no more than one wave of the device's CTA slots fits (column
// tiles x row blocks <= slots).  Long CTAs pay their load ramp once, and
// fewer block partials shorten stage 2: at 65536 x 4096 BF16 one wave ran in
// 173 us, four full waves of short CTAs in 187 us (FP32 rows, bound by DRAM,
// ran at 328 us either way).
int balanced_blocks(long long rows, int col_tiles, long long slots) {
    const int nmax = param_blocks(rows);
    if (slots <= 0) return nmax;
    const long long fit = slots / col_tiles;
    if (fit < 1) return 1;
    return fit < nmax ? static_cast<int>(fit) : nmax;
}

template <class T>
cudaError_t launch_typed(int elem, const T *x, const T *dy, const float *stats, float *dgamma,
                         float *dbeta, long long rows, int width, float *ws, unsigned int *status,
                         cudaStream_t stream) {
    const int col_tiles = (width + kCols * kThreads - 1) / (kCols * kThreads);
    const int nblk = balanced_blocks(rows, col_tiles, partial_slots_of<T>(elem));
    const int rows_per_block = static_cast<int>((rows + nblk - 1) / nblk);
    const uintptr_t a = reinterpret_cast<uintptr_t>(x), b = reinterpret_cast<uintptr_t>(dy);
    // aligned loads of 4 columns: rows of whole groups of 4, aligned to
    // 16 bytes (FP32) or 8 bytes (BF16 / FP16)
    const uintptr_t group = kCols * sizeof(T);
    const int vec = (width % kCols == 0) && (a % group == 0) && (b % group == 0);
    const dim3 grid1(col_tiles, nblk, 1);
    param_partial_kernel<T><<<grid1, kThreads, 0, stream>>>(x, dy, stats, ws, rows, width,
                                                            rows_per_block, vec,
                                                            dbeta != nullptr, status);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const dim3 grid2((width + 31) / 32, 1, 1);
    param_final_kernel<<<grid2, kThreads, 0, stream>>>(ws, nblk, width, dgamma, dbeta, status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_param_grad(int elem, const void *x, const void *dy, const float *stats,
                              float *dgamma, float *dbeta, long long rows, int width, float *ws,
                              cudaStream_t stream) {
    cudaError_t err = cudaSuccess;
    unsigned int *status = status_address(&err);
    if (status == nullptr) return err;
    switch (elem) {
        case ELEM_F32:
            return launch_typed<float>(elem, static_cast<const float *>(x),
                                       static_cast<const float *>(dy), stats, dgamma, dbeta,
                                       rows, width, ws, status, stream);
        case ELEM_BF16:
            return launch_typed<__nv_bfloat16>(elem, static_cast<const __nv_bfloat16 *>(x),
                                               static_cast<const __nv_bfloat16 *>(dy), stats,
                                               dgamma, dbeta, rows, width, ws, status, stream);
        case ELEM_F16:
            return launch_typed<__half>(elem, static_cast<const __half *>(x),
                                        static_cast<const __half *>(dy), stats, dgamma, dbeta,
                                        rows, width, ws, status, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t status_param_grad(unsigned int *value, cudaStream_t stream) {
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
