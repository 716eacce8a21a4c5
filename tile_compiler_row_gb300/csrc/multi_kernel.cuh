// Row kernel with R rows per CTA, every thread owning the same columns of
// each of them.
//
// The register kernel gives each row its own W = 32*S workers.  Here one CTA
// of W threads normalises R rows at once: worker t holds elements
// (k*W + t)*EV .. +EV-1 of every one of its R rows in an FP32 stripe
// v[R][K][EV], each input element read once (the stripe layout of
// "Immutable input reuse in Metal reductions", "What the transformation
// actually preserves", repeated per row).  Two things are shared across the
// R rows: the reduction rounds (one warp butterfly and one shared-memory
// exchange carry the partial sums of all R rows, so a CTA barrier serves R
// rows), and the per-column parameters of affine LayerNorm and weighted
// RMSNorm (each thread loads its gamma/beta columns once and applies them to
// all R rows).  A row's arithmetic is exactly that of the register kernel
// with the same S and K (same per-lane accumulators, combine order and
// output map), so the results are bitwise those of that plan.
//
// Preconditions (checked on the host): every pointer 16-byte aligned and
// width a multiple of the vector (whole 16-byte rows, no head or tail),
// K * W * EV >= width.  A CTA whose last rows fall past the end replays the
// last row and predicates only its stores, so every barrier is taken by all.
#pragma once

#include "row_kernel.cuh"

namespace tile {

// Resident CTAs the register budget must allow: 2-byte rows with at most
// 16 stripe floats a thread are held to 64 registers (32 warps per SM),
// which they fit without spilling; at 32 stripe floats the LayerNorm
// kernels would spill there, so the compiler keeps its own count.
template <class T, int S, int K, int R>
constexpr int multi_min_blocks() {
    return (sizeof(T) == 2 && R * K * 8 <= 16) ? 32 / S : 0;
}

template <int OP, class T, int S, int K, int R>
__global__ void __launch_bounds__(32 * S, (multi_min_blocks<T, S, K, R>()))
    row_multi_kernel(const RowArgs a) {
    static_assert(OP == OP_RESLN || OP == OP_LN || OP == OP_RMS || OP == OP_SOFTMAX,
                  "normalisers and softmax");
    constexpr int EV = Elem<T>::kVec;
    constexpr int W = 32 * S;
    constexpr float kFill = (OP == OP_SOFTMAX) ? -INFINITY : 0.0f;
    // packed f32x2 lane arithmetic where the register kernel uses it
    constexpr bool PK = sizeof(T) == 2 && W <= 512 && (OP == OP_LN || OP == OP_RESLN);

    __shared__ float part1[S > 1 ? R * S : 1];
    __shared__ float part2[S > 1 ? 2 * R * S : 1];

    if (blockDim.x != W) {
        if (threadIdx.x == 0) atomicOr(a.status, STATUS_BAD_LAUNCH);
        return;
    }
    const int width = a.width;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int nb = width / EV;
    const long long last = a.rows - 1;

    long long row[R];
    bool active[R];
#pragma unroll
    for (int j = 0; j < R; ++j) {
        row[j] = static_cast<long long>(blockIdx.x) * R + j;
        active[j] = row[j] <= last;
        if (!active[j]) row[j] = last;             // replay the last row
    }

    // ---- load every row once into the stripe --------------------------------
    float v[R][K][EV];
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const long long base = row[j] * static_cast<long long>(width);
        const T *xr = static_cast<const T *>(a.x) + base;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int i = k * W + tid;
            if (i < nb) {
                Elem<T>::load_vec(xr + EV * i, v[j][k]);
                if constexpr (OP == OP_RESLN) {
                    const T *rr = static_cast<const T *>(a.r) + base;
                    if constexpr (sizeof(T) == 2) {
                        add_raw_vec<T>(v[j][k], __ldcs(reinterpret_cast<const uint4 *>(rr + EV * i)));
                    } else {
                        float b[EV];
                        Elem<T>::load_vec(rr + EV * i, b);
                        vadd<PK, EV>(v[j][k], b);
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < EV; ++e) v[j][k][e] = kFill;
            }
        }
    }

    const float n = static_cast<float>(width);
    if constexpr (OP == OP_RESLN || OP == OP_LN) {
        // ---- mean estimates ---------------------------------------------------
        float s[R];
#pragma unroll
        for (int j = 0; j < R; ++j) {
            float acc[EV];
#pragma unroll
            for (int e = 0; e < EV; ++e) acc[e] = 0.0f;
#pragma unroll
            for (int k = 0; k < K; ++k) vadd<PK, EV>(acc, v[j][k]);
            s[j] = lane_total(acc);
        }
        row_allreduce<Sum, R, S, 1, 1>(s, part1, nullptr, 0, warp, lane);
        // ---- centre in place; (sum d, sum d^2) per row ---------------------
        float q[2 * R];
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const float mean0 = over_n<T>(s[j], n, a.inv_n);
            float a1[EV], a2[EV];
#pragma unroll
            for (int e = 0; e < EV; ++e) a1[e] = a2[e] = 0.0f;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const bool ok = k * W + tid < nb;
                if constexpr (PK) {
                    if (ok) {
                        vadd_c<PK, EV>(v[j][k], -mean0);
                        vadd<PK, EV>(a1, v[j][k]);
                        vsq_acc<PK, EV>(a2, v[j][k]);
                    } else {
#pragma unroll
                        for (int e = 0; e < EV; ++e) v[j][k][e] = 0.0f;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < EV; ++e) {
                        const float d = ok ? v[j][k][e] - mean0 : 0.0f;
                        v[j][k][e] = d;
                        a1[e] += d;
                        a2[e] = fmaf(d, d, a2[e]);
                    }
                }
            }
            q[2 * j] = lane_total(a1);
            q[2 * j + 1] = lane_total(a2);
        }
        row_allreduce<Sum, 2 * R, S, 1, 1>(q, part2, nullptr, 0, warp, lane);
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const float mu1 = over_n<T>(q[2 * j], n, a.inv_n);
            const float var = fmaxf(over_n<T>(q[2 * j + 1], n, a.inv_n) - mu1 * mu1, 0.0f);
            const float rstd = inv_sqrt<T>(var + a.eps);
            if constexpr (PK) {
                const float shift = -mu1 * rstd;
#pragma unroll
                for (int k = 0; k < K; ++k) vfma_c<PK, EV>(v[j][k], rstd, shift);
            } else {
#pragma unroll
                for (int k = 0; k < K; ++k)
#pragma unroll
                    for (int e = 0; e < EV; ++e) v[j][k][e] = ln_out<T>(v[j][k][e], mu1, rstd);
            }
        }
    } else if constexpr (OP == OP_RMS) {
        float s[R];
#pragma unroll
        for (int j = 0; j < R; ++j) {
            float acc[EV];
#pragma unroll
            for (int e = 0; e < EV; ++e) acc[e] = 0.0f;
#pragma unroll
            for (int k = 0; k < K; ++k) vsq_acc<PK, EV>(acc, v[j][k]);
            s[j] = lane_total(acc);
        }
        row_allreduce<Sum, R, S, 1, 1>(s, part1, nullptr, 0, warp, lane);
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const float rstd = inv_sqrt<T>(over_n<T>(s[j], n, a.inv_n) + a.eps);
#pragma unroll
            for (int k = 0; k < K; ++k) vmul_c<PK, EV>(v[j][k], rstd);
        }
    } else {
        // ---- softmax: row maxima, exponentials in place, row sums ----------
        float m[R];
#pragma unroll
        for (int j = 0; j < R; ++j) {
            float mj[EV];
#pragma unroll
            for (int e = 0; e < EV; ++e) mj[e] = kFill;
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int e = 0; e < EV; ++e) mj[e] = fmaxf(mj[e], v[j][k][e]);
            m[j] = lane_max(mj);
        }
        row_allreduce<Max, R, S, 1, 1>(m, part1, nullptr, 0, warp, lane);
        float s[R];
#pragma unroll
        for (int j = 0; j < R; ++j) {
            float acc[EV];
#pragma unroll
            for (int e = 0; e < EV; ++e) acc[e] = 0.0f;
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int e = 0; e < EV; ++e) {
                    const float x = softmax_exp<T>(v[j][k][e] - m[j]);
                    v[j][k][e] = x;
                    acc[e] += x;
                }
            s[j] = lane_total(acc);
        }
        row_allreduce<Sum, R, S, 1, 1>(s, part2, nullptr, 0, warp, lane);
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const float inv = 1.0f / s[j];
#pragma unroll
            for (int k = 0; k < K; ++k) vmul_c<PK, EV>(v[j][k], inv);
        }
    }

    // ---- per-column scale and shift: loaded once, applied to all R rows ----
    if constexpr (OP != OP_SOFTMAX) {
        if (a.gamma != nullptr) {
            const float *g = a.gamma;
            const float *b = a.beta;
            const bool g32 = EV == 8 && (reinterpret_cast<uintptr_t>(g) & 31) == 0 &&
                             (b == nullptr || (reinterpret_cast<uintptr_t>(b) & 31) == 0);
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int i = k * W + tid;
                if (i < nb) {
                    float gg[EV], bb[EV];
                    if (g32) {
                        if constexpr (EV == 8) {
                            ldg_v8(g + EV * i, gg);
                            if (b != nullptr) {
                                ldg_v8(b + EV * i, bb);
                            } else {
#pragma unroll
                                for (int e = 0; e < EV; ++e) bb[e] = 0.0f;
                            }
                        }
                    } else {
#pragma unroll
                        for (int q4 = 0; q4 < EV / 4; ++q4) {
                            const float4 g4 = __ldg(reinterpret_cast<const float4 *>(g + EV * i) + q4);
                            float4 b4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                            if (b != nullptr) b4 = __ldg(reinterpret_cast<const float4 *>(b + EV * i) + q4);
                            gg[4 * q4] = g4.x; gg[4 * q4 + 1] = g4.y;
                            gg[4 * q4 + 2] = g4.z; gg[4 * q4 + 3] = g4.w;
                            bb[4 * q4] = b4.x; bb[4 * q4 + 1] = b4.y;
                            bb[4 * q4 + 2] = b4.z; bb[4 * q4 + 3] = b4.w;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < R; ++j) vfma<PK, EV>(v[j][k], gg, bb);
                }
            }
        }
    }

    // ---- streaming stores, predicated for replayed rows -------------------
#pragma unroll
    for (int j = 0; j < R; ++j) {
        if (active[j]) {
            T *yr = static_cast<T *>(a.y) + row[j] * static_cast<long long>(width);
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int i = k * W + tid;
                if (i < nb) Elem<T>::store_vec(yr + EV * i, v[j][k]);
            }
        }
    }
}

}  // namespace tile
