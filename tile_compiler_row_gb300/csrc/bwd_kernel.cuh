// Backward row kernels: input gradients of LayerNorm, RMSNorm and softmax.
//
// Same mapping as the forward row kernel (P row programs of W = 32*S workers
// per CTA, or one row over a cluster of C CTAs), with two register stripes:
// the forward input (or softmax output) and the upstream gradient dy, each
// read from global memory once.  Row statistics are recomputed from the
// input with the forward kernel's corrected two-pass form; every reduction
// level combines in a fixed order, so a plan is bitwise deterministic.
//
//   LayerNorm:  xhat = (x - mean) rstd,  g = dy * gamma
//               dx = rstd (g - mean(g) - xhat mean(g xhat))
//   RMSNorm:    xhat = x rstd,  dx = rstd (g - xhat mean(g xhat))
//   softmax:    dx = y (dy - sum(dy y))
//
// Optionally (stats != NULL, LayerNorm / RMSNorm) the row statistics are
// written to stats[row] = (mean, rstd) (mean 0 for RMSNorm) for the
// parameter-gradient kernel (param_grad.cu).
#pragma once

#include "row_kernel.cuh"

namespace tile {

enum { BWD_LN = BWD_LN_OP, BWD_RMS = BWD_RMS_OP, BWD_SOFTMAX = BWD_SOFTMAX_OP };

template <int OP, class T, int V, int S, int P, int K, int C>
__global__ void __launch_bounds__(32 * S * P) row_bwd_kernel(const BwdArgs a) {
    static_assert(V == 1 || V == 4, "V is 1 (scalar) or 4 (16-byte vectors)");
    static_assert(C == 1 || P == 1, "a cluster row has one program per CTA");
    constexpr int W = 32 * S;
    // elements per access: one 16-byte vector (4 FP32 or 8 BF16 / FP16), or one
    constexpr int EV = (V == 4) ? Elem<T>::kVec : 1;

    // Reduction partials, one buffer per round: [N][P*S] floats (N = 2, 4).
    __shared__ float part1[S > 1 ? 2 * P * S : 1];
    __shared__ float part2[S > 1 ? 4 * P * S : 1];
    __shared__ float cpart[C > 1 ? 5 : 1];

    if (blockDim.x != 32 * S * P) {
        if (threadIdx.x == 0) atomicOr(a.status, STATUS_BAD_LAUNCH);
        return;
    }
    const int width = a.width;
    const int tid = threadIdx.x;
    const int program = tid / W;
    const int worker = tid - program * W;
    const int warp = worker >> 5;
    const int lane = tid & 31;
    int rank = 0;
    long long group = blockIdx.x;
    if constexpr (C > 1) {
        rank = static_cast<int>(cluster_rank());
        group = cluster_index();
    }
    long long row = group * P + program;
    const bool active = row < a.rows;
    if (!active) row = a.rows - 1;                // replay the last row

    const long long base = row * static_cast<long long>(width);
    const T *xr = static_cast<const T *>(a.x) + base;
    const T *dr = static_cast<const T *>(a.dy) + base;
    T *outr = static_cast<T *>(a.dx) + base;

    int h = 0, tl = 0, nb;
    if constexpr (V == 4) {
        const int mis =
            static_cast<int>((reinterpret_cast<uintptr_t>(xr) / sizeof(T)) & (EV - 1));
        h = (EV - mis) & (EV - 1);
        if (h > width) h = width;
        nb = (width - h) / EV;
        tl = width - h - nb * EV;
    } else {
        nb = width;
    }
    const int gw = rank * W + worker;

    // ---- load both stripes once ---------------------------------------
    float v[K][EV], u[K][EV];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int i = k * (C * W) + gw;
        if (i < nb) {
            if constexpr (V == 4) {
                Elem<T>::load_vec(xr + h + EV * i, v[k]);
                Elem<T>::load_vec(dr + h + EV * i, u[k]);
            } else {
                v[k][0] = Elem<T>::load(xr + i);
                u[k][0] = Elem<T>::load(dr + i);
            }
        } else {
#pragma unroll
            for (int j = 0; j < EV; ++j) {
                v[k][j] = 0.0f;
                u[k][j] = 0.0f;
            }
        }
    }
    bool has_h = false, has_t = false;
    float hv = 0.0f, tv = 0.0f, hu = 0.0f, tu = 0.0f;
    int te = 0;
    if constexpr (V == 4) {
        has_h = (rank == 0) && (worker < h);
        has_t = (rank == 0) && (worker < tl);
        te = h + EV * nb + worker;
        if (has_h) {
            hv = Elem<T>::load(xr + worker);
            hu = Elem<T>::load(dr + worker);
        }
        if (has_t) {
            tv = Elem<T>::load(xr + te);
            tu = Elem<T>::load(dr + te);
        }
    }

    const float n = static_cast<float>(width);
    const float *gam = a.gamma;
    auto col_of = [&](int i) { return (V == 4) ? h + EV * i : i; };

    if constexpr (OP == BWD_SOFTMAX) {
        // ---- sum(dy * y), then dx = y (dy - sum) -------------------------
        float s[1] = {fmaf(hu, hv, tu * tv)};
#pragma unroll
        for (int k = 0; k < K; ++k)
#pragma unroll
            for (int j = 0; j < EV; ++j) s[0] = fmaf(u[k][j], v[k][j], s[0]);
        row_allreduce<Sum, 1, S, P, C>(s, part1, cpart, program, warp, lane);
        const float dot = s[0];
#pragma unroll
        for (int k = 0; k < K; ++k)
#pragma unroll
            for (int j = 0; j < EV; ++j) v[k][j] = v[k][j] * (u[k][j] - dot);
        hv = hv * (hu - dot);
        tv = tv * (tu - dot);
    } else {
        // ---- g = dy * gamma in place (2-byte rows, bound by instruction
        // issue: gamma as float4 when its phase allows; FP32 rows, bound by
        // DRAM, measured faster with scalar loads)
        if (gam != nullptr) {
            bool gvec = false;
            if constexpr (V == 4 && sizeof(T) == 2)
                gvec = (reinterpret_cast<uintptr_t>(gam + h) & 15) == 0;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int i = k * (C * W) + gw;
                if (i < nb) {
                    if (gvec) {
#pragma unroll
                        for (int q = 0; q < EV / 4; ++q) {
                            const float4 g4 =
                                __ldg(reinterpret_cast<const float4 *>(gam + col_of(i)) + q);
                            u[k][4 * q] *= g4.x;
                            u[k][4 * q + 1] *= g4.y;
                            u[k][4 * q + 2] *= g4.z;
                            u[k][4 * q + 3] *= g4.w;
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < EV; ++j) u[k][j] *= __ldg(gam + col_of(i) + j);
                    }
                }
            }
            if (has_h) hu *= __ldg(gam + worker);
            if (has_t) tu *= __ldg(gam + te);
        }
        // ---- row statistics and the two gradient sums -----------------------
        // The gradient sums need no extra reduction round: with d = x - m0
        // (LayerNorm) sum(g xhat) = rstd (sum(g d) - mu1 sum(g)), and for
        // RMSNorm sum(g xhat) = rstd sum(g x), so they are reduced together
        // with the statistics they depend on.
        float rstd, mean = 0.0f, mean_g = 0.0f, mean_gx;
        float ca = 0.0f, cb = 0.0f;   // 2-byte rows: dx = rstd g + ca v + cb, v = d (or x)
        if constexpr (OP == BWD_LN) {
            float s[1] = {hv + tv};
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int j = 0; j < EV; ++j) s[0] += v[k][j];
            row_allreduce<Sum, 1, S, P, C>(s, part1, cpart, program, warp, lane);
            const float mean0 = over_n<T>(s[0], n, a.inv_n);
            float q[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const bool ok = k * (C * W) + gw < nb;
#pragma unroll
                for (int j = 0; j < EV; ++j) {
                    const float d = ok ? v[k][j] - mean0 : 0.0f;
                    v[k][j] = d;
                    q[0] += d;
                    q[1] = fmaf(d, d, q[1]);
                    q[2] += u[k][j];
                    q[3] = fmaf(u[k][j], d, q[3]);
                }
            }
            hv = has_h ? hv - mean0 : 0.0f;
            tv = has_t ? tv - mean0 : 0.0f;
            q[0] += hv + tv;
            q[1] = fmaf(hv, hv, fmaf(tv, tv, q[1]));
            q[2] += hu + tu;
            q[3] = fmaf(hu, hv, fmaf(tu, tv, q[3]));
            row_allreduce<Sum, 4, S, P, C>(q, part2, cpart + 1, program, warp, lane);
            const float mu1 = over_n<T>(q[0], n, a.inv_n);
            const float var = fmaxf(over_n<T>(q[1], n, a.inv_n) - mu1 * mu1, 0.0f);
            rstd = inv_sqrt<T>(var + a.eps);
            mean = mean0 + mu1;
            mean_g = over_n<T>(q[2], n, a.inv_n);
            mean_gx = over_n<T>(rstd * fmaf(-mu1, q[2], q[3]), n, a.inv_n);
            if constexpr (sizeof(T) == 2) {
                // rstd (g - mean_g - (d - mu1) rstd mean_gx)
                ca = -rstd * rstd * mean_gx;
                cb = rstd * fmaf(rstd * mean_gx, mu1, -mean_g);
            } else {
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    const bool ok = k * (C * W) + gw < nb;
#pragma unroll
                    for (int j = 0; j < EV; ++j) v[k][j] = ok ? (v[k][j] - mu1) * rstd : 0.0f;
                }
                hv = has_h ? (hv - mu1) * rstd : 0.0f;
                tv = has_t ? (tv - mu1) * rstd : 0.0f;
            }
        } else {
            float q[2] = {fmaf(hv, hv, tv * tv), fmaf(hu, hv, tu * tv)};
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int j = 0; j < EV; ++j) {
                    q[0] = fmaf(v[k][j], v[k][j], q[0]);
                    q[1] = fmaf(u[k][j], v[k][j], q[1]);
                }
            row_allreduce<Sum, 2, S, P, C>(q, part1, cpart, program, warp, lane);
            rstd = inv_sqrt<T>(over_n<T>(q[0], n, a.inv_n) + a.eps);
            mean_gx = over_n<T>(rstd * q[1], n, a.inv_n);
            if constexpr (sizeof(T) == 2) {
                ca = -rstd * rstd * mean_gx;         // rstd (g - x rstd mean_gx)
            } else {
#pragma unroll
                for (int k = 0; k < K; ++k)
#pragma unroll
                    for (int j = 0; j < EV; ++j) v[k][j] *= rstd;
                hv *= rstd;
                tv *= rstd;
            }
        }

        if (a.stats != nullptr && active && worker == 0 && rank == 0) {
            a.stats[2 * row] = mean;
            a.stats[2 * row + 1] = rstd;
        }

        // ---- dx = rstd (g - mean(g) - xhat mean(g xhat)) ----------------------
        if constexpr (sizeof(T) == 2) {
            // 2-byte rows: written in d (or x) directly, rstd g + ca v + cb,
            // two FMAs (xhat is never formed)
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int j = 0; j < EV; ++j)
                    v[k][j] = fmaf(rstd, u[k][j], fmaf(ca, v[k][j], cb));
            hv = fmaf(rstd, hu, fmaf(ca, hv, cb));
            tv = fmaf(rstd, tu, fmaf(ca, tv, cb));
        } else {
            // FP32 rows: v holds xhat
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int j = 0; j < EV; ++j)
                    v[k][j] = rstd * (u[k][j] - mean_g - v[k][j] * mean_gx);
            hv = rstd * (hu - mean_g - hv * mean_gx);
            tv = rstd * (tu - mean_g - tv * mean_gx);
        }
    }

    if constexpr (C > 1) cluster_arrive();
    if (active) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int i = k * (C * W) + gw;
            if (i < nb) {
                if constexpr (V == 4)
                    Elem<T>::store_vec(outr + h + EV * i, v[k]);
                else
                    Elem<T>::store(outr + i, v[k][0]);
            }
        }
        if constexpr (V == 4) {
            if (has_h) Elem<T>::store(outr + worker, hv);
            if (has_t) Elem<T>::store(outr + te, tv);
        }
    }
    if constexpr (C > 1) cluster_wait();
}

}  // namespace tile

namespace tile {

// The two values of a 32-bit word of 2-byte elements (lower address in the
// low half), widened exactly.  Volatile asm, so the compiler widens again in
// every phase instead of keeping the widened values live (which would take
// back the registers the raw words save).
template <class T>
__device__ __forceinline__ void widen_word(unsigned int w, float &lo, float &hi) {
    if constexpr (std::is_same<T, __half>::value) {
        asm volatile("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
                     "cvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
                     : "=f"(lo), "=f"(hi) : "r"(w));
    } else {
        unsigned int a, b;
        asm volatile("shl.b32 %0, %2, 16;\n\tand.b32 %1, %2, 0xffff0000;"
                     : "=r"(a), "=r"(b) : "r"(w));
        lo = __uint_as_float(a);
        hi = __uint_as_float(b);
    }
}

template <class T>
__device__ __forceinline__ void widen_raw8(const unsigned int (&w)[4], float (&f)[8]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) widen_word<T>(w[i], f[2 * i], f[2 * i + 1]);
}

// v[j] = element j of a raw vector of 8 + c, one mixed-precision add
// (add.rn.f32.bf16 / .f16) per element: the 2-byte value enters exactly, so
// each lane is round(x + c) as after an explicit widening.  Volatile, like
// the widening, so that no phase keeps another phase's values live.
template <class T>
__device__ __forceinline__ void add_raw8(const unsigned int (&w)[4], float c, float (&v)[8]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (std::is_same<T, __half>::value)
            asm volatile("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
                         "add.rn.f32.f16 %0, lo, %3;\n\tadd.rn.f32.f16 %1, hi, %3;\n\t}"
                         : "=f"(v[2 * i]), "=f"(v[2 * i + 1]) : "r"(w[i]), "f"(c));
        else
            asm volatile("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
                         "add.rn.f32.bf16 %0, lo, %3;\n\tadd.rn.f32.bf16 %1, hi, %3;\n\t}"
                         : "=f"(v[2 * i]), "=f"(v[2 * i + 1]) : "r"(w[i]), "f"(c));
    }
}

// s[j % 4] += element j of a raw vector of 8, one mixed-precision add each.
template <class T>
__device__ __forceinline__ void acc_raw8(const unsigned int (&w)[4], float (&s)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (std::is_same<T, __half>::value)
            asm volatile("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
                         "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
                         : "+f"(s[(2 * i) & 3]), "+f"(s[(2 * i + 1) & 3]) : "r"(w[i]));
        else
            asm volatile("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
                         "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
                         : "+f"(s[(2 * i) & 3]), "+f"(s[(2 * i + 1) & 3]) : "r"(w[i]));
    }
}

// Mixed-precision fused multiply-add on two 2-byte operands and an FP32
// addend (fma.rn.f32.bf16 / .f16): the product of two BF16 or FP16 values is
// exact in FP32, so each step rounds once.
#define TILE_MIXED_FMA(TY)                                                               \
    "{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t" \
    "fma.rn.f32." TY " %0, al, bl, %0;\n\tfma.rn.f32." TY " %1, ah, bh, %1;\n\t}"

// (s0, s1) += the products of elements 2i and 2i + 1 of two raw vectors.
template <class T>
__device__ __forceinline__ void dot_raw8(const unsigned int (&a)[4], const unsigned int (&b)[4],
                                         float &s0, float &s1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (std::is_same<T, __half>::value)
            asm volatile(TILE_MIXED_FMA("f16") : "+f"(s0), "+f"(s1) : "r"(a[i]), "r"(b[i]));
        else
            asm volatile(TILE_MIXED_FMA("bf16") : "+f"(s0), "+f"(s1) : "r"(a[i]), "r"(b[i]));
    }
}

// Backward kernel for 2-byte rows of 16-byte vectors (BF16, FP16): the
// mapping and reduction order of row_bwd_kernel, but the two stripes hold the
// raw 2-byte words (4 per vector of 8) and every phase reads them again, so
// a register carries 4 bytes of DRAM data instead of 2 and a thread keeps as
// many bytes in flight as the FP32 kernel.  Where a phase needs x - m, a sum
// of x, or a product of two 2-byte values, mixed-precision adds and FMAs take
// the raw halves directly (each exact or rounded once, as after a
// widening); elsewhere the words are widened.  gamma comes in one 256-bit
// load per vector where g is used, and the output map
// dx = rstd g + ca d + cb runs on packed f32x2 pairs per vector just before
// its store.  G: gamma may be present (the host launches G = false for
// RMSNorm without gamma, whose kernel then has no gamma code).  WH: every
// row is 16-byte aligned and holds whole vectors, so the kernel carries no
// scalar head or tail (the same results: a head and tail of no elements add
// exact +0 terms, which can change only the sign of a zero).
template <int OP, class T, int S, int P, int K, int C, bool G, bool WH = false>
__global__ void __launch_bounds__(32 * S * P) row_bwd_raw_kernel(const BwdArgs a) {
    static_assert(sizeof(T) == 2, "2-byte element types");
    constexpr bool HT = !WH;   // the row may have a scalar head and tail
    static_assert(C == 1 || P == 1, "a cluster row has one program per CTA");
    constexpr int W = 32 * S;
    constexpr int EV = 8;

    __shared__ float part1[S > 1 ? 2 * P * S : 1];
    __shared__ float part2[S > 1 ? 4 * P * S : 1];
    __shared__ float cpart[C > 1 ? 5 : 1];

    if (blockDim.x != 32 * S * P) {
        if (threadIdx.x == 0) atomicOr(a.status, STATUS_BAD_LAUNCH);
        return;
    }
    const int width = a.width;
    const int tid = threadIdx.x;
    const int program = tid / W;
    const int worker = tid - program * W;
    const int warp = worker >> 5;
    const int lane = tid & 31;
    int rank = 0;
    long long group = blockIdx.x;
    if constexpr (C > 1) {
        rank = static_cast<int>(cluster_rank());
        group = cluster_index();
    }
    long long row = group * P + program;
    const bool active = row < a.rows;
    if (!active) row = a.rows - 1;                // replay the last row

    const long long base = row * static_cast<long long>(width);
    const T *xr = static_cast<const T *>(a.x) + base;
    const T *dr = static_cast<const T *>(a.dy) + base;
    T *outr = static_cast<T *>(a.dx) + base;

    int h = 0, nb = width / EV, tl = 0;
    if constexpr (HT) {
        const int mis = static_cast<int>((reinterpret_cast<uintptr_t>(xr) / sizeof(T)) & (EV - 1));
        h = (EV - mis) & (EV - 1);
        if (h > width) h = width;
        nb = (width - h) / EV;
        tl = width - h - nb * EV;
    }
    const int gw = rank * W + worker;

    // ---- load both stripes once, as raw words --------------------------
    unsigned int xw[K][4], dw[K][4];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int i = k * (C * W) + gw;
        if (i < nb) {
            const uint4 tx = __ldcs(reinterpret_cast<const uint4 *>(xr + h + EV * i));
            const uint4 td = __ldcs(reinterpret_cast<const uint4 *>(dr + h + EV * i));
            xw[k][0] = tx.x; xw[k][1] = tx.y; xw[k][2] = tx.z; xw[k][3] = tx.w;
            dw[k][0] = td.x; dw[k][1] = td.y; dw[k][2] = td.z; dw[k][3] = td.w;
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) xw[k][q] = dw[k][q] = 0u;   // +0.0 in both types
        }
    }
    const bool has_h = HT && (rank == 0) && (worker < h);
    const bool has_t = HT && (rank == 0) && (worker < tl);
    const int te = h + EV * nb + worker;
    float hv = 0.0f, tv = 0.0f, hu = 0.0f, tu = 0.0f;
    if (has_h) {
        hv = Elem<T>::load(xr + worker);
        hu = Elem<T>::load(dr + worker);
    }
    if (has_t) {
        tv = Elem<T>::load(xr + te);
        tu = Elem<T>::load(dr + te);
    }

    const float n = static_cast<float>(width);
    // G = false: no gamma (compiled out); G = true: gamma if a.gamma is set
    const float *gam = (OP != BWD_SOFTMAX && G) ? a.gamma : nullptr;
    const bool gvec = gam != nullptr && (reinterpret_cast<uintptr_t>(gam + h) & 15) == 0;
    const bool g32 = gam != nullptr && (reinterpret_cast<uintptr_t>(gam + h) & 31) == 0;
    if (gam != nullptr) {
        if (has_h) hu *= __ldg(gam + worker);
        if (has_t) tu *= __ldg(gam + te);
    }
    // g = dy * gamma of stripe vector k (column block i)
    auto vec_g = [&](int k, int i, float (&gf)[EV]) {
        widen_raw8<T>(dw[k], gf);
        if (gam != nullptr) {
            const float *gp = gam + h + EV * i;
            if (g32) {
                float gv[EV];
                ldg_v8(gp, gv);
#pragma unroll
                for (int j = 0; j < EV; ++j) gf[j] *= gv[j];
            } else if (gvec) {
#pragma unroll
                for (int q = 0; q < EV / 4; ++q) {
                    const float4 g4 = __ldg(reinterpret_cast<const float4 *>(gp) + q);
                    gf[4 * q] *= g4.x;
                    gf[4 * q + 1] *= g4.y;
                    gf[4 * q + 2] *= g4.z;
                    gf[4 * q + 3] *= g4.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < EV; ++j) gf[j] *= __ldg(gp + j);
            }
        }
    };
    // x (or y) and g of stripe vector k
    auto vec_xg = [&](int k, int i, float (&xf)[EV], float (&gf)[EV]) {
        widen_raw8<T>(xw[k], xf);
        vec_g(k, i, gf);
    };

    float mean0 = 0.0f, rstd = 1.0f, mean = 0.0f, ca = 0.0f, cb = 0.0f, dot = 0.0f;
    if constexpr (OP == BWD_SOFTMAX) {
        // ---- sum(dy * y) ---------------------------------------------------
        float s0 = HT ? fmaf(hu, hv, tu * tv) : 0.0f, s1 = 0.0f;
#pragma unroll
        for (int k = 0; k < K; ++k) dot_raw8<T>(dw[k], xw[k], s0, s1);   // empty slots add 0
        float s[1] = {s0 + s1};
        row_allreduce<Sum, 1, S, P, C>(s, part1, cpart, program, warp, lane);
        dot = s[0];
        hv = hv * (hu - dot);
        tv = tv * (tu - dot);
    } else {
        float mean_g = 0.0f, mean_gx;
        if constexpr (OP == BWD_LN) {
            // four independent partial sums (the first estimate of the mean
            // only shifts the data; measured faster than one chain or packed
            // pairs)
            float s4[4] = {HT ? hv + tv : 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int k = 0; k < K; ++k) acc_raw8<T>(xw[k], s4);   // empty slots add 0
            float s[1] = {(s4[0] + s4[1]) + (s4[2] + s4[3])};
            row_allreduce<Sum, 1, S, P, C>(s, part1, cpart, program, warp, lane);
            mean0 = over_n<T>(s[0], n, a.inv_n);
            float q[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int i = k * (C * W) + gw;
                if (i < nb) {
                    float d[EV], gf[EV];
                    add_raw8<T>(xw[k], -mean0, d);       // d = x - mean0
                    vec_g(k, i, gf);
#pragma unroll
                    for (int j = 0; j < EV; ++j) {
                        q[0] += d[j];
                        q[1] = fmaf(d[j], d[j], q[1]);
                        q[2] += gf[j];
                        q[3] = fmaf(gf[j], d[j], q[3]);
                    }
                }
            }
            if constexpr (HT) {
                hv = has_h ? hv - mean0 : 0.0f;
                tv = has_t ? tv - mean0 : 0.0f;
                q[0] += hv + tv;
                q[1] = fmaf(hv, hv, fmaf(tv, tv, q[1]));
                q[2] += hu + tu;
                q[3] = fmaf(hu, hv, fmaf(tu, tv, q[3]));
            }
            row_allreduce<Sum, 4, S, P, C>(q, part2, cpart + 1, program, warp, lane);
            const float mu1 = over_n<T>(q[0], n, a.inv_n);
            const float var = fmaxf(over_n<T>(q[1], n, a.inv_n) - mu1 * mu1, 0.0f);
            rstd = inv_sqrt<T>(var + a.eps);
            mean = mean0 + mu1;
            mean_g = over_n<T>(q[2], n, a.inv_n);
            mean_gx = over_n<T>(rstd * fmaf(-mu1, q[2], q[3]), n, a.inv_n);
            ca = -rstd * rstd * mean_gx;
            cb = rstd * fmaf(rstd * mean_gx, mu1, -mean_g);
        } else {
            float q0 = HT ? fmaf(hv, hv, tv * tv) : 0.0f, q1 = 0.0f;
            float g0 = HT ? fmaf(hu, hv, tu * tv) : 0.0f, g1 = 0.0f;
            if (gam == nullptr) {
                // sum x^2 and sum dy x straight from the raw words (mixed
                // fma: the products are exact), two accumulators each
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    dot_raw8<T>(xw[k], xw[k], q0, q1);        // empty slots add 0
                    dot_raw8<T>(dw[k], xw[k], g0, g1);
                }
            } else {
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    const int i = k * (C * W) + gw;
                    if (i < nb) {
                        float xf[EV], gf[EV];
                        vec_xg(k, i, xf, gf);
#pragma unroll
                        for (int j = 0; j < EV; ++j) {
                            q0 = fmaf(xf[j], xf[j], q0);
                            g0 = fmaf(gf[j], xf[j], g0);
                        }
                    }
                }
            }
            float q[2] = {q0 + q1, g0 + g1};
            row_allreduce<Sum, 2, S, P, C>(q, part1, cpart, program, warp, lane);
            rstd = inv_sqrt<T>(over_n<T>(q[0], n, a.inv_n) + a.eps);
            mean_gx = over_n<T>(rstd * q[1], n, a.inv_n);
            ca = -rstd * rstd * mean_gx;
        }
        if (a.stats != nullptr && active && worker == 0 && rank == 0) {
            a.stats[2 * row] = mean;
            a.stats[2 * row + 1] = rstd;
        }
        hv = fmaf(rstd, hu, fmaf(ca, hv, cb));
        tv = fmaf(rstd, tu, fmaf(ca, tv, cb));
    }

    if constexpr (C > 1) cluster_arrive();
    // ---- dx per vector, stored at once; the output map on packed pairs
    // (the same two FMAs per element, rounded the same way) --------------
    if (active) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int i = k * (C * W) + gw;
            if (i < nb) {
                float xf[EV], gf[EV], o[EV];
                if constexpr (OP == BWD_SOFTMAX) {
                    widen_raw8<T>(xw[k], xf);
                    widen_raw8<T>(dw[k], gf);
#pragma unroll
                    for (int j = 0; j < EV; j += 2) {
                        add_x2(gf[j], gf[j + 1], -dot, -dot);
                        o[j] = xf[j];
                        o[j + 1] = xf[j + 1];
                        mul_x2(o[j], o[j + 1], gf[j], gf[j + 1]);
                    }
                } else {
                    if constexpr (OP == BWD_LN) {
                        add_raw8<T>(xw[k], -mean0, xf);  // x - mean0
                        vec_g(k, i, gf);
                    } else {
                        vec_xg(k, i, xf, gf);
                    }
#pragma unroll
                    for (int j = 0; j < EV; j += 2) {
                        o[j] = cb;
                        o[j + 1] = cb;
                        fma_x2(o[j], o[j + 1], ca, ca, xf[j], xf[j + 1]);
                        fma_x2(o[j], o[j + 1], rstd, rstd, gf[j], gf[j + 1]);
                    }
                }
                Elem<T>::store_vec(outr + h + EV * i, o);
            }
        }
        if (has_h) Elem<T>::store(outr + worker, hv);
        if (has_t) Elem<T>::store(outr + te, tv);
    }
    if constexpr (C > 1) cluster_wait();
}

}  // namespace tile
