// Fused FP32 row-normalisation kernel for sm_103a: one template, four ops.
//
// Mapping (after "Cooperating-program packing", section "Implementation
// boundary"): a CTA of T = 32*S*P threads runs P row programs of W = 32*S
// cooperating workers each.  With C > 1 one row is split over a thread-block
// cluster of C CTAs (P = 1), which is how rows too wide for one CTA's
// registers are handled.
//
// Every worker loads its elements of the row exactly once into a register
// stripe (float4 accesses where the row is 16-byte aligned, a scalar head
// and tail otherwise), and every later phase reads the stripe, never global
// memory -- the input-reuse scheme of "Immutable input reuse in Metal
// reductions" (execution map e = (chunk*W + worker)*V + v, resource map
// stripe_slot = chunk*V + v).  Reductions go warp shuffle -> P*S shared
// partials -> (C > 1) C cluster partials read through distributed shared
// memory; every level combines in a fixed order, so a plan is bitwise
// deterministic.  A packed CTA whose last programs fall past the final row
// replays the last row and predicates only its stores, so every barrier is
// unconditional.
#pragma once

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "launch.h"

namespace tile {

// Bits of the per-library device error word (read by tile_check_device_status).
enum { STATUS_BAD_LAUNCH = 1u };

// ---------------------------------------------------------------------------
// memory access.  Inputs are read once and outputs written once, so both use
// the streaming cache hint (evict-first).  Elem<T> moves one element or one
// 16-byte vector (4 FP32 or 8 BF16 values) between memory and FP32
// registers; BF16 widens exactly and narrows with round-to-nearest-even.
// ---------------------------------------------------------------------------
template <class T>
struct Elem;

template <>
struct Elem<float> {
    static constexpr int kVec = 4;
    __device__ static void load_vec(const float *p, float (&v)[4]) {
        const float4 t = __ldcs(reinterpret_cast<const float4 *>(p));
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    }
    __device__ static void store_vec(float *p, const float (&v)[4]) {
        __stcs(reinterpret_cast<float4 *>(p), make_float4(v[0], v[1], v[2], v[3]));
    }
    __device__ static float load(const float *p) { return __ldcs(p); }
    __device__ static void store(float *p, float v) { __stcs(p, v); }
};

template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kVec = 8;
    __device__ static float widen(unsigned int bits16) { return __uint_as_float(bits16 << 16); }
    __device__ static unsigned int narrow(float v) {
        return static_cast<unsigned int>(__bfloat16_as_ushort(__float2bfloat16_rn(v)));
    }
    // Two values per 32-bit word: the low half is the element at the lower
    // address; widening is a shift, narrowing one paired conversion.
    __device__ static unsigned int narrow2(float lo, float hi) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const unsigned int *>(&h);
    }
    __device__ static void load_vec(const __nv_bfloat16 *p, float (&v)[8]) {
        const uint4 t = __ldcs(reinterpret_cast<const uint4 *>(p));
        const unsigned int w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static void store_vec(__nv_bfloat16 *p, const float (&v)[8]) {
        uint4 t;
        t.x = narrow2(v[0], v[1]);
        t.y = narrow2(v[2], v[3]);
        t.z = narrow2(v[4], v[5]);
        t.w = narrow2(v[6], v[7]);
        __stcs(reinterpret_cast<uint4 *>(p), t);
    }
    __device__ static float load(const __nv_bfloat16 *p) {
        return widen(__ldcs(reinterpret_cast<const unsigned short *>(p)));
    }
    __device__ static void store(__nv_bfloat16 *p, float v) {
        __stcs(reinterpret_cast<unsigned short *>(p), static_cast<unsigned short>(narrow(v)));
    }
};

template <>
struct Elem<__half> {
    static constexpr int kVec = 8;
    // Two values per 32-bit word (lower address in the low half); widening
    // is exact, narrowing one paired round-to-nearest-even conversion.
    __device__ static float2 widen2(unsigned int w) {
        return __half22float2(*reinterpret_cast<const __half2 *>(&w));
    }
    __device__ static unsigned int narrow2(float lo, float hi) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const unsigned int *>(&h);
    }
    __device__ static void load_vec(const __half *p, float (&v)[8]) {
        const uint4 t = __ldcs(reinterpret_cast<const uint4 *>(p));
        const unsigned int w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = widen2(w[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    __device__ static void store_vec(__half *p, const float (&v)[8]) {
        uint4 t;
        t.x = narrow2(v[0], v[1]);
        t.y = narrow2(v[2], v[3]);
        t.z = narrow2(v[4], v[5]);
        t.w = narrow2(v[6], v[7]);
        __stcs(reinterpret_cast<uint4 *>(p), t);
    }
    __device__ static float load(const __half *p) {
        return __half2float(__ushort_as_half(__ldcs(reinterpret_cast<const unsigned short *>(p))));
    }
    __device__ static void store(__half *p, float v) {
        __stcs(reinterpret_cast<unsigned short *>(p), __half_as_ushort(__float2half_rn(v)));
    }
};

// exp(t), t <= 0 or -inf, for the softmax numerators.  FP32 rows call expf.
// 2-byte rows (BF16, FP16), whose outputs keep 8 or 11 significant bits,
// use the identity
// e^t = 2^(t log2 e) with the hardware base-2 exponential (PTX
// ex2.approx.ftz.f32, relative error about 2^-22; ex2(-inf) = +0): rounding
// t log2 e adds a relative error of at most |t| ln(2) 2^-24, about 1e-6 at
// t = -20, where e^t is already below 1e-8; both stay far inside half an
// ulp of the output (2^-9 BF16, 2^-12 FP16).  It takes a fraction of expf's
// instructions, which matters because 2-byte rows carry twice the elements
// per byte.
template <class T>
__device__ __forceinline__ float softmax_exp(float t) {
    if constexpr (sizeof(T) == 2) {
        float r;
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t * 1.4426950408889634f));
        return r;
    } else {
        return expf(t);
    }
}

// LayerNorm output map of a centred value d (centred on the mean estimate,
// with mu1 the remaining mean offset): (d - mu1) rstd.  FP32 rows use that
// form, which is exactly 0 for a constant row (every d equals mu1).  2-byte
// rows (BF16, FP16), whose kernels are bound by instruction issue and whose
// outputs keep 8 or 11 significant bits, use one FMA, d rstd + (-mu1 rstd):
// it differs from the
// two-step form by at most the rounding of mu1 rstd (mu1 is the rounding
// error of the mean estimate, so about 2^-24 |mean| rstd), and a constant
// row gives |y| of that order instead of an exact 0.
template <class T>
__device__ __forceinline__ float ln_out(float d, float mu1, float rstd) {
    if constexpr (sizeof(T) == 2)
        return fmaf(d, rstd, -mu1 * rstd);
    else
        return (d - mu1) * rstd;
}

// Row statistics from the reduced sums: s / n and 1 / sqrt(t).  FP32 rows
// take both as correctly rounded operations.  2-byte rows (BF16, FP16),
// whose kernels are bound by instruction issue and whose outputs keep 8 or
// 11 significant bits, multiply by 1 / n rounded once on the host (relative
// error at most 2^-23 against 2^-24 for the division) and take rsqrtf (at
// most 2 ulp, the CUDA math library's bound): one instruction each instead
// of a division or square-root sequence, with errors far inside half an ulp
// of the output.  (The mean estimate only centres the row, so its rounding
// does not reach the result.)
template <class T>
__device__ __forceinline__ float over_n(float s, float n, float inv_n) {
    if constexpr (sizeof(T) == 2)
        return s * inv_n;
    else
        return s / n;
}
template <class T>
__device__ __forceinline__ float inv_sqrt(float t) {
    if constexpr (sizeof(T) == 2)
        return rsqrtf(t);
    else
        return 1.0f / sqrtf(t);
}

// v[j] += the 16-byte vector `t` of element type T (4 FP32 or 8 BF16 / FP16
// lanes, the lower address in the lower half of each word).  2-byte lanes
// use the mixed-precision add (PTX add.rn.f32.bf16 / add.rn.f32.f16, sm_100
// and later): the 2-byte operand is widened exactly inside the instruction,
// so each lane is round(v + x) as after an explicit widening, one
// instruction instead of two.
template <class T>
__device__ __forceinline__ void add_raw_vec(float (&v)[16 / sizeof(T)], uint4 t) {
    if constexpr (sizeof(T) == 4) {
        v[0] += __uint_as_float(t.x);
        v[1] += __uint_as_float(t.y);
        v[2] += __uint_as_float(t.z);
        v[3] += __uint_as_float(t.w);
    } else {
        const unsigned int w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (std::is_same<T, __half>::value)
                asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
                    "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
                    : "+f"(v[2 * i]), "+f"(v[2 * i + 1])
                    : "r"(w[i]));
            else
                asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
                    "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
                    : "+f"(v[2 * i]), "+f"(v[2 * i + 1])
                    : "r"(w[i]));
        }
    }
}

// Eight consecutive FP32 values from a 32-byte aligned address in one
// 256-bit load (sm_100 and later): a warp's loads then cover one contiguous
// kilobyte, where two 16-byte loads per thread (32 bytes apart between
// threads) each span a kilobyte for half of it and double the L1 traffic.
// Volatile, so that no phase keeps another phase's values live.
__device__ __forceinline__ void ldg_v8(const float *p, float (&v)[8]) {
    asm volatile("ld.global.nc.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]),
                   "=f"(v[6]), "=f"(v[7])
                 : "l"(p));
}

// ---------------------------------------------------------------------------
// Lane-wise arithmetic on a vector of EV FP32 lanes.  With PK (BF16 rows,
// whose kernels are bound by instruction issue) two lanes go through one
// packed instruction (PTX add / mul / fma .rn.f32x2, sm_100 and later); each
// lane is rounded exactly as by the scalar instruction, so the results are
// the same bit for bit with half the arithmetic instructions.  Without PK
// (FP32 rows, bound by DRAM) the scalar loop is kept.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void add_x2(float &a0, float &a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb;\n\tmov.b64 ra, {%0, %1};\n\tmov.b64 rb, {%2, %3};\n\t"
        "add.rn.f32x2 ra, ra, rb;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1) : "f"(b0), "f"(b1));
}
__device__ __forceinline__ void mul_x2(float &a0, float &a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb;\n\tmov.b64 ra, {%0, %1};\n\tmov.b64 rb, {%2, %3};\n\t"
        "mul.rn.f32x2 ra, ra, rb;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1) : "f"(b0), "f"(b1));
}
// (a0, a1) = (b0 * c0 + a0, b1 * c1 + a1), fused
__device__ __forceinline__ void fma_x2(float &a0, float &a1, float b0, float b1, float c0,
                                       float c1) {
    asm("{\n\t.reg .b64 ra, rb, rc;\n\tmov.b64 ra, {%0, %1};\n\tmov.b64 rb, {%2, %3};\n\t"
        "mov.b64 rc, {%4, %5};\n\tfma.rn.f32x2 ra, rb, rc, ra;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1) : "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// a[j] += b[j]
template <bool PK, int EV>
__device__ __forceinline__ void vadd(float (&a)[EV], const float (&b)[EV]) {
    if constexpr (PK && EV % 2 == 0) {
#pragma unroll
        for (int j = 0; j < EV; j += 2) add_x2(a[j], a[j + 1], b[j], b[j + 1]);
    } else {
#pragma unroll
        for (int j = 0; j < EV; ++j) a[j] += b[j];
    }
}
// a[j] += c
template <bool PK, int EV>
__device__ __forceinline__ void vadd_c(float (&a)[EV], float c) {
    if constexpr (PK && EV % 2 == 0) {
#pragma unroll
        for (int j = 0; j < EV; j += 2) add_x2(a[j], a[j + 1], c, c);
    } else {
#pragma unroll
        for (int j = 0; j < EV; ++j) a[j] += c;
    }
}
// a[j] *= c
template <bool PK, int EV>
__device__ __forceinline__ void vmul_c(float (&a)[EV], float c) {
    if constexpr (PK && EV % 2 == 0) {
#pragma unroll
        for (int j = 0; j < EV; j += 2) mul_x2(a[j], a[j + 1], c, c);
    } else {
#pragma unroll
        for (int j = 0; j < EV; ++j) a[j] *= c;
    }
}
// acc[j] = fma(d[j], d[j], acc[j])
template <bool PK, int EV>
__device__ __forceinline__ void vsq_acc(float (&acc)[EV], const float (&d)[EV]) {
    if constexpr (PK && EV % 2 == 0) {
#pragma unroll
        for (int j = 0; j < EV; j += 2) fma_x2(acc[j], acc[j + 1], d[j], d[j + 1], d[j], d[j + 1]);
    } else {
#pragma unroll
        for (int j = 0; j < EV; ++j) acc[j] = fmaf(d[j], d[j], acc[j]);
    }
}
// a[j] = fma(a[j], b, c)
template <bool PK, int EV>
__device__ __forceinline__ void vfma_c(float (&a)[EV], float b, float c) {
    if constexpr (PK && EV % 2 == 0) {
#pragma unroll
        for (int j = 0; j < EV; j += 2) {
            float c0 = c, c1 = c;
            fma_x2(c0, c1, a[j], a[j + 1], b, b);
            a[j] = c0;
            a[j + 1] = c1;
        }
    } else {
#pragma unroll
        for (int j = 0; j < EV; ++j) a[j] = fmaf(a[j], b, c);
    }
}
// a[j] = fma(a[j], b[j], c[j])
template <bool PK, int EV>
__device__ __forceinline__ void vfma(float (&a)[EV], const float (&b)[EV], const float (&c)[EV]) {
    if constexpr (PK && EV % 2 == 0) {
#pragma unroll
        for (int j = 0; j < EV; j += 2) {
            float c0 = c[j], c1 = c[j + 1];
            fma_x2(c0, c1, a[j], a[j + 1], b[j], b[j + 1]);
            a[j] = c0;
            a[j + 1] = c1;
        }
    } else {
#pragma unroll
        for (int j = 0; j < EV; ++j) a[j] = fmaf(a[j], b[j], c[j]);
    }
}

// ---------------------------------------------------------------------------
// cluster primitives (inline PTX)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
// Read a float from the shared memory of CTA `rank` of this cluster, at the
// address `local` has in this CTA's shared window.
__device__ __forceinline__ float load_dsmem(const float *local, uint32_t rank) {
    uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t remote;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// ---------------------------------------------------------------------------
// reductions
// ---------------------------------------------------------------------------
struct Sum {
    __device__ static float apply(float a, float b) { return a + b; }
};
struct Max {
    __device__ static float apply(float a, float b) { return fmaxf(a, b); }
};

// Combine per-vector-lane accumulators in a fixed pairwise order.
template <int N>
__device__ __forceinline__ float lane_total(const float (&a)[N]) {
    if constexpr (N == 1) {
        return a[0];
    } else {
        float t[N / 2];
#pragma unroll
        for (int i = 0; i < N / 2; ++i) t[i] = a[2 * i] + a[2 * i + 1];
        return lane_total(t);
    }
}
template <int N>
__device__ __forceinline__ float lane_max(const float (&a)[N]) {
    if constexpr (N == 1) {
        return a[0];
    } else {
        float t[N / 2];
#pragma unroll
        for (int i = 0; i < N / 2; ++i) t[i] = fmaxf(a[2 * i], a[2 * i + 1]);
        return lane_max(t);
    }
}

// xor butterfly: every lane ends with the same value (IEEE + and max are
// commutative, so lane i and lane i^o compute the same pair).
template <class Op, int N>
__device__ __forceinline__ void warp_allreduce(float (&v)[N]) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int i = 0; i < N; ++i)
            v[i] = Op::apply(v[i], __shfl_xor_sync(0xffffffffu, v[i], o));
    }
}

// All-reduce of N values over one row program: warp -> S shared partials of
// this program -> C cluster partials.  part: [N][P*S] floats, cpart: [N].
// Each call site passes its own part/cpart so no phase overwrites a buffer
// another thread may still be reading.
template <class Op, int N, int S, int P, int C>
__device__ __forceinline__ void row_allreduce(float (&v)[N], float *part, float *cpart,
                                              int program, int warp, int lane) {
    warp_allreduce<Op, N>(v);
    if constexpr (S > 1) {
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < N; ++i) part[i * P * S + program * S + warp] = v[i];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < N; ++i) {
            float t = part[i * P * S + program * S];
#pragma unroll
            for (int w = 1; w < S; ++w) t = Op::apply(t, part[i * P * S + program * S + w]);
            v[i] = t;
        }
    }
    if constexpr (C > 1) {
        if (threadIdx.x == 0) {
#pragma unroll
            for (int i = 0; i < N; ++i) cpart[i] = v[i];
        }
        cluster_arrive();
        cluster_wait();
#pragma unroll
        for (int i = 0; i < N; ++i) {
            float t = load_dsmem(&cpart[i], 0);
#pragma unroll
            for (int q = 1; q < C; ++q) t = Op::apply(t, load_dsmem(&cpart[i], q));
            v[i] = t;
        }
    }
}

// Compensated (error-free) sum of pairs: (s, c) holds s + c with s the FP32
// sum and c the accumulated rounding errors.  Knuth's TwoSum gives the exact
// error of one addition (The Art of Computer Programming, vol. 2, 4.2.2);
// the combine is commutative in its result, so xor butterflies stay uniform.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
__device__ __forceinline__ void comp_add(float &s, float &c, float v) {
    float e;
    two_sum(s, v, s, e);
    c = __fadd_rn(c, e);
}
__device__ __forceinline__ void comp_merge(float &s, float &c, float s2, float c2) {
    float e;
    two_sum(s, s2, s, e);
    c = __fadd_rn(__fadd_rn(c, c2), e);
}

template <int S, int P, int C>
__device__ __forceinline__ void row_allreduce_comp(float &s, float &c, float *part, float *cpart,
                                                   int program, int warp, int lane) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        const float c2 = __shfl_xor_sync(0xffffffffu, c, o);
        comp_merge(s, c, s2, c2);
    }
    if constexpr (S > 1) {
        if (lane == 0) {
            part[program * S + warp] = s;
            part[P * S + program * S + warp] = c;
        }
        __syncthreads();
        s = part[program * S];
        c = part[P * S + program * S];
#pragma unroll
        for (int w = 1; w < S; ++w) comp_merge(s, c, part[program * S + w], part[P * S + program * S + w]);
    }
    if constexpr (C > 1) {
        if (threadIdx.x == 0) {
            cpart[0] = s;
            cpart[1] = c;
        }
        cluster_arrive();
        cluster_wait();
        s = load_dsmem(&cpart[0], 0);
        c = load_dsmem(&cpart[1], 0);
#pragma unroll
        for (int q = 1; q < C; ++q) comp_merge(s, c, load_dsmem(&cpart[0], q), load_dsmem(&cpart[1], q));
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

// Resident CTAs the register budget must allow: 2-byte rows of 16-byte
// vectors with a stripe of at most 32 floats are held to 64 registers a
// thread (the count these plans reach without gamma's 256-bit loads; at 70
// registers BF16 LayerNorm lost a CTA per SM and ran 4 % slower at 4096
// columns); other plans leave the count to the compiler.
template <class T, int V, int S, int P, int K>
constexpr int row_min_blocks() {
    return (sizeof(T) == 2 && V == 4 && K * 8 <= 32) ? 32 / (S * P) : 0;
}

// WH (whole vectors; V = 4 only): every row starts on a 16-byte boundary and
// holds whole vectors, so the row has no scalar head or tail and the kernel
// carries none of their loads, sums and stores.  The launcher takes it when
// the rows are aligned and the width is a multiple of the vector; the
// results are bitwise those of the general kernel (a head and tail of zero
// elements contribute exact +0 terms, which can change only the sign of a
// partial sum that is exactly -0, and so of a zero result).
template <int OP, class T, int V, int S, int P, int K, int C, bool WH = false>
__global__ void __launch_bounds__(32 * S * P, (row_min_blocks<T, V, S, P, K>()))
    row_kernel(const RowArgs a) {
    static_assert(V == 1 || V == 4, "V is 1 (scalar) or 4 (16-byte vectors)");
    static_assert(!WH || V == 4, "whole-vector rows are read as 16-byte vectors");
    // the row may have a scalar head and tail
    constexpr bool HT = V == 4 && !WH;
    // elements per access: one 16-byte vector (4 FP32 or 8 BF16), or one
    constexpr int EV = (V == 4) ? Elem<T>::kVec : 1;
    static_assert(C == 1 || P == 1, "a cluster row has one program per CTA");
    static_assert(32 * S * P <= 1024, "at most 1024 threads per CTA");
    constexpr int W = 32 * S;
    // Empty stripe slots hold the identity of the first reduction: -inf for
    // the softmax maximum, NaN for min/max (fmaxf ignores a NaN operand, for
    // x and for -x alike), 0 for sums.
    constexpr float kFill = (OP == OP_SOFTMAX) ? -INFINITY : (OP == OP_MINMAX) ? NAN : 0.0f;
    constexpr bool kRowOutput = (OP == OP_SUM || OP == OP_MINMAX);
    // BF16 LayerNorm rows of 16-byte vectors, the op with the most lane
    // arithmetic: packed pairs (BF16 LayerNorm 166 -> 159 us at 65536x4096),
    // except in 1024-thread CTAs, whose 64-register cap the paired operands
    // (aligned register pairs) would push into spills.  BF16 RMSNorm and
    // softmax measured no gain at 4096 columns and a loss at 12288-16384.
    constexpr bool PK = sizeof(T) == 2 && V == 4 && 32 * S * P <= 512 &&
                        (OP == OP_LN || OP == OP_RESLN);

    __shared__ float part1[S > 1 ? 2 * P * S : 1];
    __shared__ float part2[S > 1 ? 2 * P * S : 1];
    __shared__ float cpart[C > 1 ? 4 : 1];

    if (blockDim.x != 32 * S * P) {           // uniform over the grid
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
    const T *rr = (OP == OP_RESLN) ? static_cast<const T *>(a.r) + base : nullptr;
    T *yr = kRowOutput ? nullptr : static_cast<T *>(a.y) + base;

    // Row geometry.  V = 4: h scalars up to the first 16-byte boundary, then
    // nb vectors of EV elements, then tl scalars.  All row pointers share the
    // 16-byte phase.
    int h = 0, tl = 0, nb;
    if constexpr (WH) {
        nb = width / EV;
    } else if constexpr (V == 4) {
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

    // ---- a1: load the row once into the register stripe ----------------
    float v[K][EV];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int i = k * (C * W) + gw;
        if (i < nb) {
            if constexpr (V == 4) {
                Elem<T>::load_vec(xr + h + EV * i, v[k]);
                if constexpr (OP == OP_RESLN) {
                    if constexpr (sizeof(T) == 2) {
                        add_raw_vec<T>(v[k], __ldcs(reinterpret_cast<const uint4 *>(rr + h + EV * i)));
                    } else {
                        float b[EV];
                        Elem<T>::load_vec(rr + h + EV * i, b);
                        vadd<PK, EV>(v[k], b);
                    }
                }
            } else {
                float t = Elem<T>::load(xr + i);
                if constexpr (OP == OP_RESLN) t += Elem<T>::load(rr + i);
                v[k][0] = t;
            }
        } else {
#pragma unroll
            for (int j = 0; j < EV; ++j) v[k][j] = kFill;
        }
    }
    bool has_h = false, has_t = false;
    float hv = kFill, tv = kFill;
    int te = 0;
    if constexpr (HT) {
        has_h = (rank == 0) && (worker < h);
        has_t = (rank == 0) && (worker < tl);
        te = h + EV * nb + worker;
        if (has_h) {
            hv = Elem<T>::load(xr + worker);
            if constexpr (OP == OP_RESLN) hv += Elem<T>::load(rr + worker);
        }
        if (has_t) {
            tv = Elem<T>::load(xr + te);
            if constexpr (OP == OP_RESLN) tv += Elem<T>::load(rr + te);
        }
    }

    const float n = static_cast<float>(width);
    float row_out0 = 0.0f, row_out1 = 0.0f;       // per-row results (sum, min/max)
    if constexpr (OP == OP_RESLN || OP == OP_LN) {
        // ---- a2: mean estimate (one accumulator per vector lane) ----------
        float acc[EV];
#pragma unroll
        for (int j = 0; j < EV; ++j) acc[j] = 0.0f;
#pragma unroll
        for (int k = 0; k < K; ++k) vadd<PK, EV>(acc, v[k]);
        float s[1] = {HT ? lane_total(acc) + (hv + tv) : lane_total(acc)};
        row_allreduce<Sum, 1, S, P, C>(s, part1, cpart, program, warp, lane);
        const float mean0 = over_n<T>(s[0], n, a.inv_n);
        // ---- a3: centre in place; reduce (sum d, sum d^2) -----------------
        float a1[EV], a2[EV];
#pragma unroll
        for (int j = 0; j < EV; ++j) a1[j] = a2[j] = 0.0f;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const bool ok = k * (C * W) + gw < nb;
            if constexpr (PK) {
                // d = v + (-mean0) is v - mean0 exactly; empty slots give 0
                if (ok) {
                    vadd_c<PK, EV>(v[k], -mean0);
                    vadd<PK, EV>(a1, v[k]);
                    vsq_acc<PK, EV>(a2, v[k]);
                } else {
#pragma unroll
                    for (int j = 0; j < EV; ++j) v[k][j] = 0.0f;
                }
            } else {
#pragma unroll
                for (int j = 0; j < EV; ++j) {
                    const float d = ok ? v[k][j] - mean0 : 0.0f;
                    v[k][j] = d;
                    a1[j] += d;
                    a2[j] = fmaf(d, d, a2[j]);
                }
            }
        }
        hv = has_h ? hv - mean0 : 0.0f;
        tv = has_t ? tv - mean0 : 0.0f;
        float q[2] = {HT ? lane_total(a1) + (hv + tv) : lane_total(a1),
                      HT ? fmaf(hv, hv, fmaf(tv, tv, lane_total(a2))) : lane_total(a2)};
        row_allreduce<Sum, 2, S, P, C>(q, part2, cpart + 1, program, warp, lane);
        // corrected two-pass: mean = mean0 + mu1, var = E[d^2] - mu1^2
        const float mu1 = over_n<T>(q[0], n, a.inv_n);
        const float var = fmaxf(over_n<T>(q[1], n, a.inv_n) - mu1 * mu1, 0.0f);
        const float rstd = inv_sqrt<T>(var + a.eps);
        if constexpr (PK) {
            const float nb_shift = -mu1 * rstd;      // ln_out<T>: one FMA per lane
#pragma unroll
            for (int k = 0; k < K; ++k) vfma_c<PK, EV>(v[k], rstd, nb_shift);
        } else {
#pragma unroll
            for (int k = 0; k < K; ++k)
#pragma unroll
                for (int j = 0; j < EV; ++j) v[k][j] = ln_out<T>(v[k][j], mu1, rstd);
        }
        hv = ln_out<T>(hv, mu1, rstd);
        tv = ln_out<T>(tv, mu1, rstd);
    } else if constexpr (OP == OP_RMS) {
        // ---- a2: mean square ---------------------------------------------
        float acc[EV];
#pragma unroll
        for (int j = 0; j < EV; ++j) acc[j] = 0.0f;
#pragma unroll
        for (int k = 0; k < K; ++k) vsq_acc<PK, EV>(acc, v[k]);
        float s[1] = {HT ? fmaf(hv, hv, fmaf(tv, tv, lane_total(acc))) : lane_total(acc)};
        row_allreduce<Sum, 1, S, P, C>(s, part1, cpart, program, warp, lane);
        const float rstd = inv_sqrt<T>(over_n<T>(s[0], n, a.inv_n) + a.eps);
#pragma unroll
        for (int k = 0; k < K; ++k) vmul_c<PK, EV>(v[k], rstd);
        hv *= rstd;
        tv *= rstd;
    } else if constexpr (OP == OP_SOFTMAX) {
        // ---- a2: row maximum (empty slots hold -inf) ---------------------
        float mj[EV];
#pragma unroll
        for (int j = 0; j < EV; ++j) mj[j] = kFill;
#pragma unroll
        for (int k = 0; k < K; ++k)
#pragma unroll
            for (int j = 0; j < EV; ++j) mj[j] = fmaxf(mj[j], v[k][j]);
        float m[1] = {HT ? fmaxf(lane_max(mj), fmaxf(hv, tv)) : lane_max(mj)};
        row_allreduce<Max, 1, S, P, C>(m, part1, cpart, program, warp, lane);
        const float mx = m[0];
        // ---- a3: exponentiate in place (exp(-inf) = 0), reduce the sum ---
        float acc[EV];
#pragma unroll
        for (int j = 0; j < EV; ++j) acc[j] = 0.0f;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            if constexpr (PK) {
                vadd_c<PK, EV>(v[k], -mx);                      // v - mx, exactly
#pragma unroll
                for (int j = 0; j < EV; ++j) v[k][j] = softmax_exp<T>(v[k][j]);
                vadd<PK, EV>(acc, v[k]);
            } else {
#pragma unroll
                for (int j = 0; j < EV; ++j) {
                    const float e = softmax_exp<T>(v[k][j] - mx);
                    v[k][j] = e;
                    acc[j] += e;
                }
            }
        }
        hv = softmax_exp<T>(hv - mx);
        tv = softmax_exp<T>(tv - mx);
        float s[1] = {HT ? lane_total(acc) + (hv + tv) : lane_total(acc)};
        row_allreduce<Sum, 1, S, P, C>(s, part2, cpart + 1, program, warp, lane);
        const float inv = 1.0f / s[0];
#pragma unroll
        for (int k = 0; k < K; ++k) vmul_c<PK, EV>(v[k], inv);
        hv *= inv;
        tv *= inv;
    } else if constexpr (OP == OP_SUM) {
        // ---- compensated row sum (empty slots hold 0) --------------------
        float s = 0.0f, c = 0.0f;
#pragma unroll
        for (int k = 0; k < K; ++k)
#pragma unroll
            for (int j = 0; j < EV; ++j) comp_add(s, c, v[k][j]);
        if constexpr (HT) {
            comp_add(s, c, hv);
            comp_add(s, c, tv);
        }
        row_allreduce_comp<S, P, C>(s, c, part1, cpart, program, warp, lane);
        row_out0 = __fadd_rn(s, c);
    } else {
        // ---- paired min/max: max(x) and max(-x) in one reduction ---------
        float hi[EV], lo[EV];
#pragma unroll
        for (int j = 0; j < EV; ++j) hi[j] = lo[j] = kFill;
#pragma unroll
        for (int k = 0; k < K; ++k)
#pragma unroll
            for (int j = 0; j < EV; ++j) {
                hi[j] = fmaxf(hi[j], v[k][j]);
                lo[j] = fmaxf(lo[j], -v[k][j]);
            }
        float m[2] = {HT ? fmaxf(lane_max(hi), fmaxf(hv, tv)) : lane_max(hi),
                      HT ? fmaxf(lane_max(lo), fmaxf(-hv, -tv)) : lane_max(lo)};
        row_allreduce<Max, 2, S, P, C>(m, part1, cpart, program, warp, lane);
        row_out0 = -m[1];
        row_out1 = m[0];
    }

    // Our cluster partials must stay readable until every CTA of the
    // cluster has read them: arrive now (no cluster read follows), wait
    // after the stores.
    if constexpr (C > 1) cluster_arrive();

    // Optional per-column scale and shift (affine LayerNorm, weighted
    // RMSNorm): y = y * gamma[col] + beta[col], loaded through the read-only
    // cache (every row reuses them).  float4 loads when gamma/beta share the
    // row's 16-byte phase (one 256-bit load per 8-column vector of a 2-byte
    // row when they are 32-byte aligned), scalar loads otherwise.  2-byte
    // rows store each vector as soon as it is scaled, so a vector's gamma
    // and beta registers and its stripe slot are free before the next one
    // is loaded.
    bool vec_stored = false;
    if constexpr (OP == OP_RESLN || OP == OP_LN || OP == OP_RMS) {
        if (a.gamma != nullptr) {
            const float *g = a.gamma;
            const float *b = a.beta;
            bool gvec = false, g32 = false;
            if constexpr (V == 4) {
                gvec = ((reinterpret_cast<uintptr_t>(g + h) & 15) == 0) &&
                       (b == nullptr || (reinterpret_cast<uintptr_t>(b + h) & 15) == 0);
                if constexpr (EV == 8)       // 2-byte rows: one 256-bit load each
                    g32 = ((reinterpret_cast<uintptr_t>(g + h) & 31) == 0) &&
                          (b == nullptr || (reinterpret_cast<uintptr_t>(b + h) & 31) == 0);
            }
            if constexpr (EV == 8) {
                // one loop per load form, chosen once per launch; replayed
                // programs store nothing and skip it
                vec_stored = true;
                auto apply = [&](auto load) {
                    if (!active) return;
#pragma unroll
                    for (int k = 0; k < K; ++k) {
                        const int i = k * (C * W) + gw;
                        if (i < nb) {
                            float gg[EV], bb[EV];
                            load(h + EV * i, gg, bb);
                            vfma<PK, EV>(v[k], gg, bb);
                            Elem<T>::store_vec(yr + h + EV * i, v[k]);
                        }
                    }
                };
                auto scalar = [&](int col, float (&gg)[EV], float (&bb)[EV]) {
#pragma unroll
                    for (int j = 0; j < EV; ++j) {
                        gg[j] = __ldg(g + col + j);
                        bb[j] = b != nullptr ? __ldg(b + col + j) : 0.0f;
                    }
                };
                if constexpr (V == 4) {
                    auto quad = [&](int col, float (&gg)[EV], float (&bb)[EV]) {
#pragma unroll
                        for (int q = 0; q < EV / 4; ++q) {
                            const float4 g4 = __ldg(reinterpret_cast<const float4 *>(g + col) + q);
                            gg[4 * q] = g4.x; gg[4 * q + 1] = g4.y;
                            gg[4 * q + 2] = g4.z; gg[4 * q + 3] = g4.w;
                            float4 b4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                            if (b != nullptr) b4 = __ldg(reinterpret_cast<const float4 *>(b + col) + q);
                            bb[4 * q] = b4.x; bb[4 * q + 1] = b4.y;
                            bb[4 * q + 2] = b4.z; bb[4 * q + 3] = b4.w;
                        }
                    };
                    if constexpr (EV == 8) {
                        auto wide = [&](int col, float (&gg)[EV], float (&bb)[EV]) {
                            ldg_v8(g + col, gg);
                            if (b != nullptr) {
                                ldg_v8(b + col, bb);
                            } else {
#pragma unroll
                                for (int j = 0; j < EV; ++j) bb[j] = 0.0f;
                            }
                        };
                        if (g32) apply(wide);
                        else if (gvec) apply(quad);
                        else apply(scalar);
                    } else {
                        if (gvec) apply(quad);
                        else apply(scalar);
                    }
                } else {
                    apply(scalar);
                }
            } else {
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    const int i = k * (C * W) + gw;
                    if (i < nb) {
                        const int col = (V == 4) ? h + EV * i : i;
                        float gg[EV], bb[EV];
                        bool loaded = false;
                        if constexpr (V == 4 && EV == 8) {
                            if (g32) {
                                ldg_v8(g + col, gg);
                                if (b != nullptr) {
                                    ldg_v8(b + col, bb);
                                } else {
#pragma unroll
                                    for (int j = 0; j < EV; ++j) bb[j] = 0.0f;
                                }
                                loaded = true;
                            }
                        }
                        if constexpr (V == 4) {
                            if (!loaded && gvec) {
#pragma unroll
                                for (int q = 0; q < EV / 4; ++q) {
                                    const float4 g4 =
                                        __ldg(reinterpret_cast<const float4 *>(g + col) + q);
                                    gg[4 * q] = g4.x; gg[4 * q + 1] = g4.y;
                                    gg[4 * q + 2] = g4.z; gg[4 * q + 3] = g4.w;
                                    float4 b4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                                    if (b != nullptr)
                                        b4 = __ldg(reinterpret_cast<const float4 *>(b + col) + q);
                                    bb[4 * q] = b4.x; bb[4 * q + 1] = b4.y;
                                    bb[4 * q + 2] = b4.z; bb[4 * q + 3] = b4.w;
                                }
                                loaded = true;
                            }
                        }
                        if (!loaded) {
#pragma unroll
                            for (int j = 0; j < EV; ++j) {
                                gg[j] = __ldg(g + col + j);
                                bb[j] = b != nullptr ? __ldg(b + col + j) : 0.0f;
                            }
                        }
                        vfma<PK, EV>(v[k], gg, bb);
                    }
                }
            }
            if constexpr (HT) {
                if (has_h) hv = fmaf(hv, __ldg(g + worker), b != nullptr ? __ldg(b + worker) : 0.0f);
                if (has_t) tv = fmaf(tv, __ldg(g + te), b != nullptr ? __ldg(b + te) : 0.0f);
            }
        }
    }

    // ---- a4: streaming stores, predicated for replayed programs ---------
    if constexpr (kRowOutput) {
        if (active && worker == 0 && rank == 0) {
            static_cast<float *>(a.y)[row] = row_out0;
            if constexpr (OP == OP_MINMAX) a.y2[row] = row_out1;
        }
    } else {
        if (active) {
            if (!vec_stored) {
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    const int i = k * (C * W) + gw;
                    if (i < nb) {
                        if constexpr (V == 4)
                            Elem<T>::store_vec(yr + h + EV * i, v[k]);
                        else
                            Elem<T>::store(yr + i, v[k][0]);
                    }
                }
            }
            if constexpr (HT) {
                if (has_h) Elem<T>::store(yr + worker, hv);
                if (has_t) Elem<T>::store(yr + te, tv);
            }
        }
    }
    if constexpr (C > 1) cluster_wait();
}

}  // namespace tile
