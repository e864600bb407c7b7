// epilogue.cuh -- the fused epilogue applied by the fp16 kernels before their
// single rounding to half: out = act(alpha * acc + bias[n] + beta * res[m][n]),
// "第 6 章 · Shared Memory & Tile", section "6.5.4 Epilogue 融合" (bias and
// activation applied while the accumulators are still on chip, saving a
// round trip of C through HBM), with the usual GEMM scalars and residual.
//
// The epilogue warps have the length of one tile's main loop to finish a
// tile, so the residual's global-load latency must not be paid once per 8
// columns: a slab's residual loads are all issued before its accumulators are
// read, the tile's residual rows are prefetched to L2 before the accumulator
// wait, and the activations use the SFU's tanh (one instruction).
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

#include "gemm_internal.h"

namespace gb300 {

struct Epi {
    float alpha, beta;
    const __half *bias;  // [N] or null
    const __half *res;   // [M, N] or null; not read when beta == 0
    int act;             // 0 none, 1 ReLU, 2 SiLU, 3 tanh-GELU
    int on;              // 0: plain product
    int vec;             // bias and res 16-byte aligned and N % 8 == 0: vector loads
    __device__ __forceinline__ bool reads_res() const { return res != nullptr && beta != 0.f; }
};

// tanh on the special-function unit: relative error about 2^-11, the size of
// the half rounding that follows it.
__device__ __forceinline__ float tanh_sfu(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The activation, fixed at compile time in the tile kernels (one kernel per
// activation keeps each kernel's code small: the epilogue warps share the
// SM's instruction cache with the MMA and TMA warps).
template <int ACT>
__device__ __forceinline__ float epi_act(float v) {
    if constexpr (ACT == 1) {
        return fmaxf(v, 0.f);
    } else if constexpr (ACT == 2) {
        // SiLU v * sigmoid(v), with sigmoid(v) = (1 + tanh(v / 2)) / 2
        return 0.5f * v * (1.f + tanh_sfu(0.5f * v));
    } else if constexpr (ACT == 3) {
        // GELU, tanh form: 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))
        const float u = 0.7978845608028654f * fmaf(0.044715f * v, v * v, v);
        return 0.5f * v * (1.f + tanh_sfu(u));
    } else {
        return v;
    }
}

// The same chosen at run time (matrix-vector and K = 0 kernels).
__device__ __forceinline__ float epi_activate(float v, int act) {
    if (act == 1) return epi_act<1>(v);
    if (act == 2) return epi_act<2>(v);
    if (act == 3) return epi_act<3>(v);
    return v;
}

template <int ACT>
__device__ __forceinline__ float epi_value(const Epi &e, float acc, float b, float r) {
    return epi_act<ACT>(fmaf(e.beta, r, fmaf(e.alpha, acc, b)));
}

// The activation on two values at once: packed fp32 arithmetic (fma.rn.f32x2,
// each half rounded like fmaf) halves the instructions of the tile epilogue.
// GELU is evaluated as h + h tanh(u), h = v/2, u = v (c0 + c1 v^2) with
// c0 = sqrt(2/pi), c1 = 0.044715 sqrt(2/pi); SiLU as h + h tanh(h).
template <int ACT>
__device__ __forceinline__ float2 epi_act2(float2 v) {
    if constexpr (ACT == 1) {
        return make_float2(fmaxf(v.x, 0.f), fmaxf(v.y, 0.f));
    } else if constexpr (ACT == 2) {
        const float2 h = __fmul2_rn(v, make_float2(0.5f, 0.5f));
        return __ffma2_rn(h, make_float2(tanh_sfu(h.x), tanh_sfu(h.y)), h);
    } else if constexpr (ACT == 3) {
        constexpr float c0 = 0.7978845608028654f, c1 = 0.7978845608028654f * 0.044715f;
        const float2 p = __ffma2_rn(make_float2(c1, c1), __fmul2_rn(v, v), make_float2(c0, c0));
        const float2 u = __fmul2_rn(v, p);
        const float2 h = __fmul2_rn(v, make_float2(0.5f, 0.5f));
        return __ffma2_rn(h, make_float2(tanh_sfu(u.x), tanh_sfu(u.y)), h);
    } else {
        return v;
    }
}

// Halves p[n .. n+7] (zeros past N) as one 16-byte word.
__device__ __forceinline__ uint4 load_half8(const __half *p, bool vec, int n, int N) {
    if (vec && n + 8 <= N) return *reinterpret_cast<const uint4 *>(p + n);
    uint4 out;
    uint16_t *h = reinterpret_cast<uint16_t *>(&out);
#pragma unroll
    for (int j = 0; j < 8; ++j) h[j] = (n + j < N) ? __half_as_ushort(p[n + j]) : uint16_t(0);
    return out;
}

// Residual of row m, columns n .. n+7 (zeros when R is not read or m >= M).
__device__ __forceinline__ uint4 epi_load_res8(const Epi &e, int m, int n, int M, int N) {
    if (!e.reads_res() || m >= M) return make_uint4(0u, 0u, 0u, 0u);
    return load_half8(e.res + static_cast<size_t>(m) * N, e.vec, n, N);
}

// The bias of columns n0 + 8j .. n0 + 8j + 7 for the lane j < NQ (the same for
// every row): each of the first NQ lanes holds one 16-byte word, handed to
// the others with shuffles.
template <int NQ>
__device__ __forceinline__ uint4 epi_load_bias_lane(const Epi &e, int n0, int lane, int N) {
    if (e.bias == nullptr || lane >= NQ) return make_uint4(0u, 0u, 0u, 0u);
    return load_half8(e.bias, e.vec, n0 + 8 * lane, N);
}

__device__ __forceinline__ uint4 shfl_u4(const uint4 &v, int src) {
    return make_uint4(__shfl_sync(0xffffffffu, v.x, src), __shfl_sync(0xffffffffu, v.y, src),
                      __shfl_sync(0xffffffffu, v.z, src), __shfl_sync(0xffffffffu, v.w, src));
}

// Eight consecutive fp32 accumulators (raw bits) through the epilogue, in place.
template <int ACT>
__device__ __forceinline__ void epi_apply8(const Epi &e, uint32_t *acc, const uint4 &bias8,
                                           const uint4 &res8) {
    const __half2 *b2 = reinterpret_cast<const __half2 *>(&bias8);
    const __half2 *r2 = reinterpret_cast<const __half2 *>(&res8);
    const float2 alpha = make_float2(e.alpha, e.alpha), beta = make_float2(e.beta, e.beta);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 a = make_float2(__uint_as_float(acc[2 * q]), __uint_as_float(acc[2 * q + 1]));
        float2 v = __ffma2_rn(alpha, a, __half22float2(b2[q]));
        v = epi_act2<ACT>(__ffma2_rn(beta, __half22float2(r2[q]), v));
        acc[2 * q] = __float_as_uint(v.x);
        acc[2 * q + 1] = __float_as_uint(v.y);
    }
}

// One output whose bias and residual were loaded (or are 0); activation chosen at run time.
__device__ __forceinline__ float epi_apply1(const Epi &e, float acc, float b, float r) {
    return epi_activate(fmaf(e.beta, r, fmaf(e.alpha, acc, b)), e.act);
}

// Ask L2 for the residual of row m, columns [n0, n0 + ncols), ahead of use.
__device__ __forceinline__ void epi_prefetch_res(const Epi &e, int m, int n0, int ncols, int M, int N) {
    if (!e.reads_res() || m >= M || n0 >= N) return;
    const int n1 = n0 + ncols < N ? n0 + ncols : N;
    // Every address stays inside the row's range: one per 128 bytes from the
    // first byte, then the last byte (whose line the stride may have skipped).
    const char *row = reinterpret_cast<const char *>(e.res + static_cast<size_t>(m) * N);
    const char *first = row + 2 * static_cast<size_t>(n0);
    const char *last = row + 2 * static_cast<size_t>(n1) - 1;
    for (const char *a = first; a <= last; a += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(last));
}

inline Epi make_epi(const EpiSpec &s, int N) {
    Epi e;
    e.alpha = s.alpha;
    e.beta = s.beta;
    e.bias = static_cast<const __half *>(s.bias);
    e.res = static_cast<const __half *>(s.res);
    e.act = s.act;
    e.on = s.on;
    e.vec = (N % 8 == 0) &&
            ((reinterpret_cast<uintptr_t>(s.bias) | reinterpret_cast<uintptr_t>(s.res)) & 15u) == 0;
    return e;
}

}  // namespace gb300
