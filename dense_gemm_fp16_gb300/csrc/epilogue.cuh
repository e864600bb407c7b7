// epilogue.cuh -- the fused epilogue applied by the fp16 kernels before their
// single rounding to half: out = act(alpha * acc + bias[n] + beta * res[m][n]),
// "第 6 章 · Shared Memory & Tile", section "6.5.4 Epilogue 融合" (bias and
// activation applied while the accumulators are still on chip, saving a
// round trip of C through HBM), with the usual GEMM scalars and residual.
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
};

__device__ __forceinline__ float epi_activate(float v, int act) {
    if (act == 1) return fmaxf(v, 0.f);
    if (act == 2) return v / (1.f + __expf(-v));  // SiLU: v * sigmoid(v)
    if (act == 3) {
        // GELU, tanh form: 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))
        const float u = 0.7978845608028654f * fmaf(0.044715f * v, v * v, v);
        return 0.5f * v * (1.f + tanhf(u));
    }
    return v;
}

__device__ __forceinline__ void load_half8(const __half *p, bool vec, int n, int N, float (&out)[8]) {
    if (vec && n + 8 <= N) {
        const uint4 v = *reinterpret_cast<const uint4 *>(p + n);
        const __half2 *h = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 f = __half22float2(h[q]);
            out[2 * q] = f.x;
            out[2 * q + 1] = f.y;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) out[j] = (n + j < N) ? __half2float(p[n + j]) : 0.f;
    }
}

// Eight consecutive fp32 accumulators (columns n .. n+7 of row m, held as
// raw bits) through the fused epilogue, in place.
__device__ __forceinline__ void epi_apply8(const Epi &e, uint32_t *acc, int m, int n, int M, int N) {
    float b[8], r[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) b[j] = r[j] = 0.f;
    if (e.bias) load_half8(e.bias, e.vec, n, N, b);
    if (e.res && e.beta != 0.f && m < M) load_half8(e.res + static_cast<size_t>(m) * N, e.vec, n, N, r);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float v = fmaf(e.alpha, __uint_as_float(acc[j]), b[j]);
        v = fmaf(e.beta, r[j], v);
        acc[j] = __float_as_uint(epi_activate(v, e.act));
    }
}

// The same for one output.
__device__ __forceinline__ float epi_apply1(const Epi &e, float acc, int m, int n, int N) {
    float v = e.alpha * acc;
    if (e.bias) v += __half2float(e.bias[n]);
    if (e.res && e.beta != 0.f) v = fmaf(e.beta, __half2float(e.res[static_cast<size_t>(m) * N + n]), v);
    return epi_activate(v, e.act);
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
