// sgemm.cu -- C = alpha * A * B + beta * C in fp32 on the CUDA cores.
//
// Row-major A [M,K], B [K,N], C [M,N].  The operation and its alpha/beta
// epilogue are those of the gemm_cp_async kernel in "异步拷贝与 Hopper/Blackwell
// 新特性" (anrans.github.io/ai-infra-handbooks/cuda/advanced/async-hopper),
// section "cp.async 与多级流水 sm_80+"; beta == 0 follows the BLAS convention
// (C is not read).  fp32 semantics exclude TF32, so the work is plain FFMA.
//
// Design: each CTA of 256 threads owns a BM x BN tile of C; every thread owns
// a TM x TN register micro-tile made of 4 x 4 blocks spread BM/RM rows and
// BN/RN columns apart ("第 6 章 · Shared Memory & Tile", section "6.3.1 寄存器
// tile").  K is walked in BK = 8 slices through two shared-memory buffers: the
// next slice is fetched from global memory into registers while the current
// one is multiplied, then stored, so one __syncthreads per slice suffices.
// A is stored transposed (As[k][m]) so that every thread reads its rows as
// float4; the +4 padding of each As row puts the two k-halves a warp writes
// on disjoint banks (section "6.4 Bank Conflict" of the same page).  Warps
// are 4 x 8 thread blocks of the 16 x 16 thread grid, so a warp's float4 reads
// of As and Bs touch 64 B and 128 B respectively: one wavefront each.
// Out-of-range rows, columns and k are loaded as zeros and never stored, which
// makes any M, N, K exact.
#include <cuda_runtime.h>

#include "gemm.h"
#include "gemm_internal.h"

namespace gb300 {
namespace {

constexpr int kSgemmThreads = 256;
constexpr int kBK = 8;

template <int BM, int BN, int TM, int TN>
struct SgemmCfg {
    static constexpr int RM = TM / 4;  // 4-row groups per thread
    static constexpr int RN = TN / 4;  // 4-column groups per thread
    static constexpr int kAPitch = BM + 4;
    static_assert((BM / TM) * (BN / TN) == kSgemmThreads, "16 x 16 thread grid");
    static_assert(BM / TM == 16 && BN / TN == 16, "thread grid layout assumes 16 x 16");
    static_assert(TM % 4 == 0 && TN % 4 == 0, "micro-tiles are 4 x 4 blocks");
};

template <bool VEC>
__device__ __forceinline__ float4 load4(const float *__restrict__ p, bool row_ok, int col,
                                        int ncols) {
    // Four consecutive elements p[col .. col+3] of one row, zero beyond ncols.
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!row_ok) return v;
    if (VEC) {
        // ncols % 4 == 0 and col % 4 == 0: the group is entirely in or out.
        if (col < ncols) v = *reinterpret_cast<const float4 *>(p + col);
    } else {
        if (col + 0 < ncols) v.x = p[col + 0];
        if (col + 1 < ncols) v.y = p[col + 1];
        if (col + 2 < ncols) v.z = p[col + 2];
        if (col + 3 < ncols) v.w = p[col + 3];
    }
    return v;
}

template <int BM, int BN, int TM, int TN, bool VEC>
__global__ void __launch_bounds__(kSgemmThreads)
    sgemm_kernel(int M, int N, int K, float alpha, const float *__restrict__ A,
                 const float *__restrict__ B, float beta, float *__restrict__ C) {
    using Cfg = SgemmCfg<BM, BN, TM, TN>;
    constexpr int RM = Cfg::RM, RN = Cfg::RN, AP = Cfg::kAPitch;
    constexpr int A_LOADS = (BM * kBK / 4 + kSgemmThreads - 1) / kSgemmThreads;
    constexpr int B_LOADS = (BN * kBK / 4 + kSgemmThreads - 1) / kSgemmThreads;

    __shared__ __align__(16) float As[2][kBK][AP];
    __shared__ __align__(16) float Bs[2][kBK][BN];

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int ty = (warp >> 1) * 4 + (lane >> 3);  // 0..15
    const int tx = (warp & 1) * 8 + (lane & 7);    // 0..15
    const int m0 = blockIdx.y * BM;
    const int n0 = blockIdx.x * BN;

    float4 ra[A_LOADS], rb[B_LOADS];

    auto fetch = [&](int k0) {
#pragma unroll
        for (int l = 0; l < A_LOADS; ++l) {
            const int idx = tid + l * kSgemmThreads;
            if (idx < BM * kBK / 4) {
                const int row = idx / (kBK / 4), kq = idx % (kBK / 4);
                const int m = m0 + row;
                ra[l] = load4<VEC>(A + static_cast<size_t>(m < M ? m : 0) * K, m < M, k0 + kq * 4, K);
            }
        }
#pragma unroll
        for (int l = 0; l < B_LOADS; ++l) {
            const int idx = tid + l * kSgemmThreads;
            if (idx < BN * kBK / 4) {
                const int kr = idx / (BN / 4), nq = idx % (BN / 4);
                const int k = k0 + kr;
                rb[l] = load4<VEC>(B + static_cast<size_t>(k < K ? k : 0) * N, k < K, n0 + nq * 4, N);
            }
        }
    };
    auto stash = [&](int buf) {
#pragma unroll
        for (int l = 0; l < A_LOADS; ++l) {
            const int idx = tid + l * kSgemmThreads;
            if (idx < BM * kBK / 4) {
                const int row = idx / (kBK / 4), kq = idx % (kBK / 4);
                As[buf][kq * 4 + 0][row] = ra[l].x;
                As[buf][kq * 4 + 1][row] = ra[l].y;
                As[buf][kq * 4 + 2][row] = ra[l].z;
                As[buf][kq * 4 + 3][row] = ra[l].w;
            }
        }
#pragma unroll
        for (int l = 0; l < B_LOADS; ++l) {
            const int idx = tid + l * kSgemmThreads;
            if (idx < BN * kBK / 4) {
                const int kr = idx / (BN / 4), nq = idx % (BN / 4);
                *reinterpret_cast<float4 *>(&Bs[buf][kr][nq * 4]) = rb[l];
            }
        }
    };

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

    const int KT = (K + kBK - 1) / kBK;
    if (KT > 0) {
        fetch(0);
        stash(0);
    }
    __syncthreads();
    for (int kt = 0; kt < KT; ++kt) {
        const int cur = kt & 1;
        if (kt + 1 < KT) fetch((kt + 1) * kBK);
#pragma unroll
        for (int k = 0; k < kBK; ++k) {
            float a[TM], b[TN];
#pragma unroll
            for (int g = 0; g < RM; ++g) {
                const float4 v = *reinterpret_cast<const float4 *>(&As[cur][k][g * (BM / RM) + ty * 4]);
                a[g * 4 + 0] = v.x; a[g * 4 + 1] = v.y; a[g * 4 + 2] = v.z; a[g * 4 + 3] = v.w;
            }
#pragma unroll
            for (int g = 0; g < RN; ++g) {
                const float4 v = *reinterpret_cast<const float4 *>(&Bs[cur][k][g * (BN / RN) + tx * 4]);
                b[g * 4 + 0] = v.x; b[g * 4 + 1] = v.y; b[g * 4 + 2] = v.z; b[g * 4 + 3] = v.w;
            }
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (kt + 1 < KT) stash(cur ^ 1);
        __syncthreads();
    }

    // Epilogue: C = alpha * acc + beta * C, masked; C is not read when beta == 0.
#pragma unroll
    for (int gi = 0; gi < RM; ++gi) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = m0 + gi * (BM / RM) + ty * 4 + i;
            if (m >= M) continue;
            float *crow = C + static_cast<size_t>(m) * N;
#pragma unroll
            for (int gj = 0; gj < RN; ++gj) {
                const int n = n0 + gj * (BN / RN) + tx * 4;
                const float *av = &acc[gi * 4 + i][gj * 4];
                if (VEC) {
                    if (n < N) {
                        float4 o = make_float4(alpha * av[0], alpha * av[1], alpha * av[2], alpha * av[3]);
                        if (beta != 0.f) {
                            const float4 c = *reinterpret_cast<const float4 *>(crow + n);
                            o.x = fmaf(beta, c.x, o.x);
                            o.y = fmaf(beta, c.y, o.y);
                            o.z = fmaf(beta, c.z, o.z);
                            o.w = fmaf(beta, c.w, o.w);
                        }
                        *reinterpret_cast<float4 *>(crow + n) = o;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (n + j < N) {
                            float o = alpha * av[j];
                            if (beta != 0.f) o = fmaf(beta, crow[n + j], o);
                            crow[n + j] = o;
                        }
                    }
                }
            }
        }
    }
}

// C = beta * C (K == 0: the product term is an empty sum); beta == 0 writes zeros.
__global__ void scale_kernel(float *C, size_t count, float beta) {
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < count; i += stride)
        C[i] = (beta == 0.f) ? 0.f : beta * C[i];
}

template <int BM, int BN, int TM, int TN>
int launch_tile(const SgemmLaunch &L, std::string &err) {
    const dim3 grid((L.N + BN - 1) / BN, (L.M + BM - 1) / BM);
    const bool vec = (L.K % 4 == 0) && (L.N % 4 == 0) &&
                     ((reinterpret_cast<uintptr_t>(L.A) | reinterpret_cast<uintptr_t>(L.B) |
                       reinterpret_cast<uintptr_t>(L.C)) & 15u) == 0;
    if (vec)
        sgemm_kernel<BM, BN, TM, TN, true><<<grid, kSgemmThreads, 0, L.stream>>>(
            L.M, L.N, L.K, L.alpha, L.A, L.B, L.beta, L.C);
    else
        sgemm_kernel<BM, BN, TM, TN, false><<<grid, kSgemmThreads, 0, L.stream>>>(
            L.M, L.N, L.K, L.alpha, L.A, L.B, L.beta, L.C);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        err = std::string("sgemm kernel launch: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

}  // namespace

int sgemm_launch(const SgemmLaunch &L, std::string &err) {
    if (L.K == 0) {
        const size_t count = static_cast<size_t>(L.M) * L.N;
        const int blocks = static_cast<int>((count + 255) / 256 < 4096 ? (count + 255) / 256 : 4096);
        scale_kernel<<<blocks, 256, 0, L.stream>>>(L.C, count, L.beta);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) {
            err = std::string("scale launch: ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
        return GEMM_OK;
    }
    switch (L.variant) {
        case GEMM_SGEMM_128x128: return launch_tile<128, 128, 8, 8>(L, err);
        case GEMM_SGEMM_64x64: return launch_tile<64, 64, 4, 4>(L, err);
        default: err = "unknown sgemm variant"; return GEMM_ERR_INVALID_ARG;
    }
}

}  // namespace gb300
