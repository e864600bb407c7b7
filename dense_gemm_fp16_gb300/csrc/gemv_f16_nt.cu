// gemv_f16_nt.cu -- C = A * B^T for very few rows of A (M <= 8): the
// matrix-vector regime of an LLM decode step.
//
// Same operation and numerics as gemm_f16_nt (half inputs, fp32 accumulation,
// one round-to-nearest-even per output), but with M this small every element
// of B is used only M times, so the product is bound by reading B from HBM,
// not by the tensor cores ("第 6 章 · Shared Memory & Tile", section "6.5.5
// GEMV (M=1)：LLM decode 完全不能用 tile": tiling has nothing to reuse; one
// warp per output row, a shuffle reduction).
//
// Design for sm_103a's HBM: each warp owns one row of B at a time (a dot
// product of K halves with each of the M rows of A) and streams it with
// 16-byte loads that bypass L1 allocation, four in flight per lane; the M rows
// of A (at most 8 x K halves) sit in shared memory, read as 16-byte vectors;
// the grid is a whole number of CTAs per SM; partial sums meet through warp
// shuffles.  Reading B once and A once per CTA, the algorithmic bytes are
// N*K*2 + M*K*2 + M*N*2.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "gemm.h"
#include "gemm_internal.h"

namespace gb300 {
namespace {

constexpr int kGemvWarps = 8;  // 256 threads per CTA

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// acc[m] += sum over the 8 halves of b . a_m
template <int MT>
__device__ __forceinline__ void dot8(float (&acc)[MT], const uint4 &bv, const uint4 (&av)[MT]) {
    const __half2 *b2 = reinterpret_cast<const __half2 *>(&bv);
    float2 bf[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) bf[q] = __half22float2(b2[q]);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const __half2 *a2 = reinterpret_cast<const __half2 *>(&av[m]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 af = __half22float2(a2[q]);
            acc[m] = fmaf(af.x, bf[q].x, acc[m]);
            acc[m] = fmaf(af.y, bf[q].y, acc[m]);
        }
    }
}

// VEC: K % 8 == 0 and A, B 16-byte aligned (16-byte vectors); else halves one by one.
template <int MT, bool VEC>
__global__ void __launch_bounds__(kGemvWarps * 32)
    gemv_f16_nt_kernel(int M, int N, int K, const __half *__restrict__ A,
                       const __half *__restrict__ B, __half *__restrict__ C) {
    extern __shared__ __align__(16) unsigned char gemv_smem[];
    __half *As = reinterpret_cast<__half *>(gemv_smem);  // [MT][K]
    // Programmatic dependent launch: nothing global before the predecessor is done.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    for (int i = threadIdx.x; i < MT * K; i += blockDim.x) {
        const int m = i / K;
        As[i] = m < M ? A[static_cast<size_t>(m) * K + (i - m * K)] : __float2half_rn(0.f);
    }
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int warp_global = blockIdx.x * kGemvWarps + (threadIdx.x >> 5);
    const int warps_total = gridDim.x * kGemvWarps;
    for (int n = warp_global; n < N; n += warps_total) {
        const __half *brow = B + static_cast<size_t>(n) * K;
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.f;
        if (VEC) {
            const int kv = K / 8;  // 16-byte vectors per row
            int v = lane;
            // four vectors of B in flight per lane
            for (; v + 96 < kv; v += 128) {
                uint4 bv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) bv[u] = ld_stream_v4(brow + (v + 32 * u) * 8);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint4 av[MT];
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        av[m] = *reinterpret_cast<const uint4 *>(As + m * K + (v + 32 * u) * 8);
                    dot8<MT>(acc, bv[u], av);
                }
            }
            for (; v < kv; v += 32) {
                const uint4 bv = ld_stream_v4(brow + v * 8);
                uint4 av[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) av[m] = *reinterpret_cast<const uint4 *>(As + m * K + v * 8);
                dot8<MT>(acc, bv, av);
            }
        } else {
            for (int k = lane; k < K; k += 32) {
                const float b = __half2float(brow[k]);
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[m] = fmaf(__half2float(As[m * K + k]), b, acc[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], off);
        }
        if (lane < MT && lane < M) {
            float out = acc[0];
#pragma unroll
            for (int m = 1; m < MT; ++m)
                if (lane == m) out = acc[m];
            C[static_cast<size_t>(lane) * N + n] = __float2half_rn(out);
        }
    }
}

template <int MT>
int launch_mt(const GemvLaunch &L, std::string &err) {
    const bool vec = (L.K % 8 == 0) &&
                     ((reinterpret_cast<uintptr_t>(L.A) | reinterpret_cast<uintptr_t>(L.B)) & 15u) == 0;
    const size_t smem = static_cast<size_t>(MT) * L.K * sizeof(__half);
    auto kernel = vec ? gemv_f16_nt_kernel<MT, true> : gemv_f16_nt_kernel<MT, false>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) {
            err = std::string("gemv: cudaFuncSetAttribute: ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
    }
    // Whole CTAs per SM, about one warp per row of B at most.
    const long long want = (static_cast<long long>(L.N) + kGemvWarps - 1) / kGemvWarps;
    const long long cap = static_cast<long long>(L.sm_count) * L.ctas_per_sm;
    const int grid = static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGemvWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, L.M, L.N, L.K, static_cast<const __half *>(L.A),
                                       static_cast<const __half *>(L.B), static_cast<__half *>(L.C));
    if (e != cudaSuccess) {
        err = std::string("gemv kernel launch: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

}  // namespace

int gemv_launch(const GemvLaunch &L, std::string &err) {
    if (L.M <= 1) return launch_mt<1>(L, err);
    if (L.M <= 2) return launch_mt<2>(L, err);
    if (L.M <= 4) return launch_mt<4>(L, err);
    if (L.M <= 8) return launch_mt<8>(L, err);
    err = "gemv: M > 8";
    return GEMM_ERR_INVALID_ARG;
}

}  // namespace gb300
