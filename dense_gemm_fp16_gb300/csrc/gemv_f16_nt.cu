// gemv_f16_nt.cu -- C = A * B^T for one or two rows of A (M <= 2): the
// matrix-vector regime of an LLM decode step.
//
// Same operation and numerics as gemm_f16_nt (half inputs, fp32 accumulation,
// one round-to-nearest-even per output), but with M this small every element
// of B is used only M times, so the product is bound by reading B from HBM
// (from M = 3 on, the fp32 FMAs on the CUDA cores no longer keep pace with
// HBM and the tensor-core path is faster; measured at N = 16384, K = 8192),
// not by the tensor cores ("第 6 章 · Shared Memory & Tile", section "6.5.5
// GEMV (M=1)：LLM decode 完全不能用 tile": tiling has nothing to reuse; one
// warp per output row, a shuffle reduction).
//
// Design for sm_103a's HBM: B is streamed once with 16-byte loads that skip
// L1 allocation; each CTA takes a balanced block of rows (the grid is a whole
// number of CTAs per SM) and its warps split every row's K range, so no warp
// waits on a longer share of rows than the others; the M rows of A (at most
// 2 x K halves) sit in shared memory, read as 16-byte vectors; partial sums
// meet through warp shuffles and a small shared array.  Reading B once and A
// once per CTA, the algorithmic bytes are N*K*2 + M*K*2 + M*N*2.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "epilogue.cuh"
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
//
// Work split: CTA b owns rows [b*N/G, (b+1)*N/G) of B (balanced to one row),
// and all its warps share every row: warp w reads the w-th eighth of the row's
// K range.  Rows go kGemvRows at a time with kVec 16-byte vectors of each in
// flight per lane; each warp's partial dot products meet in a double-buffered
// shared array, so one barrier per group of rows suffices, and the first
// kGemvRows * M threads finish the sums.
template <int MT, int kGemvRows, int kVec, bool VEC>
__global__ void __launch_bounds__(kGemvWarps * 32)
    gemv_f16_nt_kernel(int M, int N, int K, const __half *__restrict__ A,
                       const __half *__restrict__ B, __half *__restrict__ C, const Epi epi) {
    extern __shared__ __align__(16) unsigned char gemv_smem[];
    __shared__ float red[2][kGemvWarps][kGemvRows][MT];
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
    const int warp = threadIdx.x >> 5;
    const int r0 = static_cast<int>(static_cast<long long>(blockIdx.x) * N / gridDim.x);
    const int r1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * N / gridDim.x);
    // this warp's slice of K: whole 16-byte vectors (VEC) or single halves
    const int units = VEC ? K / 8 : K;
    const int u0 = static_cast<int>(static_cast<long long>(warp) * units / kGemvWarps);
    const int u1 = static_cast<int>(static_cast<long long>(warp + 1) * units / kGemvWarps);

    int buf = 0;
    for (int n0 = r0; n0 < r1; n0 += kGemvRows, buf ^= 1) {
        // The finishing threads fetch their bias and residual now; the loads
        // complete under this group's dot products.
        float eb = 0.f, er = 0.f;
        if (epi.on && threadIdx.x < kGemvRows * MT) {
            const int r = threadIdx.x / MT, m = threadIdx.x % MT;
            if (n0 + r < r1 && m < M) {
                if (epi.bias) eb = __half2float(epi.bias[n0 + r]);
                if (epi.reads_res()) er = __half2float(epi.res[static_cast<size_t>(m) * N + n0 + r]);
            }
        }
        float acc[kGemvRows][MT];
#pragma unroll
        for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;
        if (VEC) {
            for (int u = u0 + lane; u < u1; u += 32 * kVec) {
                // up to kVec vectors of each of the rows in flight per lane
                uint4 bv[kGemvRows][kVec];
#pragma unroll
                for (int r = 0; r < kGemvRows; ++r) {
                    const int n = n0 + r < r1 ? n0 + r : r1 - 1;
                    const __half *brow = B + static_cast<size_t>(n) * K;
#pragma unroll
                    for (int h = 0; h < kVec; ++h)
                        if (u + 32 * h < u1) bv[r][h] = ld_stream_v4(brow + (u + 32 * h) * 8);
                }
#pragma unroll
                for (int h = 0; h < kVec; ++h) {
                    if (u + 32 * h >= u1) break;
                    uint4 av[MT];
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        av[m] = *reinterpret_cast<const uint4 *>(As + m * K + (u + 32 * h) * 8);
#pragma unroll
                    for (int r = 0; r < kGemvRows; ++r) dot8<MT>(acc[r], bv[r][h], av);
                }
            }
        } else {
            for (int k = u0 + lane; k < u1; k += 32) {
#pragma unroll
                for (int r = 0; r < kGemvRows; ++r) {
                    const int n = n0 + r < r1 ? n0 + r : r1 - 1;
                    const float b = __half2float(B[static_cast<size_t>(n) * K + k]);
#pragma unroll
                    for (int m = 0; m < MT; ++m) acc[r][m] = fmaf(__half2float(As[m * K + k]), b, acc[r][m]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], off);
            }
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
                for (int m = 0; m < MT; ++m) red[buf][warp][r][m] = acc[r][m];
        }
        __syncthreads();
        // Thread t < rows*MT finishes output (row t / MT, column t % MT) of
        // this pair; the next pair writes the other buffer, and the barrier
        // after it orders this read before that buffer is written again.
        if (threadIdx.x < kGemvRows * MT) {
            const int r = threadIdx.x / MT, m = threadIdx.x % MT;
            if (n0 + r < r1 && m < M) {
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < kGemvWarps; ++w) sum += red[buf][w][r][m];
                const int n = n0 + r;
                C[static_cast<size_t>(m) * N + n] =
                    __float2half_rn(epi.on ? epi_apply1(epi, sum, eb, er) : sum);
            }
        }
    }
}

template <int MT>
int launch_mt(const GemvLaunch &L, std::string &err) {
    constexpr int R = 2, V = 4;  // rows per step, vectors per row per lane in flight
    const bool vec = (L.K % 8 == 0) &&
                     ((reinterpret_cast<uintptr_t>(L.A) | reinterpret_cast<uintptr_t>(L.B)) & 15u) == 0;
    const size_t smem = static_cast<size_t>(MT) * L.K * sizeof(__half);
    auto kernel = vec ? gemv_f16_nt_kernel<MT, R, V, true> : gemv_f16_nt_kernel<MT, R, V, false>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) {
            err = std::string("gemv: cudaFuncSetAttribute: ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
    }
    // Whole CTAs per SM, at most one CTA per row of B.
    const long long cap = static_cast<long long>(L.sm_count) * L.ctas_per_sm;
    const int grid = static_cast<int>(L.N < cap ? (L.N > 0 ? L.N : 1) : cap);
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
                                       static_cast<const __half *>(L.B), static_cast<__half *>(L.C),
                                       make_epi(L.epi, L.N));
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
    err = "gemv: M > 2";
    return GEMM_ERR_INVALID_ARG;
}

}  // namespace gb300
