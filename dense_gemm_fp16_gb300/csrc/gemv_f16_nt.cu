// gemv_f16_nt.cu -- C = A * B^T for one to four rows of A (M <= 4): the
// matrix-vector regime of an LLM decode step.
//
// Same operation and numerics as gemm_f16_nt (half inputs, fp32 accumulation,
// one round-to-nearest-even per output), but with M this small every element
// of B is used only M times, so the product is bound by reading B from HBM,
// not by the tensor cores ("第 6 章 · Shared Memory & Tile", section "6.5.5
// GEMV (M=1)：LLM decode 完全不能用 tile": tiling has nothing to reuse; one
// warp per output row, a shuffle reduction).  From five rows on, the A
// vectors each B vector needs (M x 16 bytes from L1 per 16 bytes of B) bound
// the CUDA cores below HBM speed and the tensor-core path is faster
// (measured at N = K = 8192 and N = 16384, K = 8192).
//
// Design for sm_103a's HBM: B is streamed once with 16-byte loads that skip
// L1 allocation; every warp owns a balanced block of rows of B (the grid is a
// whole number of CTAs per SM, as many as the registers allow) and its lanes
// split each row's K range, two rows at a time with four 16-byte vectors of
// each in flight per lane.  A (at most 4 x K halves) is read through L1,
// where every warp of the SM finds it.  The products accumulate as packed
// fp32 pairs (fma.rn.f32x2), and each output's partial sums meet in one
// butterfly of shuffles: no shared memory, no barrier.  Reading B once, the
// algorithmic bytes are N*K*2 + M*K*2 + M*N*2.
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

// acc[r][m] += the 8 halves of row r's vector b[r] . those of A row m, as
// packed fp32 pairs: .x sums the even k, .y the odd k (fma.rn.f32x2, each
// lane rounded like fmaf).  Each half2 of A is converted once for all the
// rows of the group.
template <int MT, int R>
__device__ __forceinline__ void dot8x2(float2 (&acc)[R][MT], const uint4 (&b)[R], const uint4 (&av)[MT]) {
    float2 bf[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const __half2 *b2 = reinterpret_cast<const __half2 *>(&b[r]);
#pragma unroll
        for (int q = 0; q < 4; ++q) bf[r][q] = __half22float2(b2[q]);
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const __half2 *a2 = reinterpret_cast<const __half2 *>(&av[m]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 af = __half22float2(a2[q]);
#pragma unroll
            for (int r = 0; r < R; ++r) acc[r][m] = __ffma2_rn(af, bf[r][q], acc[r][m]);
        }
    }
}

// R rows of B at a time, kVec 16-byte vectors of each in flight per lane;
// A rows past M alias row 0 (their sums are never stored).  K % 8 == 0 and
// 16-byte aligned A and B (the entry point checks both).
template <int MT, int R, int kVec>
__global__ void __launch_bounds__(kGemvWarps * 32)
    gemv_rows_kernel(int M, int N, int K, const __half *__restrict__ A, const __half *__restrict__ B,
                     __half *__restrict__ C, const Epi epi) {
    // Programmatic dependent launch: nothing global before the predecessor is done.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int lane = threadIdx.x & 31;
    const int W = static_cast<int>(gridDim.x) * kGemvWarps;
    const int w = static_cast<int>(blockIdx.x) * kGemvWarps + (threadIdx.x >> 5);
    const int r0 = static_cast<int>(static_cast<long long>(w) * N / W);
    const int r1 = static_cast<int>(static_cast<long long>(w + 1) * N / W);
    const int nv = K / 8;  // 16-byte vectors per row
    static_assert(R * MT <= 32, "one lane per output of a row group");
    const __half *arow[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) arow[m] = A + static_cast<size_t>(m < M ? m : 0) * K;
    for (int n0 = r0; n0 < r1; n0 += R) {
        const __half *brow[R];
#pragma unroll
        for (int r = 0; r < R; ++r)  // rows past the block repeat its last row (computed, not stored)
            brow[r] = B + static_cast<size_t>(n0 + r < r1 ? n0 + r : r1 - 1) * K;
        float2 acc[R][MT];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[r][m] = make_float2(0.f, 0.f);
        for (int v = lane; v < nv; v += 32 * kVec) {
            uint4 bv[R][kVec];
#pragma unroll
            for (int h = 0; h < kVec; ++h)
                if (v + 32 * h < nv) {
#pragma unroll
                    for (int r = 0; r < R; ++r) bv[r][h] = ld_stream_v4(brow[r] + (v + 32 * h) * 8);
                }
#pragma unroll
            for (int h = 0; h < kVec; ++h) {
                if (v + 32 * h >= nv) break;
                uint4 av[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    av[m] = __ldg(reinterpret_cast<const uint4 *>(arow[m] + (v + 32 * h) * 8));
                uint4 bh[R];
#pragma unroll
                for (int r = 0; r < R; ++r) bh[r] = bv[r][h];
                dot8x2<MT, R>(acc, bh, av);
            }
        }
        // every lane ends with every sum; lane r * MT + m stores output (m, n0 + r)
        float mine = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                float x = acc[r][m].x + acc[r][m].y;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
                if (lane == r * MT + m) mine = x;
            }
        if (lane < R * MT) {
            const int r = lane / MT, m = lane % MT;
            const int n = n0 + r;
            if (m < M && n < r1) {
                float o = mine;
                if (epi.on) {
                    const float eb = epi.bias ? __half2float(epi.bias[n]) : 0.f;
                    const float er = epi.reads_res() ? __half2float(epi.res[static_cast<size_t>(m) * N + n]) : 0.f;
                    o = epi_apply1(epi, o, eb, er);
                }
                C[static_cast<size_t>(m) * N + n] = __float2half_rn(o);
            }
        }
    }
}

template <int MT>
int launch_mt(const GemvLaunch &L, std::string &err) {
    auto kernel = gemv_rows_kernel<MT, 2, 4>;
    // Whole CTAs per SM (as many as the registers allow, at most ctas_per_sm),
    // at most one warp per row of B.
    int fit = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, kernel, kGemvWarps * 32, 0);
    if (e != cudaSuccess || fit < 1) {
        err = std::string("gemv: occupancy query: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    const long long per_sm = fit < L.ctas_per_sm ? fit : L.ctas_per_sm;
    const long long cap = static_cast<long long>(L.sm_count) * per_sm;
    const long long need = (static_cast<long long>(L.N) + kGemvWarps - 1) / kGemvWarps;
    const int grid = static_cast<int>(need < cap ? (need > 0 ? need : 1) : cap);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGemvWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = L.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, L.M, L.N, L.K, static_cast<const __half *>(L.A),
                           static_cast<const __half *>(L.B), static_cast<__half *>(L.C), make_epi(L.epi, L.N));
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
    err = "gemv: M > 4";
    return GEMM_ERR_INVALID_ARG;
}

}  // namespace gb300
