// sgemm.cu -- C = alpha * A * B + beta * C in fp32 on the CUDA cores.
//
// Row-major A [M,K], B [K,N], C [M,N].  The operation and its alpha/beta
// epilogue are those of the gemm_cp_async kernel in "异步拷贝与 Hopper/Blackwell
// 新特性" (anrans.github.io/ai-infra-handbooks/cuda/advanced/async-hopper),
// section "cp.async 与多级流水 sm_80+"; beta == 0 follows the BLAS convention
// (C is not read).  fp32 semantics exclude TF32, so the work is plain FFMA.
//
// Design: each CTA owns a BM x BN tile of C; every thread owns a TM x TN
// register micro-tile ("第 6 章 · Shared Memory & Tile", section "6.3.1 寄存器
// tile"): rows ty + i * (BM/TM) + g * (BM/RM) and groups of 4 columns spread
// BN/RN apart, and a warp is 4 x 8 such threads.  K is walked in BK-deep slices through a
// STAGES-deep ring of shared memory filled by cp.async, STAGES-1 slices ahead
// of the multiply, one barrier per slice (the multi-stage scheme of
// "异步拷贝与 Hopper/Blackwell 新特性", section "cp.async 与多级流水 sm_80+",
// here with zero-filled tails).  On sm_103a the FP32 pipe retires 128 FMA per
// clock per SM, twice the rate the pages' Ampere kernels were tuned for, so
// issue slots and shared-memory wavefronts are the limits: the outer product
// uses the packed two-wide fp32 FMA (fma.rn.f32x2, each lane's two FMAs
// rounded exactly like fmaf), and the main tile's 8 x 16 micro-tile (128
// threads per 128 x 128 tile) does 5.3 FMAs per lane per 128-byte shared
// wavefront, where an 8 x 8 micro-tile's 4 would tie shared memory to the
// FMA pipe at peak.
// Out-of-range rows, columns and k are loaded as zeros and never stored, which
// makes any M, N, K exact.
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "gemm.h"
#include "gemm_internal.h"

namespace gb300 {
namespace {

// ---------------------------------------------------------------------------
// A and B slices go straight from global to shared memory
// with cp.async (16-byte copies, zero-filled past the matrix edges), STAGES-1
// slices ahead of the multiply, one barrier per slice.  A keeps its row-major
// layout in shared memory: a thread reads 4 consecutive k of one of its rows as
// a float4 (all 8 lanes of a quarter-warp read the same row: a broadcast), so
// no transpose is needed and the loads issue no register-staged stores.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 4 : 0)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int BM, int BN, int TM, int TN>
constexpr int sgemm_threads() { return (BM / TM) * (BN / TN); }

// Split-K ("第 6 章 · Shared Memory & Tile", section "6.5.6 Split-K /
// Stream-K"): with few tiles, blockIdx.z = s takes K elements
// [s * kchunk, (s + 1) * kchunk) of its tile and writes alpha times its partial
// to the tile's workspace slot s; the CTA that finishes a tile last (a
// counter per tile, reset by that CTA for the next launch) adds the slots in
// the order s = 0, 1, ... -- so the result does not depend on timing -- and
// applies beta * C.
struct SplitK {
    int splits;         // 1: no split
    int kchunk;         // K elements per split, a multiple of BK
    float *ws;          // [tiles][splits][BM * BN] partials
    unsigned *counters; // [tiles], zero between launches
};

template <int BM, int BN, int BK, int TM, int TN, int STAGES, int MINB, bool VEC, bool PADA, bool PIPE>
__global__ void __launch_bounds__(sgemm_threads<BM, BN, TM, TN>(), MINB)
    sgemm_pipe_kernel(int M, int N, int K, float alpha, const float *__restrict__ A,
                      const float *__restrict__ B, float beta, float *__restrict__ C, const SplitK sk) {
    constexpr int RM = TM / 4, RN = TN / 4;
    constexpr int kThreads = sgemm_threads<BM, BN, TM, TN>();
    constexpr int kWarpsN = (BN / TN) / 8;  // a warp is 4 thread rows x 8 thread columns
    constexpr int A_CHUNKS = BM * BK / 4, B_CHUNKS = BK * BN / 4;
    static_assert((BM / TM) % 4 == 0 && (BN / TN) % 8 == 0, "whole 4 x 8 warps");
    static_assert(BK % 4 == 0, "A is read as float4 along k");

    // PADA: A rows padded to BK + 4 floats (80 bytes for BK = 16) and a
    // thread's rows BM/TM apart, so that the four quarter-warps read four
    // consecutive rows in four different 16-byte bank groups (unpadded, with
    // a thread's 4 rows adjacent, the quarter-warps' rows are 4 apart and all
    // fall in one group).  Measured: 512^3 on 64 x 64 tiles 16.5 -> 14.4 us;
    // the 128 x 128 tile ran 2.5 % slower with it, so it keeps the plain layout.
    // Without PADA the rows stay BK floats and a row's float4 chunk q is
    // stored at chunk q ^ ((row / 4) % 4): the quarter-warps' rows are 4
    // apart, and the XOR puts their reads in four different bank groups.
    static_assert(PADA || BK == 16, "the chunk swizzle permutes 4 chunks per row");
    constexpr int BKP = PADA ? BK + 4 : BK;
    auto achunk = [](int row, int kq) { return PADA ? kq : (kq ^ ((row >> 2) & 3)); };
    __shared__ __align__(16) float As[STAGES][BM][BKP];
    __shared__ __align__(16) float Bs[STAGES][BK][BN];

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int ty = (warp / kWarpsN) * 4 + (lane >> 3);
    // tile row of this thread's row i of row group g
    auto trow = [&](int g, int i) { return g * (BM / RM) + (PADA ? i * (BM / TM) + ty : ty * 4 + i); };
    const int tx = (warp % kWarpsN) * 8 + (lane & 7);
    const int m0 = blockIdx.y * BM;
    const int n0 = blockIdx.x * BN;

    auto load_slice = [&](int buf, int k0) {
#pragma unroll
        for (int c = tid; c < A_CHUNKS; c += kThreads) {
            const int row = c / (BK / 4), kq = c % (BK / 4);
            const int m = m0 + row, k = k0 + kq * 4;
            const float *src = A + static_cast<size_t>(m < M ? m : 0) * K;
            const uint32_t dst =
                static_cast<uint32_t>(__cvta_generic_to_shared(&As[buf][row][achunk(row, kq) * 4]));
            if (VEC) {
                cp_async_16(dst, src + (k < K ? k : 0), m < M && k < K);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    cp_async_4(dst + 4 * e, src + (k + e < K ? k + e : 0), m < M && k + e < K);
            }
        }
#pragma unroll
        for (int c = tid; c < B_CHUNKS; c += kThreads) {
            const int kr = c / (BN / 4), nq = c % (BN / 4);
            const int k = k0 + kr, n = n0 + nq * 4;
            const float *src = B + static_cast<size_t>(k < K ? k : 0) * N;
            const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(&Bs[buf][kr][nq * 4]));
            if (VEC) {
                cp_async_16(dst, src + (n < N ? n : 0), k < K && n < N);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    cp_async_4(dst + 4 * e, src + (n + e < N ? n + e : 0), k < K && n + e < N);
            }
        }
    };

    // Accumulators in column pairs: accp[i][p] = (acc[i][2p], acc[i][2p+1]).
    // One packed fma.rn.f32x2 performs both fp32 FMAs (each rounded once, as
    // fmaf would), halving the FFMA issue slots of the outer product.
    float2 accp[TM][TN / 2];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) accp[i][j] = make_float2(0.f, 0.f);

    // this CTA's share of K (all of it without a split)
    const int kbeg = static_cast<int>(blockIdx.z) * sk.kchunk;
    const int kend = sk.splits > 1 ? min(K, kbeg + sk.kchunk) : K;
    const int KT = (kend - kbeg + BK - 1) / BK;
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < KT) load_slice(s, kbeg + s * BK);
        cp_async_commit();  // one group per slice, empty ones included
    }
    // One k step of the outer product: the broadcast pairs (a, a) of the
    // TM rows first, then the TM x TN/2 packed FMAs.
    auto fma_step = [&](const float4(&av)[TM], int kk, const float4(&bv)[RN]) {
        float2 bp[TN / 2];
#pragma unroll
        for (int g = 0; g < RN; ++g) {
            bp[g * 2 + 0] = make_float2(bv[g].x, bv[g].y);
            bp[g * 2 + 1] = make_float2(bv[g].z, bv[g].w);
        }
        float2 aa[TM];
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const float a = kk == 0 ? av[i].x : kk == 1 ? av[i].y : kk == 2 ? av[i].z : av[i].w;
            aa[i] = make_float2(a, a);
        }
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN / 2; ++j) accp[i][j] = __ffma2_rn(aa[i], bp[j], accp[i][j]);
    };
    auto read_a = [&](float4(&dst)[TM], int buf, int kq) {
#pragma unroll
        for (int g = 0; g < RM; ++g)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                dst[g * 4 + i] = *reinterpret_cast<const float4 *>(
                    &As[buf][trow(g, i)][achunk(trow(g, i), kq) * 4]);
    };
    auto read_b = [&](float4(&dst)[RN], int buf, int k) {
#pragma unroll
        for (int g = 0; g < RN; ++g)
            dst[g] = *reinterpret_cast<const float4 *>(&Bs[buf][k][g * (BN / RN) + tx * 4]);
    };
    if constexpr (PIPE) {
        // Register fragments read from shared memory one k step before their
        // FMAs, in double buffers.  A slice's barrier sits in its last k
        // step: after it the next slice's first fragments are read while that
        // step's FMAs run, so no step waits for a shared-memory read.  The
        // next slice's copy is then issued one slice later than in the loop
        // below, so this form wants a ring one stage deeper.
        static_assert(STAGES >= 3 && BK % 8 == 0, "fragment double buffers alternate within a slice");
        cp_async_wait<STAGES - 2>();  // slice 0 has landed (this thread's part)
        __syncthreads();              // ... everyone's part
        float4 afr[2][TM];
        float4 bfr[2][RN];
        read_a(afr[0], 0, 0);
        read_b(bfr[0], 0, 0);
        for (int kt = 0; kt < KT; ++kt) {
            const int buf = kt % STAGES;
#pragma unroll
            for (int k = 0; k < BK; ++k) {
                const int kq = k / 4, kk = k % 4, ca = kq & 1, cb = k & 1;
                if (k + 1 < BK) {
                    read_b(bfr[cb ^ 1], buf, k + 1);
                    if (kk == 3) read_a(afr[ca ^ 1], buf, kq + 1);
                } else {
                    cp_async_wait<STAGES - 3>();  // slice kt+1 has landed (this thread's part)
                    __syncthreads();              // ... everyone's; slice kt-1's buffer is free
                    const int next = kt + STAGES - 1;
                    if (next < KT) load_slice(next % STAGES, kbeg + next * BK);
                    cp_async_commit();
                    if (kt + 1 < KT) {
                        read_b(bfr[cb ^ 1], (kt + 1) % STAGES, 0);
                        read_a(afr[ca ^ 1], (kt + 1) % STAGES, 0);
                    }
                }
                fma_step(afr[ca], kk, bfr[cb]);
            }
        }
    } else {
        // One barrier at the top of each slice, then its fragments read as
        // they are used (the register file holds no second set next to the
        // 8 x 16 micro-tile's 128 accumulators).
        for (int kt = 0; kt < KT; ++kt) {
            cp_async_wait<STAGES - 2>();  // slice kt has landed (this thread's part)
            __syncthreads();              // ... everyone's part; slice kt-1 is no longer read
            const int next = kt + STAGES - 1;
            if (next < KT) load_slice(next % STAGES, kbeg + next * BK);
            cp_async_commit();
            const int buf = kt % STAGES;
#pragma unroll
            for (int kq = 0; kq < BK / 4; ++kq) {
                float4 av[TM];
                read_a(av, buf, kq);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    float4 bv[RN];
                    read_b(bv, buf, kq * 4 + kk);
                    fma_step(av, kk, bv);
                }
            }
        }
    }
    cp_async_wait<0>();
    const float(&acc)[TM][TN] = *reinterpret_cast<const float(*)[TM][TN]>(&accp[0][0]);

    if (sk.splits > 1) {
        // Partial of this split, alpha applied, into slot blockIdx.z: float4 q
        // of thread t at (q * threads + t) * 4, so a warp writes 512
        // contiguous bytes per store.
        constexpr int Q = TM * TN / 4;
        const int tile = blockIdx.y * gridDim.x + blockIdx.x;
        float4 *slots = reinterpret_cast<float4 *>(sk.ws) + static_cast<size_t>(tile) * sk.splits * (Q * kThreads);
        float4 *mine = slots + static_cast<size_t>(blockIdx.z) * (Q * kThreads);
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const float *a = &acc[q / (TN / 4)][(q % (TN / 4)) * 4];
            mine[q * kThreads + tid] = make_float4(alpha * a[0], alpha * a[1], alpha * a[2], alpha * a[3]);
        }
        __threadfence();
        __syncthreads();
        int arrived_last = 0;
        if (tid == 0) arrived_last = atomicAdd(&sk.counters[tile], 1u) == static_cast<unsigned>(sk.splits - 1);
        if (!__syncthreads_or(arrived_last)) return;
        __threadfence();  // every split's partial is visible to this CTA
        if (tid == 0) sk.counters[tile] = 0u;
        // Sum the slots in split order, QC float4 of each slot in flight at
        // once (one L2 round trip per slot and chunk, not per float4).
        constexpr int QC = Q < 16 ? Q : 16;
        const size_t sstride = static_cast<size_t>(Q) * kThreads;
#pragma unroll
        for (int qc = 0; qc < Q; qc += QC) {
            float4 o[QC];
#pragma unroll
            for (int u = 0; u < QC; ++u) o[u] = __ldcg(&slots[(qc + u) * kThreads + tid]);
            for (int sp = 1; sp < sk.splits; ++sp) {
                const float4 *src = slots + sp * sstride;
                float4 v[QC];
#pragma unroll
                for (int u = 0; u < QC; ++u) v[u] = __ldcg(&src[(qc + u) * kThreads + tid]);
#pragma unroll
                for (int u = 0; u < QC; ++u) {
                    o[u].x += v[u].x;
                    o[u].y += v[u].y;
                    o[u].z += v[u].z;
                    o[u].w += v[u].w;
                }
            }
#pragma unroll
            for (int u = 0; u < QC; ++u) {
                const int q = qc + u, r = q / (TN / 4), gj = q % (TN / 4);
                const int m = m0 + trow(r / 4, r % 4);
                if (m >= M) continue;
                float *crow = C + static_cast<size_t>(m) * N;
                const int n = n0 + gj * (BN / RN) + tx * 4;
                float4 w = o[u];
                if (VEC) {
                    if (n < N) {
                        if (beta != 0.f) {
                            const float4 c = *reinterpret_cast<const float4 *>(crow + n);
                            w.x = fmaf(beta, c.x, w.x);
                            w.y = fmaf(beta, c.y, w.y);
                            w.z = fmaf(beta, c.z, w.z);
                            w.w = fmaf(beta, c.w, w.w);
                        }
                        *reinterpret_cast<float4 *>(crow + n) = w;
                    }
                } else {
                    const float ov[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (n + j < N) crow[n + j] = beta != 0.f ? fmaf(beta, crow[n + j], ov[j]) : ov[j];
                }
            }
        }
        return;
    }

#pragma unroll
    for (int gi = 0; gi < RM; ++gi) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = m0 + trow(gi, i);
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

// Split-K workspace of one (device, stream): partial slots and per-tile
// counters (zeroed once; every launch leaves them zero), grown on demand.
// Calls on one stream run in order, so a stream has one user at a time.
struct SgWorkspace {
    float *ws = nullptr;
    unsigned *counters = nullptr;
    size_t ws_bytes = 0;
    int tiles = 0;
};

int sg_workspace(cudaStream_t stream, size_t ws_bytes, int tiles, bool capturing, SgWorkspace **out,
                 std::string &err) {
    static std::mutex mu;
    static std::map<std::pair<int, cudaStream_t>, SgWorkspace> cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        err = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(mu);
    SgWorkspace &w = cache[{dev, stream}];
    if (w.ws_bytes >= ws_bytes && w.tiles >= tiles) {
        *out = &w;
        return GEMM_OK;
    }
    *out = nullptr;
    if (capturing) return GEMM_OK;  // no allocation inside a graph capture: do not split
    // The stream may still be running a launch that uses the old buffers.
    e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && w.ws) e = cudaFree(w.ws);
    if (e == cudaSuccess && w.counters) e = cudaFree(w.counters);
    w = SgWorkspace{};
    const size_t bytes = ws_bytes > 0 ? ws_bytes : 16;
    if (e == cudaSuccess) e = cudaMalloc(&w.ws, bytes);
    if (e == cudaSuccess) e = cudaMalloc(&w.counters, static_cast<size_t>(tiles) * sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemset(w.counters, 0, static_cast<size_t>(tiles) * sizeof(unsigned));
    if (e != cudaSuccess) {
        err = std::string("sgemm split-K workspace: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    w.ws_bytes = bytes;
    w.tiles = tiles;
    *out = &w;
    return GEMM_OK;
}

template <int BM, int BN, int BK, int TM, int TN, int STAGES, int MINB, bool PADA, bool PIPE>
int launch_pipe(const SgemmLaunch &L, std::string &err) {
    dim3 grid((L.N + BN - 1) / BN, (L.M + BM - 1) / BM);
    // Split-K as planned by the caller: blockIdx.z picks a K share.
    static_assert(BK == 16, "sgemm_split_chunk rounds shares to 16-deep slices");
    SplitK sk{1, L.K, nullptr, nullptr};
    const int tiles = static_cast<int>(grid.x * grid.y);
    int kchunk = L.K;
    const int splits = sgemm_split_chunk(L.K, L.splits, &kchunk);
    if (splits > 1) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        cudaError_t e = cudaStreamIsCapturing(L.stream, &cap);
        if (e != cudaSuccess) {
            err = std::string("cudaStreamIsCapturing: ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
        SgWorkspace *w = nullptr;
        const size_t need = static_cast<size_t>(tiles) * splits * BM * BN * sizeof(float);
        const int st = sg_workspace(L.stream, need, tiles, cap != cudaStreamCaptureStatusNone, &w, err);
        if (st != GEMM_OK) return st;
        if (w) {  // null under capture when the workspace would have to grow: no split
            sk = SplitK{splits, kchunk, w->ws, w->counters};
            grid.z = splits;
        }
    }
    const bool vec = (L.K % 4 == 0) && (L.N % 4 == 0) &&
                     ((reinterpret_cast<uintptr_t>(L.A) | reinterpret_cast<uintptr_t>(L.B) |
                       reinterpret_cast<uintptr_t>(L.C)) & 15u) == 0;
    constexpr int threads = sgemm_threads<BM, BN, TM, TN>();
    auto kvec = sgemm_pipe_kernel<BM, BN, BK, TM, TN, STAGES, MINB, true, PADA, PIPE>;
    auto kscalar = sgemm_pipe_kernel<BM, BN, BK, TM, TN, STAGES, MINB, false, PADA, PIPE>;
    if (vec)
        kvec<<<grid, threads, 0, L.stream>>>(L.M, L.N, L.K, L.alpha, L.A, L.B, L.beta, L.C, sk);
    else
        kscalar<<<grid, threads, 0, L.stream>>>(L.M, L.N, L.K, L.alpha, L.A, L.B, L.beta, L.C, sk);
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
        case GEMM_SGEMM_128x128: return launch_pipe<128, 128, 16, 8, 16, 3, 2, false, false>(L, err);
        case GEMM_SGEMM_64x64: return launch_pipe<64, 64, 16, 4, 4, 3, 2, true, false>(L, err);
        case GEMM_SGEMM_128x64: return launch_pipe<128, 64, 16, 8, 8, 4, 2, false, true>(L, err);
        default: err = "unknown sgemm variant"; return GEMM_ERR_INVALID_ARG;
    }
}

}  // namespace gb300
