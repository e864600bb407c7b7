// gemm_f16_nt.cu -- C = A * B^T on the sm_103a tensor cores.
//
// A half [M,K], B half [N,K] (both row-major, i.e. both K-major), fp32
// accumulation, C half [M,N] row-major, each output rounded once to nearest
// even.  The operation is the one defined in "从零开始的 AI Infra: 算子基础与GPU架构"
// (qi-zhan.github.io/blog/2026/cuda-gemm), section "0. Naive Implementation";
// section "19. 去掉转置" is why no transpose is needed: B [N,K] row-major is
// exactly the K-major operand the tensor core reads.
//
// Design (GB300-first; the pages' Ampere kernels are prior art only):
//  * persistent grid, one CTA per SM, static round-robin over output tiles
//    ("第 6 章 · Shared Memory & Tile", section "6.5.7 持久化 kernel");
//  * warp specialisation with an mbarrier ring of STAGES shared-memory stages
//    (section "6.10.1 Warp Specialization" of the same page; "异步拷贝与
//    Hopper/Blackwell 新特性", section "wgmma 与 warp 专门化 sm_90a"):
//      warp 0     one thread issues TMA loads of the A and B tiles (128-byte
//                 swizzle, out-of-bounds rows/columns filled with zeros, which
//                 is what makes partial M, N and K tiles exact),
//      warp 1     allocates TMEM; one thread issues tcgen05.mma (M=128,
//                 N=BN, K=16) into a TMEM accumulator and tcgen05.commit's
//                 the stage back to the producer,
//      warps 2-5  epilogue: tcgen05.ld TMEM -> registers, round to half,
//                 masked stores;
//  * the accumulator is double-buffered in TMEM (2 x BN columns), so the
//    epilogue of tile i overlaps the main loop of tile i+1;
//  * programmatic dependent launch: the prologue (barrier init, TMEM alloc,
//    descriptor prefetch) of one call overlaps the tail of the previous
//    kernel in the stream; global memory is touched only after
//    griddepcontrol.wait;
//  * every wait is bounded in time: on expiry the kernel records a status
//    code, tells the other roles to stop, waits (bounded) for its own copies
//    and MMAs in flight, frees TMEM and returns.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "gemm.h"
#include "gemm_internal.h"
#include "sm103_ptx.cuh"

namespace gb300 {
namespace {

constexpr int kBM = 128;       // rows of an output tile (= MMA M, = TMEM lanes)
constexpr int kBK = 64;        // halves per k-block: one 128-byte swizzle row
constexpr int kUmmaK = 16;     // K of one kind::f16 MMA
constexpr int kThreads = 192;  // 6 warps
// Epilogue staging: each of the 4 epilogue warps owns two 4 KB buffers, each
// holding 32 rows x 64 halves (128 B per row, 128-byte swizzled) for a TMA store.
constexpr int kEpiBufBytes = 32 * 128;
constexpr int kEpiBytes = 4 * 2 * kEpiBufBytes;

// Device-side status: first timeout code recorded by any CTA (0 = none).
// 1 = producer (empty-slot wait), 2 = MMA (full-slot or accumulator-free
// wait), 3 = epilogue (accumulator-ready wait).
__device__ int g_f16_status = 0;

struct F16Args {
    __half *C;
    int M, N, K;
    int m_tiles, n_tiles, num_kb;
    int vec_store;          // N % 8 == 0 and C 16-byte aligned
    int tma_store;          // same condition: the epilogue stores through a C tensor map
    uint64_t timeout_ns;
    int debug_skip_kblock;  // -1 = none
};

template <int BN, int STAGES>
struct TileCfg {
    static constexpr int kABytes = kBM * kBK * 2;
    static constexpr int kBBytes = BN * kBK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kTmemCols = 2 * BN;  // two accumulator buffers
    static constexpr int kNumBars = 2 * STAGES + 5;
    static constexpr int kEpiOffset = STAGES * kStageBytes;
    static constexpr int kBarOffset = kEpiOffset + kEpiBytes;
    static constexpr int kSmemBytes = 1024 + kBarOffset + kNumBars * 8 + 16;
    static_assert(kSmemBytes <= 232448, "fits the 227 KB opt-in limit");
    static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "swizzle atoms stay aligned");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "valid UMMA N for M = 128");
    static_assert(kTmemCols == 256 || kTmemCols == 512, "TMEM allocation is a power of two");
};

__device__ __forceinline__ void record_timeout(int code) { atomicCAS(&g_f16_status, 0, code); }

// Round 32 consecutive fp32 accumulators of one output row to half and store
// the columns n0 .. n0+31 that lie below N (16-byte vectors when allowed).
__device__ __forceinline__ void store_row_chunk(__half *crow, bool row_ok, int n0, int N, int vec,
                                                const uint32_t (&r)[32]) {
    if (!row_ok) return;
    if (vec) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (n0 + q * 8 < N) {
                uint4 v;
                __half2 h0 = __floats2half2_rn(__uint_as_float(r[q * 8 + 0]), __uint_as_float(r[q * 8 + 1]));
                __half2 h1 = __floats2half2_rn(__uint_as_float(r[q * 8 + 2]), __uint_as_float(r[q * 8 + 3]));
                __half2 h2 = __floats2half2_rn(__uint_as_float(r[q * 8 + 4]), __uint_as_float(r[q * 8 + 5]));
                __half2 h3 = __floats2half2_rn(__uint_as_float(r[q * 8 + 6]), __uint_as_float(r[q * 8 + 7]));
                v.x = *reinterpret_cast<uint32_t *>(&h0);
                v.y = *reinterpret_cast<uint32_t *>(&h1);
                v.z = *reinterpret_cast<uint32_t *>(&h2);
                v.w = *reinterpret_cast<uint32_t *>(&h3);
                *reinterpret_cast<uint4 *>(crow + n0 + q * 8) = v;
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (n0 + j < N) crow[n0 + j] = __float2half_rn(__uint_as_float(r[j]));
    }
}

// Epilogue of one accumulator tile for one epilogue warp: output rows
// row0 .. row0+31 (lane i holds row row0+i, the TMEM lane it may read),
// columns n_base .. n_base+BN-1, read from TMEM address `taddr` onwards.
// With a C tensor map, each 64-column slab is rounded to half, written into
// one of the warp's two swizzled staging buffers and stored by one TMA
// instruction (out-of-range rows and columns are clipped by the TMA unit);
// otherwise each thread stores its own row directly.
template <int BN>
__device__ __forceinline__ void epilogue_warp_tile(const F16Args &args, const CUtensorMap *tmC,
                                                   uint32_t taddr, int row0, int n_base, int lane,
                                                   uint32_t stage_smem, uint32_t &step) {
    if (args.tma_store) {
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
            uint32_t lo[32], hi[32];
            tmem_load_32cols(taddr + static_cast<uint32_t>(c * 64), lo);
            tmem_load_32cols(taddr + static_cast<uint32_t>(c * 64 + 32), hi);
            const uint32_t buf = stage_smem + (step & 1u) * kEpiBufBytes;
            // The store issued from this buffer two slabs ago must have read it.
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
            const uint32_t row_addr = buf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t *v = j < 4 ? &lo[j * 8] : &hi[(j - 4) * 8];
                __half2 h0 = __floats2half2_rn(__uint_as_float(v[0]), __uint_as_float(v[1]));
                __half2 h1 = __floats2half2_rn(__uint_as_float(v[2]), __uint_as_float(v[3]));
                __half2 h2 = __floats2half2_rn(__uint_as_float(v[4]), __uint_as_float(v[5]));
                __half2 h3 = __floats2half2_rn(__uint_as_float(v[6]), __uint_as_float(v[7]));
                // 16-byte chunk j of row `lane` sits at chunk j ^ (lane % 8): the
                // TMA's 128-byte swizzle, which also spreads a quarter-warp's
                // writes over all 32 banks.
                st_shared_v4(row_addr + (static_cast<uint32_t>(j ^ (lane & 7)) << 4),
                             *reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1),
                             *reinterpret_cast<uint32_t *>(&h2), *reinterpret_cast<uint32_t *>(&h3));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                // A box wholly past the last row or column would store nothing.
                if (row0 < args.M && n_base + c * 64 < args.N)
                    tma_store_2d(tmC, buf, n_base + c * 64, row0);
                bulk_commit_group();
            }
            ++step;
        }
    } else {
        const int m = row0 + lane;
        __half *crow = args.C + static_cast<size_t>(m) * args.N;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_load_32cols(taddr + static_cast<uint32_t>(c * 32), r);
            store_row_chunk(crow, m < args.M, n_base + c * 32, args.N, args.vec_store, r);
        }
    }
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_f16_nt_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmC, const F16Args args) {
    using T = TileCfg<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzle atoms must sit on 1024-byte boundaries of the shared window.
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + T::kBarOffset);
    const uint32_t bar0 = smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + T::kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    __shared__ int never_abort;  // stays 0: used by drain waits that must not bail early

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (args.tma_store) tma_prefetch_desc(&tmC);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);   // producer's arrive.expect_tx + TMA bytes
            mbar_init(empty_bar(s), 1);  // one tcgen05.commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);   // one tcgen05.commit per tile
            mbar_init(acce_bar(b), 4);   // one arrive per epilogue warp
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        never_abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), T::kTmemCols);
        tmem_relinquish_alloc_permit();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // Everything above overlaps the previous kernel's tail under programmatic
    // dependent launch; A and B are read and C written only after this wait.
    pdl_launch_dependents();
    pdl_wait_prerequisites();

    const int total_tiles = args.m_tiles * args.n_tiles;
    const int num_kb = args.num_kb;

    // Producer bookkeeping kept for the teardown drain: which stages were ever
    // armed, and the parity of each stage's arm count.
    uint32_t armed = 0, arm_parity = 0;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            bool first_tile = true;
            for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
                const int mt = tile % args.m_tiles;
                const int nt = tile / args.m_tiles;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, args.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const bool skip = first_tile && kb == args.debug_skip_kblock;
                    if (!skip) {
                        const uint32_t sa = sbase + stage * T::kStageBytes;
                        const uint32_t sb = sa + T::kABytes;
                        mbar_arrive_expect_tx(full_bar(stage), T::kStageBytes);
                        tma_load_2d(sa, &tmA, full_bar(stage), kb * kBK, mt * kBM);
                        tma_load_2d(sb, &tmB, full_bar(stage), kb * kBK, nt * BN);
                        armed |= 1u << stage;
                        arm_parity ^= 1u << stage;
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                first_tile = false;
            }
            if (!ok) {
                if (!*abort_flag) record_timeout(1);
                *abort_flag = 1;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32acc(kBM, BN);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int i = 0;
            for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++i) {
                const int b = i & 1;
                const uint32_t ap = (i >> 1) & 1;
                if (!mbar_wait(acce_bar(b), ap ^ 1u, args.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(full_bar(stage), phase, args.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sa = sbase + stage * T::kStageBytes;
                    const uint64_t adesc = sw128_kmajor_desc(sa);
                    const uint64_t bdesc = sw128_kmajor_desc(sa + T::kABytes);
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        // advance the start address by k * 16 halves = 32 bytes
                        mma_f16_ss(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc,
                                   (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit(empty_bar(stage));  // frees the stage once the MMAs read it
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(accf_bar(b));  // accumulator complete
            }
            if (!ok) {
                if (!*abort_flag) record_timeout(2);
                *abort_flag = 1;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;  // TMEM lanes this warp may read: 32*quarter ..
        const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t stage_smem = sbase + T::kEpiOffset + (warp - 2) * 2 * kEpiBufBytes;
        uint32_t step = 0;
        int i = 0;
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++i) {
            const int b = i & 1;
            const uint32_t ap = (i >> 1) & 1;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(accf_bar(b), ap, args.timeout_ns, abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    if (!*abort_flag) record_timeout(3);
                    *abort_flag = 1;
                }
                break;
            }
            tc_fence_after_sync();
            const int mt = tile % args.m_tiles;
            const int nt = tile / args.m_tiles;
            epilogue_warp_tile<BN>(args, &tmC, tmem_base + lane_field + static_cast<uint32_t>(b * BN),
                                   mt * kBM + quarter * 32, nt * BN, lane, stage_smem, step);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(b));
        }
        if (lane == 0) bulk_wait_group_all();  // C fully written before the CTA retires
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    // Every role has left its loop, so abort_flag is final and uniform here.
    // After an abort, let this CTA's own asynchronous work finish before its
    // shared memory and TMEM are released: the last copy armed on each stage
    // (earlier ones were consumed before the stage could be re-armed) and all
    // MMAs issued (one commit tracks every earlier tcgen05 operation).
    if (*abort_flag) {
        if (warp == 0 && lane == 0) {
            for (int s = 0; s < STAGES; ++s)
                if (armed & (1u << s))
                    (void)mbar_wait(full_bar(s), ((arm_parity >> s) & 1u) ^ 1u, args.timeout_ns,
                                    &never_abort);
        }
        if (warp == 1 && lane == 0) {
            mma_commit(drain_bar);
            (void)mbar_wait(drain_bar, 0, args.timeout_ns, &never_abort);
        }
        __syncwarp();
        tc_fence_before_sync();
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, T::kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// CTA-pair variant: a cluster of two CTAs computes a 256 x 256 output tile
// with tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16).  CTA r of the pair
// loads rows 128r .. 128r+127 of the tile's A block and rows 128r .. 128r+127
// of its B block (the B half it contributes), so each SM brings in 32 KB per
// 64-deep k-block instead of 48 KB, and each CTA's TMEM receives its own 128
// output rows x 256 columns.  The even CTA's single MMA thread drives both
// SMs' tensor cores:
//   full[s]   (even CTA)  one arrive.expect_tx for both CTAs' bytes; the odd
//                         CTA's TMA loads complete on it across the pair,
//   empty[s]  (both CTAs) freed by a commit multicast to the pair,
//   accf[b]   (both CTAs) accumulator ready, commit multicast to the pair,
//   acce[b]   (even CTA)  accumulator drained: 4 epilogue warps x 2 CTAs.
// ---------------------------------------------------------------------------

template <int STAGES>
struct PairCfg {
    static constexpr int kBN = 256;                 // pair tile N (= MMA N)
    static constexpr int kABytes = kBM * kBK * 2;   // this CTA's 128 rows of A
    static constexpr int kBBytes = 128 * kBK * 2;   // this CTA's half of B
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kTmemCols = 512;           // two 256-column accumulators
    static constexpr int kNumBars = 2 * STAGES + 5;
    static constexpr int kEpiOffset = STAGES * kStageBytes;
    static constexpr int kBarOffset = kEpiOffset + kEpiBytes;
    static constexpr int kSmemBytes = 1024 + kBarOffset + kNumBars * 8 + 16;
    static_assert(kSmemBytes <= 232448, "fits the 227 KB opt-in limit");
};

template <int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_f16_nt_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmC, const F16Args args) {
    using T = PairCfg<STAGES>;
    constexpr int BN = T::kBN;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + T::kBarOffset);
    const uint32_t bar0 = smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + T::kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    __shared__ int never_abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0 (leader) or 1
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (args.tma_store) tma_prefetch_desc(&tmC);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 8);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        never_abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(tmem_slot), T::kTmemCols);
        tmem_relinquish_alloc_permit_pair();
    }
    tc_fence_before_sync();
    cluster_sync();  // barriers of both CTAs initialised, TMEM allocated in both
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    pdl_launch_dependents();
    pdl_wait_prerequisites();

    const int total_tiles = args.m_tiles * args.n_tiles;  // pair tiles
    const int num_kb = args.num_kb;
    uint32_t armed = 0, arm_parity = 0;

    if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            bool first_tile = true;
            for (int tile = pair; tile < total_tiles && ok; tile += num_pairs) {
                const int mt = tile % args.m_tiles;
                const int nt = tile / args.m_tiles;
                const int a_row = mt * 256 + static_cast<int>(rank) * 128;
                const int b_row = nt * BN + static_cast<int>(rank) * 128;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait_cluster(empty_bar(stage), phase ^ 1u, args.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const bool skip = first_tile && kb == args.debug_skip_kblock && leader;
                    if (!skip) {
                        const uint32_t sa = sbase + stage * T::kStageBytes;
                        const uint32_t full_leader = mapa_shared(full_bar(stage), 0);
                        if (leader) {
                            mbar_arrive_expect_tx(full_bar(stage), 2 * T::kStageBytes);
                            armed |= 1u << stage;
                            arm_parity ^= 1u << stage;
                        }
                        tma_load_2d_pair(sa, &tmA, full_leader, kb * kBK, a_row);
                        tma_load_2d_pair(sa + T::kABytes, &tmB, full_leader, kb * kBK, b_row);
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                first_tile = false;
            }
            if (!ok) {
                if (!*abort_flag) record_timeout(1);
                *abort_flag = 1;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader only)
        if (lane == 0 && leader) {
            constexpr uint32_t idesc = idesc_f16_f32acc(256, BN);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int i = 0;
            for (int tile = pair; tile < total_tiles; tile += num_pairs, ++i) {
                const int b = i & 1;
                const uint32_t ap = (i >> 1) & 1;
                if (!mbar_wait_cluster(acce_bar(b), ap ^ 1u, args.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait_cluster(full_bar(stage), phase, args.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sa = sbase + stage * T::kStageBytes;
                    const uint64_t adesc = sw128_kmajor_desc(sa);
                    const uint64_t bdesc = sw128_kmajor_desc(sa + T::kABytes);
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k)
                        mma_f16_ss_pair(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc,
                                        (kb > 0 || k > 0) ? 1u : 0u);
                    mma_commit_pair_multicast(empty_bar(stage), 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_pair_multicast(accf_bar(b), 0x3);
            }
            if (!ok) {
                if (!*abort_flag) record_timeout(2);
                *abort_flag = 1;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int quarter = warp & 3;
        const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t stage_smem = sbase + T::kEpiOffset + (warp - 2) * 2 * kEpiBufBytes;
        uint32_t step = 0;
        int i = 0;
        for (int tile = pair; tile < total_tiles; tile += num_pairs, ++i) {
            const int b = i & 1;
            const uint32_t ap = (i >> 1) & 1;
            int ok = 1;
            if (lane == 0)
                ok = mbar_wait_cluster(accf_bar(b), ap, args.timeout_ns, abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    if (!*abort_flag) record_timeout(3);
                    *abort_flag = 1;
                }
                break;
            }
            tc_fence_after_sync();
            const int mt = tile % args.m_tiles;
            const int nt = tile / args.m_tiles;
            epilogue_warp_tile<BN>(args, &tmC, tmem_base + lane_field + static_cast<uint32_t>(b * BN),
                                   mt * 256 + static_cast<int>(rank) * 128 + quarter * 32, nt * BN,
                                   lane, stage_smem, step);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(b), 0));
        }
        if (lane == 0) bulk_wait_group_all();
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (*abort_flag) {
        // The even CTA waits for the last phase armed on each stage (it counts
        // both CTAs' bytes) and for every MMA it issued; the odd CTA's copies
        // complete on those same barriers.
        if (leader && warp == 0 && lane == 0) {
            for (int s = 0; s < STAGES; ++s)
                if (armed & (1u << s))
                    (void)mbar_wait_cluster(full_bar(s), ((arm_parity >> s) & 1u) ^ 1u,
                                            args.timeout_ns, &never_abort);
        }
        if (leader && warp == 1 && lane == 0) {
            mma_commit_pair(drain_bar);
            (void)mbar_wait_cluster(drain_bar, 0, args.timeout_ns, &never_abort);
        }
        __syncwarp();
        tc_fence_before_sync();
        __syncthreads();
    }
    // Neither CTA may leave while the other can still touch its shared memory
    // (remote arrivals, pair TMA completions, pair MMA operand reads).
    cluster_sync();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, T::kTmemCols);
    }
}

// C = 0 for K == 0 (the empty sum).
__global__ void zero_half_kernel(__half *C, size_t count) {
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < count; i += stride)
        C[i] = __float2half_rn(0.0f);
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch
// ---------------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn(std::string &err) {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    static cudaError_t status = cudaSuccess;
    static cudaDriverEntryPointQueryResult qres = cudaDriverEntryPointSuccess;
    std::call_once(once, [] {
        void *p = nullptr;
        status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                  cudaEnableDefault, &qres);
        if (status == cudaSuccess && qres == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!fn) {
        err = std::string("cuTensorMapEncodeTiled unavailable: ") + cudaGetErrorString(status);
    }
    return fn;
}

// Row-major 2-D tensor of halves [rows, cols]: box = box_rows x box_cols,
// 128-byte swizzle (box_cols * 2 == 128), zero fill out of bounds on loads,
// clipping on stores.
bool encode_half_map(CUtensorMap *map, const void *ptr, int rows, int cols, int box_rows,
                     int box_cols, std::string &err) {
    EncodeTiledFn enc = get_encode_fn(err);
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    // No L2 promotion: the operands are L2-resident after their first use and
    // wider L2 fetches measured slower on this path.
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(ptr), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char buf[160];
        std::snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (CUresult %d) rows=%d cols=%d",
                      static_cast<int>(r), rows, cols);
        err = buf;
        return false;
    }
    return true;
}

template <int BN, int STAGES>
int launch_variant(const F16Launch &L, std::string &err) {
    using T = TileCfg<BN, STAGES>;
    auto kernel = gemm_f16_nt_tc_kernel<BN, STAGES>;
    // The opt-in for more than 48 KB of dynamic shared memory is per device.
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        err = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 T::kSmemBytes);
        if (e != cudaSuccess) {
            err = std::string("cudaFuncSetAttribute(max dynamic smem): ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
        if (dev >= 0 && dev < 64) configured[dev] = 1;
    }
    CUtensorMap tmA, tmB;
    if (!encode_half_map(&tmA, L.A, L.M, L.K, kBM, kBK, err)) return GEMM_ERR_CUDA;
    if (!encode_half_map(&tmB, L.B, L.N, L.K, BN, kBK, err)) return GEMM_ERR_CUDA;

    F16Args args;
    args.C = static_cast<__half *>(L.C);
    args.M = L.M;
    args.N = L.N;
    args.K = L.K;
    args.m_tiles = (L.M + kBM - 1) / kBM;
    args.n_tiles = (L.N + BN - 1) / BN;
    args.num_kb = (L.K + kBK - 1) / kBK;
    args.vec_store = (L.N % 8 == 0) && ((reinterpret_cast<uintptr_t>(L.C) & 15u) == 0);
    args.tma_store = args.vec_store;
    args.timeout_ns = L.timeout_ns;
    args.debug_skip_kblock = L.debug_skip_kblock;
    CUtensorMap tmC;
    std::memset(&tmC, 0, sizeof tmC);
    if (args.tma_store && !encode_half_map(&tmC, L.C, L.M, L.N, 32, 64, err)) return GEMM_ERR_CUDA;
    const int tiles = args.m_tiles * args.n_tiles;
    const int grid = L.grid < tiles ? L.grid : tiles;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = T::kSmemBytes;
    cfg.stream = L.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, tmC, args);
    if (e != cudaSuccess) {
        err = std::string("gemm_f16_nt kernel launch: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

template <int STAGES>
int launch_pair(const F16Launch &L, std::string &err) {
    using T = PairCfg<STAGES>;
    auto kernel = gemm_f16_nt_pair_kernel<STAGES>;
    static int max_clusters[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        err = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    const bool cached = dev >= 0 && dev < 64 && max_clusters[dev] > 0;
    if (!cached) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmemBytes);
        if (e != cudaSuccess) {
            err = std::string("cudaFuncSetAttribute(max dynamic smem): ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = T::kSmemBytes;
    cfg.stream = L.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = cached ? max_clusters[dev] : 0;
    if (!cached) {
        // How many CTA pairs can be resident at once: the persistent grid size.
        cfg.gridDim = dim3(2);
        e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
        if (e != cudaSuccess || clusters <= 0) {
            err = std::string("cudaOccupancyMaxActiveClusters: ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
        if (dev >= 0 && dev < 64) max_clusters[dev] = clusters;
    }
    CUtensorMap tmA, tmB;
    if (!encode_half_map(&tmA, L.A, L.M, L.K, kBM, kBK, err)) return GEMM_ERR_CUDA;
    if (!encode_half_map(&tmB, L.B, L.N, L.K, 128, kBK, err)) return GEMM_ERR_CUDA;

    F16Args args;
    args.C = static_cast<__half *>(L.C);
    args.M = L.M;
    args.N = L.N;
    args.K = L.K;
    args.m_tiles = (L.M + 255) / 256;
    args.n_tiles = (L.N + 255) / 256;
    args.num_kb = (L.K + kBK - 1) / kBK;
    args.vec_store = (L.N % 8 == 0) && ((reinterpret_cast<uintptr_t>(L.C) & 15u) == 0);
    args.tma_store = args.vec_store;
    args.timeout_ns = L.timeout_ns;
    args.debug_skip_kblock = L.debug_skip_kblock;
    CUtensorMap tmC;
    std::memset(&tmC, 0, sizeof tmC);
    if (args.tma_store && !encode_half_map(&tmC, L.C, L.M, L.N, 32, 64, err)) return GEMM_ERR_CUDA;
    const int tiles = args.m_tiles * args.n_tiles;
    int pairs = L.grid / 2;
    if (pairs < 1) pairs = 1;
    if (pairs > clusters) pairs = clusters;
    if (pairs > tiles) pairs = tiles;
    cfg.gridDim = dim3(2 * pairs);
    cfg.numAttrs = 2;  // cluster shape + programmatic dependent launch
    e = cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, tmC, args);
    if (e != cudaSuccess) {
        err = std::string("gemm_f16_nt pair kernel launch: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

}  // namespace

int f16_launch(const F16Launch &L, std::string &err) {
    if (L.K == 0) {
        const size_t count = static_cast<size_t>(L.M) * L.N;
        const int blocks = static_cast<int>((count + 255) / 256 < 4096 ? (count + 255) / 256 : 4096);
        zero_half_kernel<<<blocks, 256, 0, L.stream>>>(static_cast<__half *>(L.C), count);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) {
            err = std::string("zero fill launch: ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
        return GEMM_OK;
    }
    switch (L.variant) {
        case GEMM_F16_128x256: return launch_variant<256, 4>(L, err);
        case GEMM_F16_128x128: return launch_variant<128, 6>(L, err);
        case GEMM_F16_256x256_PAIR: return launch_pair<6>(L, err);
        default: err = "unknown fp16 variant"; return GEMM_ERR_INVALID_ARG;
    }
}

int f16_status_read_clear(cudaStream_t stream, int *code, std::string &err) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
        err = std::string("cudaStreamSynchronize: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_f16_status, sizeof(int));
    if (e == cudaSuccess && v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_f16_status, &zero, sizeof(int));
    }
    if (e != cudaSuccess) {
        err = std::string("status word access: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    *code = v;
    return GEMM_OK;
}

}  // namespace gb300
