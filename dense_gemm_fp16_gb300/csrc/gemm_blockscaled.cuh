// gemm_blockscaled.cuh -- block-scaled FP8 (MXFP8) and FP4 (NVFP4) NT
// products on the sm_103a tensor cores: their kernels, scale packing and
// launchers.  Included once, by gemm_f16_nt.cu, after the fp16 kernels: it
// shares that file's argument block, epilogue helpers, tensor-map encoding
// and device status word, and is compiled in the same translation unit.
#pragma once

namespace gb300 {
namespace {

// ---------------------------------------------------------------------------
// Block-scaled FP8 (MXFP8) NT product, "异步拷贝与 Hopper/Blackwell 新特性",
// section "Blackwell 概览 sm_100": E4M3 A [M,K] and B [N,K] (K-major), one
// UE8M0 scale per row per 32 elements of K, fp32 accumulation on the tensor
// cores (tcgen05.mma kind::mxf8f6f4, block_scale, scale_vec::1X), half C.
//
// The same warp roles as the 1-CTA fp16 kernel, with 128 x BN output tiles
// and 128-byte k-blocks.  With each stage's A and B boxes, the producer
// loads the k-block's scales into that stage's slot of a scale region after
// the stages: per 128-row tile a 512-byte chunk of 128 rows x 4 scales (four
// chunks for NVFP4), stored contiguously in the operand's scale array (see
// gemm_mxfp8_nt in gemm.h for the layout: byte 16*(r % 32) + 4*(r / 32) + j
// of the chunk is row r's j-th scale).  The MMA thread copies each chunk into
// TMEM (tcgen05.cp 32x128b.warpx4: TMEM lane r holds, in column c, the four
// scales of row 32c + r % 32) ahead of the k-block's four MMAs, which pick
// scale j through the descriptor's scale-factor IDs (MXFP8, K = 32) or take
// all four bytes of their own chunk (NVFP4, K = 64); copies and MMAs from one
// thread run in order, so one scale area per stage suffices.
// ---------------------------------------------------------------------------

constexpr int kMxBK = 128;       // K elements (bytes) per k-block: one 128-byte swizzle row
constexpr int kMxStages = 5;
constexpr int kMxUmmaK = 32;     // bytes of K per MMA instruction (32 E4M3 or 64 E2M1 elements)
constexpr int kMxSfChunk = 512;  // 128 rows x 4 scales

// BN output columns per tile (128 or 256: B's scales are BN/128 chunks),
// STAGES ring stages, EBUFS epilogue staging buffers per warp, ACC TMEM
// accumulators (2: the epilogue of a tile overlaps the next tile's MMAs).
// FMT: kFmtMx8 (E4M3, a UE8M0 scale per 32 of K: one 512-byte chunk per
// 128 rows per 128-byte k-block) or kFmtNv4 (E2M1 pairs, a UE4M3 scale per
// 16 of K: four chunks per 128 rows per 128-byte k-block, one per MMA).
constexpr int kFmtMx8 = 0;
constexpr int kFmtNv4 = 1;

template <int BN, int STAGES, int EBUFS, int ACC, int FMT = kFmtMx8>
struct MxCfg {
    static constexpr int kABytes = kBM * kMxBK;
    static constexpr int kBBytes = BN * kMxBK;
    static constexpr int kSfbChunks = BN / 128;                 // B's 128-row tiles
    static constexpr int kCpt = FMT == kFmtNv4 ? 4 : 1;         // chunks per row tile per k-block
    static constexpr int kSfBytes = (1 + kSfbChunks) * kCpt * kMxSfChunk;
    // operand stages (whole 1 KB multiples: the 128-byte swizzle), then each
    // stage's scale chunks, then the epilogue buffers
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kSfOffset = STAGES * kStageBytes;
    static constexpr int kTmemCols = 512;  // accumulators, then the scale columns of each stage
    static constexpr int kSfCols = 4 * (1 + kSfbChunks) * kCpt;
    static constexpr int kSfCol0 = ACC * BN;
    static constexpr int kNumBars = 2 * STAGES + 5;
    static constexpr int kEpiOffset = (kSfOffset + STAGES * kSfBytes + 1023) / 1024 * 1024;
    static constexpr int kBarOffset = kEpiOffset + 4 * EBUFS * kEpiBufBytes;
    static constexpr int kSmemBytes = 1024 + kBarOffset + kNumBars * 8 + 16;
    static_assert(kStageBytes % 1024 == 0, "stages keep the 1 KB alignment of the swizzled boxes");
    static_assert(BN == 128 || BN == 256, "B's scales come in whole 128-row chunks");
    static_assert(ACC == 1 || ACC == 2, "one or two accumulators");
    static_assert(FMT == kFmtMx8 || FMT == kFmtNv4, "MXFP8 or NVFP4");
    static_assert(kSfCol0 + kSfCols * STAGES <= kTmemCols, "scale columns fit the allocation");
    static_assert(kSmemBytes <= 232448, "fits the 227 KB opt-in limit");
};

struct MxArgs {
    const uint8_t *sfa;  // scale chunks of A: [ceil(M/128)][ceil(K/128)][512]
    const uint8_t *sfb;  // scale chunks of B: [ceil(N/128)][ceil(K/128)][512]
};

// The CTA-pair form of the NVFP4 MMA (issued by the even CTA for both).
__device__ __forceinline__ void mma_nvf4_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Stores of the 8-warp epilogue: KH accumulator columns (fp32 bits in v) of
// output row row0 + lane from column n0 on, rounded to half (NVFP4: times
// alpha first).  STAGED, and when C allows TMA stores, 32 x 32 halves at a
// time go through the warp's 2 KB buffer `buf` and one TMA store: row `lane`
// is 64 bytes, its 16-byte chunk j at chunk j ^ ((lane / 2) % 4) -- the TMA's
// 64-byte swizzle, under which every 8 lanes' stores cover all 32 banks.
// Otherwise each lane stores its own row with 16-byte stores.
template <int KH, int FMT, bool STAGED>
__device__ __forceinline__ void mx_epi8_store(const F16Args &args, const CUtensorMap *tmC, uint32_t (&v)[KH],
                                              int row0, int n0, int lane, uint32_t buf) {
    if constexpr (FMT == kFmtNv4) {
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int q = 0; q < KH / 8; ++q) epi_apply8<0>(args.epi, &v[8 * q], zero, zero);
    }
    if (STAGED && args.tma_store) {
        const uint32_t row_addr = buf + static_cast<uint32_t>(lane) * 64u;
#pragma unroll
        for (int c = 0; c < KH / 32; ++c) {
            if (lane == 0) bulk_wait_group_read<0>();  // the last store has read the buffer
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t *p = &v[32 * c + 8 * j];
                __half2 h0 = __floats2half2_rn(__uint_as_float(p[0]), __uint_as_float(p[1]));
                __half2 h1 = __floats2half2_rn(__uint_as_float(p[2]), __uint_as_float(p[3]));
                __half2 h2 = __floats2half2_rn(__uint_as_float(p[4]), __uint_as_float(p[5]));
                __half2 h3 = __floats2half2_rn(__uint_as_float(p[6]), __uint_as_float(p[7]));
                st_shared_v4(row_addr + (static_cast<uint32_t>(j ^ ((lane >> 1) & 3)) << 4),
                             *reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1),
                             *reinterpret_cast<uint32_t *>(&h2), *reinterpret_cast<uint32_t *>(&h3));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                // a box wholly past the last row or column would store nothing
                if (row0 < args.M && n0 + 32 * c < args.N) tma_store_2d(tmC, buf, n0 + 32 * c, row0);
                bulk_commit_group();
            }
        }
    } else {
        const int m = row0 + lane;
        __half *crow = args.C + static_cast<size_t>(m) * args.N;
#pragma unroll
        for (int c = 0; c < KH / 32; ++c)
            store_row_chunk(crow, m < args.M, n0 + 32 * c, args.N, args.vec_store,
                            *reinterpret_cast<const uint32_t(*)[32]>(&v[32 * c]));
    }
}

// EW epilogue warps: 4 (one per TMEM lane quarter, the tile through the
// staged TMA-store epilogue) or 8 (two per quarter, each reading its half of
// the columns into registers and releasing the accumulator before it
// converts and stores them: with one accumulator, the next tile's MMAs wait
// only for the TMEM reads).  With EW = 8, EBUFS = 1 stores 32 x 32 halves at
// a time through a 2 KB buffer per warp and one TMA store (coalesced), and
// EBUFS = 0 stores each lane's row with 16-byte stores.
template <int BN, int STAGES, int EBUFS, int ACC, int FMT = kFmtMx8, int EW = 4>
__global__ void __launch_bounds__((2 + EW) * 32, 1)
    gemm_mxfp8_nt_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmC, const F16Args args, const MxArgs mx) {
    using T = MxCfg<BN, STAGES, EBUFS, ACC, FMT>;
    static_assert(EW == 4 || (EW == 8 && (EBUFS == 0 || EBUFS == 1)),
                  "the 8-warp epilogue stores from registers, directly or through 2 KB per warp");
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

    // The A and B boxes of this CTA's first ring fill are asked of L2 before
    // the set-up and the dependent-launch wait, one per lane of warp 2.  A
    // prefetch only fills L2, where a previous kernel's writes land too.
    if (args.prefetch_first && warp == 2 && lane < 2 * STAGES && lane / 2 < args.num_kb &&
        static_cast<int>(blockIdx.x) < args.m_tiles * args.n_tiles) {
        const int mt = static_cast<int>(blockIdx.x) % args.m_tiles;
        const int nt = static_cast<int>(blockIdx.x) / args.m_tiles;
        if (lane & 1)
            tma_prefetch_l2_2d(&tmB, (lane >> 1) * kMxBK, nt * BN);
        else
            tma_prefetch_l2_2d(&tmA, (lane >> 1) * kMxBK, mt * kBM);
    }

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
            mbar_init(acce_bar(b), EW);
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
    pdl_launch_dependents();
    pdl_wait_prerequisites();

    const int total_tiles = args.m_tiles * args.n_tiles;
    const int num_kb = args.num_kb;
    uint32_t armed = 0, arm_parity = 0;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
                const int mt = tile % args.m_tiles;
                const int nt = tile / args.m_tiles;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, args.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + stage * T::kStageBytes;
                    const uint32_t sb = sa + T::kABytes;
                    const uint32_t ssf = sbase + T::kSfOffset + stage * T::kSfBytes;
                    // the k-block's scale chunks: kCpt consecutive chunks per
                    // 128-row tile; B's row tiles past N do not exist in the
                    // scale array and are not fetched (their stale values meet
                    // only output columns >= N, which the store clips)
                    constexpr uint32_t kTileSf = T::kCpt * kMxSfChunk;
                    const int b_tiles = (args.N - nt * BN + 127) / 128;
                    const int b_here = b_tiles < T::kSfbChunks ? b_tiles : T::kSfbChunks;
                    // test hook: the first tile's k-block debug_skip_kblock is never loaded
                    if (!(tile == static_cast<int>(blockIdx.x) && kb == args.debug_skip_kblock)) {
                        mbar_arrive_expect_tx(full_bar(stage),
                                              T::kABytes + T::kBBytes + (1 + b_here) * kTileSf);
                        tma_load_2d(sa, &tmA, full_bar(stage), kb * kMxBK, mt * kBM);
                        tma_load_2d(sb, &tmB, full_bar(stage), kb * kMxBK, nt * BN);
                        bulk_load(ssf, mx.sfa + (static_cast<size_t>(mt) * num_kb + kb) * kTileSf, kTileSf,
                                  full_bar(stage));
                        for (int c = 0; c < b_here; ++c)
                            bulk_load(ssf + (1 + c) * kTileSf,
                                      mx.sfb + (static_cast<size_t>(nt * T::kSfbChunks + c) * num_kb + kb) * kTileSf,
                                      kTileSf, full_bar(stage));
                        armed |= 1u << stage;
                        arm_parity ^= 1u << stage;
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                if (!*abort_flag) record_timeout(1);
                *abort_flag = 1;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ scale copies + MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int i = 0;
            for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++i) {
                const int b = i % ACC;
                const uint32_t ap = (i / ACC) & 1;
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
                    const uint32_t sb = sa + T::kABytes;
                    const uint32_t ssf = sbase + T::kSfOffset + stage * T::kSfBytes;
                    // Each chunk is 32 rows of 16 bytes (8-row core matrices 128
                    // bytes apart) and fills 4 TMEM columns.  A's chunk a lands at
                    // sfa + 4a; B's chunk a of row tile c at sfb + 4(a * tiles + c),
                    // so that each MMA's B scales (all of B's rows) are contiguous.
                    const uint32_t sfa_tmem = tmem_base + static_cast<uint32_t>(T::kSfCol0 + T::kSfCols * stage);
                    const uint32_t sfb_tmem = sfa_tmem + 4u * T::kCpt;
#pragma unroll
                    for (int a = 0; a < T::kCpt; ++a) {
                        tmem_cp_32x128b_warpx4(sfa_tmem + 4u * a, plain_kmajor_desc(ssf + a * kMxSfChunk, 128, 128));
#pragma unroll
                        for (int c = 0; c < T::kSfbChunks; ++c)
                            tmem_cp_32x128b_warpx4(
                                sfb_tmem + 4u * (a * T::kSfbChunks + c),
                                plain_kmajor_desc(ssf + ((1 + c) * T::kCpt + a) * kMxSfChunk, 128, 128));
                    }
                    const uint64_t adesc = sw128_kmajor_desc(sa);
                    const uint64_t bdesc = sw128_kmajor_desc(sb);
#pragma unroll
                    for (int j = 0; j < kMxBK / kMxUmmaK; ++j) {
                        // 32 bytes of K per MMA (32 FP8 or 64 FP4): the start
                        // address advances 32 bytes.
                        if constexpr (FMT == kFmtMx8) {
                            // scale j of each row (its 32-element block) applies
                            mma_mxf8_ss(d_tmem, adesc + 2u * j, bdesc + 2u * j, idesc_mxf8_e4m3(kBM, BN, j),
                                        sfa_tmem, sfb_tmem, (kb > 0 || j > 0) ? 1u : 0u);
                        } else {
                            // the four 16-element scales of chunk j apply
                            mma_nvf4_ss(d_tmem, adesc + 2u * j, bdesc + 2u * j, idesc_nvf4_e2m1(kBM, BN),
                                        sfa_tmem + 4u * j, sfb_tmem + 4u * T::kSfbChunks * j,
                                        (kb > 0 || j > 0) ? 1u : 0u);
                        }
                    }
                    mma_commit(empty_bar(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(accf_bar(b));
            }
            if (!ok) {
                if (!*abort_flag) record_timeout(2);
                *abort_flag = 1;
            }
        }
        __syncwarp();
    } else if constexpr (EW == 8) {
        // ------------------------------------------------------------ epilogue, 8 warps
        const int quarter = warp & 3;        // TMEM lanes this warp may read
        const int half = (warp - 2) >> 2;    // which half of the tile's columns
        const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
        int i = 0;
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++i) {
            const int b = i % ACC;
            const uint32_t ap = (i / ACC) & 1;
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
            constexpr int kHalf = BN / 2;
            uint32_t v[kHalf];
            const uint32_t taddr = tmem_base + lane_field + static_cast<uint32_t>(b * BN + half * kHalf);
#pragma unroll
            for (int c = 0; c < kHalf / 32; ++c)
                tmem_load_32cols(taddr + 32u * c, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * c]));
            // the accumulator is in registers: hand it back to the MMAs
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(b));
            const int mt = tile % args.m_tiles;
            const int nt = tile / args.m_tiles;
            mx_epi8_store<kHalf, FMT, (EBUFS > 0)>(args, &tmC, v, mt * kBM + quarter * 32, nt * BN + half * kHalf,
                                                  lane, sbase + T::kEpiOffset + static_cast<uint32_t>(warp - 2) * 2048u);
        }
        if (lane == 0) bulk_wait_group_all();
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;
        const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t stage_smem = sbase + T::kEpiOffset + (warp - 2) * EBUFS * kEpiBufBytes;
        uint32_t step = 0;
        int i = 0;
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++i) {
            const int b = i % ACC;
            const uint32_t ap = (i / ACC) & 1;
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
            // NVFP4: the tensor-level scale alpha through the epilogue (ACT 0)
            epilogue_warp_tile<BN, EBUFS, FMT == kFmtNv4 ? 0 : -1>(
                args, &tmC, tmem_base + lane_field + static_cast<uint32_t>(b * BN), mt * kBM + quarter * 32,
                nt * BN, lane, stage_smem, step);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(b));
        }
        if (lane == 0) bulk_wait_group_all();
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
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

// CTA-pair form: a 2-CTA cluster computes a 256 x 128 output tile with
// tcgen05.mma.cta_group::2 (M 256, N 128, K 32).  CTA r loads its 128 rows of
// A, its 64 rows of B and the two scale chunks its TMEM needs (its own rows
// of A; all 128 rows of B), all completing on the even CTA's full barrier;
// per k-block an SM takes 25 KB (against 33 KB for a 1-CTA 128 x 128 tile)
// for the same MMA time.  The scale chunks go through TMA (a 2D view of the
// chunk arrays as 256-byte rows) so that the odd CTA's copies can complete on
// the even CTA's barrier.  Barriers and roles as in the fp16 pair kernel.
// BN: pair tile columns (128 or 256; each CTA loads BN/2 rows of B and all
// BN/128 scale chunks of B), STAGES, EBUFS epilogue buffers per warp, ACC
// accumulators, FMT as in the 1-CTA kernel (NVFP4: four chunks per row tile
// per k-block, one TMA box of 8 rows), EW epilogue warps per CTA (4: the
// staged epilogue; 8: the register epilogue that releases the accumulator
// early, EBUFS = 1).
template <int BN, int STAGES, int EBUFS, int ACC, int FMT = kFmtMx8>
struct MxPairCfg {
    static constexpr int kABytes = kBM * kMxBK;             // this CTA's 128 rows of A
    static constexpr int kBBytes = (BN / 2) * kMxBK;        // this CTA's half of B
    static constexpr int kSfbChunks = BN / 128;
    static constexpr int kCpt = FMT == kFmtNv4 ? 4 : 1;     // chunks per row tile per k-block
    static constexpr int kSfBytes = (1 + kSfbChunks) * kCpt * kMxSfChunk;
    // operand stages (whole 1 KB multiples: the 128-byte swizzle), then each
    // stage's scale chunks, then the epilogue buffers
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kSfOffset = STAGES * kStageBytes;
    static constexpr int kTmemCols = 512;  // accumulators, then the scale columns of each stage
    static constexpr int kSfCols = 4 * (1 + kSfbChunks) * kCpt;
    static constexpr int kSfCol0 = ACC * BN;
    static constexpr int kNumBars = 2 * STAGES + 5;
    static constexpr int kEpiOffset = (kSfOffset + STAGES * kSfBytes + 1023) / 1024 * 1024;
    static constexpr int kBarOffset = kEpiOffset + 4 * EBUFS * kEpiBufBytes;
    static constexpr int kSmemBytes = 1024 + kBarOffset + kNumBars * 8 + 16;
    static_assert(kStageBytes % 1024 == 0, "stages keep the 1 KB alignment of the swizzled boxes");
    static_assert(BN == 128 || BN == 256, "B's scales come in whole 128-row chunks");
    static_assert(kSfCol0 + kSfCols * STAGES <= kTmemCols, "scale columns fit the allocation");
    static_assert(kSmemBytes <= 232448, "fits the 227 KB opt-in limit");
};

template <int BN, int STAGES, int EBUFS, int ACC, int FMT = kFmtMx8, int EW = 4>
__global__ void __launch_bounds__((2 + EW) * 32, 1)
    gemm_mxfp8_nt_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                              const __grid_constant__ CUtensorMap tmC,
                              const __grid_constant__ CUtensorMap tmSFA,
                              const __grid_constant__ CUtensorMap tmSFB, const F16Args args) {
    using T = MxPairCfg<BN, STAGES, EBUFS, ACC, FMT>;
    static_assert(EW == 4 || (EW == 8 && EBUFS == 1), "8 epilogue warps stage through 2 KB each");
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
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmSFA);
        tma_prefetch_desc(&tmSFB);
        if (args.tma_store) tma_prefetch_desc(&tmC);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 2 * EW);  // every epilogue warp of both CTAs
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
    cluster_sync();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    pdl_launch_dependents();
    pdl_wait_prerequisites();

    const int total_tiles = args.m_tiles * args.n_tiles;
    const int num_kb = args.num_kb;
    uint32_t armed = 0, arm_parity = 0;

    if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int tile = pair; tile < total_tiles && ok; tile += num_pairs) {
                const int mt = tile % args.m_tiles;
                const int nt = tile / args.m_tiles;
                const int a_tile128 = 2 * mt + static_cast<int>(rank);  // this CTA's 128-row tile of A
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait_cluster(empty_bar(stage), phase ^ 1u, args.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + stage * T::kStageBytes;
                    const uint32_t ssf = sbase + T::kSfOffset + stage * T::kSfBytes;
                    const uint32_t full_leader = mapa_shared(full_bar(stage), 0);
                    // test hook: the even CTA never arms nor loads the first
                    // tile's k-block debug_skip_kblock (the odd CTA's bytes
                    // still land, but the stage's phase can never complete)
                    const bool skip = tile == pair && kb == args.debug_skip_kblock && leader;
                    if (!skip) {
                        if (leader) {
                            // both CTAs' operand and scale bytes (the stage's padding is not loaded)
                            mbar_arrive_expect_tx(full_bar(stage), 2 * (T::kABytes + T::kBBytes + T::kSfBytes));
                            armed |= 1u << stage;
                            arm_parity ^= 1u << stage;
                        }
                        tma_load_2d_pair(sa, &tmA, full_leader, kb * kMxBK, a_tile128 * kBM);
                        tma_load_2d_pair(sa + T::kABytes, &tmB, full_leader, kb * kMxBK,
                                         nt * BN + static_cast<int>(rank) * (BN / 2));
                        // scale chunks: 512 bytes = two 256-byte rows of the 2D view;
                        // the k-block's kCpt chunks of a row tile are contiguous
                        tma_load_2d_pair(ssf, &tmSFA, full_leader, 0, 2 * T::kCpt * (a_tile128 * num_kb + kb));
#pragma unroll
                        for (int c = 0; c < T::kSfbChunks; ++c)
                            tma_load_2d_pair(ssf + (1 + c) * T::kCpt * kMxSfChunk, &tmSFB, full_leader, 0,
                                             2 * T::kCpt * ((nt * T::kSfbChunks + c) * num_kb + kb));
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                if (!*abort_flag) record_timeout(1);
                *abort_flag = 1;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ scale copies + MMA issuer (even CTA)
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            // the k-block's scale chunks into this stage's TMEM columns (the
            // chunk placement of the 1-CTA kernel)
            auto copy_scales = [&](int st) {
                const uint32_t ssf = sbase + T::kSfOffset + st * T::kSfBytes;
                const uint32_t sfa_tmem = tmem_base + static_cast<uint32_t>(T::kSfCol0 + T::kSfCols * st);
                const uint32_t sfb_tmem = sfa_tmem + 4u * T::kCpt;
#pragma unroll
                for (int a = 0; a < T::kCpt; ++a) {
                    tmem_cp_32x128b_warpx4_pair(sfa_tmem + 4u * a, plain_kmajor_desc(ssf + a * kMxSfChunk, 128, 128));
#pragma unroll
                    for (int c = 0; c < T::kSfbChunks; ++c)
                        tmem_cp_32x128b_warpx4_pair(
                            sfb_tmem + 4u * (a * T::kSfbChunks + c),
                            plain_kmajor_desc(ssf + ((1 + c) * T::kCpt + a) * kMxSfChunk, 128, 128));
                }
            };
            int i = 0;
            for (int tile = pair; tile < total_tiles; tile += num_pairs, ++i) {
                const int b = i % ACC;
                const uint32_t ap = (i / ACC) & 1;
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
                    copy_scales(stage);
                    const uint32_t sa = sbase + stage * T::kStageBytes;
                    const uint32_t sfa_tmem = tmem_base + static_cast<uint32_t>(T::kSfCol0 + T::kSfCols * stage);
                    const uint32_t sfb_tmem = sfa_tmem + 4u * T::kCpt;
                    const uint64_t adesc = sw128_kmajor_desc(sa);
                    const uint64_t bdesc = sw128_kmajor_desc(sa + T::kABytes);
#pragma unroll
                    for (int j = 0; j < kMxBK / kMxUmmaK; ++j) {
                        if constexpr (FMT == kFmtMx8)
                            mma_mxf8_ss_pair(d_tmem, adesc + 2u * j, bdesc + 2u * j, idesc_mxf8_e4m3(256, BN, j),
                                             sfa_tmem, sfb_tmem, (kb > 0 || j > 0) ? 1u : 0u);
                        else
                            mma_nvf4_ss_pair(d_tmem, adesc + 2u * j, bdesc + 2u * j, idesc_nvf4_e2m1(256, BN),
                                             sfa_tmem + 4u * j, sfb_tmem + 4u * T::kSfbChunks * j,
                                             (kb > 0 || j > 0) ? 1u : 0u);
                    }
                    const int nstage = stage + 1 == STAGES ? 0 : stage + 1;
                    const uint32_t nphase = nstage == 0 ? phase ^ 1u : phase;
                    mma_commit_pair_multicast(empty_bar(stage), 0x3);
                    stage = nstage;
                    phase = nphase;
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
        const uint32_t stage_smem = sbase + T::kEpiOffset + (warp - 2) * EBUFS * kEpiBufBytes;
        uint32_t step = 0;
        int i = 0;
        for (int tile = pair; tile < total_tiles; tile += num_pairs, ++i) {
            const int b = i % ACC;
            const uint32_t ap = (i / ACC) & 1;
            int ok = 1;
            if (lane == 0) ok = mbar_wait_cluster(accf_bar(b), ap, args.timeout_ns, abort_flag) ? 1 : 0;
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
            const int row0 = mt * 256 + static_cast<int>(rank) * 128 + quarter * 32;
            if constexpr (EW == 8) {
                // this warp's half of the columns into registers, then the
                // accumulator goes back to the MMAs before the stores
                constexpr int kHalf = BN / 2;
                const int half = (warp - 2) >> 2;
                uint32_t v[kHalf];
                const uint32_t taddr = tmem_base + lane_field + static_cast<uint32_t>(b * BN + half * kHalf);
#pragma unroll
                for (int c = 0; c < kHalf / 32; ++c)
                    tmem_load_32cols(taddr + 32u * c, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * c]));
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(b), 0));
                mx_epi8_store<kHalf, FMT, true>(args, &tmC, v, row0, nt * BN + half * kHalf, lane,
                                                sbase + T::kEpiOffset + static_cast<uint32_t>(warp - 2) * 2048u);
            } else {
                // NVFP4: the tensor-level scale alpha through the epilogue (ACT 0)
                epilogue_warp_tile<BN, EBUFS, FMT == kFmtNv4 ? 0 : -1>(
                    args, &tmC, tmem_base + lane_field + static_cast<uint32_t>(b * BN), row0, nt * BN, lane,
                    stage_smem, step);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(b), 0));
            }
        }
        if (lane == 0) bulk_wait_group_all();
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (*abort_flag) {
        if (leader && warp == 0 && lane == 0) {
            for (int s = 0; s < STAGES; ++s)
                if (armed & (1u << s))
                    (void)mbar_wait_cluster(full_bar(s), ((arm_parity >> s) & 1u) ^ 1u, args.timeout_ns,
                                            &never_abort);
        }
        if (leader && warp == 1 && lane == 0) {
            mma_commit_pair(drain_bar);
            (void)mbar_wait_cluster(drain_bar, 0, args.timeout_ns, &never_abort);
        }
        __syncwarp();
        tc_fence_before_sync();
        __syncthreads();
    }
    cluster_sync();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, T::kTmemCols);
    }
}

// Plain scales [rows][ksf] -> the kernels' chunk layout (`cpr` chunks of 4
// scales per 128-row tile), padded with `pad` (a scale of 1) past the last
// row and the last scale; one thread per output byte.
__global__ void mx_pack_scales_kernel(const uint8_t *__restrict__ plain, uint8_t *__restrict__ blocked,
                                      int rows, int ksf, int cpr, uint8_t pad, size_t total) {
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t o = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; o < total; o += stride) {
        const size_t chunk = o / kMxSfChunk;
        const int within = static_cast<int>(o % kMxSfChunk);
        const int rt = static_cast<int>(chunk / cpr), kb = static_cast<int>(chunk % cpr);
        const int r = rt * 128 + (within >> 4) + 32 * ((within >> 2) & 3);
        const int j = kb * 4 + (within & 3);
        blocked[o] = (r < rows && j < ksf) ? plain[static_cast<size_t>(r) * ksf + j] : pad;
    }
}

}  // namespace

namespace {

// The argument block of a block-scaled launch: tile_rows (128, or 256 for a
// CTA pair) by BN output tiles, num_kb 128-byte k-blocks, TMA stores when C
// allows them, and for NVFP4 the tensor-level scale alpha through the
// epilogue (C = alpha * the block-scaled product); no stream-K.
inline F16Args mx_args(const MxLaunch &L, int tile_rows, int BN, int num_kb) {
    F16Args args;
    args.C = static_cast<__half *>(L.C);
    args.M = L.M;
    args.N = L.N;
    args.K = L.K;
    args.m_tiles = (L.M + tile_rows - 1) / tile_rows;
    args.n_tiles = (L.N + BN - 1) / BN;
    args.num_kb = num_kb;
    // operand bytes: one per E4M3 element, one per E2M1 pair
    args.prefetch_first = (static_cast<size_t>(L.M) + L.N) * static_cast<size_t>(L.K) / (L.fmt == kFmtNv4 ? 2 : 1) >= kPrefetchMinBytes;
    args.vec_store = (L.N % 8 == 0) && ((reinterpret_cast<uintptr_t>(L.C) & 15u) == 0);
    args.tma_store = args.vec_store;
    EpiSpec scale;
    if (L.fmt == kFmtNv4) {
        scale.alpha = L.alpha;
        scale.on = 1;
    }
    args.epi = make_epi(scale, L.N);
    args.timeout_ns = L.timeout_ns;
    args.debug_skip_kblock = L.debug_skip_kblock;
    args.dp_tiles = 0;
    args.sk_units = 0;
    args.sk_ws = nullptr;
    args.sk_flags = nullptr;
    args.seq = 0;
    return args;
}

template <int BN, int STAGES, int EBUFS, int ACC, int FMT = kFmtMx8, int EW = 4>
int mx_launch_pair(const MxLaunch &L, std::string &err) {
    using T = MxPairCfg<BN, STAGES, EBUFS, ACC, FMT>;
    auto kernel = gemm_mxfp8_nt_pair_kernel<BN, STAGES, EBUFS, ACC, FMT, EW>;
    const int kbytes = FMT == kFmtNv4 ? L.K / 2 : L.K;  // bytes of K per row
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
    cfg.blockDim = dim3((2 + EW) * 32);
    cfg.dynamicSmemBytes = T::kSmemBytes;
    cfg.stream = L.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = cached ? max_clusters[dev] : 0;
    if (!cached) {
        cfg.gridDim = dim3(2);
        e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
        if (e != cudaSuccess || clusters <= 0) {
            err = std::string("cudaOccupancyMaxActiveClusters: ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
        if (dev >= 0 && dev < 64) max_clusters[dev] = clusters;
    }
    const int kbt = (kbytes + kMxBK - 1) / kMxBK;
    // 256-byte rows of the scale chunk arrays; a k-block's chunks of one row
    // tile are 2 * kCpt of them
    const int sfa_rows = ((L.M + 127) / 128) * kbt * T::kCpt * 2;
    const int sfb_rows = ((L.N + 127) / 128) * kbt * T::kCpt * 2;
    CUtensorMap tmA, tmB, tmC, tmSFA, tmSFB;
    std::memset(&tmC, 0, sizeof tmC);
    if (!encode_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, L.A, L.M, kbytes, kBM, kMxBK, err) ||
        !encode_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, L.B, L.N, kbytes, BN / 2, kMxBK, err) ||
        !encode_map(&tmSFA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, L.SFA, sfa_rows, 256, 2 * T::kCpt, 256, err,
                    CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_map(&tmSFB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, L.SFB, sfb_rows, 256, 2 * T::kCpt, 256, err,
                    CU_TENSOR_MAP_SWIZZLE_NONE))
        return GEMM_ERR_CUDA;
    const F16Args args = mx_args(L, 256, BN, kbt);
    if (args.tma_store && !encode_map(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, L.C, L.M, L.N, 32,
                                      EW == 8 ? 32 : 64, err,
                                      EW == 8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B))
        return GEMM_ERR_CUDA;
    const int tiles = args.m_tiles * args.n_tiles;
    int pairs = L.grid > 0 ? L.grid / 2 : clusters;
    if (pairs < 1) pairs = 1;
    if (pairs > clusters) pairs = clusters;
    if (pairs > tiles) pairs = tiles;
    cfg.gridDim = dim3(2 * pairs);
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, tmC, tmSFA, tmSFB, args);
    if (e != cudaSuccess) {
        err = std::string("gemm_mxfp8_nt pair kernel launch: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

template <int BN, int STAGES, int EBUFS, int ACC, int FMT = kFmtMx8, int EW = 4>
int mx_launch_1cta(const MxLaunch &L, std::string &err) {
    using T = MxCfg<BN, STAGES, EBUFS, ACC, FMT>;
    auto kernel = gemm_mxfp8_nt_kernel<BN, STAGES, EBUFS, ACC, FMT, EW>;
    const int kbytes = FMT == kFmtNv4 ? L.K / 2 : L.K;  // bytes of K per row
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        err = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmemBytes);
        if (e != cudaSuccess) {
            err = std::string("cudaFuncSetAttribute(max dynamic smem): ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
        if (dev >= 0 && dev < 64) configured[dev] = 1;
    }
    CUtensorMap tmA, tmB, tmC;
    std::memset(&tmC, 0, sizeof tmC);
    if (!encode_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, L.A, L.M, kbytes, kBM, kMxBK, err))
        return GEMM_ERR_CUDA;
    if (!encode_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, L.B, L.N, kbytes, BN, kMxBK, err))
        return GEMM_ERR_CUDA;
    const F16Args args = mx_args(L, kBM, BN, (kbytes + kMxBK - 1) / kMxBK);
    // C boxes: 32 rows x 64 columns (128-byte swizzle) for the 4-warp staged
    // epilogue, 32 x 32 (64-byte swizzle) for the 8-warp one
    if (args.tma_store && !encode_map(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, L.C, L.M, L.N, 32,
                                      EW == 8 ? 32 : 64, err,
                                      EW == 8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B))
        return GEMM_ERR_CUDA;
    MxArgs mx{static_cast<const uint8_t *>(L.SFA), static_cast<const uint8_t *>(L.SFB)};
    const int tiles = args.m_tiles * args.n_tiles;
    int grid = L.grid > 0 ? L.grid : L.sm_count;
    if (grid > tiles) grid = tiles;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((2 + EW) * 32);
    cfg.dynamicSmemBytes = T::kSmemBytes;
    cfg.stream = L.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, tmC, args, mx);
    if (e != cudaSuccess) {
        err = std::string("gemm_mxfp8_nt kernel launch: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

}  // namespace

int mx_launch(const MxLaunch &L, std::string &err) {
    if (L.fmt == kFmtNv4) {
        switch (L.variant) {
            // 128 x 256: the 8-warp register epilogue staging through 2 KB per
            // warp, 3 stages: 38.8 us at 5376 x 5376 x 2048 (direct 16-byte
            // stores with 4 stages: 40.3; the 4-warp staged epilogue: 50.4),
            // 118 at K = 8192 like the direct form.
            case 3: return mx_launch_1cta<256, 3, 1, 1, kFmtNv4, 8>(L, err);
            case 1: return mx_launch_1cta<128, kMxStages, 2, 2, kFmtNv4>(L, err);
            case 2: return mx_launch_pair<128, 6, 2, 2, kFmtNv4, 4>(L, err);
            case 4: return mx_launch_pair<256, 5, 1, 1, kFmtNv4, 8>(L, err);
            default: err = "unknown NVFP4 variant"; return GEMM_ERR_INVALID_ARG;
        }
    }
    switch (L.variant) {
        case 2: return mx_launch_pair<128, 7, 2, 2>(L, err);
        // 128 x 256: the 8-warp register epilogue staging through 2 KB per
        // warp: 46.1 us at 5376 x 5376 x 2048 against 52.0 for the 4-warp
        // staged one (whose single accumulator waits for the whole drain) and
        // 52 for direct 16-byte stores (uncoalesced, one row per lane); equal
        // within the spread at K = 8192.
        case 3: return mx_launch_1cta<256, 4, 1, 1, kFmtMx8, 8>(L, err);
        case 4: return mx_launch_pair<256, 6, 1, 1, kFmtMx8, 8>(L, err);
        default: return mx_launch_1cta<128, kMxStages, 2, 2>(L, err);
    }
}

int mx_pack_scales_launch(int fmt, int rows, int K, const void *plain, void *blocked, cudaStream_t stream,
                          std::string &err) {
    // MXFP8: a scale per 32 elements, one chunk per 128 of K; NVFP4: a scale
    // per 16, four chunks per 256 of K (whole 128-byte k-blocks).
    const int ksf = fmt == kFmtNv4 ? K / 16 : K / 32;
    const int cpr = fmt == kFmtNv4 ? 4 * ((K + 255) / 256) : (K + kMxBK - 1) / kMxBK;
    const uint8_t pad = fmt == kFmtNv4 ? uint8_t(0x38) : uint8_t(127);  // 1.0 in E4M3 / UE8M0
    const size_t total = static_cast<size_t>((rows + 127) / 128) * cpr * kMxSfChunk;
    if (total == 0) return GEMM_OK;
    const size_t want = (total + 255) / 256;
    const int blocks = static_cast<int>(want < 4096 ? want : 4096);
    mx_pack_scales_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint8_t *>(plain),
                                                      static_cast<uint8_t *>(blocked), rows, ksf, cpr, pad,
                                                      total);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        err = std::string("scale packing launch: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

}  // namespace gb300
