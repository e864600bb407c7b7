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
#include <map>
#include <utility>
#include <mutex>

#include "gemm.h"
#include "epilogue.cuh"
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
// wait), 3 = epilogue (accumulator-ready wait), 4 = epilogue of a stream-K
// tile's first pair (wait for the other pairs' partials).
__device__ int g_f16_status = 0;

struct F16Args {
    __half *C;
    int M, N, K;
    int m_tiles, n_tiles, num_kb;
    int vec_store;          // N % 8 == 0 and C 16-byte aligned
    int tma_store;          // same condition: the epilogue stores through a C tensor map
    Epi epi;                // fused epilogue (epi.on == 0: the plain product)
    uint64_t timeout_ns;
    int debug_skip_kblock;  // -1 = none
    int debug_skip_publish = 0;  // test hook: stream-K partials are written but never flagged
    // Stream-K (pair kernel only): tiles [0, dp_tiles) are data-parallel, one
    // whole tile per work item; the k-blocks of the remaining tiles are split
    // evenly over the pairs (sk_units k-blocks in all).  A pair whose share
    // starts inside a tile writes its fp32 partial tile to its workspace slot
    // and sets its flag to `seq`; the pair holding k-block 0 adds those partials.
    int dp_tiles;
    int sk_units;
    float *sk_ws;           // slot (pair, rank): 128 rows x 256 fp32, row-major
    uint32_t *sk_flags;     // flag (pair, rank, epilogue warp), 8 per (pair, rank)
    uint32_t seq;           // this launch's sequence number (never 0)
    int raster = 1 << 30;   // tile rows per band of the tile order
    // Ask L2 for the first ring fill's boxes at kernel entry: operands this
    // large usually come from DRAM, while small ones are likely L2-resident,
    // where the prefetch only delays the set-up (1024^3: +0.2 us).
    int prefetch_first = 0;
};

// The first-fill prefetch pays from this many bytes of A and B.
constexpr size_t kPrefetchMinBytes = size_t(16) << 20;

// Output tile `tile` of the persistent order -> its tile row and column: bands
// of `raster` tile rows (the last one shorter), each walked column by column
// with the rows of a column consecutive.  With raster >= m_tiles this is the
// plain column order (tile % m_tiles, tile / m_tiles).
__device__ __forceinline__ void tile_mn(int tile, const F16Args &a, int &mt, int &nt) {
    const int g = a.raster < a.m_tiles ? a.raster : a.m_tiles;
    const int band_tiles = g * a.n_tiles;
    const int band = tile / band_tiles;
    const int first = band * g;
    const int h = a.m_tiles - first < g ? a.m_tiles - first : g;  // this band's rows
    const int r = tile - band * band_tiles;
    mt = first + r % h;
    nt = r / h;
}

// The work items of one CTA pair: whole data-parallel tiles first, then its
// contiguous share of the stream-K k-blocks cut at tile boundaries.  Every role
// of both CTAs walks the same sequence.  Shares are handed out in reverse pair
// order (share rank = num_pairs - 1 - pair): the pair that finishes a split
// tile (it holds k-block 0, which comes last in its share) then has a higher
// block index than the pairs contributing the tile's later k-blocks, so it is
// never resident before them and its wait for their partials cannot stall the
// launch of a contributor.
struct PairWork {
    int num_pairs, dp_tiles, num_kb, sk_units;
    int next_dp, u, u_end;
    __device__ PairWork(const F16Args &a, int pair, int pairs)
        : num_pairs(pairs), dp_tiles(a.dp_tiles), num_kb(a.num_kb), sk_units(a.sk_units),
          next_dp(pair), u(sk_begin(pairs - 1 - pair)), u_end(sk_begin(pairs - pair)) {}
    // first stream-K k-block of share rank r (no 64-bit division without stream-K work)
    __device__ int sk_begin(int r) const {
        return sk_units ? static_cast<int>((static_cast<long long>(r) * sk_units) / num_pairs) : 0;
    }
    __device__ bool next(int &tile, int &kb0, int &kb1) {
        if (next_dp < dp_tiles) {
            tile = next_dp;
            kb0 = 0;
            kb1 = num_kb;
            next_dp += num_pairs;
            return true;
        }
        if (u < u_end) {
            const int tl = u / num_kb;
            kb0 = u - tl * num_kb;
            kb1 = (num_kb < kb0 + (u_end - u)) ? num_kb : kb0 + (u_end - u);
            tile = dp_tiles + tl;
            u += kb1 - kb0;
            return true;
        }
        return false;
    }
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
// Stream-K partial tiles.  A slot holds one CTA's 128 x 256 fp32 partial
// accumulators in a lane-interleaved order: the region of epilogue warp `ew`
// starts at ew * NCOLS * 32 floats and element (slab c, vector v, lane l) --
// columns 4v .. 4v+3 of the 64-column slab c of the row that lane l holds --
// sits at float4 index (c * 16 + v) * 32 + l, so every warp-wide store or load
// moves 512 contiguous bytes.  The owner's warp with the same `ew` reads what
// the contributor's warp wrote.
struct Partials {
    const float *ws;
    int count;           // 0: none
    int first_slot;      // slots first_slot, first_slot - 2, ... (pairs below this one)
    int region;          // float offset of this warp's region in a slot
    int lane;
    uint32_t dsmem = 0;  // or: this warp's region of the partner pair's share (shared::cluster); 0: none
};

constexpr size_t kSkSlotFloatsDev = 128 * 256;

__device__ __forceinline__ void add_partial_slab(const Partials &pp, int c, uint32_t (&lo)[32],
                                                 uint32_t (&hi)[32]) {
    if (pp.dsmem) {
        // the partner pair's share of the same rows and columns, from its
        // shared memory (the layout epilogue_warp_share writes)
        float4 x[16];
#pragma unroll
        for (int v = 0; v < 16; ++v)
            x[v] = ld_dsmem_f4(pp.dsmem + static_cast<uint32_t>(((c * 16 + v) * 32 + pp.lane) * 16));
#pragma unroll
        for (int v = 0; v < 16; ++v) {
            uint32_t *d = v < 8 ? &lo[v * 4] : &hi[(v - 8) * 4];
            d[0] = __float_as_uint(__uint_as_float(d[0]) + x[v].x);
            d[1] = __float_as_uint(__uint_as_float(d[1]) + x[v].y);
            d[2] = __float_as_uint(__uint_as_float(d[2]) + x[v].z);
            d[3] = __float_as_uint(__uint_as_float(d[3]) + x[v].w);
        }
        return;
    }
#pragma unroll 1
    for (int q = 0; q < pp.count; ++q) {
        const float4 *src = reinterpret_cast<const float4 *>(
                                pp.ws + static_cast<size_t>(pp.first_slot - 2 * q) * kSkSlotFloatsDev +
                                pp.region) +
                            static_cast<size_t>(c) * 16 * 32 + pp.lane;
        float4 x[16];
#pragma unroll
        for (int v = 0; v < 16; ++v) x[v] = src[v * 32];
#pragma unroll
        for (int v = 0; v < 16; ++v) {
            uint32_t *d = v < 8 ? &lo[v * 4] : &hi[(v - 8) * 4];
            d[0] = __float_as_uint(__uint_as_float(d[0]) + x[v].x);
            d[1] = __float_as_uint(__uint_as_float(d[1]) + x[v].y);
            d[2] = __float_as_uint(__uint_as_float(d[2]) + x[v].z);
            d[3] = __float_as_uint(__uint_as_float(d[3]) + x[v].w);
        }
    }
}

// This warp's rows of the accumulator, unrounded, into shared memory at
// `dst` for the partner pair of a K-split cluster: float4 v of slab c of lane
// l at ((c * 16 + v) * 32 + l) * 16 bytes, so a warp's store covers 512
// contiguous bytes (no bank conflicts), as add_partial_slab reads it back.
template <int NCOLS>
__device__ __forceinline__ void epilogue_warp_share(uint32_t dst, uint32_t taddr, int lane) {
#pragma unroll 1
    for (int c = 0; c < NCOLS / 64; ++c) {
        uint32_t lo[32], hi[32];
        tmem_load_32cols(taddr + static_cast<uint32_t>(c * 64), lo);
        tmem_load_32cols(taddr + static_cast<uint32_t>(c * 64 + 32), hi);
#pragma unroll
        for (int v = 0; v < 16; ++v) {
            const uint32_t *s = v < 8 ? &lo[v * 4] : &hi[(v - 8) * 4];
            st_shared_v4(dst + static_cast<uint32_t>(((c * 16 + v) * 32 + lane) * 16), s[0], s[1], s[2], s[3]);
        }
    }
}

// A stream-K contributor's share: the warp's 32 rows x NCOLS fp32 accumulators
// go to its region of the slot unrounded.
template <int NCOLS>
__device__ __forceinline__ void epilogue_warp_partial(float *slot, uint32_t taddr, int region,
                                                      int lane) {
#pragma unroll 1
    for (int c = 0; c < NCOLS / 64; ++c) {
        uint32_t lo[32], hi[32];
        tmem_load_32cols(taddr + static_cast<uint32_t>(c * 64), lo);
        tmem_load_32cols(taddr + static_cast<uint32_t>(c * 64 + 32), hi);
        float4 *dst = reinterpret_cast<float4 *>(slot + region) + static_cast<size_t>(c) * 16 * 32 + lane;
#pragma unroll
        for (int v = 0; v < 16; ++v) {
            const uint32_t *s = v < 8 ? &lo[v * 4] : &hi[(v - 8) * 4];
            dst[v * 32] = make_float4(__uint_as_float(s[0]), __uint_as_float(s[1]),
                                      __uint_as_float(s[2]), __uint_as_float(s[3]));
        }
    }
}

// The residual of the fused epilogue fetched by TMA (pair kernel, RES
// instances): the warp's slab s (its s-th 32 x 64 output box) has its
// residual box loaded into staging buffer s % kResBufs, completing on that
// buffer's mbarrier, kResAhead slabs before it is needed; the output is then
// written over it in place and stored from there.  Loading a 128-byte row per
// request and one instruction per box keeps the residual off the load/store
// unit, which the accumulator reads and the staging writes also use.
// Two buffers, one slab ahead: the ring then leaves room for a sixth stage of
// the main loop, which measured 3-4 % faster (75 against 78 us at 5376 x 5376
// x 2048) than four buffers two ahead with five stages.
constexpr int kResBufs = 2;
constexpr int kResAhead = 1;
static_assert(kResAhead >= 1 && kResAhead <= 2 && kResAhead < kResBufs,
              "a buffer is free for the next request; a tile starts with one or two requests");

struct ResRing {
    const CUtensorMap *map;
    uint32_t bar0;    // this warp's kResBufs mbarriers
    uint32_t issued;  // slabs requested so far (lane 0's count)
};

// Lane 0: request slab t's residual box (columns n0.., rows row0..).  PENDING
// is the number of stores committed after the one that last read buffer
// t % kResBufs (slab t - kResBufs), so after the wait that buffer is free.  A
// box wholly outside C is not fetched: a plain arrival completes its phase
// and the lanes read stale values for outputs the store clips anyway.
template <int PENDING>
__device__ __forceinline__ void res_request(ResRing &rr, const F16Args &args, uint32_t stage_smem,
                                            uint32_t t, int n0, int row0) {
    bulk_wait_group_read<PENDING>();
    const uint32_t j = t % kResBufs;
    const uint32_t bar = rr.bar0 + 8u * j;
    if (row0 < args.M && n0 < args.N) {
        mbar_arrive_expect_tx(bar, kEpiBufBytes);
        tma_load_2d(stage_smem + j * kEpiBufBytes, rr.map, bar, n0, row0);
    } else {
        mbar_arrive(bar);
    }
    ++rr.issued;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// ACT < 0: the plain product (no epilogue code); 0..3: the fused epilogue
// with that activation (0 none, 1 ReLU, 2 SiLU, 3 tanh-GELU).  RES: the
// residual comes through the TMA ring `rr` (NBUF == kResBufs); otherwise it
// is loaded into registers.  Returns false when a residual wait ran out.
template <int NCOLS, int NBUF, int ACT, bool RES = false>
__device__ __forceinline__ bool epilogue_warp_tile(const F16Args &args, const CUtensorMap *tmC,
                                                   uint32_t taddr, int row0, int n_base, int lane,
                                                   uint32_t stage_smem, uint32_t &step,
                                                   const Partials &pp = Partials{nullptr, 0, 0, 0, 0},
                                                   ResRing *rr = nullptr,
                                                   const volatile int *abort_flag = nullptr) {
    static_assert(NCOLS % 64 == 0 && (NBUF == 1 || NBUF == 2 || NBUF == kResBufs),
                  "64-column slabs, 1, 2 or 4 buffers");
    static_assert(!RES || (ACT >= 0 && NBUF == kResBufs), "the residual ring is the fused path's");
    if (args.tma_store) {
        // Fused epilogue: the row's 8 residual words of a slab are loaded
        // together, one slab ahead (issued before the previous slab's stores
        // and this slab's accumulator reads); the slab's bias is spread over
        // lanes 0..7 and handed round by shuffles.
        uint4 res8[8];
        if constexpr (ACT >= 0 && !RES) {
#pragma unroll
            for (int q = 0; q < 8; ++q) res8[q] = epi_load_res8(args.epi, row0 + lane, n_base + 8 * q, args.M, args.N);
        }
#pragma unroll 1
        for (int c = 0; c < NCOLS / 64; ++c) {
            const int n0 = n_base + c * 64;
            const uint32_t buf = stage_smem + (step % NBUF) * kEpiBufBytes;
            const uint32_t row_addr = buf + static_cast<uint32_t>(lane) * 128u;
            uint4 bias_l = make_uint4(0u, 0u, 0u, 0u);
            if constexpr (ACT >= 0) bias_l = epi_load_bias_lane<8>(args.epi, n0, lane, args.N);
            if constexpr (RES) {
                // Keep kResAhead slabs of this tile in flight, then take this
                // slab's residual row from its buffer (chunk q of row `lane` is
                // at chunk q ^ (lane % 8): the 128-byte swizzle).
                if (lane == 0 && c + kResAhead < NCOLS / 64)
                    res_request<kResBufs - 1 - kResAhead>(*rr, args, stage_smem, step + kResAhead,
                                                          n0 + 64 * kResAhead, row0);
                // Lane 0 waits (bounded) and the verdict is the warp's; then
                // every lane observes the completed phase itself (one try_wait,
                // true at once: the phase cannot move on before this buffer is
                // requested again), which makes the TMA-written bytes visible
                // to it.
                const uint32_t rbar = rr->bar0 + 8u * (step % kResBufs);
                const uint32_t rpar = (step / kResBufs) & 1u;
                int arrived = 1;
                if (lane == 0) arrived = mbar_wait(rbar, rpar, args.timeout_ns, abort_flag) ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, arrived, 0)) return false;
                (void)mbar_try_wait(rbar, rpar);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    res8[q] = ld_shared_v4(row_addr + (static_cast<uint32_t>(q ^ (lane & 7)) << 4));
            }
            uint32_t lo[32], hi[32];
            tmem_load_32cols(taddr + static_cast<uint32_t>(c * 64), lo);
            tmem_load_32cols(taddr + static_cast<uint32_t>(c * 64 + 32), hi);
            if (pp.count || pp.dsmem) add_partial_slab(pp, c, lo, hi);
            if constexpr (ACT >= 0) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    epi_apply8<ACT>(args.epi, q < 4 ? &lo[q * 8] : &hi[(q - 4) * 8], shfl_u4(bias_l, q), res8[q]);
                if (!RES && c + 1 < NCOLS / 64) {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        res8[q] = epi_load_res8(args.epi, row0 + lane, n0 + 64 + 8 * q, args.M, args.N);
                }
            }
            // The store issued from this buffer NBUF slabs ago must have read
            // it (with the residual ring that was ensured before the residual
            // was loaded into it).
            if constexpr (!RES) {
                if (lane == 0) bulk_wait_group_read<NBUF - 1>();
                __syncwarp();
            }
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
        return true;
    } else {
        const int m = row0 + lane;
        __half *crow = args.C + static_cast<size_t>(m) * args.N;
#pragma unroll 1
        for (int c = 0; c < NCOLS / 32; ++c) {
            const int n0 = n_base + c * 32;
            uint4 res8[4], bias_l = make_uint4(0u, 0u, 0u, 0u);
            if constexpr (ACT >= 0) {
#pragma unroll
                for (int q = 0; q < 4; ++q) res8[q] = epi_load_res8(args.epi, m, n0 + 8 * q, args.M, args.N);
                bias_l = epi_load_bias_lane<4>(args.epi, n0, lane, args.N);
            }
            uint32_t r[32];
            tmem_load_32cols(taddr + static_cast<uint32_t>(c * 32), r);
            if (pp.dsmem) {
                // the partner pair's share of these 32 columns: half h of
                // 64-column slab c / 2 in epilogue_warp_share's layout
                float4 x[8];
#pragma unroll
                for (int v = 0; v < 8; ++v)
                    x[v] = ld_dsmem_f4(pp.dsmem + static_cast<uint32_t>(
                                                      (((c >> 1) * 16 + (c & 1) * 8 + v) * 32 + lane) * 16));
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    r[v * 4 + 0] = __float_as_uint(__uint_as_float(r[v * 4 + 0]) + x[v].x);
                    r[v * 4 + 1] = __float_as_uint(__uint_as_float(r[v * 4 + 1]) + x[v].y);
                    r[v * 4 + 2] = __float_as_uint(__uint_as_float(r[v * 4 + 2]) + x[v].z);
                    r[v * 4 + 3] = __float_as_uint(__uint_as_float(r[v * 4 + 3]) + x[v].w);
                }
            }
            if constexpr (ACT >= 0) {
#pragma unroll
                for (int q = 0; q < 4; ++q) epi_apply8<ACT>(args.epi, &r[q * 8], shfl_u4(bias_l, q), res8[q]);
            }
            store_row_chunk(crow, m < args.M, n_base + c * 32, args.N, args.vec_store, r);
        }
        return true;
    }
}

template <int BN, int STAGES, int ACT>
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

    // The boxes of this CTA's first ring fill are asked of L2 before the
    // set-up and the dependent-launch wait, one per lane of warp 2: the first
    // loads then find them there instead of waiting on DRAM.  A prefetch only
    // fills L2, where a previous kernel's writes land too.
    if (args.prefetch_first && warp == 2 && lane < 2 * STAGES && lane / 2 < args.num_kb &&
        static_cast<int>(blockIdx.x) < args.m_tiles * args.n_tiles) {
        int mt, nt;
        tile_mn(static_cast<int>(blockIdx.x), args, mt, nt);
        if (lane & 1)
            tma_prefetch_l2_2d(&tmB, (lane >> 1) * kBK, nt * BN);
        else
            tma_prefetch_l2_2d(&tmA, (lane >> 1) * kBK, mt * kBM);
    }

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
                int mt, nt;
                tile_mn(tile, args, mt, nt);
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
            if constexpr (ACT >= 0) {
                // The residual rows of this tile (first tile only) and of the
                // next one go to L2 while the accumulators are being made.
                const int pf = i == 0 ? tile : tile + static_cast<int>(gridDim.x);
                if (pf < total_tiles) {
                    int pm, pn;
                    tile_mn(pf, args, pm, pn);
                    epi_prefetch_res(args.epi, pm * kBM + quarter * 32 + lane, pn * BN, BN, args.M, args.N);
                }
                if (i == 0 && tile + static_cast<int>(gridDim.x) < total_tiles) {
                    const int nx = tile + static_cast<int>(gridDim.x);
                    int pm, pn;
                    tile_mn(nx, args, pm, pn);
                    epi_prefetch_res(args.epi, pm * kBM + quarter * 32 + lane, pn * BN, BN, args.M, args.N);
                }
            }
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
            int mt, nt;
            tile_mn(tile, args, mt, nt);
            epilogue_warp_tile<BN, 2, ACT>(args, &tmC, tmem_base + lane_field + static_cast<uint32_t>(b * BN),
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

// EPI_BYTES: epilogue staging; RES_BARS: mbarriers of the residual rings.
template <int STAGES, int EPI_BYTES = kEpiBytes, int RES_BARS = 0>
struct PairCfg {
    static constexpr int kBN = 256;                 // pair tile N (= MMA N)
    static constexpr int kABytes = kBM * kBK * 2;   // this CTA's 128 rows of A
    static constexpr int kBBytes = 128 * kBK * 2;   // this CTA's half of B
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kTmemCols = 512;           // two 256-column accumulators
    static constexpr int kNumBars = 2 * STAGES + 5 + RES_BARS;
    static constexpr int kEpiOffset = STAGES * kStageBytes;
    static constexpr int kBarOffset = kEpiOffset + EPI_BYTES;
    static constexpr int kSmemBytes = 1024 + kBarOffset + kNumBars * 8 + 16;
    static_assert(kSmemBytes <= 232448, "fits the 227 KB opt-in limit");
};

// RES: the fused epilogue's residual comes through per-warp TMA rings
// (kResBufs staging buffers per epilogue warp; 4 epilogue warps).
//
// CL = 4 (two pairs per cluster): the pairs of a cluster compute the two
// vertically adjacent 256 x 256 tiles (2q, n) and (2q + 1, n) of quad tile
// (q, n), which need the same 256 rows of B.  CTA r of pair p loads rows
// 64p .. 64p+63 of its 128-row half of B and multicasts them to CTA r of both
// pairs, so each B byte leaves L2 once for two tiles: a quarter fewer L2 reads
// and requests per k-block (A is not shared).  The multicast bytes are counted
// on the full barrier of each receiving pair's even CTA, which arms it for its
// pair's 64 KB as before.  A stage can be refilled only when both pairs' MMAs
// have read it, so empty[s] takes one commit from each pair's MMA issuer,
// multicast to all four CTAs.
//
// KS (with CL = 4): the two pairs of a cluster compute the same 256 x 256
// tile over the two halves of its K range instead, each pair loading its own
// A and B boxes.  Pair 1's epilogue warps write their fp32 accumulator rows
// into their own CTA's (idle) ring; pair 0's warps wait on a barrier those
// writes arrive on, add them through distributed shared memory, and store.
// One tile per cluster: the ring holds the share, so no next tile may load.
template <int STAGES, int EPI, int ACT, bool RES, int CL = 2, bool KS = false>
__global__ void __launch_bounds__((2 + EPI) * 32, 1)
    gemm_f16_nt_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmC,
                            const __grid_constant__ CUtensorMap tmR, const F16Args args) {
    static_assert(!RES || EPI == 4, "residual rings are laid out for 4 epilogue warps");
    static_assert(CL == 2 || CL == 4, "a CTA pair, or two pairs sharing B");
    static_assert(!KS || CL == 4, "the K split puts two pairs in one cluster");
    constexpr int kBufs = RES ? kResBufs : 8 / EPI;
    constexpr int kResBars = RES ? EPI * kResBufs : 0;
    using T = PairCfg<STAGES, EPI * kBufs * kEpiBufBytes, kResBars + (KS ? EPI : 0)>;
    static_assert(!KS || STAGES * T::kStageBytes >= 256 * 128 * 4, "the ring holds a CTA's share");
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
    const uint32_t res_bar0 = bar0 + 8u * (2 * STAGES + 5);  // RES: kResBufs per epilogue warp
    // KS: per epilogue warp of pair 0, the partner warp's share is in place
    auto xready_bar = [&](int w) { return bar0 + 8u * (2 * STAGES + 5 + kResBars + w); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + T::kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    __shared__ int never_abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();
    const uint32_t rank = crank & 1u;          // 0 (leader) or 1 within the pair
    const uint32_t pic = crank >> 1;           // which pair of the cluster (CL = 4)
    const uint32_t lead = crank & ~1u;         // this pair's even CTA
    const bool leader = rank == 0;
    // the persistent work unit: a pair (CL = 2) or a two-pair cluster (CL = 4)
    const int pair = static_cast<int>(blockIdx.x) / CL;
    const int num_pairs = static_cast<int>(gridDim.x) / CL;
    // tile row of this pair for work-list tile row mt (quad rows hold two)
    auto pair_row = [&](int mt) { return CL == 2 || KS ? mt : 2 * mt + static_cast<int>(pic); };
    // KS: this pair's half of a tile's k-blocks [kb0, kb1)
    auto k_half = [&](int &kb0, int &kb1) {
        if constexpr (KS) {
            const int h = (kb1 - kb0 + 1) / 2;
            if (pic) kb0 += h; else kb1 = kb0 + h;
        }
    };
    // A producer work item: k-blocks [kb0, kb1) and the rows of this CTA's A
    // and B boxes.
    struct LoadItem {
        int kb0, kb1, a_row, b_row;
    };
    auto next_load_item = [&](PairWork &w, LoadItem &it) {
        int tile;
        if (!w.next(tile, it.kb0, it.kb1)) return false;
        k_half(it.kb0, it.kb1);
        int mt, nt;
        tile_mn(tile, args, mt, nt);
        mt = pair_row(mt);
        it.a_row = mt * 256 + static_cast<int>(rank) * 128;
        it.b_row = nt * BN + static_cast<int>(rank) * 128 + (CL == 4 && !KS ? 64 * static_cast<int>(pic) : 0);
        return true;
    };
    // While other warps set up: the producer finds its first item, and the
    // boxes of this CTA's first ring fill are asked of L2, one per lane of
    // warp 3, so that the first loads find them there instead of waiting on
    // DRAM (-1.1 us per launch at 5376 x 5376 x 2048).  Both precede the
    // dependent-launch wait: a prefetch only fills L2, which is where a
    // previous kernel's writes land too, so it cannot make a later load see
    // stale data.
    PairWork load_work(args, pair, num_pairs);
    LoadItem load_item{0, 0, 0, 0};
    bool load_more = threadIdx.x == 0 && next_load_item(load_work, load_item);
    if (args.prefetch_first && warp == 3 && lane < 2 * STAGES) {
        PairWork w(args, pair, num_pairs);
        LoadItem it;
        if (next_load_item(w, it) && it.kb0 + (lane >> 1) < it.kb1) {
            const int kb = it.kb0 + (lane >> 1);
            if (lane & 1)
                tma_prefetch_l2_2d(&tmB, kb * kBK, it.b_row);
            else
                tma_prefetch_l2_2d(&tmA, kb * kBK, it.a_row);
        }
    }

    if (threadIdx.x == 64) {  // (thread 0, the producer, is busy with its first item)
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (args.tma_store) tma_prefetch_desc(&tmC);
        if (RES) tma_prefetch_desc(&tmR);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), KS ? 1 : CL / 2);  // one MMA commit per pair reading the stage
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 2 * EPI);  // every epilogue warp of both CTAs
        }
        if (RES)
            for (int j = 0; j < EPI * kResBufs; ++j) mbar_init(res_bar0 + 8u * j, 1);
        if (KS)
            for (int w = 0; w < EPI; ++w) mbar_init(xready_bar(w), 32);  // every lane of the partner warp
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        never_abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(tmem_slot), T::kTmemCols);
        tmem_relinquish_alloc_permit_pair();
    }
    // This CTA's TMEM address and flags, then both CTAs' barriers initialised
    // (released by fence.mbarrier_init) and TMEM allocated in both.
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_relaxed();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    pdl_launch_dependents();
    pdl_wait_prerequisites();

    uint32_t armed = 0, arm_parity = 0;

    if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            bool first_tile = true;
            int filled = 0;  // every slot starts free: the first STAGES loads need no wait
            while (ok && load_more) {
                const int a_row = load_item.a_row, b_row = load_item.b_row;
                for (int kb = load_item.kb0; kb < load_item.kb1; ++kb) {
                    if (filled < STAGES) {
                        ++filled;
                    } else if (!mbar_wait_cluster(empty_bar(stage), phase ^ 1u, args.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const bool skip = first_tile && kb == args.debug_skip_kblock && leader;
                    if (!skip) {
                        const uint32_t sa = sbase + stage * T::kStageBytes;
                        const uint32_t full_leader = mapa_shared(full_bar(stage), lead);
                        if (leader) {
                            mbar_arrive_expect_tx(full_bar(stage), 2 * T::kStageBytes);
                            armed |= 1u << stage;
                            arm_parity ^= 1u << stage;
                        }
                        tma_load_2d_pair(sa, &tmA, full_leader, kb * kBK, a_row);
                        if constexpr (CL == 2 || KS) {
                            tma_load_2d_pair(sa + T::kABytes, &tmB, full_leader, kb * kBK, b_row);
                        } else {
                            // rows 64 pic .. of this CTA's B half, to CTA `rank` of both pairs
                            tma_load_2d_pair_multicast(sa + T::kABytes + pic * (T::kBBytes / 2), &tmB,
                                                       full_leader, kb * kBK, b_row,
                                                       static_cast<uint16_t>(0x5u << rank));
                        }
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                first_tile = false;
                load_more = next_load_item(load_work, load_item);
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
            PairWork work(args, pair, num_pairs);
            int tile, kb0, kb1;
            for (int i = 0; work.next(tile, kb0, kb1); ++i) {
                k_half(kb0, kb1);
                const int b = i & 1;
                const uint32_t ap = (i >> 1) & 1;
                if (!mbar_wait_cluster(acce_bar(b), ap ^ 1u, args.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
                for (int kb = kb0; kb < kb1; ++kb) {
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
                                        (kb > kb0 || k > 0) ? 1u : 0u);
                    // the stage is free once every pair reading it is done: this
                    // pair, or (B shared) both pairs of the cluster
                    mma_commit_pair_multicast(empty_bar(stage),
                                              KS ? static_cast<uint16_t>(0x3u << lead) : (CL == 2 ? 0x3 : 0xF));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_pair_multicast(accf_bar(b), static_cast<uint16_t>(0x3u << lead));
            }
            if (!ok) {
                if (!*abort_flag) record_timeout(2);
                *abort_flag = 1;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        // EPI warps share the tile: warp w reads TMEM lane quarter w % 4 and,
        // with 8 warps, one half of the columns.
        constexpr int kCols = BN * 4 / EPI;
        const int ew = warp - 2;
        const int quarter = warp & 3;
        const int col0 = (ew / 4) * kCols;
        const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t stage_smem = sbase + T::kEpiOffset + ew * kBufs * kEpiBufBytes;
        uint32_t step = 0;
        ResRing rr{&tmR, res_bar0 + 8u * kResBufs * ew, 0};
        PairWork work(args, pair, num_pairs);
        int tile, kb0, kb1;
        for (int i = 0; work.next(tile, kb0, kb1); ++i) {
            const int b = i & 1;
            const uint32_t ap = (i >> 1) & 1;
            int tm, tn;
            tile_mn(tile, args, tm, tn);
            tm = pair_row(tm);
            const int row0 = tm * 256 + static_cast<int>(rank) * 128 + quarter * 32;
            const int n_base = tn * BN + col0;
            if constexpr (RES) {
                // The tile's first kResAhead residual boxes load while its
                // accumulators are being made (stores of earlier slabs pending:
                // see res_request).
                if (lane == 0 && kb0 == 0) {
                    res_request<kResBufs - 1>(rr, args, stage_smem, step, n_base, row0);
                    if constexpr (kResAhead >= 2)
                        res_request<kResBufs - 2>(rr, args, stage_smem, step + 1, n_base + 64, row0);
                }
            }
            if constexpr (ACT >= 0) {
                // The residual rows of this tile (first tile only) and of the
                // next one go to L2 while the accumulators are being made.
                auto prefetch = [&](int t) {
                    int pm, pn;
                    tile_mn(t, args, pm, pn);
                    pm = pair_row(pm);
                    epi_prefetch_res(args.epi, pm * 256 + static_cast<int>(rank) * 128 + quarter * 32 + lane,
                                     pn * BN + col0, kCols, args.M, args.N);
                };
                if (i == 0 && kb0 == 0) prefetch(tile);
                PairWork peek = work;
                int t2, k0, k1;
                if (peek.next(t2, k0, k1) && k0 == 0) prefetch(t2);
            }
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
            const uint32_t taddr = tmem_base + lane_field + static_cast<uint32_t>(b * BN + col0);
            const int region = ew * kCols * 32;    // this warp's part of a partial slot
            if (KS && pic == 1) {
                // K-split partner: this warp's rows of the accumulator into
                // its own ring (idle: the pair's k-blocks are all consumed),
                // then every lane arrives, with cluster-scope release, on the
                // barrier of pair 0's matching warp (CTA `rank` of the cluster).
                epilogue_warp_share<kCols>(sbase + static_cast<uint32_t>(region) * 4u, taddr, lane);
                mbar_arrive_cluster(mapa_shared(xready_bar(ew), rank));
            } else if (kb0 > 0) {
                // Stream-K contributor: this warp publishes its rows of the
                // unrounded partial, then its own flag (no barrier between warps).
                float *slot = args.sk_ws + static_cast<size_t>(pair * 2 + rank) * kSkSlotFloatsDev;
                epilogue_warp_partial<kCols>(slot, taddr, region, lane);
                __threadfence();
                __syncwarp();
                if (lane == 0 && !args.debug_skip_publish)
                    st_release_gpu(args.sk_flags + (pair * 2 + rank) * 8 + ew, args.seq);
            } else {
                Partials pp{args.sk_ws, 0, 0, region, lane};
                if constexpr (KS) {
                    // K-split owner: wait (bounded) for the partner warp's
                    // share, then every lane acquires it before reading it
                    // through distributed shared memory.
                    const uint32_t xp = static_cast<uint32_t>(i & 1);
                    int got = 1;
                    if (lane == 0) got = mbar_wait_cluster(xready_bar(ew), xp, args.timeout_ns, abort_flag) ? 1 : 0;
                    got = __shfl_sync(0xffffffffu, got, 0);
                    if (!got) {
                        if (lane == 0) {
                            if (!*abort_flag) record_timeout(3);
                            *abort_flag = 1;
                        }
                        break;
                    }
                    (void)mbar_try_wait_cluster(xready_bar(ew), xp);
                    pp.dsmem = mapa_shared(sbase + static_cast<uint32_t>(region) * 4u, crank + 2u);
                }
                if (kb1 < args.num_kb) {
                    // Owner of a split tile: the following share ranks (pairs
                    // pair-1, pair-2, ...), whose shares begin inside this tile,
                    // hold its remaining k-blocks; every share is non-empty, so
                    // they are consecutive.  This warp waits for the flag of the
                    // warp that wrote the same rows and columns.
                    const int tile_end = (tile - args.dp_tiles + 1) * args.num_kb;
                    const int my_rank = num_pairs - 1 - pair;
                    pp.first_slot = (pair - 1) * 2 + static_cast<int>(rank);
                    while (my_rank + 1 + pp.count < num_pairs &&
                           work.sk_begin(my_rank + 1 + pp.count) < tile_end)
                        ++pp.count;
                    int fine = 1;
                    if (lane == 0)
                        for (int q = 0; q < pp.count && fine; ++q)
                            fine = wait_flag_equal(args.sk_flags + (pp.first_slot - 2 * q) * 8 + ew,
                                                   args.seq, args.timeout_ns, abort_flag) ? 1 : 0;
                    fine = __shfl_sync(0xffffffffu, fine, 0);
                    if (!fine) {
                        if (lane == 0) {
                            if (!*abort_flag) record_timeout(4);
                            *abort_flag = 1;
                        }
                        break;
                    }
                }
                const bool fine = epilogue_warp_tile<kCols, kBufs, ACT, RES>(
                    args, &tmC, taddr, row0, n_base, lane, stage_smem, step, pp, &rr, abort_flag);
                if (!fine) {
                    if (lane == 0) {
                        if (!*abort_flag) record_timeout(3);
                        *abort_flag = 1;
                    }
                    break;
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            // The MMA issuer waits for this buffer only before a later tile:
            // after the last one nothing is sent, so no arrival on the even
            // CTA can still be in flight when the pair leaves.
            PairWork more = work;
            int t2, k0, k1;
            if (lane == 0 && more.next(t2, k0, k1)) mbar_arrive_cluster(mapa_shared(acce_bar(b), lead));
        }
        if constexpr (RES) {
            // Residual loads still in flight (only after an abort) land before
            // this CTA's shared memory is released.
            if (lane == 0)
                for (uint32_t t = step; t < rr.issued; ++t)
                    (void)mbar_wait(rr.bar0 + 8u * (t % kResBufs), (t / kResBufs) & 1u, args.timeout_ns,
                                    &never_abort);
        }
        if (lane == 0) bulk_wait_group_all();
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    const bool aborted = *abort_flag != 0;
    if (aborted) {
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
    // (remote arrivals, pair TMA completions, pair MMA operand reads).  On the
    // normal path every such operation has completed on an mbarrier the other
    // CTA waited on (the last tile sends no drained-accumulator arrival; the
    // K-split partner's share was acquired and read), so the barrier only
    // orders execution.  After an abort an arrival may still be in flight, and
    // the releasing form orders it first.
    if (aborted)
        cluster_sync();
    else
        cluster_sync_relaxed();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, T::kTmemCols);
    }
}

// K == 0: the product is the empty sum; C = 0, or the fused epilogue of 0.
__global__ void zero_half_kernel(__half *C, int M, int N, Epi epi) {
    const size_t count = static_cast<size_t>(M) * N;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < count; i += stride) {
        const int n = static_cast<int>(i % N);
        float v = 0.f;
        if (epi.on) {
            const float b = epi.bias ? __half2float(epi.bias[n]) : 0.f;
            const float r = epi.reads_res() ? __half2float(epi.res[i]) : 0.f;
            v = epi_apply1(epi, 0.f, b, r);
        }
        C[i] = __float2half_rn(v);
    }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch
// ---------------------------------------------------------------------------

}  // namespace

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

// (declared in gemm_internal.h, shared with the other translation units)
bool encode_map(CUtensorMap *map, CUtensorMapDataType dtype, int elem_bytes, const void *ptr, int rows,
                int cols, int box_rows, int box_cols, std::string &err, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn enc = get_encode_fn(err);
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * elem_bytes};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    // No L2 promotion: the operands are L2-resident after their first use and
    // wider L2 fetches measured slower on this path.
    CUresult r = enc(map, dtype, 2, const_cast<void *>(ptr), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle, CU_TENSOR_MAP_L2_PROMOTION_NONE,
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

namespace {

bool encode_half_map(CUtensorMap *map, const void *ptr, int rows, int cols, int box_rows,
                     int box_cols, std::string &err) {
    return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, ptr, rows, cols, box_rows, box_cols, err);
}

template <int BN, int STAGES, int ACT>
int launch_variant(const F16Launch &L, std::string &err) {
    using T = TileCfg<BN, STAGES>;
    auto kernel = gemm_f16_nt_tc_kernel<BN, STAGES, ACT>;
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
    args.raster = L.raster > 0 ? L.raster : (1 << 30);
    args.n_tiles = (L.N + BN - 1) / BN;
    args.num_kb = (L.K + kBK - 1) / kBK;
    args.prefetch_first = (static_cast<size_t>(L.M) + L.N) * L.K * 2 >= kPrefetchMinBytes;
    args.vec_store = (L.N % 8 == 0) && ((reinterpret_cast<uintptr_t>(L.C) & 15u) == 0);
    args.tma_store = args.vec_store;
    args.epi = make_epi(L.epi, L.N);
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

// Stream-K workspace of one (device, stream): partial-tile slots and flags,
// allocated on first use and kept for the life of the process.  Calls on one
// stream run in order (the kernel touches global memory only after the
// previous grid has finished), so a stream never has two users of its slots.
struct SkWorkspace {
    float *ws = nullptr;
    uint32_t *flags = nullptr;
    int pairs = 0;
    uint32_t seq = 0;
};

constexpr size_t kSkSlotFloats = 128 * 256;  // one CTA's half of a 256 x 256 tile

int sk_workspace(cudaStream_t stream, int pairs, SkWorkspace **out, std::string &err) {
    static std::mutex mu;
    static std::map<std::pair<int, cudaStream_t>, SkWorkspace> cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        err = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(mu);
    SkWorkspace &w = cache[std::make_pair(dev, stream)];
    if (w.pairs < pairs) {
        if (w.ws) cudaFree(w.ws);
        if (w.flags) cudaFree(w.flags);
        w = SkWorkspace{};
        e = cudaMalloc(&w.ws, static_cast<size_t>(pairs) * 2 * kSkSlotFloats * sizeof(float));
        if (e == cudaSuccess)
            e = cudaMalloc(&w.flags, static_cast<size_t>(pairs) * 2 * 8 * sizeof(uint32_t));
        if (e != cudaSuccess) {
            err = std::string("stream-K workspace allocation: ") + cudaGetErrorString(e);
            w = SkWorkspace{};
            return GEMM_ERR_CUDA;
        }
        w.pairs = pairs;
    }
    if (++w.seq == 0 || w.seq == 1) {
        // first use, or the sequence number wrapped: no flag may hold a live value
        e = cudaMemsetAsync(w.flags, 0, static_cast<size_t>(w.pairs) * 2 * 8 * sizeof(uint32_t),
                            stream);
        if (e != cudaSuccess) {
            err = std::string("stream-K flag reset: ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
        w.seq = 1;
    }
    *out = &w;
    return GEMM_OK;
}

// Scratch of gemm_f16_nt_stream_k_noalloc: the same partial slots and flags as
// a stream-K workspace, in module memory instead of a cudaMalloc'd buffer, for
// up to kNoAllocMaxPairs CTA pairs (76 pairs = one GB300's 152 SMs).  Every
// GPU that loads the library holds it until the process exits.  It starts out
// zero (module memory is zero-initialised); each call tags its flags with a
// fresh per-device sequence number, so stale slots and flags from earlier
// calls are never mistaken for this call's, and only a wrap of that counter
// needs the flags cleared.  All calls on a device share it: calls whose
// kernels overlap on the GPU (on different streams) race on it.
constexpr int kNoAllocMaxPairs = 76;
constexpr size_t kNoAllocSlotBytes =
    static_cast<size_t>(kNoAllocMaxPairs) * 2 * kSkSlotFloats * sizeof(float);
constexpr size_t kNoAllocFlagBytes = static_cast<size_t>(kNoAllocMaxPairs) * 2 * 8 * sizeof(uint32_t);
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocSlotBytes + kNoAllocFlagBytes];

// Device address of the scratch array for the current device, looked up once
// per device with that device current (in host code the symbol itself is only
// a host-side stand-in).  Also advances and returns that device's sequence number.
// The address stays valid for the life of the CUDA context it was looked up
// in (a cudaDeviceReset ends that context, and the library must not be used
// on that device afterwards).
int noalloc_scratch(cudaStream_t stream, float **ws, uint32_t **flags, uint32_t *seq,
                    std::string &err) {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static void *addr[kMaxDevices] = {nullptr};
    static uint32_t counter[kMaxDevices] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        err = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        char buf[160];
        std::snprintf(buf, sizeof buf,
                      "gemm_f16_nt_stream_k_noalloc: device %d is beyond the %d devices it keeps "
                      "scratch addresses for", dev, kMaxDevices);
        err = buf;
        return GEMM_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            err = std::string("cudaGetSymbolAddress(stream-K scratch): ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
        addr[dev] = p;
    }
    uint32_t *f = reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(addr[dev]) + kNoAllocSlotBytes);
    if (++counter[dev] == 0) {
        e = cudaMemsetAsync(f, 0, kNoAllocFlagBytes, stream);  // the counter wrapped
        if (e != cudaSuccess) {
            err = std::string("stream-K scratch flag reset: ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
        counter[dev] = 1;
    }
    *ws = static_cast<float *>(addr[dev]);
    *flags = f;
    *seq = counter[dev];
    return GEMM_OK;
}

thread_local PairLaunchRecord t_last_pair;

// CL = 2: one CTA pair per 256 x 256 tile; CL = 4: two pairs per cluster
// sharing B (vertically adjacent tiles), no split; CL = 4 with KS: two pairs
// per cluster splitting one tile's K range, one tile per cluster.
template <int STAGES, int EPI, int ACT, bool RES, int CL = 2, bool KS = false>
int launch_pair(const F16Launch &L, std::string &err) {
    constexpr int kBufs = RES ? kResBufs : 8 / EPI;
    using T = PairCfg<STAGES, EPI * kBufs * kEpiBufBytes, (RES ? EPI * kResBufs : 0) + (KS ? EPI : 0)>;
    auto kernel = gemm_f16_nt_pair_kernel<STAGES, EPI, ACT, RES, CL, KS>;
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
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3((2 + EPI) * 32);
    cfg.dynamicSmemBytes = T::kSmemBytes;
    cfg.stream = L.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = cached ? max_clusters[dev] : 0;
    if (!cached) {
        // How many clusters can be resident at once: the persistent grid size.
        cfg.gridDim = dim3(CL);
        e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
        if (e != cudaSuccess || clusters <= 0) {
            err = std::string("cudaOccupancyMaxActiveClusters: ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
        if (dev >= 0 && dev < 64) max_clusters[dev] = clusters;
    }
    CUtensorMap tmA, tmB;
    if (!encode_half_map(&tmA, L.A, L.M, L.K, kBM, kBK, err)) return GEMM_ERR_CUDA;
    // (two pairs sharing B each load 64 of a CTA's 128 rows of it)
    if (!encode_half_map(&tmB, L.B, L.N, L.K, CL == 2 || KS ? 128 : 64, kBK, err)) return GEMM_ERR_CUDA;

    F16Args args;
    args.C = static_cast<__half *>(L.C);
    args.M = L.M;
    args.N = L.N;
    args.K = L.K;
    // work-list tile rows: 256 output rows per pair (or per K-split cluster),
    // 512 per two-pair cluster sharing B
    constexpr int kRowsPerUnit = CL == 2 || KS ? 256 : 512;
    args.m_tiles = (L.M + kRowsPerUnit - 1) / kRowsPerUnit;
    args.raster = L.raster > 0 ? (kRowsPerUnit == 256 ? L.raster : (L.raster + 1) / 2) : (1 << 30);
    args.n_tiles = (L.N + 255) / 256;
    args.num_kb = (L.K + kBK - 1) / kBK;
    args.prefetch_first = (static_cast<size_t>(L.M) + L.N) * L.K * 2 >= kPrefetchMinBytes;
    args.vec_store = (L.N % 8 == 0) && ((reinterpret_cast<uintptr_t>(L.C) & 15u) == 0);
    args.tma_store = args.vec_store;
    args.epi = make_epi(L.epi, L.N);
    args.timeout_ns = L.timeout_ns;
    args.debug_skip_kblock = L.debug_skip_kblock;
    args.debug_skip_publish = L.debug_skip_publish ? 1 : 0;
    CUtensorMap tmC, tmR;
    std::memset(&tmC, 0, sizeof tmC);
    std::memset(&tmR, 0, sizeof tmR);
    if (args.tma_store && !encode_half_map(&tmC, L.C, L.M, L.N, 32, 64, err)) return GEMM_ERR_CUDA;
    if (RES && !encode_half_map(&tmR, L.epi.res, L.M, L.N, 32, 64, err)) return GEMM_ERR_CUDA;
    const int tiles = args.m_tiles * args.n_tiles;
    // `pairs` counts the persistent clusters (CTA pairs, or two-pair clusters)
    int pairs = L.grid / CL;
    if (pairs < 1) pairs = 1;
    if (pairs > clusters) pairs = clusters;
    // The allocation-free entry point's static array has partial slots for
    // kNoAllocMaxPairs pairs: a larger device runs that many persistent pairs.
    if (L.static_scratch && pairs > kNoAllocMaxPairs) pairs = kNoAllocMaxPairs;
    // K split: one tile per cluster, since the partner pair's share occupies
    // its ring.  No cluster waits on another, so clusters beyond those that
    // fit at once simply start later.
    if (KS) pairs = tiles;

    // The k-blocks of some tiles shared out over several pairs (stream-K),
    // whose fp32 partials the pair holding k-block 0 adds before rounding:
    //  * split-K, by default, when the tiles would leave most pairs idle (fewer
    //    than half as many tiles as pairs, enough k-blocks per share): every
    //    tile is split, over at most kMaxSplit pairs;
    //  * on request (GEMM_F16_FLAG_STREAM_K), the last partial round of tiles
    //    when it would leave many pairs idle.
    // Both need the TMA store epilogue and a stream that is not being captured
    // (a replayed graph would reuse the sequence number baked into its
    // arguments); otherwise every tile is whole.
    args.dp_tiles = tiles;
    args.sk_units = 0;
    args.sk_ws = nullptr;
    args.sk_flags = nullptr;
    args.seq = 0;
    const int split_pairs = CL == 2 && args.tma_store ? pair_split_pairs(tiles, args.num_kb, pairs) : 0;
    int rem = 0;  // tiles of the shared round
    if (split_pairs > 0) {
        rem = tiles;
    } else {
        if (pairs > tiles) pairs = tiles;
        const int r = tiles % pairs;
        if (CL == 2 && L.allow_stream_k && args.tma_store && tiles > pairs && r != 0 &&
            10 * r < 9 * pairs && static_cast<long long>(r) * args.num_kb >= pairs)
            rem = r;
    }
    if (rem > 0) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        e = cudaStreamIsCapturing(L.stream, &cap);
        if (e != cudaSuccess) {
            err = std::string("cudaStreamIsCapturing: ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
        if (split_pairs > 0) pairs = cap == cudaStreamCaptureStatusNone ? split_pairs : (pairs < tiles ? pairs : tiles);
        if (cap == cudaStreamCaptureStatusNone && !L.static_scratch) {
            SkWorkspace *w = nullptr;
            const int st = sk_workspace(L.stream, pairs, &w, err);
            if (st != GEMM_OK) return st;
            args.dp_tiles = tiles - rem;
            args.sk_units = rem * args.num_kb;
            args.sk_ws = w->ws;
            args.sk_flags = w->flags;
            args.seq = w->seq;
        } else if (cap == cudaStreamCaptureStatusNone) {
            float *ws = nullptr;
            uint32_t *flags = nullptr;
            uint32_t seq = 0;
            const int st = noalloc_scratch(L.stream, &ws, &flags, &seq, err);
            if (st != GEMM_OK) return st;
            args.dp_tiles = tiles - rem;
            args.sk_units = rem * args.num_kb;
            args.sk_ws = ws;
            args.sk_flags = flags;
            args.seq = seq;
        }
    }
    cfg.gridDim = dim3(CL * pairs);
    cfg.numAttrs = 2;  // cluster shape + programmatic dependent launch
    e = cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, tmC, tmR, args);
    if (e != cudaSuccess) {
        err = std::string("gemm_f16_nt pair kernel launch: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    t_last_pair.valid = true;
    t_last_pair.pairs = pairs * (CL / 2);
    t_last_pair.whole_tiles = args.dp_tiles;
    t_last_pair.shared_units = args.sk_units;
    t_last_pair.scratch_kind = args.sk_units == 0 ? 0 : (L.static_scratch ? 2 : 1);
    return GEMM_OK;
}

// One kernel per epilogue: the plain product, or the fused epilogue with
// each activation.
template <int BN, int STAGES>
int launch_variant_epi(const F16Launch &L, std::string &err) {
    switch (L.epi.on ? L.epi.act : -1) {
        case 0: return launch_variant<BN, STAGES, 0>(L, err);
        case 1: return launch_variant<BN, STAGES, 1>(L, err);
        case 2: return launch_variant<BN, STAGES, 2>(L, err);
        case 3: return launch_variant<BN, STAGES, 3>(L, err);
        default: return launch_variant<BN, STAGES, -1>(L, err);
    }
}

// Pair kernels: 6-stage ring for the plain product and for epilogues without
// a residual; with a residual that TMA can fetch (16-byte aligned, N % 8 == 0,
// TMA-store epilogue) a 5-stage ring, whose 32 KB go to the residual rings.
template <bool RES>
int launch_pair_act(const F16Launch &L, std::string &err) {
    constexpr int S = 6;
    switch (L.epi.on ? L.epi.act : -1) {
        case 0: return launch_pair<S, 4, 0, RES>(L, err);
        case 1: return launch_pair<S, 4, 1, RES>(L, err);
        case 2: return launch_pair<S, 4, 2, RES>(L, err);
        case 3: return launch_pair<S, 4, 3, RES>(L, err);
        default: return launch_pair<6, 4, -1, false>(L, err);
    }
}

int launch_pair_epi(const F16Launch &L, std::string &err) {
    const bool res_tma = L.epi.on && L.epi.res != nullptr && L.epi.beta != 0.f && L.N % 8 == 0 &&
                         ((reinterpret_cast<uintptr_t>(L.C) | reinterpret_cast<uintptr_t>(L.epi.res)) & 15u) == 0;
    return res_tma ? launch_pair_act<true>(L, err) : launch_pair_act<false>(L, err);
}

}  // namespace

}  // namespace gb300

#include "gemm_blockscaled.cuh"

namespace gb300 {

int f16_launch(const F16Launch &L, std::string &err) {
    if (L.K == 0) {
        const size_t count = static_cast<size_t>(L.M) * L.N;
        const int blocks = static_cast<int>((count + 255) / 256 < 4096 ? (count + 255) / 256 : 4096);
        zero_half_kernel<<<blocks, 256, 0, L.stream>>>(static_cast<__half *>(L.C), L.M, L.N,
                                                        make_epi(L.epi, L.N));
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) {
            err = std::string("zero fill launch: ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
        return GEMM_OK;
    }
    switch (L.variant) {
        case GEMM_F16_128x256: return launch_variant_epi<256, 4>(L, err);
        case GEMM_F16_128x128: return launch_variant_epi<128, 6>(L, err);
        case GEMM_F16_256x256_PAIR: return launch_pair_epi(L, err);
        // two pairs sharing B: the plain product (a fused epilogue runs on the pair variant)
        case GEMM_F16_256x256_QUAD: return L.epi.on ? launch_pair_epi(L, err) : launch_pair<6, 4, -1, false, 4>(L, err);
        // two pairs splitting one tile's K: the plain product over at least two k-blocks
        case GEMM_F16_256x256_KSPLIT:
            return L.epi.on || L.K <= kBK ? launch_pair_epi(L, err) : launch_pair<6, 4, -1, false, 4, true>(L, err);
        case GEMM_F16_GEMV: {
            GemvLaunch G{L.M, L.N, L.K, L.A, L.B, L.C, L.stream, L.sm_count, 4, L.epi};
            return gemv_launch(G, err);
        }
        case GEMM_F16_SKINNY: {
            // the grid is the CTA count the K split aims for
            SkinnyLaunch S{L.M, L.N, L.K, L.A, L.B, L.C, L.stream,
                           L.grid > 0 ? L.grid : L.sm_count * skinny_ctas_per_sm(), L.timeout_ns, L.epi,
                           L.debug_skip_kblock};
            return skinny_launch(S, err);
        }
        default: err = "unknown fp16 variant"; return GEMM_ERR_INVALID_ARG;
    }
}

PairLaunchRecord last_pair_launch() { return t_last_pair; }

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
