// gemm_skinny.cu -- C = A * B^T on the tensor cores as the swapped product
// D = B * A^T (D = C^T), for a few rows of A or for too few tiles to fill
// the SMs without splitting K.
//
// Same operation and numerics as gemm_f16_nt (half inputs, fp32
// accumulation, one round-to-nearest-even per output).  With M this small, B
// is read once and the work is bound by HBM.  The tile kernels' 128-row tiles
// of A would leave 120 of the MMA's 128 rows empty and give one tile per
// 128 columns of C: at N = 8192, 64 CTAs for 152 SMs.  Here B's rows take the
// MMA's M = 128 and A's rows its N (16, 32, 64 or 128, the rows past M zero-filled
// by TMA), so a tile is 128 columns of C by all of its rows (by 128 of them
// per tile on the grid's third dimension when M > 128), and the K range is
// split over enough CTAs to fill the SMs ("第 6 章 · Shared Memory & Tile",
// section "6.5.6 Split-K / Stream-K").
//
// Per CTA: warp 0 issues TMA loads of B's 128 x 64 box and A's MN x 64 box
// per k-block into a ring of STAGES stages (128-byte swizzle), warp 1 issues
// the k-blocks' tcgen05.mma (M = 128, N = MN, K = 16) into one TMEM
// accumulator, warps 2-5 read it back: TMEM lane n holds D[n][0..MN), so lane
// n stores C[m][n] for every m, 32 consecutive columns of C per warp and row.
// With a split, the CTAs that share a tile's K range form one thread-block
// cluster (2, 4 or 8 CTAs): each puts its fp32 share in its own shared
// memory, and after a cluster barrier CTA r adds slice r of the tile over all
// the shares, read through distributed shared memory in split order
// ("异步拷贝与 Hopper/Blackwell 新特性", section "线程块集群与分布式共享内存
// sm_90+": CTAs of a cluster synchronise and read one another's shared
// memory), so results do not depend on timing and no share goes through HBM.
// When even 8-CTA clusters leave most SMs idle (a few tiles over a very long
// K), each tile's K range goes to several clusters ("parts"): every cluster
// sums its own shares as above and writes that fp32 partial to a workspace,
// and the cluster that finishes the tile last (a per-slice counter tagged
// with the launch's sequence number, so nothing is reset between launches)
// adds the parts in order and stores.  Nothing waits on another cluster.
// Every wait is bounded as in the other kernels.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <map>
#include <mutex>
#include <utility>

#include "gemm.h"
#include "epilogue.cuh"
#include "gemm_internal.h"
#include "sm103_ptx.cuh"

namespace gb300 {
namespace {

__device__ int g_skinny_status = 0;
__device__ __forceinline__ void skinny_timeout(int code) { atomicCAS(&g_skinny_status, 0, code); }

constexpr int kSkBM = 128;       // the MMA's M: at most this many rows of B per group
constexpr int kSkBK = 64;        // halves per k-block: one 128-byte swizzle row
constexpr int kSkThreads = 192;  // warp 0 producer, warp 1 MMA, warps 2-5 epilogue
constexpr int kSkCtasPerSm = 1;  // CTAs resident per SM (their stages keep HBM busy)

template <int MN, int STAGES>
struct SkCfg {
    static constexpr int kBBytes = kSkBM * kSkBK * 2;  // 16 KB: 128 rows of B
    static constexpr int kABytes = MN * kSkBK * 2;     // MN rows of A (zero past M)
    static constexpr int kStageBytes = kBBytes + kABytes;
    static constexpr int kTmemCols = MN < 32 ? 32 : MN;
    static constexpr int kNumBars = 2 * STAGES + 2;    // full, empty, accumulator ready, drain
    static constexpr int kBarOffset = STAGES * kStageBytes;
    static constexpr int kSmemBytes = 1024 + kBarOffset + kNumBars * 8 + 16;  // + TMEM slot and flags
    static_assert(MN == 16 || MN == 32 || MN == 64 || MN == 128, "an MMA N for M = 128");
    static_assert(kABytes % 1024 == 0, "stages keep the 1 KB alignment of the swizzled boxes");
    static_assert(kSmemBytes <= 232448, "fits the 227 KB opt-in limit");
};

// Ring stages that let kSkCtasPerSm CTAs share an SM's 228 KB (1 KB of it
// reserved per CTA), at most 8.
template <int MN>
constexpr int sk_stages() {
    constexpr int stage = kSkBM * kSkBK * 2 + MN * kSkBK * 2;
    constexpr int per_cta = 233472 / kSkCtasPerSm - 1024 - 1024 - 256;  // reserve, alignment, barriers
    return per_cta / stage > 8 ? 8 : per_cta / stage;
}

struct SkArgs {
    __half *C;
    int M, N, K;
    int num_kb;        // 64-deep k-blocks of K
    int kb_per_split;  // k-blocks per share (the last may be shorter)
    int splits;        // shares of K per group: 1, or the cluster size (2, 4, 8)
    int rows;          // rows of B (columns of C) per group: a multiple of 8, <= 128
    uint64_t timeout_ns;
    Epi epi;           // fused epilogue, applied where the fp32 sum is rounded
    int debug_skip_kblock;  // test hook: every CTA leaves out this k-block of its share (-1: none)
    // Clusters per tile (1: none): cluster p of a tile writes slice r of its
    // sum to ws[((tile * splits + r) * parts + p) * slice4 + i] (float4 i of
    // the slice) and bumps ctr[tile * splits + r], whose high 32 bits hold
    // the launch's `seq` and low 32 bits the parts counted so far.
    int parts;
    int slice4;                // float4 of a CTA's slice of the tile
    float4 *ws;
    unsigned long long *ctr;
    uint32_t seq;              // never 0
};

// Count one more part of this launch on a tagged counter; returns how many
// parts, this one included, have arrived (a stale count from an earlier
// launch counts as none).  Other parts of the same launch are the only
// contenders, so the loop ends after at most `parts` rounds; the bound is a
// guard.
__device__ __forceinline__ int count_part(unsigned long long *ctr, uint32_t seq) {
    unsigned long long cur = atomicAdd(ctr, 0ull);
    for (int i = 0; i < 1 << 16; ++i) {
        const unsigned long long want = (static_cast<uint32_t>(cur >> 32) == seq)
                                            ? cur + 1ull
                                            : ((static_cast<unsigned long long>(seq) << 32) | 1ull);
        const unsigned long long prev = atomicCAS(ctr, cur, want);
        if (prev == cur) return static_cast<int>(want & 0xffffffffull);
        cur = prev;
    }
    return 0;
}

// One output through the epilogue and rounded to half.
__device__ __forceinline__ __half skinny_out(const Epi &e, float x, int m, int n, int N) {
    if (e.on) {
        const float b = e.bias ? __half2float(e.bias[n]) : 0.f;
        const float r = e.reads_res() ? __half2float(e.res[static_cast<size_t>(m) * N + n]) : 0.f;
        x = epi_apply1(e, x, b, r);
    }
    return __float2half_rn(x);
}

// Whole warp: 16 consecutive 32-bit TMEM columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_load_16cols(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

template <int MN, int STAGES>
__global__ void __launch_bounds__(kSkThreads, 1)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmA,
                       const SkArgs args) {
    using T = SkCfg<MN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + T::kBarOffset);
    const uint32_t bar0 = smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    const uint32_t accf_bar = bar0 + 8u * (2 * STAGES);
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 1);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + T::kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    __shared__ int never_abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tile = blockIdx.x;   // group of `rows` columns of C
    const int row0 = tile * args.rows;
    const int nend = row0 + args.rows < args.N ? row0 + args.rows : args.N;
    // the B box is `rows` rows tall; the stage's rows past it keep stale data,
    // which only reaches TMEM lanes the epilogue never reads
    const uint32_t stage_tx = static_cast<uint32_t>(args.rows + MN) * (kSkBK * 2);
    const int share = blockIdx.y;                // share of K (parts x splits of them per tile)
    const int split = share % args.splits;        // this CTA's rank in its cluster
    const int part = share / args.splits;         // which cluster of the tile
    const int m0 = static_cast<int>(blockIdx.z) * MN;  // first row of A (and of C) of this tile
    const int mt = args.M - m0 < MN ? args.M - m0 : MN;  // its rows of A
    const int kb0 = share * args.kb_per_split;
    const int kb1 = kb0 + args.kb_per_split < args.num_kb ? kb0 + args.kb_per_split : args.num_kb;

    // The B boxes of this CTA's first ring fill are asked of L2 before the
    // set-up and the dependent-launch wait, one per lane of warp 2, so the
    // stream from DRAM starts earlier.  A prefetch only fills L2, where a
    // previous kernel's writes land too.
    if (warp == 2 && lane < STAGES && kb0 + lane < kb1) tma_prefetch_l2_2d(&tmB, (kb0 + lane) * kSkBK, row0);

    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmA);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(accf_bar, 1);
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

    uint32_t armed = 0, arm_parity = 0;
    uint32_t v[MN];  // epilogue warps: this lane's accumulators (fp32 bits)
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(empty_bar(stage), phase ^ 1u, args.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                if (kb - kb0 != args.debug_skip_kblock) {
                    const uint32_t sb = sbase + stage * T::kStageBytes;
                    mbar_arrive_expect_tx(full_bar(stage), stage_tx);
                    armed |= 1u << stage;
                    arm_parity ^= 1u << stage;
                    tma_load_2d(sb, &tmB, full_bar(stage), kb * kSkBK, row0);
                    tma_load_2d(sb + T::kBBytes, &tmA, full_bar(stage), kb * kSkBK, m0);
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) {
                if (!*abort_flag) skinny_timeout(1);
                *abort_flag = 1;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            constexpr uint32_t idesc = idesc_f16_f32acc(kSkBM, MN);
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(full_bar(stage), phase, args.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t sb = sbase + stage * T::kStageBytes;
                const uint64_t bdesc_rows = sw128_kmajor_desc(sb);               // B: the MMA's A operand
                const uint64_t adesc_rows = sw128_kmajor_desc(sb + T::kBBytes);  // A: the MMA's B operand
#pragma unroll
                for (int k = 0; k < kSkBK / 16; ++k)
                    mma_f16_ss(tmem_base, bdesc_rows + 2u * k, adesc_rows + 2u * k, idesc,
                               (kb > kb0 || k > 0) ? 1u : 0u);
                mma_commit(empty_bar(stage));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            // (with no k-blocks the commit arrives at once and the epilogue writes zeros)
            if (ok) mma_commit(accf_bar);
            if (!ok) {
                if (!*abort_flag) skinny_timeout(2);
                *abort_flag = 1;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue, 4 warps
        const int quarter = warp & 3;  // TMEM lanes this warp may read
        int ok = 1;
        if (lane == 0) ok = mbar_wait(accf_bar, 0, args.timeout_ns, abort_flag) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
#pragma unroll
        for (int m = 0; m < MN; ++m) v[m] = 0u;  // (stays 0 with no k-blocks)
        if (ok && kb1 > kb0) {
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
            if constexpr (MN == 16) {
                tmem_load_16cols(taddr, v);
            } else {
#pragma unroll
                for (int c = 0; c < MN / 32; ++c)
                    tmem_load_32cols(taddr + 32u * c, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * c]));
            }
        }
        if (!ok && lane == 0) {
            if (!*abort_flag) skinny_timeout(3);
            *abort_flag = 1;
        }
        const int n = row0 + quarter * 32 + lane;
        if (args.splits == 1 && ok && n < nend) {
#pragma unroll
            for (int m = 0; m < MN; ++m) {  // (a guard, not an early exit: v stays in registers)
                if (m < mt)
                    args.C[static_cast<size_t>(m0 + m) * args.N + n] =
                        skinny_out(args.epi, __uint_as_float(v[m]), m0 + m, n, args.N);
            }
        }
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (*abort_flag) {
        // let this CTA's own copies and MMAs in flight finish before its
        // shared memory and TMEM are released
        if (warp == 0 && lane == 0) {
            for (int s = 0; s < STAGES; ++s)
                if (armed & (1u << s))
                    (void)mbar_wait(full_bar(s), ((arm_parity >> s) & 1u) ^ 1u, args.timeout_ns, &never_abort);
        }
        if (warp == 1 && lane == 0) {
            mma_commit(drain_bar);
            (void)mbar_wait(drain_bar, 0, args.timeout_ns, &never_abort);
        }
        __syncwarp();
        tc_fence_before_sync();
        __syncthreads();
    }
    if (args.splits > 1) {
        // ------------------------------------------- sum of the cluster's shares
        // The ring is idle now (every load was consumed by an MMA that has
        // completed, or drained above): its start holds this CTA's share,
        // [mt][128] fp32 (at most 64 KB).  Every thread of every CTA in the
        // cluster passes both cluster barriers.
        float *share = reinterpret_cast<float *>(smem);
        if (warp >= 2) {
            const int nl = (warp & 3) * 32 + lane;
#pragma unroll
            for (int m = 0; m < MN; ++m)
                if (m < mt) share[m * kSkBM + nl] = __uint_as_float(v[m]);
        }
        cluster_sync();
        // CTA r of the cluster (r = its share of K) adds slice r of the tile,
        // four consecutive columns per thread, over the shares in order.
        const int groups = mt * (kSkBM / 4);
        const int per = (groups + args.splits - 1) / args.splits;
        const int g0 = split * per;
        const int g1 = g0 + per < groups ? g0 + per : groups;
        const bool vec = (args.N & 3) == 0 && (reinterpret_cast<uintptr_t>(args.C) & 7u) == 0;
        const int tile_slice = (static_cast<int>(blockIdx.z) * static_cast<int>(gridDim.x) + tile) * args.splits + split;
        float4 *slices = args.parts > 1 ? args.ws + static_cast<size_t>(tile_slice) * args.parts * args.slice4
                                        : nullptr;
        bool store = args.parts == 1;
        if (args.parts > 1) {
            // this cluster's part of the slice to the workspace, then count it
            for (int gi = g0 + static_cast<int>(threadIdx.x); gi < g1; gi += kSkThreads) {
                const uint32_t at = sbase + static_cast<uint32_t>(gi) * 16u;
                float4 sum = ld_dsmem_f4(mapa_shared(at, 0));
                for (int sp = 1; sp < args.splits; ++sp) {
                    const float4 x = ld_dsmem_f4(mapa_shared(at, static_cast<uint32_t>(sp)));
                    sum.x += x.x;
                    sum.y += x.y;
                    sum.z += x.z;
                    sum.w += x.w;
                }
                slices[static_cast<size_t>(part) * args.slice4 + (gi - g0)] = sum;
            }
            __threadfence();
            __syncthreads();
            __shared__ int last;
            if (threadIdx.x == 0) last = count_part(args.ctr + tile_slice, args.seq) == args.parts;
            __syncthreads();
            store = last != 0;
            if (store) __threadfence();  // every part's slice is visible to this CTA
        }
        for (int gi = g0 + static_cast<int>(threadIdx.x); store && gi < g1; gi += kSkThreads) {
            float4 sum;
            if (args.parts > 1) {
                // the parts in order p = 0, 1, ...: the sum does not depend on
                // which cluster finished last
                sum = __ldcg(&slices[gi - g0]);
                for (int p = 1; p < args.parts; ++p) {
                    const float4 x = __ldcg(&slices[static_cast<size_t>(p) * args.slice4 + (gi - g0)]);
                    sum.x += x.x;
                    sum.y += x.y;
                    sum.z += x.z;
                    sum.w += x.w;
                }
            } else {
                const uint32_t at = sbase + static_cast<uint32_t>(gi) * 16u;
                sum = ld_dsmem_f4(mapa_shared(at, 0));
                for (int sp = 1; sp < args.splits; ++sp) {
                    const float4 x = ld_dsmem_f4(mapa_shared(at, static_cast<uint32_t>(sp)));
                    sum.x += x.x;
                    sum.y += x.y;
                    sum.z += x.z;
                    sum.w += x.w;
                }
            }
            const int m = m0 + gi / (kSkBM / 4);
            const int n = row0 + (gi % (kSkBM / 4)) * 4;
            __half *out = args.C + static_cast<size_t>(m) * args.N + n;
            const float s4[4] = {sum.x, sum.y, sum.z, sum.w};
            if (vec && n + 3 < nend) {
                __half2 lo = __halves2half2(skinny_out(args.epi, s4[0], m, n, args.N),
                                            skinny_out(args.epi, s4[1], m, n + 1, args.N));
                __half2 hi = __halves2half2(skinny_out(args.epi, s4[2], m, n + 2, args.N),
                                            skinny_out(args.epi, s4[3], m, n + 3, args.N));
                uint2 w;
                w.x = *reinterpret_cast<uint32_t *>(&lo);
                w.y = *reinterpret_cast<uint32_t *>(&hi);
                *reinterpret_cast<uint2 *>(out) = w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (n + j < nend) out[j] = skinny_out(args.epi, s4[j], m, n + j, args.N);
            }
        }
        // No CTA leaves while another still reads its share.  Those reads have
        // returned their values (they feed the stores above) before a CTA
        // arrives, so the barrier only has to order execution.
        cluster_sync_relaxed();
    }
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, T::kTmemCols);
    }
}

// Clusters of `size` CTAs of this kernel the device holds at once (cached).
template <int MN, int S>
int max_clusters(int size, std::string &err) {
    static std::mutex mu;
    static std::map<std::pair<int, int>, int> cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        err = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return -1;
    }
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find({dev, size});
    if (it != cache.end()) return it->second;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = size;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(1, size);
    cfg.blockDim = dim3(kSkThreads);
    cfg.dynamicSmemBytes = SkCfg<MN, S>::kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, gemm_skinny_kernel<MN, S>, &cfg);
    if (e != cudaSuccess) {
        err = std::string("cudaOccupancyMaxActiveClusters: ") + cudaGetErrorString(e);
        return -1;
    }
    cache[{dev, size}] = n;
    return n;
}

// Workspace of the multi-cluster split, per (device, stream): partial slices
// and tagged counters, grown on demand, with the stream's launch sequence
// number (counters are cleared only when it wraps).  Calls on one stream run
// in order, so a stream has one user at a time.
struct SkWs {
    float4 *ws = nullptr;
    unsigned long long *ctr = nullptr;
    size_t ws_bytes = 0;
    int counters = 0;
    uint32_t seq = 0;
};

int skinny_workspace(cudaStream_t stream, size_t ws_bytes, int counters, SkWs **out, std::string &err) {
    static std::mutex mu;
    static std::map<std::pair<int, cudaStream_t>, SkWs> cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        err = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(mu);
    SkWs &w = cache[{dev, stream}];
    if (w.ws_bytes < ws_bytes || w.counters < counters) {
        // the stream may still be running a launch that uses the old buffers
        e = cudaStreamSynchronize(stream);
        if (e == cudaSuccess && w.ws) e = cudaFree(w.ws);
        if (e == cudaSuccess && w.ctr) e = cudaFree(w.ctr);
        w = SkWs{};
        if (e == cudaSuccess) e = cudaMalloc(&w.ws, ws_bytes);
        if (e == cudaSuccess) e = cudaMalloc(&w.ctr, static_cast<size_t>(counters) * sizeof(unsigned long long));
        if (e == cudaSuccess)
            e = cudaMemsetAsync(w.ctr, 0, static_cast<size_t>(counters) * sizeof(unsigned long long), stream);
        if (e != cudaSuccess) {
            err = std::string("skinny split workspace: ") + cudaGetErrorString(e);
            w = SkWs{};
            return GEMM_ERR_CUDA;
        }
        w.ws_bytes = ws_bytes;
        w.counters = counters;
    }
    if (++w.seq == 0) {  // the sequence number wrapped: no counter may hold a live tag
        e = cudaMemsetAsync(w.ctr, 0, static_cast<size_t>(w.counters) * sizeof(unsigned long long), stream);
        if (e != cudaSuccess) {
            err = std::string("skinny split counter reset: ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
        w.seq = 1;
    }
    *out = &w;
    return GEMM_OK;
}

template <int MN>
int launch_mn(const SkinnyLaunch &L, std::string &err) {
    constexpr int S = sk_stages<MN>();
    using T = SkCfg<MN, S>;
    auto kernel = gemm_skinny_kernel<MN, S>;
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
    // clusters of 2, 4 and 8 CTAs the device holds at once
    int cap[4] = {L.ctas, 0, 0, 0};
    for (int l = 1; l < 4; ++l) {
        cap[l] = max_clusters<MN, S>(1 << l, err);
        if (cap[l] < 0) return GEMM_ERR_CUDA;
    }
    SkinnyPlan plan;
    skinny_plan(L.M, L.N, L.K, L.ctas, cap, &plan);
    const int num_kb = (L.K + kSkBK - 1) / kSkBK;
    const int splits = plan.splits;
    // Several clusters per tile need the workspace; under stream capture (a
    // replayed graph would reuse this launch's sequence number) the tile
    // stays with one cluster.
    float4 *ws = nullptr;
    unsigned long long *ctr = nullptr;
    uint32_t seq = 0;
    const int slice4 = (MN * (kSkBM / 4) + splits - 1) / splits;
    if (plan.parts > 1) {
        cudaStreamCaptureStatus cap_status = cudaStreamCaptureStatusNone;
        e = cudaStreamIsCapturing(L.stream, &cap_status);
        if (e != cudaSuccess) {
            err = std::string("cudaStreamIsCapturing: ") + cudaGetErrorString(e);
            return GEMM_ERR_CUDA;
        }
        if (cap_status != cudaStreamCaptureStatusNone) {
            plan.parts = 1;
            plan.kb_per_split = (num_kb + splits - 1) / splits;
        } else {
            const int slices = plan.groups * plan.mtiles * splits;
            SkWs *w = nullptr;
            const int st = skinny_workspace(
                L.stream, static_cast<size_t>(slices) * plan.parts * slice4 * sizeof(float4), slices, &w, err);
            if (st != GEMM_OK) return st;
            ws = w->ws;
            ctr = w->ctr;
            seq = w->seq;
        }
    }
    const SkArgs args{static_cast<__half *>(L.C), L.M, L.N, L.K, num_kb, plan.kb_per_split, splits, plan.rows,
                      L.timeout_ns, make_epi(L.epi, L.N), L.debug_skip_kblock, plan.parts, slice4, ws, ctr,
                      seq};
    CUtensorMap tmB, tmA;
    if (!encode_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, L.B, L.N, L.K, plan.rows, kSkBK, err) ||
        !encode_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, L.A, L.M, L.K, MN, kSkBK, err))
        return GEMM_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = splits;
    attr[1].val.clusterDim.z = 1;
    cfg.gridDim = dim3(plan.groups, splits * plan.parts, plan.mtiles);
    cfg.blockDim = dim3(kSkThreads);
    cfg.dynamicSmemBytes = T::kSmemBytes;
    cfg.stream = L.stream;
    cfg.attrs = attr;
    cfg.numAttrs = splits > 1 ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kernel, tmB, tmA, args);
    if (e != cudaSuccess) {
        err = std::string("skinny kernel launch: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

}  // namespace

int skinny_ctas_per_sm() { return kSkCtasPerSm; }

void skinny_plan(int M, int N, int K, int ctas, const int *cap, SkinnyPlan *plan) {
    const int num_kb = (K + kSkBK - 1) / kSkBK;
    const int mtiles = M <= kSkBM ? 1 : (M + kSkBM - 1) / kSkBM;  // 128-row tiles of A
    const long long tiles = static_cast<long long>((N + kSkBM - 1) / kSkBM) * mtiles;
    // An SM's rate goes with the k-blocks its ring keeps in flight, not with
    // the rows each carries: shorter groups or fewer shares measured slower.
    // So the groups stay 128 rows and each tile gets the largest power of
    // two of shares (at most 8, each at least 8 k-blocks) for which all the
    // tiles' clusters are resident at once.
    int s = 1;
    for (int l = 3; l >= 1; --l) {
        const int c = 1 << l;
        int fit = ctas / c;
        if (cap && cap[l] < fit) fit = cap[l];
        if (num_kb / c >= 8 && tiles <= fit) {
            s = c;
            break;
        }
    }
    int rows = kSkBM;
    if (s == 1 && mtiles == 1 && tiles < ctas && tiles * 2 > ctas) {
        // fewer 128-row groups than CTA slots, and no split: shorter groups
        // put every slot to work on B's stream (16 x 16384 x 8192: 128 groups
        // -> 147 of 112 rows, -0.4 us; 64 x 12288 x 4096: -0.7 us)
        rows = static_cast<int>((N + ctas - 1) / ctas);
        rows = (rows + 7) & ~7;
    }
    if (s == 1 && mtiles == 1 && tiles > ctas && ctas > 0) {
        // more than one wave: spread the rows evenly over the waves, so that
        // the last wave is as full as the others
        const long long slots = ((tiles + ctas - 1) / ctas) * ctas;
        rows = static_cast<int>((N + slots - 1) / slots);
        rows = (rows + 7) & ~7;
    }
    // Still most SMs idle with the largest cluster (a few tiles over a very
    // long K): give each tile several clusters, as many as fill the SMs at
    // once (at most 8), each share still at least 8 k-blocks.
    int parts = 1;
    if (s == 8) {
        int fit = ctas / 8;
        if (cap && cap[3] < fit) fit = cap[3];
        long long p = tiles > 0 ? fit / tiles : 1;
        if (p > 8) p = 8;
        if (p > num_kb / (8 * s)) p = num_kb / (8 * s);
        if (p >= 2) parts = static_cast<int>(p);
    }
    const int kbs = (num_kb + s * parts - 1) / (s * parts);
    *plan = SkinnyPlan{s, rows, (N + rows - 1) / rows, kbs > 0 ? kbs : 1, mtiles, parts};
}

int skinny_launch(const SkinnyLaunch &L, std::string &err) {
    if (L.M < 1 || (L.M + kSkBM - 1) / kSkBM > 65535) {
        err = "skinny: M must be 1..65535*128";
        return GEMM_ERR_INVALID_ARG;
    }
    if (L.M <= 16) return launch_mn<16>(L, err);
    if (L.M <= 32) return launch_mn<32>(L, err);
    if (L.M <= 64) return launch_mn<64>(L, err);
    return launch_mn<128>(L, err);
}

int skinny_status_read_clear(cudaStream_t stream, int *code, std::string &err) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
        err = std::string("cudaStreamSynchronize: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_skinny_status, sizeof(int));
    if (e == cudaSuccess && v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_skinny_status, &zero, sizeof(int));
    }
    if (e != cudaSuccess) {
        err = std::string("status word access: ") + cudaGetErrorString(e);
        return GEMM_ERR_CUDA;
    }
    *code = v;
    return GEMM_OK;
}

}  // namespace gb300
