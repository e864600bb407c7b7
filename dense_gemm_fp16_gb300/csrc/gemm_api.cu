// gemm_api.cu -- the C ABI of libgemm.so: argument validation, shape-keyed
// selection of the kernel configuration, per-thread error messages, and the
// device-status query.  Declarations and the contract of each entry point are
// in include/gemm.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include "gemm.h"
#include "gemm_internal.h"
#include "gemm_testing.h"

namespace {

thread_local std::string t_last_error;

int fail(int status, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return status;
}

int fail_str(int status, const std::string &msg) {
    t_last_error = msg;
    return status;
}

// Bounded-wait budget inside the fp16 kernel: long enough for any legitimate
// stall (preemption by another context included), short enough that a broken
// handshake ends the kernel instead of holding the GPU.
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s

int sm_count_of_current_device(int *out) {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && cache[dev] > 0) {
        *out = cache[dev];
        return GEMM_OK;
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || n <= 0)
        return fail(GEMM_ERR_CUDA, "cudaDeviceGetAttribute(SM count): %s", cudaGetErrorString(e));
    if (dev >= 0 && dev < 64) cache[dev] = n;
    *out = n;
    return GEMM_OK;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// Persistent CTA count of an fp16 variant: one CTA (or CTA pair) per tile up
// to one per SM.
int f16_default_grid(int variant, int M, int N, int K, int sm_count) {
    long long tiles;
    if (variant == GEMM_F16_GEMV) return sm_count;  // planned per SM by the launcher
    if (variant == GEMM_F16_SKINNY) return sm_count * gb300::skinny_ctas_per_sm();  // the split's CTA target
    switch (variant) {
        case GEMM_F16_128x256: tiles = ceil_div(M, 128) * ceil_div(N, 256); break;
        case GEMM_F16_256x256_PAIR: tiles = 2 * ceil_div(M, 256) * ceil_div(N, 256); break;
        case GEMM_F16_256x256_QUAD: tiles = 4 * ceil_div(M, 512) * ceil_div(N, 256); break;
        case GEMM_F16_256x256_KSPLIT: return static_cast<int>(4 * ceil_div(M, 256) * ceil_div(N, 256));
        default: tiles = ceil_div(M, 128) * ceil_div(N, 128); break;
    }
    long long cap = sm_count;
    if (variant == GEMM_F16_256x256_QUAD) cap = sm_count & ~3;
    if (variant == GEMM_F16_256x256_PAIR) {
        cap = sm_count & ~1;
        // Split-K spreads few tiles over all the pairs.
        if (gb300::pair_split_pairs(tiles / 2, ceil_div(K, 64), sm_count / 2) > 0) return static_cast<int>(cap);
    }
    long long g = tiles < cap ? tiles : cap;
    return static_cast<int>(g > 0 ? g : 1);
}

// Thread 0 of each CTA records the SM it runs on, that SM's cycle counter
// and the global nanosecond timer, read back to back.
__global__ void sm_clock_sample_kernel(unsigned long long *out) {
    if (threadIdx.x != 0) return;
    unsigned smid;
    unsigned long long ns;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    const long long cycles = clock64();
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(ns));
    out[3 * blockIdx.x + 0] = smid;
    out[3 * blockIdx.x + 1] = static_cast<unsigned long long>(cycles);
    out[3 * blockIdx.x + 2] = ns;
}

}  // namespace

extern "C" {

const char *gemm_last_error(void) { return t_last_error.c_str(); }

// ---------------------------------------------------------------------------
// Selection (host logic only; no device call)
// ---------------------------------------------------------------------------

// Tile rows per band of the tile order.  While A and B fit comfortably in
// L2 (129 MB) the plain column order is kept; beyond that a wave of tiles
// walking every tile row would stream all of A through L2 once per wave, so
// the tiles go in bands of a few rows.
static int f16_default_raster(int variant, int M, int N, int K) {
    const double operand_bytes = 2.0 * (static_cast<double>(M) + N) * K;
    if (variant == GEMM_F16_GEMV || variant == GEMM_F16_SKINNY || operand_bytes <= 96.0 * 1024 * 1024)
        return 1 << 30;
    return variant == GEMM_F16_256x256_PAIR || variant == GEMM_F16_256x256_QUAD ? 8 : 16;
}



int gemm_f16_select(int M, int N, int K, int sm_count, gemm_f16_config *cfg) {
    if (!cfg) return fail(GEMM_ERR_INVALID_ARG, "gemm_f16_select: cfg is NULL");
    if (M < 0 || N < 0 || K < 0 || sm_count <= 0)
        return fail(GEMM_ERR_INVALID_ARG, "gemm_f16_select: bad M=%d N=%d K=%d sm_count=%d", M, N,
                    K, sm_count);
    // With a few rows of A every element of B is used only a few times:
    // reading B from HBM bounds the product.  For one row the matrix-vector
    // kernel streams B once on the CUDA cores; from two rows up to 64 the
    // skinny kernel does (B's rows on the MMA's 128-row side, A's rows on
    // its N side, K split over clusters so the tiles fill the SMs), where
    // the 128-row tiles of A would leave most of each MMA and most SMs idle.
    // The skinny kernel also takes any M whose 128 x 128 tiles are too few to
    // fill the SMs, when it can split K into 2 shares of at least 16
    // k-blocks or into 4 or more (measured 1.5-8x faster than the tile
    // kernels there: 160 x 2048 x 8192 13.3 against 29.8 us).
    int variant;
    gb300::SkinnyPlan plan;
    gb300::skinny_plan(M, N, K, sm_count * gb300::skinny_ctas_per_sm(), nullptr, &plan);
    const bool skinny_split = plan.splits >= 4 || (plan.splits == 2 && plan.kb_per_split >= 16);
    if (M <= 1) {
        variant = GEMM_F16_GEMV;
    } else if (M <= 64 || skinny_split) {
        variant = GEMM_F16_SKINNY;
    } else if (M <= 128) {
        variant = GEMM_F16_128x128;  // a pair tile would be half empty
    } else {
        // Otherwise the tile whose waves cost least: a wave of 128 x 256 tiles
        // or of 256 x 256 pair tiles takes about 1.15 and 1.1 times a wave of
        // 128 x 128 tiles (1.5 for both with K <= 512, where the wider tiles'
        // set-up and drain weigh more), fitted to a GB300 sweep of M 160-2048,
        // N 2048-28672, K 512-8192 (mean 0.5 % from the best tile).  Ties go
        // to the smaller tile.
        const long long t128 = ceil_div(M, 128) * ceil_div(N, 128);
        const long long t256 = ceil_div(M, 128) * ceil_div(N, 256);
        const long long tpair = ceil_div(M, 256) * ceil_div(N, 256);
        const bool short_k = ceil_div(K, 64) <= 8;
        const double c256 = short_k ? 1.5 : 1.15, cpair = short_k ? 1.5 : 1.1;
        const long long pairs = sm_count / 2 > 0 ? sm_count / 2 : 1;
        const double w128 = static_cast<double>(ceil_div(t128, sm_count));
        const double w256 = c256 * static_cast<double>(ceil_div(t256, sm_count));
        const double wpair = cpair * static_cast<double>(ceil_div(tpair, pairs));
        variant = GEMM_F16_128x128;
        double best = w128;
        if (w256 < best) {
            variant = GEMM_F16_128x256;
            best = w256;
        }
        if (wpair < best) variant = GEMM_F16_256x256_PAIR;
        // Rows of A and B that are not a whole number of 128-byte lines (K not
        // a multiple of 64) make every 128-byte TMA row span two L2 lines:
        // the L2 requests per byte loaded more than double and bound the pair
        // kernel (5000 x 5376 x 2040: 2.6x the requests of 5376^2 x 2048, the
        // tensor pipe 63 % busy instead of 86 %).  Two pairs sharing B through
        // multicast cut a quarter of them, which measured faster on every such
        // shape tried, even where their 36 clusters need more waves than 76
        // pairs (us, pair / two pairs: 5000 x 5376 x 2040 94 / 76, 5376^2 x 2040
        // 95 / 87, 4096^2 x 4088 116 / 93, 8192^2 x 8184 803 / 713); on rows of
        // whole lines the pair stays ahead (5376^2 x 2048 78 / 88).  With one
        // row of pair tiles (M <= 256) the second pair would have no tiles.
        if (variant == GEMM_F16_256x256_PAIR && K % 64 != 0 && M > 256) variant = GEMM_F16_256x256_QUAD;
        // Few pair tiles over a long K: two pairs per cluster split each
        // tile's K, their sums added through distributed shared memory, when
        // the tiles fill at least half of the 4-CTA clusters that fit at once
        // (36 on 152 SMs) and each half keeps 64+ k-blocks.  Measured (us,
        // that / the tile pick / cuBLAS): 1024 x 2048 x 8192 28.3 / 30.8 /
        // 23.0, 256 x 8192 x 8192 34.9 / 37.1 / 28.5, 512 x 4096 x 14336
        // 45.1 / 54.0 / 41.0; with 32 k-blocks per half it lost (1024 x 2048 x
        // 2048 14.9 / 10.6), and with more tiles than clusters too.
        const long long ks_clusters = sm_count / 4 - 2;
        if (M >= 256 && K % 64 == 0 && ceil_div(K, 64) >= 128 && 2 * tpair > ks_clusters && tpair <= ks_clusters)
            variant = GEMM_F16_256x256_KSPLIT;
    }
    cfg->variant = variant;
    cfg->grid = f16_default_grid(variant, M, N, K, sm_count);
    cfg->flags = 0;
    cfg->raster = f16_default_raster(variant, M, N, K);
    return GEMM_OK;
}

// Predicted time in microseconds of one SGEMM launch with a given tile and
// split count.  The CTAs spread over the SMs, so the busiest SM runs
// ceil(ctas / sms) of them, each over its K share; one 128 x 128 CTA costs
// about 0.090 us per K element, one 64 x 64 CTA 0.041 us (13% less each when
// two share an SM) and one 128 x 64 CTA 0.054 us (10% less each when two
// share an SM); a split adds the partial-slot writes, the fence and the last
// CTA's pass over the slots.  The constants are GB300 measurements, fitted
// to a 16-shape sweep of every tile at 1 to 8 shares: the picks land 0.3 %
// from the best measured on average, worst 2.8 %; the model only has to
// rank the candidates.
static void sgemm_tile(int variant, int *bm, int *bn) {
    *bm = variant == GEMM_SGEMM_64x64 ? 64 : 128;
    *bn = variant == GEMM_SGEMM_128x128 ? 128 : 64;
}

static double sgemm_cost(int variant, int M, int N, int sms, int splits, int chunk) {
    const bool big = variant == GEMM_SGEMM_128x128;
    int bm, bn;
    sgemm_tile(variant, &bm, &bn);
    const double tiles = static_cast<double>(ceil_div(M, bm)) * static_cast<double>(ceil_div(N, bn));
    const double per_sm = std::ceil(tiles * splits / sms);
    if (variant == GEMM_SGEMM_128x64) {
        double cost = per_sm * chunk * 0.054 * (per_sm >= 2 ? 0.9 : 1.0);
        if (splits > 1) cost += 1.0 + 0.2 * splits;
        return cost;
    }
    const double share = (!big && per_sm >= 2) ? 0.87 : 1.0;
    double cost = per_sm * chunk * (big ? 0.090 : 0.041) * share;
    if (splits > 1) cost += big ? 2.0 + 1.0 * splits : 1.0 + 0.4 * splits;
    return cost;
}

// Tile and split count of the lowest predicted time; a caller's fixed
// variant or split count (non-zero) narrows the search.  Splits are only
// considered when the tiles number at most twice the SMs: beyond that the
// last wave is a small part of the run and the slots' traffic is not.
static void sgemm_plan(int M, int N, int K, int sms, int fix_variant, int fix_splits, int *variant,
                       int *splits) {
    bool have = false;
    double best = 0.0;
    *variant = fix_variant ? fix_variant : GEMM_SGEMM_128x128;
    *splits = 1;
    for (int v = GEMM_SGEMM_128x128; v < GEMM_SGEMM_NUM_VARIANTS; ++v) {
        if (fix_variant && v != fix_variant) continue;
        int bm, bn;
        sgemm_tile(v, &bm, &bn);
        const long long tiles = ceil_div(M, bm) * ceil_div(N, bn);
        const int smax = (K > 0 && tiles <= 2LL * sms) ? gb300::kSgemmMaxSplits : 1;
        const int s_lo = fix_splits ? fix_splits : 1, s_hi = fix_splits ? fix_splits : smax;
        for (int s = s_lo; s <= s_hi; ++s) {
            int chunk = K;
            const int eff = gb300::sgemm_split_chunk(K, s, &chunk);
            if (eff != s && !fix_splits) continue;  // the same as a smaller count
            const double c = sgemm_cost(v, M, N, sms, eff, chunk);
            if (!have || c < best) {
                have = true;
                best = c;
                *variant = v;
                *splits = eff;
            }
        }
    }
}

int gemm_sgemm_select(int M, int N, int K, int sm_count, gemm_sgemm_config *cfg) {
    if (!cfg) return fail(GEMM_ERR_INVALID_ARG, "gemm_sgemm_select: cfg is NULL");
    if (M < 0 || N < 0 || K < 0 || sm_count <= 0)
        return fail(GEMM_ERR_INVALID_ARG, "gemm_sgemm_select: bad M=%d N=%d K=%d sm_count=%d", M,
                    N, K, sm_count);
    sgemm_plan(M, N, K, sm_count, 0, 0, &cfg->variant, &cfg->splits);
    return GEMM_OK;
}

// ---------------------------------------------------------------------------
// fp16 NT
// ---------------------------------------------------------------------------

static int f16_nt_impl(int M, int N, int K, const void *A, const void *B, void *C,
                       gemm_stream_t stream, const gemm_f16_config *cfg, uint64_t timeout_ns,
                       int debug_skip_kblock, bool static_scratch = false,
                       const gemm_f16_epilogue *epi = nullptr, bool debug_skip_publish = false) {
    if (M < 0 || N < 0 || K < 0)
        return fail(GEMM_ERR_INVALID_ARG, "gemm_f16_nt: negative size M=%d N=%d K=%d", M, N, K);
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C) return fail(GEMM_ERR_INVALID_ARG, "gemm_f16_nt: C is NULL");
    if (K > 0 && (!A || !B)) return fail(GEMM_ERR_INVALID_ARG, "gemm_f16_nt: A or B is NULL");
    if (K > 0 && (!aligned16(A) || !aligned16(B)))
        return fail(GEMM_ERR_MISALIGNED, "gemm_f16_nt: A and B must be 16-byte aligned");
    if (K % 8 != 0)
        return fail(GEMM_ERR_UNSUPPORTED,
                    "gemm_f16_nt: K=%d; K*2 bytes must be a multiple of 16 (K %% 8 == 0)", K);
    if (epi && (epi->activation < 0 || epi->activation >= GEMM_ACT_NUM))
        return fail(GEMM_ERR_INVALID_ARG, "gemm_f16_nt_fused: unknown activation %d", epi->activation);
    if (cfg && (cfg->variant < 0 || cfg->variant >= GEMM_F16_NUM_VARIANTS || cfg->grid < 0 ||
                (cfg->flags & ~GEMM_F16_FLAG_STREAM_K) != 0 || cfg->raster < 0))
        return fail(GEMM_ERR_INVALID_ARG, "gemm_f16_nt_ex: bad config variant=%d grid=%d flags=%d raster=%d",
                    cfg->variant, cfg->grid, cfg->flags, cfg->raster);
    int sms = 0;
    int st = sm_count_of_current_device(&sms);
    if (st != GEMM_OK) return st;
    gemm_f16_config sel;
    st = gemm_f16_select(M, N, K, sms, &sel);
    if (st != GEMM_OK) return st;
    if (cfg && cfg->variant != GEMM_F16_AUTO) {
        sel.variant = cfg->variant;
        sel.grid = f16_default_grid(sel.variant, M, N, K, sms);
        if (sel.variant == GEMM_F16_GEMV && M > 4)
            return fail(GEMM_ERR_UNSUPPORTED, "gemm_f16_nt_ex: the GEMV variant takes M <= 4 (M=%d)", M);
    }
    if (cfg && cfg->grid > 0) sel.grid = cfg->grid;
    if (cfg && cfg->variant != GEMM_F16_AUTO) sel.raster = f16_default_raster(sel.variant, M, N, K);
    if (cfg && cfg->raster > 0) sel.raster = cfg->raster;

    gb300::F16Launch L;
    L.M = M;
    L.N = N;
    L.K = K;
    L.A = A;
    L.B = B;
    L.C = C;
    L.stream = reinterpret_cast<cudaStream_t>(stream);
    L.variant = sel.variant;
    L.grid = sel.grid;
    L.timeout_ns = timeout_ns;
    L.debug_skip_kblock = debug_skip_kblock;
    L.allow_stream_k = cfg && (cfg->flags & GEMM_F16_FLAG_STREAM_K);
    L.static_scratch = static_scratch;
    L.debug_skip_publish = debug_skip_publish;
    L.raster = sel.raster;
    L.sm_count = sms;
    if (epi) {
        L.epi.alpha = epi->alpha;
        L.epi.beta = epi->beta;
        L.epi.bias = epi->bias;
        L.epi.res = epi->residual;
        L.epi.act = epi->activation;
        L.epi.on = 1;
    }
    std::string err;
    st = gb300::f16_launch(L, err);
    if (st != GEMM_OK) return fail_str(st, err);
    return GEMM_OK;
}

int gemm_f16_nt(int M, int N, int K, const void *A, const void *B, void *C, gemm_stream_t stream) {
    return f16_nt_impl(M, N, K, A, B, C, stream, nullptr, kDefaultTimeoutNs, -1);
}

int gemm_f16_nt_ex(int M, int N, int K, const void *A, const void *B, void *C,
                   gemm_stream_t stream, const gemm_f16_config *cfg) {
    return f16_nt_impl(M, N, K, A, B, C, stream, cfg, kDefaultTimeoutNs, -1);
}

int gemm_f16_nt_fused(int M, int N, int K, const void *A, const void *B, void *C,
                      const gemm_f16_epilogue *epi, gemm_stream_t stream,
                      const gemm_f16_config *cfg) {
    return f16_nt_impl(M, N, K, A, B, C, stream, cfg, kDefaultTimeoutNs, -1, false, epi);
}

// The allocation-free variant declared in gemm.h: the CTA-pair kernel with
// stream-K, its partials in the library's static scratch array.
int gemm_f16_nt_stream_k_noalloc(int M, int N, int K, const void *A, const void *B, void *C,
                                 gemm_stream_t stream) {
    const gemm_f16_config cfg = {GEMM_F16_256x256_PAIR, 0, GEMM_F16_FLAG_STREAM_K};
    return f16_nt_impl(M, N, K, A, B, C, stream, &cfg, kDefaultTimeoutNs, -1, true);
}

// Test hook declared in gemm_testing.h: one TMA load left out so that the
// kernel's bounded waits run out (`timeout_ns` each) and the status path runs.
int gemm_debug_f16_nt_skip_load(int M, int N, int K, const void *A, const void *B, void *C,
                                gemm_stream_t stream, int skip_kblock, unsigned long long timeout_ns) {
    return f16_nt_impl(M, N, K, A, B, C, stream, nullptr, timeout_ns, skip_kblock);
}

// Test hook declared in gemm_testing.h: stream-K on the pair kernel with the
// partials written but never flagged, so that each split tile's first pair
// waits for them until its bounded wait (`timeout_ns`) runs out.
int gemm_debug_f16_nt_stream_k_skip_publish(int M, int N, int K, const void *A, const void *B, void *C,
                                            gemm_stream_t stream, unsigned long long timeout_ns) {
    const gemm_f16_config cfg = {GEMM_F16_256x256_PAIR, 0, GEMM_F16_FLAG_STREAM_K, 0};
    return f16_nt_impl(M, N, K, A, B, C, stream, &cfg, timeout_ns, -1, false, nullptr, true);
}

// Test hook declared in gemm_testing.h: the last pair launch's split.
int gemm_debug_last_pair_launch(int *pairs, int *whole_tiles, int *shared_units, int *scratch_kind) {
    if (!pairs || !whole_tiles || !shared_units || !scratch_kind) return -1;
    const gb300::PairLaunchRecord r = gb300::last_pair_launch();
    if (!r.valid) return -1;
    *pairs = r.pairs;
    *whole_tiles = r.whole_tiles;
    *shared_units = r.shared_units;
    *scratch_kind = r.scratch_kind;
    return 0;
}

// Measurement hook declared in gemm_testing.h: one clock sample per CTA.
int gemm_debug_sm_clocks(unsigned long long *out, int ctas, gemm_stream_t stream) {
    if (ctas < 1 || ctas > 65535)
        return fail(GEMM_ERR_INVALID_ARG, "gemm_debug_sm_clocks: ctas=%d outside 1..65535", ctas);
    if (!out || reinterpret_cast<uintptr_t>(out) % 8 != 0)
        return fail(GEMM_ERR_INVALID_ARG, "gemm_debug_sm_clocks: out is NULL or not 8-byte aligned");
    sm_clock_sample_kernel<<<ctas, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(out);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "gemm_debug_sm_clocks: launch: %s", cudaGetErrorString(e));
    return GEMM_OK;
}

// Test hook declared in gemm_testing.h: the skinny variant's plan.
int gemm_debug_skinny_plan(int M, int N, int K, int ctas, int *rows, int *groups, int *kb_per_split) {
    if (M < 1 || N < 1 || K < 0 || ctas < 1 || !rows || !groups || !kb_per_split) return -1;
    gb300::SkinnyPlan p;
    gb300::skinny_plan(M, N, K, ctas, nullptr, &p);
    *rows = p.rows;
    *groups = p.groups;
    *kb_per_split = p.kb_per_split;
    return p.splits;
}

// Test hook declared in gemm_testing.h: clusters per tile of the same plan.
int gemm_debug_skinny_parts(int M, int N, int K, int ctas) {
    if (M < 1 || N < 1 || K < 0 || ctas < 1) return -1;
    gb300::SkinnyPlan p;
    gb300::skinny_plan(M, N, K, ctas, nullptr, &p);
    return p.parts;
}

// ---------------------------------------------------------------------------
// Block-scaled FP8 (MXFP8)
// ---------------------------------------------------------------------------

size_t gemm_mxfp8_scale_bytes(int rows, int K) {
    if (rows <= 0 || K <= 0) return 0;
    return static_cast<size_t>((rows + 127) / 128) * static_cast<size_t>((K + 127) / 128) * 512;
}

int gemm_mxfp8_pack_scales(int rows, int K, const void *plain, void *blocked, gemm_stream_t stream) {
    if (rows < 0 || K < 0)
        return fail(GEMM_ERR_INVALID_ARG, "gemm_mxfp8_pack_scales: negative size rows=%d K=%d", rows, K);
    if (K % 32 != 0)
        return fail(GEMM_ERR_UNSUPPORTED, "gemm_mxfp8_pack_scales: K=%d is not a multiple of 32", K);
    if (rows == 0 || K == 0) return GEMM_OK;
    if (!plain || !blocked) return fail(GEMM_ERR_INVALID_ARG, "gemm_mxfp8_pack_scales: NULL pointer");
    std::string err;
    const int st = gb300::mx_pack_scales_launch(0, rows, K, plain, blocked,
                                                reinterpret_cast<cudaStream_t>(stream), err);
    if (st != GEMM_OK) return fail_str(st, err);
    return GEMM_OK;
}

int gemm_mxfp8_nt(int M, int N, int K, const void *A, const void *SFA, const void *B,
                  const void *SFB, void *C, gemm_stream_t stream) {
    return gemm_mxfp8_nt_ex(M, N, K, A, SFA, B, SFB, C, stream, nullptr);
}

// Both block-scaled products: fmt 0 MXFP8 (alpha 1), 1 NVFP4.
static int mx_impl(int fmt, int M, int N, int K, const void *A, const void *SFA, const void *B,
                   const void *SFB, float alpha, void *C, gemm_stream_t stream,
                   const gemm_mxfp8_config *cfg, uint64_t timeout_ns, int debug_skip_kblock) {
    const char *name = fmt == 0 ? "gemm_mxfp8_nt" : "gemm_nvfp4_nt";
    if (cfg && (cfg->variant < 0 || cfg->variant >= GEMM_MXFP8_NUM_VARIANTS || cfg->grid < 0))
        return fail(GEMM_ERR_INVALID_ARG, "%s_ex: bad config variant=%d grid=%d", name, cfg->variant,
                    cfg->grid);
    if (M < 0 || N < 0 || K < 0)
        return fail(GEMM_ERR_INVALID_ARG, "%s: negative size M=%d N=%d K=%d", name, M, N, K);
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C) return fail(GEMM_ERR_INVALID_ARG, "%s: C is NULL", name);
    if (K % 32 != 0)
        return fmt == 0 ? fail(GEMM_ERR_UNSUPPORTED,
                               "gemm_mxfp8_nt: K=%d; the 32-element scale blocks need K %% 32 == 0", K)
                        : fail(GEMM_ERR_UNSUPPORTED,
                               "gemm_nvfp4_nt: K=%d; rows of K/2 bytes must be multiples of 16 bytes "
                               "(K %% 32 == 0)", K);
    if (K == 0) return f16_nt_impl(M, N, 0, nullptr, nullptr, C, stream, nullptr, kDefaultTimeoutNs, -1);
    if (!A || !B || !SFA || !SFB) return fail(GEMM_ERR_INVALID_ARG, "%s: NULL operand", name);
    if (!aligned16(A) || !aligned16(B) || !aligned16(SFA) || !aligned16(SFB))
        return fail(GEMM_ERR_MISALIGNED, "%s: A, B, SFA and SFB must be 16-byte aligned", name);
    int sms = 0;
    int st = sm_count_of_current_device(&sms);
    if (st != GEMM_OK) return st;
    gb300::MxLaunch L;
    L.M = M;
    L.N = N;
    L.K = K;
    L.A = A;
    L.SFA = SFA;
    L.B = B;
    L.SFB = SFB;
    L.C = C;
    L.stream = reinterpret_cast<cudaStream_t>(stream);
    L.grid = cfg ? cfg->grid : 0;
    L.timeout_ns = timeout_ns;
    L.sm_count = sms;
    // Measured on GB300 at 5376 x 5376 x 2048 / x 8192 (us): 1-CTA 128 x 256
    // with N = 256 MMAs 52 / 157, 1-CTA 128 x 128 62 / 215, CTA pair 256 x 256
    // 56 / 175, CTA pair 256 x 128 68 / 248.  The wide MMA pays more than the
    // second accumulator it costs (two 256-column accumulators and the scale
    // columns do not fit TMEM together); narrow N keeps the 128 x 128 tiles.
    L.variant = (cfg && cfg->variant != GEMM_MXFP8_AUTO) ? cfg->variant
                : (N > 128 ? GEMM_MXFP8_128x256 : GEMM_MXFP8_128x128);
    L.fmt = fmt;
    L.alpha = fmt == 0 ? 1.f : alpha;
    L.debug_skip_kblock = debug_skip_kblock;
    std::string err;
    st = gb300::mx_launch(L, err);
    if (st != GEMM_OK) return fail_str(st, err);
    return GEMM_OK;
}

int gemm_mxfp8_nt_ex(int M, int N, int K, const void *A, const void *SFA, const void *B,
                     const void *SFB, void *C, gemm_stream_t stream, const gemm_mxfp8_config *cfg) {
    return mx_impl(0, M, N, K, A, SFA, B, SFB, 1.f, C, stream, cfg, kDefaultTimeoutNs, -1);
}

// Test hook declared in gemm_testing.h: a block-scaled product with one
// k-block never loaded, so that the kernel's bounded waits run out.
int gemm_debug_blockscaled_skip_load(int fmt, int M, int N, int K, const void *A, const void *SFA,
                                     const void *B, const void *SFB, void *C, gemm_stream_t stream,
                                     const gemm_mxfp8_config *cfg, int skip_kblock,
                                     unsigned long long timeout_ns) {
    if (fmt != 0 && fmt != 1)
        return fail(GEMM_ERR_INVALID_ARG, "gemm_debug_blockscaled_skip_load: fmt %d is not 0 or 1", fmt);
    return mx_impl(fmt, M, N, K, A, SFA, B, SFB, 1.f, C, stream, cfg, timeout_ns, skip_kblock);
}

// ---------------------------------------------------------------------------
// Block-scaled FP4 (NVFP4)
// ---------------------------------------------------------------------------

size_t gemm_nvfp4_scale_bytes(int rows, int K) {
    if (rows <= 0 || K <= 0) return 0;
    return static_cast<size_t>((rows + 127) / 128) * 4 * static_cast<size_t>((K + 255) / 256) * 512;
}

int gemm_nvfp4_pack_scales(int rows, int K, const void *plain, void *blocked, gemm_stream_t stream) {
    if (rows < 0 || K < 0)
        return fail(GEMM_ERR_INVALID_ARG, "gemm_nvfp4_pack_scales: negative size rows=%d K=%d", rows, K);
    if (K % 32 != 0)
        return fail(GEMM_ERR_UNSUPPORTED, "gemm_nvfp4_pack_scales: K=%d is not a multiple of 32", K);
    if (rows == 0 || K == 0) return GEMM_OK;
    if (!plain || !blocked) return fail(GEMM_ERR_INVALID_ARG, "gemm_nvfp4_pack_scales: NULL pointer");
    std::string err;
    const int st = gb300::mx_pack_scales_launch(1, rows, K, plain, blocked,
                                                reinterpret_cast<cudaStream_t>(stream), err);
    if (st != GEMM_OK) return fail_str(st, err);
    return GEMM_OK;
}

int gemm_nvfp4_nt_ex(int M, int N, int K, const void *A, const void *SFA, const void *B,
                     const void *SFB, float alpha, void *C, gemm_stream_t stream,
                     const gemm_mxfp8_config *cfg) {
    return mx_impl(1, M, N, K, A, SFA, B, SFB, alpha, C, stream, cfg, kDefaultTimeoutNs, -1);
}

int gemm_nvfp4_nt(int M, int N, int K, const void *A, const void *SFA, const void *B, const void *SFB,
                  float alpha, void *C, gemm_stream_t stream) {
    return gemm_nvfp4_nt_ex(M, N, K, A, SFA, B, SFB, alpha, C, stream, nullptr);
}

// ---------------------------------------------------------------------------
// SGEMM
// ---------------------------------------------------------------------------

int sgemm_ex(int M, int N, int K, float alpha, const float *A, const float *B, float beta,
             float *C, gemm_stream_t stream, const gemm_sgemm_config *cfg) {
    if (M < 0 || N < 0 || K < 0)
        return fail(GEMM_ERR_INVALID_ARG, "sgemm: negative size M=%d N=%d K=%d", M, N, K);
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C) return fail(GEMM_ERR_INVALID_ARG, "sgemm: C is NULL");
    if (K > 0 && (!A || !B)) return fail(GEMM_ERR_INVALID_ARG, "sgemm: A or B is NULL");
    if (cfg && (cfg->variant < 0 || cfg->variant >= GEMM_SGEMM_NUM_VARIANTS || cfg->splits < 0 ||
                cfg->splits > gb300::kSgemmMaxSplits))
        return fail(GEMM_ERR_INVALID_ARG, "sgemm_ex: bad config variant=%d splits=%d", cfg->variant,
                    cfg->splits);
    int sms = 0;
    int st0 = sm_count_of_current_device(&sms);
    if (st0 != GEMM_OK) return st0;
    int variant = GEMM_SGEMM_128x128, splits = 1;
    sgemm_plan(M, N, K, sms, cfg ? cfg->variant : 0, cfg ? cfg->splits : 0, &variant, &splits);
    gb300::SgemmLaunch L;
    L.splits = splits;
    L.M = M;
    L.N = N;
    L.K = K;
    L.alpha = alpha;
    L.beta = beta;
    L.A = A;
    L.B = B;
    L.C = C;
    L.stream = reinterpret_cast<cudaStream_t>(stream);
    L.variant = variant;
    std::string err;
    int st = gb300::sgemm_launch(L, err);
    if (st != GEMM_OK) return fail_str(st, err);
    return GEMM_OK;
}

int sgemm(int M, int N, int K, float alpha, const float *A, const float *B, float beta, float *C,
          gemm_stream_t stream) {
    return sgemm_ex(M, N, K, alpha, A, B, beta, C, stream, nullptr);
}

// ---------------------------------------------------------------------------
// Device status
// ---------------------------------------------------------------------------

int gemm_check_device_status(gemm_stream_t stream) {
    int code = 0;
    std::string err;
    int st = gb300::f16_status_read_clear(reinterpret_cast<cudaStream_t>(stream), &code, err);
    if (st != GEMM_OK) return fail_str(st, err);
    int sk = 0;
    st = gb300::skinny_status_read_clear(reinterpret_cast<cudaStream_t>(stream), &sk, err);
    if (st != GEMM_OK) return fail_str(st, err);
    if (code == 0 && sk >= 1 && sk <= 3) code = sk;
    if (code != 0) {
        static const char *role[] = {"?", "TMA producer (free-slot wait)",
                                     "MMA issuer (data or accumulator wait)",
                                     "epilogue (accumulator-ready wait)",
                                     "epilogue (stream-K partial wait)"};
        return fail(GEMM_ERR_DEVICE_TIMEOUT,
                    "gemm_f16_nt: a bounded pipeline wait expired in the %s",
                    role[(code >= 1 && code <= 4) ? code : 0]);
    }
    return GEMM_OK;
}

}  // extern "C"
