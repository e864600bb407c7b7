// gemm_internal.h -- declarations shared by the translation units of
// libgemm.so (never installed, never part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

namespace gb300 {

// A row-major [rows][cols] matrix of `elem_bytes`-byte elements at `ptr` as a
// 2-D TMA tensor map with boxes of box_rows x box_cols (zero fill past the
// edges on loads, clipping on stores).  cuTensorMapEncodeTiled is looked up
// through the runtime once.  false, with `err` set, on failure.
bool encode_map(CUtensorMap *map, CUtensorMapDataType dtype, int elem_bytes, const void *ptr, int rows,
                int cols, int box_rows, int box_cols, std::string &err,
                CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

// Split-K for pair-tile grids the tiles alone would leave mostly idle: how
// many CTA pairs share the k-blocks of all `tiles` tiles (each tile split
// over at most kMaxSplit pairs, each share at least kMinShareKb k-blocks),
// or 0 when a split would not give every tile at least kMinSplit pairs.  The
// tile's owner adds the other shares' fp32 partials one after another, which
// costs a few microseconds per tile: measured on GB300, two-way splits lose to
// the unsplit 128 x 128 tiles, four-way and deeper ones win (up to 3.8x at
// 256 x 256 x 65536).
constexpr int kMaxSplit = 8;
constexpr int kMinSplit = 4;
constexpr int kMinShareKb = 32;
inline int pair_split_pairs(long long tiles, long long num_kb, int pairs) {
    long long p = pairs;
    if (p > tiles * kMaxSplit) p = tiles * kMaxSplit;
    if (p > tiles * num_kb / kMinShareKb) p = tiles * num_kb / kMinShareKb;
    return p >= kMinSplit * tiles ? static_cast<int>(p) : 0;
}

// Fused epilogue of the fp16 product: out = act(alpha * acc + bias[n] + beta * res[m][n]).
// act: 0 none, 1 ReLU, 2 SiLU, 3 tanh-GELU.  on == 0: out = acc (the plain product).
struct EpiSpec {
    float alpha = 1.f, beta = 0.f;
    const void *bias = nullptr;  // half [N] or null
    const void *res = nullptr;   // half [M, N] row-major or null (not read when beta == 0)
    int act = 0;
    int on = 0;
};

// One fp16 NT launch, after argument validation and selection.
struct F16Launch {
    int M, N, K;
    const void *A;
    const void *B;
    void *C;
    cudaStream_t stream;
    int variant;            // GEMM_F16_128x256 or GEMM_F16_128x128
    int grid;               // persistent CTAs (> 0)
    uint64_t timeout_ns;    // budget of every bounded wait in the kernel
    int debug_skip_kblock;  // test hook: producer skips this k-block of its first tile (-1: none)
    bool allow_stream_k;    // pair kernel: split the last partial round of tiles along K
    bool static_scratch;    // stream-K partials in the library's static array, no allocation
    int sm_count;           // SMs of the current device
    EpiSpec epi;            // fused epilogue (off by default)
    int raster = 1 << 30;   // tile rows per band of the tile order (>= tile rows: plain)
    bool debug_skip_publish = false;  // test hook: stream-K partials never flagged ready
};

int f16_launch(const F16Launch &L, std::string &err);

// What the last CTA-pair launch on this host thread chose (a test hook):
// the pair count, the tiles computed whole, the k-block units shared out, and
// where the partials went (0 nowhere, 1 an allocated workspace, 2 the static
// array of the allocation-free entry point).  valid == false before the first.
struct PairLaunchRecord {
    bool valid = false;
    int pairs = 0, whole_tiles = 0, shared_units = 0, scratch_kind = 0;
};
PairLaunchRecord last_pair_launch();

// Read-and-clear the fp16 kernel's device status word (0 = no fault).
// Block-scaled FP8 (MXFP8) NT product: E4M3 A [M,K], B [N,K], scale chunks
// SFA, SFB (the layout gemm.h documents), half C [M,N].
struct MxLaunch {
    int M, N, K;
    const void *A, *SFA, *B, *SFB;
    void *C;
    cudaStream_t stream;
    int grid;  // 0: one CTA per SM (at most one per tile)
    uint64_t timeout_ns;
    int sm_count;
    int variant;  // GEMM_MXFP8_* of gemm.h
    int fmt;      // 0: MXFP8 (E4M3, UE8M0 per 32), 1: NVFP4 (E2M1 pairs, UE4M3 per 16)
    float alpha;  // NVFP4: the tensor-level scale applied to the product
    int debug_skip_kblock = -1;  // test hook: producer skips this k-block of its first tile
};
int mx_launch(const MxLaunch &L, std::string &err);
// Plain scales [rows][K/block] -> chunk layout (device pointers, on
// `stream`); fmt as in MxLaunch.
int mx_pack_scales_launch(int fmt, int rows, int K, const void *plain, void *blocked, cudaStream_t stream,
                          std::string &err);

int f16_status_read_clear(cudaStream_t stream, int *code, std::string &err);

// One fp16 matrix-vector launch (M <= 4), after validation and selection.
struct GemvLaunch {
    int M, N, K;
    const void *A;
    const void *B;
    void *C;
    cudaStream_t stream;
    int sm_count;      // CTAs are planned per SM
    int ctas_per_sm;   // at most this many CTAs per SM (fewer if the registers do not allow them)
    EpiSpec epi;
};

int gemv_launch(const GemvLaunch &L, std::string &err);

// One fp16 product computed as B * A^T on the
// tensor cores with the K range split over CTAs, after validation.
struct SkinnyLaunch {
    int M, N, K;
    const void *A;
    const void *B;
    void *C;
    cudaStream_t stream;
    int ctas;              // CTA count the K split aims for (tiles x shares <= ctas)
    uint64_t timeout_ns;
    EpiSpec epi;           // fused epilogue (epi.on == 0: the plain product)
    int debug_skip_kblock; // test hook: each CTA leaves out this k-block of its share (-1: none)
};

// CTAs of the skinny kernel resident per SM (its default CTA target is this
// times the SM count).
int skinny_ctas_per_sm();

// How a skinny launch spreads the product: `groups` groups of `rows`
// columns of C (rows of B) times `mtiles` tiles of up to 128 rows of A, each
// tile's K range in `splits` shares of `kb_per_split` 64-deep k-blocks (the
// last may be shorter), one CTA per share, a tile's shares one cluster.
struct SkinnyPlan {
    int splits;        // 1, 2, 4 or 8: CTAs of a cluster sharing a tile's K range
    int rows;          // a multiple of 8, at most 128
    int groups;        // ceil(N / rows)
    int kb_per_split;  // k-blocks per share (a share is one CTA)
    int mtiles;        // 1 for M <= 128, else ceil(M / 128)
    int parts = 1;     // clusters per tile: its K range in parts x splits shares
};

// The plan for an M x N product of depth K on `ctas` CTA slots; cap[l] is
// the number of clusters of 2^l CTAs the device holds at once (cap[0] =
// ctas), or cap == nullptr to take ctas / 2^l.  Host logic only.
void skinny_plan(int M, int N, int K, int ctas, const int *cap, SkinnyPlan *plan);

int skinny_launch(const SkinnyLaunch &L, std::string &err);

// Read-and-clear the skinny kernel's device status word (0 = no timeout).
int skinny_status_read_clear(cudaStream_t stream, int *code, std::string &err);

// One SGEMM launch, after validation and selection.
struct SgemmLaunch {
    int M, N, K;
    float alpha, beta;
    const float *A;
    const float *B;
    float *C;
    cudaStream_t stream;
    int variant;   // GEMM_SGEMM_128x128, GEMM_SGEMM_64x64 or GEMM_SGEMM_128x64
    int splits;    // split-K depth, 1 = none (sgemm_split_chunk gives the shares)
};

// Split-K of the SGEMM path: at most this many CTAs share one tile's K.
constexpr int kSgemmMaxSplits = 8;

// K share of each of `splits` CTAs: ceil(K / splits) rounded up to the
// 16-deep k-slice and at least 64 deep; returns how many shares that makes
// (at most `splits`; 1 = no split).
inline int sgemm_split_chunk(int K, int splits, int *chunk) {
    if (splits <= 1 || K <= 0) {
        *chunk = K;
        return 1;
    }
    int c = (K + splits - 1) / splits;
    c = (c + 15) / 16 * 16;
    if (c < 64) c = 64;
    const int eff = (K + c - 1) / c;
    *chunk = eff > 1 ? c : K;
    return eff;
}

int sgemm_launch(const SgemmLaunch &L, std::string &err);

}  // namespace gb300
