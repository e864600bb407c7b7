/*
 * gemm.h -- C ABI of libgemm.so, the GB300 (sm_103a) dense matrix products.
 *
 * Two products, both on row-major, densely packed matrices in device memory:
 *
 *  gemm_f16_nt  C = A * B^T, A half [M,K], B half [N,K], fp32 accumulation,
 *               C half [M,N] (each output rounded to nearest-even once).
 *               Defined by "从零开始的 AI Infra: 算子基础与GPU架构"
 *               (qi-zhan.github.io/blog/2026/cuda-gemm), section "0. Naive
 *               Implementation" (C[m][n] = half(sum_k A[m][k] * B[n][k]) with
 *               a float accumulator) and section "19. 去掉转置" (B stored as
 *               [N,K] row-major is the right operand B^T [K,N] column-major).
 *               Runs on the 5th-generation tensor cores (tcgen05.mma, TMEM
 *               accumulators, TMA-fed 128-byte-swizzled shared-memory tiles).
 *
 *  sgemm        C = alpha * A * B + beta * C, A float [M,K], B float [K,N],
 *               C float [M,N], fp32 arithmetic on the CUDA cores (FFMA; no
 *               TF32).  Defined by "异步拷贝与 Hopper/Blackwell 新特性"
 *               (anrans.github.io/ai-infra-handbooks/cuda/advanced/
 *               async-hopper), section "cp.async 与多级流水 sm_80+": the
 *               gemm_cp_async kernel's epilogue c = alpha*acc + beta*c.
 *
 * Common rules for every entry point below:
 *  - Ownership: all matrix pointers are device memory owned by the caller;
 *    the library keeps no reference after the call returns and allocates no
 *    device memory per call.  One exception: the fp16 pair kernel's split-K
 *    and stream-K partials (see GEMM_F16_FLAG_STREAM_K) live in a workspace
 *    of about 256 KB per CTA pair (19 MiB on a 152-SM GB300), allocated once
 *    per device and stream by the first call that splits and kept for the
 *    life of the process; gemm_f16_nt_stream_k_noalloc never allocates.
 *    Likewise the skinny variant's split over several clusters per tile
 *    (GEMM_F16_SKINNY) keeps its fp32 partial sums in a workspace allocated
 *    once per device and stream (a few hundred KB; not under stream capture).
 *    C must not overlap A or B.
 *  - Asynchrony: work is enqueued on `stream` (a cudaStream_t; NULL means
 *    the legacy default stream) on the calling thread's current device.  The
 *    call returns once the work is enqueued; it does not synchronise.  Stream
 *    order holds: the fp16, matrix-vector and block-scaled kernels are
 *    launched as programmatic dependents, so their set-up (and an L2
 *    prefetch of their first operand boxes, which changes no value) may
 *    overlap the end of the previous kernel on the stream, but they read A
 *    and B and write C only after that kernel has completed.
 *  - Errors: the return value is a gemm_status.  On any non-OK status nothing
 *    was enqueued, and gemm_last_error() gives a message.  Faults found on
 *    the device (a bounded wait inside a kernel that ran out) are reported by
 *    gemm_check_device_status().
 *  - Empty problems: M == 0 or N == 0 is a no-op returning GEMM_OK.
 *  - Per-device state (SM counts, occupancy, workspaces, the static array's
 *    address) is looked up once per device and kept for the CUDA context it
 *    was made in: after cudaDeviceReset on a device, do not call the library
 *    on that device again in the same process.
 */
#ifndef DENSE_GEMM_FP16_GB300_GEMM_H
#define DENSE_GEMM_FP16_GB300_GEMM_H

#include <stddef.h> /* size_t */

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, spelled without including the CUDA headers. */
typedef struct CUstream_st *gemm_stream_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = -1,     /* negative size, NULL pointer with work to do, bad config */
    GEMM_ERR_MISALIGNED = -2,      /* a pointer the fast path needs 16-byte aligned is not   */
    GEMM_ERR_UNSUPPORTED = -3,     /* a shape the path cannot express (see each entry point) */
    GEMM_ERR_CUDA = -4,            /* a CUDA runtime/driver call failed (message has detail) */
    GEMM_ERR_DEVICE_TIMEOUT = -5   /* a kernel's bounded wait expired (device-side status)   */
} gemm_status;

/*
 * C = A * B^T in fp16 with fp32 accumulation.
 *   M, N, K  sizes, each >= 0.  A is [M,K], B is [N,K], C is [M,N]; row
 *            strides are K, K and N elements (packed).
 *   A, B     const half*, 16-byte aligned (they are read by TMA).
 *   C        half*, written; never read.
 * Constraints: K * 2 bytes must be a multiple of 16 (K % 8 == 0), the row
 * stride rule of the tensor-memory-accelerator descriptors; otherwise
 * GEMM_ERR_UNSUPPORTED.  M and N are arbitrary: partial tiles are masked.
 * K == 0 writes C = 0.  When N % 8 == 0 and C is 16-byte aligned the
 * epilogue stores 16-byte vectors, else single halves.
 * Returns GEMM_ERR_INVALID_ARG (negative size, NULL with M*N > 0),
 * GEMM_ERR_MISALIGNED (A or B not 16-byte aligned), GEMM_ERR_UNSUPPORTED,
 * GEMM_ERR_CUDA, or GEMM_OK.
 */
int gemm_f16_nt(int M, int N, int K, const void *A, const void *B, void *C,
                gemm_stream_t stream);

/*
 * C = alpha * A * B + beta * C in fp32 (FFMA only, no TF32).
 *   M, N, K  sizes, each >= 0.  A is [M,K], B is [K,N], C is [M,N], all
 *            row-major and packed.
 *   alpha, beta  scalars.  beta == 0 follows the BLAS convention: C is not
 *            read, so its prior contents (even NaN) do not matter.
 *   A, B     const float*; C float*, read (when beta != 0) and written.
 * Any alignment is accepted: 16-byte vector loads/stores are used where the
 * pointers and row strides allow, scalar ones elsewhere.  K == 0 gives
 * C = beta * C.
 * Returns GEMM_ERR_INVALID_ARG, GEMM_ERR_CUDA, or GEMM_OK.
 */
int sgemm(int M, int N, int K, float alpha, const float *A, const float *B, float beta,
          float *C, gemm_stream_t stream);

/* Message for the last non-OK status returned on this host thread ("" if none).
 * The pointer stays valid until the next call into the library on this thread. */
const char *gemm_last_error(void);

/*
 * Synchronises `stream`, then reads and clears the device-side status word
 * that kernels set when a bounded wait runs out (a pipeline handshake that
 * never completed).  Returns GEMM_OK, GEMM_ERR_DEVICE_TIMEOUT, or
 * GEMM_ERR_CUDA (for an error raised by the synchronisation itself).
 */
int gemm_check_device_status(gemm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Tile and cluster selection.                                               */
/* ------------------------------------------------------------------------ */

/*
 * One kernel configuration of the fp16 path.  `variant` names a compiled
 * instance (GEMM_F16_* below); grid is the persistent CTA count
 * (0 = choose from the device's SM count; for the pair variant it is rounded
 * down to whole pairs and capped by the pairs the device can hold at once).
 * For the skinny variant, grid is instead the number of CTA slots it plans
 * for: C's columns go in groups of 128 and each group's K range in the
 * largest of 2, 4 or 8 shares (a cluster, each share at least 8 k-blocks of
 * 64) with groups x shares <= grid whose clusters the device holds at once,
 * else 1; when the groups alone need more than one wave their height is
 * evened out over the waves (gemm_testing.h exposes the plan).
 */
typedef struct {
    int variant;
    int grid;
    int flags;      /* GEMM_F16_FLAG_* below, 0 for none */
    int raster;     /* tile order: the persistent CTAs walk the output tiles in
                       bands of `raster` tile rows (M), each band column by
                       column, so that a wave's A rows and B columns stay in
                       L2 when the operands do not fit it; 0 = the library's
                       choice, a value >= the tile rows = plain column order */
} gemm_f16_config;

/*
 * Stream-K (pair variant only): when the last round of 256 x 256 tiles would
 * leave many CTA pairs idle, split those tiles' k-blocks evenly over all
 * pairs; a pair that takes over part of a tile's k-range writes its fp32
 * partial to a workspace that the tile's first pair adds in before rounding.
 * The workspace (per device and stream, about 256 KB per CTA pair) is
 * allocated by the library on the first such call on a stream and kept; the
 * split is skipped while the stream is being captured into a graph.  Off by
 * default: on GB300 at the benchmark shapes the partial hand-off costs more
 * than the balanced last round gains.
 *
 * Split-K, by contrast, is on by default in the pair variant, with no flag:
 * when there are so few pair tiles that each would get at least four CTA
 * pairs ("第 6 章 · Shared Memory & Tile", section "6.5.6 Split-K /
 * Stream-K"), every tile's k-blocks are shared over up to 8 pairs (at least
 * 32 k-blocks each) through the same workspace.  The partials are added in a
 * fixed order: results do not depend on timing.  Also skipped under stream
 * capture.  gemm_f16_select sends such shapes to GEMM_F16_SKINNY instead,
 * whose split needs no workspace.
 *
 * Waiting between pairs (stream-K, this split-K and
 * gemm_f16_nt_stream_k_noalloc): a split tile's first pair waits, inside the
 * kernel, for the partials of the pairs that share its k-range, and those
 * always have lower cluster indices than the pair that waits.  The GPU
 * dispatches the clusters of a grid in index order (observed behaviour, not
 * a documented guarantee), so when a long kernel on another stream holds
 * some SMs, the pairs that are running form a prefix of the grid and every
 * pair they wait for is running or done.  Should a wait still not end (a
 * different dispatch order, or a preemption longer than the bound), it gives up
 * after 2 s: the call leaves C partly written and gemm_check_device_status()
 * reports GEMM_ERR_DEVICE_TIMEOUT.  The skinny and SGEMM splits never wait
 * on another CTA's progress outside their own cluster.
 */
#define GEMM_F16_FLAG_STREAM_K 1

enum {
    GEMM_F16_AUTO = 0,          /* let gemm_f16_select decide                     */
    GEMM_F16_128x256 = 1,       /* one CTA per 128 x 256 output tile, 4 stages    */
    GEMM_F16_128x128 = 2,       /* one CTA per 128 x 128 output tile, 6 stages    */
    GEMM_F16_256x256_PAIR = 3,  /* a 2-CTA cluster per 256 x 256 tile (pair MMA,  */
                                /* each CTA 128 rows of A and half of B), 6 stages */
    GEMM_F16_GEMV = 4,          /* M <= 4 (chosen for M = 1): B streamed once from */
                                /* HBM on the CUDA cores, a warp per row block, A  */
                                /* read through L1                                  */
    GEMM_F16_SKINNY = 5,        /* C^T = B A^T on the tensor cores: 128 rows of B  */
                                /* by up to 128 rows of A per tile, K split over a */
                                /* cluster of 2-8 CTAs so the tiles fill the SMs,  */
                                /* the shares added in split order through         */
                                /* distributed shared memory (no workspace; the    */
                                /* tile kernels' numerics).  Chosen for 2 <= M <=  */
                                /* 64, and for any M whose tiles it splits in two  */
                                /* shares of 16+ k-blocks or in four or more.  A   */
                                /* few tiles over a very long K get several 8-CTA  */
                                /* clusters each, their sums added in a fixed      */
                                /* order by the last to finish (a workspace)       */
    GEMM_F16_256x256_QUAD = 6,  /* a 4-CTA cluster of two CTA pairs computing two  */
                                /* vertically adjacent 256 x 256 tiles; each B     */
                                /* byte is loaded once for both (TMA multicast),   */
                                /* a quarter fewer L2 reads and requests; plain     */
                                /* product only (with a fused epilogue the pair    */
                                /* variant runs)                                    */
    GEMM_F16_256x256_KSPLIT = 7,/* a 4-CTA cluster of two CTA pairs computing one  */
                                /* 256 x 256 tile over the two halves of K, the    */
                                /* second pair's fp32 sum added by the first       */
                                /* through distributed shared memory (no           */
                                /* workspace; the sum of the two halves, each in   */
                                /* the pair kernel's order); one tile per cluster. */
                                /* For few tiles over a long K.  Plain product     */
                                /* with K > 64 only: otherwise the pair variant    */
                                /* runs                                             */
    GEMM_F16_NUM_VARIANTS = 8
};

/*
 * Shape-keyed choice of the fp16 configuration: pure host logic, no device
 * call.  sm_count is the number of SMs to plan for (> 0).  The rules, in
 * order: M = 1 takes GEMM_F16_GEMV; 2 <= M <= 64 takes GEMM_F16_SKINNY, and
 * so does any M whose 128 x 128 tiles it splits along K into 2 shares of at
 * least 16 k-blocks or into 4 or more; other M <= 128 take GEMM_F16_128x128;
 * larger M take the tile (128 x 128, 128 x 256 or the CTA pair) whose waves
 * over the SMs cost least, a wave of the wider tiles counting 1.15 / 1.1
 * waves of 128 x 128 tiles (1.5 / 1.5 when K <= 512).  When that is the pair
 * and K % 64 != 0 (rows of A and B not a whole number of 128-byte lines, so
 * every TMA row spans two L2 lines) with M > 256, GEMM_F16_256x256_QUAD
 * replaces it.  From 256 rows, when K % 64 == 0, K >= 8192 and the 256 x 256
 * tiles number more than half and at most all of the 4-CTA clusters that fit
 * at once (sm_count / 4 - 2 of them), GEMM_F16_256x256_KSPLIT takes the
 * product instead.
 * Fills *cfg and returns GEMM_OK, or GEMM_ERR_INVALID_ARG.
 */
int gemm_f16_select(int M, int N, int K, int sm_count, gemm_f16_config *cfg);

/* gemm_f16_nt with an explicit configuration (cfg == NULL or variant AUTO
 * means the selector's choice; grid 0 means the default grid; flags as
 * above).  Same argument rules and errors as gemm_f16_nt, plus
 * GEMM_ERR_INVALID_ARG for an unknown variant or flag. */
int gemm_f16_nt_ex(int M, int N, int K, const void *A, const void *B, void *C,
                   gemm_stream_t stream, const gemm_f16_config *cfg);

/*
 * gemm_f16_nt computed without any device-memory allocation by the library.
 * The pages have no counterpart: this entry point exists for callers that
 * cannot let a library call cudaMalloc -- servers that reserve their whole
 * device-memory budget in their own pool up front (a later cudaMalloc may
 * fail or break the budget), latency-critical paths (cudaMalloc and cudaFree
 * can synchronise the device and stall other streams), and frameworks whose
 * allocator must account for every byte.
 *
 * It runs the CTA-pair kernel (GEMM_F16_256x256_PAIR) with the stream-K split
 * of GEMM_F16_FLAG_STREAM_K, but keeps the partial tiles and flags in a static
 * array inside the library (19.0 MiB of device memory, enough for 76 CTA
 * pairs; every GPU that loads the library holds it until the process exits)
 * instead of a workspace it allocates.  The caller passes A, B and C exactly as
 * for gemm_f16_nt, with the same argument rules, and gets the same result up to
 * the order of the fp32 additions.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.
 *
 * Sharing: every call on a device uses the same array and leaves its contents
 * behind; each call tags its flags with a fresh sequence number, so nothing
 * has to be cleared between calls.  Calls whose kernels overlap on the GPU
 * (for example on two streams at once) race on the array and must not be
 * made; calls on one stream never overlap.
 *
 * Size limit: the array holds partial slots for 76 CTA pairs; on a device
 * that could run more pairs at once, the call runs 76 persistent pairs.
 *
 * Errors: as gemm_f16_nt, plus GEMM_ERR_UNSUPPORTED for a device id of 64 or
 * more (the library keeps the array's address for devices 0..63).
 */
int gemm_f16_nt_stream_k_noalloc(int M, int N, int K, const void *A, const void *B, void *C,
                                 gemm_stream_t stream);

/* Activation applied by the fused epilogue of gemm_f16_nt_fused. */
enum {
    GEMM_ACT_NONE = 0,
    GEMM_ACT_RELU = 1,       /* max(v, 0)                                              */
    GEMM_ACT_SILU = 2,       /* v / (1 + exp(-v))                                      */
    GEMM_ACT_GELU_TANH = 3,  /* 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))        */
    GEMM_ACT_NUM = 4
};

/* The fused epilogue: every output is
 *     C[m][n] = half_rn( act( alpha * sum_k A[m][k] B[n][k] + bias[n] + beta * residual[m][n] ) )
 * computed in fp32 from the fp32 accumulators, rounded to half once.
 *   bias      device pointer to N halves, or NULL (no bias term);
 *   residual  device pointer to an M x N row-major half matrix, or NULL; it is
 *             read only when beta != 0 and it MAY be C itself (each output
 *             reads its own residual before it is written, so in-place
 *             C = act(alpha*A*B^T + beta*C) works);
 *   activation  one of GEMM_ACT_*.
 * Bias and residual need no alignment; when both are 16-byte aligned and
 * N % 8 == 0 they are read as 16-byte vectors. */
typedef struct {
    float alpha;
    float beta;
    const void *bias;
    const void *residual;
    int activation;
} gemm_f16_epilogue;

/* gemm_f16_nt with the product passed through a fused epilogue before the
 * single rounding to half ("第 6 章 · Shared Memory & Tile", section "6.5.4
 * Epilogue 融合": bias and activation applied while the accumulators are on
 * chip, so C makes one trip to HBM instead of three).  Same arguments, layout,
 * validation and kernel choice as gemm_f16_nt_ex (cfg may be NULL); epi NULL
 * is the plain product.  epi->activation outside GEMM_ACT_* returns
 * GEMM_ERR_INVALID_ARG.  K == 0 gives act(bias + beta * residual). */
int gemm_f16_nt_fused(int M, int N, int K, const void *A, const void *B, void *C,
                      const gemm_f16_epilogue *epi, gemm_stream_t stream,
                      const gemm_f16_config *cfg);

/* Block-scaled FP8 (MXFP8) product, C = A_s * B_s^T with
 *     A_s[m][k] = e4m3(A[m][k]) * 2^(SA[m][k/32] - 127),
 *     B_s[n][k] = e4m3(B[n][k]) * 2^(SB[n][k/32] - 127),
 * accumulated in fp32 on the tensor cores and rounded once to half ("异步拷贝与
 * Hopper/Blackwell 新特性", section "Blackwell 概览 sm_100": in MXFP8 every 32
 * elements share one 8-bit exponent scale).
 *   A    device, M x K bytes, row-major: FP8 E4M3 codes (1 sign, 4 exponent
 *        bits with bias 7, 3 mantissa bits; S.1111.111 is NaN);
 *   B    device, N x K bytes, row-major (the transposed right operand, as in
 *        gemm_f16_nt);
 *   SFA, SFB  device, the UE8M0 scale codes (2^(e - 127)) of A and B in the
 *        chunk layout below, gemm_mxfp8_scale_bytes(M or N, K) bytes each;
 *   C    device, half M x N, row-major.
 * Scale chunk layout: for a matrix of `rows` rows, rows are grouped in tiles
 * of 128 and K in blocks of 128 (4 scales); chunk (t, b) is 512 bytes at
 * offset (t * ceil(K/128) + b) * 512, and byte 16*(r % 32) + 4*(r / 32) + j of
 * it holds the scale of row 128t + r for K elements 128b + 32j .. +31.
 * Entries past the last row or scale must be finite codes (the packer writes
 * 127).  gemm_mxfp8_pack_scales converts plain [rows][K/32] scales.
 * K must be a multiple of 32 (GEMM_ERR_UNSUPPORTED otherwise); A, B, SFA and
 * SFB 16-byte aligned (GEMM_ERR_MISALIGNED).  K = 0 writes C = 0. */
int gemm_mxfp8_nt(int M, int N, int K, const void *A, const void *SFA, const void *B,
                  const void *SFB, void *C, gemm_stream_t stream);

/* One kernel configuration of the MXFP8 path. */
typedef struct {
    int variant;
    int grid;  /* CTAs (a multiple of 2 for the pair kernel); 0 = one per SM */
} gemm_mxfp8_config;

enum {
    GEMM_MXFP8_AUTO = 0,
    GEMM_MXFP8_128x128 = 1,       /* 1-CTA 128 x 128 tiles, 5 stages (default for N <= 128) */
    GEMM_MXFP8_256x128_PAIR = 2,  /* CTA pair (cta_group::2) 256 x 128 tiles, 7 stages
                                     (NVFP4: 6)                                            */
    GEMM_MXFP8_128x256 = 3,       /* 1-CTA 128 x 256 tiles, N = 256 MMAs, one accumulator
                                     that 8 epilogue warps release from registers, 4 stages
                                     (NVFP4: 3); default for N > 128                        */
    GEMM_MXFP8_256x256_PAIR = 4,  /* CTA pair 256 x 256 tiles, one accumulator released by
                                     8 epilogue warps, 6 stages (NVFP4: 5)                  */
    GEMM_MXFP8_NUM_VARIANTS = 5
};

/* gemm_mxfp8_nt with an explicit kernel configuration (NULL or AUTO: the
 * library's choice). */
int gemm_mxfp8_nt_ex(int M, int N, int K, const void *A, const void *SFA, const void *B,
                     const void *SFB, void *C, gemm_stream_t stream, const gemm_mxfp8_config *cfg);

/* Bytes of the chunk layout of the scales of a `rows` x K MXFP8 matrix:
 * ceil(rows/128) * ceil(K/128) * 512.  0 for an empty matrix. */
size_t gemm_mxfp8_scale_bytes(int rows, int K);

/* Device-side conversion of plain row-major UE8M0 scales [rows][K/32]
 * (`plain`) into the chunk layout (`blocked`, gemm_mxfp8_scale_bytes(rows,
 * K) bytes), padding with 127; enqueued on `stream`.  K % 32 != 0 ->
 * GEMM_ERR_UNSUPPORTED. */
int gemm_mxfp8_pack_scales(int rows, int K, const void *plain, void *blocked, gemm_stream_t stream);

/* Block-scaled FP4 (NVFP4) product, C = alpha * A_s * B_s^T with
 *     A_s[m][k] = e2m1(A, m, k) * e4m3(SA[m][k/16]),
 *     B_s[n][k] = e2m1(B, n, k) * e4m3(SB[n][k/16]),
 * accumulated in fp32 on the tensor cores (tcgen05.mma kind::mxf4nvf4,
 * block_scale, scale_vec::4X) and rounded once to half ("异步拷贝与
 * Hopper/Blackwell 新特性", section "Blackwell 概览 sm_100": in NVFP4 every 16
 * elements share one FP8 scale, plus a tensor-level FP32 scale).
 *   A    device, M x K/2 bytes, row-major: FP4 E2M1 codes (1 sign, 2 exponent
 *        bits with bias 1, 1 mantissa bit), two per byte, element 2i of a
 *        row in the low 4 bits of byte i;
 *   B    device, N x K/2 bytes, row-major (the transposed right operand);
 *   SFA, SFB  device, the E4M3 block scales (positive codes) of A and B in
 *        the chunk layout below, gemm_nvfp4_scale_bytes(M or N, K) bytes each;
 *   alpha  the tensor-level scale (the product of A's and B's);
 *   C    device, half M x N, row-major.
 * Scale chunk layout: rows in tiles of 128, K in blocks of 256 split into four
 * 64-element chunks; chunk (t, c) (c counts 64-element blocks, 4 per 256)
 * is 512 bytes at offset (t * 4 * ceil(K/256) + c) * 512, and byte
 * 16*(r % 32) + 4*(r / 32) + j of it holds the scale of row 128t + r for K
 * elements 64c + 16j .. +15.  Entries past the last row or scale must be
 * finite (the packer writes 0x38 = 1.0).  gemm_nvfp4_pack_scales converts
 * plain [rows][K/16] scales.  K must be a multiple of 32
 * (GEMM_ERR_UNSUPPORTED otherwise); A, B, SFA and SFB 16-byte aligned
 * (GEMM_ERR_MISALIGNED).  K = 0 writes C = 0. */
int gemm_nvfp4_nt(int M, int N, int K, const void *A, const void *SFA, const void *B,
                  const void *SFB, float alpha, void *C, gemm_stream_t stream);

/* gemm_nvfp4_nt with a kernel configuration: any GEMM_MXFP8_* variant
 * (the same tile shapes, with four scale chunks per 128 rows per 256 of K). */
int gemm_nvfp4_nt_ex(int M, int N, int K, const void *A, const void *SFA, const void *B,
                     const void *SFB, float alpha, void *C, gemm_stream_t stream,
                     const gemm_mxfp8_config *cfg);

/* Bytes of the NVFP4 scale chunk layout: ceil(rows/128) * 4 * ceil(K/256) * 512. */
size_t gemm_nvfp4_scale_bytes(int rows, int K);

/* Device-side conversion of plain [rows][K/16] E4M3 scales into the chunk
 * layout (padding 0x38), enqueued on `stream`.  K % 32 != 0 ->
 * GEMM_ERR_UNSUPPORTED. */
int gemm_nvfp4_pack_scales(int rows, int K, const void *plain, void *blocked, gemm_stream_t stream);

/* One kernel configuration of the SGEMM path.  splits: how many CTAs share
 * each tile's K (split-K, "第 6 章 · Shared Memory & Tile", section "6.5.6
 * Split-K / Stream-K"): 0 = the library's choice (gemm_sgemm_select), 1 =
 * never, 2..8 = that many (each share at least 64 deep, so fewer when K is
 * short).  variant 0 with splits n picks the tile for that split count.
 * The last CTA of a tile adds the
 * shares in a fixed order, so results do not depend on timing.  The partials
 * live in a workspace allocated once per device and stream (the first call
 * that splits) and kept; under stream capture a split that would need it is
 * not taken. */
typedef struct {
    int variant;
    int splits;
} gemm_sgemm_config;

enum {
    GEMM_SGEMM_AUTO = 0,
    GEMM_SGEMM_128x128 = 1,     /* 128 x 128 CTA tile, 8 x 16 per thread, BK 16, 3 stages */
    GEMM_SGEMM_64x64 = 2,       /* 64 x 64 CTA tile, 4 x 4 per thread, BK 16, 3 stages   */
    GEMM_SGEMM_128x64 = 3,      /* 128 x 64 CTA tile, 8 x 8 per thread, BK 16, 3 stages  */
    GEMM_SGEMM_NUM_VARIANTS = 4
};

/* Shape-keyed choice of the SGEMM tile (128 x 128, 64 x 64 or 128 x 64) and
 * split count (host logic only): the pair with the lowest predicted time,
 * where a launch takes as long as its busiest SM (ceil(CTAs / sm_count) CTAs,
 * each over its K share) plus the cost of adding the split partials.  Splits are only considered when the
 * tiles number at most 2 * sm_count.  Fills cfg->variant and cfg->splits
 * (>= 1). */
int gemm_sgemm_select(int M, int N, int K, int sm_count, gemm_sgemm_config *cfg);

/* sgemm with an explicit configuration (NULL or AUTO = selector's choice). */
int sgemm_ex(int M, int N, int K, float alpha, const float *A, const float *B, float beta,
             float *C, gemm_stream_t stream, const gemm_sgemm_config *cfg);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_FP16_GB300_GEMM_H */
