/*
 * gemm_testing.h -- test hooks exported by libgemm.so in addition to the
 * public C ABI of gemm.h.  Not for production callers.
 */
#ifndef DENSE_GEMM_FP16_GB300_GEMM_TESTING_H
#define DENSE_GEMM_FP16_GB300_GEMM_TESTING_H

#include "gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * gemm_f16_nt with one TMA load deliberately left out: the producer skips
 * k-block `skip_kblock` of the first tile each CTA processes, so the MMA
 * issuer's wait for that shared-memory stage can never succeed.  Every wait in
 * the kernel is bounded by `timeout_ns`; on expiry the kernel records a status
 * code, stops its other roles, lets the copies and MMAs it already issued
 * finish, frees its Tensor Memory and exits.  The launch itself returns
 * GEMM_OK; the fault is then reported by gemm_check_device_status() as
 * GEMM_ERR_DEVICE_TIMEOUT and the CUDA context stays usable.  C is left
 * partially written.  Same argument rules as gemm_f16_nt.  When the
 * selector picks the skinny variant (2 <= M <= 128), every CTA leaves out
 * k-block `skip_kblock` of its own share of K instead, so the CTAs of a split
 * cluster all give up and still meet at the cluster barriers.
 */
int gemm_debug_f16_nt_skip_load(int M, int N, int K, const void *A, const void *B, void *C,
                                gemm_stream_t stream, int skip_kblock,
                                unsigned long long timeout_ns);

/*
 * How the skinny fp16 variant (GEMM_F16_SKINNY) spreads an M x N product of
 * depth K over `ctas` CTA slots: pure host logic, no device call, assuming
 * every slot can hold a cluster of each size (the launch uses the device's
 * own cluster counts).  A's rows go in tiles of 128 (one tile for M <= 128),
 * C's columns in *groups groups of *rows (128, or, when M <= 128 and 128-row
 * groups need more than one wave, the multiple of 8 that fills every wave
 * evenly); each tile's K range in the returned number of shares (the largest
 * of 2, 4, 8 with tiles x shares <= ctas and at least 8 k-blocks of 64 a
 * share, else 1) of *kb_per_split k-blocks, one CTA per share.  Returns -1
 * for M < 1, N < 1, K < 0, ctas < 1 or a NULL output pointer.
 */
int gemm_debug_skinny_plan(int M, int N, int K, int ctas, int *rows, int *groups, int *kb_per_split);

/*
 * How many clusters the same plan gives each tile: when even 8-CTA clusters
 * leave most slots idle, each tile's K range goes to several clusters
 * (parts), as many as the slots hold at once, at most 8, each share still at
 * least 8 k-blocks; *kb_per_split above is then per share of parts x 8.  The
 * parts' fp32 sums meet in a workspace the library allocates per device and
 * stream (skipped under stream capture, where each tile keeps one cluster).
 * Returns the parts (1 = one cluster per tile), or -1 for bad arguments.
 */
int gemm_debug_skinny_parts(int M, int N, int K, int ctas);

/*
 * A block-scaled product (fmt 0: gemm_mxfp8_nt_ex, 1: gemm_nvfp4_nt_ex with
 * alpha = 1) with one k-block deliberately never loaded: each CTA (the even
 * CTA of each pair, for the pair variants) neither arms nor loads k-block
 * `skip_kblock` of the first tile it processes, so the MMA issuer's wait for
 * that stage can never succeed.  Every wait is bounded by `timeout_ns`; the
 * kernel then records a status code, drains its own copies and MMAs, frees
 * its Tensor Memory and exits, and gemm_check_device_status() reports
 * GEMM_ERR_DEVICE_TIMEOUT.  C is left partially written.  Same argument rules
 * as gemm_mxfp8_nt_ex / gemm_nvfp4_nt_ex (cfg may be NULL), plus
 * GEMM_ERR_INVALID_ARG for another fmt.
 */
int gemm_debug_blockscaled_skip_load(int fmt, int M, int N, int K, const void *A, const void *SFA,
                                     const void *B, const void *SFB, void *C, gemm_stream_t stream,
                                     const gemm_mxfp8_config *cfg, int skip_kblock,
                                     unsigned long long timeout_ns);

/*
 * gemm_f16_nt_ex on the CTA-pair variant with GEMM_F16_FLAG_STREAM_K, where
 * every pair that takes over part of a tile's k-range writes its fp32
 * partial but never flags it ready.  The tile's first pair then waits for
 * the flags until its bounded wait (`timeout_ns`) runs out, and
 * gemm_check_device_status() reports GEMM_ERR_DEVICE_TIMEOUT.  Whether the
 * launch splits at all follows the stream-K rule (gemm_debug_last_pair_launch
 * tells); the shape must have a partial last round of 256 x 256 tiles.
 */
int gemm_debug_f16_nt_stream_k_skip_publish(int M, int N, int K, const void *A, const void *B, void *C,
                                            gemm_stream_t stream, unsigned long long timeout_ns);

/*
 * How the last launch of the CTA-pair kernel (GEMM_F16_256x256_PAIR) made on
 * the calling host thread split its work: *pairs CTA pairs, *whole_tiles
 * 256 x 256 tiles computed whole, *shared_units k-blocks of 64 shared out
 * over the pairs (stream-K or split-K; 0 when nothing was split), and where
 * the fp32 partials of the shared tiles went: *scratch_kind 0 nowhere, 1 the
 * workspace the library allocates per device and stream, 2 the static array
 * of gemm_f16_nt_stream_k_noalloc.  Host state only, no device call.
 * Returns 0, or -1 (outputs untouched) when no pair launch has been made on
 * this thread or an output pointer is NULL.
 */
int gemm_debug_last_pair_launch(int *pairs, int *whole_tiles, int *shared_units, int *scratch_kind);

/*
 * A clock sample for measurement: launches `ctas` CTAs of 32 threads on
 * `stream`; thread 0 of CTA b writes out[3b] = the SM it ran on (%smid),
 * out[3b + 1] = that SM's cycle counter (clock64) and out[3b + 2] = the
 * global nanosecond timer (%globaltimer), read back to back.  Two samples
 * enqueued around a stretch of work give each SM seen in both its mean clock
 * over that stretch: the cycle difference over the nanosecond difference.
 * Which SMs the CTAs land on is up to the hardware; twice the SM count of
 * CTAs usually reaches every SM.  `out`: caller-owned device memory of
 * 3 * ctas 64-bit words, 8-byte aligned.  Returns GEMM_OK,
 * GEMM_ERR_INVALID_ARG (ctas outside 1..65535, out NULL or misaligned;
 * nothing enqueued) or GEMM_ERR_CUDA (the launch failed).
 */
int gemm_debug_sm_clocks(unsigned long long *out, int ctas, gemm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_FP16_GB300_GEMM_TESTING_H */
