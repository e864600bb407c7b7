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

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_FP16_GB300_GEMM_TESTING_H */
