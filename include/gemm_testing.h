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
 * selector picks the skinny variant (2 <= M <= 64), every CTA leaves out
 * k-block `skip_kblock` of its own share of K instead, so the CTAs of a split
 * cluster all give up and still meet at the cluster barriers.
 */
int gemm_debug_f16_nt_skip_load(int M, int N, int K, const void *A, const void *B, void *C,
                                gemm_stream_t stream, int skip_kblock,
                                unsigned long long timeout_ns);

/*
 * The K split the skinny fp16 variant (GEMM_F16_SKINNY) plans for a product
 * with N columns of C and depth K, aiming at `ctas` CTAs: pure host logic,
 * no device call.  Returns the shares of K per 128-column tile (1, 2, 4 or 8:
 * the largest power of two with tiles x shares <= ctas and at least 8
 * k-blocks of 64 per share; 1 when none fits) and stores the k-blocks per
 * share in *kb_per_split (the last share may be shorter).  The launch halves
 * the shares further while the device cannot hold all the clusters at once.
 * Returns -1 for N < 1, K < 0, ctas < 1 or a NULL kb_per_split.
 */
int gemm_debug_skinny_split_plan(int N, int K, int ctas, int *kb_per_split);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_FP16_GB300_GEMM_TESTING_H */
