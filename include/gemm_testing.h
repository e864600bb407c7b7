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
 * partially written.  Same argument rules as gemm_f16_nt.
 */
int gemm_debug_f16_nt_skip_load(int M, int N, int K, const void *A, const void *B, void *C,
                                gemm_stream_t stream, int skip_kblock,
                                unsigned long long timeout_ns);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_FP16_GB300_GEMM_TESTING_H */
