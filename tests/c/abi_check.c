/*
 * abi_check.c -- a plain C99 caller of libgemm.so, built against include/gemm.h
 * and include/gemm_testing.h with gcc -std=c99 -Wall -Wextra -Werror.
 *
 *   abi_check host
 *       Host-only calls (no device needed): the selectors, the scale-layout
 *       sizes, the skinny plan and the argument checks.  Prints key=value
 *       lines for the Python side to compare with its own calls; exits
 *       non-zero if a call breaks its documented contract.
 *
 *   abi_check gpu DIR
 *       DIR/params.txt holds "M N K Ms Ns Ks alpha beta".  Reads half
 *       DIR/A.bin [M,K] and DIR/B.bin [N,K], float DIR/As.bin [Ms,Ks],
 *       DIR/Bs.bin [Ks,Ns] and DIR/C0.bin [Ms,Ns]; runs gemm_f16_nt and sgemm
 *       on cudaMalloc'd buffers (the legacy default stream), checks
 *       gemm_check_device_status, and writes DIR/C.bin (half [M,N]) and
 *       DIR/Cs.bin (float [Ms,Ns]).
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "gemm.h"
#include "gemm_testing.h"

static int failures = 0;

#define EXPECT(cond, ...)                                   \
    do {                                                    \
        if (!(cond)) {                                      \
            fprintf(stderr, "FAILED %s: ", #cond);          \
            fprintf(stderr, __VA_ARGS__);                   \
            fprintf(stderr, "\n");                          \
            ++failures;                                     \
        }                                                   \
    } while (0)

static int host_checks(void)
{
    gemm_f16_config f;
    gemm_sgemm_config s;
    int st, rows = 0, groups = 0, kb = 0, splits;

    memset(&f, 0, sizeof f);
    st = gemm_f16_select(5376, 5376, 2048, 152, &f);
    EXPECT(st == GEMM_OK, "gemm_f16_select status %d", st);
    printf("f16_select_5376x5376x2048=%d,%d,%d\n", f.variant, f.grid, f.raster);
    st = gemm_f16_select(1, 16384, 8192, 152, &f);
    EXPECT(st == GEMM_OK && f.variant == GEMM_F16_GEMV, "M = 1 takes the GEMV (%d, %d)", st, f.variant);
    printf("f16_select_1x16384x8192=%d,%d,%d\n", f.variant, f.grid, f.raster);
    st = gemm_f16_select(-1, 4, 8, 152, &f);
    EXPECT(st == GEMM_ERR_INVALID_ARG, "negative M in the selector: %d", st);

    memset(&s, 0, sizeof s);
    st = gemm_sgemm_select(4096, 4096, 4096, 152, &s);
    EXPECT(st == GEMM_OK && s.splits >= 1, "gemm_sgemm_select status %d splits %d", st, s.splits);
    printf("sgemm_select_4096=%d,%d\n", s.variant, s.splits);
    st = gemm_sgemm_select(256, 256, 256, 152, &s);
    EXPECT(st == GEMM_OK, "gemm_sgemm_select(256^3) status %d", st);
    printf("sgemm_select_256=%d,%d\n", s.variant, s.splits);

    /* argument checks return before any device work */
    st = gemm_f16_nt(-1, 4, 8, NULL, NULL, NULL, NULL);
    EXPECT(st == GEMM_ERR_INVALID_ARG, "gemm_f16_nt(M = -1) returned %d", st);
    EXPECT(gemm_last_error() != NULL && strlen(gemm_last_error()) > 0, "empty gemm_last_error");
    printf("f16_negative_m=%d:%s\n", st, gemm_last_error());
    st = sgemm(4, -2, 4, 1.0f, NULL, NULL, 0.0f, NULL, NULL);
    EXPECT(st == GEMM_ERR_INVALID_ARG, "sgemm(N = -2) returned %d", st);
    printf("sgemm_negative_n=%d:%s\n", st, gemm_last_error());
    st = gemm_f16_nt(0, 4, 8, NULL, NULL, NULL, NULL);
    EXPECT(st == GEMM_OK, "an empty product is a no-op: %d", st);

    splits = gemm_debug_skinny_plan(16, 16384, 8192, 152, &rows, &groups, &kb);
    EXPECT(splits >= 1 && rows > 0 && groups > 0, "skinny plan %d %d %d %d", splits, rows, groups, kb);
    printf("skinny_plan_16x16384x8192=%d,%d,%d,%d\n", splits, rows, groups, kb);
    EXPECT(gemm_debug_skinny_plan(0, 1, 1, 1, &rows, &groups, &kb) == -1, "bad plan arguments");

    printf("mxfp8_scale_bytes_5376x2048=%zu\n", gemm_mxfp8_scale_bytes(5376, 2048));
    printf("nvfp4_scale_bytes_5376x2048=%zu\n", gemm_nvfp4_scale_bytes(5376, 2048));
    EXPECT(gemm_mxfp8_scale_bytes(0, 2048) == 0, "empty matrix scale bytes");
    return failures == 0 ? 0 : 1;
}

/* ---------------------------------------------------------------------- */
/* gpu mode: the CUDA runtime for device memory only                        */
/* ---------------------------------------------------------------------- */
#ifdef ABI_CHECK_GPU
#include <cuda_runtime_api.h>

static void *read_file(const char *dir, const char *name, size_t bytes)
{
    char path[1024];
    FILE *f;
    void *p = malloc(bytes ? bytes : 1);
    snprintf(path, sizeof path, "%s/%s", dir, name);
    f = fopen(path, "rb");
    if (!f || !p || fread(p, 1, bytes, f) != bytes) {
        fprintf(stderr, "cannot read %zu bytes from %s\n", bytes, path);
        exit(2);
    }
    fclose(f);
    return p;
}

static void write_file(const char *dir, const char *name, const void *p, size_t bytes)
{
    char path[1024];
    FILE *f;
    snprintf(path, sizeof path, "%s/%s", dir, name);
    f = fopen(path, "wb");
    if (!f || fwrite(p, 1, bytes, f) != bytes) {
        fprintf(stderr, "cannot write %s\n", path);
        exit(2);
    }
    fclose(f);
}

static void *to_device(const void *h, size_t bytes)
{
    void *d = NULL;
    if (cudaMalloc(&d, bytes ? bytes : 16) != cudaSuccess ||
        cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
        fprintf(stderr, "device upload of %zu bytes failed\n", bytes);
        exit(2);
    }
    return d;
}

static int gpu_checks(const char *dir)
{
    char path[1024];
    FILE *f;
    int M, N, K, Ms, Ns, Ks, st;
    float alpha, beta;
    size_t a_b, b_b, c_b, as_b, bs_b, cs_b;
    void *hA, *hB, *hAs, *hBs, *hC0, *hC, *hCs, *dA, *dB, *dC, *dAs, *dBs, *dCs;

    snprintf(path, sizeof path, "%s/params.txt", dir);
    f = fopen(path, "r");
    if (!f || fscanf(f, "%d %d %d %d %d %d %f %f", &M, &N, &K, &Ms, &Ns, &Ks, &alpha, &beta) != 8) {
        fprintf(stderr, "cannot parse %s\n", path);
        return 2;
    }
    fclose(f);
    a_b = (size_t)M * K * 2;
    b_b = (size_t)N * K * 2;
    c_b = (size_t)M * N * 2;
    as_b = (size_t)Ms * Ks * 4;
    bs_b = (size_t)Ks * Ns * 4;
    cs_b = (size_t)Ms * Ns * 4;
    hA = read_file(dir, "A.bin", a_b);
    hB = read_file(dir, "B.bin", b_b);
    hAs = read_file(dir, "As.bin", as_b);
    hBs = read_file(dir, "Bs.bin", bs_b);
    hC0 = read_file(dir, "C0.bin", cs_b);
    dA = to_device(hA, a_b);
    dB = to_device(hB, b_b);
    dAs = to_device(hAs, as_b);
    dBs = to_device(hBs, bs_b);
    dCs = to_device(hC0, cs_b);
    if (cudaMalloc(&dC, c_b) != cudaSuccess) return 2;

    st = gemm_f16_nt(M, N, K, dA, dB, dC, NULL);
    EXPECT(st == GEMM_OK, "gemm_f16_nt: %d %s", st, gemm_last_error());
    st = sgemm(Ms, Ns, Ks, alpha, (const float *)dAs, (const float *)dBs, beta, (float *)dCs, NULL);
    EXPECT(st == GEMM_OK, "sgemm: %d %s", st, gemm_last_error());
    st = gemm_check_device_status(NULL);
    EXPECT(st == GEMM_OK, "gemm_check_device_status: %d %s", st, gemm_last_error());

    hC = malloc(c_b);
    hCs = malloc(cs_b);
    if (!hC || !hCs || cudaMemcpy(hC, dC, c_b, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(hCs, dCs, cs_b, cudaMemcpyDeviceToHost) != cudaSuccess) {
        fprintf(stderr, "device download failed\n");
        return 2;
    }
    write_file(dir, "C.bin", hC, c_b);
    write_file(dir, "Cs.bin", hCs, cs_b);
    cudaFree(dA);
    cudaFree(dB);
    cudaFree(dC);
    cudaFree(dAs);
    cudaFree(dBs);
    cudaFree(dCs);
    free(hA);
    free(hB);
    free(hAs);
    free(hBs);
    free(hC0);
    free(hC);
    free(hCs);
    return failures == 0 ? 0 : 1;
}
#endif

int main(int argc, char **argv)
{
    if (argc >= 2 && strcmp(argv[1], "host") == 0) return host_checks();
#ifdef ABI_CHECK_GPU
    if (argc >= 3 && strcmp(argv[1], "gpu") == 0) return gpu_checks(argv[2]);
#endif
    fprintf(stderr, "usage: %s host | gpu DIR\n", argv[0]);
    return 2;
}
