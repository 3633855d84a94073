/*
 * The C ABI used from plain C (C99): the three public headers compile as C,
 * and a program that owns its device memory through the CUDA runtime calls
 * gemm_create / gemm_run / gemm_run_host / gemm_sync_status / gemm_destroy.
 * Inputs are small integers, so every product and sum is exact in FP32 and
 * the result must equal an integer triple loop bit for bit.
 *
 * Build: gcc -std=c99 -Wall -Werror -I include -isystem <cuda>/include \
 *        gemm_abi_check.c -L <lib dir> -ldense_gemm_gb300 -L <cuda>/lib64 -lcudart
 * Exit status 0 and "C ABI OK" on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "gemm.h"
#include "gemm_ladder.h"
#include "gemm_peaks.h"

static float value(int64_t i, int64_t j, int salt)
{
    return (float)(((i * 7 + j * 13 + salt * 5) % 17) - 8); /* integers in [-8, 8] */
}

static int check(const char *what, const float *C, int64_t M, int64_t N, int64_t K, const float *A,
                 const float *Bl)
{
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            int64_t s = 0;
            for (int64_t k = 0; k < K; ++k) s += (int64_t)A[i * K + k] * (int64_t)Bl[k * N + j];
            if (C[i * N + j] != (float)s) {
                fprintf(stderr, "%s: C[%lld][%lld] = %g, expected %lld\n", what, (long long)i, (long long)j,
                        (double)C[i * N + j], (long long)s);
                return 1;
            }
        }
    return 0;
}

int main(void)
{
    const int64_t M = 300, N = 260, K = 200;
    float *A = malloc(sizeof(float) * M * K), *Bl = malloc(sizeof(float) * K * N);
    float *Bc = malloc(sizeof(float) * N * K), *C = malloc(sizeof(float) * M * N);
    if (!A || !Bl || !Bc || !C) return 2;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t k = 0; k < K; ++k) A[i * K + k] = value(i, k, 1);
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < N; ++j) {
            Bl[k * N + j] = value(k, j, 2);
            Bc[j * K + k] = Bl[k * N + j]; /* the same logical B, column-major */
        }

    gemm_handle_t h = NULL;
    int rc = gemm_create(&h, 0);
    if (rc != GEMM_OK) {
        fprintf(stderr, "gemm_create: %s\n", gemm_status_string(rc));
        return 1;
    }
    float *dA, *dB, *dC;
    if (cudaMalloc((void **)&dA, sizeof(float) * M * K) != cudaSuccess ||
        cudaMalloc((void **)&dB, sizeof(float) * K * N) != cudaSuccess ||
        cudaMalloc((void **)&dC, sizeof(float) * M * N) != cudaSuccess)
        return 1;
    cudaMemcpy(dA, A, sizeof(float) * M * K, cudaMemcpyHostToDevice);
    int fails = 0;
    const int modes[3] = {GEMM_F32, GEMM_TF32, GEMM_F32};
    for (int t = 0; t < 3; ++t) {
        const int layout = t == 2 ? GEMM_B_COL_MAJOR : GEMM_B_ROW_MAJOR;
        cudaMemcpy(dB, layout == GEMM_B_ROW_MAJOR ? Bl : Bc, sizeof(float) * K * N, cudaMemcpyHostToDevice);
        cudaMemset(dC, 0xff, sizeof(float) * M * N);
        rc = gemm_run(h, layout, M, N, K, dA, K, dB, layout == GEMM_B_ROW_MAJOR ? N : K, dC, N, modes[t], 0);
        if (rc == GEMM_OK) rc = gemm_sync_status(h, 0);
        if (rc != GEMM_OK) {
            fprintf(stderr, "gemm_run: %s (%s)\n", gemm_status_string(rc), gemm_last_error_string(h));
            return 1;
        }
        cudaMemcpy(C, dC, sizeof(float) * M * N, cudaMemcpyDeviceToHost);
        fails += check(gemm_last_path(h), C, M, N, K, A, Bl);
    }
    /* host buffers (pageable here) */
    for (int64_t i = 0; i < M * N; ++i) C[i] = -1.0f;
    rc = gemm_run_host(h, GEMM_B_COL_MAJOR, M, N, K, A, K, Bc, K, C, N, GEMM_F32, 0);
    if (rc == GEMM_OK) rc = gemm_sync_status(h, 0);
    if (rc != GEMM_OK) {
        fprintf(stderr, "gemm_run_host: %s\n", gemm_status_string(rc));
        return 1;
    }
    fails += check(gemm_last_path(h), C, M, N, K, A, Bl);
    /* argument errors come back as codes */
    if (gemm_run(h, 2, M, N, K, dA, K, dB, N, dC, N, GEMM_F32, 0) != GEMM_ERR_INVALID) ++fails;
    if (gemm_validate(GEMM_B_ROW_MAJOR, M, N, K, dA, K - 1, dB, N, dC, N, GEMM_F32) != GEMM_ERR_INVALID) ++fails;
    cudaFree(dA);
    cudaFree(dB);
    cudaFree(dC);
    gemm_destroy(h);
    free(A);
    free(Bl);
    free(Bc);
    free(C);
    if (fails) {
        fprintf(stderr, "%d check(s) failed\n", fails);
        return 1;
    }
    printf("C ABI OK\n");
    return 0;
}
