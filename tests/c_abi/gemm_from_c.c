/*
 * gemm_from_c.c -- drives the GEMM library through its C ABI from plain C.
 *
 * Usage: gemm_from_c <abt|ab> <f16|bf16> M N K A.bin B.bin D.bin
 *        gemm_from_c fp8 <e4m3|e5m2> M N K A.bin B.bin D.bin alpha
 *        gemm_from_c mx <e4m3|e5m2> M N K A.bin B.bin D.bin alpha SA.bin SB.bin
 * Reads A (M x K) and B (N x K for abt / fp8 / mx, K x N for ab) as raw 16-bit
 * patterns (bytes for fp8 and mx; for mx also the row-major scale bytes, M and
 * N rows of ceil(K / 32)), runs gemm_abt / gemm_ab / gemm_fp8_abt /
 * gemm_mx_abt (BF16 D; mx packs the scales with gemm_mx_pack_scales[_b]
 * first) on cudaMalloc'd buffers on a created stream, writes D (M x N, 16-bit)
 * to D.bin, and checks that a few invalid calls return the documented status
 * codes.  Exit status 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "gemm.h"

static void* read_file(const char* path, size_t bytes) {
    FILE* f = fopen(path, "rb");
    if (!f) return NULL;
    void* p = malloc(bytes ? bytes : 1);
    size_t got = fread(p, 1, bytes, f);
    fclose(f);
    if (got != bytes) {
        free(p);
        return NULL;
    }
    return p;
}

#define CHECK_CUDA(x)                                                       \
    do {                                                                    \
        cudaError_t e_ = (x);                                               \
        if (e_ != cudaSuccess) {                                            \
            fprintf(stderr, "%s failed: %s\n", #x, cudaGetErrorString(e_)); \
            return 2;                                                       \
        }                                                                   \
    } while (0)

int main(int argc, char** argv) {
    const int mx = argc >= 2 && strcmp(argv[1], "mx") == 0;
    const int fp8 = mx || (argc >= 2 && strcmp(argv[1], "fp8") == 0);
    if (argc != (mx ? 12 : fp8 ? 10 : 9)) {
        fprintf(stderr, "usage: %s <abt|ab> <f16|bf16> M N K A.bin B.bin D.bin\n"
                        "       %s fp8 <e4m3|e5m2> M N K A.bin B.bin D.bin alpha\n"
                        "       %s mx <e4m3|e5m2> M N K A.bin B.bin D.bin alpha SA.bin SB.bin\n",
                argv[0], argv[0], argv[0]);
        return 2;
    }
    const int ab = strcmp(argv[1], "ab") == 0;
    const int dtype = fp8 ? GEMM_BF16 : strcmp(argv[2], "bf16") == 0 ? GEMM_BF16 : GEMM_F16;
    const int fmt = strcmp(argv[2], "e5m2") == 0 ? GEMM_E5M2 : GEMM_E4M3;
    const float alpha = fp8 ? (float)atof(argv[9]) : 1.0f;
    const int64_t M = atoll(argv[3]), N = atoll(argv[4]), K = atoll(argv[5]);
    const size_t esize = fp8 ? 1 : 2;
    const size_t a_bytes = (size_t)(M * K) * esize, b_bytes = (size_t)(N * K) * esize,
                 d_bytes = (size_t)(M * N) * 2;
    void* hA = read_file(argv[6], a_bytes);
    void* hB = read_file(argv[7], b_bytes);
    if (!hA || !hB) {
        fprintf(stderr, "cannot read inputs\n");
        return 2;
    }
    void *dA, *dB, *dD;
    cudaStream_t s;
    CHECK_CUDA(cudaMalloc(&dA, a_bytes));
    CHECK_CUDA(cudaMalloc(&dB, b_bytes));
    CHECK_CUDA(cudaMalloc(&dD, d_bytes));
    CHECK_CUDA(cudaStreamCreate(&s));
    CHECK_CUDA(cudaMemcpy(dA, hA, a_bytes, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dB, hB, b_bytes, cudaMemcpyHostToDevice));

    void *dSA = NULL, *dSB = NULL;
    if (mx) {
        /* row-major scales -> device -> the layouts gemm_mx_abt reads */
        const int64_t groups = (K + 31) / 32;
        size_t sa_bytes = 0, sb_bytes = 0;
        if (gemm_mx_scales_size(M, K, &sa_bytes) != GEMM_OK ||
            gemm_mx_scales_b_size(N, K, &sb_bytes) != GEMM_OK)
            return 1;
        void* hSA = read_file(argv[10], (size_t)(M * groups));
        void* hSB = read_file(argv[11], (size_t)(N * groups));
        if (!hSA || !hSB) {
            fprintf(stderr, "cannot read scales\n");
            return 2;
        }
        void *rawA, *rawB;
        CHECK_CUDA(cudaMalloc(&rawA, (size_t)(M * groups)));
        CHECK_CUDA(cudaMalloc(&rawB, (size_t)(N * groups)));
        CHECK_CUDA(cudaMalloc(&dSA, sa_bytes));
        CHECK_CUDA(cudaMalloc(&dSB, sb_bytes));
        CHECK_CUDA(cudaMemcpy(rawA, hSA, (size_t)(M * groups), cudaMemcpyHostToDevice));
        CHECK_CUDA(cudaMemcpy(rawB, hSB, (size_t)(N * groups), cudaMemcpyHostToDevice));
        if (gemm_mx_pack_scales(rawA, M, K, groups, dSA, s) != GEMM_OK ||
            gemm_mx_pack_scales_b(rawB, N, K, groups, dSB, s) != GEMM_OK)
            return 1;
        CHECK_CUDA(cudaStreamSynchronize(s));
        cudaFree(rawA);
        cudaFree(rawB);
        free(hSA);
        free(hSB);
    }
    int st = mx    ? gemm_mx_abt(dA, dB, dSA, dSB, dD, M, N, K, K, K, N, fmt, dtype, alpha, s)
             : fp8 ? gemm_fp8_abt(dA, dB, dD, M, N, K, K, K, N, fmt, dtype, alpha, s)
             : ab  ? gemm_ab(dA, dB, dD, M, N, K, K, N, N, dtype, s)
                   : gemm_abt(dA, dB, dD, M, N, K, K, K, N, dtype, s);
    if (st != GEMM_OK) {
        fprintf(stderr, "gemm: %s\n", gemm_status_string(st));
        return 1;
    }
    CHECK_CUDA(cudaStreamSynchronize(s));
    uint32_t word = 1;
    if (gemm_device_status(&word, 1) != GEMM_OK || word != 0) {
        fprintf(stderr, "device status %u\n", word);
        return 1;
    }
    void* hD = malloc(d_bytes ? d_bytes : 1);
    CHECK_CUDA(cudaMemcpy(hD, dD, d_bytes, cudaMemcpyDeviceToHost));
    FILE* f = fopen(argv[8], "wb");
    if (!f || fwrite(hD, 1, d_bytes, f) != d_bytes) return 2;
    fclose(f);

    /* documented errors */
    if (mx) {
        if (gemm_mx_abt(dA, dB, NULL, dSB, dD, M, N, K, K, K, N, fmt, dtype, 1.0f, s) != GEMM_ERR_NULL)
            return 3;
        if (gemm_mx_abt(dA, dB, (char*)dSA + 4, dSB, dD, M, N, K, K, K, N, fmt, dtype, 1.0f, s) !=
            GEMM_ERR_ALIGN)
            return 3;
        cudaFree(dSA);
        cudaFree(dSB);
    }
    if (fp8) {
        if (gemm_fp8_abt(dA, dB, dD, M, N, K, K, K, N, GEMM_F16, dtype, 1.0f, s) != GEMM_ERR_DTYPE)
            return 3;
        if (gemm_fp8_abt(dA, dB, dD, M, N, K, K + 8, K, N, fmt, dtype, 1.0f, s) != GEMM_ERR_ALIGN)
            return 3;
        if (gemm_abt(dA, dB, dD, M, N, K, K, K, N, fmt, s) != GEMM_ERR_DTYPE) return 3;
    }
    if (gemm_abt(dA, dB, dD, M, N, K, K, K, N, 7, s) != GEMM_ERR_DTYPE) return 3;
    if (gemm_abt(NULL, dB, dD, M, N, K, K, K, N, dtype, s) != GEMM_ERR_NULL) return 3;
    if (gemm_abt((char*)dA + 2, dB, dD, M, N, K, K, K, N, dtype, s) != GEMM_ERR_ALIGN) return 3;
    if (gemm_abt(dA, dB, dA, M, N, K, K, K, N, dtype, s) != GEMM_ERR_ALIAS) return 3;
    if (gemm_status_string(GEMM_ERR_SHAPE)[0] == '\0') return 3;

    cudaFree(dA);
    cudaFree(dB);
    cudaFree(dD);
    cudaStreamDestroy(s);
    free(hA);
    free(hB);
    free(hD);
    printf("ok\n");
    return 0;
}
