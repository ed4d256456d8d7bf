/*
 * A plain C client of libtg: no Python, no PyTorch.  It allocates device memory
 * with the CUDA runtime, runs tg_gemm (bias epilogue, fp32 out) and
 * tg_grouped_gemm on small integer-valued problems, whose fp32 results are exact,
 * and compares every element with a C loop.  Exit status 0 = all equal.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "tg.h"

static uint16_t bf16_of_int(int v) {           /* small integers are exact in bf16 */
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

#define CHECK_CUDA(x)                                                              \
    do {                                                                           \
        cudaError_t e_ = (x);                                                      \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));               \
            return 2;                                                              \
        }                                                                          \
    } while (0)

#define CHECK_TG(x)                                                                \
    do {                                                                           \
        tg_status s_ = (x);                                                        \
        if (s_ != TG_OK) {                                                         \
            fprintf(stderr, "%s: %s: %s\n", #x, tg_status_string(s_), tg_last_error_message()); \
            return 3;                                                              \
        }                                                                          \
    } while (0)

static int run_dense(int M, int N, int K) {
    size_t na = (size_t)M * K, nb = (size_t)K * N, nc = (size_t)M * N;
    uint16_t *ha = malloc(na * 2), *hb = malloc(nb * 2), *hbias = malloc((size_t)N * 2);
    float *hc = malloc(nc * 4);
    int *ia = malloc(na * sizeof(int)), *ib = malloc(nb * sizeof(int)), *ibias = malloc(N * sizeof(int));
    for (size_t i = 0; i < na; ++i) { ia[i] = (int)((i * 7 + 3) % 9) - 4; ha[i] = bf16_of_int(ia[i]); }
    for (size_t i = 0; i < nb; ++i) { ib[i] = (int)((i * 5 + 1) % 7) - 3; hb[i] = bf16_of_int(ib[i]); }
    for (int j = 0; j < N; ++j) { ibias[j] = (j % 5) - 2; hbias[j] = bf16_of_int(ibias[j]); }
    void *da, *db, *dbias, *dc;
    CHECK_CUDA(cudaMalloc(&da, na * 2));
    CHECK_CUDA(cudaMalloc(&db, nb * 2));
    CHECK_CUDA(cudaMalloc(&dbias, (size_t)N * 2));
    CHECK_CUDA(cudaMalloc(&dc, nc * 4));
    CHECK_CUDA(cudaMemcpy(da, ha, na * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(db, hb, nb * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dbias, hbias, (size_t)N * 2, cudaMemcpyHostToDevice));
    /* A row-major [M][K], B row-major [K][N], C fp32 row-major [M][N] */
    CHECK_TG(tg_gemm(da, TG_ROW_MAJOR, K, db, TG_ROW_MAJOR, N, dc, TG_F32, N, M, N, K, TG_EPI_BIAS, dbias, NULL));
    CHECK_TG(tg_device_status(NULL));
    CHECK_CUDA(cudaMemcpy(hc, dc, nc * 4, cudaMemcpyDeviceToHost));
    long bad = 0;
    for (int i = 0; i < M; ++i)
        for (int j = 0; j < N; ++j) {
            long ref = ibias[j];
            for (int k = 0; k < K; ++k) ref += (long)ia[(size_t)i * K + k] * ib[(size_t)k * N + j];
            if (hc[(size_t)i * N + j] != (float)ref) ++bad;
        }
    cudaFree(da); cudaFree(db); cudaFree(dbias); cudaFree(dc);
    free(ha); free(hb); free(hbias); free(hc); free(ia); free(ib); free(ibias);
    printf("dense %dx%dx%d: %ld mismatches\n", M, N, K, bad);
    return bad ? 1 : 0;
}

static int run_grouped(void) {
    enum { G = 3, N = 136, K = 200 };
    const int Ms[G] = {37, 0, 300};
    tg_group_problem table[G];
    memset(table, 0, sizeof table);
    void *da[G], *db[G], *dc[G];
    int *ia[G], *ib[G];
    for (int g = 0; g < G; ++g) {
        int M = Ms[g];
        size_t na = (size_t)M * K, nb = (size_t)K * N;
        ia[g] = malloc((na ? na : 1) * sizeof(int));
        ib[g] = malloc(nb * sizeof(int));
        uint16_t *ha = malloc((na ? na : 1) * 2), *hb = malloc(nb * 2);
        for (size_t i = 0; i < na; ++i) { ia[g][i] = (int)((i * 3 + g) % 5) - 2; ha[i] = bf16_of_int(ia[g][i]); }
        for (size_t i = 0; i < nb; ++i) { ib[g][i] = (int)((i * 11 + g) % 7) - 3; hb[i] = bf16_of_int(ib[g][i]); }
        CHECK_CUDA(cudaMalloc(&da[g], (na ? na : 8) * 2));
        CHECK_CUDA(cudaMalloc(&db[g], nb * 2));
        CHECK_CUDA(cudaMalloc(&dc[g], (size_t)(M ? M : 1) * N * 4));
        if (na) CHECK_CUDA(cudaMemcpy(da[g], ha, na * 2, cudaMemcpyHostToDevice));
        CHECK_CUDA(cudaMemcpy(db[g], hb, nb * 2, cudaMemcpyHostToDevice));
        free(ha); free(hb);
        table[g].M = M; table[g].N = N; table[g].K = K;
        table[g].A = da[g]; table[g].lda = K; table[g].layout_a = TG_ROW_MAJOR;
        table[g].B = db[g]; table[g].ldb = N; table[g].layout_b = TG_ROW_MAJOR;
        table[g].C = dc[g]; table[g].ldc = N; table[g].c_dtype = TG_F32;
        table[g].epi = TG_EPI_NONE; table[g].bias = NULL; table[g].ab_dtype = TG_BF16;
    }
    CHECK_TG(tg_grouped_gemm(table, G, NULL));
    CHECK_TG(tg_device_status(NULL));
    long bad = 0;
    for (int g = 0; g < G; ++g) {
        int M = Ms[g];
        if (M == 0) continue;
        float *hc = malloc((size_t)M * N * 4);
        CHECK_CUDA(cudaMemcpy(hc, dc[g], (size_t)M * N * 4, cudaMemcpyDeviceToHost));
        for (int i = 0; i < M; ++i)
            for (int j = 0; j < N; ++j) {
                long ref = 0;
                for (int k = 0; k < K; ++k) ref += (long)ia[g][(size_t)i * K + k] * ib[g][(size_t)k * N + j];
                if (hc[(size_t)i * N + j] != (float)ref) ++bad;
            }
        free(hc);
    }
    for (int g = 0; g < G; ++g) { cudaFree(da[g]); cudaFree(db[g]); cudaFree(dc[g]); free(ia[g]); free(ib[g]); }
    printf("grouped (37, 0, 300 rows): %ld mismatches\n", bad);
    return bad ? 1 : 0;
}

int main(void) {
    int rc = run_dense(300, 264, 640);
    if (!rc) rc = run_dense(1000, 512, 1024);
    if (!rc) rc = run_grouped();
    printf("libtg version %u.%u: %s\n", tg_version() >> 16, tg_version() & 0xffffu, rc ? "FAIL" : "ok");
    return rc;
}
