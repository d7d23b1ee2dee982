/*
 * c_abi_client.c -- a plain C (C99) client of libtb.so.
 *
 * It includes nothing of the library but include/tb.h (and, for the GPU part,
 * the CUDA runtime's C API), so it shows that the boundary is usable from C
 * with no C++ and no Python in between.
 *
 *   ./c_abi_client        argument checks, which return before any CUDA call
 *   ./c_abi_client gpu    also a softmax backward and a LayerNorm backward on the
 *                         GPU, compared with the CPU oracle (liboracle.so)
 *
 * Test infrastructure: built and run by tests/test_c_abi.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "tb.h"

#define CHECK(cond)                                                              \
    do {                                                                         \
        if (!(cond)) {                                                           \
            fprintf(stderr, "%s:%d: check failed: %s\n", __FILE__, __LINE__, #cond); \
            return 1;                                                            \
        }                                                                        \
    } while (0)

static int cpu_checks(void) {
    size_t bytes = 123;
    CHECK(tb_version() >= 100);
    CHECK(strcmp(tb_status_string(TB_ERR_ALIAS), "TB_ERR_ALIAS") == 0);
    CHECK(strcmp(tb_status_string(TB_OK), "TB_OK") == 0);
    CHECK(tb_adamw_plan_destroy(NULL) == TB_OK);
    CHECK(tb_softmax_bwd(NULL, NULL, NULL, 4, 4, TB_F32, NULL) == TB_ERR_INVALID_VALUE);
    CHECK(tb_softmax_bwd((void*)0x1000, (void*)0x2000, (void*)0x3000, 4, 4, (tb_dtype)9, NULL) ==
          TB_ERR_UNSUPPORTED_DTYPE);
    CHECK(tb_layernorm_bwd_workspace_size(-1, 16, TB_F32, &bytes) == TB_ERR_INVALID_VALUE);
    CHECK(tb_layernorm_bwd_workspace_size(0, 16, TB_F32, &bytes) == TB_OK && bytes == 0);
    CHECK(tb_cast_from_f32((const float*)0x1000, (void*)0x1002, TB_BF16, 4, NULL) == TB_ERR_ALIAS);
    return 0;
}

#ifdef WITH_CUDA
#include <cuda_runtime_api.h>

/* The CPU oracle's entry points (oracle/oracle.c), linked for this test only. */
void orc_softmax_bwd_f64(int64_t rows, int64_t cols, const double* dY, const double* P, double* dX);
void orc_layernorm_bwd_f64(int64_t rows, int64_t D, const double* dY, const double* x,
                           const double* mean, const double* inv_std, const double* gamma,
                           double* dX, double* dgamma, double* dbeta);

/* Seeded uniform in [-1, 1): a 64-bit linear congruential generator. */
static uint64_t g_state = 0x2545F4914F6CDD1Dull;
static double uniform(void) {
    g_state = g_state * 6364136223846793005ull + 1442695040888963407ull;
    return (double)(g_state >> 11) / 9007199254740992.0 * 2.0 - 1.0;
}

static int softmax_check(void) {
    const int64_t rows = 257, cols = 1000, n = rows * cols;
    float *P = malloc(n * sizeof(float)), *dY = malloc(n * sizeof(float)), *dX = malloc(n * sizeof(float));
    double *Pd = malloc(n * sizeof(double)), *dYd = malloc(n * sizeof(double)), *ref = malloc(n * sizeof(double));
    void *gP = NULL, *gdY = NULL, *gdX = NULL;
    double err = 0.0;
    int64_t r, j;
    CHECK(P && dY && dX && Pd && dYd && ref);
    for (r = 0; r < rows; ++r) { /* P = softmax of random logits, in double, rounded to float */
        double mx = -1e300, s = 0.0;
        for (j = 0; j < cols; ++j) { Pd[r * cols + j] = 4.0 * uniform(); if (Pd[r * cols + j] > mx) mx = Pd[r * cols + j]; }
        for (j = 0; j < cols; ++j) { Pd[r * cols + j] = exp(Pd[r * cols + j] - mx); s += Pd[r * cols + j]; }
        for (j = 0; j < cols; ++j) P[r * cols + j] = (float)(Pd[r * cols + j] / s);
    }
    for (j = 0; j < n; ++j) { dY[j] = (float)uniform(); Pd[j] = P[j]; dYd[j] = dY[j]; }
    CHECK(cudaMalloc(&gP, n * sizeof(float)) == cudaSuccess);
    CHECK(cudaMalloc(&gdY, n * sizeof(float)) == cudaSuccess);
    CHECK(cudaMalloc(&gdX, n * sizeof(float)) == cudaSuccess);
    CHECK(cudaMemcpy(gP, P, n * sizeof(float), cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(gdY, dY, n * sizeof(float), cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(tb_softmax_bwd(gdY, gP, gdX, rows, cols, TB_F32, NULL) == TB_OK);
    CHECK(cudaMemcpy(dX, gdX, n * sizeof(float), cudaMemcpyDeviceToHost) == cudaSuccess);
    orc_softmax_bwd_f64(rows, cols, dYd, Pd, ref);
    for (j = 0; j < n; ++j) { double e = fabs((double)dX[j] - ref[j]); if (e > err) err = e; }
    printf("softmax bwd 257 x 1000 fp32 through the C ABI: max |dX - oracle| = %.3g\n", err);
    CHECK(err <= 1e-5);
    cudaFree(gP); cudaFree(gdY); cudaFree(gdX);
    free(P); free(dY); free(dX); free(Pd); free(dYd); free(ref);
    return 0;
}

static int layernorm_check(void) {
    const int64_t rows = 300, D = 768, n = rows * D;
    float *x = malloc(n * 4), *dY = malloc(n * 4), *dX = malloc(n * 4);
    float *mean = malloc(rows * 4), *rstd = malloc(rows * 4), *gamma = malloc(D * 4);
    float *dg = malloc(D * 4), *db = malloc(D * 4);
    double *xd = malloc(n * 8), *dYd = malloc(n * 8), *md = malloc(rows * 8), *rd = malloc(rows * 8);
    double *gd = malloc(D * 8), *rdx = malloc(n * 8), *rdg = malloc(D * 8), *rdb = malloc(D * 8);
    void *gx = NULL, *gdY = NULL, *gdX = NULL, *gm = NULL, *gr = NULL, *gg = NULL, *gdg = NULL, *gdb = NULL, *ws = NULL;
    size_t ws_bytes = 0;
    double ex = 0.0, sx = 0.0, eg = 0.0, sg = 0.0, eb = 0.0, sb = 0.0;
    int64_t r, j;
    CHECK(x && dY && dX && mean && rstd && gamma && dg && db && xd && dYd && md && rd && gd && rdx && rdg && rdb);
    for (j = 0; j < n; ++j) { x[j] = (float)(2.0 * uniform()); dY[j] = (float)uniform(); xd[j] = x[j]; dYd[j] = dY[j]; }
    for (j = 0; j < D; ++j) { gamma[j] = (float)(1.0 + 0.1 * uniform()); gd[j] = gamma[j]; }
    for (r = 0; r < rows; ++r) { /* saved statistics of the forward, in double, rounded to float */
        double mu = 0.0, var = 0.0;
        for (j = 0; j < D; ++j) mu += xd[r * D + j];
        mu /= (double)D;
        for (j = 0; j < D; ++j) var += (xd[r * D + j] - mu) * (xd[r * D + j] - mu);
        mean[r] = (float)mu;
        rstd[r] = (float)(1.0 / sqrt(var / (double)D + 1e-5));
        md[r] = mean[r];
        rd[r] = rstd[r];
    }
    CHECK(tb_layernorm_bwd_workspace_size(rows, D, TB_F32, &ws_bytes) == TB_OK);
    CHECK(cudaMalloc(&gx, n * 4) == cudaSuccess && cudaMalloc(&gdY, n * 4) == cudaSuccess);
    CHECK(cudaMalloc(&gdX, n * 4) == cudaSuccess && cudaMalloc(&gm, rows * 4) == cudaSuccess);
    CHECK(cudaMalloc(&gr, rows * 4) == cudaSuccess && cudaMalloc(&gg, D * 4) == cudaSuccess);
    CHECK(cudaMalloc(&gdg, D * 4) == cudaSuccess && cudaMalloc(&gdb, D * 4) == cudaSuccess);
    CHECK(cudaMalloc(&ws, ws_bytes) == cudaSuccess);
    CHECK(cudaMemcpy(gx, x, n * 4, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(gdY, dY, n * 4, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(gm, mean, rows * 4, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(gr, rstd, rows * 4, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(gg, gamma, D * 4, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(tb_layernorm_bwd(gdY, gx, gm, gr, gg, gdX, gdg, gdb, rows, D, TB_F32, ws, ws_bytes, NULL) == TB_OK);
    CHECK(cudaMemcpy(dX, gdX, n * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(dg, gdg, D * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(db, gdb, D * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
    orc_layernorm_bwd_f64(rows, D, dYd, xd, md, rd, gd, rdx, rdg, rdb);
    for (j = 0; j < n; ++j) { ex = fmax(ex, fabs(dX[j] - rdx[j])); sx = fmax(sx, fabs(rdx[j])); }
    for (j = 0; j < D; ++j) {
        eg = fmax(eg, fabs(dg[j] - rdg[j])); sg = fmax(sg, fabs(rdg[j]));
        eb = fmax(eb, fabs(db[j] - rdb[j])); sb = fmax(sb, fabs(rdb[j]));
    }
    printf("LayerNorm bwd 300 x 768 fp32 through the C ABI: rel. err dX %.3g, dgamma %.3g, dbeta %.3g\n",
           ex / sx, eg / sg, eb / sb);
    CHECK(ex <= 1e-4 * sx && eg <= 1e-3 * sg && eb <= 1e-3 * sb);
    cudaFree(gx); cudaFree(gdY); cudaFree(gdX); cudaFree(gm); cudaFree(gr); cudaFree(gg);
    cudaFree(gdg); cudaFree(gdb); cudaFree(ws);
    free(x); free(dY); free(dX); free(mean); free(rstd); free(gamma); free(dg); free(db);
    free(xd); free(dYd); free(md); free(rd); free(gd); free(rdx); free(rdg); free(rdb);
    return 0;
}
#endif

int main(int argc, char** argv) {
    int rc = cpu_checks();
    if (rc == 0) printf("argument checks through the C ABI: ok\n");
#ifdef WITH_CUDA
    if (rc == 0 && argc > 1 && strcmp(argv[1], "gpu") == 0) {
        int code = -1;
        rc = softmax_check();
        if (rc == 0) rc = layernorm_check();
        if (rc == 0 && (tb_device_error(&code, 1) != TB_OK || code != 0)) rc = 1;
    }
#else
    (void)argc;
    (void)argv;
#endif
    return rc;
}
