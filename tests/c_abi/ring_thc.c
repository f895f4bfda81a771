/* A plain-C consumer of libgar.so: no Python, no PyTorch.  Four workers'
 * buffers in cudaMalloc'ed memory go through the ring all-reduce (average),
 * one uniform THC round (range, fused encode -> aggregate -> decode, NMSE),
 * one non-uniform THC round (a table on a granularity-36 grid) and a round
 * trip through the randomized Hadamard transform, through the C ABI of gar.h
 * alone.  Inputs are small integers, so the ring average (a sum of integers
 * divided by 4) is exact and checked exactly; the THC averages are checked
 * within the widest quantization interval of their round, the round trip
 * within the transform's fp32 error bound.  Prints "c abi ok" and exits 0 on
 * success. */
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include "gar.h"

#define CHECK_GAR(call)                                                         \
    do {                                                                        \
        int rc_ = (call);                                                       \
        if (rc_ != GAR_OK) {                                                    \
            fprintf(stderr, "%s: %d (%s)\n", #call, rc_, gar_last_error());     \
            return 1;                                                           \
        }                                                                       \
    } while (0)
#define CHECK_CUDA(call)                                                        \
    do {                                                                        \
        cudaError_t e_ = (call);                                                \
        if (e_ != cudaSuccess) {                                                \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));         \
            return 1;                                                           \
        }                                                                       \
    } while (0)

enum { P = 4 };
static const int64_t N = 100003; /* ragged: not a multiple of the chunk or vector sizes */

int main(void) {
    float *host = (float *)malloc(sizeof(float) * (size_t)N * P);
    float *back = (float *)malloc(sizeof(float) * (size_t)N);
    float *x[P], *y[P];
    if (!host || !back) return 1;
    for (int w = 0; w < P; ++w)
        for (int64_t i = 0; i < N; ++i) host[(size_t)w * N + i] = (float)((i * 7 + w * 13) % 101 - 50);
    for (int w = 0; w < P; ++w) {
        CHECK_CUDA(cudaMalloc((void **)&x[w], sizeof(float) * (size_t)N));
        CHECK_CUDA(cudaMalloc((void **)&y[w], sizeof(float) * (size_t)N));
        CHECK_CUDA(cudaMemcpy(x[w], host + (size_t)w * N, sizeof(float) * (size_t)N, cudaMemcpyHostToDevice));
        CHECK_CUDA(cudaMemcpy(y[w], host + (size_t)w * N, sizeof(float) * (size_t)N, cudaMemcpyHostToDevice));
    }

    /* ring all-reduce, in place: every worker ends with the average */
    CHECK_GAR(gar_ring_allreduce_sim((void *const *)y, P, N, GAR_F32, GAR_AVG, NULL));
    for (int w = 0; w < P; ++w) {
        CHECK_CUDA(cudaMemcpy(back, y[w], sizeof(float) * (size_t)N, cudaMemcpyDeviceToHost));
        for (int64_t i = 0; i < N; ++i) {
            float s = 0.0f;
            for (int v = 0; v < P; ++v) s += host[(size_t)v * N + i];
            if (back[i] != s / (float)P) {
                fprintf(stderr, "ring: worker %d element %lld: %g != %g\n", w, (long long)i, back[i], s / P);
                return 1;
            }
        }
    }

    /* one uniform THC round, b = 4, with the wire vectors */
    const int b = 4;
    const int64_t words = gar_thc_words(N, b);
    float *d_mM, *avg, *exact;
    uint32_t *packed[P];
    double *d_nmse;
    void *ws;
    const size_t ws_bytes = gar_nmse_workspace_bytes(N);
    CHECK_CUDA(cudaMalloc((void **)&d_mM, 2 * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void **)&avg, sizeof(float) * (size_t)N));
    CHECK_CUDA(cudaMalloc((void **)&d_nmse, sizeof(double)));
    CHECK_CUDA(cudaMalloc(&ws, ws_bytes));
    for (int w = 0; w < P; ++w) CHECK_CUDA(cudaMalloc((void **)&packed[w], sizeof(uint32_t) * (size_t)words));
    CHECK_GAR(gar_thc_range((const float *const *)x, P, N, d_mM, NULL));
    CHECK_GAR(gar_thc_allreduce_fused((const float *const *)x, P, N, b, 0x5EEDull, d_mM, avg, packed, NULL));
    exact = y[0]; /* the exact average from the ring above */
    CHECK_GAR(gar_nmse(exact, avg, N, d_nmse, ws, ws_bytes, NULL));
    uint32_t status = 0;
    CHECK_GAR(gar_sync_status(NULL, &status, 1));
    float mM[2];
    double nmse = 0.0;
    CHECK_CUDA(cudaMemcpy(mM, d_mM, sizeof(mM), cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(&nmse, d_nmse, sizeof(double), cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(back, avg, sizeof(float) * (size_t)N, cudaMemcpyDeviceToHost));
    if (mM[0] != -50.0f || mM[1] != 50.0f || status != 0) {
        fprintf(stderr, "range [%g, %g], status %u\n", mM[0], mM[1], status);
        return 1;
    }
    /* every worker's rounding moves its value by less than one step (M - m) / 15,
     * so the average moves by less than one step too */
    const double step = (mM[1] - mM[0]) / 15.0;
    for (int64_t i = 0; i < N; ++i) {
        double s = 0.0;
        for (int v = 0; v < P; ++v) s += host[(size_t)v * N + i];
        if (fabs(back[i] - s / P) > step * (1.0 + 1e-6)) {
            fprintf(stderr, "thc: element %lld: %g against %g\n", (long long)i, back[i], s / P);
            return 1;
        }
    }
    if (!(nmse > 0.0 && nmse < 1.0)) {
        fprintf(stderr, "nmse %g\n", nmse);
        return 1;
    }

    /* one non-uniform THC round, b = 4, granularity 36, the table 0, 2, 5, ..., 36 */
    const int g = 36;
    uint16_t table[16];
    int widest = 0;
    for (int z = 0; z < 16; ++z) table[z] = (uint16_t)((z * g * 2 + 15) / 30); /* round(z * 36 / 15) */
    for (int z = 0; z < 15; ++z)
        if (table[z + 1] - table[z] > widest) widest = table[z + 1] - table[z];
    CHECK_GAR(gar_nuhc_allreduce_fused((const float *const *)x, P, N, b, g, table, 0x5EEDull, d_mM, avg, packed,
                                       NULL));
    CHECK_CUDA(cudaMemcpy(back, avg, sizeof(float) * (size_t)N, cudaMemcpyDeviceToHost));
    const double interval = widest * (mM[1] - mM[0]) / g;
    for (int64_t i = 0; i < N; ++i) {
        double s = 0.0;
        for (int v = 0; v < P; ++v) s += host[(size_t)v * N + i];
        if (fabs(back[i] - s / P) > interval * (1.0 + 1e-6)) {
            fprintf(stderr, "non-uniform thc: element %lld: %g against %g\n", (long long)i, back[i], s / P);
            return 1;
        }
    }

    /* the randomized Hadamard transform there and back: n = 2^20 (tile pass
     * and cluster pass), the first worker's values repeated */
    const int64_t n = (int64_t)1 << 20;
    float *hx = (float *)malloc(sizeof(float) * (size_t)n), *hz = (float *)malloc(sizeof(float) * (size_t)n);
    float *dx, *dy, *dz;
    if (!hx || !hz) return 1;
    double norm2 = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        hx[i] = host[i % N] * 0.01f;
        norm2 += (double)hx[i] * hx[i];
    }
    CHECK_CUDA(cudaMalloc((void **)&dx, sizeof(float) * (size_t)n));
    CHECK_CUDA(cudaMalloc((void **)&dy, sizeof(float) * (size_t)n));
    CHECK_CUDA(cudaMalloc((void **)&dz, sizeof(float) * (size_t)n));
    CHECK_CUDA(cudaMemcpy(dx, hx, sizeof(float) * (size_t)n, cudaMemcpyHostToDevice));
    CHECK_GAR(gar_rht(dx, dy, n, 7, 0, NULL));
    CHECK_GAR(gar_rht(dy, dz, n, 7, 1, NULL));
    CHECK_CUDA(cudaMemcpy(hz, dz, sizeof(float) * (size_t)n, cudaMemcpyDeviceToHost));
    double err2 = 0.0;
    for (int64_t i = 0; i < n; ++i) err2 += ((double)hz[i] - hx[i]) * ((double)hz[i] - hx[i]);
    /* each direction within (log2 n + 2) 2^-24 ||x|| of the exact transform (orthogonal) */
    const double bound = 2.0 * (20 + 2) * ldexp(1.0, -24) * sqrt(norm2);
    if (!(sqrt(err2) <= bound)) {
        fprintf(stderr, "rht round trip: error %g above %g\n", sqrt(err2), bound);
        return 1;
    }
    CHECK_GAR(gar_sync_status(NULL, &status, 1));
    if (status != 0) {
        fprintf(stderr, "status %u\n", status);
        return 1;
    }
    printf("c abi ok: ring exact, THC b=4 within one step, NMSE %.4g; non-uniform THC within its widest "
           "interval; RHT round trip within its bound\n",
           nmse);
    return 0;
}
