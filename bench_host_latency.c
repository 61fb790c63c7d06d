/* bench_host_latency.c -- wall-clock latency of a whole-array sum returned to
 * the host through the C ABI (ak_reduce with dst_host), without any binding
 * in between: the library's own time, launches and synchronization included.
 *
 * Built and run by bench.py:  bench_host_latency N REPS
 * Prints one JSON object: medians / minima in microseconds of calls made
 * after an L2 flush ("flushed") and back to back on a warm L2 ("warm"). The
 * input is N floats of a fixed pattern (the values do not affect the time).
 */
#define _POSIX_C_SOURCE 200809L
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <time.h>

#include <cuda_runtime_api.h>

#include "ak.h"

static double now_us(void) {
    struct timespec t;
    clock_gettime(CLOCK_MONOTONIC, &t);
    return (double)t.tv_sec * 1e6 + (double)t.tv_nsec * 1e-3;
}

static int cmp_double(const void* a, const void* b) {
    const double x = *(const double*)a, y = *(const double*)b;
    return (x > y) - (x < y);
}

#define CK(call)                                                          \
    do {                                                                  \
        cudaError_t e_ = (call);                                          \
        if (e_ != cudaSuccess) {                                          \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_)); \
            return 1;                                                     \
        }                                                                 \
    } while (0)

int main(int argc, char** argv) {
    const int64_t n = argc > 1 ? atoll(argv[1]) : 1000000;
    const int reps = argc > 2 ? atoi(argv[2]) : 300;
    float* h = (float*)malloc((size_t)n * sizeof(float));
    double* ts = (double*)malloc((size_t)reps * sizeof(double));
    if (!h || !ts || n < 1 || reps < 1) return 1;
    for (int64_t i = 0; i < n; ++i) h[i] = (float)((i % 2001) - 1000) * (1.0f / 1024.0f);
    float* x = NULL;
    void* flush = NULL;
    const size_t flush_bytes = (size_t)256 << 20;
    cudaStream_t s;
    CK(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
    CK(cudaMalloc((void**)&x, (size_t)n * sizeof(float)));
    CK(cudaMalloc(&flush, flush_bytes));
    CK(cudaMemcpy(x, h, (size_t)n * sizeof(float), cudaMemcpyHostToDevice));
    size_t wsb = 0;
    if (ak_reduce_workspace_size(n, AK_F32, AK_F32, NULL, &wsb) != AK_OK) return 1;
    void* ws = NULL;
    CK(cudaMalloc(&ws, wsb));
    const float init = 0.0f;
    float res = 0.0f;
    double med[2], mn[2];
    for (int pass = 0; pass < 2; ++pass) {  /* 0: flushed, 1: warm */
        for (int w = 0; w < 20; ++w)
            if (ak_reduce(x, n, AK_F32, AK_MAP_IDENTITY, AK_OP_ADD, AK_F32, AK_F32, &init, AK_STORE_INIT, NULL,
                          &res, ws, wsb, NULL, s) != AK_OK)
                return 1;
        for (int r = 0; r < reps; ++r) {
            if (pass == 0) CK(cudaMemsetAsync(flush, r & 0xFF, flush_bytes, s));
            CK(cudaStreamSynchronize(s));
            const double t0 = now_us();
            const ak_status st = ak_reduce(x, n, AK_F32, AK_MAP_IDENTITY, AK_OP_ADD, AK_F32, AK_F32, &init,
                                           AK_STORE_INIT, NULL, &res, ws, wsb, NULL, s);
            ts[r] = now_us() - t0;
            if (st != AK_OK) return 1;
        }
        qsort(ts, (size_t)reps, sizeof(double), cmp_double);
        med[pass] = ts[reps / 2];
        mn[pass] = ts[0];
    }
    double want = 0.0;
    for (int64_t i = 0; i < n; ++i) want += h[i];
    printf("{\"n\": %lld, \"reps\": %d, \"flushed_us_median\": %.2f, \"flushed_us_min\": %.2f, "
           "\"warm_us_median\": %.2f, \"warm_us_min\": %.2f, \"result\": %.9g, \"expected\": %.9g}\n",
           (long long)n, reps, med[0], mn[0], med[1], mn[1], (double)res, want);
    cudaFree(ws);
    cudaFree(flush);
    cudaFree(x);
    cudaStreamDestroy(s);
    free(h);
    free(ts);
    return 0;
}
