/* Host cost of one ar_reduce call from C, for decode-sized calls (R = 4,
 * 4099 floats, 4 destinations): the time to validate, pick the launch and
 * enqueue it, measured two ways.
 *   eager:   500 calls on a stream (fewer than the launch queue holds, so
 *            the host does not wait for the GPU);
 *   capture: 10 000 calls recorded into a CUDA graph (nothing runs).
 * Prints "ok eager_us=<per call> capture_us=<per call>". */
#define _POSIX_C_SOURCE 199309L /* clock_gettime under -std=c11 */
#include <cuda_runtime.h>
#include <stdio.h>
#include <time.h>

#include "ar.h"

#define R 4
#define ND 4
#define N 4099
#define ROW 4100 /* rows padded so that every buffer starts on a 16-byte boundary */

static double now_us(void) {
    struct timespec t;
    clock_gettime(CLOCK_MONOTONIC, &t);
    return (double)t.tv_sec * 1e6 + (double)t.tv_nsec * 1e-3;
}

int main(void) {
    float *buf = NULL;
    if (cudaMalloc((void **)&buf, sizeof(float) * ROW * (R + ND)) != cudaSuccess) return 2;
    if (cudaMemset(buf, 0, sizeof(float) * ROW * (R + ND)) != cudaSuccess) return 2;
    const void *srcs[R];
    void *dsts[ND];
    for (int r = 0; r < R; ++r) srcs[r] = buf + (size_t)r * ROW;
    for (int d = 0; d < ND; ++d) dsts[d] = buf + (size_t)(R + d) * ROW;
    cudaStream_t s;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return 2;
    if (ar_init(R, N) != AR_OK) return 3;
    for (int k = 0; k < 100; ++k)
        if (ar_reduce(srcs, dsts, ND, N, AR_F32, AR_F16, s) != AR_OK) return 4;
    if (cudaStreamSynchronize(s) != cudaSuccess) return 2;

    double t0 = now_us();
    for (int k = 0; k < 500; ++k)
        if (ar_reduce(srcs, dsts, ND, N, AR_F32, AR_F16, s) != AR_OK) return 4;
    const double eager = (now_us() - t0) / 500;
    if (cudaStreamSynchronize(s) != cudaSuccess) return 2;

    cudaGraph_t g;
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return 2;
    t0 = now_us();
    for (int k = 0; k < 10000; ++k)
        if (ar_reduce(srcs, dsts, ND, N, AR_F32, AR_F16, s) != AR_OK) return 4;
    const double capture = (now_us() - t0) / 10000;
    if (cudaStreamEndCapture(s, &g) != cudaSuccess) return 2;
    cudaGraphDestroy(g);

    ar_free();
    cudaStreamDestroy(s);
    cudaFree(buf);
    printf("ok eager_us=%.3f capture_us=%.3f\n", eager, capture);
    return 0;
}
