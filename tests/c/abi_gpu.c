/* Plain C use of the C ABI on a GPU: device buffers from cudaMalloc, one
 * reduction, and small integers whose sum is exact (so the expected value
 * needs no oracle): 3 ranks of f32 values in [-100, 100], bf16 wire
 * (exact for |v| <= 256), 2 destinations. */
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "ar.h"

#define N 100003

int main(void) {
    static float h[3][N], out[2][N];
    for (int r = 0; r < 3; ++r)
        for (int i = 0; i < N; ++i) h[r][i] = (float)((i * (r + 7) + 13 * r) % 201 - 100);
    void *d_src[3], *d_dst[2];
    for (int r = 0; r < 3; ++r) {
        if (cudaMalloc(&d_src[r], sizeof h[r]) != cudaSuccess) return 2;
        cudaMemcpy(d_src[r], h[r], sizeof h[r], cudaMemcpyHostToDevice);
    }
    for (int d = 0; d < 2; ++d)
        if (cudaMalloc(&d_dst[d], sizeof out[d]) != cudaSuccess) return 2;
    int st = ar_init(3, N);
    if (st != AR_OK) {
        printf("ar_init: %s\n", ar_status_string(st));
        return 3;
    }
    st = ar_reduce((const void *const *)d_src, d_dst, 2, N, AR_F32, AR_BF16, (cudaStream_t)0);
    if (st != AR_OK) {
        printf("ar_reduce: %s\n", ar_status_string(st));
        return 4;
    }
    cudaDeviceSynchronize();
    long bad = 0;
    for (int d = 0; d < 2; ++d) {
        cudaMemcpy(out[d], d_dst[d], sizeof out[d], cudaMemcpyDeviceToHost);
        for (int i = 0; i < N; ++i)
            if (out[d][i] != h[0][i] + h[1][i] + h[2][i]) bad++;
    }
    ar_free();
    for (int r = 0; r < 3; ++r) cudaFree(d_src[r]);
    for (int d = 0; d < 2; ++d) cudaFree(d_dst[d]);
    printf("%s (%ld mismatches)\n", bad ? "FAIL" : "ok", bad);
    return bad ? 1 : 0;
}
