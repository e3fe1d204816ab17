/* ar_reduce_host_noalloc across a device reset.  One call, then ar_free,
 * cudaDeviceReset (which ends this process's context on the device, and with
 * it the loaded module that holds the staging area), ar_init, and a second
 * call with other data: the second call must find the staging area where
 * the new context holds it.  Small integers make every sum exact (3 ranks
 * of f32 values in [-100, 100] through a bf16 wire, exact for |v| <= 256),
 * so the expected values need no oracle. */
#include <stdio.h>

#include <cuda_runtime_api.h>

#include "ar.h"

#define N 100003

static float h[3][N], out[2][N];

/* Number of wrong output elements of one call, or -1 when a call failed. */
static long one_call(int call) {
    for (int r = 0; r < 3; ++r)
        for (int i = 0; i < N; ++i) h[r][i] = (float)(((i + 17 * call) * (r + 7) + 13 * r) % 201 - 100);
    for (int d = 0; d < 2; ++d)
        for (int i = 0; i < N; ++i) out[d][i] = -1e30f;
    const void *srcs[3] = {h[0], h[1], h[2]};
    void *dsts[2] = {out[0], out[1]};
    const int st = ar_reduce_host_noalloc(srcs, dsts, 2, N, AR_F32, AR_BF16, (cudaStream_t)0);
    if (st != AR_OK) {
        printf("call %d: %s\n", call, ar_status_string(st));
        return -1;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    long bad = 0;
    for (int d = 0; d < 2; ++d)
        for (int i = 0; i < N; ++i)
            if (out[d][i] != h[0][i] + h[1][i] + h[2][i]) bad++;
    return bad;
}

int main(void) {
    if (ar_init(3, N) != AR_OK) return 3;
    const long before = one_call(0);
    ar_free();
    if (cudaDeviceReset() != cudaSuccess) return 5;
    if (ar_init(3, N) != AR_OK) return 3;
    const long after = one_call(1);
    ar_free();
    const int ok = before == 0 && after == 0;
    printf("%s (mismatches before the reset %ld, after %ld)\n", ok ? "ok" : "FAIL", before, after);
    return ok ? 0 : 1;
}
