/* Plain C use of the C ABI without a GPU: the header compiles as C11 on
 * its own and the host-only calls behave as documented. */
#include <stdio.h>
#include <string.h>

#include "ar.h"

int main(void) {
    const void *srcs[2] = {(const void *)0x100000, (const void *)0x200000};
    void *dsts[1] = {(void *)0x300000};
    int fails = 0;
    if (ar_check_args(2, srcs, dsts, 1, 64, 1024, AR_F32, AR_BF16) != AR_OK) fails++;
    if (ar_check_args(2, srcs, dsts, 1, 2048, 1024, AR_F32, AR_BF16) != AR_ERR_TOO_LARGE) fails++;
    if (ar_check_args(0, srcs, dsts, 1, 64, 1024, AR_F32, AR_BF16) != AR_ERR_INVALID_ARG) fails++;
    ar_layout L;
    memset(&L, 0, sizeof L);
    L.ne0 = 16;
    L.ne1 = 4;
    if (ar_check_layout(2, srcs, dsts, 1, &L, 1024, AR_F16, AR_F16) != AR_OK) fails++;
    if (strcmp(ar_status_string(AR_ERR_OVERLAP), "ok") == 0) fails++;
    int64_t v = 0;
    if (ar_query(AR_Q_RANKS, &v) != AR_ERR_NOT_INITIALIZED) fails++;
    ar_free();
    printf("%s\n", fails ? "FAIL" : "ok");
    return fails;
}
