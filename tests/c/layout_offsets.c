/* Prints the size and field offsets of ar_layout as a C compiler lays it out
 * from include/ar.h, for the binding's ctypes mirror to be checked against. */
#include <stddef.h>
#include <stdio.h>

#include "ar.h"

int main(void) {
    printf("size %zu\n", sizeof(ar_layout));
    printf("ne0 %zu\n", offsetof(ar_layout, ne0));
    printf("ne1 %zu\n", offsetof(ar_layout, ne1));
    printf("src_row_bytes %zu\n", offsetof(ar_layout, src_row_bytes));
    printf("dst_row_bytes %zu\n", offsetof(ar_layout, dst_row_bytes));
    printf("residual %zu\n", offsetof(ar_layout, residual));
    printf("residual_row_bytes %zu\n", offsetof(ar_layout, residual_row_bytes));
    printf("inactive_mask %zu\n", offsetof(ar_layout, inactive_mask));
    return 0;
}
