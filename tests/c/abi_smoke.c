/* A plain C99 caller of libattn.so: compiled by the CPU test suite against
 * include/attn.h (no C++, no torch), it checks the calls a host program
 * makes before any device work -- status strings, sizes, the chunk plan of
 * the host-buffer prefill, and host-side argument rejection. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "attn.h"

static int fails = 0;
#define CHECK(cond)                                                   \
    do {                                                              \
        if (!(cond)) {                                                \
            fprintf(stderr, "FAILED %s:%d: %s\n", __FILE__, __LINE__, #cond); \
            ++fails;                                                  \
        }                                                             \
    } while (0)

int main(void) {
    CHECK(strcmp(attn_status_str(ATTN_OK), "ATTN_OK") == 0);
    CHECK(strcmp(attn_status_str(ATTN_ERR_TIMEOUT), "ATTN_ERR_TIMEOUT") == 0);
    CHECK(strcmp(attn_status_str((attn_status)99), "ATTN_UNKNOWN_STATUS") == 0);

    /* workspace sizes: positive for valid sizes, 0 for invalid ones */
    CHECK(attn_decode_workspace_bytes(64, 32, 128, 32768) > 0);
    CHECK(attn_decode_workspace_bytes(0, 32, 128, 32768) == 0);
    CHECK(attn_backward_workspace_bytes(1, 64, 32768) == (size_t)64 * 32768 * 4);

    /* 64 query heads, 8 KV heads, 32768 rows: two heads per chunk by default */
    CHECK(attn_prefill_from_host_heads_per_chunk(1, 64, 8, 32768, 128, 0, 148) == 2);
    CHECK(attn_prefill_from_host_heads_per_chunk(1, 64, 8, 32768, 128, 8, 148) == 8);
    CHECK(attn_prefill_from_host_heads_per_chunk(1, 4, 3, 128, 128, 0, 148) == 0);

    /* host-side rejection before any launch (no device is touched) */
    void *fake = (void *)(uintptr_t)(1u << 20);
    CHECK(attn_prefill(NULL, fake, fake, fake, NULL, 1, 4, 2, 128, 128, 128, 1, 0.1f, ATTN_BF16,
                       ATTN_BF16, NULL, NULL, NULL, NULL) == ATTN_ERR_INVALID);
    CHECK(attn_prefill(fake, fake, fake, fake, NULL, 1, 4, 2, 128, 128, 96, 1, 0.1f, ATTN_BF16,
                       ATTN_BF16, NULL, NULL, NULL, NULL) == ATTN_ERR_UNSUPPORTED);
    CHECK(attn_prefill(fake, fake, fake, fake, NULL, 1, 4, 2, 256, 128, 128, 1, 0.1f, ATTN_BF16,
                       ATTN_BF16, NULL, NULL, NULL, NULL) == ATTN_ERR_INVALID);
    CHECK(attn_prefill_from_host(fake, fake, fake, fake, NULL, fake, fake, fake, fake, NULL, 1, 4,
                                 2, 128, 128, 128, 1, 0.1f, ATTN_BF16, ATTN_BF16, NULL, NULL,
                                 NULL, -1, NULL) == ATTN_ERR_INVALID);
    CHECK(attn_last_launch_count() == 0);

    if (fails == 0)
        printf("c abi ok\n");
    return fails == 0 ? 0 : 1;
}
