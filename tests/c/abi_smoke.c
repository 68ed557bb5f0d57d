/* Plain C99 user of the swap-in library's C ABI (host-only calls: no GPU
 * needed).  Compiled with -std=c99 -Wall -Wextra -Werror -pedantic by the
 * test-suite and linked against the in-tree library; prints "ok" and exits 0
 * when every checked value matches. */
#include <stdio.h>
#include <string.h>

#include "hisparse_swap.h"

static int failures = 0;

static void expect(int cond, const char* what) {
    if (!cond) {
        fprintf(stderr, "FAILED: %s\n", what);
        ++failures;
    }
}

int main(void) {
    hs_config c;
    memset(&c, 0, sizeof(c));
    c.num_requests = 64;
    c.max_seq_len = 32768;
    c.item_size_bytes = 656;
    c.hot_buffer_size = 4096;
    c.top_k = 2048;
    c.max_steps = 1;
    c.num_layers = 2;
    c.max_batch = 64;
    c.index_kind = HS_INDEX_DENSE;
    c.extra_page_size = 256;
    expect(hs_config_check(&c) == HS_OK, "config accepted");
    expect(hs_device_kv_bytes(&c) == (size_t)64 * (4096 + 2048 + 256) * 656, "device kv bytes");
    expect(hs_host_pool_bytes(&c) == (size_t)64 * 32768 * 656, "host pool bytes");
    expect(hs_hash_size(&c) == 0, "no hash bank with the dense index");
    expect(hs_state_bytes(&c) > 0 && hs_workspace_bytes(&c) > 0, "state and workspace sizes");
    c.index_kind = HS_INDEX_HASH;
    expect(hs_hash_size(&c) == 8192, "hash bank of 2H entries");
    c.item_size_bytes = 650;
    expect(hs_config_check(&c) == HS_ERR_INVALID_ARG, "row size not a multiple of 16");
    expect(hs_state_bytes(&c) == 0, "no sizes for a rejected config");
    c.item_size_bytes = 656;
    c.hot_buffer_size = HS_MAX_HOT_BUFFER + 1;
    expect(hs_config_check(&c) == HS_ERR_UNSUPPORTED, "hot buffer above the limit");
    expect(hs_config_check(NULL) == HS_ERR_INVALID_ARG, "null config");
    expect(hs_swap_in(NULL, NULL, NULL, NULL, 1, 1, 0, NULL, NULL, NULL, NULL, NULL, NULL) ==
               HS_ERR_INVALID_ARG,
           "swap-in without a handle");
    expect(hs_append_rows(NULL, 0, NULL, NULL, NULL, NULL, 1, NULL) == HS_ERR_INVALID_ARG,
           "append without a handle");
    expect(strcmp(hs_status_string(HS_OK), "ok") == 0, "status string");
    expect(hs_version() == 20000, "version");
    hs_destroy_state(NULL);
    if (failures) return 1;
    printf("ok\n");
    return 0;
}
