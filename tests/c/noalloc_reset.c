/* hs_swap_in_noalloc across a reset of the device's context, from plain C99
 * with buffers from the CUDA runtime alone.  The entry point keeps the
 * device address of its scratch array per device and context; after
 * cudaDeviceReset the primary context is created anew and the array must
 * be looked up again.  The program runs the same session twice with a
 * cudaDeviceReset in between.  A session creates a state, makes two
 * no-alloc calls over the same top-k and checks them against the host pool
 * it filled: the first call misses every token and each returned location
 * holds the token's host row, the second call hits every token.
 * Compiled by the test-suite with -std=c99 -Wall -Wextra -Werror -pedantic;
 * prints "ok" and exits 0 when every check passes. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "hisparse_swap.h"

enum { R = 3, L = 512, W = 656, H = 48, K = 40, B = 3 };

static int failures = 0;

static void expect(int cond, const char* what) {
    if (!cond) {
        fprintf(stderr, "FAILED: %s\n", what);
        ++failures;
    }
}

static uint8_t row_byte(int q, int t, int j) {
    return (uint8_t)((q * 29 + t * 11 + j * 3) & 0xff);
}

#define CK(call)                                                                   \
    do {                                                                           \
        cudaError_t e_ = (call);                                                   \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "CUDA error %s at %s\n", cudaGetErrorString(e_), #call); \
            return 2;                                                              \
        }                                                                          \
    } while (0)

static int session(int round) {
    hs_config c;
    memset(&c, 0, sizeof(c));
    c.num_requests = R;
    c.max_seq_len = L;
    c.item_size_bytes = W;
    c.hot_buffer_size = H;
    c.top_k = K;
    c.max_steps = 1;
    c.num_layers = 1;
    c.max_batch = B;
    c.index_kind = HS_INDEX_DENSE;
    if (hs_config_check(&c) != HS_OK) {
        fprintf(stderr, "config rejected\n");
        return 1;
    }
    const size_t pool_bytes = hs_host_pool_bytes(&c);
    const size_t kv_bytes = hs_device_kv_bytes(&c);
    const size_t st_bytes = hs_state_bytes(&c);
    const size_t ws_bytes = hs_workspace_bytes(&c);

    CK(cudaSetDevice(0));
    uint8_t* pool = NULL;
    CK(cudaHostAlloc((void**)&pool, pool_bytes, cudaHostAllocMapped));
    for (int q = 0; q < R; ++q)
        for (int t = 0; t < L; ++t)
            for (int j = 0; j < W; ++j) pool[((size_t)q * L + t) * W + j] = row_byte(q, t, j);
    void *kv = NULL, *state = NULL, *ws = NULL;
    CK(cudaMalloc(&kv, kv_bytes));
    CK(cudaMemset(kv, 0, kv_bytes));
    CK(cudaMalloc(&state, st_bytes));
    CK(cudaMalloc(&ws, ws_bytes));
    void* pools[1];
    void* kvs[1];
    pools[0] = pool;
    kvs[0] = kv;
    hs_state* st = NULL;
    expect(hs_create_state(&c, pools, kvs, state, st_bytes, ws, ws_bytes, NULL, &st) == HS_OK &&
               st != NULL,
           "state created");
    if (st == NULL) return 1;

    int32_t rpi[B], sl[B], topk[B * K];
    for (int b = 0; b < B; ++b) {
        rpi[b] = (b + round) % R;
        sl[b] = L;
        for (int k = 0; k < K; ++k) topk[b * K + k] = (b * 53 + k * 7 + round * 101) % L;
    }
    int32_t *d_rpi = NULL, *d_sl = NULL, *d_topk = NULL, *d_locs = NULL, *d_stats = NULL;
    CK(cudaMalloc((void**)&d_rpi, sizeof(rpi)));
    CK(cudaMalloc((void**)&d_sl, sizeof(sl)));
    CK(cudaMalloc((void**)&d_topk, sizeof(topk)));
    CK(cudaMalloc((void**)&d_locs, sizeof(int32_t) * B * K));
    CK(cudaMalloc((void**)&d_stats, sizeof(int32_t) * B * HS_NUM_STATS));
    CK(cudaMemcpy(d_rpi, rpi, sizeof(rpi), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_sl, sl, sizeof(sl), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_topk, topk, sizeof(topk), cudaMemcpyHostToDevice));

    int32_t locs[B * K], stats[B * HS_NUM_STATS];
    uint8_t* kv_host = (uint8_t*)malloc(kv_bytes);
    uint8_t want[W];
    if (kv_host == NULL) return 1;
    for (int call = 0; call < 2; ++call) {
        expect(hs_swap_in_noalloc(st, d_rpi, d_sl, d_topk, B, 1, 0, d_locs, d_stats, NULL, NULL,
                                  NULL, NULL) == HS_OK,
               "no-alloc swap-in accepted");
        CK(cudaDeviceSynchronize());
        uint32_t flags = 1u;
        expect(hs_get_status(st, &flags, NULL) == HS_OK && flags == 0u, "no device status flags");
        CK(cudaMemcpy(locs, d_locs, sizeof(locs), cudaMemcpyDeviceToHost));
        CK(cudaMemcpy(stats, d_stats, sizeof(stats), cudaMemcpyDeviceToHost));
        CK(cudaMemcpy(kv_host, kv, kv_bytes, cudaMemcpyDeviceToHost));
        for (int b = 0; b < B; ++b) {
            const int32_t* s = stats + b * HS_NUM_STATS;
            if (call == 0)
                expect(s[HS_STAT_UNIQUE_MISSES] == K && s[HS_STAT_ADMITTED] == K,
                       "first call: every token a miss, all admitted");
            else
                expect(s[HS_STAT_HITS] == K && s[HS_STAT_UNIQUE_MISSES] == 0,
                       "second call: every token a hit");
            const int q = rpi[b];
            for (int k = 0; k < K; ++k) {
                const int32_t loc = locs[b * K + k];
                if (loc < q * (H + K) || loc >= (q + 1) * (H + K)) {
                    expect(0, "location inside the request's rows");
                    continue;
                }
                for (int j = 0; j < W; ++j) want[j] = row_byte(q, topk[b * K + k], j);
                expect(memcmp(kv_host + (size_t)loc * W, want, W) == 0,
                       "the location holds the token's host row");
            }
        }
    }
    hs_destroy_state(st);
    free(kv_host);
    CK(cudaFree(d_rpi));
    CK(cudaFree(d_sl));
    CK(cudaFree(d_topk));
    CK(cudaFree(d_locs));
    CK(cudaFree(d_stats));
    CK(cudaFree(kv));
    CK(cudaFree(state));
    CK(cudaFree(ws));
    CK(cudaFreeHost(pool));
    return 0;
}

int main(void) {
    int rc = session(0);
    if (rc) return rc;
    if (cudaDeviceReset() != cudaSuccess) {
        fprintf(stderr, "cudaDeviceReset failed\n");
        return 2;
    }
    rc = session(1);
    if (rc) return rc;
    if (failures) return 1;
    printf("ok\n");
    return 0;
}
