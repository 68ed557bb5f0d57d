/*
 * CPU oracle of the decode KV swap-in (test infrastructure only).
 *
 * This header belongs to the oracle, a plain, slow, obviously correct CPU
 * restatement of the swap-in that the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg compare the CUDA library against.  Nothing in
 * the product path includes, links or loads it, and it shares no code with
 * the CUDA library.
 *
 * All arguments are host pointers.  Sizes and layouts match the library's
 * public contract: top-k indices int32 [B, S, K]; host pool uint8
 * [R, L_max, W] per layer; device-buffer mirror uint8 [R * (H + C + E), W]
 * per layer with C = max_steps * top_k and E = extra_page_size: rows
 * q * (H + C) + p of the hot slots and scratch ring, then the extra-page
 * rows R * (H + C) + q * E + (t mod E); returned locations are rows of that
 * buffer.
 */
#ifndef HS_ORACLE_H
#define HS_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HSO_OK 0
#define HSO_ERR_ARG (-1)
#define HSO_ERR_DUPLICATE_REQUEST (-2)

/* Per-request counters of one call, in this order. */
#define HSO_STAT_HITS 0          /* valid entries whose token was resident */
#define HSO_STAT_HIT_SLOTS 1     /* distinct hot slots referenced by hits */
#define HSO_STAT_DUP_MISSES 2    /* miss entries repeating an earlier miss */
#define HSO_STAT_UNIQUE_MISSES 3 /* U: distinct non-resident valid tokens */
#define HSO_STAT_ADMITTED 4      /* m = min(U, H - hit slots) */
#define HSO_STAT_EVICTED 5       /* admitted into a slot that held a token */
#define HSO_STAT_OVERFLOW 6      /* U - m: misses served but not admitted */
#define HSO_STAT_INVALID 7       /* entries outside [0, min(seq_len, L_max)) */
#define HSO_STAT_EXTRA 8         /* valid entries served by the extra page */
#define HSO_NUM_STATS 9

typedef struct hso_oracle hso_oracle;

hso_oracle* hso_create(int32_t num_requests, int32_t max_seq_len, int32_t item_size_bytes,
                       int32_t hot_buffer_size, int32_t top_k, int32_t max_steps,
                       int32_t num_layers, int32_t extra_page_size);
void hso_destroy(hso_oracle* o);

/* One swap-in call for `layer`.  `stats` [B, HSO_NUM_STATS], `miss_src`/`miss_dst`
 * [B, C] and `miss_count` [B] may be NULL.  num_threads <= 1 runs the
 * requests one after the other; more splits them over std::threads. */
int hso_swap_in(hso_oracle* o, int32_t layer, const uint8_t* host_pool, uint8_t* device_kv,
                const int32_t* req_pool_indices, const int32_t* seq_lens,
                const int32_t* topk, int32_t batch, int32_t num_steps,
                int32_t* device_locs, int32_t* stats, int64_t* miss_src,
                int64_t* miss_dst, int32_t* miss_count, int32_t num_threads);

/* Write-back of newly decoded rows of `layer`: for each i with request
 * q = req[i] in [0, R) and position t = tok[i] in [0, min(seq_lens[i], L_max)):
 * host row (q, t) := rows[i]; the extra-page row of t := rows[i] when E > 0
 * and t lies in the extra page of length seq_lens[i]; the hot row of t :=
 * rows[i] when t is resident.  Other entries are skipped.  Entries are
 * applied in order.  Returns the number skipped, or HSO_ERR_ARG. */
int hso_append_rows(hso_oracle* o, int32_t layer, uint8_t* host_pool, uint8_t* device_kv,
                    const int32_t* req, const int32_t* tok, const int32_t* seq_lens,
                    const uint8_t* rows, int32_t n);

/* Copies the policy state of (layer, q): tok [H], ep [H], phys [H + C], epoch. */
int hso_get_request_state(const hso_oracle* o, int32_t layer, int32_t q, int32_t* tok,
                          int32_t* ep, int32_t* phys, int32_t* epoch);

/* Returns requests to the empty state in every layer. */
int hso_reset_requests(hso_oracle* o, const int32_t* req_pool_indices, int32_t n);

/* Sparse page table of one call (independent of the cache state).  An entry
 * is valid iff 0 <= t < min(seq_len, max_seq_len), as in hso_swap_in. */
int hso_page_table(const int32_t* topk, const int32_t* seq_lens, int32_t batch,
                   int32_t num_steps, int32_t top_k, int32_t max_seq_len, int32_t page_size,
                   int32_t* pages, int32_t* num_pages, int32_t* token_page);

#ifdef __cplusplus
}
#endif

#endif /* HS_ORACLE_H */
