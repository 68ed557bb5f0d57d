/*
 * hisparse_swap.h -- C ABI of the GB300 decode KV swap-in library.
 *
 * The library resolves, for each decode step and layer, every request's
 * indexer top-k token indices against a per-request device hot buffer that
 * is backed by a pinned host KV pool, and returns the device row of every
 * selected token (plus, on request, a sparse page table).  One call:
 *   0. serves tokens on the request's extra page (its newest, still-filling
 *      page, when configured) without a lookup,
 *   1. looks the others up in the request's token -> slot index (hash bank
 *      or dense map),
 *   2. de-duplicates misses within and across the speculative steps,
 *   3. copies each unique miss's KV row from mapped pinned host memory into a
 *      scratch row of the device buffer,
 *   4. commits: marks the referenced hot slots, evicts the least recently
 *      referenced slots (epoch-CLOCK), rotates the scratch rows into the
 *      victims' hot slots and updates the hash.
 * Sources: "[HiSparse] Support hisparse multi-step swap io kernel" (PR
 * #32162 report), sections 功能与动机, 实现拆解 item 1-2, 关键源码片段
 * (HiSparseSpecState) and 风险与影响; PR #20343 summary, 实现拆解
 * (swap_in_selected_pages, device/host mapped pool); "SGLang HiSparse:
 * 当稀疏注意力从算法变为系统组件", sections 2.1 and 2.3.
 *
 * Conventions for every call:
 *  - Pointers named *_dev are device pointers; *_host are host pointers.
 *    A device pointer may also address mapped pinned host memory (with
 *    unified addressing, the pinned buffer's own address): the kernels then
 *    read or write it across the host link, e.g. NVLink-C2C on Grace.
 *    Arrays must be aligned to their element type (4 bytes for int32_t, 8
 *    for int64_t); a misaligned one returns HS_ERR_INVALID_ARG before any
 *    launch.
 *    The caller owns every buffer (pinned host pool, device KV buffers,
 *    state, workspace, inputs, outputs).  The library owns only the small
 *    host handle `hs_state`.  Buffer sizes follow from the config and the
 *    call's arguments as each function states; the kernels trust them (the
 *    Python binding checks tensor shapes before calling).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls are asynchronous on that stream unless stated.  Calls
 *    that share one hs_state must be ordered on one stream (or by events):
 *    they share the state and the workspace.  Separate handles are
 *    independent: their calls may run concurrently from several host
 *    threads and on several streams.
 *  - A handle belongs to the device that was current at hs_create_state.
 *    Every call on it must be made with that device current (and a stream
 *    of that device); otherwise it returns HS_ERR_INVALID_ARG and launches
 *    nothing.
 *  - Return value: HS_OK (0) or a negative HS_ERR_* code; nothing aborts or
 *    throws.  Argument errors are detected on the host before any launch.
 *    Data-dependent problems found by the kernels (request index out of
 *    range, a request twice in one call, seq_len above max_seq_len, hash
 *    probe limit) set bits in a device status word read by hs_get_status.
 *  - Token index t of batch row b is valid iff 0 <= t < min(seq_lens[b],
 *    max_seq_len); invalid entries get location -1 and change nothing.
 *  - Layouts (row-major, densest index last):
 *      host pool of layer l      uint8 [R, max_seq_len, W], row (q, t)
 *      device KV buffer of layer uint8 [R * (H + C) + R * E, W] with
 *                                C = max_steps * top_k, E = extra_page_size:
 *                                first request q's H hot + C scratch rows at
 *                                q * (H + C) + p, then request q's extra page
 *                                at R * (H + C) + q * E + (t mod E)
 *      top-k indices             int32 [B, S, top_k]
 *      device_locs               int32 [B, S, top_k]: row index into the
 *                                layer's device KV buffer
 */
#ifndef HISPARSE_SWAP_H
#define HISPARSE_SWAP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------ */
#define HS_OK 0
#define HS_ERR_INVALID_ARG (-1)   /* bad pointer, size, index or config      */
#define HS_ERR_UNSUPPORTED (-2)   /* valid but beyond this build's limits    */
#define HS_ERR_CUDA (-3)          /* a CUDA runtime call or launch failed    */
#define HS_ERR_DEVICE_STATUS (-4) /* hs_get_status found device flags set    */
#define HS_ERR_TIMEOUT (-5)       /* a bounded device wait gave up           */

/* ---- device status flags (hs_get_status) -------------------------------- */
#define HS_STATUS_BAD_REQUEST 0x1u       /* req_pool_indices[b] outside [0, R) */
#define HS_STATUS_DUPLICATE_REQUEST 0x2u /* a request twice in one call        */
#define HS_STATUS_SEQ_LEN_CLAMPED 0x4u   /* seq_lens[b] > max_seq_len          */
#define HS_STATUS_PROBE_LIMIT 0x8u       /* hash probe exceeded the table      */
#define HS_STATUS_TABLE_FULL 0x10u       /* hash insert found no free entry    */
#define HS_STATUS_BAD_APPEND 0x20u       /* hs_append_rows entry out of range  */
#define HS_STATUS_BAD_PLAN 0x40u         /* hs_copy_planned row/count out of range */

/* ---- per-request counters of one call (int32 [B, HS_NUM_STATS]) -------- */
#define HS_STAT_HITS 0          /* valid entries whose token was resident   */
#define HS_STAT_HIT_SLOTS 1     /* distinct hot slots those hits referenced */
#define HS_STAT_DUP_MISSES 2    /* miss entries repeating an earlier miss   */
#define HS_STAT_UNIQUE_MISSES 3 /* U: distinct non-resident valid tokens    */
#define HS_STAT_ADMITTED 4      /* m = min(U, H - hit slots)                */
#define HS_STAT_EVICTED 5       /* admitted into a slot that held a token   */
#define HS_STAT_OVERFLOW 6      /* U - m: served this call, not admitted    */
#define HS_STAT_INVALID 7       /* entries outside [0, min(seq_len, L_max)) */
#define HS_STAT_EXTRA 8         /* valid entries served by the extra page   */
#define HS_NUM_STATS 9

/* Limits of this build. */
#define HS_MAX_HOT_BUFFER 32768  /* hot_buffer_size upper bound (PR #32162 report, 风险与影响) */
#define HS_MAX_STEPS 4           /* speculative steps per call (same report, 实现拆解 item 2) */
#define HS_MAX_ENTRIES 8192      /* max_steps * top_k per request per call */
#define HS_MAX_PAGES 262144      /* ceil(max_seq_len / page_size) for hs_page_table */
#define HS_MAX_EXTRA_PAGE 65536  /* extra_page_size upper bound */
#define HS_MAX_ITEM_BYTES 65536  /* item_size_bytes upper bound (MLA rows are 656) */

typedef struct hs_config {
    int32_t num_requests;    /* R: request-pool slots (req_pool_indices range)    */
    int32_t max_seq_len;     /* L_max: host rows per request and layer            */
    int32_t item_size_bytes; /* W: bytes per KV row; a multiple of 16, at most
                                HS_MAX_ITEM_BYTES (656 = MLA)                     */
    int32_t hot_buffer_size; /* H: hot slots per request and layer, 1..32768      */
    int32_t top_k;           /* K: indices per request and step                   */
    int32_t max_steps;       /* S_max: 1..4 speculative steps                     */
    int32_t num_layers;      /* layers sharing one state object                   */
    int32_t max_batch;       /* B_max: requests per call, <= num_requests         */
    int32_t index_kind;      /* token -> slot index: HS_INDEX_HASH (0, default) or
                                HS_INDEX_DENSE (1); see below                       */
    int32_t extra_page_size; /* E: rows of each request's extra page, 0 = none;
                                see below                                          */
} hs_config;

/* Extra page (the first lookup of the report's gather, ahead of the hot-cache hash: "[HiSparse]
 * Support hisparse multi-step swap io kernel", 实现拆解 item 1; the page does not
 * define it, and this library reads it as the request's newest, still-filling
 * page).  With E > 0 every request q owns E device rows, and for a call with
 * n = min(seq_len, max_seq_len) the positions [floor((n - 1) / E) * E, n) are
 * the extra page: a selected token t there gets location
 * R * (H + C) + q * E + (t mod E) without a lookup, is neither a hit nor a
 * miss, changes no policy state and counts as HS_STAT_EXTRA.  The caller
 * fills those rows with hs_append_rows as decode produces them (and once for
 * the partial last page after prefill); the library never copies them from
 * the host pool. */

/* Token -> hot-slot index of each (layer, request).
 *   HS_INDEX_HASH: an open-addressing hash bank of hash_size int64 entries,
 *     (t << 32) | slot (the pages' per-request hash banks, PR #32162 report,
 *     关键源码片段).  Memory per (layer, request): 16 * H bytes or more; a
 *     lookup probes a short chain; evictions leave deleted entries that a
 *     rebuild clears.
 *   HS_INDEX_DENSE: a direct int16 map over the request's positions,
 *     slot_of[t] (-1 = not resident).  Memory per (layer, request):
 *     2 * max_seq_len bytes; a lookup is one load, an eviction or admission
 *     one store.  Results are identical; only speed and memory differ. */
#define HS_INDEX_HASH 0
#define HS_INDEX_DENSE 1

typedef struct hs_state hs_state; /* opaque host handle */

/* Returns HS_OK if `cfg` is valid and supported, else the error code.
 * Host only; no CUDA call.  The limits are the multi-step swap report's
 * (section 风险与影响: hot_buffer_size up to 32768; 实现拆解 item 2: up to 4
 * speculative steps) and this build's (HS_MAX_*). */
int hs_config_check(const hs_config* cfg);

/* Sizes the caller must allocate (0 if the config is not accepted).
 * Host only; no CUDA call.  The state holds what the multi-step swap
 * report's HiSparseSpecState holds (section 关键源码片段: the per-request
 * hash banks of cache_index, the reference epochs of cache_policy, the
 * reusable scratch locations and counters of scratch_locs / scratch_state),
 * in this library's layout; the host pool is the pinned pool that PR #20343
 * maps between device and host (PR #20343 summary, 实现拆解: the memory
 * pool extended with a device-host mapping).
 *   state:      device bytes, persistent cache state of all layers
 *               (hash banks, slot epochs, slot tokens, position table,
 *               control words)
 *   workspace:  device bytes, per-call scratch shared by all layers
 *   device_kv:  device bytes of ONE layer's KV buffer, R * (H + C + E) * W
 *   host_pool:  pinned host bytes of ONE layer's pool, R * L_max * W
 * `hash_size` is the entries of one request's hash bank (power of two), or 0
 * with HS_INDEX_DENSE. */
size_t hs_state_bytes(const hs_config* cfg);
size_t hs_workspace_bytes(const hs_config* cfg);
size_t hs_device_kv_bytes(const hs_config* cfg);
size_t hs_host_pool_bytes(const hs_config* cfg);
int32_t hs_hash_size(const hs_config* cfg);

/* Creates the host handle and initialises the state on `stream`: every
 * request empty, no token resident, position table the identity, epoch 0
 * (the persistent state of HiSparseSpecState, multi-step swap report,
 * section 关键源码片段; the pages do not state an initial value, and this
 * library reads it as an empty cache).
 *   host_pool_host[l]: host pool of layer l, 16-byte aligned.  Pinned memory
 *     (cudaHostAlloc'd or cudaHostRegister'ed) is used through its device
 *     mapping (cudaHostGetDevicePointer).  Plain pageable memory is accepted
 *     only on devices that read host page tables directly
 *     (cudaDevAttrPageableMemoryAccess, e.g. Grace NVLink-C2C systems);
 *     elsewhere it fails with HS_ERR_INVALID_ARG.
 *   device_kv_dev[l]: device KV buffer of layer l, 16-byte aligned.
 *   state_dev / workspace_dev: 256-byte aligned device memory of at least
 *     hs_state_bytes / hs_workspace_bytes.
 * The pointer arrays are copied; the memory they point to must outlive the
 * handle.  Synchronous with respect to the host only for the pointer
 * queries; the initialisation kernel runs on `stream`. */
int hs_create_state(const hs_config* cfg, void* const* host_pool_host,
                    void* const* device_kv_dev, void* state_dev, size_t state_bytes,
                    void* workspace_dev, size_t workspace_bytes, void* stream,
                    hs_state** out);

/* Frees the host handle only (never the caller's memory). NULL is a no-op.
 * (Lifetime of the handle of hs_create_state; no counterpart on the pages,
 * whose state object is a Python tuple of tensors.) */
void hs_destroy_state(hs_state* st);

/* One per-layer swap-in call (the page's swap_in_selected_pages(
 * req_pool_indices, seq_lens, topk_indices, layer_id)).
 *   req_pool_indices_dev int32 [batch]: distinct request slots in [0, R)
 *   seq_lens_dev         int32 [batch]
 *   topk_dev             int32 [batch, num_steps, top_k]
 *   batch                0..max_batch (0 is a no-op)
 *   num_steps            1..max_steps (1 = single-step decode)
 *   device_locs_dev      int32 [batch, num_steps, top_k] out
 *   stats_dev            int32 [batch, HS_NUM_STATS] out, or NULL
 *   miss_src_dev         int64 [batch, C] out or NULL: host row
 *                        (q * max_seq_len + t) of unique miss j
 *   miss_dst_dev         int64 [batch, C] out or NULL: device row it was
 *                        copied to (the location returned for it)
 *   miss_count_dev       int32 [batch] out or NULL: unique misses U
 *   (the three miss-plan pointers are all NULL or all non-NULL; entries
 *    j >= U are left untouched)
 * Locations stay valid until the next call on the same layer (extra-page
 * locations: until hs_append_rows rewrites that row).  Launches one kernel
 * on `stream`: each batch row's thread-block cluster looks up, de-duplicates
 * and locates its entries, then commits the request's policy state while
 * its other warps copy the request's miss rows. */
int hs_swap_in(hs_state* st, const int32_t* req_pool_indices_dev, const int32_t* seq_lens_dev,
               const int32_t* topk_dev, int32_t batch, int32_t num_steps, int32_t layer_id,
               int32_t* device_locs_dev, int32_t* stats_dev, int64_t* miss_src_dev,
               int64_t* miss_dst_dev, int32_t* miss_count_dev, void* stream);

/* Sparse page table of one call (PAGED mode: token -> page + in-page
 * offset; only pages holding selected tokens; "SGLang HiSparse" sections
 * 1.2, 2.1 and 2.3).  Stateless.  For batch row b:
 *   pages_dev      int32 [batch, num_steps * top_k]: the distinct pages
 *                  t / page_size of b's valid tokens, ascending, then -1
 *   num_pages_dev  int32 [batch]
 *   token_page_dev int32 [batch, num_steps, top_k]: for a valid token,
 *                  (index of its page in pages[b]) * page_size +
 *                  t % page_size; -1 for an invalid one.
 * Validity as in hs_swap_in with L_max = max_seq_len.  Requires
 * ceil(max_seq_len / page_size) <= HS_MAX_PAGES and num_steps * top_k <=
 * HS_MAX_ENTRIES. */
int hs_page_table(const int32_t* topk_dev, const int32_t* seq_lens_dev, int32_t batch,
                  int32_t num_steps, int32_t top_k, int32_t max_seq_len, int32_t page_size,
                  int32_t* pages_dev, int32_t* num_pages_dev, int32_t* token_page_dev,
                  void* stream);

/* Write-back of newly decoded KV rows of layer `layer_id` (decode keeps idle
 * KV in host memory: PR #20343 summary, 功能与动机).
 *   req_dev      int32 [n]: request slot q of entry i
 *   tok_dev      int32 [n]: position t of entry i
 *   seq_lens_dev int32 [n]: the request's length once entry i is in (t < it)
 *   rows_dev     uint8 [n, W], 16-byte aligned, device memory: the KV rows
 * For every entry with 0 <= q < R and 0 <= t < min(seq_len, max_seq_len):
 *   - host pool row (q, t) := the row (written through the pool's device
 *     mapping; the caller's pool memory is modified);
 *   - if E > 0 and t lies on the extra page of length seq_len: extra-page
 *     row R * (H + C) + q * E + (t mod E) := the row;
 *   - if t is resident in a hot slot of (layer_id, q): that slot's device
 *     row := the row.
 * So every copy of (q, t) stays equal.  Other entries are skipped and set
 * HS_STATUS_BAD_APPEND.  The (q, t) pairs of one call must be distinct
 * (with duplicates the rows written are unspecified).  Order it on the same
 * stream as the swap-ins of the layer: before the swap-in whose selection
 * may include the appended tokens.  Asynchronous on `stream`; n = 0 is a
 * no-op. */
int hs_append_rows(hs_state* st, int32_t layer_id, const int32_t* req_dev,
                   const int32_t* tok_dev, const int32_t* seq_lens_dev, const void* rows_dev,
                   int32_t n, void* stream);

/* Returns requests to the empty state in every layer (use when a request
 * slot is given to a new sequence; order it after the previous user's last
 * call and before the new user's first call on `stream`: the PR #20343
 * summary, sections 评论区精华 and 风险与影响, reports an illegal-address
 * crash when admitting a request into staging was not ordered by a stream
 * wait under overlapped scheduling).  Only policy
 * state is reset: KV rows (host pool, device buffer, extra page) are left as
 * they are, and the new sequence's rows arrive through its own prefill and
 * hs_append_rows. */
int hs_reset_requests(hs_state* st, const int32_t* req_pool_indices_dev, int32_t n,
                      void* stream);

/* Synchronises `stream`, returns the device status flags (HS_STATUS_*) in
 * *flags_out and clears them.  Returns HS_ERR_DEVICE_STATUS if any flag was
 * set, HS_OK otherwise.  (No counterpart on the pages: the kernels record
 * out-of-range request slots, duplicate requests and probe limits here
 * instead of touching memory out of bounds, the kind of fault the PR #20343
 * summary, section 评论区精华, reports as cudaErrorIllegalAddress.) */
int hs_get_status(hs_state* st, uint32_t* flags_out, void* stream);

/* Running sums of the per-request counters (HS_STAT_*) of layer `layer_id`
 * (the pages count a call's unique cross-step misses in their test: the
 * multi-step swap report, section 实现拆解 item 4, 782 unique misses)
 * over every swap-in call since the handle was created or last read with
 * `reset` (a monitoring aid: hit rate, misses, evictions, overflow).  Rows
 * rejected on the device add nothing.  Copies HS_NUM_STATS int64 values to
 * totals_host (indexed by HS_STAT_*) and synchronises `stream`; reset != 0
 * then sets the sums to zero (ordered on `stream`). */
int hs_get_stats(hs_state* st, int32_t layer_id, int64_t* totals_host, int32_t reset,
                 void* stream);

/* Copies one request's policy state of one layer to host memory and
 * synchronises `stream` (checkpointing and tests; the state is that of
 * HiSparseSpecState, multi-step swap report, section 关键源码片段, in this
 * library's layout).  Any output may be NULL.
 *   tok_host  int32 [H]: token held by each hot slot, -1 if empty
 *   ep_host   int32 [H]: epoch of the slot's last reference, -1 if never
 *   phys_host int32 [H + C]: physical row of each position (a permutation)
 *   ctrl_host int32 [8]: {next epoch, resident count, used hash entries, ...}
 *   bank_host int64 [hash_size]: hash entries (t << 32 | slot), -1 empty,
 *             -2 deleted; with HS_INDEX_DENSE it receives the request's map
 *             instead, widened: int64 [max_seq_len], slot or -1 */
int hs_export_request_state(hs_state* st, int32_t layer_id, int32_t request, int32_t* tok_host,
                            int32_t* ep_host, int32_t* phys_host, int32_t* ctrl_host,
                            int64_t* bank_host, void* stream);

/* Deferred-copy mode of the miss-plan protocol (the multi-step swap report,
 * sections 实现拆解 item 2 and 风险与影响: the miss_src / miss_dst /
 * miss_count plan lets the row copies be replayed by a prefetch path).
 * When `defer` is non-zero, later hs_swap_in calls on this handle must be
 * given the three miss-plan outputs and do not copy rows: they resolve
 * locations and commit the policy state only.  The caller then runs
 * hs_copy_planned with that plan, on any stream, ordered after the call and
 * before (a) anything that reads the returned rows and (b) the next
 * hs_swap_in on the same layer (whose scratch rows may be the same).
 * 0 restores copying inside hs_swap_in.  Host only. */
int hs_set_defer_copy(hs_state* st, int32_t defer);

/* Copies the rows of a recorded miss plan: for batch row b and j <
 * miss_count[b], host row miss_src[b, j] of layer `layer_id`'s pool to
 * device row miss_dst[b, j] of its device buffer (W bytes each).  The plan
 * is exactly what hs_swap_in wrote ([batch, C] with C = max_steps * top_k).
 * A count outside [0, C] is clamped and a row outside the pool or the
 * device buffer is skipped; either sets HS_STATUS_BAD_PLAN.  Asynchronous on
 * `stream`. */
int hs_copy_planned(hs_state* st, int32_t layer_id, const int64_t* miss_src_dev,
                    const int64_t* miss_dst_dev, const int32_t* miss_count_dev, int32_t batch,
                    void* stream);

/* Profiling (no counterpart on the pages): when `timeline_dev` is non-NULL,
 * every later hs_swap_in (and hs_swap_in_noalloc) on this handle writes the
 * phase times of its CTAs there, as uint64 [batch][8][16] indexed by batch
 * row, cluster rank and word (8-byte aligned device memory of at least
 * max_batch * 128 words; rows of ranks the call does not use are left
 * untouched).  Words 0-10 are nanoseconds of the GPU's global timer, taken
 * by the CTA's first thread once the data named has arrived: 0 CTA start,
 * 1 its index probes answered, 2 past the first cluster barrier (the
 * de-duplication tables cleared), 3 its de-duplication inserts issued,
 * 4 past the second barrier (the tables complete), 5 its first-occurrence
 * flags known, 6 past the third barrier (flag words and counts exchanged),
 * 7 its hit and miss rows loaded, 8 past the fourth barrier (locations and
 * miss lists written), 9 commit done (rank 0 only), 10 its last warp done
 * copying.  Word 15 is the cluster size; words 11-14 are unused.  A
 * rejected batch row writes words 0-4 and 15 only.  Recording costs a few
 * instructions of each CTA's first thread.  NULL turns it off.  Host only. */
int hs_set_timeline(hs_state* st, uint64_t* timeline_dev);

/* Tuning: CTAs of hs_copy_planned.  0 restores the default (twice the SM
 * count); otherwise 1..65535.  Host only.  (The pages flag a hard-coded
 * launch shape as a risk on other hardware: PR #20343 summary, 风险与影响,
 * block_size=256; this keeps the replay's grid a parameter.) */
int hs_set_copy_ctas(hs_state* st, int32_t copy_ctas);

/* Size of the per-call scratch array of hs_swap_in_noalloc (16 MiB). */
#define HS_NOALLOC_SCRATCH_BYTES (16u << 20)

/* hs_swap_in for callers that cannot allocate device memory.  The pages have
 * no counterpart to this entry point.
 *
 * Some callers cannot call cudaMalloc, or any routine that allocates, on the
 * path that issues swap-ins.  Examples: a plugin that a serving runtime hands
 * only its input and output tensors, and a runtime whose device memory all
 * comes from its own pool, reserved up front, where an allocation behind its
 * back could fail or fragment that pool.  This call takes the same arguments
 * as hs_swap_in and gives the same results.  Its per-call scratch (miss
 * lists, admission list, per-batch-row words) lives in one
 * file-scope device array of HS_NOALLOC_SCRATCH_BYTES, not in the handle's
 * workspace.  Every GPU that loads the library holds that array until the
 * process exits.  The call allocates nothing.
 *   - A call needs 4 * align256(4 * batch * C) + align256(64 * batch) bytes
 *     (C = max_steps * top_k).  A larger call returns HS_ERR_UNSUPPORTED
 *     before any launch; e.g. batch 64 with C = 8192 needs 8.4 MB.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and so does the first
 *     call after the device's context was created again (for example after
 *     cudaDeviceReset): an address is kept per device and context.  Make
 *     that first call before any stream capture.
 *   - All calls share the array, and it keeps the last call's contents.
 *     Nothing in it needs clearing: a call zeroes the words it counts with
 *     and writes every list entry before it reads it.  Calls whose kernels
 *     can overlap on the GPU (other streams, other handles, no ordering
 *     between them) race on the array: order them.
 *   - Device status flags still go to the handle (read with hs_get_status).
 * Everything else (state, host pool, device buffer, deferred-copy and
 * timeline settings) is the handle's, as for hs_swap_in. */
int hs_swap_in_noalloc(hs_state* st, const int32_t* req_pool_indices_dev,
                       const int32_t* seq_lens_dev, const int32_t* topk_dev, int32_t batch,
                       int32_t num_steps, int32_t layer_id, int32_t* device_locs_dev,
                       int32_t* stats_dev, int64_t* miss_src_dev, int64_t* miss_dst_dev,
                       int32_t* miss_count_dev, void* stream);

/* Static string for a return code (no counterpart on the pages). */
const char* hs_status_string(int code);

/* Library ABI version (major * 10000 + minor * 100 + patch; no counterpart
 * on the pages). */
int32_t hs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HISPARSE_SWAP_H */
