// Gather kernel of the decode KV swap-in (sm_103a).
//
// A thread-block cluster of P CTAs resolves one batch row b (request
// q = req_pool_indices[b]): its S x K top-k entries form one working set (the
// multi-step swap report "[HiSparse] Support hisparse multi-step swap io
// kernel", section 实现拆解 item 1: gather flattens [batch, steps, top_k],
// looks tokens up in the hot cache's token -> slot hash and de-duplicates
// misses across steps).  CTA rank c owns the c-th contiguous slice of the
// flattened entries.  P is chosen so that B * P CTAs about fill the GPU.
//   1. each thread loads up to RMAX entries; an entry on the request's extra
//      page (its newest, still-filling page, the first lookup the same report
//      lists) is served from its extra row and skips everything below; the
//      others probe the request's token -> slot index (hash bank: linear
//      probing, all first probes issued before any resolves; or dense map);
//   2. misses are de-duplicated in a table distributed over the cluster's
//      shared memory: a token's home CTA and start position come from its
//      hash, its probe chain stays in the home CTA, and remote atomics keep
//      the smallest flat index and the set of steps it occurs in.
//      __match_any_sync first merges equal tokens inside a warp;
//   3. first occurrences are numbered j = 0, 1, ... in (step, k) order: a
//      block scan inside each CTA plus the totals of lower-ranked CTAs;
//   4. every entry gets its device row: q * (H + C) + phys[slot] for a hit,
//      q * (H + C) + phys[H + j] for miss j, R * (H + C) + q * E + t mod E
//      on the extra page.  Hit slots take the call's epoch;
//      unique misses are listed for the commit (token, last step) and the
//      copy (destination row).
// The row copy itself runs in the second kernel, spread over the whole GPU.
#include <cooperative_groups.h>

#include "hs_internal.cuh"

namespace cg = cooperative_groups;

namespace hs {
namespace {

constexpr int kMissPending = -2;  // code of an entry that missed the hash bank
// Entry codes: >= 0 hit slot; -1 invalid; <= -3 miss at dedup position (-3 - p),
// where p = home * sub_table_size + position in the home CTA's sub-table.
__device__ __forceinline__ int miss_code(int p) { return -3 - p; }
__device__ __forceinline__ int miss_pos(int code) { return -3 - code; }

// Inserts token t (flat index i, step-bit set `steps`) into its home CTA's
// sub-table (already mapped into this CTA's view); returns the position in
// that sub-table.  The whole table has at least twice as many entries as the
// request has entries, so a free position always exists.
__device__ __forceinline__ int dedup_insert(int* keys, int* first, unsigned* smask, int size,
                                            unsigned start, int t, int i, unsigned steps,
                                            uint32_t* status) {
    const unsigned mask = (unsigned)size - 1u;
    unsigned p = start;
    for (int n = 0; n < size; ++n) {
        const int k = atomicCAS(&keys[p], -1, t);
        if (k == -1 || k == t) {
            atomicMin(&first[p], i);
            atomicOr(&smask[p >> 2], steps << ((p & 3u) * 8u));
            return (int)p;
        }
        p = (p + 1u) & mask;
    }
    atomicOr(status, HS_STATUS_TABLE_FULL);
    return -1;
}

template <int RMAX>
__global__ void __launch_bounds__(1024, 1) gather_kernel(const SwapArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int P = (int)cluster.num_blocks();
    const int c = (int)cluster.block_rank();
    const int TS = a.dedup_size / P;  // this CTA's share of the dedup table
    const int ts_log = __ffs(TS) - 1;
    int* keys = reinterpret_cast<int*>(smem);
    int* first = keys + TS;                                     // first index, later ordinal
    unsigned* smask = reinterpret_cast<unsigned*>(first + TS);  // 8 step bits per position
    int* wcount = reinterpret_cast<int*>(smask + (TS >> 2));    // [RMAX][32] warp counts
    __shared__ int s_ok, s_epoch, s_total, s_cnt[4];

    const Dims& d = a.d;
    const int b = blockIdx.x / P;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int BD = blockDim.x, nwarps = BD >> 5;
    const int N = a.S * d.K;
    const int per = (N + P - 1) / P;
    const int lo = c * per, hi = min(N, lo + per);

    // ---- 0. independent loads first: request slot, length, this CTA's entries
    const int q = __ldg(a.rpi + b);
    const int sl = __ldg(a.seq_lens + b);
    const int32_t* topk_b = a.topk + (long long)b * N;
    int t[RMAX], code[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
        const int i = lo + r * BD + tid;
        t[r] = (i < hi) ? __ldg(topk_b + i) : -1;
    }
    const bool q_ok = q >= 0 && q < d.R;
    const int limit = sl < d.L ? sl : d.L;
    // first position of the extra page (past every valid token if none)
    const int xstart = (d.E > 0 && limit > 0) ? (limit - 1) / d.E * d.E : 0x7fffffff;
    unsigned xbits = 0u;  // bit r: entry r is on the extra page
    const long long base = (long long)q * (d.H + d.C);
    const int32_t* phys = a.lv.phys + base;
    for (int i = tid; i < TS; i += BD) {
        keys[i] = -1;
        first[i] = 0x7fffffff;
    }
    for (int i = tid; i < (TS >> 2); i += BD) smask[i] = 0u;
    if (tid < 4) s_cnt[tid] = 0;
    cluster.sync();  // every CTA of the cluster runs and its sub-table is empty
    // Let the commit + copy kernel launch now: its CTAs warm L2 with their
    // request's state while this grid works, and wait for this grid's
    // completion before reading anything it writes.
    pdl_trigger();

    // ---- 1. probe the hash bank (all first probes issued before any resolves)
    const long long* bank = a.lv.bank + (long long)(q_ok ? q : 0) * d.hash_size;
    const unsigned hmask = (unsigned)d.hash_size - 1u;
    {
        long long e[RMAX];
        unsigned pos[RMAX];
        const int16_t* map = a.lv.map + (long long)(q_ok ? q : 0) * d.L;
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
            const bool in_range = q_ok && (lo + r * BD + tid < hi) && t[r] >= 0 && t[r] < limit;
            const bool extra = in_range && t[r] >= xstart;
            const bool valid = in_range && !extra;  // goes through the index
            if (extra) xbits |= 1u << r;
            code[r] = valid ? kMissPending : -1;
            if (d.dense) {  // dense index: the slot is one load away, no chain
                e[r] = kEmpty;
                if (valid) {
                    const int slot = map[t[r]];
                    if (slot >= 0 && slot < d.H) code[r] = slot;
                }
                continue;
            }
            pos[r] = hash_token(t[r], d.hash_shift);
            e[r] = valid ? bank[pos[r]] : kEmpty;
        }
        if (c == 0 && tid == 0) {
            // The request lock and epoch, decided once and sent to every CTA.
            int ok = 1;
            if (!q_ok) {
                atomicOr(a.ws.status, HS_STATUS_BAD_REQUEST);
                ok = 0;
            } else if (atomicCAS(&a.lv.ctrl[(long long)q * kCtrlWords + CTRL_LOCK], 0, 1) != 0) {
                atomicOr(a.ws.status, HS_STATUS_DUPLICATE_REQUEST);
                ok = 0;
            }
            if (sl > d.L) atomicOr(a.ws.status, HS_STATUS_SEQ_LEN_CLAMPED);
            const int E = ok ? a.lv.ctrl[(long long)q * kCtrlWords + CTRL_EPOCH] : 0;
            for (int r = 0; r < P; ++r) {
                *cluster.map_shared_rank(&s_ok, r) = ok;
                *cluster.map_shared_rank(&s_epoch, r) = E;
            }
        }
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
            if (code[r] == -1) continue;
            for (int n = 0;; ++n) {
                const long long x = e[r];
                if (x == kEmpty) break;  // not resident
                if (x >= 0 && (int)(x >> 32) == t[r]) {
                    const int slot = (int)(x & 0xffffffffll);
                    if (slot < d.H) code[r] = slot;
                    else atomicOr(a.ws.status, HS_STATUS_PROBE_LIMIT);  // corrupt entry
                    break;
                }
                if (n + 1 >= d.hash_size) {
                    atomicOr(a.ws.status, HS_STATUS_PROBE_LIMIT);
                    break;
                }
                pos[r] = (pos[r] + 1u) & hmask;
                e[r] = bank[pos[r]];
            }
        }
    }
    // Hits: fetch the slot's physical row now (the epoch stamp waits for the lock).
    int hrow[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) hrow[r] = code[r] >= 0 ? phys[code[r]] : 0;

    // ---- 2. de-duplicate misses into the cluster-wide table ------------------
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
        const int i = lo + r * BD + tid;
        const bool miss = code[r] == kMissPending;
        const unsigned grp = __match_any_sync(0xffffffffu, miss ? t[r] : (-2 - lane));
        if (miss) {
            const int leader = __ffs(grp) - 1;
            const unsigned steps = __reduce_or_sync(grp, 1u << (i / d.K));
            int p = -1;
            if (lane == leader) {
                const unsigned h = hash_token(t[r], a.dedup_shift);
                const int home = (int)(h >> ts_log);
                const int lp = dedup_insert(cluster.map_shared_rank(keys, home),
                                            cluster.map_shared_rank(first, home),
                                            cluster.map_shared_rank(smask, home), TS,
                                            h & (unsigned)(TS - 1), t[r], i, steps, a.ws.status);
                p = lp >= 0 ? home * TS + lp : -1;
            }
            p = __shfl_sync(grp, p, leader);
            code[r] = p >= 0 ? miss_code(p) : -1;
        }
    }
    cluster.sync();  // the table is complete, s_ok / s_epoch have arrived

    int32_t* locs_b = a.locs + (long long)b * N;
    int32_t* cnt = a.ws.cnt + (long long)b * kCntWords;
    if (!s_ok) {
        // Rejected batch row: no location, no state change, nothing to copy.
        for (int i = lo + tid; i < hi; i += BD) locs_b[i] = -1;
        if (c == 0) {
            if (tid < kCntWords) cnt[tid] = (tid == CNT_SKIP) ? 1 : 0;
            if (a.stats && tid < HS_NUM_STATS) a.stats[(long long)b * HS_NUM_STATS + tid] = 0;
            if (a.plan_count && tid == 0) a.plan_count[b] = 0;
        }
        return;
    }
    const int E = s_epoch;
    int32_t* ep = a.lv.ep + (long long)q * d.H;
#pragma unroll
    for (int r = 0; r < RMAX; ++r)
        if (code[r] >= 0) ep[code[r]] = E;  // hit slots take the call's epoch

    // ---- 3. number the unique misses in (step, k) order ---------------------
    unsigned firstbits = 0u;
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
        const int i = lo + r * BD + tid;
        bool f = false;
        if (code[r] <= -3) {
            const int p = miss_pos(code[r]);
            f = *cluster.map_shared_rank(first + (p & (TS - 1)), p >> ts_log) == i;
        }
        const unsigned bal = __ballot_sync(0xffffffffu, f);
        if (lane == 0) wcount[r * nwarps + warp] = __popc(bal);
        if (f) firstbits |= 1u << r;
    }
    __syncthreads();
    if (warp == 0) {
        // exclusive scan of RMAX * nwarps warp counts in (r, warp) order
        const int n = RMAX * nwarps;
        const int per_lane = (n + 31) >> 5;
        int loc[RMAX];
        int sum = 0;
#pragma unroll
        for (int k = 0; k < RMAX; ++k) {
            const int idx = lane * per_lane + k;
            loc[k] = (k < per_lane && idx < n) ? wcount[idx] : 0;
            sum += loc[k];
        }
        const int inc = warp_inclusive_scan(sum);
        int run = inc - sum;
#pragma unroll
        for (int k = 0; k < RMAX; ++k) {
            const int idx = lane * per_lane + k;
            if (k < per_lane && idx < n) {
                wcount[idx] = run;
                run += loc[k];
            }
        }
        if (lane == 31) s_total = inc;
    }
    cluster.sync();  // every CTA's count of first occurrences is known
    int offset = 0, U = 0;
    for (int r = 0; r < P; ++r) {
        const int n = *cluster.map_shared_rank(&s_total, r);
        offset += r < c ? n : 0;
        U += n;
    }
    // First index -> ordinal (every read of the first indices is done).
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
        const bool f = (firstbits >> r) & 1u;
        const unsigned bal = __ballot_sync(0xffffffffu, f);
        if (f) {
            const int p = miss_pos(code[r]);
            *cluster.map_shared_rank(first + (p & (TS - 1)), p >> ts_log) =
                offset + wcount[r * nwarps + warp] + __popc(bal & lanemask_lt());
        }
    }
    cluster.sync();  // ordinals are in place

    // ---- 4. locations, miss lists, counters --------------------------------
    const long long wbase = (long long)b * d.C;
    int n_hit = 0, n_inv = 0, n_miss = 0, n_ext = 0;
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
        const int i = lo + r * BD + tid;
        if (i >= hi) continue;
        int loc;
        if ((xbits >> r) & 1u) {
            loc = (int)((long long)d.R * (d.H + d.C) + (long long)q * d.E + t[r] % d.E);
            ++n_ext;
        } else if (code[r] >= 0) {
            loc = (int)(base + hrow[r]);
            ++n_hit;
        } else if (code[r] == -1) {
            loc = -1;
            ++n_inv;
        } else {
            const int p = miss_pos(code[r]);
            const int home = p >> ts_log, lp = p & (TS - 1);
            const int j = *cluster.map_shared_rank(first + lp, home);
            loc = (int)(base + phys[d.H + j]);
            ++n_miss;
            if ((firstbits >> r) & 1u) {
                const unsigned m8 =
                    (*cluster.map_shared_rank(smask + (lp >> 2), home) >> ((lp & 3) * 8)) & 0xffu;
                a.ws.miss_tok[wbase + j] = t[r];
                a.ws.miss_last[wbase + j] = 31 - __clz((int)m8);
                a.ws.miss_dst[wbase + j] = loc;
                if (a.plan_src) {
                    a.plan_src[wbase + j] = (long long)q * d.L + t[r];
                    a.plan_dst[wbase + j] = loc;
                }
            }
        }
        locs_b[i] = loc;
    }
    n_hit = __reduce_add_sync(0xffffffffu, n_hit);
    n_inv = __reduce_add_sync(0xffffffffu, n_inv);
    n_miss = __reduce_add_sync(0xffffffffu, n_miss);
    n_ext = __reduce_add_sync(0xffffffffu, n_ext);
    if (lane == 0) {
        int* rc = cluster.map_shared_rank(s_cnt, 0);
        atomicAdd(&rc[0], n_hit);
        atomicAdd(&rc[1], n_inv);
        atomicAdd(&rc[2], n_miss);
        if (n_ext) atomicAdd(&rc[3], n_ext);
    }
    cluster.sync();  // counters complete; no remote access after this point
    if (c == 0 && tid == 0) {
        n_hit = s_cnt[0];
        n_inv = s_cnt[1];
        n_miss = s_cnt[2];
        cnt[CNT_U] = U;
        cnt[CNT_HITS] = n_hit;
        cnt[CNT_MISSES] = n_miss;
        cnt[CNT_INVALID] = n_inv;
        cnt[CNT_SKIP] = 0;
        cnt[CNT_Q] = q;
        if (a.stats) {
            int32_t* st = a.stats + (long long)b * HS_NUM_STATS;
            st[HS_STAT_HITS] = n_hit;
            st[HS_STAT_DUP_MISSES] = n_miss - U;
            st[HS_STAT_UNIQUE_MISSES] = U;
            st[HS_STAT_INVALID] = n_inv;
            st[HS_STAT_EXTRA] = s_cnt[3];
        }
        unsigned long long* tot = a.lv.totals;  // the layer's running sums
        atomicAdd(tot + HS_STAT_HITS, (unsigned long long)n_hit);
        atomicAdd(tot + HS_STAT_DUP_MISSES, (unsigned long long)(n_miss - U));
        atomicAdd(tot + HS_STAT_UNIQUE_MISSES, (unsigned long long)U);
        atomicAdd(tot + HS_STAT_INVALID, (unsigned long long)n_inv);
        atomicAdd(tot + HS_STAT_EXTRA, (unsigned long long)s_cnt[3]);
        if (a.plan_count) a.plan_count[b] = U;
    }
}

template <int RMAX>
cudaError_t launch_rmax(const SwapArgs& a, int cluster, int block, size_t smem, cudaStream_t s) {
    static SmemOptIn opt_in;
    cudaError_t e = ensure_smem(gather_kernel<RMAX>, smem, &opt_in);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.B * cluster);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gather_kernel<RMAX>, a);
}

}  // namespace

// CTAs per request: the largest power of two <= 8 with B * P CTAs still
// within one wave of `sms` SMs and at least 256 entries per CTA, but never
// more than 4096 entries per CTA (4 per thread).
int gather_cluster_size(int batch, int entries, int sms) {
    int p = 1;
    while (p < 8 && batch * (2 * p) <= sms && entries / (2 * p) >= 256) p *= 2;
    while (p < 8 && (entries + p - 1) / p > 4096) p *= 2;
    return p;
}

// Dynamic shared memory of one gather CTA: its 1/P share of a dedup table
// (keys, first index, step bits) with at least twice `entries` positions in
// all, and the warp counts.
size_t gather_smem_bytes(int entries, int cluster, int* dedup_size) {
    int t1 = 64;
    while (t1 < 2 * entries) t1 <<= 1;
    if (dedup_size) *dedup_size = t1;
    return (size_t)(t1 / cluster) * 9 + 8 * 32 * 4;
}

cudaError_t launch_gather(const SwapArgs& a, int sms, cudaStream_t s) {
    const int N = a.S * a.d.K;
    const int P = gather_cluster_size(a.B, N, sms);
    int t1 = 0;
    const size_t smem = gather_smem_bytes(N, P, &t1);
    SwapArgs g = a;
    g.dedup_size = t1;
    g.dedup_shift = 32 - __builtin_ctz((unsigned)t1);
    const int per = (N + P - 1) / P;  // entries per CTA
    if (per <= 1024) {
        const int block = ((per + 31) / 32) * 32 < 64 ? 64 : ((per + 31) / 32) * 32;
        return launch_rmax<1>(g, P, block, smem, s);
    }
    if (per <= 2048) return launch_rmax<2>(g, P, 1024, smem, s);
    return launch_rmax<4>(g, P, 1024, smem, s);  // per <= 4096 by the choice of P
}

}  // namespace hs
