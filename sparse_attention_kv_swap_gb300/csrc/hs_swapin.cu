// Swap-in kernel of the decode KV swap-in (sm_103a): one launch per
// layer-call does the lookup, the miss de-duplication, the locations, the
// policy commit and the miss-row copy.
//
// A thread-block cluster of P CTAs serves one batch row b (request
// q = req_pool_indices[b]).  Its S x K top-k entries form one working set
// (the multi-step swap report "[HiSparse] Support hisparse multi-step swap io
// kernel", section 实现拆解 item 1: the gather flattens [batch, steps, top_k],
// looks tokens up in the hot cache's token -> slot index and de-duplicates
// misses across steps; the commit updates CLOCK state, rotates scratch and
// hot locations and updates the index).  CTA rank c owns the c-th contiguous
// slice of the flattened entries; entry (s, k) has flat index i = s * K + k.
//   1. each thread loads up to RMAX entries; an entry on the request's extra
//      page (its newest, still-filling page, the first lookup the same
//      report lists) is served from its extra row; the others probe the
//      request's token -> slot index (dense map: one load; hash bank: linear
//      probing with every first probe issued before any resolves);
//   2. misses go into a de-duplication table spread over the cluster's
//      shared memory, which keeps for each token the smallest key (rank and
//      local index, ordered as flat indices are) of the entries at which it
//      occurs and the set of steps it occurs in.  When the table
//      fits, it is indexed by the token's position (home CTA t mod P, entry
//      t / P) and an insert is one fire-and-forget atomic (two in a
//      multi-step call that may overflow); otherwise it is a hash table
//      with linear probing (compare-and-swap inserts).  Step 1 touches no
//      other CTA's shared memory, so it runs inside the first cluster
//      barrier; hit slots are marked in a shared-memory bitmap inside the
//      second;
//   3. an entry is the first occurrence of its token iff the table holds its
//      own key.  Each CTA turns its first-occurrence flags into 64-bit words
//      (running count << 32 | flags of 32 entries) and sends them and its
//      total to every CTA of the cluster, its entry counters and hit bits to
//      the leader;
//   4. the ordinal j of a miss is the number of first occurrences before
//      its token's first occurrence: the totals of lower-ranked CTAs plus
//      that CTA's running count and flags up to it, all read from local
//      shared memory.  Every entry gets its device row (q * (H + C) +
//      phys[slot] for a hit, q * (H + C) + phys[H + j] for miss j,
//      R * (H + C) + q * E + t mod E on the extra page); first occurrences
//      list their token, last step and device row, and every location is
//      stored inside the last cluster barrier;
//   5. the leader CTA (rank 0) commits the request's policy state
//      (epoch-CLOCK victims, admission, rotation, index update), while the
//      other CTAs of the cluster copy the request's miss rows from the
//      mapped pinned host pool in chunks of 16-byte pieces (each warp's
//      first chunk by its index, the rest claimed from a per-batch-row
//      counter); the leader joins the copy when it is done.  A cluster of one
//      CTA commits on 16 of its warps and copies on the others.
// A request's copy thus starts as soon as its own lookup is complete; no
// CTA waits for another batch row.  The commit rewrites only policy state,
// the copy only device KV rows, so the two never touch the same memory.
#include <cooperative_groups.h>

#include "hs_internal.cuh"

namespace cg = cooperative_groups;

namespace hs {
namespace {

constexpr int kMaxCluster = 8;
constexpr int kMissPending = -2;    // code of an entry that missed the index
constexpr int kNoFirst = 0x7fffffff;  // de-duplication entry not yet seen
constexpr int kCopyUnroll = 4;
constexpr int kWarpPieces = 32 * kCopyUnroll;  // 16-byte pieces a warp takes at once
constexpr int kCommitWarps = 16;               // the leader CTA's commit warps (at most)
constexpr unsigned kHitKey = 0xffffffffu;      // radix key of a slot referenced by the call
constexpr int kKeyBatch = 8;                    // epochs a commit thread loads at once
// Shared memory one CTA may spend on its share of a position-indexed
// de-duplication table (4 bytes a position, 8 when the call may overflow);
// longer sequences use the hashed table.
constexpr int kPositionTableBytes = 160 * 1024;

// Entry keys: the entry at local index l (flat index lo + l) of cluster
// rank c has key c * kKeyStride + l.  Keys order entries as their flat
// indices do (l < per <= HS_MAX_ENTRIES = kKeyStride), fit in 16 bits for
// up to 8 ranks, and give the owning rank and local index by shift and
// mask, where the flat index would need a division by per.
constexpr int kKeyShift = 13;
constexpr int kKeyStride = 1 << kKeyShift;
static_assert(kKeyStride >= HS_MAX_ENTRIES && kMaxCluster * kKeyStride <= 0x10000,
              "entry keys must cover a rank's entries and fit in 16 bits");

// Entry codes: >= 0 hit slot; -1 invalid; kMissPending; after step 2
// <= -3 a miss in the de-duplication table at entry (u * 8 + home); after
// step 3 <= -3 a miss whose token first occurs at the entry with key
// (-3 - code) & 0xffff and last occurs in step (-3 - code) >> 16.
__device__ __forceinline__ int miss_code(int x) { return -3 - x; }
__device__ __forceinline__ int miss_value(int code) { return -3 - code; }

// The two halves of a cluster barrier (barrier.cluster.arrive / wait, with
// release and acquire semantics): a thread arrives once its writes for the
// other CTAs are issued and waits only where it needs theirs, so work that
// needs neither runs in between.  Called by whole warps.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Step of flat index i < S * K (S <= HS_MAX_STEPS = 4), without a division.
__device__ __forceinline__ int step_of(int i, int K) {
    return (i >= K) + (i >= 2 * K) + (i >= 3 * K);
}
static_assert(HS_MAX_STEPS <= 4, "step_of covers four steps");

// Timeline stamp once the values in v (loads in flight) have arrived: the
// empty asm consumes each value, so the timer is read after the data.
template <int N>
__device__ __forceinline__ void stamp_after(unsigned long long* tl, int word, const int (&v)[N]) {
#pragma unroll
    for (int r = 0; r < N; ++r) asm volatile("" ::"r"(v[r]));
    tl[word] = global_timer();
}

// Warps [0, n / 32) of the CTA, synchronising on named barrier 1 (the
// leader CTA's commit warps, while its other warps copy).
struct Group {
    int tid, n;
    __device__ void sync() const { asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory"); }
};

// Exclusive scan of one int per group thread; returns the prefix and the
// group total.  `tmp` needs 33 ints of shared memory.
__device__ int group_exclusive_scan(const Group& g, int x, int* tmp, int* total) {
    const int lane = g.tid & 31, warp = g.tid >> 5, nwarps = g.n >> 5;
    const int inc = warp_inclusive_scan(x);
    if (lane == 31) tmp[warp] = inc;
    g.sync();
    if (warp == 0) {
        const int w = lane < nwarps ? tmp[lane] : 0;
        const int wi = warp_inclusive_scan(w);
        tmp[lane] = wi - w;
        if (lane == 31) tmp[32] = wi;
    }
    g.sync();
    const int r = tmp[warp] + inc - x;
    *total = tmp[32];
    g.sync();
    return r;
}

__device__ int group_sum(const Group& g, int x, int* tmp) {
    int total;
    group_exclusive_scan(g, x, tmp, &total);
    return total;
}

// Hashed de-duplication: inserts token t (entry key `key`, step bits `steps`)
// into its home CTA's share (already mapped into this CTA's view) starting
// at `start`; returns the entry.  The whole table has at least twice as
// many entries as the request has entries, so a free one always exists.
__device__ __forceinline__ int dedup_insert(int* keys, int* first, unsigned* smask, int size,
                                            unsigned start, int t, int key, unsigned steps,
                                            uint32_t* status) {
    const unsigned mask = (unsigned)size - 1u;
    unsigned p = start;
    for (int n = 0; n < size; ++n) {
        const int k = atomicCAS(&keys[p], -1, t);
        if (k == -1 || k == t) {
            atomicMin(&first[p], key);
            atomicOr(&smask[p >> 2], steps << ((p & 3u) * 8u));
            return (int)p;
        }
        p = (p + 1u) & mask;
    }
    atomicOr(status, HS_STATUS_TABLE_FULL);
    return -1;
}

// ---- commit (policy state of one request) -----------------------------------

// Deletes token t from a request's hash bank (the entry must exist).
__device__ void bank_delete(long long* bank, int shift, unsigned mask, int32_t t,
                            uint32_t* status) {
    unsigned p = hash_token(t, shift);
    for (unsigned n = 0; n <= mask; ++n) {
        const long long x = bank[p];
        if (x == kEmpty) break;
        if (x >= 0 && (int)(x >> 32) == t) {
            bank[p] = kDeleted;
            return;
        }
        p = (p + 1u) & mask;
    }
    atomicOr(status, HS_STATUS_PROBE_LIMIT);
}

// Inserts (t, slot) at the first empty or deleted entry of t's probe
// sequence; returns 1 if the entry was never used before.
__device__ int bank_insert(long long* bank, int shift, unsigned mask, int32_t t, int32_t slot,
                           uint32_t* status) {
    const long long e = make_entry(t, slot);
    unsigned p = hash_token(t, shift);
    for (unsigned n = 0; n <= mask; ++n) {
        long long x = bank[p];
        while (x < 0) {
            const long long y = atomicCAS(reinterpret_cast<unsigned long long*>(&bank[p]),
                                          (unsigned long long)x, (unsigned long long)e);
            if (y == x) return x == kEmpty ? 1 : 0;
            x = y;
        }
        p = (p + 1u) & mask;
    }
    atomicOr(status, HS_STATUS_TABLE_FULL);
    return 0;
}

// Finds the `need`-th smallest key (1-based) among keys[0..n) that are not
// kHitKey, by most-significant-digit radix select over `bits` bits.
// Returns the key; *need_out is how many keys equal to it to take.
__device__ unsigned radix_select(const Group& g, const unsigned* keys, int n, int need, int bits,
                                 int* hist, int* sh, int* need_out) {
    unsigned prefix = 0u;
    const int top = ((bits + 7) / 8) * 8;
    for (int shift = top - 8; shift >= 0; shift -= 8) {
        for (int i = g.tid; i < 256; i += g.n) hist[i] = 0;
        g.sync();
        for (int v = g.tid; v < n; v += g.n) {
            const unsigned k = keys[v];
            if (k == kHitKey) continue;
            if (shift + 8 < 32 && (k >> (shift + 8)) != prefix) continue;
            atomicAdd(&hist[(k >> shift) & 255u], 1);
        }
        g.sync();
        if (g.tid < 32) {
            const int lane = g.tid;
            int c[8];
            int sum = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                c[k] = hist[lane * 8 + k];
                sum += c[k];
            }
            const int inc = warp_inclusive_scan(sum);
            const int exc = inc - sum;
            if (exc < need && need <= inc) {
                int run = exc;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    if (run < need && need <= run + c[k]) {
                        sh[0] = lane * 8 + k;
                        sh[1] = need - run;
                    }
                    run += c[k];
                }
            }
        }
        g.sync();
        prefix = (prefix << 8) | (unsigned)sh[0];
        need = sh[1];
        g.sync();
    }
    *need_out = need;
    return prefix;
}

// Commit of batch row b (request q, epoch E, U unique misses) by group g
// (section 实现拆解 item 1 of the multi-step swap report; overflow admission
// prefers the latest step: section 风险与影响):
//   - `hits` has a bit for every hot slot the call referenced: those slots
//     take epoch E (in the same pass that builds the keys), cap = H - #hits
//     and m = min(U, cap);
//   - victims: the m non-hit slots with the smallest (epoch, slot); a radix
//     select over epoch + 1 finds the threshold epoch and how many slots at
//     the threshold to take (the lowest ones);
//   - admitted misses: all if U <= cap, otherwise the m best by (last step
//     descending, ordinal ascending);
//   - the i-th admitted miss (ascending ordinal) takes the i-th victim
//     (ascending slot): its old token leaves the index, phys[v] and
//     phys[H + j] swap (the copied row becomes the hot row, no second copy),
//     the new token enters the index and the slot takes epoch E.
// `keys` is H + C words of shared memory: the keys, then the victims.
__device__ void commit_request(const SwapArgs& a, const Group& g, int b, int q, int U, int E,
                               const unsigned* hits, unsigned* keys) {
    __shared__ int s_tmp[33];
    __shared__ int s_hist[256];
    __shared__ int s_sel[2];
    __shared__ int s_misc[8];

    const Dims& d = a.d;
    const int tid = g.tid, BD = g.n;
    const int H = d.H;
    int32_t* ctrl = a.lv.ctrl + (long long)q * kCtrlWords;
    int32_t* ep = a.lv.ep + (long long)q * H;
    int32_t* tok = a.lv.tok + (long long)q * H;
    int32_t* phys = a.lv.phys + (long long)q * (H + d.C);
    long long* bank = a.lv.bank + (long long)q * d.hash_size;
    const unsigned hmask = (unsigned)d.hash_size - 1u;
    const long long wbase = (long long)b * d.C;
    int* vict = reinterpret_cast<int*>(keys + H);  // victims in ascending slot order
    int32_t* adm = a.ws.adm + wbase;

    // The request's use counters, read now so that their load is done by
    // the time the commit updates them (nothing else writes them while the
    // request is locked).
    int used0 = 0, resident0 = 0;
    if (tid == 0) {
        used0 = ctrl[CTRL_USED];
        resident0 = ctrl[CTRL_RESIDENT];
    }
    // Keys for victim selection: epoch + 1 (0 = never used), or kHitKey for
    // a slot the call referenced, which takes epoch E in the same pass.
    // Each thread loads kKeyBatch epochs before it stores any, so the loads
    // are in flight together.
    int nhit = 0;
    for (int v0 = tid; v0 < H; v0 += kKeyBatch * BD) {
        int e[kKeyBatch];
#pragma unroll
        for (int u = 0; u < kKeyBatch; ++u) {
            const int v = v0 + u * BD;
            e[u] = v < H ? ep[v] : 0;
        }
#pragma unroll
        for (int u = 0; u < kKeyBatch; ++u) {
            const int v = v0 + u * BD;
            if (v < H) {
                const bool hit = (hits[v >> 5] >> (v & 31)) & 1u;
                keys[v] = hit ? kHitKey : (unsigned)(e[u] + 1);
                if (hit) ep[v] = E;
                nhit += hit;
            }
        }
    }
    nhit = group_sum(g, nhit, s_tmp);  // includes the barrier that publishes keys
    const int cap = H - nhit;
    const int m = U < cap ? U : cap;

    int evicted = 0;
    if (m > 0) {
        // ---- victims: m smallest (key, slot) among non-hit slots ------------
        const int bits = 32 - __clz(E);  // keys lie in [0, E]
        int need = m;
        unsigned thr = 0u;
        if (bits > 0) thr = radix_select(g, keys, H, m, bits, s_hist, s_sel, &need);
        // Each warp owns a contiguous chunk of slots, read lane by lane, so
        // ballots keep ascending slot order without shared-memory conflicts.
        // One pass counts each chunk's keys below and at the threshold, one
        // scan of both counts (packed: each is at most H <= 32768, and fewer
        // than m keys lie below the threshold) places every chunk, and a
        // second pass writes the victims: every key below the threshold,
        // then the lowest `need` slots at it.
        const int lane = tid & 31, warp = tid >> 5, nw = BD >> 5;
        const int chunk = ((H + nw - 1) / nw + 31) & ~31;
        const int w0 = warp * chunk, w1 = min(H, w0 + chunk);
        int lt = 0, eq = 0;
        for (int v0 = w0; v0 < w1; v0 += 32) {
            const int v = v0 + lane;
            const unsigned k = v < w1 ? keys[v] : kHitKey;
            lt += __popc(__ballot_sync(0xffffffffu, k < thr));
            eq += __popc(__ballot_sync(0xffffffffu, k == thr));
        }
        int packed_total;
        const int packed_before =
            group_exclusive_scan(g, lane == 0 ? (lt << 16) | eq : 0, s_tmp, &packed_total);
        const int pw = __shfl_sync(0xffffffffu, packed_before, 0);
        {
            int er = pw & 0xffff;                        // keys at the threshold before the chunk
            int vpos = (pw >> 16) + (er < need ? er : need);  // victims before the chunk
            for (int v0 = w0; v0 < w1; v0 += 32) {
                const int v = v0 + lane;
                const unsigned k = v < w1 ? keys[v] : kHitKey;
                const unsigned em = __ballot_sync(0xffffffffu, k == thr);
                const bool take = k < thr || (k == thr && er + __popc(em & lanemask_lt()) < need);
                const unsigned tm = __ballot_sync(0xffffffffu, take);
                if (take) vict[vpos + __popc(tm & lanemask_lt())] = v;
                vpos += __popc(tm);
                er += __popc(em);
            }
        }
        // ---- admitted misses ---------------------------------------------------
        if (U > cap) {
            const int* last = a.ws.miss_last + wbase;
            if (tid < 8) s_misc[tid] = 0;
            g.sync();
            for (int x0 = tid & ~31; x0 < U; x0 += BD) {  // per-step counts, one add per warp
                const int j = x0 + lane;
                const int l = j < U ? last[j] : -1;
                for (int st = 0; st < a.S; ++st) {
                    const int c = __popc(__ballot_sync(0xffffffffu, l == st));
                    if (lane == 0 && c) atomicAdd(&s_misc[st], c);
                }
            }
            g.sync();
            // threshold step: walk from the latest step down
            int s_thr = 0, need_s = m, acc = 0;
            for (int s = a.S - 1; s >= 0; --s) {
                if (acc + s_misc[s] >= m) {
                    s_thr = s;
                    need_s = m - acc;
                    break;
                }
                acc += s_misc[s];
            }
            const int cj = ((U + nw - 1) / nw + 31) & ~31;
            const int j0 = warp * cj, j1 = min(U, j0 + cj);
            int eqs = 0;
            for (int x0 = j0; x0 < j1; x0 += 32) {
                const int j = x0 + lane;
                eqs += __popc(__ballot_sync(0xffffffffu, j < j1 && last[j] == s_thr));
            }
            int eqs_total;
            const int es_before = group_exclusive_scan(g, lane == 0 ? eqs : 0, s_tmp, &eqs_total);
            const int es_w = __shfl_sync(0xffffffffu, es_before, 0);
            int na = 0;
            {
                int er = es_w;
                for (int x0 = j0; x0 < j1; x0 += 32) {
                    const int j = x0 + lane;
                    const int l = j < j1 ? last[j] : -1;
                    const unsigned em = __ballot_sync(0xffffffffu, l == s_thr);
                    const bool take =
                        l > s_thr || (l == s_thr && er + __popc(em & lanemask_lt()) < need_s);
                    na += __popc(__ballot_sync(0xffffffffu, take));
                    er += __popc(em);
                }
            }
            int na_total;
            const int a_before = group_exclusive_scan(g, lane == 0 ? na : 0, s_tmp, &na_total);
            {
                int er = es_w;
                int apos = __shfl_sync(0xffffffffu, a_before, 0);
                for (int x0 = j0; x0 < j1; x0 += 32) {
                    const int j = x0 + lane;
                    const int l = j < j1 ? last[j] : -1;
                    const unsigned em = __ballot_sync(0xffffffffu, l == s_thr);
                    const bool take =
                        l > s_thr || (l == s_thr && er + __popc(em & lanemask_lt()) < need_s);
                    const unsigned tm = __ballot_sync(0xffffffffu, take);
                    if (take) adm[apos + __popc(tm & lanemask_lt())] = j;
                    apos += __popc(tm);
                    er += __popc(em);
                }
            }
        }
        g.sync();
        // ---- evict, rotate and admit ------------------------------------------
        // A pair's four loads are independent.  Deletions and insertions may
        // interleave: a deletion only rewrites an entry that holds its own
        // (live) key and an insertion only claims empty or deleted entries,
        // so an insertion that probes past a live entry being deleted just
        // lands further along its chain.
        int fresh = 0;
        const int32_t* mtok = a.ws.miss_tok + wbase;
        for (int i = tid; i < m; i += BD) {
            const int v = vict[i];
            const int j = (U > cap) ? adm[i] : i;
            const int old = tok[v];
            const int pv = phys[v];
            const int ps = phys[H + j];
            const int t = mtok[j];
            phys[v] = ps;
            phys[H + j] = pv;
            tok[v] = t;
            ep[v] = E;
            if (d.dense) {  // dense index: one store each (old != t: resident vs not)
                int16_t* map = a.lv.map + (long long)q * d.L;
                if (old >= 0) {
                    map[old] = -1;
                    ++evicted;
                }
                map[t] = (int16_t)v;
                continue;
            }
            if (old >= 0) {
                bank_delete(bank, d.hash_shift, hmask, old, a.ws.status);
                ++evicted;
            }
            fresh += bank_insert(bank, d.hash_shift, hmask, t, v, a.ws.status);
        }
        {  // one scan of both counts (each at most m <= C <= HS_MAX_ENTRIES = 8192)
            const int both = group_sum(g, (fresh << 16) | evicted, s_tmp);
            evicted = both & 0xffff;
            fresh = both >> 16;
        }
        if (tid == 0) {
            s_misc[0] = used0 + fresh;
            s_misc[1] = resident0 + m - evicted;
        }
        g.sync();
        // ---- rebuild the bank once deleted entries pile up ---------------------
        if (!d.dense && s_misc[0] > (d.hash_size / 4) * 3) {
            for (int p = tid; p < d.hash_size; p += BD) bank[p] = kEmpty;
            g.sync();
            for (int v = tid; v < H; v += BD) {
                const int t = tok[v];
                if (t >= 0) bank_insert(bank, d.hash_shift, hmask, t, v, a.ws.status);
            }
            if (tid == 0) {
                s_misc[0] = s_misc[1];
                ctrl[CTRL_REBUILDS] += 1;
            }
        }
        g.sync();
        if (tid == 0) {
            ctrl[CTRL_USED] = s_misc[0];
            ctrl[CTRL_RESIDENT] = s_misc[1];
        }
    }
    if (tid == 0) {
        ctrl[CTRL_EPOCH] = E + 1;
        ctrl[CTRL_LOCK] = 0;
        if (a.stats) {
            int32_t* st = a.stats + (long long)b * HS_NUM_STATS;
            st[HS_STAT_HIT_SLOTS] = nhit;
            st[HS_STAT_ADMITTED] = m;
            st[HS_STAT_EVICTED] = evicted;
            st[HS_STAT_OVERFLOW] = U - m;
        }
        unsigned long long* tot = a.lv.totals;  // the layer's running sums
        atomicAdd(tot + HS_STAT_HIT_SLOTS, (unsigned long long)nhit);
        atomicAdd(tot + HS_STAT_ADMITTED, (unsigned long long)m);
        atomicAdd(tot + HS_STAT_EVICTED, (unsigned long long)evicted);
        atomicAdd(tot + HS_STAT_OVERFLOW, (unsigned long long)(U - m));
    }
}

// ---- copy (miss rows of one request) -----------------------------------------

// Copies the U miss rows of one request (W bytes each) from its host pool
// rows to their device rows, one warp at a time: a warp takes kWarpPieces
// consecutive 16-byte pieces of the flattened (miss, piece) space, issues
// all its loads, then its stores, and takes more until the pieces run out.
// The first `nfixed` chunks go to the warps that start copying at once, by
// their index `fixed` (-1 for a warp that starts later), so that their first
// loads wait for no atomic; every other chunk is claimed from `claim`.
// `mtok` and `mdst` were written earlier in this kernel, so they are read
// with plain (coherent) loads.
__device__ void copy_request(const uint8_t* pool_q, uint8_t* kv, const int32_t* mtok,
                             const int32_t* mdst, int U, int W, unsigned* claim, int fixed,
                             int nfixed) {
    const int lane = threadIdx.x & 31;
    const unsigned nv = (unsigned)W >> 4;  // 16-byte pieces per row
    const unsigned total = (unsigned)U * nv;
    for (;;) {
        unsigned start;
        if (fixed >= 0) {
            start = (unsigned)fixed * kWarpPieces;
            fixed = -1;
        } else {
            start = 0;
            if (lane == 0) start = atomicAdd(claim, (unsigned)kWarpPieces);
            start = __shfl_sync(0xffffffffu, start, 0) + (unsigned)nfixed * kWarpPieces;
        }
        if (start >= total) break;
        uint4 v[kCopyUnroll];
        long long dst[kCopyUnroll];  // destination byte offset of each piece, -1 if none
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const unsigned p = start + (unsigned)(u * 32 + lane);
            dst[u] = -1;
            if (p < total) {
                const unsigned row = p / nv;
                const unsigned piece = p - row * nv;
                dst[u] = (long long)mdst[row] * W + ((long long)piece << 4);
                v[u] = ld_stream_v4(pool_q + (long long)mtok[row] * W + ((long long)piece << 4));
            }
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u)
            if (dst[u] >= 0) st_v4(kv + dst[u], v[u]);
    }
}

// ---- the kernel ----------------------------------------------------------------

template <int RMAX, bool BY_POSITION>
__global__ void __launch_bounds__(1024, 1) swapin_kernel(const SwapArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_ok, s_epoch, s_done;
    __shared__ int s_tot[kMaxCluster];     // first occurrences of each rank
    __shared__ int s_cnt[kMaxCluster][4];  // leader: each rank's hit / invalid / miss / extra entries
    __shared__ int s_wcnt[32][4];          // the same counts per warp of this CTA
    // Hot slots referenced by this CTA's entries, one bit a slot; the
    // leader's copy collects every CTA's bits for the commit.
    __shared__ unsigned s_hits[HS_MAX_HOT_BUFFER / 32];
    cg::cluster_group cluster = cg::this_cluster();
    const int P = (int)cluster.num_blocks();
    const int c = (int)cluster.block_rank();
    const int plog = __ffs(P) - 1;

    const Dims& d = a.d;
    const int b = blockIdx.x >> plog;  // clusters are P consecutive CTAs
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int BD = blockDim.x, nwarps = BD >> 5;
    const int N = a.S * d.K;
    const int per = (N + P - 1) / P;
    const int lo = c * per, hi = min(N, lo + per);
    unsigned long long* tl =
        a.timeline ? a.timeline + ((long long)b * kTimelineCtas + c) * kTimelineWords : nullptr;
    if (tl && tid == 0) {
        tl[TL_START] = global_timer();
        tl[TL_CLUSTER_SIZE] = (unsigned long long)P;
    }

    // This CTA's share of the de-duplication table, then the flag words.
    // Indexed by position, an entry is the smallest entry key of the token
    // (int) and, when the call may overflow, the OR of its step bits next to
    // it (one 8-byte word, read by one load); hashed, the table keeps the
    // tokens, the smallest keys and 8 step bits an entry apart.
    // Only overflow admission reads a miss's last step, and a call with
    // S * K <= H cannot overflow: its distinct tokens, hits and misses
    // together, are at most S * K, so U <= H - #hit slots.
    const int TS = a.dedup_entries;
    const bool pairs = BY_POSITION && a.step_bits;
    int* first = reinterpret_cast<int*>(smem);
    unsigned* smask = reinterpret_cast<unsigned*>(first + TS);  // hashed table only
    int* keys = reinterpret_cast<int*>(smask + (TS >> 2));      // hashed table only
    const int table_bytes = BY_POSITION ? (pairs ? 8 : 4) * TS : (9 * TS + 15) & ~15;
    // Bitmap words of every rank of the cluster (each CTA sends its own to
    // all): fw[c' * NW + w], word w = r * nwarps + warp of rank c''s
    // entries, (running count << 32) | first-occurrence flags.
    const int NW = RMAX * nwarps;
    unsigned long long* fw = reinterpret_cast<unsigned long long*>(smem + table_bytes);

    // ---- 0. loads first (request slot, length, this CTA's entries), then
    // the table clear, which depends on none of them
    const int q = __ldg(a.rpi + b);
    const int sl = __ldg(a.seq_lens + b);
    const int32_t* topk_b = a.topk + (long long)b * N;
    int t[RMAX], code[RMAX], aux[RMAX], hrow[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
        const int i = lo + r * BD + tid;
        t[r] = (i < hi) ? __ldg(topk_b + i) : -1;
    }
    {
        int4* f4 = reinterpret_cast<int4*>(first);
        if (pairs) {
            for (int x = tid; x < (TS >> 1); x += BD) f4[x] = make_int4(kNoFirst, 0, kNoFirst, 0);
        } else {
            for (int x = tid; x < (TS >> 2); x += BD)
                f4[x] = make_int4(kNoFirst, kNoFirst, kNoFirst, kNoFirst);
        }
        if (!BY_POSITION) {
            int4* m4 = reinterpret_cast<int4*>(smask);
            for (int x = tid; x < (TS >> 4); x += BD) m4[x] = make_int4(0, 0, 0, 0);
            int4* k4 = reinterpret_cast<int4*>(keys);
            for (int x = tid; x < (TS >> 2); x += BD) k4[x] = make_int4(-1, -1, -1, -1);
        }
    }
    // The batch row's copy claim counter (16-byte pieces of its miss rows
    // handed out so far), zeroed by the leader after the first barrier (a
    // global store before that barrier's release would hold it back).
    unsigned* claim = reinterpret_cast<unsigned*>(a.ws.cnt + (long long)b * kCntWords + CNT_CLAIM);
    if (tid == 0) s_done = 0;
    for (int x = tid; x < ((d.H + 31) >> 5); x += BD) s_hits[x] = 0u;
    // First barrier, first half: this CTA runs and its table share is
    // empty.  The second half waits after the probe, which needs no other
    // CTA, so the barrier costs the probe nothing.
    cluster_arrive();
    const bool q_ok = q >= 0 && q < d.R;
    const int limit = sl < d.L ? sl : d.L;
    // first position of the extra page (past every valid token if none)
    const int xstart = (d.E > 0 && limit > 0) ? (limit - 1) / d.E * d.E : 0x7fffffff;
    unsigned xbits = 0u;  // bit r: entry r is on the extra page
    const long long base = (long long)q * (d.H + d.C);
    const int32_t* phys = a.lv.phys + base;
    // ---- 1. probe the token -> slot index: global memory only, so it runs
    // inside the first cluster barrier, beside the other CTAs' table clear
    int lock_old = 0, epoch0 = 0;
    {
        const long long* bank = a.lv.bank + (long long)(q_ok ? q : 0) * d.hash_size;
        const unsigned hmask = (unsigned)d.hash_size - 1u;
        const int16_t* map = a.lv.map + (long long)(q_ok ? q : 0) * d.L;
        long long e[RMAX];
        unsigned pos[RMAX];
        // The request lock and epoch, read by the leader's first thread
        // together with its index loads (the epoch only matters if the lock
        // is won, and nothing else changes it while the lock is held).
        if (c == 0 && tid == 0 && q_ok) {
            int32_t* ctrl_q = a.lv.ctrl + (long long)q * kCtrlWords;
            epoch0 = ctrl_q[CTRL_EPOCH];
            lock_old = atomicCAS(ctrl_q + CTRL_LOCK, 0, 1);
        }
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
            const bool in_range = q_ok && (lo + r * BD + tid < hi) && t[r] >= 0 && t[r] < limit;
            const bool extra = in_range && t[r] >= xstart;
            const bool valid = in_range && !extra;  // goes through the index
            if (extra) xbits |= 1u << r;
            code[r] = valid ? kMissPending : -1;
            e[r] = kEmpty;
            pos[r] = 0u;
            if (d.dense) {  // dense index: the slot is one load away, no chain
                if (valid) {
                    const int slot = map[t[r]];
                    if (slot >= 0 && slot < d.H) code[r] = slot;
                }
                continue;
            }
            pos[r] = hash_token(t[r], d.hash_shift);
            if (valid) e[r] = bank[pos[r]];
        }
        if (!d.dense) {
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
    }
    if (tl && tid == 0) stamp_after(tl, TL_PROBED, code);
    cluster_wait();  // every CTA of the cluster runs and its table share is empty
    if (tl && tid == 0) tl[TL_BARRIER0] = global_timer();
    if (c == 0 && tid == 0) *claim = 0u;  // read by the copy, after the last barrier

    if (c == 0 && tid == 0) {
        // The lock decision and the epoch, sent to every CTA.
        int ok = 1;
        if (!q_ok) {
            atomicOr(a.ws.status, HS_STATUS_BAD_REQUEST);
            ok = 0;
        } else if (lock_old != 0) {
            atomicOr(a.ws.status, HS_STATUS_DUPLICATE_REQUEST);
            ok = 0;
        }
        if (sl > d.L) atomicOr(a.ws.status, HS_STATUS_SEQ_LEN_CLAMPED);
        const int E = ok ? epoch0 : 0;
        for (int r = 0; r < P; ++r) {
            *cluster.map_shared_rank(&s_ok, r) = ok;
            *cluster.map_shared_rank(&s_epoch, r) = E;
        }
    }
    // ---- 2. de-duplicate misses into the cluster-wide table ------------------
    if (BY_POSITION) {
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
            if (code[r] != kMissPending) continue;
            const int home = t[r] & (P - 1);
            const int u = t[r] >> plog;
            int* f = cluster.map_shared_rank(first, home) + (pairs ? 2 * u : u);
            atomicMin(f, c * kKeyStride + r * BD + tid);
            if (pairs)  // else the last step is never read (recorded as step 0)
                atomicOr(reinterpret_cast<unsigned*>(f + 1),
                         1u << step_of(lo + r * BD + tid, d.K));
            code[r] = miss_code(u * kMaxCluster + home);
        }
    } else {
        const int ts_log = __ffs(TS) - 1;
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
            const bool miss = code[r] == kMissPending;
            // equal tokens of one warp insert once, by their lowest lane
            const unsigned grp = __match_any_sync(0xffffffffu, miss ? t[r] : (-2 - lane));
            if (miss) {
                const int leader = __ffs(grp) - 1;
                const unsigned steps =
                    __reduce_or_sync(grp, 1u << step_of(lo + r * BD + tid, d.K));
                int x = -1;
                if (lane == leader) {
                    const unsigned h = hash_token(t[r], a.dedup_shift);
                    const int home = (int)(h >> ts_log);
                    const int u = dedup_insert(cluster.map_shared_rank(keys, home),
                                               cluster.map_shared_rank(first, home),
                                               cluster.map_shared_rank(smask, home), TS,
                                               h & (unsigned)(TS - 1), t[r],
                                               c * kKeyStride + r * BD + tid, steps,
                                               a.ws.status);
                    x = u >= 0 ? u * kMaxCluster + home : -1;
                }
                x = __shfl_sync(grp, x, leader);
                code[r] = x >= 0 ? miss_code(x) : -1;
            }
        }
    }
    if (tl && tid == 0) tl[TL_INSERTED] = global_timer();
    // Second barrier, first half: this CTA's inserts (and, from the leader,
    // the lock decision) are sent.  Inside it, the work on hits, which needs
    // no other CTA: mark the slot for the commit and load its physical row
    // (used by the next step's locations).
    cluster_arrive();
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
        hrow[r] = 0;
        if (code[r] >= 0) {
            atomicOr(&s_hits[code[r] >> 5], 1u << (code[r] & 31));
            hrow[r] = phys[code[r]];
        }
    }
    if (q_ok) {
        // Warm L2 for later steps: the scratch positions (miss locations,
        // step 4) and the epochs (the commit).
        l2_prefetch(phys + d.H, (size_t)d.C * 4, c * BD + tid, P * BD);
        if (c == 0) l2_prefetch(a.lv.ep + (long long)q * d.H, (size_t)d.H * 4, tid, BD);
    }
    cluster_wait();  // the table is complete, s_ok / s_epoch have arrived
    if (tl && tid == 0) tl[TL_BARRIER_A] = global_timer();

    int32_t* locs_b = a.locs + (long long)b * N;
    if (!s_ok) {
        // Rejected batch row: no location, no state change, nothing to copy.
        for (int i = lo + tid; i < hi; i += BD) locs_b[i] = -1;
        if (c == 0) {
            if (a.stats && tid < HS_NUM_STATS) a.stats[(long long)b * HS_NUM_STATS + tid] = 0;
            if (a.plan_count && tid == 0) a.plan_count[b] = 0;
        }
        return;
    }
    const int E = s_epoch;

    // ---- 3. first occurrences: flags, running counts, totals -----------------
    {
        unsigned mw[RMAX];
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {  // all remote loads in flight together
            mw[r] = 0u;
            if (code[r] <= -3) {
                const int x = miss_value(code[r]);
                const int home = x & (kMaxCluster - 1), u = x >> 3;
                if (!BY_POSITION) {
                    aux[r] = *(cluster.map_shared_rank(first, home) + u);
                    mw[r] = *(cluster.map_shared_rank(smask, home) + (u >> 2));
                    mw[r] = (mw[r] >> ((u & 3) * 8)) & 0xffu;
                } else if (pairs) {  // first index and step bits in one load
                    const unsigned long long v = *reinterpret_cast<const unsigned long long*>(
                        cluster.map_shared_rank(first, home) + 2 * u);
                    aux[r] = (int)(unsigned)v;
                    mw[r] = (unsigned)(v >> 32);
                } else {
                    aux[r] = *(cluster.map_shared_rank(first, home) + u);
                    mw[r] = 1u;
                }
            }
        }
        int n_hit = 0, n_inv = 0, n_miss = 0, n_ext = 0;
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
            const int i = lo + r * BD + tid;
            const bool f = code[r] <= -3 && aux[r] == c * kKeyStride + r * BD + tid;
            if (i < hi) {  // the counters of this CTA's entries
                if ((xbits >> r) & 1u) ++n_ext;
                else if (code[r] >= 0) ++n_hit;
                else if (code[r] == -1) ++n_inv;
                else ++n_miss;
            }
            if (code[r] <= -3)  // now: the token's first index and last step
                code[r] = miss_code(aux[r] | ((31 - __clz((int)mw[r])) << 16));
            const unsigned bal = __ballot_sync(0xffffffffu, f);
            if (lane == 0) fw[c * NW + r * nwarps + warp] = bal;
        }
        n_hit = __reduce_add_sync(0xffffffffu, n_hit);
        n_inv = __reduce_add_sync(0xffffffffu, n_inv);
        n_miss = __reduce_add_sync(0xffffffffu, n_miss);
        n_ext = __reduce_add_sync(0xffffffffu, n_ext);
        if (lane == 0) {
            s_wcnt[warp][0] = n_hit;
            s_wcnt[warp][1] = n_inv;
            s_wcnt[warp][2] = n_miss;
            s_wcnt[warp][3] = n_ext;
        }
    }
    if (tl && tid == 0) stamp_after(tl, TL_FLAGGED, code);
    __syncthreads();
    // Warp 0 sends the flag words and the total, warp 1 the entry counters,
    // the other warps the hit bits (a CTA has at least 8 warps).
    if (c != 0 && warp >= 2) {  // this CTA's hit slots, into the leader's bitmap
        unsigned* lead = cluster.map_shared_rank(s_hits, 0);
        for (int x = tid - 64; x < ((d.H + 31) >> 5); x += BD - 64)
            if (s_hits[x]) atomicOr(lead + x, s_hits[x]);
    }
    if (warp == 1) {  // this CTA's entry counters, to the leader
        int n[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            n[k] = __reduce_add_sync(0xffffffffu, lane < nwarps ? s_wcnt[lane][k] : 0);
        if (lane < 4)
            *cluster.map_shared_rank(&s_cnt[c][lane], 0) =
                lane == 0 ? n[0] : lane == 1 ? n[1] : lane == 2 ? n[2] : n[3];
    }
    if (warp == 0) {
        // Running counts over this CTA's RMAX * nwarps words in (r, warp)
        // order; each finished word goes to every CTA of the cluster, so
        // that step 4 reads any rank's words from its own shared memory.
        const int per_lane = (NW + 31) >> 5;
        unsigned bw[RMAX];
        int sum = 0;
#pragma unroll
        for (int k = 0; k < RMAX; ++k) {
            const int idx = lane * per_lane + k;
            bw[k] = (k < per_lane && idx < NW) ? (unsigned)fw[c * NW + idx] : 0u;
            sum += __popc(bw[k]);
        }
        const int inc = warp_inclusive_scan(sum);
        int run = inc - sum;
#pragma unroll
        for (int k = 0; k < RMAX; ++k) {
            const int idx = lane * per_lane + k;
            if (k < per_lane && idx < NW) {
                fw[c * NW + idx] = ((unsigned long long)(unsigned)run << 32) | bw[k];
                run += __popc(bw[k]);
            }
        }
        __syncwarp();
        for (int rk = 1; rk < P; ++rk) {
            unsigned long long* dst = cluster.map_shared_rank(fw + c * NW, (c + rk) & (P - 1));
            for (int idx = lane; idx < NW; idx += 32) dst[idx] = fw[c * NW + idx];
        }
        const int total = __shfl_sync(0xffffffffu, inc, 31);
        if (lane < P) *cluster.map_shared_rank(&s_tot[c], lane) = total;
    }
    cluster.sync();  // every CTA's words, totals and counters are in place
    if (tl && tid == 0) tl[TL_BARRIER_B] = global_timer();

    // ---- 4. ordinals, miss lists, locations ---------------------------------
    // Lane k < P: the first occurrences of the ranks below k (ranks P .. 7
    // add none); U, all of them.
    const int tot_k = lane < P ? s_tot[lane] : 0;
    int incl = tot_k;
#pragma unroll
    for (int o = 1; o < kMaxCluster; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const int U = __shfl_sync(0xffffffffu, incl, kMaxCluster - 1);
    const int excl = incl - tot_k;
    const long long wbase = (long long)b * d.C;
    {
        int j[RMAX];
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {  // ordinal of the token's first occurrence
            // Rank c1 and local index l1 of the first occurrence, from its
            // key; computed for every entry (the shuffle needs all lanes)
            // and used for misses only.
            const bool m = code[r] <= -3;
            const int key = miss_value(code[r]) & 0xffff;
            const int c1 = key >> kKeyShift, l1 = key & (kKeyStride - 1);
            const int off = __shfl_sync(0xffffffffu, excl, c1 & (kMaxCluster - 1));
            const unsigned long long wd = m ? fw[c1 * NW + (l1 >> 5)] : 0ull;
            j[r] = m ? off + (int)(wd >> 32) + __popc((unsigned)wd & ((1u << (l1 & 31)) - 1u)) : 0;
        }
        // Every position load in flight before any store below: a store
        // might alias phys as far as the compiler knows, so loads mixed
        // with the stores would each wait for the previous round trip.
        int row[RMAX];
#pragma unroll
        for (int r = 0; r < RMAX; ++r)
            row[r] = code[r] >= 0 ? hrow[r] : (code[r] <= -3 ? phys[d.H + j[r]] : 0);
        if (tl && tid == 0) stamp_after(tl, TL_ROWS, row);
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {  // first occurrences: list the miss
            if (code[r] <= -3 &&
                (miss_value(code[r]) & 0xffff) == c * kKeyStride + r * BD + tid) {
                const int loc = (int)(base + row[r]);
                a.ws.miss_tok[wbase + j[r]] = t[r];
                a.ws.miss_last[wbase + j[r]] = miss_value(code[r]) >> 16;
                a.ws.miss_dst[wbase + j[r]] = loc;
                if (a.plan_src) {
                    a.plan_src[wbase + j[r]] = (long long)q * d.L + t[r];
                    a.plan_dst[wbase + j[r]] = loc;
                }
            }
        }
        // Last barrier, first half: the miss lists are written.  Inside it,
        // the locations, which no CTA reads.
        cluster_arrive();
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
            const int i = lo + r * BD + tid;
            if (i >= hi) continue;
            int loc = code[r] == -1 ? -1 : (int)(base + row[r]);
            if ((xbits >> r) & 1u)
                loc = (int)((long long)d.R * (d.H + d.C) + (long long)q * d.E + t[r] % d.E);
            locs_b[i] = loc;
        }
    }
    // Miss lists visible to the whole cluster; no shared memory of another
    // CTA is touched after this point.
    cluster_wait();
    if (tl && tid == 0) tl[TL_BARRIER_C] = global_timer();
    if (c == 0 && tid == 0) {
        int n_hit = 0, n_inv = 0, n_miss = 0, n_ext = 0;
        for (int k = 0; k < P; ++k) {
            n_hit += s_cnt[k][0];
            n_inv += s_cnt[k][1];
            n_miss += s_cnt[k][2];
            n_ext += s_cnt[k][3];
        }
        if (a.stats) {
            int32_t* st = a.stats + (long long)b * HS_NUM_STATS;
            st[HS_STAT_HITS] = n_hit;
            st[HS_STAT_DUP_MISSES] = n_miss - U;
            st[HS_STAT_UNIQUE_MISSES] = U;
            st[HS_STAT_INVALID] = n_inv;
            st[HS_STAT_EXTRA] = n_ext;
        }
        unsigned long long* tot = a.lv.totals;  // the layer's running sums
        atomicAdd(tot + HS_STAT_HITS, (unsigned long long)n_hit);
        atomicAdd(tot + HS_STAT_DUP_MISSES, (unsigned long long)(n_miss - U));
        atomicAdd(tot + HS_STAT_UNIQUE_MISSES, (unsigned long long)U);
        atomicAdd(tot + HS_STAT_INVALID, (unsigned long long)n_inv);
        atomicAdd(tot + HS_STAT_EXTRA, (unsigned long long)n_ext);
        if (a.plan_count) a.plan_count[b] = U;
    }

    // ---- 5. commit on the leader, copy everywhere else ----------------------
    // With other CTAs in the cluster to copy, the whole leader commits (and
    // copies once it is done); a lone CTA splits its warps between the two.
    const int commit_warps = P > 1 ? nwarps : (nwarps < kCommitWarps ? nwarps : kCommitWarps);
    if (c == 0 && warp < commit_warps) {
        commit_request(a, Group{tid, commit_warps * 32}, b, q, U, E, s_hits,
                       reinterpret_cast<unsigned*>(smem));
        if (tl && tid == 0) tl[TL_COMMITTED] = global_timer();
    }
    if (!a.defer_copy && U > 0) {
        // Warps that copy from the start: every warp of the other CTAs (of
        // all but the commit warps in a cluster of one); the leader's commit
        // warps join when done.
        const int nfixed = P > 1 ? (P - 1) * nwarps : nwarps - commit_warps;
        const int fixed = P > 1 ? (c > 0 ? (c - 1) * nwarps + warp : -1)
                                : (warp >= commit_warps ? warp - commit_warps : -1);
        copy_request(a.lv.host_pool + (long long)q * d.L * d.W, a.lv.device_kv,
                     a.ws.miss_tok + wbase, a.ws.miss_dst + wbase, U, d.W, claim, fixed,
                     nfixed);
    }
    if (tl && lane == 0 && atomicAdd(&s_done, 1) == nwarps - 1) tl[TL_COPIED] = global_timer();
}

template <int RMAX, bool BY_POSITION>
SmemOptIn* smem_opt_in() {
    static SmemOptIn opt_in;
    return &opt_in;
}

// The launch configuration of a shape (attrs: one cluster-dimension attribute).
inline cudaLaunchConfig_t launch_config(const SwapinShape& sh, int batch, cudaStream_t s,
                                        cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(batch * sh.P);
    cfg.blockDim = dim3(sh.block);
    cfg.dynamicSmemBytes = sh.smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = sh.P;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <int RMAX, bool BY_POSITION>
cudaError_t launch_one(const SwapArgs& a, const SwapinShape& sh, cudaStream_t s) {
    cudaError_t e = ensure_smem(swapin_kernel<RMAX, BY_POSITION>, sh.smem,
                                smem_opt_in<RMAX, BY_POSITION>());
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = launch_config(sh, a.B, s, attr);
    return cudaLaunchKernelEx(&cfg, swapin_kernel<RMAX, BY_POSITION>, a);
}

// How many clusters of this shape the current device runs at once (0 if
// the query fails).
template <int RMAX, bool BY_POSITION>
int max_clusters_one(const SwapinShape& sh) {
    if (ensure_smem(swapin_kernel<RMAX, BY_POSITION>, sh.smem, smem_opt_in<RMAX, BY_POSITION>()) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = launch_config(sh, 1, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, swapin_kernel<RMAX, BY_POSITION>, &cfg) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// max_clusters_one, remembered per device and shape (a host query per
// distinct shape, not per call).
int max_clusters(const SwapinShape& sh) {
    struct Entry {
        int device, rmax, by_position, P, block;
        size_t smem;
        int clusters;
    };
    static std::mutex m;
    static Entry cache[128];
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    {
        std::lock_guard<std::mutex> lock(m);
        for (int i = 0; i < used; ++i) {
            const Entry& e = cache[i];
            if (e.device == dev && e.rmax == sh.rmax && e.by_position == (int)sh.by_position &&
                e.P == sh.P && e.block == sh.block && e.smem == sh.smem)
                return e.clusters;
        }
    }
    int n = 0;
    if (sh.by_position)
        n = sh.rmax == 1 ? max_clusters_one<1, true>(sh)
                         : (sh.rmax == 2 ? max_clusters_one<2, true>(sh) : max_clusters_one<4, true>(sh));
    else
        n = sh.rmax == 1 ? max_clusters_one<1, false>(sh)
                         : (sh.rmax == 2 ? max_clusters_one<2, false>(sh) : max_clusters_one<4, false>(sh));
    std::lock_guard<std::mutex> lock(m);
    if (n > 0 && used < 128)
        cache[used++] = Entry{dev, sh.rmax, (int)sh.by_position, sh.P, sh.block, sh.smem, n};
    return n;
}

}  // namespace

// Whether a call must record each miss's last step: only overflow
// admission reads it, and a call of S * K <= H entries cannot overflow.
bool step_bits_needed(const Dims& d, int steps) {
    return steps > 1 && (long long)steps * d.K > d.H;
}

// Launch shape of a call with `batch` rows of `steps * K` entries:
//   - P, the CTAs per batch row: the largest power of two <= p_cap with
//     batch * P CTAs still within one wave of `sms` SMs and at least 256
//     entries per CTA, but never more than 4096 entries per CTA (4 a
//     thread); then raised (up to p_cap) until a position-indexed
//     de-duplication table over max_seq_len positions fits
//     kPositionTableBytes per CTA.  If it never fits, the table is hashed.
//     The launcher lowers p_cap while the device cannot hold the batch's
//     clusters at once.
//   - threads: 1024 for more than 1024 entries per CTA, else the entries
//     rounded up to whole warps, at least 256 (512 with H >= 2048, since
//     the leader CTA's threads also run the commit over the H slots).  More
//     threads than entries would not pay: with one 1024-thread CTA per SM,
//     clusters of 8 no longer all fit at once (16 of them in a 152-SM
//     GB300 ran in two waves).
//   - shared memory: the table share plus the flag words of every rank,
//     or the commit's H keys and up to C victims if larger.
SwapinShape swapin_shape(const Dims& d, int batch, int steps, int sms, int p_cap) {
    const int N = steps * d.K;
    int p = 1;
    while (p < p_cap && batch * (2 * p) <= sms && N / (2 * p) >= 256) p *= 2;
    while (p < kMaxCluster && (N + p - 1) / p > 4096) p *= 2;
    auto pos_entries = [&](int pp) { return ((d.L + pp - 1) / pp + 15) & ~15; };
    const int entry_bytes = step_bits_needed(d, steps) ? 8 : 4;  // first index (+ step bits)
    int pp = p;
    while (pp < p_cap && entry_bytes * pos_entries(pp) > kPositionTableBytes) pp *= 2;
    SwapinShape sh;
    sh.by_position = entry_bytes * pos_entries(pp) <= kPositionTableBytes;
    if (sh.by_position) p = pp;
    sh.P = p;
    if (sh.by_position) {
        sh.dedup_entries = pos_entries(p);
    } else {
        int t1 = 128;
        while (t1 < 2 * N) t1 <<= 1;
        sh.dedup_entries = t1 / p;
    }
    const int per = (N + p - 1) / p;
    const int min_block = d.H >= 2048 ? 512 : 256;
    if (per <= 1024) {
        sh.rmax = 1;
        const int w = ((per + 31) / 32) * 32;
        sh.block = w < min_block ? min_block : w;
    } else {
        sh.rmax = per <= 2048 ? 2 : 4;
        sh.block = 1024;
    }
    const size_t table = sh.by_position ? (size_t)entry_bytes * sh.dedup_entries
                                        : (size_t)((9 * sh.dedup_entries + 15) & ~15);
    const size_t words = (size_t)p * sh.rmax * (sh.block / 32) * 8;  // every rank's words
    const size_t commit = (size_t)(d.H + d.C) * 4;  // keys and victims
    sh.smem = table + words > commit ? table + words : commit;
    return sh;
}

cudaError_t launch_swapin(const SwapArgs& a, int sms, cudaStream_t s) {
    SwapinShape sh = swapin_shape(a.d, a.B, a.S, sms, kMaxCluster);
    // A shape counts CTAs against SMs, but whether clusters of P large CTAs
    // are co-resident depends on how the SMs group: while the batch would
    // need more than one wave of clusters, try half the cluster size.
    while (sh.P > 1) {
        const int fit = max_clusters(sh);
        if (fit <= 0 || a.B <= fit) break;
        const SwapinShape smaller = swapin_shape(a.d, a.B, a.S, sms, sh.P / 2);
        if (smaller.P >= sh.P) break;
        const int fit2 = max_clusters(smaller);
        if (fit2 <= 0 || (a.B + fit2 - 1) / fit2 >= (a.B + fit - 1) / fit) break;  // no fewer waves
        sh = smaller;
    }
    SwapArgs g = a;
    g.step_bits = step_bits_needed(a.d, a.S) ? 1 : 0;
    g.dedup_entries = sh.dedup_entries;
    g.dedup_shift = 32 - __builtin_ctz((unsigned)(sh.dedup_entries * sh.P));
    if (sh.by_position) {
        if (sh.rmax == 1) return launch_one<1, true>(g, sh, s);
        if (sh.rmax == 2) return launch_one<2, true>(g, sh, s);
        return launch_one<4, true>(g, sh, s);
    }
    if (sh.rmax == 1) return launch_one<1, false>(g, sh, s);
    if (sh.rmax == 2) return launch_one<2, false>(g, sh, s);
    return launch_one<4, false>(g, sh, s);
}

}  // namespace hs
