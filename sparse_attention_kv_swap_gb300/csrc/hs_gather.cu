// Gather kernel of the decode KV swap-in (sm_103a).
//
// One CTA per batch row b (request q = req_pool_indices[b]) resolves the
// row's S x K top-k entries as one working set (the multi-step swap report
// "[HiSparse] Support hisparse multi-step swap io kernel", section 实现拆解
// item 1: gather flattens [batch, steps, top_k], looks tokens up in the hot
// cache's token -> slot hash and de-duplicates misses across steps):
//   1. each thread loads up to RMAX entries and probes the request's hash
//      bank (linear probing, all first probes issued before any is resolved);
//      a hit stamps its slot with the call's epoch;
//   2. misses are de-duplicated: __match_any_sync merges equal tokens inside
//      a warp, then the group leader inserts the token into a shared-memory
//      table, keeping the smallest flat index and the set of steps it occurs in;
//   3. a block scan over "first occurrence" flags numbers the unique misses
//      j = 0, 1, ... in (step, k) order;
//   4. every entry gets its device row: q * (H + C) + phys[slot] for a hit,
//      q * (H + C) + phys[H + j] for miss j.  Unique misses are listed for the
//      commit (token, last step) and the copy (destination row).
// The row copy itself runs in the second kernel, spread over the whole GPU.
#include "hs_internal.cuh"

namespace hs {
namespace {

constexpr int kMissPending = -2;  // code of an entry that missed the hash bank
// Entry codes: >= 0 hit slot; -1 invalid; <= -3 miss at dedup position (-3 - p).
__device__ __forceinline__ int miss_code(int p) { return -3 - p; }
__device__ __forceinline__ int miss_pos(int code) { return -3 - code; }

// Inserts token t (flat index i, step-bit set `steps`) into the shared
// de-duplication table; returns its position.  The table has at least twice
// as many entries as the CTA has entries, so a free position always exists.
__device__ __forceinline__ int dedup_insert(int* keys, int* first, unsigned* smask, int size,
                                            int shift, int t, int i, unsigned steps,
                                            uint32_t* status) {
    const unsigned mask = (unsigned)size - 1u;
    unsigned p = hash_token(t, shift);
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
    const int T1 = a.dedup_size;
    int* keys = reinterpret_cast<int*>(smem);
    int* first = keys + T1;                                    // first index, later ordinal
    unsigned* smask = reinterpret_cast<unsigned*>(first + T1);  // 8 step bits per position
    int* wcount = reinterpret_cast<int*>(smask + (T1 >> 2));   // [RMAX][32] warp counts
    __shared__ int s_tmp[33];
    __shared__ int s_q, s_ok, s_epoch, s_limit, s_total;

    const Dims& d = a.d;
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int BD = blockDim.x, nwarps = BD >> 5;
    const int N = a.S * d.K;

    for (int i = tid; i < T1; i += BD) {
        keys[i] = -1;
        first[i] = 0x7fffffff;
    }
    for (int i = tid; i < (T1 >> 2); i += BD) smask[i] = 0u;
    if (tid == 0) {
        const int q = a.rpi[b];
        int ok = 1;
        if (q < 0 || q >= d.R) {
            atomicOr(a.ws.status, HS_STATUS_BAD_REQUEST);
            ok = 0;
        } else if (atomicCAS(&a.lv.ctrl[(long long)q * kCtrlWords + CTRL_LOCK], 0, 1) != 0) {
            atomicOr(a.ws.status, HS_STATUS_DUPLICATE_REQUEST);
            ok = 0;
        }
        const int sl = a.seq_lens[b];
        if (sl > d.L) atomicOr(a.ws.status, HS_STATUS_SEQ_LEN_CLAMPED);
        s_limit = sl < d.L ? sl : d.L;
        s_q = q;
        s_ok = ok;
        s_epoch = ok ? a.lv.ctrl[(long long)q * kCtrlWords + CTRL_EPOCH] : 0;
    }
    __syncthreads();

    int32_t* locs_b = a.locs + (long long)b * N;
    int32_t* cnt = a.ws.cnt + (long long)b * kCntWords;
    if (!s_ok) {
        // Rejected batch row: no location, no state change, nothing to copy.
        for (int i = tid; i < N; i += BD) locs_b[i] = -1;
        if (tid < kCntWords) cnt[tid] = (tid == CNT_SKIP) ? 1 : 0;
        if (a.stats && tid < HS_NUM_STATS) a.stats[(long long)b * HS_NUM_STATS + tid] = 0;
        if (a.plan_count && tid == 0) a.plan_count[b] = 0;
        pdl_trigger();
        return;
    }

    const int q = s_q, E = s_epoch, limit = s_limit;
    const long long base = (long long)q * (d.H + d.C);
    const long long* bank = a.lv.bank + (long long)q * d.hash_size;
    const int32_t* phys = a.lv.phys + base;
    int32_t* ep = a.lv.ep + (long long)q * d.H;
    const int32_t* topk_b = a.topk + (long long)b * N;
    const unsigned hmask = (unsigned)d.hash_size - 1u;

    // ---- 1. probe the hash bank -------------------------------------------
    int t[RMAX], code[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
        const int i = r * BD + tid;
        t[r] = (i < N) ? __ldg(topk_b + i) : -1;
    }
    {
        long long e[RMAX];
        unsigned pos[RMAX];
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
            const bool valid = (r * BD + tid < N) && t[r] >= 0 && t[r] < limit;
            code[r] = valid ? kMissPending : -1;
            pos[r] = hash_token(t[r], d.hash_shift);
            e[r] = valid ? bank[pos[r]] : kEmpty;
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
    // Hits: stamp the slot with this call's epoch and fetch its physical row.
    int hrow[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
        hrow[r] = 0;
        if (code[r] >= 0) {
            ep[code[r]] = E;
            hrow[r] = phys[code[r]];
        }
    }

    // ---- 2. de-duplicate misses -------------------------------------------
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
        const int i = r * BD + tid;
        const bool miss = code[r] == kMissPending;
        const unsigned grp = __match_any_sync(0xffffffffu, miss ? t[r] : (-2 - lane));
        if (miss) {
            const int leader = __ffs(grp) - 1;
            const unsigned steps = __reduce_or_sync(grp, 1u << (i / d.K));
            int p = -1;
            if (lane == leader)
                p = dedup_insert(keys, first, smask, T1, a.dedup_shift, t[r], i, steps,
                                 a.ws.status);
            p = __shfl_sync(grp, p, leader);
            code[r] = p >= 0 ? miss_code(p) : -1;
        }
    }
    __syncthreads();

    // ---- 3. number the unique misses in (step, k) order ---------------------
    unsigned firstbits = 0u;
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
        const int i = r * BD + tid;
        const bool f = code[r] <= -3 && first[miss_pos(code[r])] == i;
        const unsigned bal = __ballot_sync(0xffffffffu, f);
        if (lane == 0) wcount[r * nwarps + warp] = __popc(bal);
        if (f) firstbits |= 1u << r;
    }
    __syncthreads();
    if (warp == 0) {
        // exclusive scan of RMAX * nwarps warp counts in (r, warp) order
        const int n = RMAX * nwarps;
        const int per = (n + 31) >> 5;
        int loc[RMAX];
        int sum = 0;
#pragma unroll
        for (int k = 0; k < RMAX; ++k) {
            const int idx = lane * per + k;
            loc[k] = (k < per && idx < n) ? wcount[idx] : 0;
            sum += loc[k];
        }
        const int inc = warp_inclusive_scan(sum);
        int run = inc - sum;
#pragma unroll
        for (int k = 0; k < RMAX; ++k) {
            const int idx = lane * per + k;
            if (k < per && idx < n) {
                wcount[idx] = run;
                run += loc[k];
            }
        }
        if (lane == 31) s_total = inc;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
        const bool f = (firstbits >> r) & 1u;
        const unsigned bal = __ballot_sync(0xffffffffu, f);
        if (f) first[miss_pos(code[r])] = wcount[r * nwarps + warp] + __popc(bal & lanemask_lt());
    }
    __syncthreads();

    // ---- 4. locations, miss lists, counters --------------------------------
    const int U = s_total;
    const long long wbase = (long long)b * d.C;
    int n_hit = 0, n_inv = 0, n_miss = 0;
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
        const int i = r * BD + tid;
        if (i >= N) continue;
        int loc;
        if (code[r] >= 0) {
            loc = (int)(base + hrow[r]);
            ++n_hit;
        } else if (code[r] == -1) {
            loc = -1;
            ++n_inv;
        } else {
            const int p = miss_pos(code[r]);
            const int j = first[p];
            loc = (int)(base + phys[d.H + j]);
            ++n_miss;
            if ((firstbits >> r) & 1u) {
                const unsigned m8 = (smask[p >> 2] >> ((p & 3) * 8)) & 0xffu;
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
    n_hit = block_sum(n_hit, s_tmp);
    n_inv = block_sum(n_inv, s_tmp);
    n_miss = block_sum(n_miss, s_tmp);
    if (tid == 0) {
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
        }
        if (a.plan_count) a.plan_count[b] = U;
    }
    pdl_trigger();
}

template <int RMAX>
cudaError_t launch_rmax(const SwapArgs& a, int block, size_t smem, cudaStream_t s) {
    static int cached = 48 * 1024;
    cudaError_t e = ensure_smem(gather_kernel<RMAX>, smem, &cached);
    if (e != cudaSuccess) return e;
    gather_kernel<RMAX><<<a.B, block, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

size_t gather_smem_bytes(int entries, int* dedup_size) {
    int t1 = 64;
    while (t1 < 2 * entries) t1 <<= 1;
    if (dedup_size) *dedup_size = t1;
    // keys + first + step masks + warp counts (8 x 32)
    return (size_t)t1 * 4 * 2 + (size_t)t1 + 8 * 32 * 4;
}

cudaError_t launch_gather(const SwapArgs& a, cudaStream_t s) {
    const int N = a.S * a.d.K;
    int t1 = 0;
    const size_t smem = gather_smem_bytes(N, &t1);
    SwapArgs g = a;
    g.dedup_size = t1;
    g.dedup_shift = 32 - __builtin_ctz((unsigned)t1);
    if (N <= 1024) {
        const int block = ((N + 31) / 32) * 32 < 64 ? 64 : ((N + 31) / 32) * 32;
        return launch_rmax<1>(g, block, smem, s);
    }
    if (N <= 2048) return launch_rmax<2>(g, 1024, smem, s);
    if (N <= 4096) return launch_rmax<4>(g, 1024, smem, s);
    return launch_rmax<8>(g, 1024, smem, s);
}

}  // namespace hs
