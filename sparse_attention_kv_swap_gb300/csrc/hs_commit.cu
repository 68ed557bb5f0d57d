// Commit + copy kernel of the decode KV swap-in (sm_103a).
//
// Launched right behind the gather kernel with programmatic dependent
// launch; every CTA first waits for the gather grid's results.  The grid has
// two kinds of CTA that run side by side:
//
//  * CTAs 0..B-1 commit one request each (the multi-step swap report,
//    section 实现拆解 item 1: CLOCK update, rotation of scratch and hot
//    locations, token -> slot hash update, resolution of overflowing misses;
//    section 风险与影响: overflow admission prefers the latest step):
//      - hot slots referenced by the call already carry its epoch E (the
//        gather stamped them), so cap = H - #{ep == E} and m = min(U, cap);
//      - victims: the m non-hit slots with the smallest (epoch, slot); a
//        radix select over epoch + 1 finds the threshold epoch and how many
//        slots at the threshold to take (the lowest ones);
//      - admitted misses: all if U <= cap, otherwise the m best by (last step
//        descending, ordinal ascending);
//      - the i-th admitted miss (ascending ordinal) takes the i-th victim
//        (ascending slot): its old token leaves the token -> slot index
//        (hash bank or dense map), phys[v] and phys[H + j] swap (the copied
//        row becomes the hot row, no second copy), the new token enters the
//        index and the slot takes epoch E.
//  * the other CTAs copy every unique miss's KV row from the mapped pinned
//    host pool to the device row the gather returned for it: 16-byte
//    vectors, consecutive threads on consecutive 16-byte pieces of a row,
//    all of a thread's loads issued before its stores.
// The two never touch the same memory: the copy reads the miss lists and
// writes device KV rows, the commit rewrites only the policy state.
#include "hs_internal.cuh"

namespace hs {
namespace {

constexpr int kBlock = 512;
constexpr int kCopyUnroll = 6;
constexpr unsigned kHitKey = 0xffffffffu;  // radix key of a slot referenced by the call

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void* p, const uint4& v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Non-binding prefetch of [p, p + bytes) into L2, one 128-byte line per thread.
__device__ __forceinline__ void l2_prefetch(const void* p, size_t bytes) {
    const char* c = static_cast<const char*>(p);
    for (size_t off = (size_t)threadIdx.x * 128; off < bytes; off += (size_t)blockDim.x * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(c + off));
}

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
__device__ unsigned radix_select(const unsigned* keys, int n, int need, int bits, int* hist,
                                 int* sh, int* need_out) {
    unsigned prefix = 0u;
    int top = ((bits + 7) / 8) * 8;
    for (int shift = top - 8; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int v = threadIdx.x; v < n; v += blockDim.x) {
            const unsigned k = keys[v];
            if (k == kHitKey) continue;
            if (shift + 8 < 32 && (k >> (shift + 8)) != prefix) continue;
            atomicAdd(&hist[(k >> shift) & 255u], 1);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            int c[8];
            int sum = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                c[k] = hist[lane * 8 + k];
                sum += c[k];
            }
            const int inc = warp_inclusive_scan(sum);
            const int exc = inc - sum;
            const bool here = exc < need && need <= inc;
            if (here) {
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
        __syncthreads();
        prefix = (prefix << 8) | (unsigned)sh[0];
        need = sh[1];
        __syncthreads();
    }
    *need_out = need;
    return prefix;
}

__device__ void commit_request(const SwapArgs& a, int b, unsigned* keys) {
    __shared__ int s_tmp[33];
    __shared__ int s_hist[256];
    __shared__ int s_sel[2];
    __shared__ int s_misc[8];

    const Dims& d = a.d;
    const int32_t* cnt = a.ws.cnt + (long long)b * kCntWords;
    if (cnt[CNT_SKIP]) return;
    const int tid = threadIdx.x, BD = blockDim.x;
    const int q = cnt[CNT_Q];
    const int U = cnt[CNT_U];
    const int H = d.H;
    int32_t* ctrl = a.lv.ctrl + (long long)q * kCtrlWords;
    const int E = ctrl[CTRL_EPOCH];
    int32_t* ep = a.lv.ep + (long long)q * H;
    int32_t* tok = a.lv.tok + (long long)q * H;
    int32_t* phys = a.lv.phys + (long long)q * (H + d.C);
    long long* bank = a.lv.bank + (long long)q * d.hash_size;
    const unsigned hmask = (unsigned)d.hash_size - 1u;
    const long long wbase = (long long)b * d.C;
    int32_t* vict = a.ws.vict + wbase;
    int32_t* adm = a.ws.adm + wbase;

    // Keys for victim selection: epoch + 1 (0 = never used), or kHitKey.
    int nhit = 0;
    for (int v = tid; v < H; v += BD) {
        const int e = ep[v];
        const bool hit = (e == E);
        keys[v] = hit ? kHitKey : (unsigned)(e + 1);
        nhit += hit;
    }
    nhit = block_sum(nhit, s_tmp);  // includes the barrier that publishes keys
    const int cap = H - nhit;
    const int m = U < cap ? U : cap;

    int evicted = 0;
    if (m > 0) {
        // ---- victims: m smallest (key, slot) among non-hit slots ------------
        const int bits = 32 - __clz(E);  // keys lie in [0, E]
        int need = m;
        unsigned thr = 0u;
        if (bits > 0) thr = radix_select(keys, H, m, bits, s_hist, s_sel, &need);
        // Each warp owns a contiguous chunk of slots, read lane by lane, so
        // ballots keep ascending slot order without shared-memory conflicts.
        const int lane = tid & 31, warp = tid >> 5, nw = BD >> 5;
        const int chunk = ((H + nw - 1) / nw + 31) & ~31;
        const int w0 = warp * chunk, w1 = min(H, w0 + chunk);
        int eq = 0;
        for (int v0 = w0; v0 < w1; v0 += 32) {
            const int v = v0 + lane;
            eq += __popc(__ballot_sync(0xffffffffu, v < w1 && keys[v] == thr));
        }
        int eq_total;
        const int eq_before = block_exclusive_scan(lane == 0 ? eq : 0, s_tmp, &eq_total);
        const int eq_w = __shfl_sync(0xffffffffu, eq_before, 0);
        int nv = 0;
        {
            int er = eq_w;
            for (int v0 = w0; v0 < w1; v0 += 32) {
                const int v = v0 + lane;
                const unsigned k = v < w1 ? keys[v] : kHitKey;
                const unsigned em = __ballot_sync(0xffffffffu, k == thr);
                const bool take = k < thr || (k == thr && er + __popc(em & lanemask_lt()) < need);
                nv += __popc(__ballot_sync(0xffffffffu, take));
                er += __popc(em);
            }
        }
        int nv_total;
        const int v_before = block_exclusive_scan(lane == 0 ? nv : 0, s_tmp, &nv_total);
        {
            int er = eq_w;
            int vpos = __shfl_sync(0xffffffffu, v_before, 0);
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
            __syncthreads();
            for (int x0 = tid & ~31; x0 < U; x0 += BD) {  // per-step counts, one add per warp
                const int j = x0 + lane;
                const int l = j < U ? last[j] : -1;
                for (int st = 0; st < a.S; ++st) {
                    const int c = __popc(__ballot_sync(0xffffffffu, l == st));
                    if (lane == 0 && c) atomicAdd(&s_misc[st], c);
                }
            }
            __syncthreads();
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
            const int es_before = block_exclusive_scan(lane == 0 ? eqs : 0, s_tmp, &eqs_total);
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
            const int a_before = block_exclusive_scan(lane == 0 ? na : 0, s_tmp, &na_total);
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
        __syncthreads();
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
        evicted = block_sum(evicted, s_tmp);
        fresh = block_sum(fresh, s_tmp);
        if (tid == 0) {
            s_misc[0] = ctrl[CTRL_USED] + fresh;
            s_misc[1] = ctrl[CTRL_RESIDENT] + m - evicted;
        }
        __syncthreads();
        // ---- rebuild the bank once deleted entries pile up ---------------------
        if (!d.dense && s_misc[0] > (d.hash_size / 4) * 3) {
            for (int p = tid; p < d.hash_size; p += BD) bank[p] = kEmpty;
            __syncthreads();
            for (int v = tid; v < H; v += BD) {
                const int t = tok[v];
                if (t >= 0) bank_insert(bank, d.hash_shift, hmask, t, v, a.ws.status);
            }
            if (tid == 0) {
                s_misc[0] = s_misc[1];
                ctrl[CTRL_REBUILDS] += 1;
            }
        }
        __syncthreads();
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

// Where a unique miss's row comes from and goes to: the gather's workspace
// lists (token -> host row of request q) ...
struct WorkspaceRows {
    const int32_t* cnt;
    const int32_t* miss_tok;
    const int32_t* miss_dst;
    int32_t L, C;
    __device__ int count(int b) const { return cnt[(long long)b * kCntWords + CNT_U]; }
    __device__ void rows(int b, int j, long long* src, long long* dst) const {
        const long long wi = (long long)b * C + j;
        *src = (long long)cnt[(long long)b * kCntWords + CNT_Q] * L + miss_tok[wi];
        *dst = miss_dst[wi];
    }
    __device__ bool valid(long long, long long) const { return true; }  // written by the gather
};

// ... or a recorded miss plan (host row, device row, count per batch row).
struct RecordedRows {
    const long long* src;
    const long long* dst;
    const int32_t* count_;
    int32_t C;
    long long src_rows, dst_rows;  // rows of the host pool and of the device buffer
    uint32_t* status;
    // The plan comes from the caller: a count outside [0, C] is clamped and a
    // row outside its buffer is skipped, both flagged, never accessed.
    __device__ int count(int b) const {
        const int n = count_[b];
        if (n >= 0 && n <= C) return n;
        atomicOr(status, HS_STATUS_BAD_PLAN);
        return n < 0 ? 0 : C;
    }
    __device__ void rows(int b, int j, long long* s, long long* d) const {
        *s = src[(long long)b * C + j];
        *d = dst[(long long)b * C + j];
    }
    __device__ bool valid(long long s, long long d) const {
        if (s >= 0 && s < src_rows && d >= 0 && d < dst_rows) return true;
        atomicOr(status, HS_STATUS_BAD_PLAN);
        return false;
    }
};

// Copies every listed row (W bytes) from the host pool to the device buffer.
// The rows of all batch rows are flattened; CTA `cta` of `ncta` takes one
// contiguous span of 16-byte pieces, consecutive threads on consecutive
// pieces, each thread issuing kCopyUnroll loads before its stores.
template <typename Rows>
__device__ void copy_rows(const Rows& plan, int B, int W, const uint8_t* pool, uint8_t* kv,
                          int cta, int ncta, int* pre) {
    __shared__ int s_tmp[33];
    const int tid = threadIdx.x, BD = blockDim.x;
    // Exclusive prefix of the per-row counts over the batch rows.
    const int per = (B + BD - 1) / BD;
    const int b0 = tid * per, b1 = min(B, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; ++b) sum += plan.count(b);
    int total;
    int run = block_exclusive_scan(sum, s_tmp, &total);
    for (int b = b0; b < b1; ++b) {
        pre[b] = run;
        run += plan.count(b);
    }
    if (tid == 0) pre[B] = total;
    __syncthreads();
    if (total == 0) return;

    const int nv = W >> 4;  // 16-byte pieces per row
    const long long chunks = (long long)total * nv;
    const long long span = (chunks + ncta - 1) / ncta;
    const long long c0 = (long long)cta * span;
    const long long c1 = min(chunks, c0 + span);
    for (long long g = c0; g < c1; g += (long long)BD * kCopyUnroll) {
        uint4 v[kCopyUnroll];
        long long dst[kCopyUnroll];  // destination byte offset of each piece, -1 if none
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const long long c = g + (long long)u * BD + tid;
            dst[u] = -1;
            if (c < c1) {
                const int row = (int)(c / nv);
                const int piece = (int)(c - (long long)row * nv);
                int lo = 0, hi = B;  // last b with pre[b] <= row
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (pre[mid] <= row) lo = mid;
                    else hi = mid;
                }
                long long srow, drow;
                plan.rows(lo, row - pre[lo], &srow, &drow);
                if (plan.valid(srow, drow)) {
                    dst[u] = drow * W + ((long long)piece << 4);
                    v[u] = ld_stream_v4(pool + srow * W + ((long long)piece << 4));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u)
            if (dst[u] >= 0) st_v4(kv + dst[u], v[u]);
    }
}

__global__ void __launch_bounds__(kBlock, 2) commit_copy_kernel(const SwapArgs a, int copy_ctas) {
    extern __shared__ __align__(16) unsigned char smem[];
    if ((int)blockIdx.x < a.B) {
        // Before the gather finishes: pull this request's policy state into
        // L2 (a prefetch only; nothing is read before the wait below).
        const int q = a.rpi[blockIdx.x];
        if (q >= 0 && q < a.d.R) {
            const Dims& d = a.d;
            l2_prefetch(a.lv.ep + (long long)q * d.H, (size_t)d.H * 4);
            l2_prefetch(a.lv.tok + (long long)q * d.H, (size_t)d.H * 4);
            l2_prefetch(a.lv.phys + (long long)q * (d.H + d.C), (size_t)(d.H + d.C) * 4);
            l2_prefetch(a.lv.bank + (long long)q * d.hash_size, (size_t)d.hash_size * 8);
        }
    }
    pdl_wait();  // the gather grid's results are visible after this
    if ((int)blockIdx.x < a.B) {
        commit_request(a, blockIdx.x, reinterpret_cast<unsigned*>(smem));
    } else {
        const WorkspaceRows plan{a.ws.cnt, a.ws.miss_tok, a.ws.miss_dst, a.d.L, a.d.C};
        copy_rows(plan, a.B, a.d.W, a.lv.host_pool, a.lv.device_kv, blockIdx.x - a.B, copy_ctas,
                  reinterpret_cast<int*>(smem));
    }
}

// Replays a recorded miss plan (the deferred copy of a swap-in call).
__global__ void __launch_bounds__(kBlock, 2) planned_copy_kernel(const RecordedRows plan, int B,
                                                                  int W, const uint8_t* pool,
                                                                  uint8_t* kv) {
    extern __shared__ __align__(16) unsigned char smem[];
    copy_rows(plan, B, W, pool, kv, blockIdx.x, gridDim.x, reinterpret_cast<int*>(smem));
}

}  // namespace

size_t commit_smem_bytes(const Dims& d) {
    const size_t keys = (size_t)d.H * 4;
    const size_t pre = (size_t)(d.B_max + 1) * 4;
    return keys > pre ? keys : pre;
}

cudaError_t launch_commit_copy(const SwapArgs& a, int copy_ctas, bool pdl, cudaStream_t s) {
    static SmemOptIn opt_in;
    const size_t smem = commit_smem_bytes(a.d);
    cudaError_t e = ensure_smem(commit_copy_kernel, smem, &opt_in);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.B + copy_ctas);
    cfg.blockDim = dim3(kBlock);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, commit_copy_kernel, a, copy_ctas);
}

cudaError_t launch_planned_copy(const long long* src, const long long* dst, const int32_t* count,
                                int32_t B, int32_t C, int32_t W, const uint8_t* pool,
                                long long pool_rows, uint8_t* kv, long long kv_rows,
                                uint32_t* status, int ctas, cudaStream_t s) {
    static SmemOptIn opt_in;
    const size_t smem = (size_t)(B + 1) * 4;
    cudaError_t e = ensure_smem(planned_copy_kernel, smem, &opt_in);
    if (e != cudaSuccess) return e;
    const RecordedRows plan{src, dst, count, C, pool_rows, kv_rows, status};
    planned_copy_kernel<<<ctas, kBlock, smem, s>>>(plan, B, W, pool, kv);
    return cudaGetLastError();
}

}  // namespace hs
