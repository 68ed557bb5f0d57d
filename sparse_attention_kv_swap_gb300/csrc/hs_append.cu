// Write-back of newly decoded KV rows (sm_103a).
//
// Decode keeps idle KV in host memory (PR #20343 summary, 功能与动机), so
// every row that decode produces is written to the request's host pool row;
// the same row also goes to the request's extra page (its newest,
// still-filling page, which the swap-in serves without a lookup: "[HiSparse]
// Support hisparse multi-step swap io kernel", 实现拆解 item 1) when the
// position lies on it, and to the token's hot row when the token is
// resident, so that every copy of (q, t) stays equal.
//
// One warp per entry, in 16-byte vectors.  The warp loads the row while
// lane 0 validates the entry; it then stores the host pool row (over the host
// link, into the mapped pool) and the extra-page row, which follow from
// (q, t) alone, and only then resolves the hot row through the token -> slot
// index and the position table, so that the index lookups overlap the stores
// in flight.
#include "hs_internal.cuh"

namespace hs {
namespace {

constexpr int kAppendWarps = 8;  // entries per CTA

struct AppendArgs {
    Dims d;
    LayerView lv;
    uint8_t* pool;  // device mapping of the layer's host pool [R][L][W], written
    const int32_t* req;
    const int32_t* tok;
    const int32_t* seq_lens;
    const uint8_t* rows;  // [n][W] device
    int32_t n;
    uint32_t* status;
};

// Hot slot holding token t of request q, or -1 (bounded probe of the hash
// bank, or one load of the dense map).
__device__ int resident_slot(const Dims& d, const LayerView& lv, int q, int t,
                             uint32_t* status) {
    if (d.dense) {
        const int slot = lv.map[(long long)q * d.L + t];
        return (slot >= 0 && slot < d.H) ? slot : -1;
    }
    const long long* bank = lv.bank + (long long)q * d.hash_size;
    const unsigned mask = (unsigned)d.hash_size - 1u;
    unsigned p = hash_token(t, d.hash_shift);
    for (int n = 0; n < d.hash_size; ++n) {
        const long long x = bank[p];
        if (x == kEmpty) return -1;
        if (x >= 0 && (int)(x >> 32) == t) {
            const int slot = (int)(x & 0xffffffffll);
            if (slot < d.H) return slot;
            atomicOr(status, HS_STATUS_PROBE_LIMIT);  // corrupt entry
            return -1;
        }
        p = (p + 1u) & mask;
    }
    atomicOr(status, HS_STATUS_PROBE_LIMIT);
    return -1;
}

__global__ void __launch_bounds__(kAppendWarps * 32) append_kernel(const AppendArgs a) {
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
    if (i >= a.n) return;
    const Dims& d = a.d;
    const int vecs = d.W >> 4;
    const int4* src = reinterpret_cast<const int4*>(a.rows + (long long)i * d.W);
    // The first 64 vectors of the row (1 KB) are loaded at once, alongside
    // the entry itself: neither depends on the other.
    int4 x0 = make_int4(0, 0, 0, 0), x1 = x0;
    if (lane < vecs) x0 = __ldg(src + lane);
    if (lane + 32 < vecs) x1 = __ldg(src + lane + 32);
    int q = 0, t = 0, limit = 0;
    if (lane == 0) {
        q = __ldg(a.req + i);
        t = __ldg(a.tok + i);
        const int sl = __ldg(a.seq_lens + i);
        limit = sl < d.L ? sl : d.L;
        if (q < 0 || q >= d.R || t < 0 || t >= limit) {
            atomicOr(a.status, HS_STATUS_BAD_APPEND);
            q = -1;
        }
    }
    q = __shfl_sync(0xffffffffu, q, 0);
    t = __shfl_sync(0xffffffffu, t, 0);
    limit = __shfl_sync(0xffffffffu, limit, 0);
    if (q < 0) return;
    // Host row and extra-page row follow from (q, t) alone: store them first.
    int4* dst_host = reinterpret_cast<int4*>(a.pool + ((long long)q * d.L + t) * d.W);
    int4* dst_x = nullptr;
    if (d.E > 0 && t >= (limit - 1) / d.E * d.E)
        dst_x = reinterpret_cast<int4*>(
            a.lv.device_kv + ((long long)d.R * (d.H + d.C) + (long long)q * d.E + t % d.E) * d.W);
    if (lane < vecs) {
        dst_host[lane] = x0;
        if (dst_x) dst_x[lane] = x0;
    }
    if (lane + 32 < vecs) {
        dst_host[lane + 32] = x1;
        if (dst_x) dst_x[lane + 32] = x1;
    }
    // The hot copy, if the token is resident: index lookup, then its row.
    long long hrow = -1;
    if (lane == 0) {
        const int slot = resident_slot(d, a.lv, q, t, a.status);
        if (slot >= 0) {
            const long long base = (long long)q * (d.H + d.C);
            hrow = base + a.lv.phys[base + slot];
        }
    }
    hrow = __shfl_sync(0xffffffffu, hrow, 0);
    int4* dst_h = hrow >= 0 ? reinterpret_cast<int4*>(a.lv.device_kv + hrow * d.W) : nullptr;
    if (dst_h) {
        if (lane < vecs) dst_h[lane] = x0;
        if (lane + 32 < vecs) dst_h[lane + 32] = x1;
    }
    // Rows longer than 1 KB: the rest, vector by vector.
    for (int v = lane + 64; v < vecs; v += 32) {
        const int4 x = __ldg(src + v);
        dst_host[v] = x;
        if (dst_x) dst_x[v] = x;
        if (dst_h) dst_h[v] = x;
    }
}

}  // namespace

cudaError_t launch_append(const Dims& d, const LayerView& lv, uint8_t* host_pool,
                          const int32_t* req, const int32_t* tok, const int32_t* seq_lens,
                          const uint8_t* rows, int32_t n, uint32_t* status, cudaStream_t s) {
    AppendArgs a;
    a.d = d;
    a.lv = lv;
    a.pool = host_pool;
    a.req = req;
    a.tok = tok;
    a.seq_lens = seq_lens;
    a.rows = rows;
    a.n = n;
    a.status = status;
    const int grid = (n + kAppendWarps - 1) / kAppendWarps;
    append_kernel<<<grid, kAppendWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace hs
