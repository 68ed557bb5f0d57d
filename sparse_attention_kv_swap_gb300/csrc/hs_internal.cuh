// Internal layout and launch interface of the GB300 swap-in library.
//
// Device memory is caller-owned and carved here into:
//   state (persistent, per layer l and request q):
//     bank  int64 [layers][R][hash_size]  token -> slot hash, (t << 32) | slot;
//                                         -1 never used, -2 deleted
//     map   int16 [layers][R][L]          dense index instead of the bank:
//                                         slot of each position, -1 absent
//     ep    int32 [layers][R][H]          epoch of the slot's last reference
//     tok   int32 [layers][R][H]          token held by the slot (-1 empty)
//     phys  int32 [layers][R][H + C]      physical row of each position
//     ctrl  int32 [layers][R][8]          control words (see Ctrl)
//     totals uint64 [layers][16]          running sums of the HS_STAT_* counters
//   workspace (one call at a time, shared by all layers):
//     miss_tok / miss_last / miss_dst / adm  int32 [B_max][C]
//     cnt   int32 [B_max][16]             per-batch-row words (copy claim counter)
//     status uint32                       sticky device status flags
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "hisparse_swap.h"

namespace hs {

constexpr long long kEmpty = -1;    // hash entry never used
constexpr long long kDeleted = -2;  // hash entry deleted (probe continues)

constexpr int kCtrlWords = 8;
enum Ctrl : int {
    CTRL_EPOCH = 0,     // epoch of the next call
    CTRL_RESIDENT = 1,  // tokens resident in the hot slots
    CTRL_USED = 2,      // hash entries not empty (live + deleted)
    CTRL_LOCK = 3,      // held from the lookup to the commit of one call
    CTRL_REBUILDS = 4,  // hash rebuilds so far (diagnostic)
};

constexpr int kTotalsWords = 16;  // per layer; the first HS_NUM_STATS are used
constexpr int kCntWords = 16;
enum Cnt : int {
    CNT_CLAIM = 0,  // 16-byte pieces of the batch row's miss rows claimed by copying warps
};

// Words of the optional per-CTA timeline (hs_set_timeline): [b][rank][16],
// global-timer nanoseconds unless noted.
constexpr int kTimelineCtas = 8;    // cluster ranks per batch row (P <= 8)
constexpr int kTimelineWords = 16;  // words per CTA
enum TimelineWord : int {
    TL_START = 0,         // CTA start
    TL_PROBED = 1,        // its index probes answered
    TL_BARRIER0 = 2,      // past the first cluster barrier (tables cleared)
    TL_INSERTED = 3,      // its de-duplication inserts issued
    TL_BARRIER_A = 4,     // past the second (tables complete)
    TL_FLAGGED = 5,       // its first-occurrence flags known
    TL_BARRIER_B = 6,     // past the third (flag words and counts exchanged)
    TL_ROWS = 7,          // its hit and miss rows loaded
    TL_BARRIER_C = 8,     // past the fourth (locations and miss lists written)
    TL_COMMITTED = 9,     // commit done (leader only)
    TL_COPIED = 10,       // its last warp done copying
    TL_CLUSTER_SIZE = 15  // P (a count, not a time)
};

struct Dims {
    int32_t R, L, W, H, K, S_max, C, layers, B_max;
    int32_t hash_size;   // entries per request bank, power of two (>= 32); 0 if dense
    int32_t hash_shift;  // 32 - log2(hash_size)
    int32_t dense;       // 1: token -> slot index is the dense map, not the hash bank
    int32_t E;           // extra-page rows per request (0 = no extra page)
};

struct LayerView {
    long long* bank;           // [R][hash_size] (hash index)
    int16_t* map;              // [R][L] slot of each position, -1 if absent (dense index)
    int32_t* ep;               // [R][H]
    int32_t* tok;              // [R][H]
    int32_t* phys;             // [R][H + C]
    int32_t* ctrl;             // [R][kCtrlWords]
    unsigned long long* totals;  // [kTotalsWords] running sums of the HS_STAT_* counters
    const uint8_t* host_pool;  // device mapping of the pinned pool [R][L][W]
    uint8_t* device_kv;        // [R * (H + C) + R * E][W]: hot + scratch rows, extra pages
};

struct Workspace {
    int32_t* miss_tok;   // [B_max][C] token of unique miss j
    int32_t* miss_last;  // [B_max][C] last step in which miss j occurs
    int32_t* miss_dst;   // [B_max][C] device row miss j was written to
    int32_t* adm;        // [B_max][C] admitted ordinals in ascending order
    int32_t* cnt;        // [B_max][kCntWords]
    uint32_t* status;    // sticky HS_STATUS_* flags
};

struct SwapArgs {
    Dims d;
    LayerView lv;
    Workspace ws;
    const int32_t* rpi;       // [B]
    const int32_t* seq_lens;  // [B]
    const int32_t* topk;      // [B][S][K]
    int32_t B, S;
    int32_t* locs;      // [B][S][K]
    int32_t* stats;     // [B][HS_NUM_STATS] or null
    long long* plan_src;  // [B][C] or null
    long long* plan_dst;  // [B][C] or null
    int32_t* plan_count;  // [B] or null
    int32_t defer_copy;   // 1: record the plan only, copy no rows
    unsigned long long* timeline;  // [B][kTimelineCtas][kTimelineWords] or null
    // set by the launcher:
    int32_t step_bits;      // 1: record each miss's last step (the call may overflow)
    int32_t dedup_entries;  // entries of one CTA's share of the miss de-duplication table
    int32_t dedup_shift;    // hash de-duplication: 32 - log2(P * dedup_entries)
};

// Byte offsets of the state and workspace regions (256-byte aligned).
struct StateLayout {
    size_t bank, map, ep, tok, phys, ctrl, totals, total;
};
struct WorkspaceLayout {
    size_t miss_tok, miss_last, miss_dst, adm, cnt, status, total;
};

StateLayout state_layout(const Dims& d);
WorkspaceLayout workspace_layout(const Dims& d);
LayerView layer_view(const Dims& d, uint8_t* state, int layer, const uint8_t* host_pool,
                     uint8_t* device_kv);
Workspace workspace_view(const Dims& d, uint8_t* ws);

// The dynamic shared-memory size a kernel has been opened up to, per device
// (cudaFuncSetAttribute acts on the calling thread's current device).  Reads
// are lock-free; raising the limit takes the mutex, so that concurrent host
// threads leave the attribute and the remembered size equal.  Nothing is
// assumed open at first: without the attribute, static plus dynamic shared
// memory must stay within 48 KB, so the limit a kernel starts with depends
// on its own static arrays.
struct SmemOptIn {
    static constexpr int kMaxDevices = 64;
    std::atomic<int> bytes[kMaxDevices];
    std::mutex raise;
    SmemOptIn() {
        for (auto& b : bytes) b.store(0, std::memory_order_relaxed);
    }
};

// Raises a kernel's dynamic shared-memory limit on the current device to at
// least `bytes`; repeated calls cost one atomic load.
template <typename F>
cudaError_t ensure_smem(F* kernel, size_t bytes, SmemOptIn* opt) {
    if (bytes == 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= SmemOptIn::kMaxDevices)
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)bytes);
    if ((int)bytes <= opt->bytes[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(opt->raise);
    if ((int)bytes <= opt->bytes[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) opt->bytes[dev].store((int)bytes, std::memory_order_release);
    return e;
}

// Launch shape of one swap-in call (see swapin_shape in hs_swapin.cu).
struct SwapinShape {
    int P;          // CTAs per batch row (thread-block cluster size), power of two <= 8
    int rmax;       // entries per thread (1, 2 or 4)
    int block;      // threads per CTA
    bool by_position;  // miss de-duplication table indexed by token position (else hashed)
    int dedup_entries; // entries of one CTA's share of that table
    size_t smem;    // dynamic shared memory per CTA
};
SwapinShape swapin_shape(const Dims& d, int batch, int steps, int sms, int p_cap);
bool step_bits_needed(const Dims& d, int steps);

// Launchers (each returns the launch's error code).
cudaError_t launch_swapin(const SwapArgs& a, int sms, cudaStream_t s);
cudaError_t launch_planned_copy(const long long* src, const long long* dst, const int32_t* count,
                                int32_t B, int32_t C, int32_t W, const uint8_t* pool,
                                long long pool_rows, uint8_t* kv, long long kv_rows,
                                uint32_t* status, int ctas, cudaStream_t s);
cudaError_t launch_append(const Dims& d, const LayerView& lv, uint8_t* host_pool,
                          const int32_t* req, const int32_t* tok, const int32_t* seq_lens,
                          const uint8_t* rows, int32_t n, uint32_t* status, cudaStream_t s);
cudaError_t launch_reset(const Dims& d, uint8_t* state, const int32_t* rpi, int32_t n,
                         cudaStream_t s);
cudaError_t launch_page_table(const int32_t* topk, const int32_t* seq_lens, int32_t B,
                              int32_t S, int32_t K, int32_t L_max, int32_t page_size,
                              int32_t* pages, int32_t* num_pages, int32_t* token_page,
                              cudaStream_t s);

// ---- device helpers shared by the kernels -----------------------------------
#ifdef __CUDACC__

// Multiplicative (Fibonacci) hash of a token into a table of 2^(32 - shift)
// entries: the top bits of t * 2^32 / golden ratio.
__device__ __forceinline__ uint32_t hash_token(int32_t t, int shift) {
    return ((uint32_t)t * 0x9E3779B9u) >> shift;
}

__device__ __forceinline__ long long make_entry(int32_t t, int32_t slot) {
    return ((long long)t << 32) | (uint32_t)slot;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Nanoseconds of the GPU's global timer (timeline stamps).
__device__ __forceinline__ unsigned long long global_timer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// 16-byte load that bypasses L1 (each host row is read once).
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

// Non-binding prefetch into L2 of the 128-byte lines of [p, p + bytes) that
// fall to this thread when `nthreads` threads numbered `first` on share them.
__device__ __forceinline__ void l2_prefetch(const void* p, size_t bytes, int first, int nthreads) {
    const char* c = static_cast<const char*>(p);
    for (size_t off = (size_t)first * 128; off < bytes; off += (size_t)nthreads * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(c + off));
}

// Inclusive warp scan.
__device__ __forceinline__ int warp_inclusive_scan(int x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// Exclusive block scan of one int per thread; returns the prefix and the
// block total.  `tmp` needs 33 ints of shared memory.  All threads call it.
__device__ __forceinline__ int block_exclusive_scan(int x, int* tmp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    int inc = warp_inclusive_scan(x);
    if (lane == 31) tmp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nwarps ? tmp[lane] : 0;
        int wi = warp_inclusive_scan(w);
        tmp[lane] = wi - w;
        if (lane == 31) tmp[32] = wi;
    }
    __syncthreads();
    int r = tmp[warp] + inc - x;
    *total = tmp[32];
    __syncthreads();
    return r;
}

__device__ __forceinline__ int block_sum(int x, int* tmp) {
    int total;
    block_exclusive_scan(x, tmp, &total);
    return total;
}

#endif  // __CUDACC__

}  // namespace hs

#include <vector>

// The host handle behind the C ABI's opaque hs_state.
struct hs_state {
    hs_config cfg;
    hs::Dims d;
    hs::StateLayout sl;
    hs::WorkspaceLayout wl;
    uint8_t* state;
    uint8_t* ws;
    std::vector<const uint8_t*> host_pool_dev;  // device mapping of each layer's pool
    std::vector<uint8_t*> device_kv;
    int device;
    int num_sms;
    int copy_ctas;            // CTAs of hs_copy_planned
    unsigned long long* timeline;  // per-CTA phase stamps of later calls, or null
    int defer_copy;           // 1: hs_swap_in records the miss plan but copies nothing
};

// True for a null pointer or one aligned to `bytes` (the element size of an
// int32 or int64 argument; the kernels load these arrays element by element).
inline bool null_or_aligned(const void* p, size_t bytes) {
    return ((uintptr_t)p % bytes) == 0;
}

// True when the calling thread's current device is the one the handle was
// created on.  Every entry point that launches or copies checks it, so that a
// call made while another device is current fails instead of running there.
inline bool on_handle_device(const hs_state* st) {
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess && dev == st->device;
}
