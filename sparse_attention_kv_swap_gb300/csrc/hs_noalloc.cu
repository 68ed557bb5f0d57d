// hs_swap_in_noalloc: the swap-in for callers that cannot allocate device
// memory.  It has no counterpart in the pages this library follows.
//
// Some callers cannot call cudaMalloc (or any routine that allocates) on the
// path that issues swap-ins.  Examples are a plugin that a serving runtime
// hands only its input and output tensors, and a runtime whose device memory
// all comes from its own pool, reserved up front, so that an allocation
// behind its back could fail or fragment that pool.  This entry point behaves
// exactly like hs_swap_in, but the per-call scratch of the kernel (miss
// lists, admission list, per-batch-row words) lives in one
// file-scope device array of fixed size, not in the handle's workspace.
// Every GPU that loads the library holds the array until the process exits.
#include <cuda.h>  // CUcontext and CUresult only: the two driver calls below come
                   // from the runtime's entry-point query, so nothing links libcuda

#include <mutex>

#include "hs_internal.cuh"

namespace hs {
namespace {

// The shared per-call scratch.  In host code this name is only a host-side
// stand-in; kernels get its device address from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[HS_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
struct ScratchAddress {
    unsigned long long context;  // id of the context the address belongs to (0: none)
    void* addr;
};
ScratchAddress g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current CUDA context, or 0 if there is
// none yet or it cannot be read.  A device's primary context gets a new id
// when it is created again (after cudaDeviceReset, for example), and a
// symbol's address is only valid in the context it was looked up in.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
        cudaGetLastError();  // a failed query is not sticky; clear it
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Device address of the scratch array on `device` (the current device).
// Looked up once per device and context: the first call on a device, and
// the first after its context was created again, asks the runtime
// (cudaGetSymbolAddress, which also makes the context current on this
// thread if it was not); later calls reuse the address.
cudaError_t scratch_address(int device, unsigned char** out) {
    if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    unsigned long long ctx = current_context_id();
    ScratchAddress& slot = g_scratch[device];
    if (ctx == 0 || slot.addr == nullptr || slot.context != ctx) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (ctx == 0) ctx = current_context_id();  // the lookup made the context current
        slot.context = ctx;
        slot.addr = ctx ? p : nullptr;  // without a context id, look it up every call
        *out = static_cast<unsigned char*>(p);
        return cudaSuccess;
    }
    *out = static_cast<unsigned char*>(slot.addr);
    return cudaSuccess;
}

}  // namespace

// Bytes of per-call scratch a call with `batch` rows needs (same regions as
// the handle's workspace, sized for `batch` rather than max_batch).  The
// kernel zeroes the per-batch-row words it counts with before using them,
// and writes every list entry before reading it, so nothing needs clearing.
static size_t noalloc_bytes(const Dims& d, int batch) {
    const size_t bc = align256((size_t)batch * d.C * 4);
    return 4 * bc + align256((size_t)batch * kCntWords * 4);
}

}  // namespace hs

using namespace hs;

extern "C" int hs_swap_in_noalloc(hs_state* st, const int32_t* req_pool_indices_dev,
                                  const int32_t* seq_lens_dev, const int32_t* topk_dev,
                                  int32_t batch, int32_t num_steps, int32_t layer_id,
                                  int32_t* device_locs_dev, int32_t* stats_dev,
                                  int64_t* miss_src_dev, int64_t* miss_dst_dev,
                                  int32_t* miss_count_dev, void* stream) {
    if (!st) return HS_ERR_INVALID_ARG;
    const Dims& d = st->d;
    if (batch < 0 || batch > d.B_max) return HS_ERR_INVALID_ARG;
    if (num_steps < 1 || num_steps > d.S_max) return HS_ERR_INVALID_ARG;
    if (layer_id < 0 || layer_id >= d.layers) return HS_ERR_INVALID_ARG;
    const int plan = (miss_src_dev != nullptr) + (miss_dst_dev != nullptr) +
                     (miss_count_dev != nullptr);
    if (plan != 0 && plan != 3) return HS_ERR_INVALID_ARG;
    if (st->defer_copy && plan == 0) return HS_ERR_INVALID_ARG;
    if (noalloc_bytes(d, batch) > HS_NOALLOC_SCRATCH_BYTES) return HS_ERR_UNSUPPORTED;
    if (batch == 0) return HS_OK;
    if (!req_pool_indices_dev || !seq_lens_dev || !topk_dev || !device_locs_dev)
        return HS_ERR_INVALID_ARG;
    if (!null_or_aligned(req_pool_indices_dev, 4) || !null_or_aligned(seq_lens_dev, 4) ||
        !null_or_aligned(topk_dev, 4) || !null_or_aligned(device_locs_dev, 4) ||
        !null_or_aligned(stats_dev, 4) || !null_or_aligned(miss_count_dev, 4) ||
        !null_or_aligned(miss_src_dev, 8) || !null_or_aligned(miss_dst_dev, 8))
        return HS_ERR_INVALID_ARG;

    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return HS_ERR_CUDA;
    if (device != st->device) return HS_ERR_INVALID_ARG;
    unsigned char* scratch = nullptr;
    if (scratch_address(device, &scratch) != cudaSuccess) return HS_ERR_CUDA;

    // Carve the scratch like the workspace; the status word stays the
    // handle's, so hs_get_status reports this call's device flags too.
    const size_t bc = align256((size_t)batch * d.C * 4);
    Workspace ws;
    ws.miss_tok = reinterpret_cast<int32_t*>(scratch);
    ws.miss_last = reinterpret_cast<int32_t*>(scratch + bc);
    ws.miss_dst = reinterpret_cast<int32_t*>(scratch + 2 * bc);
    ws.adm = reinterpret_cast<int32_t*>(scratch + 3 * bc);
    ws.cnt = reinterpret_cast<int32_t*>(scratch + 4 * bc);
    ws.status = reinterpret_cast<uint32_t*>(st->ws + st->wl.status);

    SwapArgs a = {};
    a.d = d;
    a.lv = layer_view(d, st->state, layer_id, st->host_pool_dev[layer_id],
                      st->device_kv[layer_id]);
    a.ws = ws;
    a.rpi = req_pool_indices_dev;
    a.seq_lens = seq_lens_dev;
    a.topk = topk_dev;
    a.B = batch;
    a.S = num_steps;
    a.locs = device_locs_dev;
    a.stats = stats_dev;
    a.plan_src = reinterpret_cast<long long*>(miss_src_dev);
    a.plan_dst = reinterpret_cast<long long*>(miss_dst_dev);
    a.plan_count = miss_count_dev;
    a.defer_copy = st->defer_copy;
    a.timeline = st->timeline;
    return launch_swapin(a, st->num_sms, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? HS_OK
               : HS_ERR_CUDA;
}
