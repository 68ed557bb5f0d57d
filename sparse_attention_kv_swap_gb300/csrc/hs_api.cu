// Host side of the C ABI declared in include/hisparse_swap.h: argument
// validation, state and workspace layout, and the launch of one swap-in call
// (one kernel: lookup, de-duplication, locations, commit and miss-row copy)
// on the caller's stream.
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "hs_internal.cuh"

namespace hs {

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static int32_t hash_size_for(int32_t H) {
    int32_t h = 32;
    while (h < 2 * H) h <<= 1;
    return h;
}

static Dims dims_of(const hs_config& c) {
    Dims d;
    d.R = c.num_requests;
    d.L = c.max_seq_len;
    d.W = c.item_size_bytes;
    d.H = c.hot_buffer_size;
    d.K = c.top_k;
    d.S_max = c.max_steps;
    d.C = c.max_steps * c.top_k;
    d.layers = c.num_layers;
    d.B_max = c.max_batch;
    d.dense = c.index_kind == HS_INDEX_DENSE ? 1 : 0;
    d.hash_size = d.dense ? 0 : hash_size_for(c.hot_buffer_size);
    d.hash_shift = d.dense ? 0 : 32 - __builtin_ctz((unsigned)d.hash_size);
    d.E = c.extra_page_size;
    return d;
}

StateLayout state_layout(const Dims& d) {
    StateLayout s;
    const size_t lr = (size_t)d.layers * d.R;
    size_t o = 0;
    s.bank = o;
    o = align256(o + lr * d.hash_size * 8);
    s.map = o;
    o = align256(o + (d.dense ? lr * d.L * 2 : 0));
    s.ep = o;
    o = align256(o + lr * d.H * 4);
    s.tok = o;
    o = align256(o + lr * d.H * 4);
    s.phys = o;
    o = align256(o + lr * (size_t)(d.H + d.C) * 4);
    s.ctrl = o;
    o = align256(o + lr * kCtrlWords * 4);
    s.totals = o;
    o = align256(o + (size_t)d.layers * kTotalsWords * 8);
    s.total = o;
    return s;
}

WorkspaceLayout workspace_layout(const Dims& d) {
    WorkspaceLayout w;
    const size_t bc = (size_t)d.B_max * d.C * 4;
    size_t o = 0;
    w.miss_tok = o;
    o = align256(o + bc);
    w.miss_last = o;
    o = align256(o + bc);
    w.miss_dst = o;
    o = align256(o + bc);
    w.adm = o;
    o = align256(o + bc);
    w.cnt = o;
    o = align256(o + (size_t)d.B_max * kCntWords * 4);
    w.status = o;
    o = align256(o + 4);
    w.total = o;
    return w;
}

LayerView layer_view(const Dims& d, uint8_t* state, int layer, const uint8_t* host_pool,
                     uint8_t* device_kv) {
    const StateLayout s = state_layout(d);
    const size_t lq = (size_t)layer * d.R;
    LayerView v;
    v.bank = reinterpret_cast<long long*>(state + s.bank) + lq * d.hash_size;
    v.map = reinterpret_cast<int16_t*>(state + s.map) + (d.dense ? lq * d.L : 0);
    v.ep =reinterpret_cast<int32_t*>(state + s.ep) + lq * d.H;
    v.tok = reinterpret_cast<int32_t*>(state + s.tok) + lq * d.H;
    v.phys = reinterpret_cast<int32_t*>(state + s.phys) + lq * (d.H + d.C);
    v.ctrl = reinterpret_cast<int32_t*>(state + s.ctrl) + lq * kCtrlWords;
    v.totals = reinterpret_cast<unsigned long long*>(state + s.totals) +
               (size_t)layer * kTotalsWords;
    v.host_pool = host_pool;
    v.device_kv = device_kv;
    return v;
}

Workspace workspace_view(const Dims& d, uint8_t* ws) {
    const WorkspaceLayout w = workspace_layout(d);
    Workspace v;
    v.miss_tok = reinterpret_cast<int32_t*>(ws + w.miss_tok);
    v.miss_last = reinterpret_cast<int32_t*>(ws + w.miss_last);
    v.miss_dst = reinterpret_cast<int32_t*>(ws + w.miss_dst);
    v.adm = reinterpret_cast<int32_t*>(ws + w.adm);
    v.cnt = reinterpret_cast<int32_t*>(ws + w.cnt);
    v.status = reinterpret_cast<uint32_t*>(ws + w.status);
    return v;
}

}  // namespace hs

using namespace hs;

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

extern "C" {

int hs_config_check(const hs_config* c) {
    if (!c) return HS_ERR_INVALID_ARG;
    if (c->num_requests <= 0 || c->max_seq_len <= 0 || c->item_size_bytes <= 0 ||
        c->hot_buffer_size <= 0 || c->top_k <= 0 || c->max_steps <= 0 || c->num_layers <= 0 ||
        c->max_batch <= 0)
        return HS_ERR_INVALID_ARG;
    if (c->item_size_bytes % 16 != 0) return HS_ERR_INVALID_ARG;
    if (c->item_size_bytes > HS_MAX_ITEM_BYTES) return HS_ERR_UNSUPPORTED;
    if (c->max_batch > c->num_requests) return HS_ERR_INVALID_ARG;
    if (c->hot_buffer_size > HS_MAX_HOT_BUFFER) return HS_ERR_UNSUPPORTED;
    if (c->max_steps > HS_MAX_STEPS) return HS_ERR_UNSUPPORTED;
    if ((long long)c->max_steps * c->top_k > HS_MAX_ENTRIES) return HS_ERR_UNSUPPORTED;
    if (c->max_batch > 65535 || c->num_layers > 65535) return HS_ERR_UNSUPPORTED;
    if (c->index_kind != HS_INDEX_HASH && c->index_kind != HS_INDEX_DENSE)
        return HS_ERR_INVALID_ARG;
    if (c->extra_page_size < 0) return HS_ERR_INVALID_ARG;
    if (c->extra_page_size > HS_MAX_EXTRA_PAGE) return HS_ERR_UNSUPPORTED;
    // device rows and host rows must be addressable by int32 indices
    const long long dev_rows =
        (long long)c->num_requests * (c->hot_buffer_size + (long long)c->max_steps * c->top_k +
                                      c->extra_page_size);
    if (dev_rows > 0x7fffffffLL) return HS_ERR_UNSUPPORTED;
    if ((long long)c->num_requests * c->max_seq_len > 0x7fffffffffffLL) return HS_ERR_UNSUPPORTED;
    return HS_OK;
}

size_t hs_state_bytes(const hs_config* c) {
    if (hs_config_check(c) != HS_OK) return 0;
    return state_layout(dims_of(*c)).total;
}

size_t hs_workspace_bytes(const hs_config* c) {
    if (hs_config_check(c) != HS_OK) return 0;
    return workspace_layout(dims_of(*c)).total;
}

size_t hs_device_kv_bytes(const hs_config* c) {
    if (hs_config_check(c) != HS_OK) return 0;
    const Dims d = dims_of(*c);
    return (size_t)d.R * (d.H + d.C + d.E) * d.W;
}

size_t hs_host_pool_bytes(const hs_config* c) {
    if (hs_config_check(c) != HS_OK) return 0;
    return (size_t)c->num_requests * c->max_seq_len * c->item_size_bytes;
}

int32_t hs_hash_size(const hs_config* c) {
    if (hs_config_check(c) != HS_OK) return 0;
    return dims_of(*c).hash_size;
}

int hs_create_state(const hs_config* cfg, void* const* host_pool_host, void* const* device_kv_dev,
                    void* state_dev, size_t state_bytes, void* workspace_dev,
                    size_t workspace_bytes, void* stream, hs_state** out) {
    if (!out) return HS_ERR_INVALID_ARG;
    *out = nullptr;
    const int rc = hs_config_check(cfg);
    if (rc != HS_OK) return rc;
    if (!host_pool_host || !device_kv_dev || !state_dev || !workspace_dev)
        return HS_ERR_INVALID_ARG;
    const Dims d = dims_of(*cfg);
    const StateLayout sl = state_layout(d);
    const WorkspaceLayout wl = workspace_layout(d);
    if (state_bytes < sl.total || workspace_bytes < wl.total) return HS_ERR_INVALID_ARG;
    if (!aligned(state_dev, 256) || !aligned(workspace_dev, 256)) return HS_ERR_INVALID_ARG;
    for (int l = 0; l < d.layers; ++l) {
        if (!host_pool_host[l] || !device_kv_dev[l]) return HS_ERR_INVALID_ARG;
        if (!aligned(host_pool_host[l], 16) || !aligned(device_kv_dev[l], 16))
            return HS_ERR_INVALID_ARG;
    }
    hs_state* st = new (std::nothrow) hs_state;
    if (!st) return HS_ERR_INVALID_ARG;
    st->cfg = *cfg;
    st->d = d;
    st->sl = sl;
    st->wl = wl;
    st->state = static_cast<uint8_t*>(state_dev);
    st->ws = static_cast<uint8_t*>(workspace_dev);
    if (cudaGetDevice(&st->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&st->num_sms, cudaDevAttrMultiProcessorCount, st->device) !=
            cudaSuccess) {
        delete st;
        return HS_ERR_CUDA;
    }
    st->copy_ctas = 2 * st->num_sms;
    st->timeline = nullptr;
    st->defer_copy = 0;
    int pageable_ok = 0;
    cudaDeviceGetAttribute(&pageable_ok, cudaDevAttrPageableMemoryAccess, st->device);
    cudaGetLastError();
    for (int l = 0; l < d.layers; ++l) {
        // Pinned (page-locked, mapped) memory: use its device mapping.  Plain
        // pageable memory only where the device reads host page tables
        // directly (e.g. NVLink-C2C systems with address translation).
        void* dp = nullptr;
        cudaPointerAttributes attr;
        const bool known = cudaPointerGetAttributes(&attr, host_pool_host[l]) == cudaSuccess;
        cudaGetLastError();  // a failed query is not sticky; clear it
        if (known && attr.type == cudaMemoryTypeHost) {
            if (cudaHostGetDevicePointer(&dp, host_pool_host[l], 0) != cudaSuccess) dp = nullptr;
            cudaGetLastError();
        } else if (known && attr.type == cudaMemoryTypeUnregistered && pageable_ok) {
            dp = host_pool_host[l];
        }
        if (!dp) {
            delete st;
            return HS_ERR_INVALID_ARG;
        }
        st->host_pool_dev.push_back(static_cast<const uint8_t*>(dp));
        st->device_kv.push_back(static_cast<uint8_t*>(device_kv_dev[l]));
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(st->ws + wl.status, 0, 4, s) != cudaSuccess ||
        cudaMemsetAsync(st->ws + wl.cnt, 0, (size_t)d.B_max * kCntWords * 4, s) != cudaSuccess ||
        cudaMemsetAsync(st->state + sl.totals, 0, (size_t)d.layers * kTotalsWords * 8, s) !=
            cudaSuccess ||
        launch_reset(d, st->state, nullptr, d.R, s) != cudaSuccess) {
        delete st;
        return HS_ERR_CUDA;
    }
    *out = st;
    return HS_OK;
}

void hs_destroy_state(hs_state* st) { delete st; }

int hs_swap_in(hs_state* st, const int32_t* req_pool_indices_dev, const int32_t* seq_lens_dev,
               const int32_t* topk_dev, int32_t batch, int32_t num_steps, int32_t layer_id,
               int32_t* device_locs_dev, int32_t* stats_dev, int64_t* miss_src_dev,
               int64_t* miss_dst_dev, int32_t* miss_count_dev, void* stream) {
    if (!st) return HS_ERR_INVALID_ARG;
    if (!on_handle_device(st)) return HS_ERR_INVALID_ARG;
    const Dims& d = st->d;
    if (batch < 0 || batch > d.B_max) return HS_ERR_INVALID_ARG;
    if (num_steps < 1 || num_steps > d.S_max) return HS_ERR_INVALID_ARG;
    if (layer_id < 0 || layer_id >= d.layers) return HS_ERR_INVALID_ARG;
    const int plan = (miss_src_dev != nullptr) + (miss_dst_dev != nullptr) +
                     (miss_count_dev != nullptr);
    if (plan != 0 && plan != 3) return HS_ERR_INVALID_ARG;
    if (st->defer_copy && plan == 0) return HS_ERR_INVALID_ARG;
    if (batch == 0) return HS_OK;
    if (!req_pool_indices_dev || !seq_lens_dev || !topk_dev || !device_locs_dev)
        return HS_ERR_INVALID_ARG;
    if (!null_or_aligned(req_pool_indices_dev, 4) || !null_or_aligned(seq_lens_dev, 4) ||
        !null_or_aligned(topk_dev, 4) || !null_or_aligned(device_locs_dev, 4) ||
        !null_or_aligned(stats_dev, 4) || !null_or_aligned(miss_count_dev, 4) ||
        !null_or_aligned(miss_src_dev, 8) || !null_or_aligned(miss_dst_dev, 8))
        return HS_ERR_INVALID_ARG;

    SwapArgs a;
    std::memset(&a, 0, sizeof(a));
    a.d = d;
    a.lv = layer_view(d, st->state, layer_id, st->host_pool_dev[layer_id],
                      st->device_kv[layer_id]);
    a.ws = workspace_view(d, st->ws);
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

int hs_append_rows(hs_state* st, int32_t layer_id, const int32_t* req_dev,
                   const int32_t* tok_dev, const int32_t* seq_lens_dev, const void* rows_dev,
                   int32_t n, void* stream) {
    if (!st) return HS_ERR_INVALID_ARG;
    if (!on_handle_device(st)) return HS_ERR_INVALID_ARG;
    const Dims& d = st->d;
    if (layer_id < 0 || layer_id >= d.layers || n < 0) return HS_ERR_INVALID_ARG;
    if (n == 0) return HS_OK;
    if (!req_dev || !tok_dev || !seq_lens_dev || !rows_dev || !aligned(rows_dev, 16) ||
        !null_or_aligned(req_dev, 4) || !null_or_aligned(tok_dev, 4) ||
        !null_or_aligned(seq_lens_dev, 4))
        return HS_ERR_INVALID_ARG;
    const LayerView lv = layer_view(d, st->state, layer_id, st->host_pool_dev[layer_id],
                                    st->device_kv[layer_id]);
    // The pool is the caller's writable memory; the view holds it as const
    // because the swap-in only reads it.
    uint8_t* pool = const_cast<uint8_t*>(st->host_pool_dev[layer_id]);
    const Workspace ws = workspace_view(d, st->ws);
    return launch_append(d, lv, pool, req_dev, tok_dev, seq_lens_dev,
                         static_cast<const uint8_t*>(rows_dev), n, ws.status,
                         static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? HS_OK
               : HS_ERR_CUDA;
}

int hs_set_defer_copy(hs_state* st, int32_t defer) {
    if (!st) return HS_ERR_INVALID_ARG;
    st->defer_copy = defer ? 1 : 0;
    return HS_OK;
}

int hs_copy_planned(hs_state* st, int32_t layer_id, const int64_t* miss_src_dev,
                    const int64_t* miss_dst_dev, const int32_t* miss_count_dev, int32_t batch,
                    void* stream) {
    if (!st) return HS_ERR_INVALID_ARG;
    if (!on_handle_device(st)) return HS_ERR_INVALID_ARG;
    const Dims& d = st->d;
    if (layer_id < 0 || layer_id >= d.layers || batch < 0 || batch > d.B_max)
        return HS_ERR_INVALID_ARG;
    if (batch == 0) return HS_OK;
    if (!miss_src_dev || !miss_dst_dev || !miss_count_dev) return HS_ERR_INVALID_ARG;
    if (!null_or_aligned(miss_src_dev, 8) || !null_or_aligned(miss_dst_dev, 8) ||
        !null_or_aligned(miss_count_dev, 4))
        return HS_ERR_INVALID_ARG;
    return launch_planned_copy(reinterpret_cast<const long long*>(miss_src_dev),
                               reinterpret_cast<const long long*>(miss_dst_dev), miss_count_dev,
                               batch, d.C, d.W, st->host_pool_dev[layer_id],
                               (long long)d.R * d.L, st->device_kv[layer_id],
                               (long long)d.R * (d.H + d.C + d.E),
                               reinterpret_cast<uint32_t*>(st->ws + st->wl.status), st->copy_ctas,
                               static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? HS_OK
               : HS_ERR_CUDA;
}

int hs_set_timeline(hs_state* st, uint64_t* timeline_dev) {
    if (!st || !null_or_aligned(timeline_dev, 8)) return HS_ERR_INVALID_ARG;
    st->timeline = reinterpret_cast<unsigned long long*>(timeline_dev);
    return HS_OK;
}

int hs_set_copy_ctas(hs_state* st, int32_t copy_ctas) {
    if (!st || copy_ctas < 0 || copy_ctas > 65535) return HS_ERR_INVALID_ARG;
    st->copy_ctas = copy_ctas ? copy_ctas : 2 * st->num_sms;
    return HS_OK;
}

int hs_page_table(const int32_t* topk_dev, const int32_t* seq_lens_dev, int32_t batch,
                  int32_t num_steps, int32_t top_k, int32_t max_seq_len, int32_t page_size,
                  int32_t* pages_dev, int32_t* num_pages_dev, int32_t* token_page_dev,
                  void* stream) {
    if (batch < 0 || num_steps < 1 || top_k < 1 || max_seq_len < 1 || page_size < 1)
        return HS_ERR_INVALID_ARG;
    if ((long long)num_steps * top_k > HS_MAX_ENTRIES) return HS_ERR_UNSUPPORTED;
    if (((long long)max_seq_len + page_size - 1) / page_size > HS_MAX_PAGES)
        return HS_ERR_UNSUPPORTED;
    if (batch > 65535 * 32) return HS_ERR_UNSUPPORTED;
    if (batch == 0) return HS_OK;
    if (!topk_dev || !seq_lens_dev || !pages_dev || !num_pages_dev || !token_page_dev)
        return HS_ERR_INVALID_ARG;
    if (!null_or_aligned(topk_dev, 4) || !null_or_aligned(seq_lens_dev, 4) ||
        !null_or_aligned(pages_dev, 4) || !null_or_aligned(num_pages_dev, 4) ||
        !null_or_aligned(token_page_dev, 4))
        return HS_ERR_INVALID_ARG;
    return launch_page_table(topk_dev, seq_lens_dev, batch, num_steps, top_k, max_seq_len,
                             page_size, pages_dev, num_pages_dev, token_page_dev,
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? HS_OK
               : HS_ERR_CUDA;
}

int hs_reset_requests(hs_state* st, const int32_t* req_pool_indices_dev, int32_t n,
                      void* stream) {
    if (!st || n < 0) return HS_ERR_INVALID_ARG;
    if (!on_handle_device(st)) return HS_ERR_INVALID_ARG;
    if (n == 0) return HS_OK;
    if (!req_pool_indices_dev || n > st->d.R || !null_or_aligned(req_pool_indices_dev, 4))
        return HS_ERR_INVALID_ARG;
    return launch_reset(st->d, st->state, req_pool_indices_dev, n,
                        static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? HS_OK
               : HS_ERR_CUDA;
}

int hs_get_status(hs_state* st, uint32_t* flags_out, void* stream) {
    if (!st || !flags_out) return HS_ERR_INVALID_ARG;
    if (!on_handle_device(st)) return HS_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t flags = 0;
    if (cudaMemcpyAsync(&flags, st->ws + st->wl.status, 4, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return HS_ERR_CUDA;
    if (cudaMemsetAsync(st->ws + st->wl.status, 0, 4, s) != cudaSuccess) return HS_ERR_CUDA;
    *flags_out = flags;
    return flags ? HS_ERR_DEVICE_STATUS : HS_OK;
}

int hs_get_stats(hs_state* st, int32_t layer_id, int64_t* totals_host, int32_t reset,
                 void* stream) {
    if (!st || !totals_host) return HS_ERR_INVALID_ARG;
    if (!on_handle_device(st)) return HS_ERR_INVALID_ARG;
    if (layer_id < 0 || layer_id >= st->d.layers) return HS_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char* src = st->state + st->sl.totals + (size_t)layer_id * kTotalsWords * 8;
    unsigned long long buf[HS_NUM_STATS];
    if (cudaMemcpyAsync(buf, src, sizeof(buf), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return HS_ERR_CUDA;
    if (reset && cudaMemsetAsync(src, 0, sizeof(buf), s) != cudaSuccess) return HS_ERR_CUDA;
    for (int k = 0; k < HS_NUM_STATS; ++k) totals_host[k] = (int64_t)buf[k];
    return HS_OK;
}

int hs_export_request_state(hs_state* st, int32_t layer_id, int32_t request, int32_t* tok_host,
                            int32_t* ep_host, int32_t* phys_host, int32_t* ctrl_host,
                            int64_t* bank_host, void* stream) {
    if (!st) return HS_ERR_INVALID_ARG;
    if (!on_handle_device(st)) return HS_ERR_INVALID_ARG;
    const Dims& d = st->d;
    if (layer_id < 0 || layer_id >= d.layers || request < 0 || request >= d.R)
        return HS_ERR_INVALID_ARG;
    const LayerView v = layer_view(d, st->state, layer_id, nullptr, nullptr);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long q = request;
    cudaError_t e = cudaSuccess;
    if (tok_host && e == cudaSuccess)
        e = cudaMemcpyAsync(tok_host, v.tok + q * d.H, (size_t)d.H * 4, cudaMemcpyDeviceToHost, s);
    if (ep_host && e == cudaSuccess)
        e = cudaMemcpyAsync(ep_host, v.ep + q * d.H, (size_t)d.H * 4, cudaMemcpyDeviceToHost, s);
    if (phys_host && e == cudaSuccess)
        e = cudaMemcpyAsync(phys_host, v.phys + q * (d.H + d.C), (size_t)(d.H + d.C) * 4,
                            cudaMemcpyDeviceToHost, s);
    if (ctrl_host && e == cudaSuccess)
        e = cudaMemcpyAsync(ctrl_host, v.ctrl + q * kCtrlWords, kCtrlWords * 4,
                            cudaMemcpyDeviceToHost, s);
    std::vector<int16_t> map;
    if (bank_host && e == cudaSuccess) {
        if (d.dense) {
            map.resize((size_t)d.L);
            e = cudaMemcpyAsync(map.data(), v.map + q * d.L, (size_t)d.L * 2,
                                cudaMemcpyDeviceToHost, s);
        } else {
            e = cudaMemcpyAsync(bank_host, v.bank + q * d.hash_size, (size_t)d.hash_size * 8,
                                cudaMemcpyDeviceToHost, s);
        }
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    for (size_t i = 0; i < map.size(); ++i) bank_host[i] = map[i];  // dense map, widened
    return e == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

const char* hs_status_string(int code) {
    switch (code) {
        case HS_OK: return "ok";
        case HS_ERR_INVALID_ARG: return "invalid argument";
        case HS_ERR_UNSUPPORTED: return "unsupported by this build";
        case HS_ERR_CUDA: return "CUDA runtime error";
        case HS_ERR_DEVICE_STATUS: return "device status flags set";
        case HS_ERR_TIMEOUT: return "bounded device wait timed out";
        default: return "unknown status";
    }
}

int32_t hs_version(void) { return 20000; }

}  // extern "C"
