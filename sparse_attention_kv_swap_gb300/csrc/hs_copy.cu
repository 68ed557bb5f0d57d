// Planned copy of the decode KV swap-in (sm_103a): replays a recorded miss
// plan, i.e. copies host pool row miss_src[b, j] to device row
// miss_dst[b, j] for j < miss_count[b] (the miss-plan protocol of the
// multi-step swap report "[HiSparse] Support hisparse multi-step swap io
// kernel", sections 实现拆解 item 2 and 风险与影响, which lets the row copies
// run apart from the lookup, e.g. on another stream while the next layer
// resolves).  The rows of all batch rows are flattened and split evenly over
// the grid: 16-byte vectors, consecutive threads on consecutive 16-byte
// pieces of a row, all of a thread's loads issued before its stores.
#include "hs_internal.cuh"

namespace hs {
namespace {

constexpr int kBlock = 512;
constexpr int kCopyUnroll = 6;

// A recorded miss plan (host row, device row, count per batch row).
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
__device__ void copy_rows(const RecordedRows& plan, int B, int W, const uint8_t* pool, uint8_t* kv,
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

// Replays a recorded miss plan (the deferred copy of a swap-in call).
__global__ void __launch_bounds__(kBlock, 2) planned_copy_kernel(const RecordedRows plan, int B,
                                                                  int W, const uint8_t* pool,
                                                                  uint8_t* kv) {
    extern __shared__ __align__(16) unsigned char smem[];
    copy_rows(plan, B, W, pool, kv, blockIdx.x, gridDim.x, reinterpret_cast<int*>(smem));
}

}  // namespace

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
