// Sparse page table kernel and state reset kernel (sm_103a).
//
// Page table ("SGLang HiSparse: 当稀疏注意力从算法变为系统组件", sections 1.2
// and 2.3: the coordinator turns token-level top-k into the list of pages
// that hold selected tokens; in PAGED mode a token is addressed by its page
// and in-page offset).  One CTA per batch row:
//   1. set one bit per page t / page_size of every valid token (shared-memory
//      bitmap of ceil(max_seq_len / page_size) bits);
//   2. exclusive scan of the words' population counts: a page's rank in the
//      ascending page list is its word's prefix plus the set bits below it;
//   3. write the ascending page list (padded with -1) and, per entry,
//      rank * page_size + t % page_size.
//
// Reset: returns (layer, request) states to empty: hash bank unused or dense
// map all -1, epochs and tokens -1, position table the identity, control
// words zero.
#include "hs_internal.cuh"

namespace hs {
namespace {

constexpr int kPtBlock = 512;

__global__ void __launch_bounds__(kPtBlock) page_table_kernel(
    const int32_t* __restrict__ topk, const int32_t* __restrict__ seq_lens, int32_t S, int32_t K,
    int32_t L_max, int32_t page_size, int32_t nwords, int32_t* __restrict__ pages,
    int32_t* __restrict__ num_pages, int32_t* __restrict__ token_page) {
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned* bits = reinterpret_cast<unsigned*>(smem);
    int* pre = reinterpret_cast<int*>(bits + nwords);
    __shared__ int s_tmp[33];

    const int b = blockIdx.x;
    const int tid = threadIdx.x, BD = blockDim.x;
    const int N = S * K;
    const int32_t* t_b = topk + (long long)b * N;
    const int sl = seq_lens[b];
    const int limit = sl < L_max ? sl : L_max;

    for (int w = tid; w < nwords; w += BD) bits[w] = 0u;
    __syncthreads();
    for (int i = tid; i < N; i += BD) {
        const int t = t_b[i];
        if (t >= 0 && t < limit) {
            const int p = t / page_size;
            atomicOr(&bits[p >> 5], 1u << (p & 31));
        }
    }
    __syncthreads();
    const int per = (nwords + BD - 1) / BD;
    const int w0 = tid * per, w1 = min(nwords, w0 + per);
    int c = 0;
    for (int w = w0; w < w1; ++w) c += __popc(bits[w]);
    int total;
    int run = block_exclusive_scan(c, s_tmp, &total);
    int32_t* pages_b = pages + (long long)b * N;
    for (int w = w0; w < w1; ++w) {
        pre[w] = run;
        unsigned x = bits[w];
        while (x) {
            const int k = __ffs(x) - 1;
            pages_b[run++] = w * 32 + k;
            x &= x - 1u;
        }
    }
    if (tid == 0) num_pages[b] = total;
    for (int i = total + tid; i < N; i += BD) pages_b[i] = -1;
    __syncthreads();
    int32_t* tp_b = token_page + (long long)b * N;
    for (int i = tid; i < N; i += BD) {
        const int t = t_b[i];
        int out = -1;
        if (t >= 0 && t < limit) {
            const int p = t / page_size;
            const int rank = pre[p >> 5] + __popc(bits[p >> 5] & ((1u << (p & 31)) - 1u));
            out = rank * page_size + (t - p * page_size);
        }
        tp_b[i] = out;
    }
}

__global__ void reset_kernel(const Dims d, uint8_t* state, StateLayout sl,
                             const int32_t* __restrict__ rpi, int32_t n) {
    // blockIdx.x: request list index; blockIdx.y: layer
    const int i = blockIdx.x, layer = blockIdx.y;
    const int q = rpi ? rpi[i] : i;
    if (q < 0 || q >= d.R) return;
    const long long lq = (long long)layer * d.R + q;
    long long* bank = reinterpret_cast<long long*>(state + sl.bank) + lq * d.hash_size;
    int32_t* ep = reinterpret_cast<int32_t*>(state + sl.ep) + lq * d.H;
    int32_t* tok = reinterpret_cast<int32_t*>(state + sl.tok) + lq * d.H;
    int32_t* phys = reinterpret_cast<int32_t*>(state + sl.phys) + lq * (d.H + d.C);
    int32_t* ctrl = reinterpret_cast<int32_t*>(state + sl.ctrl) + lq * kCtrlWords;
    for (int p = threadIdx.x; p < d.hash_size; p += blockDim.x) bank[p] = kEmpty;
    if (d.dense) {
        int16_t* map = reinterpret_cast<int16_t*>(state + sl.map) + lq * d.L;
        for (int p = threadIdx.x; p < d.L; p += blockDim.x) map[p] = -1;
    }
    for (int v = threadIdx.x; v < d.H; v += blockDim.x) {
        ep[v] = -1;
        tok[v] = -1;
    }
    for (int p = threadIdx.x; p < d.H + d.C; p += blockDim.x) phys[p] = p;
    if (threadIdx.x < kCtrlWords) ctrl[threadIdx.x] = 0;
}

}  // namespace

cudaError_t launch_page_table(const int32_t* topk, const int32_t* seq_lens, int32_t B, int32_t S,
                              int32_t K, int32_t L_max, int32_t page_size, int32_t* pages,
                              int32_t* num_pages, int32_t* token_page, cudaStream_t s) {
    const long long npages = ((long long)L_max + page_size - 1) / page_size;
    const int nwords = (int)((npages + 31) / 32);
    const size_t smem = (size_t)nwords * 8;
    static SmemOptIn opt_in;
    cudaError_t e = ensure_smem(page_table_kernel, smem, &opt_in);
    if (e != cudaSuccess) return e;
    page_table_kernel<<<B, kPtBlock, smem, s>>>(topk, seq_lens, S, K, L_max, page_size, nwords,
                                                 pages, num_pages, token_page);
    return cudaGetLastError();
}

cudaError_t launch_reset(const Dims& d, uint8_t* state, const int32_t* rpi, int32_t n,
                         cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    reset_kernel<<<dim3(n, d.layers), 256, 0, s>>>(d, state, state_layout(d), rpi, n);
    return cudaGetLastError();
}

}  // namespace hs
