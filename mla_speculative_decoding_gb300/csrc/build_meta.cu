// Index + tree-mask builder for the verify call.
//
// Builds, on the device and in one launch, what the page "The Custom sm_120
// Verify Kernel: From 0.7 tok/s to 3-6x Decode Speedup on Blackwell Consumer
// GPUs" (Part IX, bug 2 and its fix) says the verify kernel consumes: the
// per-request key list = prefix slots (from req_to_token) followed by the
// draft-token slots (out_cache_loc), its offsets, and the tree visibility
// mask -- here a 64-bit ancestor-or-self set per tree token. The pages'
// reference did this on the host (tree-build 1.8 ms, mask-build 0.18 ms;
// "The Capstone Report", section 2); here it is a capture-safe kernel.
//
// Grid: (batch, blocks per request sized from the host bound on the list
// length). Each block recomputes its request's list
// offset from prefix_lens (an integer block reduction over earlier
// requests), so there is no inter-block communication and no atomics other
// than the error word. Bit-exact and deterministic.
#include "common.cuh"

namespace mlav {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxBlocksPerReq = 256;

__device__ __forceinline__ int32_t clamp_prefix(const int32_t* prefix_lens,
                                                const int32_t* req_pool_indices, int b,
                                                int64_t stride, int64_t rows, int* bad) {
    int32_t L = prefix_lens[b];
    const int32_t r = req_pool_indices[b];
    if (r < 0 || r >= rows) {
        *bad |= MLA_STATUS_BAD_PREFIX;
        return 0;
    }
    if (L < 0) {
        *bad |= MLA_STATUS_BAD_PREFIX;
        L = 0;
    } else if (L > stride) {
        *bad |= MLA_STATUS_BAD_PREFIX;
        L = (int32_t)stride;
    }
    return L;
}

__global__ void __launch_bounds__(kThreads)
build_meta_kernel(const int32_t* __restrict__ req_to_token, int64_t stride, int64_t rows,
                  const int32_t* __restrict__ req_pool_indices,
                  const int32_t* __restrict__ prefix_lens,
                  const int32_t* __restrict__ out_cache_loc,
                  const int32_t* __restrict__ tree_parent, int batch, int T, int64_t capacity,
                  int32_t* __restrict__ kv_indptr, int32_t* __restrict__ kv_indices,
                  uint64_t* __restrict__ anc, int32_t* status) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    const int b = blockIdx.x;
    __shared__ int64_t s_base;
    __shared__ int32_t s_L;
    __shared__ int64_t s_warp[kThreads / 32];
    __shared__ uint64_t s_anc[MLA_MAX_TREE];
    __shared__ int s_ptr[MLA_MAX_TREE];
    // Offset of this request's list: sum over earlier requests of (L_c + T),
    // with the same clamping those requests' own blocks apply (their errors
    // are reported by those blocks). Integer sum: exact in any order.
    {
        int ignored = 0;
        int64_t part = 0;
        for (int c = threadIdx.x; c < b; c += kThreads)
            part += (int64_t)clamp_prefix(prefix_lens, req_pool_indices, c, stride, rows,
                                          &ignored) + T;
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = part;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int64_t base = 0;
        for (int w = 0; w < kThreads / 32; ++w) base += s_warp[w];
        int bad = 0;
        const int32_t L = clamp_prefix(prefix_lens, req_pool_indices, b, stride, rows, &bad);
        s_base = base;
        s_L = L;
        if (blockIdx.y == 0) {
            const int64_t end = base + L + T;
            if (end > capacity) bad |= MLA_STATUS_CAPACITY;
            kv_indptr[b + 1] = (int32_t)min(end, capacity);
            if (b == 0) kv_indptr[0] = 0;
            status_or(status, bad);
        }
    }
    __syncthreads();
    const int64_t base = s_base;
    const int32_t L = s_L;
    const int64_t K = (int64_t)L + T;
    const int32_t* row = req_to_token + (L > 0 ? (int64_t)req_pool_indices[b] * stride : 0);
    const int32_t* tree_slots = out_cache_loc + (int64_t)b * T;
    for (int64_t j = (int64_t)blockIdx.y * kThreads + threadIdx.x; j < K;
         j += (int64_t)gridDim.y * kThreads) {
        const int64_t dst = base + j;
        if (dst >= capacity) break;
        kv_indices[dst] = (j < L) ? row[j] : tree_slots[j - L];
    }
    // The tree's ancestor-or-self sets, by the first warp of the request's
    // first block once its share of the list is written.
    if (anc != nullptr && blockIdx.y == 0 && threadIdx.x < 32) {
        const int bad = build_anc_warp(tree_parent + (int64_t)b * T, T, s_anc, s_ptr);
        for (int t = threadIdx.x; t < T; t += 32) anc[(int64_t)b * T + t] = s_anc[t];
        if (threadIdx.x == 0) status_or(status, bad);
    }
}

}  // namespace

cudaError_t launch_build_meta(const int32_t* req_to_token, int64_t stride, int64_t rows,
                              const int32_t* req_pool_indices, const int32_t* prefix_lens,
                              const int32_t* out_cache_loc, const int32_t* tree_parent,
                              int batch, int T, int64_t capacity, int32_t* kv_indptr,
                              int32_t* kv_indices, uint64_t* anc, int32_t* status,
                              cudaStream_t stream) {
    // Blocks per request from host-side bounds only (no device reads): enough
    // that each thread copies about two entries of the longest possible list.
    const int64_t per_req = stride + T;
    const int64_t want = (per_req + 2 * kThreads - 1) / (2 * kThreads);
    const int by = (int)(want < 1 ? 1 : (want > kMaxBlocksPerReq ? kMaxBlocksPerReq : want));
    dim3 grid(batch, by);
    return launch_pdl(build_meta_kernel, grid, dim3(kThreads), 0, stream, req_to_token, stride, rows,
                      req_pool_indices, prefix_lens, out_cache_loc, tree_parent, batch, T, capacity,
                      kv_indptr, kv_indices, anc, status);
}

}  // namespace mlav
