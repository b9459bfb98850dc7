// Allocation-free variant of the verify call.
//
// Some callers cannot obtain device memory at the point where they run the
// verify step: for example a plugin's enqueue callback inside an inference
// runtime that owns and pre-partitions all device memory, or code that runs
// while the application's allocator is locked or being torn down. They can
// still hand over their inputs and outputs, but not the workspace that
// mla_verify_attention needs for its per-split partial results.
//
// For them this file keeps one fixed scratch area in device global memory,
// declared at file scope. Every GPU that loads the library reserves it (for
// the lifetime of the process), so its size is capped at a modest 32 MiB:
// enough for rows * nsplit up to about 16k partials (e.g. 128 query rows x 128
// splits, or 256 rows x 64 splits).
//
// Host code cannot use the array's name as a device address (on the host it
// names a shadow object), so the first call on each device looks up the
// real address with cudaGetSymbolAddress, with that device current, and
// caches it. That first call must therefore happen outside stream capture.
// All calls share the one area: calls whose GPU work overlaps (different
// streams, or different host threads, on the same device) race on it.
#include <mutex>

#include "common.cuh"

#define MLA_NOALLOC_SCRATCH_BYTES (32u << 20)

static __device__ __align__(256) unsigned char g_mla_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDev = 64;
void* g_scratch_addr[kMaxDev];
std::mutex g_scratch_mutex;

// Device address of the scratch area on the current device (set-up on first
// use; refused during stream capture). Returns an mla_status_t.
int scratch_address(cudaStream_t stream, void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return MLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return MLA_ERR_CUDA;
        if (cs != cudaStreamCaptureStatusNone) return MLA_ERR_NOT_INITIALIZED;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_mla_noalloc_scratch) != cudaSuccess || p == nullptr)
            return MLA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MLA_OK;
}

}  // namespace

MLAV_API size_t mla_verify_noalloc_scratch_bytes(void) { return MLA_NOALLOC_SCRATCH_BYTES; }

MLAV_API int mla_verify_attention_noalloc(const void* q, const void* kv_pool,
                                          const int32_t* kv_indices, const int32_t* kv_indptr,
                                          const int32_t* prefix_lens, const int32_t* tree_parent,
                                          int T, int nsplit, void* out, float* lse, int batch,
                                          int num_heads, int64_t pool_slots, float softmax_scale,
                                          int32_t* status, cudaStream_t stream) {
    const size_t need = mla_verify_workspace_bytes(batch, T, num_heads, nsplit);
    if (need == 0) return MLA_ERR_INVALID_ARG;
    if (need > MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE_TOO_SMALL;
    if (status != nullptr && (reinterpret_cast<uintptr_t>(status) & 3u) != 0)
        return MLA_ERR_INVALID_ARG;
    void* ws = nullptr;
    int rc = scratch_address(stream, &ws);
    if (rc != MLA_OK) return rc;
    // The status word lives in the shared area and keeps the previous call's
    // bits: clear it so this call reports only its own.
    int32_t* ws_status = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(ws) +
                                                    mla_verify_status_offset());
    if (cudaMemsetAsync(ws_status, 0, sizeof(int32_t), stream) != cudaSuccess) return MLA_ERR_CUDA;
    rc = mla_verify_attention(q, kv_pool, kv_indices, kv_indptr, prefix_lens, tree_parent, T,
                              nsplit, ws, out, lse, batch, num_heads, pool_slots, softmax_scale,
                              need, stream);
    if (rc != MLA_OK) return rc;
    if (status != nullptr &&
        cudaMemcpyAsync(status, ws_status, sizeof(int32_t), cudaMemcpyDeviceToDevice, stream) !=
            cudaSuccess)
        return MLA_ERR_CUDA;
    return MLA_OK;
}
