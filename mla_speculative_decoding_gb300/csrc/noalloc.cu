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
// declared at file scope, capped at a modest 32 MiB because every GPU that
// loads this part of the library holds it until the process exits. The
// workspace of a shape is 256 + round_up(4 p, 256) + 2048 p bytes for
// p = batch * T * num_heads * nsplit partials, so the area takes at most
// p = 16,351 partials: 128 query rows x 127 splits fit, 128 x 128 do not.
//
// Host code cannot use the array's name as a device address (on the host it
// names a shadow object), so the library's per-device set-up
// (mla_verify_init, with that device current) looks up the real address
// with cudaGetSymbolAddress and caches it; the look-up also loads this
// file's module, which is when the device reserves the area. The first
// noalloc call on a device runs that set-up if it has not run yet, so that
// first call must happen outside stream capture. All calls share the one
// area: calls whose GPU work overlaps (different streams, or different host
// threads, on the same device) race on it.
#include <mutex>

#include "common.cuh"

#define MLA_NOALLOC_SCRATCH_BYTES (32u << 20)

static __device__ __align__(256) unsigned char g_mla_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDev = 64;
void* g_scratch_addr[kMaxDev];
std::mutex g_scratch_mutex;

// Cached device address of the scratch area on `dev`, or nullptr before the
// set-up has run there.
void* scratch_of(int dev) {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    return g_scratch_addr[dev];
}

}  // namespace

namespace mlav {

// Per-device set-up, called by mla_verify_init with `device` current.
cudaError_t setup_noalloc(int device) {
    if (device < 0 || device >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[device] != nullptr) return cudaSuccess;
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_mla_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_addr[device] = p;
    return cudaSuccess;
}

}  // namespace mlav

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
    // Every host-side check runs before anything is queued. A stand-in
    // pointer with the area's alignment takes the workspace's place in them.
    const void* ws_probe = reinterpret_cast<const void*>(uintptr_t{256});
    int rc = mlav::check_attention_args(q, kv_pool, kv_indices, kv_indptr, prefix_lens, tree_parent,
                                        T, nsplit, ws_probe, out, lse, batch, num_heads, pool_slots,
                                        softmax_scale, need);
    if (rc != MLA_OK) return rc;
    rc = mlav::ensure_device_ready(stream);  // the set-up (and the scratch look-up) if not yet run
    if (rc != MLA_OK) return rc;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return MLA_ERR_CUDA;
    void* ws = scratch_of(dev);
    if (ws == nullptr) return MLA_ERR_CUDA;
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
