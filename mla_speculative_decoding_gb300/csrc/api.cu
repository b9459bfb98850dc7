// C ABI entry points (declared in include/mla_verify.h): host-side argument
// checks, per-device set-up, and the launch sequence of each call.
//
// Capture safety follows the page "The Custom sm_120 Verify Kernel..."
// (Part VII, "Making the Kernel CUDA Graph Capture-Safe"): no host-device
// synchronisation, no allocation, static caller-owned buffers, and a fixed
// split count, so every entry point but mla_verify_init can be recorded in a
// CUDA graph. Device data is never read back on the host; sizes come from
// host-side upper bounds ("One Blocking Memcpy Per Verify Step", "The sync,
// and the bound that replaced it").
#include <math.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "mla_decode_steps.h"
#include "partial_kernels.cuh"

namespace mlav {
namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_ready[kMaxDevices];
int g_sm_count[kMaxDevices];
std::mutex g_init_mutex;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int init_device(int device) {
    if (device < 0 || device >= kMaxDevices) return MLA_ERR_INVALID_ARG;
    if (g_ready[device].load(std::memory_order_acquire)) return MLA_OK;
    std::lock_guard<std::mutex> lock(g_init_mutex);
    if (g_ready[device].load(std::memory_order_acquire)) return MLA_OK;
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return MLA_ERR_CUDA;
    if (prev != device && cudaSetDevice(device) != cudaSuccess) return MLA_ERR_CUDA;
    int rc = MLA_OK;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        rc = MLA_ERR_CUDA;
    } else if (major != 10 || minor != 3) {
        rc = MLA_ERR_UNSUPPORTED;  // the library carries sm_103a code only
    } else if (setup_partial_pair() != cudaSuccess || setup_partial_quad() != cudaSuccess ||
               setup_fp8_indexer() != cudaSuccess || setup_noalloc(device) != cudaSuccess) {
        rc = MLA_ERR_CUDA;
    }
    if (rc == MLA_OK) {
        g_sm_count[device] = sms;
        g_ready[device].store(1, std::memory_order_release);
    }
    if (prev != device) cudaSetDevice(prev);
    return rc;
}

// Lazy set-up on the current device; refused inside stream capture.
int ensure_ready(cudaStream_t stream, int* sm_count) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
    if (!g_ready[dev].load(std::memory_order_acquire)) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return MLA_ERR_CUDA;
        if (cs != cudaStreamCaptureStatusNone) return MLA_ERR_NOT_INITIALIZED;
        const int rc = init_device(dev);
        if (rc != MLA_OK) return rc;
    }
    if (sm_count) *sm_count = g_sm_count[dev];
    return MLA_OK;
}

bool shape_ok(int batch, int T, int num_heads, int nsplit) {
    if (batch < 1 || batch > 65535) return false;
    if (T < 1 || T > MLA_MAX_TREE) return false;
    if (num_heads < 1 || num_heads > MLA_MAX_HEADS) return false;
    if (nsplit < 1 || nsplit > MLA_MAX_NSPLIT) return false;
    // Row ids and partial ids are kept in 32-bit grids / 64-bit offsets.
    const int64_t rows = (int64_t)batch * T * num_heads;
    return rows <= (int64_t)INT32_MAX / MLA_MAX_NSPLIT;
}

int check_partial_args(const void* q, const void* kv_pool, const int32_t* kv_indices,
                       const int32_t* kv_indptr, const int32_t* prefix_lens,
                       const int32_t* tree_parent, const uint64_t* anc_mask, int T, int nsplit,
                       const void* workspace, int batch, int num_heads, int64_t pool_slots,
                       float softmax_scale, size_t workspace_bytes) {
    if (!q || !kv_pool || !kv_indices || !kv_indptr || !prefix_lens || !workspace)
        return MLA_ERR_INVALID_ARG;
    if ((tree_parent == nullptr) == (anc_mask == nullptr)) return MLA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(kv_pool, 16) || !aligned(workspace, 256))
        return MLA_ERR_INVALID_ARG;
    if (anc_mask && !aligned(anc_mask, 8)) return MLA_ERR_INVALID_ARG;
    if (!shape_ok(batch, T, num_heads, nsplit)) return MLA_ERR_INVALID_ARG;
    if (pool_slots < 1 || pool_slots > (int64_t)INT32_MAX + 1) return MLA_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return MLA_ERR_INVALID_ARG;
    if (workspace_bytes < ws_layout(batch, T, num_heads, nsplit).total)
        return MLA_ERR_WORKSPACE_TOO_SMALL;
    return MLA_OK;
}

int check_combine_args(const void* workspace, int batch, int T, int num_heads, int nsplit,
                       const void* out, const float* lse, size_t workspace_bytes) {
    if (!workspace || !out || !lse) return MLA_ERR_INVALID_ARG;
    if (!aligned(workspace, 256) || !aligned(out, 16) || !aligned(lse, 4))
        return MLA_ERR_INVALID_ARG;
    if (!shape_ok(batch, T, num_heads, nsplit)) return MLA_ERR_INVALID_ARG;
    if (workspace_bytes < ws_layout(batch, T, num_heads, nsplit).total)
        return MLA_ERR_WORKSPACE_TOO_SMALL;
    return MLA_OK;
}

PartialArgs make_partial_args(const void* q, const void* kv_pool, const int32_t* kv_indices,
                              const int32_t* kv_indptr, const int32_t* prefix_lens,
                              const int32_t* tree_parent, const uint64_t* anc_mask, int T,
                              int nsplit, void* workspace, int batch, int num_heads,
                              int64_t pool_slots, float softmax_scale) {
    const WsLayout w = ws_layout(batch, T, num_heads, nsplit);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    PartialArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.kv = static_cast<const __nv_bfloat16*>(kv_pool);
    a.kv_indices = kv_indices;
    a.kv_indptr = kv_indptr;
    a.prefix_lens = prefix_lens;
    a.tree_parent = tree_parent;
    a.anc_mask = anc_mask;
    a.lse_part = reinterpret_cast<float*>(ws + w.lse_off);
    a.o_part = reinterpret_cast<float*>(ws + w.o_off);
    a.status = reinterpret_cast<int32_t*>(ws);
    a.batch = batch;
    a.T = T;
    a.H = num_heads;
    a.nsplit = nsplit;
    a.pool_slots = pool_slots;
    a.scale_log2 = softmax_scale * kLog2e;
    a.wave_full = 0x7fffffff;  // no wave shaping unless a launcher sets it
    a.parts = 0;
    a.req_to_token = nullptr;  // the combined-list form
    a.r2t_stride = a.r2t_rows = 0;
    a.req_pool_indices = nullptr;
    a.out_cache_loc = nullptr;
    return a;
}

int run_partial(const PartialArgs& a, unsigned flags, cudaStream_t stream) {
    cudaError_t e;
    if ((flags & MLA_PARTIAL_PAIR) || (!(flags & MLA_PARTIAL_QUAD) && a.T * a.H <= 128))
        e = launch_partial_pair(a, stream);
    else
        e = launch_partial_quad(a, stream);
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int run_combine(const void* workspace, int batch, int T, int num_heads, int nsplit, void* out,
                float* lse, cudaStream_t stream) {
    const WsLayout w = ws_layout(batch, T, num_heads, nsplit);
    const unsigned char* ws = static_cast<const unsigned char*>(workspace);
    const cudaError_t e = launch_combine(
        reinterpret_cast<const float*>(ws + w.lse_off), reinterpret_cast<const float*>(ws + w.o_off),
        batch * T * num_heads, nsplit,
        T * num_heads <= 128 ? pair_expected_parts(batch, T, num_heads, nsplit)
                             : quad_expected_parts(batch, T, num_heads, nsplit),
        static_cast<__nv_bfloat16*>(out), lse,
        const_cast<int32_t*>(reinterpret_cast<const int32_t*>(ws)), stream);
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int attention_impl(const void* q, const void* kv_pool, const int32_t* kv_indices,
                   const int32_t* kv_indptr, const int32_t* prefix_lens,
                   const int32_t* tree_parent, const uint64_t* anc_mask, int T, int nsplit,
                   void* workspace, void* out, float* lse, int batch, int num_heads,
                   int64_t pool_slots, float softmax_scale, size_t workspace_bytes,
                   cudaStream_t stream) {
    int rc = check_partial_args(q, kv_pool, kv_indices, kv_indptr, prefix_lens, tree_parent,
                                anc_mask, T, nsplit, workspace, batch, num_heads, pool_slots,
                                softmax_scale, workspace_bytes);
    if (rc != MLA_OK) return rc;
    rc = check_combine_args(workspace, batch, T, num_heads, nsplit, out, lse, workspace_bytes);
    if (rc != MLA_OK) return rc;
    rc = ensure_ready(stream, nullptr);
    if (rc != MLA_OK) return rc;
    const PartialArgs a =
        make_partial_args(q, kv_pool, kv_indices, kv_indptr, prefix_lens, tree_parent, anc_mask,
                          T, nsplit, workspace, batch, num_heads, pool_slots, softmax_scale);
    rc = run_partial(a, 0u, stream);
    if (rc != MLA_OK) return rc;
    return run_combine(workspace, batch, T, num_heads, nsplit, out, lse, stream);
}

}  // namespace

int check_attention_args(const void* q, const void* kv_pool, const int32_t* kv_indices,
                         const int32_t* kv_indptr, const int32_t* prefix_lens,
                         const int32_t* tree_parent, int T, int nsplit, const void* workspace,
                         const void* out, const float* lse, int batch, int num_heads,
                         int64_t pool_slots, float softmax_scale, size_t workspace_bytes) {
    if (!tree_parent) return MLA_ERR_INVALID_ARG;
    const int rc = check_partial_args(q, kv_pool, kv_indices, kv_indptr, prefix_lens, tree_parent,
                                      nullptr, T, nsplit, workspace, batch, num_heads, pool_slots,
                                      softmax_scale, workspace_bytes);
    if (rc != MLA_OK) return rc;
    return check_combine_args(workspace, batch, T, num_heads, nsplit, out, lse, workspace_bytes);
}

int ensure_device_ready(cudaStream_t stream) { return ensure_ready(stream, nullptr); }

}  // namespace mlav

using namespace mlav;

MLAV_API const char* mla_verify_status_string(int status) {
    switch (status) {
        case MLA_OK: return "MLA_OK";
        case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
        case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
        case MLA_ERR_WORKSPACE_TOO_SMALL: return "MLA_ERR_WORKSPACE_TOO_SMALL";
        case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
        case MLA_ERR_NOT_INITIALIZED: return "MLA_ERR_NOT_INITIALIZED";
        default: return "MLA_ERR_UNKNOWN";
    }
}

MLAV_API int mla_verify_version(void) { return 100; }

MLAV_API int mla_verify_init(int device) { return init_device(device); }

MLAV_API size_t mla_verify_workspace_bytes(int batch, int T, int num_heads, int nsplit) {
    if (!shape_ok(batch, T, num_heads, nsplit)) return 0;
    return ws_layout(batch, T, num_heads, nsplit).total;
}

MLAV_API size_t mla_verify_status_offset(void) { return 0; }

MLAV_API int mla_verify_reset_status(int32_t* status, cudaStream_t stream) {
    if (!status || !aligned(status, 4)) return MLA_ERR_INVALID_ARG;
    return cudaMemsetAsync(status, 0, sizeof(int32_t), stream) == cudaSuccess ? MLA_OK
                                                                             : MLA_ERR_CUDA;
}

MLAV_API int mla_build_verify_meta(const int32_t* req_to_token, int64_t req_to_token_stride,
                                   int64_t req_to_token_rows, const int32_t* req_pool_indices,
                                   const int32_t* prefix_lens, const int32_t* out_cache_loc,
                                   const int32_t* tree_parent, int batch, int T,
                                   int64_t kv_indices_capacity, int32_t* kv_indptr,
                                   int32_t* kv_indices, uint64_t* anc_mask, int32_t* status,
                                   cudaStream_t stream) {
    if (!req_to_token || !req_pool_indices || !prefix_lens || !out_cache_loc || !tree_parent ||
        !kv_indptr || !kv_indices || !status)
        return MLA_ERR_INVALID_ARG;
    if (batch < 1 || batch > 65535 || T < 1 || T > MLA_MAX_TREE) return MLA_ERR_INVALID_ARG;
    if (req_to_token_stride < 1 || req_to_token_rows < 1) return MLA_ERR_INVALID_ARG;
    if (kv_indices_capacity < 1 || kv_indices_capacity > (int64_t)INT32_MAX)
        return MLA_ERR_INVALID_ARG;
    if (anc_mask && !aligned(anc_mask, 8)) return MLA_ERR_INVALID_ARG;
    const cudaError_t e = launch_build_meta(
        req_to_token, req_to_token_stride, req_to_token_rows, req_pool_indices, prefix_lens,
        out_cache_loc, tree_parent, batch, T, kv_indices_capacity, kv_indptr, kv_indices, anc_mask,
        status, stream);
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

MLAV_API int mla_verify_attention(const void* q, const void* kv_pool, const int32_t* kv_indices,
                                  const int32_t* kv_indptr, const int32_t* prefix_lens,
                                  const int32_t* tree_parent, int T, int nsplit, void* workspace,
                                  void* out, float* lse, int batch, int num_heads,
                                  int64_t pool_slots, float softmax_scale,
                                  size_t workspace_bytes, cudaStream_t stream) {
    if (!tree_parent) return MLA_ERR_INVALID_ARG;
    return attention_impl(q, kv_pool, kv_indices, kv_indptr, prefix_lens, tree_parent, nullptr,
                          T, nsplit, workspace, out, lse, batch, num_heads, pool_slots,
                          softmax_scale, workspace_bytes, stream);
}

MLAV_API int mla_verify_attention_anc(const void* q, const void* kv_pool,
                                      const int32_t* kv_indices, const int32_t* kv_indptr,
                                      const int32_t* prefix_lens, const uint64_t* anc_mask, int T,
                                      int nsplit, void* workspace, void* out, float* lse,
                                      int batch, int num_heads, int64_t pool_slots,
                                      float softmax_scale, size_t workspace_bytes,
                                      cudaStream_t stream) {
    if (!anc_mask) return MLA_ERR_INVALID_ARG;
    return attention_impl(q, kv_pool, kv_indices, kv_indptr, prefix_lens, nullptr, anc_mask, T,
                          nsplit, workspace, out, lse, batch, num_heads, pool_slots,
                          softmax_scale, workspace_bytes, stream);
}

namespace mlav {
namespace {
int paged_partial(const void* q, const void* kv_pool, const int32_t* req_to_token,
                  int64_t req_to_token_stride, int64_t req_to_token_rows,
                  const int32_t* req_pool_indices, const int32_t* prefix_lens,
                  const int32_t* out_cache_loc, const int32_t* tree_parent, int T, int nsplit,
                  void* workspace, int batch, int num_heads, int64_t pool_slots,
                  float softmax_scale, size_t workspace_bytes, cudaStream_t stream) {
    if (!req_to_token || !req_pool_indices || !out_cache_loc || !tree_parent)
        return MLA_ERR_INVALID_ARG;
    if (req_to_token_stride < 1 || req_to_token_stride > (int64_t)INT32_MAX - MLA_MAX_TREE ||
        req_to_token_rows < 1)
        return MLA_ERR_INVALID_ARG;
    // The list-form checks, with the table standing in for the list.
    int rc = check_partial_args(q, kv_pool, req_to_token, req_pool_indices, prefix_lens, tree_parent,
                                nullptr, T, nsplit, workspace, batch, num_heads, pool_slots,
                                softmax_scale, workspace_bytes);
    if (rc != MLA_OK) return rc;
    rc = ensure_ready(stream, nullptr);
    if (rc != MLA_OK) return rc;
    PartialArgs a = make_partial_args(q, kv_pool, nullptr, nullptr, prefix_lens, tree_parent, nullptr,
                                      T, nsplit, workspace, batch, num_heads, pool_slots,
                                      softmax_scale);
    a.req_to_token = req_to_token;
    a.r2t_stride = req_to_token_stride;
    a.r2t_rows = req_to_token_rows;
    a.req_pool_indices = req_pool_indices;
    a.out_cache_loc = out_cache_loc;
    return run_partial(a, 0u, stream);
}
}  // namespace
}  // namespace mlav

MLAV_API int mla_verify_partial_paged(const void* q, const void* kv_pool, const int32_t* req_to_token,
                                      int64_t req_to_token_stride, int64_t req_to_token_rows,
                                      const int32_t* req_pool_indices, const int32_t* prefix_lens,
                                      const int32_t* out_cache_loc, const int32_t* tree_parent,
                                      int T, int nsplit, void* workspace, int batch, int num_heads,
                                      int64_t pool_slots, float softmax_scale,
                                      size_t workspace_bytes, cudaStream_t stream) {
    return paged_partial(q, kv_pool, req_to_token, req_to_token_stride, req_to_token_rows,
                         req_pool_indices, prefix_lens, out_cache_loc, tree_parent, T, nsplit,
                         workspace, batch, num_heads, pool_slots, softmax_scale, workspace_bytes,
                         stream);
}

MLAV_API int mla_verify_attention_paged(const void* q, const void* kv_pool,
                                        const int32_t* req_to_token, int64_t req_to_token_stride,
                                        int64_t req_to_token_rows, const int32_t* req_pool_indices,
                                        const int32_t* prefix_lens, const int32_t* out_cache_loc,
                                        const int32_t* tree_parent, int T, int nsplit,
                                        void* workspace, void* out, float* lse, int batch,
                                        int num_heads, int64_t pool_slots, float softmax_scale,
                                        size_t workspace_bytes, cudaStream_t stream) {
    int rc = check_combine_args(workspace, batch, T, num_heads, nsplit, out, lse, workspace_bytes);
    if (rc != MLA_OK) return rc;
    rc = paged_partial(q, kv_pool, req_to_token, req_to_token_stride, req_to_token_rows,
                       req_pool_indices, prefix_lens, out_cache_loc, tree_parent, T, nsplit,
                       workspace, batch, num_heads, pool_slots, softmax_scale, workspace_bytes,
                       stream);
    if (rc != MLA_OK) return rc;
    return run_combine(workspace, batch, T, num_heads, nsplit, out, lse, stream);
}

MLAV_API int mla_verify_partial(const void* q, const void* kv_pool, const int32_t* kv_indices,
                                const int32_t* kv_indptr, const int32_t* prefix_lens,
                                const int32_t* tree_parent, const uint64_t* anc_mask, int T,
                                int nsplit, void* workspace, int batch, int num_heads,
                                int64_t pool_slots, float softmax_scale, size_t workspace_bytes,
                                unsigned flags, cudaStream_t stream) {
    int rc = check_partial_args(q, kv_pool, kv_indices, kv_indptr, prefix_lens, tree_parent,
                                anc_mask, T, nsplit, workspace, batch, num_heads, pool_slots,
                                softmax_scale, workspace_bytes);
    if (rc != MLA_OK) return rc;
    if ((flags & ~(MLA_PARTIAL_PAIR | MLA_PARTIAL_QUAD)) ||
        (flags & (MLA_PARTIAL_PAIR | MLA_PARTIAL_QUAD)) == (MLA_PARTIAL_PAIR | MLA_PARTIAL_QUAD))
        return MLA_ERR_INVALID_ARG;
    rc = ensure_ready(stream, nullptr);
    if (rc != MLA_OK) return rc;
    const PartialArgs a =
        make_partial_args(q, kv_pool, kv_indices, kv_indptr, prefix_lens, tree_parent, anc_mask,
                          T, nsplit, workspace, batch, num_heads, pool_slots, softmax_scale);
    return run_partial(a, flags, stream);
}

MLAV_API int mla_verify_combine(const void* workspace, int batch, int T, int num_heads,
                                int nsplit, void* out, float* lse, size_t workspace_bytes,
                                cudaStream_t stream) {
    int rc = check_combine_args(workspace, batch, T, num_heads, nsplit, out, lse,
                                workspace_bytes);
    if (rc != MLA_OK) return rc;
    rc = ensure_ready(stream, nullptr);
    if (rc != MLA_OK) return rc;
    return run_combine(workspace, batch, T, num_heads, nsplit, out, lse, stream);
}

// ---------------------------------------------------------------- decode steps
namespace {
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

MLAV_API int mla_tree_accept(const int32_t* tree_parent, const int32_t* draft_tokens,
                             const int32_t* target_argmax, const int32_t* out_cache_loc, int batch,
                             int T, int32_t* commit_len, int32_t* accepted_nodes,
                             int32_t* kept_slots, int32_t* next_tokens, int32_t* status,
                             cudaStream_t stream) {
    if (!tree_parent || !draft_tokens || !target_argmax || !out_cache_loc || !commit_len ||
        !accepted_nodes || !kept_slots || !next_tokens || !status)
        return MLA_ERR_INVALID_ARG;
    if (batch < 1 || batch > 65535 || T < 1 || T > MLA_MAX_TREE) return MLA_ERR_INVALID_ARG;
    int rc = ensure_ready(stream, nullptr);
    if (rc != MLA_OK) return rc;
    return launch_tree_accept(tree_parent, draft_tokens, target_argmax, out_cache_loc, batch, T,
                              commit_len, accepted_nodes, kept_slots, next_tokens, status,
                              stream) == cudaSuccess
               ? MLA_OK
               : MLA_ERR_CUDA;
}

MLAV_API int mla_kv_relocate(void* kv_pool, int64_t pool_slots, int32_t* req_to_token,
                             int64_t req_to_token_stride, const int32_t* req_pool_indices,
                             const int32_t* prefix_lens, const int32_t* dst_start, int32_t* progress,
                             int batch, int budget, int32_t* status, cudaStream_t stream) {
    if (!kv_pool || !req_to_token || !req_pool_indices || !prefix_lens || !dst_start || !progress ||
        !status || !al16(kv_pool))
        return MLA_ERR_INVALID_ARG;
    if (pool_slots < 1 || pool_slots > ((int64_t)1 << 31) || req_to_token_stride < 1 || batch < 1 ||
        batch > 65535 || budget < 1 || budget > (1 << 20))
        return MLA_ERR_INVALID_ARG;
    int rc = ensure_ready(stream, nullptr);
    if (rc != MLA_OK) return rc;
    return launch_kv_relocate(kv_pool, pool_slots, req_to_token, req_to_token_stride,
                              req_pool_indices, prefix_lens, dst_start, progress, batch, budget,
                              status, stream) == cudaSuccess
               ? MLA_OK
               : MLA_ERR_CUDA;
}

MLAV_API int mla_fp8_indexer_logits(const void* q, const float* weights, const void* kv_blocks,
                                    int64_t nblocks, const int32_t* block_table,
                                    const int32_t* seq_lens, int batch, int num_heads,
                                    int max_pages, float* logits, int32_t* status,
                                    cudaStream_t stream) {
    if (!q || !weights || !kv_blocks || !block_table || !seq_lens || !logits || !status ||
        !al16(q) || !al16(kv_blocks) || !al16(logits))
        return MLA_ERR_INVALID_ARG;
    if (batch < 1 || batch > 65535 || num_heads < 1 || num_heads > MLA_MAX_HEADS || max_pages < 0 ||
        max_pages > 65535 || nblocks < 0 || nblocks > 0x7fffffffLL)
        return MLA_ERR_INVALID_ARG;
    if (max_pages == 0) return MLA_OK;
    int sms = 0;
    int rc = ensure_ready(stream, &sms);
    if (rc != MLA_OK) return rc;
    return launch_fp8_indexer(q, weights, kv_blocks, nblocks, block_table, seq_lens, batch,
                              num_heads, max_pages, logits, status, sms, stream) == cudaSuccess
               ? MLA_OK
               : MLA_ERR_CUDA;
}
