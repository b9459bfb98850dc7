/*
 * mla_verify.h -- C ABI of the MLA tree-verify attention library
 * (libmlaverify.so, sm_103a).
 *
 * The operation. Speculative decoding verifies a whole draft tree in one
 * target-model pass: every draft-tree token of a request attends over that
 * request's full cached prefix plus the tree tokens on its own root path.
 * Sources (page title, section):
 *   [VK] "The Custom sm_120 Verify Kernel: From 0.7 tok/s to 3-6x Decode
 *        Speedup on Blackwell Consumer GPUs"
 *          Part VI   -- verify attention over a page_size-1 (token-granular,
 *                       scattered) KV pool, custom tree mask;
 *          Part VII  -- prefix unmasked, tree block masked; KV-split
 *                       "partial + reduce" design; NSPLIT; 128-bit KV loads;
 *                       CUDA-graph capture safety (static buffers, no host
 *                       sync, no cudaMalloc, caller-provided workspace);
 *          Part IX   -- the key list of a request is its prefix slots
 *                       followed by its draft-token slots (out_cache_loc);
 *                       mask row stride is prefix + q_len.
 *   [CR] "The Capstone Report: When Kernel Engineering Meets Honest
 *        Bottleneck Analysis", section 1 (capture-safe, fixed NSPLIT,
 *        torch-allocated workspace) and section 2 (grid = batch x tokens x
 *        heads x NSPLIT; mask build as a separate step).
 *   [BM] "One Blocking Memcpy Per Verify Step", "The sync, and the bound that
 *        replaced it": size buffers on the host by a provable upper bound,
 *        keep exact lengths on the device.
 *   [IX] "The Indexer Breakthrough: Implementing a Capture-Safe Triton Kernel
 *        for O(actual_seq) Inference", "The Technical Context": fixed grid,
 *        per-block early exit, work proportional to the actual length.
 *
 * Absorbed-latent MLA shapes: every query head and every cached token is a
 * 576-wide bf16 latent row (512 latent + 64 RoPE dims); V is the first 512
 * dims of the cached row; all heads of a request share the same KV rows.
 *
 * Semantics (row n = (b*T + t)*H + h, key j of request b at pool slot
 * kv_indices[kv_indptr[b] + j], j in [0, L_b + T)):
 *   visible(n) = { j < L_b }  U  { L_b + u : u is t or an ancestor of t }
 *   s_j        = softmax_scale * dot(q[n][0:576], K_j[0:576])
 *   lse[n]     = ln sum_{j visible} exp(s_j)            (natural log)
 *   out[n][d]  = sum_{j visible} exp(s_j - lse[n]) * K_j[d],  d < 512
 *
 * Conventions for every entry point:
 *   - All pointers are DEVICE pointers unless stated otherwise. The caller
 *     owns every buffer. The library never allocates, frees or synchronises;
 *     it only launches kernels on `stream`. Every call below except
 *     mla_verify_init is safe inside CUDA stream capture (call
 *     mla_verify_init for the device first).
 *   - The kernels are launched with programmatic dependent launch: each may
 *     start its set-up while the kernel before it on `stream` is still
 *     running, but reads and writes global memory only after that kernel
 *     (and so all earlier work on `stream`) has completed. Stream order is
 *     kept for the caller; nothing is needed on its side.
 *   - Host-checkable arguments (sizes, null/alignment, finite scale) are
 *     checked before any launch and give a negative mla_status_t.
 *   - Device data is never read on the host. Bad device data never traps:
 *     it sets bits in a device status word (MLA_STATUS_*) and the affected
 *     keys/nodes are handled as documented. The word is sticky (bits are
 *     only ever OR'd in); the caller reads it whenever it synchronises and
 *     clears it with mla_verify_reset_status.
 */
#ifndef MLA_VERIFY_H
#define MLA_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = -1,         /* bad size, null or misaligned pointer, bad scale */
    MLA_ERR_UNSUPPORTED = -2,         /* device is not sm_103 / shape outside limits */
    MLA_ERR_WORKSPACE_TOO_SMALL = -3, /* workspace_bytes < mla_verify_workspace_bytes(...) */
    MLA_ERR_CUDA = -4,                /* a CUDA runtime call or launch failed */
    MLA_ERR_NOT_INITIALIZED = -5      /* called inside stream capture before mla_verify_init */
} mla_status_t;

/* Limits checked on the host. T <= 64 because tree visibility is a 64-bit
 * ancestor mask per tree token. */
#define MLA_MAX_TREE 64
#define MLA_MAX_NSPLIT 128
#define MLA_MAX_HEADS 128
#define MLA_D_QK 576
#define MLA_D_V 512

/* Device status bits (OR'd into an int32 word on the device). */
#define MLA_STATUS_BAD_SLOT 0x1    /* kv_indices entry outside [0, pool_slots): that key is
                                      masked out and its row is never read */
#define MLA_STATUS_BAD_PARENT 0x2  /* tree_parent[b][0] != -1 or tree_parent[b][i] outside
                                      [0, i): that node is treated as a root */
#define MLA_STATUS_BAD_INDPTR 0x4  /* kv_indptr[b+1] - kv_indptr[b] != prefix_lens[b] + T:
                                      missing keys are masked, surplus keys ignored */
#define MLA_STATUS_CAPACITY 0x8    /* builder: list longer than kv_indices_capacity; the
                                      list is truncated at the capacity */
#define MLA_STATUS_BAD_PREFIX 0x10 /* builder: prefix_lens[b] outside [0, stride] or
                                      req_pool_indices[b] outside [0, rows): clamped */
#define MLA_STATUS_EMPTY_ROW 0x20  /* a query row had no valid visible key: out row = 0,
                                      lse = -inf */
#define MLA_STATUS_TIMEOUT 0x40    /* a bounded wait inside a kernel gave up (never expected);
                                      that call's outputs are invalid */

/* Human-readable name of an mla_status_t (static string, never NULL). */
const char *mla_verify_status_string(int status);

/* Library version, e.g. 100 for 1.0.0. */
int mla_verify_version(void);

/* One-time per-device set-up: checks the device is sm_103, sets kernel
 * attributes (dynamic shared memory), caches the resident cluster counts,
 * and looks up the allocation-free entry point's scratch area (see
 * mla_verify_attention_noalloc; the device reserves its 32 MiB here). Call
 * it once per device, with that device current, OUTSIDE stream capture. The
 * other calls run it lazily on first use when not capturing.
 * Returns MLA_OK, MLA_ERR_UNSUPPORTED or MLA_ERR_CUDA. */
int mla_verify_init(int device);

/* Bytes of workspace mla_verify_attention needs for this shape (a host-side
 * upper bound, [BM]): a 256-byte header holding the status word, then the
 * per-split partial results. 0 if the shape is outside the limits. */
size_t mla_verify_workspace_bytes(int batch, int T, int num_heads, int nsplit);

/* Byte offset of the int32 device status word inside the workspace. */
size_t mla_verify_status_offset(void);

/* Clears the status word at `status` (device int32) on `stream`
 * (a memset node when captured). */
int mla_verify_reset_status(int32_t *status, cudaStream_t stream);

/*
 * Index + mask builder ([VK] Part IX; [CR] section 2). One launch:
 *   kv_indptr[0] = 0, kv_indptr[b+1] = kv_indptr[b] + prefix_lens[b] + T
 *   kv_indices[kv_indptr[b] + j] = req_to_token[req_pool_indices[b]][j]   (j < L_b)
 *   kv_indices[kv_indptr[b] + L_b + u] = out_cache_loc[b*T + u]           (u < T)
 *   anc_mask[b*T + t] = bit set of t and its ancestors in tree b
 * Arguments:
 *   req_to_token      int32 [req_to_token_rows][req_to_token_stride], row-major
 *   req_pool_indices  int32 [batch]   table row of request b
 *   prefix_lens       int32 [batch]   L_b (cached prefix length)
 *   out_cache_loc     int32 [batch*T] pool slots of the draft-tree tokens
 *   tree_parent       int32 [batch][T]; parent[b][0] = -1, parent[b][i] in [0, i)
 *   kv_indices_capacity  host upper bound on sum_b (L_b + T), e.g.
 *                     batch * (req_to_token_stride + T) ([BM])
 *   kv_indptr         int32 [batch+1]  (out)
 *   kv_indices        int32 [kv_indices_capacity] (out)
 *   anc_mask          uint64 [batch*T] (out; may be NULL to skip)
 *   status            int32 device word, bits OR'd in (may point into a workspace)
 * Bit-exact and deterministic. Errors: MLA_ERR_INVALID_ARG for null pointers,
 * batch < 1, T outside [1, 64], non-positive stride/rows/capacity. */
int mla_build_verify_meta(const int32_t *req_to_token, int64_t req_to_token_stride,
                          int64_t req_to_token_rows, const int32_t *req_pool_indices,
                          const int32_t *prefix_lens, const int32_t *out_cache_loc,
                          const int32_t *tree_parent, int batch, int T,
                          int64_t kv_indices_capacity, int32_t *kv_indptr, int32_t *kv_indices,
                          uint64_t *anc_mask, int32_t *status, cudaStream_t stream);

/*
 * Tree-verify attention = split-KV partial kernel + log-sum-exp combine
 * ([VK] Part VII; [CR] sections 1-2). Two launches on `stream`.
 *   q            bf16 [batch*T][num_heads][576], contiguous, 16-byte aligned
 *   kv_pool      bf16 [pool_slots][576], one row per slot (page_size 1),
 *                16-byte aligned
 *   kv_indices   int32, the combined key list (see mla_build_verify_meta)
 *   kv_indptr    int32 [batch+1]
 *   prefix_lens  int32 [batch]
 *   tree_parent  int32 [batch][T] (visibility is built in-kernel from it)
 *   T            tree tokens per request, 1..64
 *   nsplit       KV partitions per request, 1..128: request b's L_b + T keys
 *                are cut into at most nsplit contiguous ranges (the pages cut
 *                ceil((L_b+T)/nsplit)-key chunks; the kernels balance the
 *                ranges over the SMs, mostly at 256-key tiles, and may use
 *                fewer ranges, depending on the launch); each range gives
 *                one partial result per query row and empty ranges give
 *                lse = -inf ([VK] Part VII: NSPLIT multiplies the number of
 *                partials)
 *   workspace    device buffer of >= mla_verify_workspace_bytes(batch, T,
 *                num_heads, nsplit) bytes, 256-byte aligned; holds the status
 *                word and the partials; contents need no initialisation
 *   out          bf16 [batch*T][num_heads][512] (out), round-to-nearest-even
 *   lse          fp32 [batch*T][num_heads] (out), natural log of the scaled
 *                partition sum
 *   softmax_scale finite, > 0 (e.g. 1/sqrt(192))
 * Returns MLA_OK or a negative mla_status_t (nothing launched on error). */
int mla_verify_attention(const void *q, const void *kv_pool, const int32_t *kv_indices,
                         const int32_t *kv_indptr, const int32_t *prefix_lens,
                         const int32_t *tree_parent, int T, int nsplit, void *workspace,
                         void *out, float *lse, int batch, int num_heads, int64_t pool_slots,
                         float softmax_scale, size_t workspace_bytes, cudaStream_t stream);

/* Same as mla_verify_attention, but tree visibility is read from a mask that
 * mla_build_verify_meta prebuilt (anc_mask uint64 [batch*T]) instead of being
 * rebuilt from tree_parent. Both forms give bit-identical results. */
int mla_verify_attention_anc(const void *q, const void *kv_pool, const int32_t *kv_indices,
                             const int32_t *kv_indptr, const int32_t *prefix_lens,
                             const uint64_t *anc_mask, int T, int nsplit, void *workspace,
                             void *out, float *lse, int batch, int num_heads,
                             int64_t pool_slots, float softmax_scale, size_t workspace_bytes,
                             cudaStream_t stream);

/* The same verify attention with the index build fused into the gathers:
 * the partial kernels read each key's pool slot straight from the page
 * table (mla_build_verify_meta's inputs) instead of from a prebuilt combined
 * list, and build the tree's visibility in-kernel from tree_parent, so a
 * call is two launches (partial, combine) with no kv_indptr / kv_indices /
 * anc_mask buffers ([VK] Part IX: combined indices = prefix slots ++
 * out_cache_loc; [CR] section 2: the build is memory-trivial).
 *   req_to_token      int32 [req_to_token_rows][req_to_token_stride], the
 *                     request-to-slot table; stride in [1, 2^31 - 65]
 *   req_pool_indices  int32 [batch]  table row of request b
 *   prefix_lens       int32 [batch]  L_b; keys 0..L_b-1 are the row's first
 *                     L_b entries, keys L_b..L_b+T-1 are out_cache_loc[b*T..]
 *   out_cache_loc     int32 [batch*T] pool slots of the draft-tree tokens
 * Everything else is as in mla_verify_attention (the default kernels, the
 * same workspace). A row index outside the table or L_b outside [0,
 * stride] is clamped as the builder clamps it and flagged with
 * MLA_STATUS_BAD_PREFIX in the workspace status word (that request's
 * keys are then its draft keys, resp. its whole row). On valid inputs the
 * results are bit-identical to mla_build_verify_meta +
 * mla_verify_attention. */
int mla_verify_attention_paged(const void *q, const void *kv_pool, const int32_t *req_to_token,
                               int64_t req_to_token_stride, int64_t req_to_token_rows,
                               const int32_t *req_pool_indices, const int32_t *prefix_lens,
                               const int32_t *out_cache_loc, const int32_t *tree_parent, int T,
                               int nsplit, void *workspace, void *out, float *lse, int batch,
                               int num_heads, int64_t pool_slots, float softmax_scale,
                               size_t workspace_bytes, cudaStream_t stream);

/* The partial half of mla_verify_attention_paged (the split partials into
 * the workspace, as mla_verify_partial writes them with flags 0);
 * mla_verify_combine finishes the call. */
int mla_verify_partial_paged(const void *q, const void *kv_pool, const int32_t *req_to_token,
                             int64_t req_to_token_stride, int64_t req_to_token_rows,
                             const int32_t *req_pool_indices, const int32_t *prefix_lens,
                             const int32_t *out_cache_loc, const int32_t *tree_parent, int T,
                             int nsplit, void *workspace, int batch, int num_heads,
                             int64_t pool_slots, float softmax_scale, size_t workspace_bytes,
                             cudaStream_t stream);

/*
 * The two halves of mla_verify_attention, for callers that schedule them
 * separately (e.g. to merge partials gathered from elsewhere).
 *
 * mla_verify_partial writes, for every query row n and split s:
 *   lse_part[n*nsplit + s]          fp32, natural-log partition sum of the
 *                                   split's visible keys (-inf if none)
 *   o_part[(n*nsplit + s)*512 + d]  fp32, that split's softmax-weighted V
 *                                   (normalised within the split); where
 *                                   lse_part is -inf its contents are
 *                                   unspecified (not read by the combine)
 * at workspace + 256 (lse_part, padded to 256 bytes) and right after it
 * (o_part). Exactly one of tree_parent / anc_mask must be non-NULL.
 * flags: 0 = default kernel (for requests with more than 128 rows T*H, four
 * SMs per 256-row block with 2-SM MMAs; otherwise two SMs per 128-row
 * block); MLA_PARTIAL_PAIR forces the two-SM kernel, MLA_PARTIAL_QUAD the
 * four-SM one (rows past T*H are padding). Both give results within the
 * documented tolerance of each other. Any other bit, or both bits, is
 * MLA_ERR_INVALID_ARG.
 *
 * mla_verify_combine merges them ([VK] Part VII "reduce"):
 *   lse[n] = ln sum_s exp(lse_part[n,s]);  out[n] = sum_s exp(lse_part[n,s] - lse[n]) o_part[n,s]
 * rounded to bf16 (nearest even); splits with lse_part = -inf get weight 0.
 */
#define MLA_PARTIAL_PAIR 0x4u
#define MLA_PARTIAL_QUAD 0x8u
int mla_verify_partial(const void *q, const void *kv_pool, const int32_t *kv_indices,
                       const int32_t *kv_indptr, const int32_t *prefix_lens,
                       const int32_t *tree_parent, const uint64_t *anc_mask, int T, int nsplit,
                       void *workspace, int batch, int num_heads, int64_t pool_slots,
                       float softmax_scale, size_t workspace_bytes, unsigned flags,
                       cudaStream_t stream);

int mla_verify_combine(const void *workspace, int batch, int T, int num_heads, int nsplit,
                       void *out, float *lse, size_t workspace_bytes, cudaStream_t stream);

/*
 * Allocation-free verify call. The pages have no counterpart to this entry
 * point; it exists for callers that cannot allocate device memory where
 * they run the verify step (for example a plugin enqueue callback inside an
 * inference runtime that owns all device memory, or code running while the
 * application's allocator is locked), and so cannot provide the workspace
 * that mla_verify_attention needs.
 *
 * Same inputs, outputs and results as mla_verify_attention (the same
 * kernels, bit for bit), but the per-split partials live in one fixed
 * scratch area in device global memory, mla_verify_noalloc_scratch_bytes()
 * bytes (32 MiB), that a device holds from its set-up to process exit.
 *   - Shapes whose mla_verify_workspace_bytes(batch, T, num_heads, nsplit)
 *     exceeds that size are rejected with MLA_ERR_WORKSPACE_TOO_SMALL before
 *     anything is launched: at most 16,351 partials (batch * T * num_heads *
 *     nsplit), e.g. 128 query rows with 127 splits.
 *   - Nothing is allocated: no cudaMalloc/cudaFree, no allocating library
 *     call. All host-side checks run first; then the call enqueues a 4-byte
 *     memset (clearing the area's status word), the two kernels, and, if
 *     `status` is not NULL, a 4-byte device-to-device copy of this call's
 *     status bits into *status (overwriting it; NULL discards them).
 *   - The area's device address is looked up (cudaGetSymbolAddress) by the
 *     library's per-device set-up, mla_verify_init, which is also when the
 *     device reserves the area. If mla_verify_init has not run on the
 *     current device, the first call runs it; make that first call outside
 *     stream capture (inside capture it returns MLA_ERR_NOT_INITIALIZED).
 *   - All calls share the one area and it keeps the previous call's
 *     contents: calls whose GPU work overlaps on the same device (other
 *     streams, other host threads) race on it and must be serialised by the
 *     caller.
 */
size_t mla_verify_noalloc_scratch_bytes(void);

int mla_verify_attention_noalloc(const void *q, const void *kv_pool, const int32_t *kv_indices,
                                 const int32_t *kv_indptr, const int32_t *prefix_lens,
                                 const int32_t *tree_parent, int T, int nsplit, void *out,
                                 float *lse, int batch, int num_heads, int64_t pool_slots,
                                 float softmax_scale, int32_t *status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_VERIFY_H */
