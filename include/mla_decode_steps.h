/*
 * Capture-safe decode steps beside the MLA tree-verify attention
 * (libmlaverify.so, sm_103a): greedy acceptance along the draft trees, KV
 * relocation into contiguous slots, and the fp8 paged MQA indexer logits.
 *
 * Conventions (as in mla_verify.h): every pointer is device memory owned by
 * the caller; nothing is allocated, freed or synchronised; work is launched
 * on `stream` only; grids depend on host scalars only (capture-safe; the
 * one-time set-up of mla_verify_init must have run before capture). Host-
 * checkable arguments return a negative MLA_ERR_* code before any launch;
 * bad device data never traps: it sets bits in the caller's device status
 * word (int32, OR of MLA_STATUS_* bits, which the caller resets). Kernels
 * use programmatic dependent launch as in mla_verify.h (stream order kept).
 *
 * Sources: [VK] "The Custom sm_120 Verify Kernel: From 0.7 tok/s to 3-6x
 * Decode Speedup on Blackwell Consumer GPUs"; [CR] "The Capstone Report";
 * [OM] "One Blocking Memcpy Per Verify Step"; [IX] "The Indexer
 * Breakthrough".
 */
#ifndef MLA_DECODE_STEPS_H
#define MLA_DECODE_STEPS_H

#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Greedy acceptance of each request's draft tree after verification
 * ([VK] Parts II-III report the commit length; [OM] asks for fixed-shape,
 * device-side accept and commit). The pages give no algorithm; the reading
 * implemented: from the root (node 0, the last committed token) move to the
 * child whose draft token equals the target model's argmax at the current
 * node, taking the lowest-numbered such child when siblings repeat a token;
 * stop when no child matches; the argmax at the final node is a bonus token.
 *
 * Inputs, int32 [batch][T], T in [1, 64]: tree_parent (parent[0] = -1,
 * parent[i] in [0, i)), draft_tokens, target_argmax, out_cache_loc (node
 * slots). Outputs (fixed shapes, padded with -1):
 *   commit_len     [batch]     accepted drafts + 1
 *   accepted_nodes [batch][T]  accepted nodes in path order
 *   kept_slots     [batch][T]  slots to keep: the root's, then the accepted nodes'
 *   next_tokens    [batch][T]  accepted draft tokens, then the bonus token
 * A parent outside [0, i) makes node i unreachable and sets
 * MLA_STATUS_BAD_PARENT. One warp per request.
 */
int mla_tree_accept(const int32_t *tree_parent, const int32_t *draft_tokens,
                    const int32_t *target_argmax, const int32_t *out_cache_loc, int batch, int T,
                    int32_t *commit_len, int32_t *accepted_nodes, int32_t *kept_slots,
                    int32_t *next_tokens, int32_t *status, cudaStream_t stream);

/*
 * KV relocation ("Tier 1" defragmentation, [VK] Part VIII, [CR] Defrag):
 * moves request b's prefix rows j in [progress[b], progress[b] + n_b), with
 * n_b = min(budget, prefix_lens[b] - progress[b]), from their current slots
 * req_to_token[req_pool_indices[b]][j] to dst_start[b] + j: each 576-value
 * bf16 row (1152 bytes) is copied within kv_pool [pool_slots][576], the
 * table entry is rewritten, and progress[b] advances by n_b (two launches on
 * `stream`; the grid covers `budget` rows per request whatever the device
 * progress, so the call can be captured and replayed until done).
 *
 * Contract: destination slots are free (disjoint from every source slot
 * still to be moved and from each other); rows already in place (source ==
 * destination) are left as they are. An out-of-range source or destination
 * skips that row and sets MLA_STATUS_BAD_SLOT. budget in [1, 2^20].
 */
int mla_kv_relocate(void *kv_pool, int64_t pool_slots, int32_t *req_to_token,
                    int64_t req_to_token_stride, const int32_t *req_pool_indices,
                    const int32_t *prefix_lens, const int32_t *dst_start, int32_t *progress,
                    int batch, int budget, int32_t *status, cudaStream_t stream);

/*
 * fp8 paged MQA indexer logits ([IX] "The Technical Context", "Design
 * Decisions"): for request b and position p*64 + i < seq_lens[b],
 *   logits[b][p*64 + i] = s * sum_h weights[b][h] * max(0, sum_d q[b][h][d] * k[d])
 * where k (128 fp8 e4m3 values) and s (fp32) are row i and scale i of block
 * block_table[b][p] of kv_blocks [nblocks][8448] (64 x 128 fp8 values, then
 * 64 fp32 scales); q is fp8 e4m3 [batch][num_heads][128], weights fp32
 * [batch][num_heads]. Every other position of logits [batch][max_pages*64]
 * is -inf. The dot products run on the tensor cores (fp8 e4m3 operands, fp32
 * accumulation; products of two e4m3 values are exact in fp32) in one
 * persistent launch of one CTA per SM: the 128-position tiles the device
 * lengths call for are split evenly over the CTAs, so work scales with the
 * actual lengths while the grid depends on host sizes only. A block index
 * outside [0, nblocks) gives -inf for that page and sets MLA_STATUS_BAD_SLOT.
 * num_heads in [1, 128]; nblocks in [0, 2^31); q, kv_blocks and logits
 * 16-byte aligned (MLA_ERR_INVALID_ARG otherwise).
 */
int mla_fp8_indexer_logits(const void *q, const float *weights, const void *kv_blocks,
                           int64_t nblocks, const int32_t *block_table, const int32_t *seq_lens,
                           int batch, int num_heads, int max_pages, float *logits, int32_t *status,
                           cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_STEPS_H */
