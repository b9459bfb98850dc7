/*
 * CPU oracle for the steps beside the verify attention: greedy tree
 * acceptance, KV relocation into contiguous slots, and the fp8 paged MQA
 * indexer logits. Plain loops, fp64 where arithmetic is involved.
 *
 * TEST INFRASTRUCTURE: built and called only by the tests, the smoke check
 * and the benchmark's CPU leg; the CUDA library never links or runs it, and
 * the two share no code.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- tree acceptance
 * "The Custom sm_120 Verify Kernel..." reports the speculative drafter's
 * commit length (Part II: avg_commit_len; Part III: commit-length probe) and
 * "One Blocking Memcpy Per Verify Step" says the accept computation and the
 * state commit have data-dependent shapes that need fixed-shape
 * reformulations for graph capture. The pages give no algorithm; the
 * plainest reading is greedy verification along the tree: starting at the
 * root (node 0, the last committed token), repeatedly move to the child
 * whose draft token equals the target's argmax at the current node (the
 * lowest-numbered such child when siblings repeat a token); stop when no
 * child matches. The target's argmax at the final node is the bonus token.
 *
 * Per request b (row-major [B][T] inputs):
 *   commit_len[b]                     = accepted drafts + 1 (the bonus token)
 *   accepted_nodes[b][0 .. n-1]       = accepted tree nodes in path order, then -1
 *   kept_slots[b][0 .. n]             = KV slots to keep: the root's, then the
 *                                       accepted nodes', then -1
 *   next_tokens[b][0 .. n]            = accepted draft tokens, then the bonus,
 *                                       then -1
 * Returns 0, or -2 if a parent array is not a tree rooted at node 0 with
 * parent[i] in [0, i).
 */
int oracle_tree_accept(const int32_t *tree_parent, const int32_t *draft_tokens,
                       const int32_t *target_argmax, const int32_t *out_cache_loc, int B, int T,
                       int32_t *commit_len, int32_t *accepted_nodes, int32_t *kept_slots,
                       int32_t *next_tokens) {
    if (B < 0 || T < 1) return -1;
    for (int b = 0; b < B; ++b) {
        const int32_t *par = tree_parent + (int64_t)b * T;
        const int32_t *tok = draft_tokens + (int64_t)b * T;
        const int32_t *tgt = target_argmax + (int64_t)b * T;
        const int32_t *loc = out_cache_loc + (int64_t)b * T;
        if (par[0] != -1) return -2;
        for (int i = 1; i < T; ++i)
            if (par[i] < 0 || par[i] >= i) return -2;
        int32_t *an = accepted_nodes + (int64_t)b * T;
        int32_t *ks = kept_slots + (int64_t)b * T;
        int32_t *nt = next_tokens + (int64_t)b * T;
        for (int i = 0; i < T; ++i) an[i] = ks[i] = nt[i] = -1;
        int cur = 0, n = 0;
        ks[0] = loc[0];
        for (;;) {
            int nxt = -1;
            for (int c = 1; c < T; ++c) {
                if (par[c] == cur && tok[c] == tgt[cur]) {
                    nxt = c;
                    break;
                }
            }
            if (nxt < 0) break;
            an[n] = nxt;
            nt[n] = tok[nxt];
            ++n;
            ks[n] = loc[nxt];
            cur = nxt;
        }
        nt[n] = tgt[cur];
        commit_len[b] = n + 1;
    }
    return 0;
}

/* ---------------------------------------------------------------- KV relocation
 * "The Custom sm_120 Verify Kernel..." Part VIII and "The Capstone Report"
 * (Defrag): Tier 1 defragmentation is live relocation of a request's
 * scattered KV slots into contiguous ones under a copy budget, rewriting the
 * request's req_to_token row. The pages defer it without giving details; the
 * plainest reading: request b's prefix rows j = 0 .. L_b-1 move to the
 * caller-allocated contiguous range dst_start[b] + j; one call moves at most
 * `budget` rows per request, continuing from progress[b] (rows already
 * moved), copying each 576-value row and rewriting req_to_token[rpi[b]][j].
 *
 * The destination slots must be free: disjoint from every source slot of
 * the batch still to be moved and from each other (else -5). Returns 0, -1
 * for bad arguments or -3 for an out-of-range slot.
 */
int oracle_kv_relocate(uint16_t *kv_pool, int64_t pool_slots, int32_t *req_to_token,
                       int64_t stride, const int32_t *req_pool_indices,
                       const int32_t *prefix_lens, const int32_t *dst_start, int32_t *progress,
                       int B, int budget) {
    if (B < 0 || budget < 0 || pool_slots < 1 || stride < 1) return -1;
    /* destination / source disjointness over the rows this call moves */
    unsigned char *mark = (unsigned char *)calloc((size_t)pool_slots, 1);
    if (!mark) return -4;
    int rc = 0;
    for (int b = 0; b < B && rc == 0; ++b) {
        const int32_t L = prefix_lens[b], j0 = progress[b];
        if (L < 0 || j0 < 0 || j0 > L) { rc = -1; break; }
        const int32_t n = (L - j0 < budget) ? L - j0 : budget;
        const int32_t *row = req_to_token + (int64_t)req_pool_indices[b] * stride;
        for (int32_t j = j0; j < L; ++j) {       /* every source still to be moved */
            const int32_t s = row[j];
            if (s < 0 || (int64_t)s >= pool_slots) { rc = -3; break; }
            mark[s] |= 1;
        }
        for (int32_t j = 0; j < j0 && rc == 0; ++j) {  /* rows already moved are live */
            const int64_t d = (int64_t)dst_start[b] + j;
            if (d < 0 || d >= pool_slots) { rc = -3; break; }
            mark[d] |= 1;
        }
        for (int32_t j = j0; j < j0 + n && rc == 0; ++j) {
            const int64_t d = (int64_t)dst_start[b] + j;
            if (d < 0 || d >= pool_slots) { rc = -3; break; }
            if (mark[d] & 2) rc = -5;             /* two rows aimed at one slot */
            mark[d] |= 2;
        }
    }
    if (rc == 0) {
        for (int b = 0; b < B && rc == 0; ++b) {
            const int32_t L = prefix_lens[b], j0 = progress[b];
            const int32_t n = (L - j0 < budget) ? L - j0 : budget;
            const int32_t *row = req_to_token + (int64_t)req_pool_indices[b] * stride;
            for (int32_t j = j0; j < j0 + n; ++j) {
                const int64_t d = (int64_t)dst_start[b] + j;
                if ((mark[d] & 1) && row[j] != (int32_t)d) { rc = -5; break; }  /* live source */
            }
        }
    }
    free(mark);
    if (rc != 0) return rc;
    for (int b = 0; b < B; ++b) {
        const int32_t L = prefix_lens[b], j0 = progress[b];
        const int32_t n = (L - j0 < budget) ? L - j0 : budget;
        int32_t *row = req_to_token + (int64_t)req_pool_indices[b] * stride;
        for (int32_t j = j0; j < j0 + n; ++j) {
            const int64_t s = row[j], d = (int64_t)dst_start[b] + j;
            if (s != d) memcpy(kv_pool + d * 576, kv_pool + s * 576, 576 * sizeof(uint16_t));
            row[j] = (int32_t)d;
        }
        progress[b] = j0 + n;
    }
    return 0;
}

/* ---------------------------------------------------------------- fp8 paged MQA indexer
 * "The Indexer Breakthrough..." (The Technical Context; Design Decisions):
 * the DSA indexer scores every cached position of a request: a batched
 * product of the queries with the cached keys, ReLU, weighting by per-head
 * weights, a sum over heads, and a per-position scale. KV cache blocks are
 * 8448 bytes: 64 positions x 128 fp8 (e4m3) values, then 64 fp32 scales.
 * Queries are raw fp8 converted without scaling. Positions past the
 * request's length get -inf (the fixed grid's fast path).
 *
 *   logits[b][p*64 + i] = s * sum_h w[b][h] * max(0, sum_d q[b][h][d] k[d])
 * where k and s are row i and scale i of block block_table[b][p], for
 * p*64 + i < seq_len[b]; else -inf. (The scale is applied after the head
 * sum; as scales are positive, the order does not change the value.)
 */
static double e4m3_to_double(uint8_t v) {
    const int s = v >> 7, e = (v >> 3) & 15, m = v & 7;
    double x;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        x = ldexp((double)m / 8.0, -6);
    else
        x = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -x : x;
}

int oracle_fp8_indexer_logits(const uint8_t *q, const float *weights, const uint8_t *kv_blocks,
                              int64_t nblocks, const int32_t *block_table, const int32_t *seq_lens,
                              int B, int H, int max_pages, double *logits) {
    if (B < 0 || H < 1 || max_pages < 0 || nblocks < 0) return -1;
    for (int b = 0; b < B; ++b) {
        const int32_t len = seq_lens[b];
        for (int p = 0; p < max_pages; ++p) {
            const int32_t blk = block_table[(int64_t)b * max_pages + p];
            for (int i = 0; i < 64; ++i) {
                const int64_t pos = (int64_t)p * 64 + i;
                double *o = logits + (int64_t)b * max_pages * 64 + pos;
                if (pos >= len) {
                    *o = -INFINITY;
                    continue;
                }
                if (blk < 0 || blk >= nblocks) return -3;
                const uint8_t *base = kv_blocks + blk * (int64_t)8448;
                float sf;
                memcpy(&sf, base + 8192 + 4 * i, 4);
                double acc = 0.0;
                for (int h = 0; h < H; ++h) {
                    const uint8_t *qh = q + ((int64_t)b * H + h) * 128;
                    double dot = 0.0;
                    for (int d = 0; d < 128; ++d)
                        dot += e4m3_to_double(qh[d]) * e4m3_to_double(base[i * 128 + d]);
                    acc += (double)weights[(int64_t)b * H + h] * (dot > 0.0 ? dot : 0.0);
                }
                *o = (double)sf * acc;
            }
        }
    }
    return 0;
}

/* Exposed for the tests' check of the fp8 decoding against its definition. */
double oracle_e4m3_value(int v) { return e4m3_to_double((uint8_t)v); }
