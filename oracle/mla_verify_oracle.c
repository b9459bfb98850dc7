/*
 * CPU fp64 oracle for MLA tree-verify attention.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference leg load this library. The product
 * path (the CUDA library) never calls it and shares no code with it.
 *
 * What it computes, from the page "The Custom sm_120 Verify Kernel: From
 * 0.7 tok/s to 3-6x Decode Speedup on Blackwell Consumer GPUs":
 *   - Part VI: the target model verifies all draft-tree tokens in one pass;
 *     the KV cache has page_size 1, so every key is a scattered pool slot.
 *   - Part VII: the prefix needs no mask; only the tree block is masked.
 *   - Part IX (bug 2 and its fix): each request's key list is its prefix
 *     slots followed by the slots of its draft tokens (out_cache_loc), and a
 *     draft token's visibility row covers prefix + q_len keys.
 *   - absorbed-latent MLA: q and every latent KV row are 576 wide
 *     (512 latent + 64 RoPE dims); V is the first 512 dims of the row.
 *
 * Definition written out (row n = (b*T + t)*H + h):
 *   keys      K_j = kv_pool[kv_indices[kv_indptr[b] + j]],  j in [0, L_b + T)
 *   anc*(t)   = {t, parent(t), parent(parent(t)), ...} up to the root
 *   visible   V(n) = {0..L_b-1}  U  {L_b + u : u in anc*(t)}
 *   s_j       = scale * sum_{d<576} q[n][d] * K_j[d]          (j in V(n))
 *   m         = max_j s_j,   Z = sum_j exp(s_j - m)
 *   lse[n]    = m + ln Z                          (natural log, scaled scores)
 *   out[n][d] = sum_j exp(s_j - m) * K_j[d] / Z    (d < 512)
 * Two plain passes over the visible keys: no online softmax, no splits, no
 * tiling. Readings where the pages are silent (self-visibility, the LSE
 * convention, the root) are the ones listed in the design notes.
 *
 * The combined index list and the ancestor sets are also produced here
 * (oracle_build_meta) with plain loops; the ancestor set is found by
 * walking parent links, not by a recurrence over earlier nodes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define D_QK 576
#define D_V 512

/* Error codes (negative); 0 = success. */
#define ORC_OK 0
#define ORC_BAD_ARG -1
#define ORC_BAD_TREE -2
#define ORC_BAD_INDEX -3
#define ORC_NO_MEM -4

static double bf16_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* A tree is valid when parent[0] = -1 and 0 <= parent[i] < i for i > 0. */
static int tree_valid(const int32_t *par, int T)
{
    if (T <= 0 || par[0] != -1) return 0;
    for (int i = 1; i < T; ++i)
        if (par[i] < 0 || par[i] >= i) return 0;
    return 1;
}

/* Ancestor-or-self set of node t as a bit set (T <= 64), by walking parents. */
static uint64_t ancestor_set(const int32_t *par, int t)
{
    uint64_t s = 0;
    for (int v = t; v != -1; v = par[v]) s |= (uint64_t)1 << v;
    return s;
}

int oracle_build_meta(const int32_t *req_to_token, int64_t req_to_token_stride,
                      const int32_t *req_pool_indices, const int32_t *prefix_lens,
                      const int32_t *out_cache_loc, const int32_t *tree_parent, int batch, int T,
                      int32_t *kv_indptr, int32_t *kv_indices, uint64_t *anc)
{
    if (batch < 0 || T < 1 || T > 64) return ORC_BAD_ARG;
    kv_indptr[0] = 0;
    for (int b = 0; b < batch; ++b) {
        if (prefix_lens[b] < 0 || prefix_lens[b] > req_to_token_stride) return ORC_BAD_ARG;
        kv_indptr[b + 1] = kv_indptr[b] + prefix_lens[b] + T;
    }
    for (int b = 0; b < batch; ++b) {
        const int32_t *row = req_to_token + (int64_t)req_pool_indices[b] * req_to_token_stride;
        int32_t *dst = kv_indices + kv_indptr[b];
        for (int j = 0; j < prefix_lens[b]; ++j) dst[j] = row[j];
        for (int u = 0; u < T; ++u) dst[prefix_lens[b] + u] = out_cache_loc[(int64_t)b * T + u];
        const int32_t *par = tree_parent + (int64_t)b * T;
        if (!tree_valid(par, T)) return ORC_BAD_TREE;
        for (int t = 0; t < T; ++t) anc[(int64_t)b * T + t] = ancestor_set(par, t);
    }
    return ORC_OK;
}

/* One query row: two passes over its visible keys. */
static int one_row(const uint16_t *q, const uint16_t *kv_pool, int64_t pool_slots,
                   const int32_t *kv_indices, const int32_t *kv_indptr, const int32_t *prefix_lens,
                   const int32_t *tree_parent, int T, int H, double scale, int64_t n,
                   double *s_buf, int32_t *key_buf, double *out_row, double *lse_out)
{
    const int h = (int)(n % H);
    const int64_t bt = n / H;
    const int b = (int)(bt / T);
    const int t = (int)(bt % T);
    (void)h;
    const int32_t Lb = prefix_lens[b];
    const int64_t base = kv_indptr[b];
    if (kv_indptr[b + 1] - base != (int64_t)Lb + T) return ORC_BAD_INDEX;
    const int32_t *par = tree_parent + (int64_t)b * T;
    if (!tree_valid(par, T)) return ORC_BAD_TREE;

    /* Visible key positions, in logical order: the whole prefix, then the
     * tree keys of t's ancestors-or-self. */
    int64_t nvis = 0;
    for (int32_t j = 0; j < Lb; ++j) key_buf[nvis++] = j;
    const uint64_t a = ancestor_set(par, t);
    for (int u = 0; u < T; ++u)
        if ((a >> u) & 1) key_buf[nvis++] = Lb + u;

    double qd[D_QK];
    const uint16_t *qrow = q + n * D_QK;
    for (int d = 0; d < D_QK; ++d) qd[d] = bf16_to_double(qrow[d]);

    /* Pass 1: scaled scores and their maximum. */
    double m = -INFINITY;
    for (int64_t i = 0; i < nvis; ++i) {
        const int32_t slot = kv_indices[base + key_buf[i]];
        if (slot < 0 || slot >= pool_slots) return ORC_BAD_INDEX;
        const uint16_t *k = kv_pool + (int64_t)slot * D_QK;
        double acc = 0.0;
        for (int d = 0; d < D_QK; ++d) acc += qd[d] * bf16_to_double(k[d]);
        s_buf[i] = scale * acc;
        if (s_buf[i] > m) m = s_buf[i];
    }

    /* Pass 2: normaliser and the weighted sum of the V rows. */
    double Z = 0.0;
    for (int d = 0; d < D_V; ++d) out_row[d] = 0.0;
    for (int64_t i = 0; i < nvis; ++i) {
        const int32_t slot = kv_indices[base + key_buf[i]];
        const uint16_t *k = kv_pool + (int64_t)slot * D_QK;
        const double w = exp(s_buf[i] - m);
        Z += w;
        for (int d = 0; d < D_V; ++d) out_row[d] += w * bf16_to_double(k[d]);
    }
    for (int d = 0; d < D_V; ++d) out_row[d] /= Z;
    *lse_out = m + log(Z);
    return ORC_OK;
}

int oracle_verify_attention(const uint16_t *q, const uint16_t *kv_pool, int64_t pool_slots,
                            const int32_t *kv_indices, const int32_t *kv_indptr,
                            const int32_t *prefix_lens, const int32_t *tree_parent, int batch,
                            int T, int num_heads, double scale, const int64_t *rows, int64_t nrows,
                            double *out, double *lse, int nthreads)
{
    if (batch < 1 || T < 1 || T > 64 || num_heads < 1 || !(scale > 0.0)) return ORC_BAD_ARG;
    int64_t max_keys = 0;
    for (int b = 0; b < batch; ++b) {
        if (prefix_lens[b] < 0) return ORC_BAD_ARG;
        if ((int64_t)prefix_lens[b] + T > max_keys) max_keys = (int64_t)prefix_lens[b] + T;
    }
    const int64_t total_rows = (int64_t)batch * T * num_heads;
    for (int64_t i = 0; i < nrows; ++i)
        if (rows && (rows[i] < 0 || rows[i] >= total_rows)) return ORC_BAD_ARG;

    int status = ORC_OK;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double *s_buf = (double *)malloc((size_t)max_keys * sizeof(double));
        int32_t *key_buf = (int32_t *)malloc((size_t)max_keys * sizeof(int32_t));
        if (!s_buf || !key_buf) {
#pragma omp atomic write
            status = ORC_NO_MEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < nrows; ++i) {
                const int64_t n = rows ? rows[i] : i;
                int rc = one_row(q, kv_pool, pool_slots, kv_indices, kv_indptr, prefix_lens,
                                 tree_parent, T, num_heads, scale, n, s_buf, key_buf,
                                 out + i * D_V, lse + i);
                if (rc != ORC_OK) {
#pragma omp atomic write
                    status = rc;
                }
            }
        }
        free(s_buf);
        free(key_buf);
    }
    return status;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
