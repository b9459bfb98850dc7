// Split-KV partial attention on tcgen05 tensor cores, two SMs per work item.
//
// The verify attention of "The Custom sm_120 Verify Kernel..." (Parts VI,
// VII, IX): every tree-token x head row of a request attends over the
// request's scattered latent KV rows (prefix unmasked, tree block masked),
// in a KV-split "partial + reduce" design.
//
// Work item = (128-row block of the request's T*H rows, split s, request b),
// run by a cluster of two CTAs on two SMs. TMEM holds 512 fp32 columns per
// SM; an accumulator for all 512 V dims of 128 rows fills one SM's TMEM, so
// the scores and the output live on different SMs:
//
//   S-CTA (rank 0): S = Q K^T for 256-key tiles (one N = 256 MMA per 16 dims,
//     36 per tile). TMEM: Q's 512 latent dims [0, 256) as the A operand, S
//     [256, 512). Q's 64 RoPE dims are an A operand in shared memory. K is
//     streamed in 64-dim blocks of 256 keys (32 KB, 6-stage ring), gathered
//     from the scattered rows by six warps of 16-byte cp.async copies
//     (eight lanes per 128-byte row segment; measured faster than TMA gather4
//     for this pattern). Eight softmax warps (two per
//     TMEM lane quarter, one per 128-key half) copy S out of TMEM at once
//     (freeing it for the next tile's MMAs), mask it (tree mask only past the
//     prefix), exchange the per-row tile maximum, keep a lazily updated
//     reference maximum (rescaling only when the tile maximum exceeds it by
//     2^8), and store P as bf16 straight into the O-CTA's shared memory
//     (distributed shared memory), with the per-row rescale factor.
//   O-CTA (rank 1): O += P V with TMEM O = [0, 512) (two N = 256 accumulator
//     chains, one per half of the V dims). V rows are gathered by ten
//     warps of cp.async copies in 32-key stages (32 KB, 4-stage ring). Four
//     correction warps apply the rare
//     rescales to O between tiles and, at the end, normalise O and write the
//     partial (o, lse).
//
// In both CTAs warp 0 only stages the tiles' pool rows (from the key list or
// the page table), up to four tiles ahead of the copy warps, so that the
// slot look-ups are off the copies' path.
//
// A partly filled tile (a partition's last) costs in proportion to its keys:
// only their rows are gathered, the score MMAs use N = the keys rounded up
// to 16, the V stages and P V steps stop at the last 16-key step, and a
// softmax half or 64-key block without keys is skipped. The launcher picks
// the partitions: when every (request, row block) pair of the launch can
// have a cluster of one wave, min(nsplit, resident clusters / pairs) per
// pair, all launched at once (split_range_one_wave); otherwise all nsplit,
// with the wave-shaped split over several waves.
//
// 16 warps: the producer and MMA warpgroups give registers to the softmax
// warpgroups (setmaxnreg). Every wait is bounded; on a timeout a CTA drains
// its MMAs, frees TMEM, reaches the final cluster barrier and flags
// MLA_STATUS_TIMEOUT.
#include "partial_kernels.cuh"
#include "tc_ptx.cuh"

namespace mlav {
namespace {

using namespace tc;

constexpr int kM = 128;
constexpr int kNT = 256;          // keys per tile
constexpr int kThreads = 512;     // 16 warps = 4 warpgroups
constexpr int kWarpMMA = 4;
constexpr int kSProd = 6;         // S-side copy warps: 1-3, 5-7 (warp 0 stages the rows)
constexpr int kOProd = 10;        // O-side copy warps: 1-3, 5-7, 12-15 (warp 0 stages the rows)
constexpr int kRowsRing = 4;      // tiles of pool rows staged ahead of the copies
// Register budget: launched at 128 per thread (512 x 128 = 65,536). S-CTA:
// warpgroups 0-1 drop to 64, the two softmax warpgroups rise to 192
// (256 x 64 + 256 x 192 = 65,536). O-CTA: warpgroups 0, 1, 3 drop to 64.
constexpr int kRegsLow = 64, kRegsSoftmax = 192;
constexpr int kKStages = 6;
constexpr uint32_t kKBlock = kNT * 128;        // 256 keys x 64 dims (bf16)
constexpr int kMetaRing = 4;
constexpr int kVKeys = 32;
constexpr int kVStages = 4;
constexpr uint32_t kVBlock = kVKeys * 128;     // 32 keys x 64 dims
constexpr uint32_t kVStage = 8 * kVBlock;      // 32 keys x 512 dims
constexpr int kOTileStride = 36;               // floats per row of the epilogue's write tile
static_assert(4 * 32 * kOTileStride * 4 <= kVStages * kVStage, "epilogue tiles fit in the V ring");
constexpr uint32_t kPBlock = kM * 128;         // 128 rows x 64 keys (bf16)
constexpr uint32_t kColQ = 0, kColS = 256;     // S-CTA TMEM map
constexpr float kRescaleLog2 = 8.0f;

struct SmemS {
    unsigned char q_rope[kM * 128];            // [128 rows x 64 dims], 128B-swizzled
    unsigned char kring[kKStages][kKBlock];    // [256 keys x 64 dims] per stage
    uint32_t valid[kMetaRing][kNT / 32];
    int32_t rows[kRowsRing][kNT];              // pool rows of the tiles being gathered
    float mx[2][2][kM];
    uint64_t anc[MLA_MAX_TREE];
    int32_t par[MLA_MAX_TREE];
    uint64_t k_full[kKStages], k_empty[kKStages];
    uint64_t meta_full[kMetaRing], meta_free[kMetaRing];
    uint64_t s_full, s_free, q_ready, mx_bar[2];
    uint64_t rows_full[kRowsRing], rows_free[kRowsRing];
};
struct SmemO {
    unsigned char p[4 * kPBlock];              // [128 rows x 256 keys], 4 swizzled 64-key blocks
    unsigned char vring[kVStages][kVStage];    // [32 keys x 512 dims] per stage
    int32_t rows[kRowsRing][kNT];
    float alpha[kM];
    float fin_m[kM];
    float fin_l[2][kM];
    uint64_t v_full[kVStages], v_empty[kVStages];
    uint64_t o_gate, o_prog;
    uint64_t rows_full[kRowsRing], rows_free[kRowsRing];
};
// The header sits at the same offset in both CTAs: the S-CTA arrives on the
// O-CTA's p_full / fin and the O-CTA on the S-CTA's p_free.
struct Header {
    uint64_t p_full, p_free, fin, drain;
    uint32_t tmem_base;
    int abort_flag;
    int no_abort;
};
struct __align__(1024) SmemPair {
    union {
        SmemS s;
        SmemO o;
    } u;
    Header h;
};

constexpr size_t kSmemBytes = sizeof(SmemPair) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ uint32_t ba(const uint64_t& b) { return smem_u32(&b); }

// Keys of tile i of the partition [kb, ke) (a prefix of the tile; >= 1 for
// i < the partition's tile count).
__device__ __forceinline__ int tile_keys(int kb, int ke, int i) { return min(kNT, ke - kb - i * kNT); }
// V stages (32 keys each) holding keys of that tile: the V producers and the
// P V issuer both walk exactly these.
__device__ __forceinline__ int tile_vstages(int kb, int ke, int i) { return (tile_keys(kb, ke, i) + 31) >> 5; }

__device__ __forceinline__ bool warp_wait(const uint64_t& bar, uint32_t parity,
                                          volatile int* abort) {
    const bool ok = mbar_wait(ba(bar), parity, abort);
    return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ bool warp_wait_cluster(const uint64_t& bar, uint32_t parity,
                                                  volatile int* abort) {
    const bool ok = mbar_wait_cluster(ba(bar), parity, abort);
    return __all_sync(0xffffffffu, ok);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
partial_pair_kernel(const PartialArgs a) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    extern __shared__ __align__(1024) unsigned char raw[];
    unsigned char* base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
    SmemPair& sm = *reinterpret_cast<SmemPair*>(base);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const int rb = blockIdx.x >> 1;
    // partition-major dispatch: every request's first partitions launch first
    const int b = blockIdx.y, s = blockIdx.z;
    const int T = a.T, H = a.H, rows_req = T * H;

    int Lb, K;
    int bad = request_keys(a, b, Lb, K);
    int kb, ke;
    const int nrb_req = (a.T * a.H + kM - 1) / kM;
    if (a.parts > 0)  // one wave; partitions past a.parts not launched
        split_range_one_wave(K, a.parts, s, kNT, kb, ke);
    else
        split_range_waves(K, a.nsplit, s, kNT, b * nrb_req + rb, a.batch * nrb_req, a.wave_full, kb, ke);
    const int ntiles = (ke - kb + kNT - 1) / kNT;
    const int64_t kbase = key_base(a, b);

    // lse = -inf for this item's empty partitions: its own if it has no
    // keys, and the unlaunched partitions s + parts, s + 2 parts, ... (the
    // combine reads no o of a split whose lse is -inf)
    if (rank == 1 && warp >= 8 && warp < 12) {
        const int grow = rb * kM + 32 * (warp & 3) + lane;
        if (grow < rows_req) {
            float* lp = a.lse_part + ((int64_t)b * rows_req + grow) * a.nsplit;
            if (ntiles <= 0) lp[s] = -INFINITY;
            if (a.parts > 0)
                for (int s2 = s + a.parts; s2 < a.nsplit; s2 += a.parts) lp[s2] = -INFINITY;
        }
    }
    if (ntiles <= 0) {  // empty split (fixed grid, early exit)
        if (rank == 0 && tid == 0) status_or(a.status, bad);
        return;
    }
    if (rank != 0) bad &= ~MLA_STATUS_BAD_INDPTR;  // reported once, by the S-CTA

    if (warp == kWarpMMA) {
        tmem_alloc(smem_u32(&sm.h.tmem_base), 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(ba(sm.h.p_full), 256);
        mbar_init(ba(sm.h.p_free), 1);
        mbar_init(ba(sm.h.fin), 256);
        mbar_init(ba(sm.h.drain), 1);
        if (rank == 0) {
            SmemS& S = sm.u.s;
            for (int i = 0; i < kKStages; ++i) {
                mbar_init(ba(S.k_full[i]), 32 * kSProd);
                mbar_init(ba(S.k_empty[i]), 1);
            }
            for (int i = 0; i < kMetaRing; ++i) {
                mbar_init(ba(S.meta_full[i]), 1);
                mbar_init(ba(S.meta_free[i]), 256);
            }
            mbar_init(ba(S.s_full), 1);
            mbar_init(ba(S.s_free), 256);
            mbar_init(ba(S.q_ready), 256);
            mbar_init(ba(S.mx_bar[0]), 256);
            mbar_init(ba(S.mx_bar[1]), 256);
            for (int i = 0; i < kRowsRing; ++i) {
                mbar_init(ba(S.rows_full[i]), 1);
                mbar_init(ba(S.rows_free[i]), kSProd);
            }
        } else {
            SmemO& O = sm.u.o;
            for (int i = 0; i < kVStages; ++i) {
                mbar_init(ba(O.v_full[i]), 32 * kOProd);
                mbar_init(ba(O.v_empty[i]), 1);
            }
            mbar_init(ba(O.o_gate), 128);
            mbar_init(ba(O.o_prog), 1);
            for (int i = 0; i < kRowsRing; ++i) {
                mbar_init(ba(O.rows_full[i]), 1);
                mbar_init(ba(O.rows_free[i]), kOProd);
            }
        }
        sm.h.abort_flag = 0;
        sm.h.no_abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tbase = sm.h.tmem_base;
    volatile int* abort_p = &sm.h.abort_flag;
    const uint32_t peer = rank ^ 1u;

    const int wg = warp >> 2;
    if (rank == 0 && wg < 2) {
        regs_dec<kRegsLow>();
        SmemS& S = sm.u.s;
        if (warp == 0) {
            // ------------------------------------------------ S row stager
            // Each tile's pool rows (and the key-validity bits for the
            // softmax), up to kRowsRing tiles ahead of the copies.
            key_prefetch(a, b, kbase, Lb, kb + kNT, ke, lane);  // later tiles' slots
            for (int i = 0; i < ntiles; ++i) {
                const int rb2 = i % kRowsRing, mi = i % kMetaRing;
                if (i >= kRowsRing && !warp_wait(S.rows_free[rb2], ((i / kRowsRing) - 1) & 1, abort_p)) break;
                if (i >= kMetaRing && !warp_wait(S.meta_free[mi], ((i / kMetaRing) - 1) & 1, abort_p)) break;
                bad |= stage_rows<kNT>(a, b, kbase, Lb, kb + i * kNT, ke, lane, S.rows[rb2], S.valid[mi]);
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(ba(S.meta_full[mi]));
                    mbar_arrive(ba(S.rows_full[rb2]));
                }
            }
        } else if (warp != kWarpMMA) {
            // ------------------------------------------------ S copy warps: K blocks
            // Warps 1-3 and 5-7 split the 16-byte copies, eight lanes per
            // 128-byte row segment.
            const int pw = (warp < kWarpMMA ? warp : warp - 1) - 1;  // 0..5
            bool ok = true;
            for (int i = 0; ok && i < ntiles; ++i) {
                const int rb2 = i % kRowsRing;
                if (!warp_wait(S.rows_full[rb2], (i / kRowsRing) & 1, abort_p)) {
                    ok = false;
                    break;
                }
                const int nit = (tile_keys(kb, ke, i) + 3) >> 2;  // 4 keys per warp step
                for (int kbk = 0; kbk < kDqk / 64; ++kbk) {
                    const int g = i * (kDqk / 64) + kbk;
                    const int st = g % kKStages;
                    if (g >= kKStages && !warp_wait(S.k_empty[st], ((g / kKStages) - 1) & 1, abort_p)) {
                        ok = false;
                        break;
                    }
                    // Only the rows up to the tile's last key (rounded up to a
                    // warp step) are copied; the rest of the stage keeps stale
                    // data, whose scores are masked.
                    const uint32_t dst0 = smem_u32(S.kring[st]);
                    for (int it = pw; it < nit; it += kSProd) {
                        const int key = it * 4 + (lane >> 3), c = lane & 7;
                        const int32_t slot = S.rows[rb2][key];
                        const __nv_bfloat16* src =
                            a.kv + (slot >= 0 ? (int64_t)slot * kDqk : 0) + kbk * 64 + c * 8;
                        cp_async_16_zfill_nc(dst0 + sw128_offset(key, c), src, slot >= 0);
                    }
                    cp_async_mbar_arrive_noinc(ba(S.k_full[st]));
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(ba(S.rows_free[rb2]));
            }
            cp_async_wait_all();
        } else {
            // ------------------------------------------------ S MMA issuer
            if (lane == 0) {
                const uint32_t idesc = make_idesc_bf16(kM, kNT, false, false);
                bool ok = mbar_wait(ba(S.q_ready), 0, abort_p);
                fence_proxy_async_smem();
                tc_fence_after();
                const uint32_t dS = tbase + kColS;
                // descriptors precomputed; the loop only adds offsets
                const uint64_t kdesc0 = make_sdesc(smem_u32(S.kring[0]), 16, 1024, kSwizzle128B);
                const uint64_t qrdesc = make_sdesc(smem_u32(S.q_rope), 16, 1024, kSwizzle128B);
                for (int i = 0; ok && i < ntiles; ++i) {
                    if (i >= 1 && !mbar_wait(ba(S.s_free), (i - 1) & 1, abort_p)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // a partly filled tile: N = its keys rounded up to 16 (the
                    // score columns past them keep stale values, all masked)
                    const int nv = tile_keys(kb, ke, i);
                    const uint32_t idt = nv >= kNT ? idesc : make_idesc_bf16(kM, (nv + 15) & ~15, false, false);
                    for (int kbk = 0; kbk < kDqk / 64; ++kbk) {
                        const int g = i * (kDqk / 64) + kbk;
                        const int st = g % kKStages;
                        if (!mbar_wait(ba(S.k_full[st]), (g / kKStages) & 1, abort_p)) {
                            ok = false;
                            break;
                        }
                        fence_proxy_async_smem();
                        tc_fence_after();
                        const uint64_t bd = kdesc0 + (uint64_t)st * (kKBlock >> 4);
                        if (kbk < 8) {
                            const uint32_t aa = tbase + kColQ + kbk * 32;
                            mma_ts(dS, aa, bd, idt, kbk > 0 ? 1u : 0u);
                            mma_ts(dS, aa + 8, bd + 2, idt, 1u);
                            mma_ts(dS, aa + 16, bd + 4, idt, 1u);
                            mma_ts(dS, aa + 24, bd + 6, idt, 1u);
                        } else {
                            mma_ss(dS, qrdesc, bd, idt, 1u);
                            mma_ss(dS, qrdesc + 2, bd + 2, idt, 1u);
                            mma_ss(dS, qrdesc + 4, bd + 4, idt, 1u);
                            mma_ss(dS, qrdesc + 6, bd + 6, idt, 1u);
                        }
                        mma_commit(ba(S.k_empty[st]));
                    }
                    if (ok) mma_commit(ba(S.s_full));
                }
                mma_commit(ba(sm.h.drain));
                mbar_wait(ba(sm.h.drain), 0, &sm.h.no_abort);
            }
            __syncwarp();
        }
    } else if (rank == 0) {
        regs_inc<kRegsSoftmax>();
        SmemS& S = sm.u.s;
        {
            // ------------------------------------------------ softmax (warps 8-15)
            const int quarter = warp & 3;
            const int half = (warp - 8) >> 2;     // 128-key half of the tile
            const int r = 32 * quarter + lane;     // row = TMEM lane
            const int grow = rb * kM + r;
            const bool row_ok = grow < rows_req;
            const int t = row_ok ? grow / H : 0;
            const uint32_t lb = (uint32_t)(32 * quarter) << 16;
            const int stid = tid - 256;            // 0..255

            // Q staging: RoPE dims into their swizzled A-operand tile by
            // cp.async; latent dims straight from global memory into TMEM (each
            // thread its row's 256 dims of this half), so the K ring is never
            // used for Q and the copy warps start on the keys at once.
            {
                const __nv_bfloat16* q0 = a.q + ((int64_t)b * rows_req + rb * kM) * kDqk;
                for (int f = stid; f < kM * 8; f += 256) {
                    const int rr = f >> 3, c = f & 7;
                    const bool v = rb * kM + rr < rows_req;
                    const __nv_bfloat16* src = v ? q0 + (int64_t)rr * kDqk + 512 + c * 8 : a.q;
                    cp_async_16_zfill(smem_u32(S.q_rope) + sw128_offset(rr, c), src, v);
                }
                if (stid < T) {
                    if (a.anc_mask != nullptr)
                        S.anc[stid] = a.anc_mask[(int64_t)b * T + stid];
                    else
                        S.par[stid] = a.tree_parent[(int64_t)b * T + stid];
                }
                {
                    const uint4* src = reinterpret_cast<const uint4*>(q0 + (int64_t)r * kDqk + half * 256);
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {  // 64 dims (eight 16-byte loads) at a time
                        uint32_t w[32];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const uint4 x = row_ok ? __ldg(src + 8 * c + u) : make_uint4(0, 0, 0, 0);
                            w[4 * u] = x.x;
                            w[4 * u + 1] = x.y;
                            w[4 * u + 2] = x.z;
                            w[4 * u + 3] = x.w;
                        }
                        tmem_st32(tbase + lb + kColQ + half * 128 + c * 32, w);
                    }
                    tmem_wait_st();
                }
                cp_async_wait_all();
                asm volatile("bar.sync 1, 256;" ::: "memory");
                if (stid == 0 && a.anc_mask == nullptr) bad |= build_anc_serial(S.par, T, S.anc);
                fence_proxy_async_smem();
                tc_fence_before();
                asm volatile("bar.sync 1, 256;" ::: "memory");
                mbar_arrive(ba(S.q_ready));
            }
            const uint64_t anc_t = S.anc[t] & tree_bits(T);
            const uint32_t p_peer = mapa_shared(smem_u32(sm.u.o.p), peer);
            const uint32_t alpha_peer = mapa_shared(smem_u32(&sm.u.o.alpha[r]), peer);
            const uint32_t pfull_peer = mapa_shared(ba(sm.h.p_full), peer);
            float m_ref = -INFINITY, l_part = 0.f;
            bool ok = true;
            for (int i = 0; i < ntiles; ++i) {
                if (!warp_wait(S.s_full, i & 1, abort_p)) {
                    ok = false;
                    break;
                }
                // Keys of this half of the tile: a half without any has no
                // scores to read and no P that the P V steps read.
                const int hk = tile_keys(kb, ke, i) - 128 * half;
                tc_fence_after();
                float sc[128];
                if (hk > 0) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t w[32];
                        tmem_ld32(tbase + lb + kColS + half * 128 + c * 32, w);
                        tmem_wait_ld();
#pragma unroll
                        for (int u = 0; u < 32; ++u) sc[c * 32 + u] = __uint_as_float(w[u]);
                    }
                }
                tc_fence_before();
                mbar_arrive(ba(S.s_free));
                const int mi = i % kMetaRing;
                if (!warp_wait(S.meta_full[mi], (i / kMetaRing) & 1, abort_p)) {
                    ok = false;
                    break;
                }
                uint32_t vw[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) vw[q] = row_ok ? S.valid[mi][4 * half + q] : 0u;
                mbar_arrive(ba(S.meta_free[mi]));
                const int k0 = kb + i * kNT + 128 * half;
                if (k0 + 128 > Lb) {  // this half reaches the tree keys
#pragma unroll
                    for (int q = 0; q < 4; ++q) vw[q] &= tree_keep_word(anc_t, k0 + 32 * q - Lb);
                }
                // Max over the raw scores (the scale is positive, so scaling
                // the max is exact); masked keys become -inf only where this
                // row's half-tile has any.
                float mx = -INFINITY;
                if (hk > 0 && (vw[0] & vw[1] & vw[2] & vw[3]) != 0xffffffffu) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (!((vw[c >> 5] >> (c & 31)) & 1u)) sc[c] = -INFINITY;
                }
                if (hk > 0) {  // eight independent chains, then a tree
                    float m8[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) m8[j] = sc[j];
#pragma unroll
                    for (int c = 8; c < 128; ++c) m8[c & 7] = fmaxf(m8[c & 7], sc[c]);
                    mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
                }
                mx *= a.scale_log2;
                S.mx[i & 1][half][r] = mx;
                mbar_arrive(ba(S.mx_bar[i & 1]));
                if (!warp_wait(S.mx_bar[i & 1], (i >> 1) & 1, abort_p)) {
                    ok = false;
                    break;
                }
                const float mt = fmaxf(mx, S.mx[i & 1][half ^ 1][r]);
                float alpha = 1.f;
                if (mt > -INFINITY) {
                    if (m_ref == -INFINITY) {
                        m_ref = mt;
                    } else if (mt > m_ref + kRescaleLog2) {
                        alpha = ex2_approx(m_ref - mt);
                        m_ref = mt;
                        l_part *= alpha;
                    }
                }
                if (i >= 1 && !warp_wait_cluster(sm.h.p_free, (i - 1) & 1, abort_p)) {
                    ok = false;
                    break;
                }
                // P (bf16) -> the O-CTA's A-operand tile, 8 keys (16 bytes) at a time.
                // p = 2^(s * scale_log2 - m_ref) in one FMA per key; masked
                // keys (-inf) give 2^-inf = 0; a row with no visible key yet
                // (m_ref = -inf) writes zeros.
                float ps8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // eight chains
                const float sl = a.scale_log2;
                const float nm = m_ref == -INFINITY ? 0.f : -m_ref;
                const bool any = m_ref != -INFINITY;
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    if (hk <= 64 * blk) break;  // keys from here on are past the tile's last 16-key step
                    const uint32_t pb = p_peer + (2 * half + blk) * kPBlock;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint32_t w[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int k = blk * 64 + c * 8 + 2 * u;
                            const float p0 = any ? ex2_approx(fmaf(sc[k], sl, nm)) : 0.f;
                            const float p1 = any ? ex2_approx(fmaf(sc[k + 1], sl, nm)) : 0.f;
                            ps8[(c & 3) * 2 + (u & 1)] += p0 + p1;
                            w[u] = pack_bf16x2(p0, p1);
                        }
                        st_cluster_v4(pb + sw128_offset(r, c), w[0], w[1], w[2], w[3]);
                    }
                }
                l_part += ((ps8[0] + ps8[1]) + (ps8[2] + ps8[3])) + ((ps8[4] + ps8[5]) + (ps8[6] + ps8[7]));
                if (half == 0) st_cluster_f32(alpha_peer, alpha);
                fence_proxy_async_all();
                mbar_arrive_cluster(pfull_peer);
            }
            if (ok) {
                if (half == 0) {
                    st_cluster_f32(mapa_shared(smem_u32(&sm.u.o.fin_m[r]), peer), m_ref);
                    st_cluster_f32(mapa_shared(smem_u32(&sm.u.o.fin_l[0][r]), peer), l_part);
                } else {
                    st_cluster_f32(mapa_shared(smem_u32(&sm.u.o.fin_l[1][r]), peer), l_part);
                }
                mbar_arrive_cluster(mapa_shared(ba(sm.h.fin), peer));
            }
        }
    } else if (wg != 2) {
        regs_dec<kRegsLow>();
        SmemO& O = sm.u.o;
        if (warp == 0) {
            // ------------------------------------------------ O row stager
            // Each tile's pool rows, up to kRowsRing tiles ahead of the copies.
            for (int i = 0; i < ntiles; ++i) {
                const int rb2 = i % kRowsRing;
                if (i >= kRowsRing && !warp_wait(O.rows_free[rb2], ((i / kRowsRing) - 1) & 1, abort_p)) break;
                (void)stage_rows<kNT>(a, b, kbase, Lb, kb + i * kNT, ke, lane, O.rows[rb2], nullptr);  // the S-CTA reports
                __syncwarp();
                if (lane == 0) mbar_arrive(ba(O.rows_full[rb2]));
            }
        } else if (warp != kWarpMMA) {
            // ------------------------------------------------ O copy warps: V rows
            // Warps 1-3, 5-7 and 12-15 split the 16-byte copies (32 lanes =
            // one half of a 1024-byte V row).
            const int pw = (warp < kWarpMMA ? warp : (warp < 8 ? warp - 1 : warp - 5)) - 1;  // 0..9
            bool ok = true;
            int g = 0;  // V stages so far (a tile takes only the stages holding its keys)
            for (int i = 0; ok && i < ntiles; ++i) {
                const int rb2 = i % kRowsRing;
                if (!warp_wait(O.rows_full[rb2], (i / kRowsRing) & 1, abort_p)) {
                    ok = false;
                    break;
                }
                // keys the P V steps read: the tile's keys rounded up to 16
                // (zeros where there is no pool row, so that p = 0 adds 0)
                const int nv16 = (tile_keys(kb, ke, i) + 15) & ~15;
                const int nq = tile_vstages(kb, ke, i);
                for (int q = 0; q < nq; ++q, ++g) {
                    const int st = g % kVStages;
                    if (g >= kVStages && !warp_wait(O.v_empty[st], ((g / kVStages) - 1) & 1, abort_p)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst0 = smem_u32(O.vring[st]);
                    const int nit = 2 * min(kVKeys, nv16 - kVKeys * q);  // two lanes' chunks per key
                    for (int it = pw; it < nit; it += kOProd) {
                        const int kl = it >> 1;                 // key within the stage
                        const int c = (it & 1) * 32 + lane;     // 16-byte chunk of the V row
                        const int32_t slot = O.rows[rb2][32 * q + kl];
                        const __nv_bfloat16* src = a.kv + (slot >= 0 ? (int64_t)slot * kDqk : 0) + c * 8;
                        cp_async_16_zfill_nc(dst0 + (c >> 3) * kVBlock + sw128_offset(kl, c & 7), src,
                                             slot >= 0);
                    }
                    cp_async_mbar_arrive_noinc(ba(O.v_full[st]));
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(ba(O.rows_free[rb2]));
            }
            cp_async_wait_all();
        } else {
            // ------------------------------------------------ O MMA issuer
            if (lane == 0) {
                const uint32_t idesc = make_idesc_bf16(kM, 256, false, true);
                const uint32_t pfree_peer = mapa_shared(ba(sm.h.p_free), peer);
                // descriptors precomputed: only the low word (start address) moves
                const uint64_t pdesc0 = make_sdesc(smem_u32(O.p), 16, 1024, kSwizzle128B);
                const uint64_t vdesc0 = make_sdesc(smem_u32(O.vring[0]), kVBlock, 1024, kSwizzle128B);
                const uint32_t plo = (uint32_t)pdesc0, phi = (uint32_t)(pdesc0 >> 32);
                const uint32_t vlo = (uint32_t)vdesc0, vhi = (uint32_t)(vdesc0 >> 32);
                auto dsc = [](uint32_t lo, uint32_t hi) { return ((uint64_t)hi << 32) | lo; };
                bool ok = true;
                int g = 0;  // V stages so far, as counted by the V producers
                for (int i = 0; ok && i < ntiles; ++i) {
                    if (!mbar_wait_cluster(ba(sm.h.p_full), i & 1, abort_p) ||
                        !mbar_wait(ba(O.o_gate), i & 1, abort_p)) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async_smem();
                    tc_fence_after();
                    const int nv = tile_keys(kb, ke, i);
                    const int nq = tile_vstages(kb, ke, i);
                    for (int q = 0; q < nq; ++q, ++g) {
                        const int st = g % kVStages;
                        if (!mbar_wait(ba(O.v_full[st]), (g / kVStages) & 1, abort_p)) {
                            ok = false;
                            break;
                        }
                        fence_proxy_async_smem();
                        tc_fence_after();
                        const uint32_t vd = vlo + (uint32_t)st * (kVStage >> 4);
                        // keys q*32 .. q*32+31 of the tile: P block q / 2, 16-key steps
                        const uint32_t pd = plo + (uint32_t)((q >> 1) * kPBlock + (q & 1) * 64) / 16;
                        const uint32_t acc0 = (i > 0 || q > 0) ? 1u : 0u;
                        if (kVKeys * q < nv) {  // 16-key steps holding keys of the tile
                            mma_ss(tbase, dsc(pd, phi), dsc(vd, vhi), idesc, acc0);
                            mma_ss(tbase + 256, dsc(pd, phi), dsc(vd + (4 * kVBlock) / 16, vhi), idesc, acc0);
                        }
                        if (kVKeys * q + 16 < nv) {
                            mma_ss(tbase, dsc(pd + 2, phi), dsc(vd + 2048 / 16, vhi), idesc, 1u);
                            mma_ss(tbase + 256, dsc(pd + 2, phi), dsc(vd + (4 * kVBlock + 2048) / 16, vhi), idesc, 1u);
                        }
                        mma_commit(ba(O.v_empty[st]));
                    }
                    if (!ok) break;
                    mma_commit(ba(O.o_prog));
                    // P is single-buffered: hand it back once this tile's P V is done.
                    if (!mbar_wait(ba(O.o_prog), i & 1, abort_p)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_cluster(pfree_peer);
                }
                mma_commit(ba(sm.h.drain));
                mbar_wait(ba(sm.h.drain), 0, &sm.h.no_abort);
            }
            __syncwarp();
        }
    } else {
        SmemO& O = sm.u.o;
        {
            // ------------------------------------------------ correction + epilogue
            const int quarter = warp & 3;
            const int r = 32 * quarter + lane;
            const int grow = rb * kM + r;
            const bool row_ok = grow < rows_req;
            const uint32_t lb = (uint32_t)(32 * quarter) << 16;
            bool ok = true;
            for (int i = 0; i < ntiles; ++i) {
                if (!warp_wait_cluster(sm.h.p_full, i & 1, abort_p)) {
                    ok = false;
                    break;
                }
                const float alpha = O.alpha[r];
                if (__any_sync(0xffffffffu, alpha != 1.f) && i > 0) {
                    if (!warp_wait(O.o_prog, (i - 1) & 1, abort_p)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int c0 = 0; c0 < 512; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(tbase + lb + c0, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
                        tmem_st32(tbase + lb + c0, o);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                mbar_arrive(ba(O.o_gate));
            }
            if (ok) ok = warp_wait_cluster(sm.h.fin, 0, abort_p);
            if (ok) ok = warp_wait(O.o_prog, (ntiles - 1) & 1, abort_p);
            tc_fence_after();
            if (ok) {
                const float l = O.fin_l[0][r] + O.fin_l[1][r];
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const int64_t pid = ((int64_t)b * rows_req + (row_ok ? grow : 0)) * a.nsplit + s;
                // Coalesced partial write: each 32-row x 32-column chunk goes
                // through a padded tile in the (now idle) V ring and out again
                // with eight lanes per row, so every store instruction writes
                // four whole 128-byte lines instead of 32 lines in part.
                float* tile = reinterpret_cast<float*>(O.vring[0]) + quarter * (32 * kOTileStride);
                const int jr = lane >> 3, jc = 4 * (lane & 7);  // row in a group of 4, column
                const int rj0 = rb * kM + 32 * quarter + jr;       // this lane's row of group 0
                float* const o0 = a.o_part + (((int64_t)b * rows_req + rj0) * a.nsplit + s) * kDv + jc;
                const int64_t gstep = (int64_t)4 * a.nsplit * kDv;   // four rows on
#pragma unroll 1
                for (int c0 = 0; c0 < 512; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(tbase + lb + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        *reinterpret_cast<float4*>(tile + lane * kOTileStride + 4 * u) = make_float4(
                            __uint_as_float(o[4 * u]) * inv, __uint_as_float(o[4 * u + 1]) * inv,
                            __uint_as_float(o[4 * u + 2]) * inv, __uint_as_float(o[4 * u + 3]) * inv);
                    __syncwarp();
                    // all eight tile reads before the first store (the stores
                    // may not be ordered ahead of later reads of the tile)
                    float4 v[8];
#pragma unroll
                    for (int g = 0; g < 8; ++g)
                        v[g] = *reinterpret_cast<const float4*>(tile + (4 * g + jr) * kOTileStride + jc);
#pragma unroll
                    for (int g = 0; g < 8; ++g)
                        if (rj0 + 4 * g < rows_req) *reinterpret_cast<float4*>(o0 + g * gstep + c0) = v[g];
                    __syncwarp();
                }
                if (row_ok)
                    a.lse_part[pid] = l > 0.f ? (O.fin_m[r] + log2f(l)) * kLn2 : -INFINITY;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // no CTA leaves while its peer may still touch its shared memory
    if (warp == kWarpMMA) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
    if (sm.h.abort_flag) bad |= MLA_STATUS_TIMEOUT;
    status_or(a.status, bad);
}

}  // namespace

// Resident 2-CTA clusters per device, for the wave shaping of the partitions.
int g_pair_clusters[64];

cudaError_t setup_partial_pair() {
    cudaError_t e = cudaFuncSetAttribute(partial_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    int dev = -1;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, partial_pair_kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();  // unknown: plain even partitions
        n = 0;
    }
    g_pair_clusters[dev] = n;
    return cudaSuccess;
}

static int pair_resident() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    return g_pair_clusters[dev];
}

int pair_expected_parts(int batch, int T, int H, int nsplit) {
    const int p = one_wave_parts((long long)batch * ((T * H + kM - 1) / kM), pair_resident(), nsplit);
    return p > 0 ? p : nsplit;
}

cudaError_t launch_partial_pair(const PartialArgs& a, cudaStream_t stream) {
    const int rows_req = a.T * a.H;
    const int nrb = (rows_req + kM - 1) / kM;
    const int resident = pair_resident();
    PartialArgs w = a;
    // When every (request, row block) pair can take at least one cluster of
    // one wave, the keys are split evenly over as many partitions as the
    // wave holds (up to nsplit), and only those are launched; otherwise all
    // nsplit partitions are, with the wave-shaped split.
    w.parts = one_wave_parts((long long)a.batch * nrb, resident, a.nsplit);
    w.wave_full = wave_full_items((long long)a.batch * a.nsplit * nrb, resident);
    const dim3 grid(2 * nrb, a.batch, w.parts > 0 ? w.parts : a.nsplit);
    return launch_pdl(partial_pair_kernel, grid, dim3(kThreads), kSmemBytes, stream, w);
}

}  // namespace mlav
