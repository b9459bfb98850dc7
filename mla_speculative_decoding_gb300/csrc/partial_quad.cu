// Split-KV partial attention on two pairs of SMs with 2-SM (cta_group::2)
// tensor-core MMAs: four SMs per 256-row work item.
//
// The verify attention of "The Custom sm_120 Verify Kernel..." (Parts VI,
// VII, IX): every tree-token x head row of a request attends over the
// request's scattered latent KV rows (prefix unmasked, tree block masked),
// in a KV-split "partial + reduce" design.
//
// Work item = (256-row block of the request's T*H rows, split s, request b),
// run by a cluster of four CTAs. A pair MMA (M = 256) keeps 128 rows of the
// accumulator in each SM of the pair and reads half of the B operand's N
// columns from each SM's shared memory, so every gathered byte feeds 256
// rows while each SM gathers only half of the tile:
//
//   S pair (ranks 0, 1): S = Q K^T for 256-key tiles, M = 256, N = 256
//     (36 pair MMAs per tile, issued by rank 0). Rank r holds rows
//     [128r, 128r + 128) of the block (Q's 512 latent dims in TMEM [0, 256)
//     as the A operand, the 64 RoPE dims in shared memory) and gathers keys
//     [128r, 128r + 128) of every tile (all 576 dims, 64-dim blocks of 16 KB
//     in an 8-stage ring). S lands in TMEM [256, 512) of each SM: 128 rows x
//     256 keys. Eight softmax warps per SM copy S out of TMEM, mask it, keep
//     a lazily rescaled running maximum, and write P (bf16) into a local
//     staging tile, which one thread sends to the O partner of the same rows
//     (rank r + 2) with a bulk shared-memory copy.
//   O pair (ranks 2, 3): O += P V, M = 256, two N = 256 chains (V dims
//     [0, 256) and [256, 512)), issued by rank 2; rank 2 + r holds O for rows
//     [128r, 128r + 128) in TMEM [0, 512) and gathers, for all 256 keys of a
//     tile, its half of each chain's V columns: 64-dim segments
//     {2r, 2r + 1, 4 + 2r, 5 + 2r}. P arrives double-buffered, so P of the
//     next tile is written while this tile's P V runs. Four correction warps
//     per SM apply the rare rescales to O and write the partial (o, lse).
//
// Operand readiness across a pair: each CTA's copies land on its own
// mbarrier; one thread per CTA (the odd CTA's MMA warp, a spare warp of the
// even CTA) waits for each landed stage, fences it for the tensor cores
// (proxy fence) and arrives on the even CTA's ready barrier, which the MMA
// issuer waits for, so no fence sits in the issue loop. MMA completion is committed to
// the barriers of both CTAs of the pair (multicast). Barriers that only
// signal completed work (landed copies, finished TMEM reads, completed
// MMAs) use default (CTA-scope) arrive and wait semantics, which cost far
// less than cluster-scope release/acquire; the one hand-over of data stored
// into another CTA's shared memory (the final row maxima and sums) uses
// cluster scope.
//
// Persistent clusters: the launch holds one cluster per resident slot. By
// default (the balanced plan) the key tiles of all (request, row block)
// pairs form one sequence and each cluster takes one contiguous range of it,
// each range's part of a pair being one partition (the pair's unused
// partitions get lse = -inf); where that plan does not fit (more than 128
// requests, or a pair cut into more than nsplit parts), cluster c takes the
// work items of rounds k = 0, 1, ... at position (c + k) mod C of each round
// of C items. Every ring, slot and barrier phase counts over the cluster's
// whole tile sequence, so one item's drain (last softmax, P hand-over, last
// P V and the partial write) overlaps the next item's start.
//
// Each tile's pool slots come from the combined key list or, in the paged
// form, from the request's page-table row and its draft slots; control
// warps stage them a few tiles ahead of the copies.
//
// Every wait is bounded; on a timeout a CTA drains its MMAs, reaches the
// final cluster barrier, frees TMEM and flags MLA_STATUS_TIMEOUT.
#include "partial_kernels.cuh"
#include "tc_ptx.cuh"

namespace mlav {
namespace {

using namespace tc;

constexpr int kRowsBlk = 256;     // rows per work item
constexpr int kMh = 128;          // rows per CTA
constexpr int kNT = 256;          // keys per tile
constexpr int kNh = 128;          // keys per S-CTA per tile
constexpr int kThreads = 640;     // 20 warps = 5 warpgroups
constexpr int kWarpMMA = 4;
constexpr int kWarpCtl = 7;       // P sender (S CTAs) / P slot release (O pair)
constexpr int kSProd = 8;         // S-side producer warps: 0-3, 5, 6, 16, 17
constexpr int kWarpFwd = 18;      // rank 0: fences each landed K stage for the MMA issuer
constexpr int kSGroup = 2;        // producer warps per K stage (stages go round-robin to groups)
constexpr int kOProd = 14;        // O-side producer warps: 0-3, 5, 6, 12-19
// Launched at 96 registers per thread (640 x 96 = 61,440). S CTAs:
// warpgroups 0, 1, 4 drop to 48 and the softmax warpgroups (2, 3) rise to
// 168 (384 x 48 + 256 x 168 = 61,440). O CTAs: warpgroups 0, 1, 3, 4 drop
// to 48; the correction warpgroup keeps 96.
constexpr int kRegsLow = 48, kRegsSoftmax = 168;
constexpr int kKStages = 8;
// A producer group waits for the release of the stage one lap back; with more
// groups than stages it could pass a whole lap (parity aliasing) and reuse a
// stage still in use.
static_assert(kSProd / kSGroup <= kKStages, "producer groups must not exceed the K stages");
constexpr uint32_t kKBlock = kNh * 128;        // 128 keys x 64 dims (bf16) = 16 KB
constexpr int kMetaRing = 4;
constexpr int kRowsRing = 4;       // pool-row staging, up to three tiles ahead of the copies
constexpr int kVKeys = 32;
constexpr int kVStages = 4;
constexpr uint32_t kVSub = kVKeys * 128;       // 32 keys x 64 dims = 4 KB
constexpr uint32_t kVStage = 4 * kVSub;        // [chain][segment][32 keys][64 dims]
constexpr int kOTileStride = 36;               // floats per row of the epilogue's write tile
constexpr uint32_t kPBlock = kMh * 128;        // 128 rows x 64 keys (bf16)
constexpr uint32_t kPBytes = 4 * kPBlock;      // 128 rows x 256 keys
constexpr uint32_t kPXfer = kPBytes + kMh * 4; // P + per-row rescale factors
constexpr uint32_t kPSlot = 67584;             // 1024-aligned P slot
constexpr uint32_t kColQ = 0, kColS = 256;     // S-CTA TMEM map
constexpr float kRescaleLog2 = 8.0f;

struct SmemS {
    unsigned char q_rope[kMh * 128];            // [128 rows x 64 dims], 128B-swizzled
    unsigned char kring[kKStages][kKBlock];     // [128 keys x 64 dims] per stage
    unsigned char pstage[kPXfer];               // P [4 x (128 rows x 64 keys)] + alpha[128]
    uint32_t valid[kMetaRing][kNT / 32];
    int32_t rows[kRowsRing][kNT];               // pool rows of the tiles being gathered
    float mx[2][2][kMh];
    uint64_t anc[MLA_MAX_TREE];
    int32_t par[MLA_MAX_TREE];
    uint64_t k_full[kKStages], k_empty[kKStages];
    uint64_t k_ready[kKStages];  // rank 0: both CTAs' stage landed and fenced (two forwarders)
    uint64_t meta_full[kMetaRing], meta_free[kMetaRing];
    uint64_t s_full, s_free, q_landed, q_ready, q_peer, mx_bar[2], pw_bar[2], pstage_free;
    uint64_t rows_full[kRowsRing];
    uint64_t p_free[2];
    uint64_t fin_free[2];                       // the O partner has read fin[slot]
};
struct SmemO {
    unsigned char pbuf[2][kPSlot];              // P + alpha, one slot per tile parity
    unsigned char vring[kVStages][kVStage];
    int32_t rows[kRowsRing][kNT];
    float otile[4][32 * kOTileStride];          // the epilogue's write tiles, one per warp
    float fin_m[2][kMh];                        // per item parity: row maxima
    float fin_l[2][2][kMh];                     //   and the two key halves' sums
    uint64_t v_full[kVStages], v_empty[kVStages];
    uint64_t p_full[2], o_gate[2], o_done[2], fin[2];
    uint64_t rows_full[kRowsRing], rows_free[kRowsRing];
};
constexpr int kPlanMaxReq = 128;  // requests the balanced plan tabulates
struct Header {
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int no_abort;
    int balanced;                       // 1: balanced tile ranges, 0: rotated rounds
    int w;                              // balanced: tiles over all (request, row block)
    int ptile[kPlanMaxReq + 1];         // balanced: first tile of request b (row block 0)
};
struct __align__(1024) SmemQuad {
    union {
        SmemS s;
        SmemO o;
    } u;
    Header h;
};

constexpr size_t kSmemBytes = sizeof(SmemQuad) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kPXfer <= kPSlot && kPSlot % 1024 == 0, "P slot");

__device__ __forceinline__ uint32_t ba(const uint64_t& b) { return smem_u32(&b); }

// Whole warps park in try_wait; the single-thread hand-over roles (MMA
// issuers, forwarders, the P sender and slot release) poll with
// mbar_wait_spin, since their resume latency is on a pipeline's critical path.
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

// One work item of a cluster's sequence: request b, partition s and row
// block rb, with its key range [kb, ke) in ntiles tiles.
struct QuadItem {
    int b, s, rb, kb, ke, ntiles, Lb, bad;
};

// Rotated rounds (the fallback plan): item k of cluster `cid` of `C` is the
// item at position (cid + k) mod C of round k; false past the last item.
// Items are numbered partition-major, ((s * batch + b) * nrb + rb), so every
// request's first partitions come first, and the partitions are the
// wave-shaped split of the request's tiles.
__device__ __forceinline__ bool quad_item(const PartialArgs& a, int nrb, int n_items, int C, int cid,
                                          int k, QuadItem& it) {
    const long long j = (long long)k * C + (cid + k) % C;
    if (j >= n_items) return false;
    const int jj = (int)j;
    it.rb = jj % nrb;
    const int t = jj / nrb;
    it.b = t % a.batch;
    it.s = t / a.batch;
    int K;
    it.bad = request_keys(a, it.b, it.Lb, K);
    split_range_waves(K, a.nsplit, it.s, kNT, it.b * nrb + it.rb, a.batch * nrb, a.wave_full, it.kb, it.ke);
    it.ntiles = (it.ke - it.kb + kNT - 1) / kNT;
    return true;
}

// Built by one warp of every CTA (all CTAs reach the same plan): the first
// tile of each request and the choice of plan. The balanced plan (the key
// tiles of all (request, row block) pairs cut into one contiguous range per
// cluster, each cluster's part of a pair one partition of it) needs at most
// kPlanMaxReq requests and plan_fits; otherwise the rotated rounds run.
// (Not inlined: its registers stay out of the roles' budgets; it takes the
// few arguments it reads by value so that the kernel parameters stay in
// parameter space.)
__device__ __noinline__ void build_plan(const int32_t* prefix_lens, const int32_t* kv_indptr,
                                        const int32_t* kv_indices, const int32_t* req_pool_indices,
                                        int64_t r2t_rows, int64_t r2t_stride, int batch, int T,
                                        int nsplit, int nrb, int C, int lane, Header& h) {
    PartialArgs a;
    a.prefix_lens = prefix_lens;
    a.kv_indptr = kv_indptr;
    a.kv_indices = kv_indices;
    a.req_pool_indices = req_pool_indices;
    a.r2t_rows = r2t_rows;
    a.r2t_stride = r2t_stride;
    a.batch = batch;
    a.T = T;
    a.nsplit = nsplit;
    if (a.batch > kPlanMaxReq) {
        if (lane == 0) h.balanced = 0;
        return;
    }
    long long run = 0;
    int tmax = 0;
    for (int b0 = 0; b0 < a.batch; b0 += 32) {
        const int b = b0 + lane;
        int t = 0;
        if (b < a.batch) {
            int Lb, K;
            (void)request_keys(a, b, Lb, K);
            t = (K + kNT - 1) / kNT;
        }
        tmax = max(tmax, t);
        int incl = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (b < a.batch) h.ptile[b] = (int)min(run + (long long)(incl - t) * nrb, 1ll << 30);
        run += (long long)__shfl_sync(0xffffffffu, incl, 31) * nrb;
    }
    tmax = __reduce_max_sync(0xffffffffu, tmax);
    if (lane == 0) {
        const bool fits = plan_fits(run, tmax, C, a.nsplit);
        h.ptile[a.batch] = fits ? (int)run : 0;
        h.w = fits ? (int)run : 0;
        h.balanced = fits ? 1 : 0;
    }
}

// A cluster's walk over its items under either plan.
struct ItemWalk {
    int x, xend;        // balanced: the cluster's next tile and the end of its range
    int b;              // balanced: request holding tile x
    int k;              // rotated rounds: next round
};
__device__ __forceinline__ ItemWalk walk_init(const Header& h, int cid, int C) {
    ItemWalk w;
    w.k = 0;
    w.b = 0;
    w.x = h.balanced ? plan_begin(cid, C, h.w) : 0;
    w.xend = h.balanced ? plan_begin(cid + 1, C, h.w) : 0;
    return w;
}
__device__ __forceinline__ bool walk_next(ItemWalk& w, const PartialArgs& a, const Header& h, int nrb,
                                          int n_items, int C, int cid, QuadItem& it) {
    if (!h.balanced) return quad_item(a, nrb, n_items, C, cid, w.k++, it);
    if (w.x >= w.xend) return false;
    int u0, u1;
    const int n = plan_step(h.ptile, nrb, C, h.w, cid, w.x, w.xend, w.b, it.rb, u0, u1, it.s);
    it.b = w.b;
    int K;
    it.bad = request_keys(a, it.b, it.Lb, K);
    it.kb = u0 * kNT;
    it.ke = min(K, u1 * kNT);
    it.ntiles = n;
    w.x += n;
    return true;
}

// The cluster's tiles in order over its non-empty items (what the row
// staging needs of each: request, key range, tile count).
struct TileCursor {
    ItemWalk w;
    int b, kb, ke, Lb, ntiles, i, bad;
};
__device__ __forceinline__ void cursor_init(TileCursor& c, const Header& h, int cid, int C) {
    c.w = walk_init(h, cid, C);
    c.i = 0;
    c.ntiles = 0;
    c.bad = 0;
}
// Moves to the next tile; false past the last one.
__device__ __forceinline__ bool cursor_next(TileCursor& c, const PartialArgs& a, const Header& h, int nrb,
                                            int n_items, int C, int cid) {
    if (++c.i < c.ntiles) return true;
    for (;;) {
        QuadItem it;
        if (!walk_next(c.w, a, h, nrb, n_items, C, cid, it)) return false;
        c.bad |= it.bad;
        if (it.ntiles > 0) {
            c.b = it.b;
            c.kb = it.kb;
            c.ke = it.ke;
            c.Lb = it.Lb;
            c.ntiles = it.ntiles;
            c.i = 0;
            return true;
        }
    }
}

// Columns [c0, c1) of one warp's 32 rows (the TMEM lanes of its quarter) of
// an item's partial o, scaled by the lane's 1/l: each 32-row x 32-column
// chunk goes through a padded tile and out again with eight lanes per row,
// so every store instruction writes four whole 128-byte lines.
__device__ __forceinline__ void write_o_cols(const PartialArgs& a, const QuadItem& it, int rows_req,
                                             int row0w, uint32_t taddr, float inv, float* tile, int lane,
                                             int c0, int c1) {
    const int jr = lane >> 3, jc = 4 * (lane & 7);  // row in a group of 4, column
    const int rj0 = row0w + jr;                     // this lane's row of group 0
    float* const o0 = a.o_part + (((int64_t)it.b * rows_req + rj0) * a.nsplit + it.s) * kDv + jc;
    const int64_t gstep = (int64_t)4 * a.nsplit * kDv;  // four rows on
#pragma unroll 1
    for (int c = c0; c < c1; c += 32) {
        uint32_t o[32];
        tmem_ld32(taddr + c, o);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 8; ++u)
            *reinterpret_cast<float4*>(tile + lane * kOTileStride + 4 * u) = make_float4(
                __uint_as_float(o[4 * u]) * inv, __uint_as_float(o[4 * u + 1]) * inv,
                __uint_as_float(o[4 * u + 2]) * inv, __uint_as_float(o[4 * u + 3]) * inv);
        __syncwarp();
        // all eight tile reads before the first store (the stores may not be
        // ordered ahead of later reads of the tile)
        float4 v[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) v[g] = *reinterpret_cast<const float4*>(tile + (4 * g + jr) * kOTileStride + jc);
#pragma unroll
        for (int g = 0; g < 8; ++g)
            if (rj0 + 4 * g < rows_req) *reinterpret_cast<float4*>(o0 + g * gstep + c) = v[g];
        __syncwarp();
    }
}

__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(kThreads, 1)
partial_quad_kernel(const PartialArgs a) {
    pdl_launch_dependents();
    extern __shared__ __align__(1024) unsigned char raw[];
    unsigned char* base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
    SmemQuad& sm = *reinterpret_cast<SmemQuad*>(base);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const bool sside = rank < 2;
    const uint32_t hr = rank & 1u;            // row half (and B-operand half) of this CTA
    const int cid = blockIdx.x >> 2, C = gridDim.x >> 2;
    const int T = a.T, H = a.H, rows_req = T * H;
    const int nrb = (rows_req + kRowsBlk - 1) / kRowsBlk;
    const int n_items = a.batch * a.nsplit * nrb;
    int bad = 0;

    if (warp == kWarpMMA) {  // both CTAs of each pair allocate together
        tmem_alloc_pair(smem_u32(&sm.h.tmem_base), 512);
        tmem_relinquish_pair();
    }
    if (tid == 0) {
        mbar_init(ba(sm.h.drain), 1);
        if (sside) {
            SmemS& S = sm.u.s;
            for (int i = 0; i < kKStages; ++i) {
                mbar_init(ba(S.k_full[i]), 32 * kSGroup);
                mbar_init(ba(S.k_empty[i]), 1);
                mbar_init(ba(S.k_ready[i]), 2);
            }
            for (int i = 0; i < kMetaRing; ++i) {
                mbar_init(ba(S.meta_full[i]), 1);
                mbar_init(ba(S.meta_free[i]), 8);   // one arrival per softmax warp
            }
            mbar_init(ba(S.s_full), 1);
            mbar_init(ba(S.s_free), 16);  // rank 0's: the softmax warps of both S CTAs
            mbar_init(ba(S.pstage_free), 1);
            mbar_init(ba(S.q_landed), 256);
            mbar_init(ba(S.q_ready), 256);
            mbar_init(ba(S.q_peer), 1);
            for (int i = 0; i < 2; ++i) {
                mbar_init(ba(S.mx_bar[i]), 8);
                mbar_init(ba(S.pw_bar[i]), 8);
                mbar_init(ba(S.p_free[i]), 1);
                mbar_init(ba(S.fin_free[i]), 4);  // the O partner's four correction warps
            }
            for (int i = 0; i < kRowsRing; ++i) {
                mbar_init(ba(S.rows_full[i]), 1);
            }
        } else {
            SmemO& O = sm.u.o;
            for (int i = 0; i < kVStages; ++i) {
                mbar_init(ba(O.v_full[i]), 32 * kOProd + (rank == 2 ? 1 : 0));
                mbar_init(ba(O.v_empty[i]), 1);
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(ba(O.p_full[i]), 1);
                mbar_init(ba(O.o_gate[i]), 8);
                mbar_init(ba(O.o_done[i]), 1);
                mbar_init(ba(O.fin[i]), 256);
            }
            for (int i = 0; i < kRowsRing; ++i) {
                mbar_init(ba(O.rows_full[i]), 1);
                mbar_init(ba(O.rows_free[i]), kOProd);
            }
        }
        sm.h.abort_flag = 0;
        sm.h.no_abort = 0;
        fence_mbar_init();
    }
    pdl_wait();  // the set-up above touches no global memory
    if (warp == 1)
        build_plan(a.prefix_lens, a.kv_indptr, a.kv_indices, a.req_pool_indices, a.r2t_rows, a.r2t_stride,
                   a.batch, T, a.nsplit, nrb, C, lane, sm.h);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // every CTA's barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tbase = sm.h.tmem_base;
    volatile int* abort_p = &sm.h.abort_flag;

    const int wg = warp >> 2;
    if (sside && wg != 2 && wg != 3) {
        regs_dec<kRegsLow>();
        SmemS& S = sm.u.s;
        if ((warp < 8 && warp != kWarpMMA && warp != kWarpCtl) || warp == 16 || warp == 17) {
            // ------------------------------------------------ S producers: K blocks
            // The eight producer warps form four groups of two; fill g of the
            // cluster's sequence (this CTA's 128 keys x 64 dims of one tile)
            // is copied by group g mod 4, eight lanes per 128-byte row
            // segment, so that stages complete independently of one another.
            const int pw = warp < kWarpMMA ? warp : (warp < 8 ? warp - 1 : warp - 10);  // 0..7
            const int grp = pw / kSGroup, gw = pw % kSGroup;
            constexpr int kNGroups = kSProd / kSGroup;
            constexpr int kFills = kDqk / 64;  // per tile
            bool ok = true;
            int g0 = 0, j0 = 0;  // fills and tiles so far
            QuadItem it;
            for (ItemWalk wk = walk_init(sm.h, cid, C); ok && walk_next(wk, a, sm.h, nrb, n_items, C, cid, it);) {
                if (it.ntiles <= 0) continue;
                const int nfill = it.ntiles * kFills;
                int seen = -1;  // last tile whose pool rows this warp has waited for
                for (int g = g0 + (grp - g0 % kNGroups + kNGroups) % kNGroups; ok && g < g0 + nfill;
                     g += kNGroups) {
                    const int jt = j0 + (g - g0) / kFills, kbk = (g - g0) % kFills;
                    const int rs = jt % kRowsRing;
                    const int st = g % kKStages;
                    if (jt != seen) {
                        if (!warp_wait(S.rows_full[rs], (jt / kRowsRing) & 1, abort_p)) {
                            ok = false;
                            break;
                        }
                        seen = jt;
                    }
                    if (g >= kKStages && !warp_wait(S.k_empty[st], ((g / kKStages) - 1) & 1, abort_p)) {
                        ok = false;
                        break;
                    }
                    const int32_t* my_rows = S.rows[rs] + hr * kNh;
                    const uint32_t dst0 = smem_u32(S.kring[st]);
                    for (int r = gw; r < kNh / 4; r += kSGroup) {
                        const int key = r * 4 + (lane >> 3), c = lane & 7;
                        const int32_t slot = my_rows[key];
                        const __nv_bfloat16* src =
                            a.kv + (slot >= 0 ? (int64_t)slot * kDqk : 0) + kbk * 64 + c * 8;
                        cp_async_16_zfill_nc(dst0 + sw128_offset(key, c), src, slot >= 0);
                    }
                    cp_async_mbar_arrive_noinc(ba(S.k_full[st]));
                }
                g0 += nfill;
                j0 += it.ntiles;
            }
            cp_async_wait_all();
        } else if (warp == kWarpCtl) {
            // ------------------------------------------------ tile metadata + P sender
            // The warp stages each tile's pool rows (all 256, with validity
            // bits for the softmax) three tiles ahead of the P it sends, across
            // item boundaries; lane 0 sends each tile's P (and rescale
            // factors) from the staging tile to the O partner's slot once that
            // slot is free, then hands the staging tile back to the softmax.
            // Slot j % 4 last held tile j - 4; the softmax has released that
            // tile's validity bits only after its S tile was complete, i.e.
            // after every producer had issued every stage of it, so the pool
            // rows are free as well.
            static_assert(kRowsRing == kMetaRing, "rows and metadata share the release");
            TileCursor cur;
            cursor_init(cur, sm.h, cid, C);
            int staged = 0;
            auto stage_next = [&]() -> int {  // 1: staged, 0: no tile left, -1: timed out
                if (!cursor_next(cur, a, sm.h, nrb, n_items, C, cid)) return 0;
                const int j = staged;
                const int rs = j % kRowsRing, mi = j % kMetaRing;
                if (j >= kMetaRing && !warp_wait(S.meta_free[mi], ((j / kMetaRing) - 1) & 1, abort_p))
                    return -1;
                bad |= stage_rows<kNT>(a, cur.b, key_base(a, cur.b), cur.Lb, cur.kb + cur.i * kNT, cur.ke, lane,
                                  S.rows[rs], S.valid[mi]);
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(ba(S.meta_full[mi]));
                    mbar_arrive(ba(S.rows_full[rs]));
                }
                ++staged;
                return 1;
            };
            const uint32_t p_local = smem_u32(S.pstage);
            const uint32_t orank = 2u + hr;
            // Slot j % 4 is restaged for tile j + 3 once the softmax has read
            // tile j - 1's bits, which it has when P of tile j - 1 is sent.
            int more = stage_next();
            if (more > 0) more = stage_next();
            if (more > 0) more = stage_next();
            bool ok = more >= 0;
            for (int j = 0; ok && j < staged; ++j) {
                if (more > 0) {
                    more = stage_next();
                    if (more < 0) break;
                }
                int sent = 1;
                if (lane == 0) {
                    const int slot = j & 1;
                    sent = mbar_wait_spin(ba(S.pw_bar[slot]), (j >> 1) & 1, abort_p);
                    if (sent && j >= 2) sent = mbar_wait_spin(ba(S.p_free[slot]), ((j - 2) >> 1) & 1, abort_p);
                    if (sent) {
                        const uint32_t dst = mapa_shared(smem_u32(sm.u.o.pbuf[slot]), orank);
                        const uint32_t bar = mapa_shared(ba(sm.u.o.p_full[slot]), orank);
                        mbar_arrive_expect_tx_remote(bar, kPXfer);
#pragma unroll
                        for (int blk = 0; blk < 4; ++blk)
                            bulk_copy_to_peer(dst + blk * kPBlock, p_local + blk * kPBlock, kPBlock, bar);
                        bulk_copy_to_peer(dst + kPBytes, p_local + kPBytes, kMh * 4, bar);
                        bulk_commit();
                        bulk_wait_read<0>();
                        mbar_arrive(ba(S.pstage_free));
                    }
                }
                ok = __shfl_sync(0xffffffffu, sent, 0) != 0;
            }
            if (lane == 0) bulk_wait_all();
            bad |= cur.bad;
        } else if (warp == kWarpMMA && rank == 0) {
            // ------------------------------------------------ S MMA issuer (pair)
            // The issue loop is kept free of per-MMA descriptor construction
            // and branches: a pair MMA takes about 128 cycles, and any work the
            // issuing thread does between MMAs is lost tensor time.
            if (lane == 0) {
                const uint32_t idesc = make_idesc_bf16(kRowsBlk, kNT, false, false);
                const uint32_t dS = tbase + kColS;
                const uint64_t kdesc0 = make_sdesc(smem_u32(S.kring[0]), 16, 1024, kSwizzle128B);
                const uint64_t qrdesc = make_sdesc(smem_u32(S.q_rope), 16, 1024, kSwizzle128B);
                const uint32_t kready0 = ba(S.k_ready[0]), kempty0 = ba(S.k_empty[0]);
                int st = 0, jt = 0, ne = 0;  // ring stage, tiles and non-empty items so far
                uint32_t ph = 0;
                bool ok = true;
                QuadItem it;
                for (ItemWalk wk = walk_init(sm.h, cid, C); ok && walk_next(wk, a, sm.h, nrb, n_items, C, cid, it);) {
                    if (it.ntiles <= 0) continue;
                    ok = mbar_wait_spin(ba(S.q_ready), ne & 1, abort_p) &&
                         mbar_wait_spin(ba(S.q_peer), ne & 1, abort_p);
                    fence_proxy_async_smem();
                    tc_fence_after();
                    for (int i = 0; ok && i < it.ntiles; ++i, ++jt) {
                        if (jt >= 1 && !mbar_wait_spin(ba(S.s_free), (jt - 1) & 1, abort_p)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll 1
                        for (int kbk = 0; kbk < kDqk / 64; ++kbk) {
                            // both CTAs' copies landed, each fenced for the
                            // tensor cores by its forwarder
                            if (!mbar_wait_spin(kready0 + 8 * st, ph, abort_p)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint64_t bd = kdesc0 + (uint64_t)(st * (kKBlock >> 4));
                            if (kbk < 8) {  // latent dims: A = Q from TMEM
                                const uint32_t aa = tbase + kColQ + kbk * 32;
                                mma_ts_pair(dS, aa, bd, idesc, kbk > 0 ? 1u : 0u);
                                mma_ts_pair(dS, aa + 8, bd + 2, idesc, 1u);
                                mma_ts_pair(dS, aa + 16, bd + 4, idesc, 1u);
                                mma_ts_pair(dS, aa + 24, bd + 6, idesc, 1u);
                            } else {        // RoPE dims: A = Q's RoPE tile in shared memory
                                mma_ss_pair(dS, qrdesc, bd, idesc, 1u);
                                mma_ss_pair(dS, qrdesc + 2, bd + 2, idesc, 1u);
                                mma_ss_pair(dS, qrdesc + 4, bd + 4, idesc, 1u);
                                mma_ss_pair(dS, qrdesc + 6, bd + 6, idesc, 1u);
                            }
                            mma_commit_pair_mc(kempty0 + 8 * st, 0x3);
                            if (++st == kKStages) {
                                st = 0;
                                ph ^= 1u;
                            }
                        }
                        if (ok) mma_commit_pair_mc(ba(S.s_full), 0x3);
                    }
                    ++ne;
                }
                mma_commit_pair_mc(ba(sm.h.drain), 0x1);
                mbar_wait(ba(sm.h.drain), 0, &sm.h.no_abort);
            }
        } else if (warp == kWarpFwd && rank == 0) {
            // ------------------------------------------------ rank 0: fence each landed stage
            // Copies complete on this CTA's own barriers; this thread orders
            // each filled stage for the tensor cores (proxy fence) and tells
            // the MMA issuer, off the issuer's path.
            if (lane == 0) {
                int g = 0;
                bool ok = true;
                QuadItem it;
                for (ItemWalk wk = walk_init(sm.h, cid, C); ok && walk_next(wk, a, sm.h, nrb, n_items, C, cid, it);) {
                    if (it.ntiles <= 0) continue;
                    const int gend = g + it.ntiles * (kDqk / 64);
                    for (; ok && g < gend; ++g) {
                        const int st = g % kKStages;
                        if (!mbar_wait_spin(ba(S.k_full[st]), (g / kKStages) & 1, abort_p)) {
                            ok = false;
                            break;
                        }
                        fence_proxy_async_smem();
                        mbar_arrive(ba(S.k_ready[st]));
                    }
                }
            }
        } else if (warp == kWarpMMA) {
            // ------------------------------------------------ rank 1: forward readiness to rank 0
            // Copies complete on this CTA's own barriers; rank 0's MMA issuer
            // learns of each filled K stage (and of this CTA's Q) through
            // this thread.
            if (lane == 0) {
                int g = 0, ne = 0;
                bool ok = true;
                QuadItem it;
                for (ItemWalk wk = walk_init(sm.h, cid, C); ok && walk_next(wk, a, sm.h, nrb, n_items, C, cid, it);) {
                    if (it.ntiles <= 0) continue;
                    ok = mbar_wait_spin(ba(S.q_ready), ne & 1, abort_p);
                    tc_fence_after();
                    tc_fence_before();
                    if (ok) mbar_arrive_remote(mapa_shared(ba(S.q_peer), 0));
                    const int gend = g + it.ntiles * (kDqk / 64);
                    for (; ok && g < gend; ++g) {
                        const int st = g % kKStages;
                        if (!mbar_wait_spin(ba(S.k_full[st]), (g / kKStages) & 1, abort_p)) {
                            ok = false;
                            break;
                        }
                        fence_proxy_async_smem();
                        mbar_arrive_remote(mapa_shared(ba(S.k_ready[st]), 0));
                    }
                    ++ne;
                }
            }
        }
        __syncwarp();
    } else if (sside) {
        regs_inc<kRegsSoftmax>();
        SmemS& S = sm.u.s;
        {
            // ------------------------------------------------ softmax (warps 8-15)
            const int quarter = warp & 3;
            const int half = (warp - 8) >> 2;     // 128-key half of the tile
            const int r = 32 * quarter + lane;     // row = TMEM lane
            const uint32_t lb = (uint32_t)(32 * quarter) << 16;
            const int stid = tid - 256;            // 0..255
            const uint32_t orank = 2u + hr;        // O partner holding the same rows
            const uint32_t sfree0 = mapa_shared(ba(S.s_free), 0);
            const uint32_t p_local = smem_u32(S.pstage);
            float* alpha_local = reinterpret_cast<float*>(S.pstage + kPBytes);
            const float sl = a.scale_log2;
            bool ok = true;
            int jt = 0, ne = 0;  // tiles and non-empty items so far
            QuadItem it;
            for (ItemWalk wk = walk_init(sm.h, cid, C); ok && walk_next(wk, a, sm.h, nrb, n_items, C, cid, it);) {
                if (it.ntiles <= 0) continue;
                const int b = it.b;
                const int row0 = it.rb * kRowsBlk + (int)hr * kMh;  // first request row of this CTA
                const int grow = row0 + r;
                const bool row_ok = grow < rows_req;
                const int t = row_ok ? grow / H : 0;
                // Q staging: RoPE dims into their swizzled A-operand tile by
                // cp.async; latent dims straight from global memory into TMEM
                // (each thread its row's 256 dims of this half), so the K ring
                // is never used for Q and the copy warps run on into the next
                // item's keys. The previous item's MMAs are complete (its last
                // S tile was waited for), so neither TMEM's Q columns nor the
                // RoPE tile are still being read.
                {
                    // the item's key slots into L2 for the row staging of its tiles
                    if (warp == 8) key_prefetch(a, b, key_base(a, b), it.Lb, it.kb, it.ke, lane);
                    const __nv_bfloat16* q0 = a.q + ((int64_t)b * rows_req + row0) * kDqk;
                    for (int f = stid; f < kMh * 8; f += 256) {
                        const int rr = f >> 3, c = f & 7;
                        const bool v = row0 + rr < rows_req;
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
                    // The softmax warps meet on mbarriers (bounded waits), not
                    // on a named barrier: a warp that gave up on a timed-out
                    // wait must not leave the others blocked for good.
                    cp_async_wait_all();
                    mbar_arrive(ba(S.q_landed));
                    if (!warp_wait(S.q_landed, ne & 1, abort_p)) {
                        ok = false;
                        break;
                    }
                    if (stid == 0 && a.anc_mask == nullptr) bad |= build_anc_serial(S.par, T, S.anc);
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(ba(S.q_ready));  // also orders the masks built above
                    if (!warp_wait(S.q_ready, ne & 1, abort_p)) {
                        ok = false;
                        break;
                    }
                }
                const uint64_t anc_t = S.anc[t] & tree_bits(T);
                float m_ref = -INFINITY, l_part = 0.f;
                for (int i = 0; i < it.ntiles; ++i, ++jt) {
                    if (!warp_wait(S.s_full, jt & 1, abort_p)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    float sc[128];
                    {
                        uint32_t w[4][32];
#pragma unroll
                        for (int c = 0; c < 4; ++c) tmem_ld32(tbase + lb + kColS + half * 128 + c * 32, w[c]);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int u = 0; u < 32; ++u) sc[c * 32 + u] = __uint_as_float(w[c][u]);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_remote(sfree0);
                    const int mi = jt % kMetaRing;
                    if (!warp_wait(S.meta_full[mi], (jt / kMetaRing) & 1, abort_p)) {
                        ok = false;
                        break;
                    }
                    uint32_t vw[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) vw[q] = row_ok ? S.valid[mi][4 * half + q] : 0u;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ba(S.meta_free[mi]));
                    const int k0 = it.kb + i * kNT + 128 * half;
                    if (k0 + 128 > it.Lb) {  // this half reaches the tree keys
#pragma unroll
                        for (int q = 0; q < 4; ++q) vw[q] &= tree_keep_word(anc_t, k0 + 32 * q - it.Lb);
                    }
                    // Max over the raw scores (the scale is positive, so scaling
                    // the max is exact); masked keys become -inf only where this
                    // row's half-tile has any.
                    float mx = -INFINITY;
                    if ((vw[0] & vw[1] & vw[2] & vw[3]) != 0xffffffffu) {
#pragma unroll
                        for (int c = 0; c < 128; ++c)
                            if (!((vw[c >> 5] >> (c & 31)) & 1u)) sc[c] = -INFINITY;
                    }
                    mx = max128(sc);
                    mx *= sl;
                    S.mx[jt & 1][half][r] = mx;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ba(S.mx_bar[jt & 1]));
                    if (!warp_wait(S.mx_bar[jt & 1], (jt >> 1) & 1, abort_p)) {
                        ok = false;
                        break;
                    }
                    const float mt = fmaxf(mx, S.mx[jt & 1][half ^ 1][r]);
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
                    // P (bf16) -> local staging tile (the O pair's A-operand
                    // layout), once the previous tile's P has been read out of it.
                    if (jt >= 1 && !warp_wait(S.pstage_free, (jt - 1) & 1, abort_p)) {
                        ok = false;
                        break;
                    }
                    // p = 2^(s * scale_log2 - m_ref), one packed FMA per two
                    // keys; masked keys (-inf) give 2^-inf = 0, and a row with
                    // no visible key yet (m_ref = -inf: every key of the tile
                    // masked) writes zeros. Sums in four chains of key pairs.
                    const float nm = m_ref == -INFINITY ? 0.f : -m_ref;
                    const uint64_t sl2 = f2_pack(sl, sl), nm2 = f2_pack(nm, nm);
                    uint64_t ps4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                    for (int blk = 0; blk < 2; ++blk) {
                        const uint32_t pb = p_local + (2 * half + blk) * kPBlock;
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            uint32_t w[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int kk = blk * 64 + c * 8 + 2 * u;
                                float y0, y1;
                                f2_unpack(f2_fma(f2_pack(sc[kk], sc[kk + 1]), sl2, nm2), y0, y1);
                                const float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
                                uint64_t& acc = ps4[(c & 1) * 2 + (u & 1)];
                                acc = f2_add(acc, f2_pack(p0, p1));
                                w[u] = pack_bf16x2(p0, p1);
                            }
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(pb + sw128_offset(r, c)),
                                         "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                                         : "memory");
                        }
                    }
                    {
                        float q[8];
#pragma unroll
                        for (int j = 0; j < 4; ++j) f2_unpack(ps4[j], q[2 * j], q[2 * j + 1]);
                        l_part += ((q[0] + q[1]) + (q[2] + q[3])) + ((q[4] + q[5]) + (q[6] + q[7]));
                    }
                    if (half == 0) alpha_local[r] = alpha;
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ba(S.pw_bar[jt & 1]));
                }
                if (!ok) break;
                // The item's row maxima and sums go to the O partner's slot of
                // this item's parity, once the partner has read what the item
                // two before left there.
                const int fs = ne & 1;
                if (ne >= 2 && !warp_wait(S.fin_free[fs], ((ne - 2) >> 1) & 1, abort_p)) {
                    ok = false;
                    break;
                }
                if (half == 0) {
                    st_cluster_f32(mapa_shared(smem_u32(&sm.u.o.fin_m[fs][r]), orank), m_ref);
                    st_cluster_f32(mapa_shared(smem_u32(&sm.u.o.fin_l[fs][0][r]), orank), l_part);
                } else {
                    st_cluster_f32(mapa_shared(smem_u32(&sm.u.o.fin_l[fs][1][r]), orank), l_part);
                }
                mbar_arrive_cluster(mapa_shared(ba(sm.u.o.fin[fs]), orank));
                ++ne;
            }
        }
    } else if (wg != 2) {
        // (the O CTAs keep the 96 launch registers: no role there needs more)
        SmemO& O = sm.u.o;
        if (warp != kWarpMMA && warp != kWarpCtl) {
            // ------------------------------------------------ O producers: V segments
            // Warps 0-3, 5, 6 and 12-19 copy, for 32 keys per stage, this
            // CTA's four 64-dim segments (eight lanes per 128-byte segment).
            const int pw = warp < kWarpMMA ? warp : (warp < 8 ? warp - 1 : warp - 6);  // 0..13
            bool ok = true;
            int jt = 0;  // tiles so far
            QuadItem it;
            for (ItemWalk wk = walk_init(sm.h, cid, C); ok && walk_next(wk, a, sm.h, nrb, n_items, C, cid, it);) {
                for (int i = 0; ok && i < it.ntiles; ++i, ++jt) {
                    const int rs = jt % kRowsRing;
                    if (!warp_wait(O.rows_full[rs], (jt / kRowsRing) & 1, abort_p)) {
                        ok = false;
                        break;
                    }
                    for (int q = 0; q < kNT / kVKeys; ++q) {
                        const int g = jt * (kNT / kVKeys) + q;
                        const int st = g % kVStages;
                        if (g >= kVStages && !warp_wait(O.v_empty[st], ((g / kVStages) - 1) & 1, abort_p)) {
                            ok = false;
                            break;
                        }
                        const uint32_t dst0 = smem_u32(O.vring[st]);
                        for (int x = pw; x < kVKeys * 4 * 8 / 32; x += kOProd) {
                            const int idx = x * 32 + lane;
                            const int chunk = idx & 7, pair = idx >> 3;
                            const int kl = pair >> 2, sel = pair & 3;   // key in stage; (chain, segment)
                            const int seg = 4 * (sel >> 1) + 2 * (int)hr + (sel & 1);
                            const int32_t slot = O.rows[rs][kVKeys * q + kl];
                            const __nv_bfloat16* src =
                                a.kv + (slot >= 0 ? (int64_t)slot * kDqk : 0) + seg * 64 + chunk * 8;
                            cp_async_16_zfill_nc(dst0 + sel * kVSub + sw128_offset(kl, chunk), src, slot >= 0);
                        }
                        cp_async_mbar_arrive_noinc(ba(O.v_full[st]));
                    }
                    if (!ok) break;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ba(O.rows_free[rs]));
                }
            }
            cp_async_wait_all();
        } else if (warp == kWarpCtl) {
            // ------------------------------------------------ tile rows + P slot release
            // The warp stages each tile's pool rows two tiles ahead of the
            // copies, across item boundaries; on rank 2, lane 0 frees P
            // slots: once P V of tile j is complete, its slot may take tile
            // j + 2.
            TileCursor cur;
            cursor_init(cur, sm.h, cid, C);
            int staged = 0;
            auto stage_next = [&]() -> int {  // 1: staged, 0: no tile left, -1: timed out
                if (!cursor_next(cur, a, sm.h, nrb, n_items, C, cid)) return 0;
                const int j = staged;
                const int rs = j % kRowsRing;
                if (j >= kRowsRing && !warp_wait(O.rows_free[rs], ((j / kRowsRing) - 1) & 1, abort_p))
                    return -1;
                (void)stage_rows<kNT>(a, cur.b, key_base(a, cur.b), cur.Lb, cur.kb + cur.i * kNT, cur.ke, lane,
                                 O.rows[rs], nullptr);
                __syncwarp();
                if (lane == 0) mbar_arrive(ba(O.rows_full[rs]));
                ++staged;
                return 1;
            };
            int more = stage_next();
            if (more > 0) more = stage_next();
            bool ok = more >= 0;
            for (int j = 0; ok && j < staged; ++j) {
                if (more > 0) {
                    more = stage_next();
                    if (more < 0) break;
                }
                int rel = 1;
                if (rank == 2 && lane == 0 && j + 2 < staged) {
                    rel = mbar_wait_spin(ba(O.o_done[j & 1]), (j >> 1) & 1, abort_p);
                    if (rel) {
                        mbar_arrive_remote(mapa_shared(ba(sm.u.s.p_free[j & 1]), 0));
                        mbar_arrive_remote(mapa_shared(ba(sm.u.s.p_free[j & 1]), 1));
                    }
                }
                ok = __shfl_sync(0xffffffffu, rel, 0) != 0;
            }
        } else if (rank == 2) {
            // ------------------------------------------------ O MMA issuer (pair)
            // Descriptors are precomputed; the loop only adds offsets.
            if (lane == 0) {
                const uint32_t idesc = make_idesc_bf16(kRowsBlk, 256, false, true);
                const uint64_t pdesc0 = make_sdesc(smem_u32(O.pbuf[0]), 16, 1024, kSwizzle128B);
                const uint64_t vdesc0 = make_sdesc(smem_u32(O.vring[0]), kVSub, 1024, kSwizzle128B);
                const uint32_t vfull0 = ba(O.v_full[0]), vempty0 = ba(O.v_empty[0]);
                const uint32_t d0 = tbase, d1 = tbase + 256;
                int st = 0, jt = 0;
                uint32_t ph = 0;
                bool ok = true;
                QuadItem it;
                for (ItemWalk wk = walk_init(sm.h, cid, C); ok && walk_next(wk, a, sm.h, nrb, n_items, C, cid, it);) {
                    for (int i = 0; ok && i < it.ntiles; ++i, ++jt) {
                        const int slot = jt & 1;
                        if (!mbar_wait_spin(ba(O.o_gate[slot]), (jt >> 1) & 1, abort_p)) {
                            ok = false;
                            break;
                        }
                        fence_proxy_async_smem();
                        tc_fence_after();
                        const uint64_t pd = pdesc0 + (uint64_t)(slot * (kPSlot >> 4));
#pragma unroll 1
                        for (int q = 0; q < kNT / kVKeys; ++q) {
                            if (!mbar_wait_spin(vfull0 + 8 * st, ph, abort_p)) {
                                ok = false;
                                break;
                            }
                            fence_proxy_async_smem();
                            tc_fence_after();
                            const uint64_t vd = vdesc0 + (uint64_t)(st * (kVStage >> 4));
                            // keys q*32 .. q*32+31 of the tile: P block q/2, 32-byte K steps
                            const uint64_t ad = pd + (uint64_t)((q >> 1) * (kPBlock >> 4) + (q & 1) * 4);
                            const uint32_t acc0 = (i > 0 || q > 0) ? 1u : 0u;  // each item starts afresh
                            mma_ss_pair(d0, ad, vd, idesc, acc0);
                            mma_ss_pair(d1, ad, vd + (2 * kVSub >> 4), idesc, acc0);
                            mma_ss_pair(d0, ad + 2, vd + (2048 >> 4), idesc, 1u);
                            mma_ss_pair(d1, ad + 2, vd + ((2 * kVSub + 2048) >> 4), idesc, 1u);
                            mma_commit_pair_mc(vempty0 + 8 * st, 0xC);
                            if (++st == kVStages) {
                                st = 0;
                                ph ^= 1u;
                            }
                        }
                        if (!ok) break;
                        mma_commit_pair_mc(ba(O.o_done[slot]), 0xC);
                    }
                }
                mma_commit_pair_mc(ba(sm.h.drain), 0x4);
                mbar_wait(ba(sm.h.drain), 0, &sm.h.no_abort);
            }
        } else {
            // ------------------------------------------------ rank 3: forward V readiness to rank 2
            if (lane == 0) {
                int g = 0;
                bool ok = true;
                QuadItem it;
                for (ItemWalk wk = walk_init(sm.h, cid, C); ok && walk_next(wk, a, sm.h, nrb, n_items, C, cid, it);) {
                    const int gend = g + it.ntiles * (kNT / kVKeys);
                    for (; g < gend; ++g) {
                        const int st = g % kVStages;
                        if (!mbar_wait_spin(ba(O.v_full[st]), (g / kVStages) & 1, abort_p)) {
                            ok = false;
                            break;
                        }
                        fence_proxy_async_smem();
                        mbar_arrive_remote(mapa_shared(ba(O.v_full[st]), 2));
                    }
                }
            }
        }
        __syncwarp();
    } else {
        SmemO& O = sm.u.o;
        {
            // ------------------------------------------------ correction + epilogue
            const int quarter = warp & 3;
            const int r = 32 * quarter + lane;
            const uint32_t lb = (uint32_t)(32 * quarter) << 16;
            const uint32_t srank = hr;  // S partner holding the same rows
            float* tile = O.otile[quarter];
            if (sm.h.balanced) {
                // The partitions past a (request, row block) pair's last
                // part get lse = -inf; the cluster holding the pair's first
                // tile writes them (or, for a pair without tiles, the
                // cluster holding the tile at its place in the sequence).
                const int w = sm.h.w;
                const int e1 = plan_begin(cid + 1, C, w);
                for (int b = 0; b < a.batch; ++b) {
                    const int p0 = sm.h.ptile[b], p1 = sm.h.ptile[b + 1];
                    if (p0 >= e1 && !(p0 >= w && cid == C - 1)) break;  // pairs start in order
                    if (p1 <= plan_begin(cid, C, w) && p1 > p0) continue;
                    const int t = (p1 - p0) / nrb;
                    for (int rb = 0; rb < nrb; ++rb) {
                        const int s0 = p0 + rb * t;
                        if (plan_pair_owner(s0, t, C, w) != cid) continue;
                        const int parts = plan_pair_parts(s0, t, C, w);
                        const int grow = rb * kRowsBlk + (int)hr * kMh + r;
                        if (grow >= rows_req) continue;
                        float* lp = a.lse_part + ((int64_t)b * rows_req + grow) * a.nsplit;
                        for (int p = parts; p < a.nsplit; ++p) lp[p] = -INFINITY;
                    }
                }
            }
            bool ok = true;
            int jt = 0, ne = 0;  // tiles and non-empty items so far
            QuadItem it;
            for (ItemWalk wk = walk_init(sm.h, cid, C); ok && walk_next(wk, a, sm.h, nrb, n_items, C, cid, it);) {
                const int row0 = it.rb * kRowsBlk + (int)hr * kMh;
                const int grow = row0 + r;
                const bool row_ok = grow < rows_req;
                if (it.ntiles <= 0) {  // empty split: lse = -inf, o = 0
                    if (row_ok) {
                        const int64_t pid = ((int64_t)it.b * rows_req + grow) * a.nsplit + it.s;
                        float4* o = reinterpret_cast<float4*>(a.o_part + pid * kDv);
                        for (int c = 0; c < kDv / 4; ++c) o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                        a.lse_part[pid] = -INFINITY;
                    }
                    continue;
                }
                for (int i = 0; i < it.ntiles; ++i, ++jt) {
                    const int slot = jt & 1;
                    if (!warp_wait(O.p_full[slot], (jt >> 1) & 1, abort_p)) {
                        ok = false;
                        break;
                    }
                    const float alpha = reinterpret_cast<const float*>(O.pbuf[slot] + kPBytes)[r];
                    if (__any_sync(0xffffffffu, alpha != 1.f) && i > 0) {
                        if (!warp_wait(O.o_done[slot ^ 1], ((jt - 1) >> 1) & 1, abort_p)) {
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
                    __syncwarp();
                    if (lane == 0) mbar_arrive_remote(mapa_shared(ba(O.o_gate[slot]), 2));
                }
                if (!ok) break;
                const int fs = ne & 1;
                ok = warp_wait_cluster(O.fin[fs], (ne >> 1) & 1, abort_p) &&
                     warp_wait(O.o_done[(jt - 1) & 1], ((jt - 1) >> 1) & 1, abort_p);
                if (!ok) break;
                tc_fence_after();
                const float l = O.fin_l[fs][0][r] + O.fin_l[fs][1][r];
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const float lse = l > 0.f ? (O.fin_m[fs][r] + log2f(l)) * kLn2 : -INFINITY;
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(mapa_shared(ba(sm.u.s.fin_free[fs]), srank));
                // The partial write, coalesced through the warp's transpose
                // tile. (Spreading the last item's write over the idle copy
                // warps as well was measured slower: the write is bound by
                // the SM's store throughput, not by the issuing warps.)
                write_o_cols(a, it, rows_req, row0 + 32 * quarter, tbase + lb, inv, tile, lane, 0, 512);
                if (row_ok) a.lse_part[((int64_t)it.b * rows_req + grow) * a.nsplit + it.s] = lse;
                ++ne;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // no CTA leaves while another may still touch its shared memory
    if (warp == kWarpMMA) {
        tc_fence_after();
        tmem_dealloc_pair(tbase, 512);
    }
    if (sm.h.abort_flag) bad |= MLA_STATUS_TIMEOUT;
    status_or(a.status, bad);
}

}  // namespace

// Resident 4-CTA clusters per device: the persistent launch's cluster count.
int g_quad_clusters[64];

cudaError_t setup_partial_quad() {
    cudaError_t e = cudaFuncSetAttribute(partial_quad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    int dev = -1;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(4, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, partial_quad_kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();  // unknown: one cluster per item
        n = 0;
    }
    g_quad_clusters[dev] = n;
    return cudaSuccess;
}

int quad_expected_parts(int batch, int T, int H, int nsplit) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nsplit;
    const int C = g_quad_clusters[dev];
    const long long pairs = (long long)batch * ((T * H + kRowsBlk - 1) / kRowsBlk);
    if (C <= 0 || batch > kPlanMaxReq) return nsplit;  // rotated rounds: any partition may hold keys
    const long long est = (C + pairs - 1) / pairs + 2;  // one range per cluster, plus its cut ends
    return est < nsplit ? (int)est : nsplit;
}

cudaError_t launch_partial_quad(const PartialArgs& a, cudaStream_t stream) {
    const int rows_req = a.T * a.H;
    const int nrb = (rows_req + kRowsBlk - 1) / kRowsBlk;
    const long long items = (long long)a.batch * a.nsplit * nrb;
    if (items <= 0 || items > (1ll << 30)) return cudaErrorInvalidValue;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
    const int resident = dev >= 0 && dev < 64 ? g_quad_clusters[dev] : 0;
    const int clusters = resident > 0 && resident < items ? resident : (int)items;
    PartialArgs w = a;
    w.wave_full = wave_full_items(items, clusters);
    return launch_pdl(partial_quad_kernel, dim3(4 * clusters, 1, 1), dim3(kThreads), kSmemBytes, stream, w);
}

}  // namespace mlav
