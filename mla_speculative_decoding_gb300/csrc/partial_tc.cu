// Split-KV partial attention on the tcgen05 tensor cores (TMEM accumulators).
//
// The verify attention of "The Custom sm_120 Verify Kernel..." (Parts VI,
// VII, IX): every tree token x head row of a request attends over the
// request's scattered latent KV rows; the pages' kernel is a KV-split
// "partial + reduce" design with 128-bit KV loads. Here the dense
// contractions S = Q K^T (576 dims) and O += P V (512 dims) run on tcgen05
// MMAs, and one gathered KV tile feeds all 128 query rows of a CTA.
//
// CTA = (128-row block of the request's T*H rows, one quarter of the 512 V
// columns, split s, request b). TMEM (512 columns x 128 lanes, lane = row):
//   Q  [0, 288)   the CTA's 128 query rows, bf16 pairs (A operand of Q K^T)
//   O  [288, 416) fp32 accumulator of this CTA's 128 V columns
//   S  [416, 480) two fp32 score buffers of 32 keys (double-buffered)
//   P  [480, 512) two bf16 probability buffers (A operand of P V)
// Q alone fills 288 columns and O for all 512 V columns would fill the whole
// TMEM, so the V columns are split over 4 CTAs that each recompute S.
//
// Warp roles (192 threads):
//   warp 0     producer: per tile of 32 keys, reads the slots, checks them,
//              and gathers the 1152-byte rows with 16-byte cp.async into a
//              128-byte-swizzled K-major tile (5-stage ring);
//   warp 1     TMEM owner and MMA issuer (one thread): S(i) = Q K_i^T,
//              then O += P(i-1) V_{i-1}, committing to mbarriers;
//   warps 2-5  softmax (thread = query row): read S(i) from TMEM, apply the
//              prefix/tree mask (tree mask only past the prefix, Part VII),
//              online softmax with a lazily updated reference max (O and l
//              are rescaled only when the tile max exceeds it by 2^8), write
//              P(i) as bf16 into TMEM; at the end normalise O and write the
//              partial (o, lse).
// Every wait is bounded (globaltimer); on a timeout the CTA drains its
// MMAs, frees TMEM, and flags MLA_STATUS_TIMEOUT instead of hanging.
#include "partial_tc.cuh"
#include "tc_ptx.cuh"

namespace mlav {
namespace {

using namespace tc;

constexpr int kM = 128;                 // query rows per CTA (MMA M)
constexpr int kDvPart = 128;            // V columns per CTA
constexpr int kParts = kDv / kDvPart;   // CTAs per row block
constexpr int kNK = 32;                 // keys per tile
constexpr int kStages = 5;
constexpr int kThreads = 192;
constexpr int kChunksPerRow = kDqk / 8;                // 72 x 16 B
constexpr uint32_t kKBlock = kNK * 128;                // one 64-dim block of a tile
constexpr uint32_t kStageBytes = (kDqk / 64) * kKBlock;  // 36,864
constexpr uint32_t kColQ = 0, kColO = 288, kColS = 416, kColP = 480, kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;

struct __align__(1024) SmemTC {
    unsigned char kv[kStages][kStageBytes];
    int32_t slot[kStages][kNK];
    uint32_t kvalid[kStages];
    uint64_t anc[MLA_MAX_TREE];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2];
    uint64_t q_ready, o_done, drain;
    uint32_t tmem_base;
    int abort_flag;
    int no_abort;
};

constexpr size_t kSmemBytes = sizeof(SmemTC) + 1024;

__device__ __forceinline__ uint32_t bar_addr(uint64_t& b) { return smem_u32(&b); }

// Warp-uniform bounded wait: all lanes wait, then agree.
__device__ __forceinline__ bool warp_wait(uint64_t& bar, uint32_t parity, volatile int* abort) {
    const bool ok = mbar_wait(bar_addr(bar), parity, abort);
    return __all_sync(0xffffffffu, ok);
}

__global__ void __launch_bounds__(kThreads, 1) partial_tc_kernel(const PartialArgs a) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    extern __shared__ __align__(1024) unsigned char raw[];
    unsigned char* base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
    SmemTC& sm = *reinterpret_cast<SmemTC*>(base);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int part = blockIdx.x % kParts;
    const int rb = blockIdx.x / kParts;
    const int s = blockIdx.y, b = blockIdx.z;
    const int T = a.T, H = a.H, rows_req = T * H;

    int Lb, K;
    int bad = request_keys(a, b, Lb, K);
    int kb, ke;
    split_range(K, a.nsplit, s, kb, ke);
    const int ntiles = (ke - kb + kNK - 1) / kNK;
    const int64_t kbase = key_base(a, b);

    if (ntiles <= 0) {  // empty split: lse = -inf, o = 0 (fixed grid, early exit)
        if (warp >= 2) {
            const int grow = rb * kM + 32 * (warp & 3) + lane;
            if (grow < rows_req) {
                const int64_t pid = ((int64_t)b * rows_req + grow) * a.nsplit + s;
                float4* o = reinterpret_cast<float4*>(a.o_part + pid * kDv + part * kDvPart);
                for (int c = 0; c < kDvPart / 4; ++c) o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (part == 0) a.lse_part[pid] = -INFINITY;
            }
        }
        if (tid == 0) status_or(a.status, bad);
        return;
    }

    if (warp == 1) {
        tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int st = 0; st < kStages; ++st) {
            mbar_init(bar_addr(sm.full[st]), 33);  // 32 cp.async arrivals + 1 for the slot mask
            mbar_init(bar_addr(sm.empty[st]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_addr(sm.s_full[i]), 1);
            mbar_init(bar_addr(sm.s_empty[i]), 128);
            mbar_init(bar_addr(sm.p_full[i]), 128);
            mbar_init(bar_addr(sm.p_empty[i]), 1);
        }
        mbar_init(bar_addr(sm.q_ready), 128);
        mbar_init(bar_addr(sm.o_done), 1);
        mbar_init(bar_addr(sm.drain), 1);
        sm.abort_flag = 0;
        sm.no_abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sm.tmem_base;
    volatile int* abort_p = &sm.abort_flag;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        for (int i = 0; i < ntiles; ++i) {
            const int st = i % kStages;
            if (i >= kStages && !warp_wait(sm.empty[st], ((i / kStages) - 1) & 1, abort_p)) break;
            const int j = kb + i * kNK + lane;
            int32_t sl = -1;
            if (j < ke) {
                sl = key_slot(a, b, kbase, Lb, j);
                if (sl < 0 || (int64_t)sl >= a.pool_slots) {
                    bad |= MLA_STATUS_BAD_SLOT;
                    sl = -1;
                }
            }
            sm.slot[st][lane] = sl;
            const uint32_t valid = __ballot_sync(0xffffffffu, sl >= 0);
            __syncwarp();
            const uint32_t dst0 = smem_u32(sm.kv[st]);
#pragma unroll 4
            for (int it = 0; it < kNK * kChunksPerRow / 32; ++it) {
                const int f = it * 32 + lane;
                const int key = f / kChunksPerRow, ch = f - key * kChunksPerRow;
                const int32_t ksl = sm.slot[st][key];
                const __nv_bfloat16* src = a.kv + (ksl >= 0 ? (int64_t)ksl * kDqk : 0) + ch * 8;
                cp_async_16_zfill(dst0 + (ch >> 3) * kKBlock + sw128_offset(key, ch & 7), src,
                                  ksl >= 0);
            }
            cp_async_mbar_arrive_noinc(bar_addr(sm.full[st]));
            if (lane == 0) {
                sm.kvalid[st] = valid;
                mbar_arrive(bar_addr(sm.full[st]));
            }
        }
        cp_async_wait_all();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc_qk = make_idesc_bf16(kM, kNK, false, false);
            const uint32_t idesc_pv = make_idesc_bf16(kM, kDvPart, false, true);
            bool ok = mbar_wait(bar_addr(sm.q_ready), 0, abort_p);
            tc_fence_after();
            auto issue_pv = [&](int jt) -> bool {
                const int pb = jt & 1;
                if (!mbar_wait(bar_addr(sm.p_full[pb]), (jt >> 1) & 1, abort_p)) return false;
                tc_fence_after();
                const uint32_t vbase = smem_u32(sm.kv[jt % kStages]) + part * 2 * kKBlock;
#pragma unroll
                for (int kk = 0; kk < kNK / 16; ++kk) {
                    const uint64_t bd = make_sdesc(vbase + kk * 16 * 128, kKBlock, 1024, kSwizzle128B);
                    mma_ts(tbase + kColO, tbase + kColP + pb * 16 + kk * 8, bd, idesc_pv,
                           (jt > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar_addr(sm.p_empty[pb]));
                mma_commit(bar_addr(sm.empty[jt % kStages]));
                return true;
            };
            for (int i = 0; ok && i < ntiles; ++i) {
                const int st = i % kStages;
                if (!mbar_wait(bar_addr(sm.full[st]), (i / kStages) & 1, abort_p)) {
                    ok = false;
                    break;
                }
                fence_proxy_async_smem();
                if (i >= 2 && !mbar_wait(bar_addr(sm.s_empty[i & 1]), ((i >> 1) - 1) & 1, abort_p)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t kt = smem_u32(sm.kv[st]);
                const uint32_t dS = tbase + kColS + (i & 1) * kNK;
#pragma unroll 4
                for (int ks = 0; ks < kDqk / 16; ++ks) {
                    const uint64_t bd =
                        make_sdesc(kt + (ks >> 2) * kKBlock + (ks & 3) * 32, 16, 1024, kSwizzle128B);
                    mma_ts(dS, tbase + kColQ + ks * 8, bd, idesc_qk, ks > 0 ? 1u : 0u);
                }
                mma_commit(bar_addr(sm.s_full[i & 1]));
                if (i >= 1 && !issue_pv(i - 1)) {
                    ok = false;
                    break;
                }
            }
            if (ok) issue_pv(ntiles - 1);
            mma_commit(bar_addr(sm.o_done));
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int quarter = warp & 3;
        const int r = 32 * quarter + lane;
        const int grow = rb * kM + r;
        const bool row_ok = grow < rows_req;
        const int t = row_ok ? grow / H : 0;
        const uint32_t lb = (uint32_t)(32 * quarter) << 16;

        if (warp == 2 && lane == 0) {
            if (a.anc_mask != nullptr) {
                for (int u = 0; u < T; ++u) sm.anc[u] = a.anc_mask[(int64_t)b * T + u];
            } else {
                bad |= build_anc_serial(a.tree_parent + (int64_t)b * T, T, sm.anc);
            }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");

        // This thread's query row -> TMEM (A operand of Q K^T).
        {
            const uint4* qsrc = reinterpret_cast<const uint4*>(
                a.q + ((int64_t)b * rows_req + (row_ok ? grow : 0)) * kDqk);
#pragma unroll 1
            for (int c = 0; c < kDqk / 64; ++c) {
                uint32_t w[32];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const uint4 v = row_ok ? __ldg(qsrc + c * 8 + u) : make_uint4(0, 0, 0, 0);
                    w[4 * u + 0] = v.x;
                    w[4 * u + 1] = v.y;
                    w[4 * u + 2] = v.z;
                    w[4 * u + 3] = v.w;
                }
                tmem_st32(tbase + lb + kColQ + c * 32, w);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar_addr(sm.q_ready));
        }
        const uint64_t anc_t = sm.anc[t];
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int i = 0; i < ntiles; ++i) {
            const int bi = i & 1;
            if (!warp_wait(sm.s_full[bi], (i >> 1) & 1, abort_p)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[32];
            tmem_ld32(tbase + lb + kColS + bi * kNK, sr);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar_addr(sm.s_empty[bi]));
            if (!warp_wait(sm.full[i % kStages], (i / kStages) & 1, abort_p)) {
                ok = false;
                break;
            }
            uint32_t vm = row_ok ? sm.kvalid[i % kStages] : 0u;
            const int k0 = kb + i * kNK;
            if (vm != 0u && k0 + kNK > Lb) {  // the tile reaches the tree keys: apply the tree mask
#pragma unroll
                for (int c = 0; c < kNK; ++c) {
                    const int u = k0 + c - Lb;
                    if (u >= 0 && !(u < T && ((anc_t >> u) & 1ull))) vm &= ~(1u << c);
                }
            }
            float sv[kNK];
            float mt = -INFINITY;
#pragma unroll
            for (int c = 0; c < kNK; ++c) {
                sv[c] = ((vm >> c) & 1u) ? __uint_as_float(sr[c]) * a.scale_log2 : -INFINITY;
                mt = fmaxf(mt, sv[c]);
            }
            float alpha = 1.f;
            bool need = false;
            if (mt > -INFINITY) {
                if (m_ref == -INFINITY) {
                    m_ref = mt;
                } else if (mt > m_ref + kRescaleLog2) {
                    alpha = exp2f(m_ref - mt);
                    m_ref = mt;
                    l *= alpha;
                    need = true;
                }
            }
            if (__any_sync(0xffffffffu, need)) {
                // Rescale this warp's O rows before P(i) V(i) accumulates into them;
                // the previous P V must have landed first.
                if (i >= 1 && !warp_wait(sm.p_empty[(i - 1) & 1], ((i - 1) >> 1) & 1, abort_p)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c0 = 0; c0 < kDvPart; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(tbase + lb + kColO + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                    tmem_st32(tbase + lb + kColO + c0, o);
                }
                tmem_wait_st();
            }
            uint32_t pk[kNK / 2];
            float psum = 0.f;
#pragma unroll
            for (int c = 0; c < kNK / 2; ++c) {
                const float p0 = ((vm >> (2 * c)) & 1u) ? exp2f(sv[2 * c] - m_ref) : 0.f;
                const float p1 = ((vm >> (2 * c + 1)) & 1u) ? exp2f(sv[2 * c + 1] - m_ref) : 0.f;
                psum += p0 + p1;
                pk[c] = pack_bf16x2(p0, p1);
            }
            l += psum;
            if (i >= 2 && !warp_wait(sm.p_empty[bi], ((i >> 1) - 1) & 1, abort_p)) {
                ok = false;
                break;
            }
            tc_fence_after();
            tmem_st16(tbase + lb + kColP + bi * 16, pk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar_addr(sm.p_full[bi]));
        }
        ok = warp_wait(sm.o_done, 0, abort_p) && ok;
        tc_fence_after();
        if (ok) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int64_t pid = ((int64_t)b * rows_req + (row_ok ? grow : 0)) * a.nsplit + s;
            float4* dst = reinterpret_cast<float4*>(a.o_part + pid * kDv + part * kDvPart);
#pragma unroll 1
            for (int c0 = 0; c0 < kDvPart; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(tbase + lb + kColO + c0, o);
                tmem_wait_ld();
                if (row_ok) {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        dst[c0 / 4 + u] = make_float4(
                            __uint_as_float(o[4 * u]) * inv, __uint_as_float(o[4 * u + 1]) * inv,
                            __uint_as_float(o[4 * u + 2]) * inv, __uint_as_float(o[4 * u + 3]) * inv);
                }
            }
            if (row_ok && part == 0)
                a.lse_part[pid] = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (sm.abort_flag) {
            // Make sure no MMA of this CTA is still in flight before freeing TMEM.
            if (lane == 0) {
                mma_commit(bar_addr(sm.drain));
                mbar_wait(bar_addr(sm.drain), 0, &sm.no_abort);
            }
            __syncwarp();
        }
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
    if (sm.abort_flag) bad |= MLA_STATUS_TIMEOUT;
    status_or(a.status, bad);
}

}  // namespace

bool partial_tc_supported(const PartialArgs&) { return true; }

cudaError_t setup_partial_tc() {
    return cudaFuncSetAttribute(partial_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemBytes);
}

cudaError_t launch_partial_tc(const PartialArgs& a, int /*sm_count*/, cudaStream_t stream) {
    const int rows_req = a.T * a.H;
    const int nrb = (rows_req + kM - 1) / kM;
    dim3 grid(nrb * kParts, a.nsplit, a.batch);
    return launch_pdl(partial_tc_kernel, grid, dim3(kThreads), kSmemBytes, stream, a);
}

}  // namespace mlav
