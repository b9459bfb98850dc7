// fp8 paged MQA indexer logits on the tcgen05 tensor cores (the operation is
// defined in mla_decode_steps.h; page "The Indexer Breakthrough", sections
// "The Technical Context" and "Design Decisions").
//
// One persistent CTA per SM. The work is the list of 128-position tiles (two
// 64-position pages) of every request, split evenly and contiguously over
// the CTAs. Per tile, one kind::f8f6f4 MMA chain computes
//   D[position][head] = sum_d k[position][d] * q[head][d]
// with M = 128 positions (TMEM lane = position), N = heads rounded up to 16,
// K = 128 (four MMAs of K = 32); the epilogue thread of each lane then forms
// scale * sum_h w[h] * max(0, D[h]) in a fixed order (four interleaved
// partial sums over the heads, then added pairwise). Nothing is
// reshaped to reach the tensor cores: the indexer's dot products are the
// contraction, and the kernel stays bound by the cache stream from HBM.
//
// Warp roles (320 threads):
//   warps 0-7  epilogue, two groups of four (TMEM lane quarters) taking
//              alternate tiles; first they write -inf over every position
//              past the last tile of each request
//   warp 8     producer: walks the tile list 32 tiles at a time (block-table
//              reads in parallel across lanes), loads each tile's two pages
//              by TMA (8 KB boxes, 128-byte swizzle) and their 256-byte scale
//              vectors by bulk copy into an 8-stage ring, and a request's
//              query rows into one of two B buffers when the request changes
//   warp 9     TMEM allocation; lane 0 issues the MMAs (four accumulators)
#include <cuda.h>

#include "common.cuh"
#include "mla_decode_steps.h"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace mlav {
namespace {

using namespace tc;

constexpr int kIxStages = 8;
constexpr int kIxAcc = 4;
constexpr int kIxEpiWarps = 8;
constexpr int kIxWarpProd = 8;
constexpr int kIxWarpMma = 9;
constexpr int kIxThreads = 320;
constexpr int kIxPage = 8192;              // 64 rows x 128 fp8 keys
constexpr int kIxBlock = 8448;             // + 64 fp32 scales
constexpr int kIxTile = 2 * kIxPage;

struct alignas(1024) IxSmem {
    uint8_t a[kIxStages][kIxTile];         // A: page 0 in rows 0-63, page 1 in rows 64-127
    uint8_t bq[2][128 * 128];              // B: query rows, rows >= H zero
    float scale[kIxStages][128];
    int4 tinfo[64];                        // tile k % 64: request, tile, good-page mask, length
    int2 tblk[64];                         // tile k % 64: the two pages' blocks
    int2 win[2][33];                       // producer's tile window (request, tile)
    uint64_t full[kIxStages], empty[kIxStages], bfull[2], bempty[2];
    uint64_t accfull[kIxAcc], accempty[kIxAcc], drain;
    uint32_t tmem;
    int abort;
    int b0, t0, n;
};

__device__ __forceinline__ int ix_pages(int len, int P) {
    return len <= 0 ? 0 : min((len >> 6) + ((len & 63) != 0), P);
}
__device__ __forceinline__ int ix_tiles(const int32_t* lens, int b, int P) {
    return (ix_pages(__ldg(lens + b), P) + 1) >> 1;
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += t;
    }
    return v;
}

// SM100 K-major 128-byte-swizzle operand: 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t ix_desc(uint32_t saddr) {
    return make_sdesc(saddr, 16, 1024, kSwizzle128B);
}

template <int NCH>  // 32-column chunks of the accumulator: H <= 32 * NCH
__global__ void __launch_bounds__(kIxThreads, 1)
fp8_indexer_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                      const uint8_t* __restrict__ kv, const float* __restrict__ w,
                      int64_t nblocks, const int32_t* __restrict__ bt,
                      const int32_t* __restrict__ lens, int batch, int H, int P,
                      float* __restrict__ out, int32_t* status) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    constexpr int kCols = 32 * NCH;                       // columns per accumulator
    constexpr uint32_t kAlloc = kCols * kIxAcc <= 128 ? 128 : (kCols * kIxAcc <= 256 ? 256 : 512);
    extern __shared__ uint8_t ix_raw[];
    IxSmem& S = *reinterpret_cast<IxSmem*>((reinterpret_cast<uintptr_t>(ix_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abort = &S.abort;
    const int N = (H + 15) & ~15;

    // ---------------------------------------------------------------- set-up
    if (warp == 0) {
        // total tiles, this CTA's contiguous share, and its first (request, tile)
        int total = 0;
        for (int base = 0; base < batch; base += 32) {
            int v = base + lane < batch ? ix_tiles(lens, base + lane, P) : 0;
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
            total += v;
        }
        int beg, end;
        split_range_tiles(total, gridDim.x, blockIdx.x, 1, beg, end);
        int b0 = batch, t0 = 0, run = 0;
        for (int base = 0; base < batch && b0 == batch && beg < end; base += 32) {
            const int v = base + lane < batch ? ix_tiles(lens, base + lane, P) : 0;
            const int incl = warp_incl_scan(v, lane);
            const unsigned m = __ballot_sync(0xffffffffu, run + incl > beg);
            if (m) {
                const int l = __ffs(m) - 1;
                b0 = base + l;
                t0 = beg - (run + __shfl_sync(0xffffffffu, incl - v, l));
            }
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            S.b0 = b0;
            S.t0 = t0;
            S.n = end - beg;
        }
    } else if (warp == kIxWarpProd) {
        if (lane == 0) {
            for (int i = 0; i < kIxStages; ++i) {
                mbar_init(smem_u32(&S.full[i]), 1);
                mbar_init(smem_u32(&S.empty[i]), 1 + 4);   // MMA commit + the epilogue group's warps
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(smem_u32(&S.bfull[i]), 1);
                mbar_init(smem_u32(&S.bempty[i]), 1);
            }
            for (int i = 0; i < kIxAcc; ++i) {
                mbar_init(smem_u32(&S.accfull[i]), 1);
                mbar_init(smem_u32(&S.accempty[i]), 4);
            }
            mbar_init(smem_u32(&S.drain), 1);
            S.abort = 0;
            fence_mbar_init();
            prefetch_tmap(&kmap);
            prefetch_tmap(&qmap);
        }
    } else if (warp == kIxWarpMma) {
        tmem_alloc(smem_u32(&S.tmem), kAlloc);
        tmem_relinquish();
    } else {
        // zero the query rows the TMA box does not cover (H..127) in both buffers
        const int t = tid - 32, nt = 7 * 32;
        const int chunks = (128 - H) * 8;
        for (int i = t; i < 2 * chunks; i += nt) {
            const int j = i / chunks, c = i - j * chunks;
            *reinterpret_cast<uint4*>(&S.bq[j][H * 128 + c * 16]) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;
    const int n = S.n;

    if (warp < kIxEpiWarps) {
        // ------------------------------------------------------------ epilogue
        // -inf over [128 * tiles_b, 64 * P) of every request, in float4s:
        // each CTA walks a contiguous share of the output rows.
        {
            const int64_t per = (int64_t)P * 16;
            const int64_t total = (int64_t)batch * per;
            const int64_t base = total / gridDim.x, rem = total % gridDim.x;
            const int64_t f1 = (int64_t)blockIdx.x * base + min((int64_t)blockIdx.x, rem) + base +
                               ((int64_t)blockIdx.x < rem ? 1 : 0);
            int64_t f = f1 - base - ((int64_t)blockIdx.x < rem ? 1 : 0) + tid;
            if (f < f1) {
                const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                float4* o4 = reinterpret_cast<float4*>(out);
                int b = (int)(f / per);
                int64_t j = f - (int64_t)b * per;
                int lim = 32 * ix_tiles(lens, b, P);
                for (; f < f1; f += kIxEpiWarps * 32) {
                    if (j >= lim) o4[f] = ninf;
                    j += kIxEpiWarps * 32;
                    while (j >= per) {
                        j -= per;
                        if (++b < batch) lim = 32 * ix_tiles(lens, b, P);
                    }
                }
            }
        }
        const int grp = warp >> 2, quarter = warp & 3;
        const int row = quarter * 32 + lane;              // TMEM lane = tile row
        // Weights of the current request: up to 64 heads held whole in every
        // thread (broadcast once per request), more lane-distributed (lane l:
        // heads l, l + 32, ...) and broadcast per use.
        constexpr bool kWholeW = NCH <= 2;
        int wreq = -1;
        float wl[NCH];
        float wr[kWholeW ? 32 * NCH : 1];
        for (int k = grp; k < n; k += 2) {
            const int s = k % kIxStages, a = k % kIxAcc;
            if (!mbar_wait_parked(smem_u32(&S.full[s]), (k / kIxStages) & 1, abort)) break;
            const int4 m = S.tinfo[k & 63];
            const float sc = S.scale[s][row];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&S.empty[s]));
            if (m.x != wreq) {                            // new request: its weights, one load per lane
                wreq = m.x;
#pragma unroll
                for (int c = 0; c < NCH; ++c)
                    wl[c] = 32 * c + lane < H ? __ldg(w + (int64_t)m.x * H + 32 * c + lane) : 0.f;
                if constexpr (kWholeW) {
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
#pragma unroll
                        for (int j = 0; j < 32; ++j) wr[32 * c + j] = __shfl_sync(0xffffffffu, wl[c], j);
                }
            }
            if (!mbar_wait_parked(smem_u32(&S.accfull[a]), (k / kIxAcc) & 1, abort)) break;
            tc_fence_after();
            uint32_t d[NCH][32];
            const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(a * kCols);
#pragma unroll
            for (int c = 0; c < NCH; ++c) tmem_ld32(ta + 32 * c, d[c]);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < NCH; ++c) tmem_reg_fence(d[c]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&S.accempty[a]));
            // four partial sums over heads h = 4i + r, added at the end
            float acc4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    float wh;
                    if constexpr (kWholeW) wh = wr[32 * c + j];
                    else wh = __shfl_sync(0xffffffffu, wl[c], j);
                    if (32 * c + j < H)
                        acc4[j & 3] = fmaf(wh, fmaxf(__uint_as_float(d[c][j]), 0.f), acc4[j & 3]);
                }
            }
            const float acc = (acc4[0] + acc4[1]) + (acc4[2] + acc4[3]);
            const int pos = 128 * m.y + row;
            if (pos < 64 * P) {
                const bool ok = pos < m.w && ((m.z >> (row >> 6)) & 1);
                out[(int64_t)m.x * P * 64 + pos] = ok ? sc * acc : -INFINITY;
            }
        }
    } else if (warp == kIxWarpProd) {
        // ------------------------------------------------------------ producer
        int wb = S.b0, wt = S.t0;
        int cur_b = -1, nb = 0, bad = 0;
        bool ok = true;
        int k = 0;
        for (int k0 = 0; k0 < n && ok; k0 += 32) {
            const int cnt = min(32, n - k0);
            int2* win = S.win[(k0 >> 5) & 1];
            // (request, tile) of window offsets 0..cnt, scattered by the requests covering them
            if (lane == 0) win[cnt] = make_int2(batch, 0);
            __syncwarp();
            int off = -wt;
            for (int rb = wb; rb < batch && off <= cnt; rb += 32) {
                const int r = rb + lane;
                const int v = r < batch ? ix_tiles(lens, r, P) : 0;
                const int incl = warp_incl_scan(v, lane);
                const int lo = off + incl - v, hi = off + incl;
                for (int o = max(lo, 0); o < min(hi, cnt + 1); ++o) win[o] = make_int2(r, o - lo);
                off += __shfl_sync(0xffffffffu, incl, 31);
            }
            __syncwarp();
            // this lane's tile: both pages' blocks and the good-page mask
            int tb = 0, tt = 0, len = 0, blk0 = -1, blk1 = -1, mask = 0;
            if (lane < cnt) {
                const int2 e = win[lane];
                tb = e.x;
                tt = e.y;
                len = __ldg(lens + tb);
                const int pages = ix_pages(len, P);
                const int32_t* row = bt + (int64_t)tb * P;
                if (2 * tt < pages) {
                    blk0 = __ldg(row + 2 * tt);
                    if (blk0 >= 0 && blk0 < nblocks) mask |= 1;
                    else bad = MLA_STATUS_BAD_SLOT;
                }
                if (2 * tt + 1 < pages) {
                    blk1 = __ldg(row + 2 * tt + 1);
                    if (blk1 >= 0 && blk1 < nblocks) mask |= 2;
                    else bad = MLA_STATUS_BAD_SLOT;
                }
            }
            const int2 nx = win[cnt];
            wb = nx.x;
            wt = nx.y;
            // The window's tile table, read by lane 0 below and by the MMA and
            // epilogue roles once the tile's stage is full. Entry k % 64 is
            // rewritten two windows later, after tile k + 32 was issued; that
            // needed tile k + 24's stage back (its MMA done), and that MMA
            // needed the accumulator of tile k + 20 released by the epilogue
            // group of tile k (same parity, in order): every reader is done.
            if (lane < cnt) {
                S.tinfo[(k0 + lane) & 63] = make_int4(tb, tt, mask, len);
                S.tblk[(k0 + lane) & 63] = make_int2(blk0, blk1);
            }
            __syncwarp();
            if (lane == 0) {
                for (int i = 0; i < cnt; ++i, ++k) {
                    const int4 ti = S.tinfo[k & 63];
                    const int2 tk = S.tblk[k & 63];
                    if (ti.x != cur_b) {
                        const int jb = nb & 1;
                        if (nb >= 2 && !mbar_wait(smem_u32(&S.bempty[jb]), ((nb >> 1) - 1) & 1, abort)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(smem_u32(&S.bfull[jb]), (uint32_t)H * 128);
                        tma_load_3d(smem_u32(S.bq[jb]), &qmap, 0, 0, ti.x, smem_u32(&S.bfull[jb]));
                        cur_b = ti.x;
                        ++nb;
                    }
                    const int s = k % kIxStages, lap = k / kIxStages;
                    if (lap >= 1 && !mbar_wait(smem_u32(&S.empty[s]), (lap - 1) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&S.full[s]);
                    mbar_arrive_expect_tx(fb, (uint32_t)__popc(ti.z) * (kIxPage + 256));
                    if (ti.z & 1) {
                        tma_load_3d(smem_u32(S.a[s]), &kmap, 0, 0, tk.x, fb);
                        bulk_load_g2s(smem_u32(S.scale[s]), kv + (int64_t)tk.x * kIxBlock + kIxPage, 256, fb);
                    }
                    if (ti.z & 2) {
                        tma_load_3d(smem_u32(S.a[s] + kIxPage), &kmap, 0, 0, tk.y, fb);
                        bulk_load_g2s(smem_u32(S.scale[s] + 64), kv + (int64_t)tk.y * kIxBlock + kIxPage, 256, fb);
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();
        }
        bad = __reduce_or_sync(0xffffffffu, bad);
        if (lane == 0) {
            if (bad) status_or(status, bad);
            // every issued copy has landed before the CTA may exit (only ever
            // waits on the abort path: consumers observed them all otherwise);
            // bounded on its own, whatever the abort flag says
            volatile int own = 0;
            for (int j = max(0, k - kIxStages); j < k; ++j)
                mbar_wait(smem_u32(&S.full[j % kIxStages]), (j / kIxStages) & 1, &own, 100000000ull);
            if (nb >= 1)
                mbar_wait(smem_u32(&S.bfull[(nb - 1) & 1]), ((nb - 1) >> 1) & 1, &own, 100000000ull);
            if (own) *abort = 1;
        }
    } else if (warp == kIxWarpMma && lane == 0) {
        // ------------------------------------------------------------ MMA issue
        const uint32_t idesc = make_idesc_e4m3(128, N);
        const uint64_t adesc0 = ix_desc(smem_u32(S.a[0]));
        const uint64_t bdesc0 = ix_desc(smem_u32(S.bq[0]));
        constexpr uint64_t kStageStep = kIxTile >> 4, kBStep = (128 * 128) >> 4;
        int cur_b = -1, nb = 0, jb = 0;
        for (int k = 0; k < n; ++k) {
            const int s = k % kIxStages, a = k % kIxAcc;
            if (!mbar_wait(smem_u32(&S.full[s]), (k / kIxStages) & 1, abort)) break;
            const int b = S.tinfo[k & 63].x;
            if (b != cur_b) {
                if (nb >= 1) mma_commit(smem_u32(&S.bempty[(nb - 1) & 1]));
                jb = nb & 1;
                if (!mbar_wait(smem_u32(&S.bfull[jb]), (nb >> 1) & 1, abort)) break;
                cur_b = b;
                ++nb;
            }
            if (k >= kIxAcc && !mbar_wait(smem_u32(&S.accempty[a]), ((k / kIxAcc) - 1) & 1, abort))
                break;
            tc_fence_after();
            const uint64_t ad = adesc0 + (uint64_t)s * kStageStep;
            const uint64_t bd = bdesc0 + (uint64_t)jb * kBStep;
            const uint32_t dt = tmem + (uint32_t)(a * kCols);
            mma_ss_f8(dt, ad, bd, idesc, 0);
            mma_ss_f8(dt, ad + 2, bd + 2, idesc, 1);
            mma_ss_f8(dt, ad + 4, bd + 4, idesc, 1);
            mma_ss_f8(dt, ad + 6, bd + 6, idesc, 1);
            mma_commit(smem_u32(&S.empty[s]));
            mma_commit(smem_u32(&S.accfull[a]));
        }
        // all MMAs complete before TMEM is released
        volatile int own = 0;
        mma_commit(smem_u32(&S.drain));
        mbar_wait(smem_u32(&S.drain), 0, &own, 100000000ull);
        if (own) *abort = 1;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kIxWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kAlloc);
    }
    if (tid == 0 && S.abort) status_or(status, MLA_STATUS_TIMEOUT);
}

template <int NCH>
size_t ix_smem() {
    return sizeof(IxSmem) + 1024;
}

template <int NCH>
cudaError_t ix_setup() {
    return cudaFuncSetAttribute(fp8_indexer_tc_kernel<NCH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)ix_smem<NCH>());
}

}  // namespace

cudaError_t setup_fp8_indexer() {
    cudaError_t e = ix_setup<1>();
    if (e == cudaSuccess) e = ix_setup<2>();
    if (e == cudaSuccess) e = ix_setup<3>();
    if (e == cudaSuccess) e = ix_setup<4>();
    return e;
}

cudaError_t launch_fp8_indexer(const void* q, const float* w, const void* kv, int64_t nblocks,
                               const int32_t* bt, const int32_t* lens, int batch, int H, int P,
                               float* out, int32_t* status, int grid, cudaStream_t stream) {
    CUtensorMap kmap, qmap;
    if (!make_fp8_block_map(&kmap, kv, nblocks) || !make_fp8_query_map(&qmap, q, batch, H))
        return cudaErrorInvalidValue;
    const uint8_t* kvb = static_cast<const uint8_t*>(kv);
#define MLAV_IX_LAUNCH(NCH)                                                                       \
    launch_pdl(fp8_indexer_tc_kernel<NCH>, dim3(grid), dim3(kIxThreads), ix_smem<NCH>(), stream, kmap, \
               qmap, kvb, w, nblocks, bt, lens, batch, H, P, out, status)
    cudaError_t e;
    if (H <= 32)
        e = MLAV_IX_LAUNCH(1);
    else if (H <= 64)
        e = MLAV_IX_LAUNCH(2);
    else if (H <= 96)
        e = MLAV_IX_LAUNCH(3);
    else
        e = MLAV_IX_LAUNCH(4);
#undef MLAV_IX_LAUNCH
    return e;
}

}  // namespace mlav
