// Layout self-test of the tcgen05 building blocks used by the tensor-core
// partial kernel (test-only library, libmlaselftest.so).
//
// One CTA computes D = A * B (M = 128, K = 64, N in {32, 64, 128, 256})
// with the same wrappers, descriptors and 128-byte-swizzled shared-memory
// layouts as the kernel, and writes D (fp32) back for comparison on the host:
//   mode 0: A smem K-major,  B smem K-major ([N][64])
//   mode 1: A in TMEM,       B smem K-major
//   mode 2: A smem K-major,  B smem MN-major ([64][N], 64-wide atom columns)
//   mode 3: A in TMEM,       B smem MN-major
// For the MN-major modes `variant` selects which descriptor field carries
// the atom-column stride (0: leading, 1: stride). Every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../tc_ptx.cuh"
#include "../tmap.cuh"

using namespace mlav::tc;

namespace {

constexpr int kM = 128, kK = 64;
constexpr uint32_t kAcol = 256;  // TMEM column of A (modes 1, 3); D uses [0, N)

struct __align__(1024) ProbeSmem {
    unsigned char a[kM * 128];   // [128 rows][64 bf16], swizzled
    unsigned char b[256 * 128];  // K-major [N][64] or MN-major [N/64][64 k][64 n]
    uint64_t bar;
    uint32_t tmem;
    int abort_flag;
};

__global__ void __launch_bounds__(128, 1)
probe_kernel(const __nv_bfloat16* __restrict__ A, const __nv_bfloat16* __restrict__ B,
             float* __restrict__ D, int N, int mode, int variant, int* err) {
    extern __shared__ __align__(1024) unsigned char raw[];
    // The 128-byte swizzle keys on absolute shared-memory address bits, so
    // the tiles must start on 1024-byte boundaries.
    unsigned char* base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
    ProbeSmem& sm = *reinterpret_cast<ProbeSmem*>(base);
    const int tid = threadIdx.x, warp = tid >> 5;
    const bool a_tmem = (mode == 1 || mode == 3);
    const bool b_mn = (mode == 2 || mode == 3);

    for (int i = tid; i < kM * 8; i += 128) {
        const int r = i >> 3, c = i & 7;
        *reinterpret_cast<uint4*>(sm.a + sw128_offset(r, c)) =
            *reinterpret_cast<const uint4*>(A + r * kK + c * 8);
    }
    if (!b_mn) {
        for (int i = tid; i < N * 8; i += 128) {
            const int n = i >> 3, c = i & 7;
            *reinterpret_cast<uint4*>(sm.b + sw128_offset(n, c)) =
                *reinterpret_cast<const uint4*>(B + n * kK + c * 8);
        }
    } else {
        const int nchunks = N / 8;
        for (int i = tid; i < kK * nchunks; i += 128) {
            const int k = i / nchunks, n0 = (i % nchunks) * 8;
            *reinterpret_cast<uint4*>(sm.b + (n0 / 64) * (kK * 128) + sw128_offset(k, (n0 % 64) / 8)) =
                *reinterpret_cast<const uint4*>(B + k * N + n0);
        }
    }
    fence_proxy_async_smem();
    if (warp == 0) {
        tmem_alloc(smem_u32(&sm.tmem), 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(smem_u32(&sm.bar), 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = sm.tmem;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

    if (a_tmem) {
        uint32_t w[32];
        const uint32_t* src = reinterpret_cast<const uint32_t*>(A + tid * kK);
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = src[i];
        tmem_st32(taddr + lane_base + kAcol, w);
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (tid == 0) {
        const uint32_t idesc = make_idesc_bf16(kM, N, false, b_mn);
        const uint32_t a0 = smem_u32(sm.a), b0 = smem_u32(sm.b);
        for (int ks = 0; ks < kK / 16; ++ks) {
            uint64_t bd;
            if (!b_mn) {
                bd = make_sdesc(b0 + ks * 32, 16, 1024, kSwizzle128B);
            } else {
                const uint32_t col_stride = kK * 128, kgrp_stride = 1024;
                bd = variant == 0 ? make_sdesc(b0 + ks * 2048, col_stride, kgrp_stride, kSwizzle128B)
                                  : make_sdesc(b0 + ks * 2048, kgrp_stride, col_stride, kSwizzle128B);
            }
            if (a_tmem)
                mma_ts(taddr, taddr + kAcol + ks * 8, bd, idesc, ks > 0);
            else
                mma_ss(taddr, make_sdesc(a0 + ks * 32, 16, 1024, kSwizzle128B), bd, idesc, ks > 0);
        }
        mma_commit(smem_u32(&sm.bar));
    }
    const bool ok = mbar_wait(smem_u32(&sm.bar), 0, &sm.abort_flag);
    tc_fence_after();
    if (ok) {
        for (int c0 = 0; c0 < N; c0 += 32) {
            uint32_t r[32];
            tmem_ld32(taddr + lane_base + c0, r);
            tmem_wait_ld();
            for (int j = 0; j < 32; ++j) D[tid * N + c0 + j] = __uint_as_float(r[j]);
        }
    } else if (tid == 0) {
        atomicExch(err, 1);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(taddr, 512);
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int mlav_umma_probe(
    const void* A, const void* B, float* D, int N, int mode, int variant, int* err) {
    if (N != 32 && N != 64 && N != 128 && N != 256) return -1;
    if (mode < 0 || mode > 3) return -1;
    if ((mode >= 2) && N < 64) return -1;
    cudaError_t e = cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(ProbeSmem) + 1024);
    if (e != cudaSuccess) return (int)e;
    probe_kernel<<<1, 128, sizeof(ProbeSmem) + 1024>>>(
        static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B), D, N, mode,
        variant, err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    return (int)cudaDeviceSynchronize();
}

namespace {

// Throughput probe: one thread issues `reps` rounds of MMAs (M = 128, K = 16,
// N = n) cycling over `nacc` independent accumulators, with A from shared
// memory or TMEM; reports the cycles from the first issue to the commit.
__global__ void __launch_bounds__(128, 1)
mma_rate_kernel(int N, int a_tmem, int reps, int nacc, int overwrite, long long* out, int* err) {
    extern __shared__ __align__(1024) unsigned char raw[];
    unsigned char* base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
    ProbeSmem& sm = *reinterpret_cast<ProbeSmem*>(base);
    const int tid = threadIdx.x, warp = tid >> 5;
    for (int i = tid; i < (int)(sizeof(sm.a) / 16); i += 128)
        reinterpret_cast<uint4*>(sm.a)[i] = make_uint4(0x3f803f80u, 0, 0, 0);
    for (int i = tid; i < (int)(sizeof(sm.b) / 16); i += 128)
        reinterpret_cast<uint4*>(sm.b)[i] = make_uint4(0x3f803f80u, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 0) {
        tmem_alloc(smem_u32(&sm.tmem), 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(smem_u32(&sm.bar), 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = sm.tmem;
    if (tid == 0) {
        const uint32_t idesc = make_idesc_bf16(kM, N, false, false);
        const uint32_t a0 = smem_u32(sm.a), b0 = smem_u32(sm.b);
        const long long t0 = clock64();
        for (int r = 0; r < reps; ++r) {
            const int ks = r & 3;
            const uint64_t bd = make_sdesc(b0 + ks * 32, 16, 1024, kSwizzle128B);
            const uint64_t ad = make_sdesc(a0 + ks * 32, 16, 1024, kSwizzle128B);
            for (int c = 0; c < nacc; ++c) {
                const uint32_t acc = overwrite ? 0u : 1u;
                if (a_tmem)
                    mma_ts(taddr + c * N, taddr + kAcol + ks * 8, bd, idesc, acc);
                else
                    mma_ss(taddr + c * N, ad, bd, idesc, acc);
            }
        }
        mma_commit(smem_u32(&sm.bar));
        const bool ok = mbar_wait(smem_u32(&sm.bar), 0, &sm.abort_flag);
        const long long t1 = clock64();
        out[0] = t1 - t0;
        if (!ok) atomicExch(err, 1);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(taddr, 512);
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int mlav_mma_rate(int N, int a_tmem, int reps,
                                                                    int nacc, int overwrite,
                                                                    long long* out, int* err) {
    if (N < 16 || N > 256 || (N % 16) != 0 || nacc < 1 || reps < 1) return -1;
    if (N * nacc > (a_tmem ? 256 : 512)) return -1;
    cudaError_t e = cudaFuncSetAttribute(mma_rate_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(ProbeSmem) + 1024);
    if (e != cudaSuccess) return (int)e;
    mma_rate_kernel<<<1, 128, sizeof(ProbeSmem) + 1024>>>(N, a_tmem, reps, nacc, overwrite, out, err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    return (int)cudaDeviceSynchronize();
}

namespace {

struct GatherRows {
    int r[8];
};

// TMA gather check: two tile::gather4 loads of 4 rows x 64 columns each into
// a 1024-byte-aligned tile; the raw shared-memory bytes are copied out.
__global__ void __launch_bounds__(128, 1)
gather_probe_kernel(const __grid_constant__ CUtensorMap map, GatherRows rows, int x,
                    uint4* out, int* err) {
    __shared__ __align__(1024) unsigned char buf[1024];
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    const int tid = threadIdx.x;
    if (tid == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(smem_u32(&bar), 1024);
        tma_gather4(smem_u32(buf), &map, x, rows.r[0], rows.r[1], rows.r[2], rows.r[3], smem_u32(&bar));
        tma_gather4(smem_u32(buf) + 512, &map, x, rows.r[4], rows.r[5], rows.r[6], rows.r[7],
                    smem_u32(&bar));
    }
    const bool ok = mbar_wait(smem_u32(&bar), 0, &abort_flag);
    if (!ok && tid == 0) atomicExch(err, 1);
    if (ok && tid < 64) out[tid] = reinterpret_cast<const uint4*>(buf)[tid];
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int mlav_gather_probe(const void* kv,
                                                                        long long slots,
                                                                        const int* rows_host, int x,
                                                                        void* out, int* err) {
    CUtensorMap map;
    if (!mlav::make_kv_gather_map(&map, kv, slots)) return -2;
    if (x < 0 || x > 512 || (x % 8) != 0) return -1;
    GatherRows rows;
    for (int i = 0; i < 8; ++i) rows.r[i] = rows_host[i];
    gather_probe_kernel<<<1, 128>>>(map, rows, x, static_cast<uint4*>(out), err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    return (int)cudaDeviceSynchronize();
}

namespace {

// Gather-throughput probe. Every CTA streams `ntile` tiles of 256 scattered
// latent rows through a 4-stage ring of [256 keys x 64 dims] blocks (9 blocks
// per tile), the layout the S side of the pair kernel consumes; a consumer
// warp releases each stage as soon as it lands. The tile's slots are staged
// in shared memory before its blocks are issued. Methods:
//   0: cp.async, 8 lanes per key (one 128-byte line per 8 lanes), `nw` warps
//   1: cp.async, one lane per key (8 slot registers per lane), `nw` warps
//   2: tile::gather4 issued by the 32 lanes of one warp
//   3: tile::gather4 issued by one thread
constexpr int kGStages = 4;
struct __align__(1024) GatherSmem {
    unsigned char ring[kGStages][256 * 128];
    int32_t rows[2][256];
    uint64_t full[kGStages], empty[kGStages], rows_bar[2];
    int abort_flag;
};

__global__ void __launch_bounds__(512, 1)
gather_rate_kernel(const __grid_constant__ CUtensorMap map, const __nv_bfloat16* kv,
                   const int32_t* slots, int ntile, int method, int nw, int tma_rows, long long* cycles,
                   int* err) {
    extern __shared__ __align__(1024) unsigned char raw[];
    unsigned char* base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
    GatherSmem& g = *reinterpret_cast<GatherSmem*>(base);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // method 4: warps 0..nw-1 copy keys [0, 256 - tma_rows) with cp.async (as
    // method 0) while warp 4 issues gather4 for the last tma_rows keys.
    const int nprod = (method <= 1 || method == 4) ? nw : 1;
    const int cp_keys = method == 4 ? 256 - tma_rows : 256;
    if (tid == 0) {
        for (int i = 0; i < kGStages; ++i) {
            mbar_init(smem_u32(&g.full[i]), method <= 1 ? 32 * nprod : method == 4 ? 32 * nprod + 1 : 1);
            mbar_init(smem_u32(&g.empty[i]), 1);
        }
        g.abort_flag = 0;
        fence_mbar_init();
    }
    // all tiles' slots for this CTA fit two buffers only; preload tile 0 and 1 here
    __syncthreads();
    const int32_t* my = slots + (size_t)blockIdx.x * ntile * 256;
    const long long t0 = clock64();
    if (method == 4 && warp == 4) {
        if (lane == 0) {
            for (int t = 0; t < ntile; ++t) {
                // the rows of tile t are read straight from global memory here
                for (int blk = 0; blk < 9; ++blk) {
                    const int u = t * 9 + blk, st = u % kGStages;
                    if (u >= kGStages && !mbar_wait(smem_u32(&g.empty[st]), ((u / kGStages) - 1) & 1, &g.abort_flag)) {
                        atomicExch(err, 1);
                        break;
                    }
                    const uint32_t dst0 = smem_u32(g.ring[st]);
                    mbar_arrive_expect_tx(smem_u32(&g.full[st]), (uint32_t)tma_rows * 128u);
                    for (int k0 = cp_keys; k0 < 256; k0 += 4) {
                        const int32_t* r = my + t * 256 + k0;
                        tma_gather4(dst0 + k0 * 128, &map, blk * 64, r[0], r[1], r[2], r[3], smem_u32(&g.full[st]));
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp < nprod) {
        for (int t = 0; t < ntile; ++t) {
            // stage this tile's slots (each producer warp keeps its own copy in registers
            // where needed; the shared copy serves methods 0, 2, 3)
            __syncwarp();
            if (warp == 0) {
                for (int k = lane; k < 256; k += 32) g.rows[t & 1][k] = my[t * 256 + k];
            }
            asm volatile("bar.sync 2, %0;" ::"r"(32 * nprod) : "memory");
            int32_t own[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) own[q] = g.rows[t & 1][32 * q + lane];
            for (int blk = 0; blk < 9; ++blk) {
                const int u = t * 9 + blk, st = u % kGStages;
                if (u >= kGStages && !mbar_wait(smem_u32(&g.empty[st]), ((u / kGStages) - 1) & 1, &g.abort_flag)) {
                    atomicExch(err, 1);
                    goto done;
                }
                const uint32_t dst0 = smem_u32(g.ring[st]);
                if (method == 0 || method == 4) {
                    for (int it = warp; it < cp_keys / 4; it += nprod) {
                        const int key = it * 4 + (lane >> 3), c = lane & 7;
                        const int32_t sl = g.rows[t & 1][key];
                        cp_async_16_zfill_nc(dst0 + sw128_offset(key, c),
                                             kv + (int64_t)sl * 576 + blk * 64 + c * 8, true);
                    }
                    cp_async_mbar_arrive_noinc(smem_u32(&g.full[st]));
                } else if (method == 1) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        if ((q % nprod) != warp) continue;
                        const int key = 32 * q + lane;
                        const __nv_bfloat16* src = kv + (int64_t)own[q] * 576 + blk * 64;
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            cp_async_16_zfill_nc(dst0 + sw128_offset(key, c), src + c * 8, true);
                    }
                    cp_async_mbar_arrive_noinc(smem_u32(&g.full[st]));
                } else if (method == 2) {
                    if (lane == 0) mbar_arrive_expect_tx(smem_u32(&g.full[st]), 256 * 128);
                    __syncwarp();
                    for (int v = 0; v < 2; ++v) {
                        const int gi = lane + 32 * v;
                        const int32_t* r = &g.rows[t & 1][4 * gi];
                        tma_gather4(dst0 + gi * 512, &map, blk * 64, r[0], r[1], r[2], r[3], smem_u32(&g.full[st]));
                    }
                } else {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(smem_u32(&g.full[st]), 256 * 128);
                        for (int gi = 0; gi < 64; ++gi) {
                            const int32_t* r = &g.rows[t & 1][4 * gi];
                            tma_gather4(dst0 + gi * 512, &map, blk * 64, r[0], r[1], r[2], r[3], smem_u32(&g.full[st]));
                        }
                    }
                    __syncwarp();
                }
            }
        }
        if (method <= 1) cp_async_wait_all();
    } else if (warp == 15 && lane == 0) {
        for (int u = 0; u < ntile * 9; ++u) {
            const int st = u % kGStages;
            if (!mbar_wait(smem_u32(&g.full[st]), (u / kGStages) & 1, &g.abort_flag)) {
                atomicExch(err, 1);
                break;
            }
            mbar_arrive(smem_u32(&g.empty[st]));
        }
        cycles[blockIdx.x] = clock64() - t0;
    }
done:
    __syncthreads();
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int mlav_gather_rate(
    const void* kv, long long pool, const int32_t* slots, int nblocks, int ntile, int method,
    int nw, int tma_rows, long long* cycles, int* err) {
    CUtensorMap map;
    if (!mlav::make_kv_gather_map(&map, kv, pool)) return -2;
    if (nw < 1 || nw > 12 || (method != 0 && nw > 4) || method < 0 || method > 4) return -1;
    if (method == 4 && (tma_rows < 4 || tma_rows > 252 || tma_rows % 4 != 0)) return -1;
    const int smem = (int)sizeof(GatherSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(gather_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return (int)e;
    gather_rate_kernel<<<nblocks, 512, smem>>>(map, static_cast<const __nv_bfloat16*>(kv), slots, ntile,
                                               method, nw, tma_rows, cycles, err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    return (int)cudaDeviceSynchronize();
}

namespace {

// DSMEM bulk-copy throughput: CTA 0 of each 2-CTA cluster sends `nchunk`
// chunks of `chunk` bytes from its shared memory into CTA 1's, through a
// 4-slot ring (CTA 1 releases a slot once it has landed, by a remote arrive).
// Reports cycles per sending CTA. The payload is checked on the receiver.
struct __align__(1024) BulkSmem {
    unsigned char buf[4][32768];
    uint64_t full[4], empty[4];
    int abort_flag;
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
bulk_rate_kernel(int chunk, int nchunk, long long* cycles, int* err) {
    extern __shared__ __align__(1024) unsigned char raw[];
    unsigned char* base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
    BulkSmem& b = *reinterpret_cast<BulkSmem*>(base);
    const uint32_t rank = cluster_ctarank();
    const int tid = threadIdx.x;
    for (int i = tid; i < 4 * 32768 / 16; i += 128)
        reinterpret_cast<uint4*>(b.buf)[i] = make_uint4(rank == 0 ? (uint32_t)i : 0u, 7u, 0, 0);
    if (tid == 0) {
        for (int i = 0; i < 4; ++i) {
            mbar_init(smem_u32(&b.full[i]), 1);
            mbar_init(smem_u32(&b.empty[i]), 1);
        }
        b.abort_flag = 0;
        fence_mbar_init();
    }
    fence_proxy_async_smem();
    __syncthreads();
    cluster_sync_all();
    if (tid == 0) {
        const long long t0 = clock64();
        if (rank == 0) {
            for (int c = 0; c < nchunk; ++c) {
                const int st = c & 3;
                if (c >= 4 && !mbar_wait(smem_u32(&b.empty[st]), ((c >> 2) - 1) & 1, &b.abort_flag)) {
                    atomicExch(err, 1);
                    break;
                }
                bulk_copy_to_peer(mapa_shared(smem_u32(b.buf[st]), 1), smem_u32(b.buf[st]),
                                  (uint32_t)chunk, mapa_shared(smem_u32(&b.full[st]), 1));
            }
            // the receiver's last release marks the end
            const int c = nchunk + 3;
            if (nchunk >= 1) mbar_wait(smem_u32(&b.empty[(nchunk - 1) & 3]), ((nchunk - 1) >> 2) & 1, &b.abort_flag);
            (void)c;
            cycles[blockIdx.x / 2] = clock64() - t0;
        } else {
            for (int c = 0; c < nchunk; ++c) {
                const int st = c & 3;
                mbar_arrive_expect_tx(smem_u32(&b.full[st]), (uint32_t)chunk);
                if (!mbar_wait(smem_u32(&b.full[st]), (c >> 2) & 1, &b.abort_flag)) {
                    atomicExch(err, 1);
                    break;
                }
                if (c == nchunk - 1) {
                    const uint4 v = reinterpret_cast<const uint4*>(b.buf[st])[chunk / 16 - 1];
                    if (v.y != 7u) atomicExch(err, 2);
                }
                mbar_arrive_cluster(mapa_shared(smem_u32(&b.empty[st]), 0));
            }
        }
    }
    __syncthreads();
    cluster_sync_all();
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int mlav_bulk_rate(int nclusters, int chunk,
                                                                     int nchunk, long long* cycles,
                                                                     int* err) {
    if (chunk < 16 || chunk > 32768 || (chunk % 16) != 0 || nchunk < 1 || nclusters < 1) return -1;
    const int smem = (int)sizeof(BulkSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(bulk_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return (int)e;
    bulk_rate_kernel<<<2 * nclusters, 128, smem>>>(chunk, nchunk, cycles, err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    return (int)cudaDeviceSynchronize();
}

namespace {

// CTA-pair (cta_group::2) layout self-test. A cluster of two CTAs computes
// D = A * B with M = 256, K = 64: CTA r holds A rows [128r, 128r + 128) and
// B rows (N) [r N/2, (r + 1) N/2), each in the same 128-byte-swizzled layouts
// as the single-CTA probe; CTA 0 issues the MMAs and commits to the
// mbarrier of both CTAs; each CTA reads its 128 rows of D from its own TMEM.
//   mode 0: A smem K-major, B smem K-major      (N = 128 or 256)
//   mode 1: A in TMEM,      B smem K-major      (N = 128 or 256)
//   mode 2: A smem K-major, B smem MN-major     (N = 256)
// The pair allocates 512 columns together (D at column 0, A at column 256).
// addr[r] receives CTA r's copy of the allocation result.
// `reps` > 1 repeats the MMA sequence (rate measurement); cycles[0] is CTA 0's
// issue-to-commit time.
struct __align__(1024) PairSmem {
    unsigned char a[128 * 128];  // [128 rows][64 bf16]
    unsigned char b[128 * 128];  // K-major [N/2][64] or MN-major [N/2 / 64][64 k][64 n]
    uint64_t bar, tick;
    uint32_t tmem;
    int abort_flag;
};

template <bool kATmem, int kVar>
__device__ __forceinline__ void pair_issue(uint32_t taddr, uint32_t acol, uint32_t a0, uint32_t b0,
                                           bool b_mn, uint32_t idesc, int reps, uint32_t tick) {
    const uint64_t bd0 = b_mn ? make_sdesc(b0, 64 * 128, 1024, kSwizzle128B)
                              : make_sdesc(b0, 16, 1024, kSwizzle128B);
    const uint64_t bstep = b_mn ? (2048 >> 4) : (32 >> 4);
    const uint64_t ad0 = make_sdesc(a0, 16, 1024, kSwizzle128B);
    for (int rep = 0; rep < reps; ++rep) {
        if (kVar == 2) {
            (void)mbar_test_wait(tick, 0);
            fence_proxy_async_smem();
            tc_fence_after();
        }
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            if (kATmem)
                mma_ts_pair(taddr, taddr + acol + ks * 8, bd0 + bstep * ks, idesc, ks > 0);
            else
                mma_ss_pair(taddr, ad0 + 2 * ks, bd0 + bstep * ks, idesc, ks > 0);
        }
        if (kVar >= 1) mma_commit_pair_mc(tick, (uint16_t)3);
    }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
pair_probe_kernel(const __nv_bfloat16* __restrict__ A, const __nv_bfloat16* __restrict__ B,
                  float* __restrict__ D, int N, int mode, int reps, int commit_every,
                  uint32_t* addr, long long* cycles, int* err) {
    extern __shared__ __align__(1024) unsigned char raw[];
    unsigned char* base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
    PairSmem& sm = *reinterpret_cast<PairSmem*>(base);
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t rank = cluster_ctarank();
    const bool a_tmem = mode == 1;
    const bool b_mn = mode == 2;
    const int nh = N / 2;
    constexpr uint32_t kAcolP = 256;

    const __nv_bfloat16* Ar = A + (size_t)rank * 128 * 64;
    for (int i = tid; i < 128 * 8; i += 128) {
        const int r = i >> 3, c = i & 7;
        *reinterpret_cast<uint4*>(sm.a + sw128_offset(r, c)) =
            *reinterpret_cast<const uint4*>(Ar + r * 64 + c * 8);
    }
    if (!b_mn) {
        const __nv_bfloat16* Br = B + (size_t)rank * nh * 64;
        for (int i = tid; i < nh * 8; i += 128) {
            const int n = i >> 3, c = i & 7;
            *reinterpret_cast<uint4*>(sm.b + sw128_offset(n, c)) =
                *reinterpret_cast<const uint4*>(Br + n * 64 + c * 8);
        }
    } else {
        // B is [64 k][N]; this CTA holds columns [rank * nh, rank * nh + nh).
        const int nchunks = nh / 8;
        for (int i = tid; i < 64 * nchunks; i += 128) {
            const int k = i / nchunks, n0 = (i % nchunks) * 8;
            *reinterpret_cast<uint4*>(sm.b + (n0 / 64) * (64 * 128) + sw128_offset(k, (n0 % 64) / 8)) =
                *reinterpret_cast<const uint4*>(B + k * N + rank * nh + n0);
        }
    }
    fence_proxy_async_smem();
    if (warp == 0) {
        tmem_alloc_pair(smem_u32(&sm.tmem), 512);
        tmem_relinquish_pair();
    }
    if (tid == 0) {
        mbar_init(smem_u32(&sm.bar), 1);
        mbar_init(smem_u32(&sm.tick), 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t my_addr = sm.tmem;
    if (tid == 0) addr[rank] = my_addr;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    if (a_tmem) {
        uint32_t w[32];
        const uint32_t* src = reinterpret_cast<const uint32_t*>(Ar + tid * 64);
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = src[i];
        tmem_st32(my_addr + lane_base + kAcolP, w);
        tmem_wait_st();
    }
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();

    if (rank == 0 && tid == 0) {
        const uint32_t idesc = make_idesc_bf16(256, N, false, b_mn);
        const uint32_t a0 = smem_u32(sm.a), b0 = smem_u32(sm.b);
        const long long t0 = clock64();
        // Issue variants (selected outside the loop): 0 plain; 1 commit after
        // every 4 MMAs; 2 per 4 MMAs an mbarrier test, the proxy and tcgen05
        // fences and a commit (the partial kernel's per-stage work).
        const int var = commit_every;
        if (a_tmem) {
            if (var == 0) pair_issue<true, 0>(my_addr, kAcolP, a0, b0, b_mn, idesc, reps, smem_u32(&sm.tick));
            else if (var == 1) pair_issue<true, 1>(my_addr, kAcolP, a0, b0, b_mn, idesc, reps, smem_u32(&sm.tick));
            else pair_issue<true, 2>(my_addr, kAcolP, a0, b0, b_mn, idesc, reps, smem_u32(&sm.tick));
        } else {
            if (var == 0) pair_issue<false, 0>(my_addr, kAcolP, a0, b0, b_mn, idesc, reps, smem_u32(&sm.tick));
            else if (var == 1) pair_issue<false, 1>(my_addr, kAcolP, a0, b0, b_mn, idesc, reps, smem_u32(&sm.tick));
            else pair_issue<false, 2>(my_addr, kAcolP, a0, b0, b_mn, idesc, reps, smem_u32(&sm.tick));
        }
        mma_commit_pair_mc(smem_u32(&sm.bar), (uint16_t)3);
        if (mbar_wait(smem_u32(&sm.bar), 0, &sm.abort_flag)) cycles[0] = clock64() - t0;
    }
    const bool ok = mbar_wait(smem_u32(&sm.bar), 0, &sm.abort_flag);
    tc_fence_after();
    if (ok) {
        for (int c0 = 0; c0 < N; c0 += 32) {
            uint32_t r[32];
            tmem_ld32(my_addr + lane_base + c0, r);
            tmem_wait_ld();
            float* drow = D + (size_t)(rank * 128 + tid) * N + c0;
            for (int j = 0; j < 32; ++j) drow[j] = __uint_as_float(r[j]);
        }
    } else if (tid == 0) {
        atomicExch(err, 1 + (int)rank);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 0) tmem_dealloc_pair(my_addr, 512);
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int mlav_pair_probe(
    const void* A, const void* B, float* D, int N, int mode, int reps, int commit_every,
    uint32_t* addr, long long* cycles, int* err) {
    if (mode < 0 || mode > 2 || reps < 1 || reps > 4096) return -1;
    if (mode == 0 && N != 128 && N != 256) return -1;
    if (mode == 1 && N != 128 && N != 256) return -1;
    if (mode == 2 && N != 256) return -1;
    const int smem = (int)sizeof(PairSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(pair_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return (int)e;
    pair_probe_kernel<<<2, 128, smem>>>(static_cast<const __nv_bfloat16*>(A),
                                        static_cast<const __nv_bfloat16*>(B), D, N, mode, reps,
                                        commit_every, addr, cycles, err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    return (int)cudaDeviceSynchronize();
}

namespace {

// Round trip of an empty producer/consumer ring (no data): one producer warp
// signals stage g full, one consumer thread waits for it and releases the
// stage; the producer waits for the release of stage g - depth before
// signalling stage g. Measures the signalling latency alone.
//   prod_mode 0: mbarrier.arrive by lane 0 (count 1)
//   prod_mode 1: cp.async.mbarrier.arrive.noinc by all 32 lanes (count 32)
//   cons_mode 0: mbarrier.arrive (count 1)
//   cons_mode 1: tcgen05.commit (1-CTA) with no MMA in flight
struct RingSmem {
    uint64_t full[16], empty[16];
    uint32_t tmem;
    int abort_flag;
};

__global__ void __launch_bounds__(64, 1)
ring_probe_kernel(int depth, int n, int prod_mode, int cons_mode, long long* cycles, int* err) {
    __shared__ RingSmem r;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp == 1) {
        tmem_alloc(smem_u32(&r.tmem), 32);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < depth; ++i) {
            mbar_init(smem_u32(&r.full[i]), prod_mode == 1 ? 32 : 1);
            mbar_init(smem_u32(&r.empty[i]), 1);
        }
        r.abort_flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const long long t0 = clock64();
    if (warp == 0) {
        for (int g = 0; g < n; ++g) {
            const int st = g % depth;
            if (g >= depth) {
                const bool ok = mbar_wait(smem_u32(&r.empty[st]), ((g / depth) - 1) & 1, &r.abort_flag);
                if (!__all_sync(0xffffffffu, ok)) {
                    if (lane == 0) atomicExch(err, 1);
                    break;
                }
            }
            if (prod_mode == 1)
                cp_async_mbar_arrive_noinc(smem_u32(&r.full[st]));
            else if (lane == 0)
                mbar_arrive(smem_u32(&r.full[st]));
            __syncwarp();
        }
    } else if (lane == 0) {
        for (int g = 0; g < n; ++g) {
            const int st = g % depth;
            if (!mbar_wait(smem_u32(&r.full[st]), (g / depth) & 1, &r.abort_flag)) {
                atomicExch(err, 2);
                break;
            }
            if (cons_mode == 1)
                mma_commit(smem_u32(&r.empty[st]));
            else
                mbar_arrive(smem_u32(&r.empty[st]));
        }
        cycles[0] = clock64() - t0;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(r.tmem, 32);
    }
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int mlav_ring_probe(int depth, int n, int prod_mode,
                                                                      int cons_mode, long long* cycles,
                                                                      int* err) {
    if (depth < 1 || depth > 16 || n < 1 || prod_mode < 0 || prod_mode > 1 || cons_mode < 0 ||
        cons_mode > 1)
        return -1;
    ring_probe_kernel<<<1, 64>>>(depth, n, prod_mode, cons_mode, cycles, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    return (int)cudaDeviceSynchronize();
}

namespace {

// Cost of single mbarrier operations issued back to back by one thread:
//   op 0: try_wait.parity on a completed phase
//   op 1: test_wait.parity on a completed phase
//   op 2: arrive on a barrier whose phase does not complete (count 8192,
//         n <= 4096 arrivals; counts must stay within the hardware range
//         [1, 2^20 - 1])
//   op 3: try_wait.parity.acquire.cluster on a completed phase
//   op 4: arrive + try_wait on the next (completing) phase, count 1
__global__ void __launch_bounds__(32, 1) mbar_cost_kernel(int op, int n, long long* cycles,
                                                          int* sink) {
    __shared__ uint64_t bar[2];
    if (threadIdx.x != 0) return;
    mbar_init(smem_u32(&bar[0]), 1);
    mbar_init(smem_u32(&bar[1]), 8192);
    fence_mbar_init();
    mbar_arrive(smem_u32(&bar[0]));  // phase 0 of bar[0] completes
    int acc = 0;
    const long long t0 = clock64();
    if (op == 0) {
        for (int i = 0; i < n; ++i) acc += mbar_try_wait(smem_u32(&bar[0]), 0) ? 1 : 0;
    } else if (op == 1) {
        for (int i = 0; i < n; ++i) acc += mbar_test_wait(smem_u32(&bar[0]), 0) ? 1 : 0;
    } else if (op == 2) {
        for (int i = 0; i < n; ++i) mbar_arrive(smem_u32(&bar[1]));
    } else if (op == 3) {
        for (int i = 0; i < n; ++i) acc += mbar_try_wait_cluster(smem_u32(&bar[0]), 0) ? 1 : 0;
    } else {
        for (int i = 0; i < n; ++i) {
            mbar_arrive(smem_u32(&bar[0]));  // phase i + 1 completes
            acc += mbar_try_wait(smem_u32(&bar[0]), (uint32_t)((i + 1) & 1)) ? 1 : 0;
        }
    }
    cycles[0] = clock64() - t0;
    sink[0] = acc;
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int mlav_mbar_cost(int op, int n, long long* cycles,
                                                                     int* sink) {
    if (op < 0 || op > 4 || n < 1 || n > 4096) return -1;
    mbar_cost_kernel<<<1, 32>>>(op, n, cycles, sink);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    return (int)cudaDeviceSynchronize();
}

namespace {

// Block-stream probe: every CTA streams `ntile` stages of two random 8 KB
// blocks of an fp8 indexer cache ([nblk][8448] bytes: 64 rows of 128 bytes,
// then 256 scale bytes) through an 8-stage ring of 16 KB stages in the
// 128-byte-swizzled layout; a consumer thread releases each stage as soon as
// it lands. The CTA's block indices are staged in shared memory first, so
// only the copies are timed. Methods:
//   0: two TMA 3-D boxes (64 rows x 128 bytes) per stage, one issuing thread
//   1: cp.async 16-byte pieces by `nw` warps (all warps share every stage)
//   2: two 1-D bulk copies of 8 KB per stage (unswizzled), one issuing thread
//   3: TMA box for the first block, cp.async by `nw` warps for the second
//   4: ld.global 16-byte loads into registers, then st.shared, `nw` warps
//      (warp w owns stages u = w mod nw, a whole stage per warp)
//   5: as 0, plus each block's 256 scale bytes by a 1-D bulk copy
//   6: as 0, plus each block's 256 scale bytes by a TMA box of an
//      unswizzled map (rows 64-65 of the block viewed as 66 rows of 128 bytes)
//   7: latent-cache rows instead of blocks: each stage holds 14 whole rows
//      of 1152 bytes from random slots of a [row_pool][1152-byte] pool,
//      cp.async by `nw` warps (16128 bytes per stage)
//   8: as 7 but one 128-byte segment (segment u mod 9) from each of 126
//      random rows per stage (the same bytes per stage)
//   9: as 7 but each row by one 1-D bulk copy of 1152 bytes (lanes 0-13 of
//      one warp issue a stage's 14 copies)
// Methods 7, 8 and 9 read their slots (126 per stage, 14 used by method 7) from
// `blocks` [CTA][stage][126], staged in shared memory like the block indices.
constexpr int kBStages = 8;
constexpr int kBMaxIdx = 16384;
struct __align__(1024) BlockSmem {
    unsigned char ring[kBStages][16384];
    unsigned char scale[kBStages][512];
    int32_t idx[kBMaxIdx];
    uint64_t full[kBStages], empty[kBStages];
    int abort_flag;
};

__global__ void __launch_bounds__(512, 1)
block_rate_kernel(const __grid_constant__ CUtensorMap map, const __grid_constant__ CUtensorMap smap,
                  const unsigned char* kv,
                  const int32_t* blocks, int ntile, int method, int nw, long long row_pool,
                  long long* cycles, int* err) {
    extern __shared__ __align__(1024) unsigned char raw[];
    unsigned char* base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
    BlockSmem& g = *reinterpret_cast<BlockSmem*>(base);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool cp_side = method == 1 || method == 3 || method == 7 || method == 8;
    if (tid == 0) {
        const uint32_t cnt = method == 0 || method == 2 || method == 5 || method == 6 || method == 9 ? 1u
                             : method == 1 || method >= 7 ? 32u * nw
                             : method == 3          ? 1u + 32u * nw
                                                    : 1u;
        for (int i = 0; i < kBStages; ++i) {
            mbar_init(smem_u32(&g.full[i]), cnt);
            mbar_init(smem_u32(&g.empty[i]), 1);
        }
        g.abort_flag = 0;
        fence_mbar_init();
    }
    const int nidx = (method >= 7 ? 126 : 2) * ntile;
    for (int i = tid; i < nidx; i += 512) g.idx[i] = blocks[(size_t)blockIdx.x * nidx + i];
    __syncthreads();
    const long long t0 = clock64();
    // TMA / bulk issuer: methods 0, 2, 3, 5, 6 only (7 and 8 are cp.async alone;
    // an issuer arrival there would exceed the barrier's expected count)
    if (warp == 14 && (method == 0 || method == 2 || method == 3 || method == 5 || method == 6)) {
        if (lane == 0) {
            for (int u = 0; u < ntile; ++u) {
                const int st = u % kBStages;
                if (u >= kBStages &&
                    !mbar_wait(smem_u32(&g.empty[st]), ((u / kBStages) - 1) & 1, &g.abort_flag)) {
                    atomicExch(err, 1);
                    break;
                }
                const uint32_t fb = smem_u32(&g.full[st]), dst = smem_u32(g.ring[st]);
                const int b0 = g.idx[2 * u], b1 = g.idx[2 * u + 1];
                if (method == 0) {
                    mbar_arrive_expect_tx(fb, 16384);
                    tma_load_3d(dst, &map, 0, 0, b0, fb);
                    tma_load_3d(dst + 8192, &map, 0, 0, b1, fb);
                } else if (method >= 5) {
                    const uint32_t sd = smem_u32(g.scale[st]);
                    mbar_arrive_expect_tx(fb, 16384 + 512);
                    tma_load_3d(dst, &map, 0, 0, b0, fb);
                    if (method == 5)
                        bulk_load_g2s(sd, kv + (int64_t)b0 * 8448 + 8192, 256, fb);
                    else
                        tma_load_3d(sd, &smap, 0, 64, b0, fb);
                    tma_load_3d(dst + 8192, &map, 0, 0, b1, fb);
                    if (method == 5)
                        bulk_load_g2s(sd + 256, kv + (int64_t)b1 * 8448 + 8192, 256, fb);
                    else
                        tma_load_3d(sd + 256, &smap, 0, 64, b1, fb);
                } else if (method == 2) {
                    mbar_arrive_expect_tx(fb, 16384);
                    bulk_load_g2s(dst, kv + (int64_t)b0 * 8448, 8192, fb);
                    bulk_load_g2s(dst + 8192, kv + (int64_t)b1 * 8448, 8192, fb);
                } else {
                    mbar_arrive_expect_tx(fb, 8192);
                    tma_load_3d(dst, &map, 0, 0, b0, fb);
                }
            }
        }
        __syncwarp();
    } else if (method == 9 && warp == 14) {
        for (int u = 0; u < ntile; ++u) {
            const int st = u % kBStages;
            if (u >= kBStages &&
                !mbar_wait(smem_u32(&g.empty[st]), ((u / kBStages) - 1) & 1, &g.abort_flag)) {
                if (lane == 0) atomicExch(err, 1);
                break;
            }
            const uint32_t fb = smem_u32(&g.full[st]);
            if (lane == 0) mbar_arrive_expect_tx(fb, 14 * 1152);
            __syncwarp();
            if (lane < 14)
                bulk_load_g2s(smem_u32(g.ring[st]) + lane * 1152, kv + (int64_t)g.idx[u * 126 + lane] * 1152,
                              1152, fb);
            __syncwarp();
        }
    } else if (cp_side && warp < nw) {
        const int first = method == 3 ? 1 : 0;
        for (int u = 0; u < ntile; ++u) {
            const int st = u % kBStages;
            if (u >= kBStages &&
                !mbar_wait(smem_u32(&g.empty[st]), ((u / kBStages) - 1) & 1, &g.abort_flag)) {
                atomicExch(err, 1);
                break;
            }
            const uint32_t dst = smem_u32(g.ring[st]);
            if (method >= 7) {
                // 1008 pieces of 16 bytes: 14 rows x 72 (method 7) or 126 rows x 8 (method 8)
                const int per = method == 7 ? 72 : 8;
                for (int i = warp * 32 + lane; i < 1008; i += 32 * nw) {
                    const int r = i / per, c = i - r * per;
                    const int64_t slot = g.idx[u * 126 + r];
                    const int seg = method == 7 ? c : (u % 9) * 8 + c;
                    cp_async_16_zfill_nc(dst + i * 16, kv + slot * 1152 + seg * 16, true);
                }
                cp_async_mbar_arrive_noinc(smem_u32(&g.full[st]));
                continue;
            }
            for (int i = first * 512 + warp * 32 + lane; i < 1024; i += 32 * nw) {
                const int j = i >> 9, r = (i >> 3) & 63, c = i & 7;
                cp_async_16_zfill_nc(dst + j * 8192 + sw128_offset(r, c),
                                     kv + (int64_t)g.idx[2 * u + j] * 8448 + r * 128 + c * 16, true);
            }
            cp_async_mbar_arrive_noinc(smem_u32(&g.full[st]));
        }
        cp_async_wait_all();
    } else if (method == 4 && warp < nw) {
        for (int u = warp; u < ntile; u += nw) {
            const int st = u % kBStages;
            if (u >= kBStages &&
                !mbar_wait(smem_u32(&g.empty[st]), ((u / kBStages) - 1) & 1, &g.abort_flag)) {
                atomicExch(err, 1);
                break;
            }
            uint4 v[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                const int i = q * 32 + lane, j = i >> 9, r = (i >> 3) & 63, c = i & 7;
                v[q] = __ldg(reinterpret_cast<const uint4*>(kv + (int64_t)g.idx[2 * u + j] * 8448 +
                                                            r * 128 + c * 16));
            }
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                const int i = q * 32 + lane, j = i >> 9, r = (i >> 3) & 63, c = i & 7;
                *reinterpret_cast<uint4*>(g.ring[st] + j * 8192 + sw128_offset(r, c)) = v[q];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&g.full[st]));
        }
    } else if (warp == 15 && lane == 0) {
        for (int u = 0; u < ntile; ++u) {
            const int st = u % kBStages;
            if (!mbar_wait(smem_u32(&g.full[st]), (u / kBStages) & 1, &g.abort_flag)) {
                atomicExch(err, 1);
                break;
            }
            mbar_arrive(smem_u32(&g.empty[st]));
        }
        cycles[blockIdx.x] = clock64() - t0;
    }
    __syncthreads();
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int mlav_block_rate(
    const void* kv, long long nblk, const int32_t* blocks, int nctas, int ntile, int method, int nw,
    long long row_pool, long long* cycles, int* err) {
    CUtensorMap map, smap;
    if (!mlav::make_fp8_block_map(&map, kv, nblk) || !mlav::make_fp8_scale_map(&smap, kv, nblk))
        return -2;
    if (method < 0 || method > 9 || ntile < 1 || (method >= 7 ? 126 : 2) * ntile > kBMaxIdx ||
        nctas < 1)
        return -1;
    if ((method == 1 || method == 3 || method == 4 || method >= 7) && (nw < 1 || nw > 12)) return -1;
    if (method >= 7 && (row_pool < 1 || row_pool * 1152 > nblk * 8448 || row_pool > 0xffffffffLL))
        return -1;
    const int smem = (int)sizeof(BlockSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(block_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return (int)e;
    block_rate_kernel<<<nctas, 512, smem>>>(map, smap, static_cast<const unsigned char*>(kv), blocks, ntile,
                                            method, nw, row_pool, cycles, err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    return (int)cudaDeviceSynchronize();
}
