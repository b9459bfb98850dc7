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
