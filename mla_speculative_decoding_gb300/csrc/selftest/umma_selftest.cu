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
