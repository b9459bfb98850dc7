// Split-KV partial attention on CUDA cores (fp32 FMA), the plain path.
//
// One block per (row block of 16 query rows, split s, request b). The
// block walks its split's keys in tiles of 32: it gathers the 32 scattered
// 1152-byte latent rows into shared memory with 16-byte loads (the pages'
// "128-bit vectorized bf16 KV loads", The Custom sm_120 Verify Kernel...,
// Part VII), scores them against its 16 rows, applies the tree mask only to
// keys past the prefix (Part VII), keeps an online softmax per row, and
// accumulates the first 512 dims as V. It writes one partial (normalised
// o, natural-log lse) per (row, split) for the combine kernel.
//
// This is the shape-agnostic path (any T, H, nsplit within the limits);
// the tensor-core kernel is the fast path.
#include "common.cuh"

namespace mlav {
namespace {

constexpr int kThreads = 256;  // 8 warps
constexpr int kRows = 16;      // query rows per block, 2 per warp
constexpr int kKeys = 32;      // keys per tile, one per lane when scoring
constexpr int kChunks = kDqk / 8;    // 16-byte chunks per latent row (72)
constexpr int kKvStride = kDqk + 8;  // padded smem row: 1168 B, conflict-free 16-B reads

struct SmemSimt {
    __nv_bfloat16 q[kRows][kDqk];
    __nv_bfloat16 kv[kKeys][kKvStride];
    float p[kRows][kKeys];
    float alpha[kRows];
    float row_m[kRows];
    float row_l[kRows];
    int32_t slot[kKeys];
    uint64_t anc[MLA_MAX_TREE];
};

__device__ __forceinline__ float warp_max(float v) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float dot8(const uint4& a, const uint4& b, float acc) {
    const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 fx = __bfloat1622float2(x[i]);
        const float2 fy = __bfloat1622float2(y[i]);
        acc = fmaf(fx.x, fy.x, acc);
        acc = fmaf(fx.y, fy.y, acc);
    }
    return acc;
}

__global__ void __launch_bounds__(kThreads) partial_simt_kernel(const PartialArgs a) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SmemSimt& sm = *reinterpret_cast<SmemSimt*>(smem_raw);
    const int rb = blockIdx.x, s = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.T, H = a.H;
    const int rows_req = T * H;
    const int row0 = rb * kRows;
    int bad = 0;

    int Lb, K;
    bad |= request_keys(a, b, Lb, K);
    const int64_t kbase = key_base(a, b);
    int kb, ke;
    split_range(K, a.nsplit, s, kb, ke);

    if (tid == 0) {
        if (a.anc_mask != nullptr) {
            for (int t = 0; t < T; ++t) sm.anc[t] = a.anc_mask[(int64_t)b * T + t];
        } else {
            bad |= build_anc_serial(a.tree_parent + (int64_t)b * T, T, sm.anc);
        }
    }
    for (int c = tid; c < kRows * kChunks; c += kThreads) {
        const int r = c / kChunks, ch = c % kChunks;
        const int row = row0 + r;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < rows_req)
            v = __ldg(reinterpret_cast<const uint4*>(a.q + ((int64_t)b * rows_req + row) * kDqk) + ch);
        *reinterpret_cast<uint4*>(&sm.q[r][ch * 8]) = v;
    }

    float m[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.f, 0.f};
    float acc[kRows][2];
#pragma unroll
    for (int r = 0; r < kRows; ++r) acc[r][0] = acc[r][1] = 0.f;

    // Token index of the two rows this warp scores (-1 = padding row).
    int tok[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int row = row0 + 2 * warp + rr;
        tok[rr] = row < rows_req ? row / H : -1;
    }
    __syncthreads();

    for (int k0 = kb; k0 < ke; k0 += kKeys) {
        if (tid < kKeys) {
            const int j = k0 + tid;
            int32_t sl = -1;
            if (j < ke) {
                sl = key_slot(a, b, kbase, Lb, j);
                if (sl < 0 || (int64_t)sl >= a.pool_slots) {
                    bad |= MLA_STATUS_BAD_SLOT;
                    sl = -1;
                }
            }
            sm.slot[tid] = sl;
        }
        __syncthreads();
        for (int c = tid; c < kKeys * kChunks; c += kThreads) {
            const int k = c / kChunks, ch = c % kChunks;
            const int32_t sl = sm.slot[k];
            uint4 v = make_uint4(0, 0, 0, 0);
            if (sl >= 0) v = __ldg(reinterpret_cast<const uint4*>(a.kv + (int64_t)sl * kDqk) + ch);
            *reinterpret_cast<uint4*>(&sm.kv[k][ch * 8]) = v;
        }
        __syncthreads();

        const int j = k0 + lane;
        const bool key_ok = (j < ke) && sm.slot[lane] >= 0;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int r = 2 * warp + rr;
            float dot = 0.f;
            const uint4* qr = reinterpret_cast<const uint4*>(&sm.q[r][0]);
            const uint4* kr = reinterpret_cast<const uint4*>(&sm.kv[lane][0]);
#pragma unroll 8
            for (int ch = 0; ch < kChunks; ++ch) dot = dot8(qr[ch], kr[ch], dot);
            bool vis = key_ok && tok[rr] >= 0;
            if (vis && j >= Lb) {
                const int u = j - Lb;
                vis = (u < T) && ((sm.anc[tok[rr]] >> u) & 1ull);
            }
            const float sv = vis ? dot * a.scale_log2 : -INFINITY;
            const float m_new = fmaxf(m[rr], warp_max(sv));
            const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m[rr] - m_new);
            const float p = vis ? exp2f(sv - m_new) : 0.f;
            l[rr] = l[rr] * alpha + warp_sum(p);
            m[rr] = m_new;
            sm.p[r][lane] = p;
            if (lane == 0) sm.alpha[r] = alpha;
        }
        __syncthreads();

#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const float al = sm.alpha[r];
            acc[r][0] *= al;
            acc[r][1] *= al;
        }
        for (int k = 0; k < kKeys; ++k) {
            const float2 v = __bfloat1622float2(
                *reinterpret_cast<const __nv_bfloat162*>(&sm.kv[k][2 * tid]));
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const float p = sm.p[r][k];
                acc[r][0] = fmaf(p, v.x, acc[r][0]);
                acc[r][1] = fmaf(p, v.y, acc[r][1]);
            }
        }
        __syncthreads();
    }

    if (lane == 0) {
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            sm.row_m[2 * warp + rr] = m[rr];
            sm.row_l[2 * warp + rr] = l[rr];
        }
    }
    __syncthreads();
    for (int r = 0; r < kRows; ++r) {
        const int row = row0 + r;
        if (row >= rows_req) break;
        const int64_t part = ((int64_t)b * rows_req + row) * a.nsplit + s;
        const float lr = sm.row_l[r];
        const float inv = lr > 0.f ? 1.f / lr : 0.f;
        float2 o = make_float2(acc[r][0] * inv, acc[r][1] * inv);
        reinterpret_cast<float2*>(a.o_part + part * kDv)[tid] = o;
        if (tid == 0) a.lse_part[part] = lr > 0.f ? (sm.row_m[r] + log2f(lr)) * kLn2 : -INFINITY;
    }
    status_or(a.status, bad);
}

}  // namespace

cudaError_t setup_partial_simt() {
    return cudaFuncSetAttribute(partial_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sizeof(SmemSimt));
}

cudaError_t launch_partial_simt(const PartialArgs& a, cudaStream_t stream) {
    const int rows_req = a.T * a.H;
    dim3 grid((rows_req + kRows - 1) / kRows, a.nsplit, a.batch);
    return launch_pdl(partial_simt_kernel, grid, dim3(kThreads), sizeof(SmemSimt), stream, a);
}

}  // namespace mlav
