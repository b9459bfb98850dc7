// Log-sum-exp combine of the split-KV partials.
//
// The pages' verify kernel is a "partial + reduce" design (The Custom
// sm_120 Verify Kernel..., Part VII); the reduce is written out here as the
// log-sum-exp merge: with per-split (o_s, lse_s),
//   lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s,
// splits with lse_s = -inf weighing 0.
//
// A block takes max(1, 4 / P) query rows with 64 * P threads per row (256
// threads; 512 for P = 8, 1024 for P = 16): one warp per row first reads the row's split lse
// values (max and sum by warp shuffles) and lists the splits with non-zero
// weight, in index order, in shared memory; then each of the row's P split
// groups takes every P-th listed split, each thread 8 output dims (two
// 16-byte loads per split, up to four splits in flight), and group 0 adds
// the groups' sums in group order (deterministic), rounds to bf16 (nearest
// even) and stores. P is chosen from the splits a row is expected to hold
// (the launcher's estimate) so that a row's loads go out in one or two
// rounds: few for the four-SM kernel's balanced plan on many requests, up to
// nsplit for the two-SM kernel's partitions.
#include "common.cuh"

namespace mlav {
namespace {

constexpr int kMaxPerLane = MLA_MAX_NSPLIT / 32;   // split lse values held per lane
constexpr int kInFlight = 4;                       // splits in flight per thread

template <int P>
__global__ void __launch_bounds__(P > 4 ? 64 * P : 256)
combine_kernel(const float* __restrict__ lse_part, const float* __restrict__ o_part, int rows,
               int nsplit, __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
               int32_t* status) {
    constexpr int kThreads = P > 4 ? 64 * P : 256;
    constexpr int kRowsPerBlock = kThreads / (64 * P);
    __shared__ int live_s[kRowsPerBlock][MLA_MAX_NSPLIT];
    __shared__ float w_s[kRowsPerBlock][MLA_MAX_NSPLIT];
    __shared__ int nlive_s[kRowsPerBlock];
    __shared__ float4 part_s[P > 1 ? (P - 1) * kRowsPerBlock * 64 * 2 : 1];
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- weights: one warp per row
    if (warp < kRowsPerBlock) {
        const int64_t n = (int64_t)blockIdx.x * kRowsPerBlock + warp;
        int nlive = 0;
        if (n < rows) {
            const float* lp = lse_part + n * nsplit;
            float v[kMaxPerLane];
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < kMaxPerLane; ++i) {
                const int s = lane + 32 * i;
                v[i] = s < nsplit ? lp[s] : -INFINITY;
                mx = fmaxf(mx, v[i]);
            }
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (mx == -INFINITY) {  // no split saw a visible key: empty row
                if (lane == 0) {
                    lse[n] = -INFINITY;
                    status_or(status, MLA_STATUS_EMPTY_ROW);
                }
            } else {
                float w[kMaxPerLane];
                float sum = 0.f;
#pragma unroll
                for (int i = 0; i < kMaxPerLane; ++i) {
                    w[i] = (v[i] == -INFINITY) ? 0.f : expf(v[i] - mx);
                    sum += w[i];
                }
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                const float inv = 1.f / sum;
                if (lane == 0) lse[n] = mx + logf(sum);
#pragma unroll
                for (int i = 0; i < kMaxPerLane; ++i) {  // list the weighted splits in index order
                    const uint32_t m = __ballot_sync(0xffffffffu, w[i] != 0.f);
                    if (w[i] != 0.f) {
                        const int at = nlive + __popc(m & ((1u << lane) - 1u));
                        live_s[warp][at] = lane + 32 * i;
                        w_s[warp][at] = w[i] * inv;
                    }
                    nlive += __popc(m);
                }
            }
        }
        if (lane == 0) nlive_s[warp] = nlive;
    }
    __syncthreads();

    // ---- weighted sum: P split groups per row, 8 dims per thread
    const int rl = tid / (64 * P);
    const int g = (tid / 64) % P;
    const int q = tid & 63;
    const int64_t n = (int64_t)blockIdx.x * kRowsPerBlock + rl;
    const bool row_ok = n < rows;  // a missing row's threads still reach the barrier below
    const int nlive = row_ok ? nlive_s[rl] : 0;
    const float4* op =
        reinterpret_cast<const float4*>(o_part + (row_ok ? n : 0) * nsplit * (int64_t)kDv) + 2 * q;
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
    for (int i0 = g; i0 < nlive; i0 += kInFlight * P) {
        float4 x0[kInFlight], x1[kInFlight];
        float ws[kInFlight];
#pragma unroll
        for (int u = 0; u < kInFlight; ++u) {
            const int i = i0 + u * P;
            const bool have = i < nlive;
            ws[u] = have ? w_s[rl][i] : 0.f;
            const float4* src = op + (have ? (int64_t)live_s[rl][i] * (kDv / 4) : 0);
            x0[u] = have ? src[0] : make_float4(0.f, 0.f, 0.f, 0.f);
            x1[u] = have ? src[1] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kInFlight; ++u) {
            a0.x = fmaf(ws[u], x0[u].x, a0.x);
            a0.y = fmaf(ws[u], x0[u].y, a0.y);
            a0.z = fmaf(ws[u], x0[u].z, a0.z);
            a0.w = fmaf(ws[u], x0[u].w, a0.w);
            a1.x = fmaf(ws[u], x1[u].x, a1.x);
            a1.y = fmaf(ws[u], x1[u].y, a1.y);
            a1.z = fmaf(ws[u], x1[u].z, a1.z);
            a1.w = fmaf(ws[u], x1[u].w, a1.w);
        }
    }
    if constexpr (P > 1) {
        if (g > 0) {
            float4* ps = part_s + (((g - 1) * kRowsPerBlock + rl) * 64 + q) * 2;
            ps[0] = a0;
            ps[1] = a1;
        }
        __syncthreads();
        if (g > 0) return;
#pragma unroll
        for (int gg = 1; gg < P; ++gg) {
            const float4* ps = part_s + (((gg - 1) * kRowsPerBlock + rl) * 64 + q) * 2;
            const float4 b0 = ps[0], b1 = ps[1];
            a0.x += b0.x; a0.y += b0.y; a0.z += b0.z; a0.w += b0.w;
            a1.x += b1.x; a1.y += b1.y; a1.z += b1.z; a1.w += b1.w;
        }
    }
    if (!row_ok) return;
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(a0.x, a0.y);
    const __nv_bfloat162 h1 = __floats2bfloat162_rn(a0.z, a0.w);
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(a1.x, a1.y);
    const __nv_bfloat162 h3 = __floats2bfloat162_rn(a1.z, a1.w);
    uint4 pk;
    pk.x = *reinterpret_cast<const uint32_t*>(&h0);
    pk.y = *reinterpret_cast<const uint32_t*>(&h1);
    pk.z = *reinterpret_cast<const uint32_t*>(&h2);
    pk.w = *reinterpret_cast<const uint32_t*>(&h3);
    *reinterpret_cast<uint4*>(out + n * kDv + 8 * q) = pk;  // zeros for an empty row
}

}  // namespace

cudaError_t launch_combine(const float* lse_part, const float* o_part, int rows, int nsplit,
                           int live_hint, __nv_bfloat16* out, float* lse, int32_t* status,
                           cudaStream_t stream) {
    if (live_hint <= 4)
        return launch_pdl(combine_kernel<1>, dim3((rows + 3) / 4), dim3(256), 0, stream, lse_part,
                          o_part, rows, nsplit, out, lse, status);
    if (live_hint <= 8)
        return launch_pdl(combine_kernel<2>, dim3((rows + 1) / 2), dim3(256), 0, stream, lse_part,
                          o_part, rows, nsplit, out, lse, status);
    if (live_hint <= 16)
        return launch_pdl(combine_kernel<4>, dim3(rows), dim3(256), 0, stream, lse_part, o_part, rows,
                          nsplit, out, lse, status);
    if (live_hint <= 32)
        return launch_pdl(combine_kernel<8>, dim3(rows), dim3(512), 0, stream, lse_part, o_part, rows,
                          nsplit, out, lse, status);
    return launch_pdl(combine_kernel<16>, dim3(rows), dim3(1024), 0, stream, lse_part, o_part, rows,
                      nsplit, out, lse, status);
}

}  // namespace mlav
