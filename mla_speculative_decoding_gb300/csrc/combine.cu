// Log-sum-exp combine of the split-KV partials.
//
// The pages' verify kernel is a "partial + reduce" design (The Custom
// sm_120 Verify Kernel..., Part VII); the reduce is written out here as the
// log-sum-exp merge: with per-split (o_s, lse_s),
//   lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s,
// splits with lse_s = -inf weighing 0. One warp per query row: lanes hold
// the split lse values (max and sum by warp shuffles), then sweep the 512
// output dims with 16-byte loads, summing splits in index order
// (deterministic), and round to bf16 (nearest even).
#include "common.cuh"

namespace mlav {
namespace {

constexpr int kWarps = 8;
constexpr int kMaxPerLane = MLA_MAX_NSPLIT / 32;  // split lse values held per lane

__global__ void __launch_bounds__(kWarps * 32)
combine_kernel(const float* __restrict__ lse_part, const float* __restrict__ o_part, int rows,
               int nsplit, __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
               int32_t* status) {
    const int lane = threadIdx.x & 31;
    const int64_t n = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (n >= rows) return;
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
    __nv_bfloat16* dst = out + n * kDv;
    if (mx == -INFINITY) {
        // No split saw a visible key: empty row.
        for (int d = lane * 4; d < kDv; d += 128) {
            *reinterpret_cast<uint2*>(dst + d) = make_uint2(0, 0);
        }
        if (lane == 0) {
            lse[n] = -INFINITY;
            status_or(status, MLA_STATUS_EMPTY_ROW);
        }
        return;
    }
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

    float4 acc[kDv / 128];
#pragma unroll
    for (int i = 0; i < kDv / 128; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4* op = reinterpret_cast<const float4*>(o_part + n * nsplit * (int64_t)kDv);
#pragma unroll
    for (int g = 0; g < kMaxPerLane; ++g) {
        for (int sl = 0; sl < 32; ++sl) {
            const int s = g * 32 + sl;
            if (s >= nsplit) break;
            const float ws = __shfl_sync(0xffffffffu, w[g], sl) * inv;
            if (ws == 0.f) continue;  // uniform across the warp
#pragma unroll
            for (int i = 0; i < kDv / 128; ++i) {
                const float4 x = op[s * (kDv / 4) + lane + 32 * i];
                acc[i].x = fmaf(ws, x.x, acc[i].x);
                acc[i].y = fmaf(ws, x.y, acc[i].y);
                acc[i].z = fmaf(ws, x.z, acc[i].z);
                acc[i].w = fmaf(ws, x.w, acc[i].w);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kDv / 128; ++i) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[i].x, acc[i].y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[i].z, acc[i].w);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t*>(&lo);
        pk.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(dst + 4 * (lane + 32 * i)) = pk;
    }
}

}  // namespace

cudaError_t launch_combine(const float* lse_part, const float* o_part, int rows, int nsplit,
                           __nv_bfloat16* out, float* lse, int32_t* status, cudaStream_t stream) {
    const int blocks = (rows + kWarps - 1) / kWarps;
    combine_kernel<<<blocks, kWarps * 32, 0, stream>>>(lse_part, o_part, rows, nsplit, out, lse,
                                                      status);
    return cudaGetLastError();
}

}  // namespace mlav
