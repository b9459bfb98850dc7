// Log-sum-exp combine of the split-KV partials.
//
// The pages' verify kernel is a "partial + reduce" design (The Custom
// sm_120 Verify Kernel..., Part VII); the reduce is written out here as the
// log-sum-exp merge: with per-split (o_s, lse_s),
//   lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s,
// splits with lse_s = -inf weighing 0. Four warps per query row, one per
// 128 output dims: lanes hold the split lse values (max and sum by warp
// shuffles), then each lane streams its 4 dims of every split with weight
// with 16-byte loads (coalesced 512 bytes per warp and split, sixteen
// splits in flight; sparse groups of splits visit only the weighted ones),
// summing splits in index order (deterministic), and rounds to bf16
// (nearest even).
#include "common.cuh"

namespace mlav {
namespace {

constexpr int kWarps = 8;
constexpr int kParts = 4;                          // warps per row
constexpr int kMaxPerLane = MLA_MAX_NSPLIT / 32;   // split lse values held per lane
constexpr int kUnroll = 16;                        // splits in flight per lane

__global__ void __launch_bounds__(kWarps * 32)
combine_kernel(const float* __restrict__ lse_part, const float* __restrict__ o_part, int rows,
               int nsplit, __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
               int32_t* status) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t n = gw / kParts;
    const int part = (int)(gw % kParts);
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
    __nv_bfloat16* dst = out + n * kDv + part * 128 + 4 * lane;
    if (mx == -INFINITY) {  // no split saw a visible key: empty row
        *reinterpret_cast<uint2*>(dst) = make_uint2(0, 0);
        if (lane == 0 && part == 0) {
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
    if (lane == 0 && part == 0) lse[n] = mx + logf(sum);

    // Splits in index order, sixteen loads in flight. A group of 32 with
    // more than sixteen weighted splits is streamed whole (zero weights skip
    // their loads); a sparser one visits only its weighted splits (a ballot),
    // which is what the balanced four-SM plan leaves (most splits empty).
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4* op = reinterpret_cast<const float4*>(o_part + n * nsplit * (int64_t)kDv) +
                       part * 32 + lane;
    auto accumulate = [&](const float (&ws)[kUnroll], const float4 (&x)[kUnroll]) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            acc.x = fmaf(ws[u], x[u].x, acc.x);
            acc.y = fmaf(ws[u], x[u].y, acc.y);
            acc.z = fmaf(ws[u], x[u].z, acc.z);
            acc.w = fmaf(ws[u], x[u].w, acc.w);
        }
    };
#pragma unroll
    for (int g = 0; g < kMaxPerLane; ++g) {
        if (g * 32 >= nsplit) break;
        uint32_t live = __ballot_sync(0xffffffffu, w[g] != 0.f);  // warp-uniform
        if (__popc(live) > kUnroll) {
            for (int s0 = 0; s0 < 32; s0 += kUnroll) {
                if (g * 32 + s0 >= nsplit) break;
                float4 x[kUnroll];
                float ws[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int s = g * 32 + s0 + u;
                    ws[u] = __shfl_sync(0xffffffffu, w[g], s0 + u) * inv;
                    x[u] = (s < nsplit && ws[u] != 0.f) ? op[s * (kDv / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                accumulate(ws, x);
            }
        } else if (live != 0u) {
            float4 x[kUnroll];
            float ws[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const bool have = live != 0u;
                const int j = have ? __ffs((int)live) - 1 : 0;
                const float wj = __shfl_sync(0xffffffffu, w[g], j) * inv;
                ws[u] = have ? wj : 0.f;
                x[u] = have ? op[(g * 32 + j) * (kDv / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
                live &= live - 1u;  // next set bit (no change once empty)
            }
            accumulate(ws, x);
        }
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t*>(&lo);
    pk.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst) = pk;
}

}  // namespace

cudaError_t launch_combine(const float* lse_part, const float* o_part, int rows, int nsplit,
                           __nv_bfloat16* out, float* lse, int32_t* status, cudaStream_t stream) {
    const int64_t warps = (int64_t)rows * kParts;
    const int blocks = (int)((warps + kWarps - 1) / kWarps);
    return launch_pdl(combine_kernel, dim3(blocks), dim3(kWarps * 32), 0, stream, lse_part, o_part, rows,
                      nsplit, out, lse, status);
}

}  // namespace mlav
