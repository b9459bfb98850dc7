// Decode steps beside the verify attention: greedy tree acceptance and KV
// relocation (see mla_decode_steps.h; the fp8 indexer is in fp8_indexer.cu).

#include "common.cuh"
#include "mla_decode_steps.h"

namespace mlav {
namespace {

// ---------------------------------------------------------------- tree acceptance
// One warp per request; lane l holds nodes l and l + 32. Each step ballots
// the children of the current node whose draft token equals the target's
// choice there and takes the lowest-numbered one.
__global__ void __launch_bounds__(32)
tree_accept_kernel(const int32_t* __restrict__ par, const int32_t* __restrict__ tok,
                   const int32_t* __restrict__ tgt, const int32_t* __restrict__ loc, int T,
                   int32_t* __restrict__ commit, int32_t* __restrict__ an, int32_t* __restrict__ ks,
                   int32_t* __restrict__ nt, int32_t* status) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    const int b = blockIdx.x, lane = threadIdx.x;
    const int64_t base = (int64_t)b * T;
    int p[2], k[2];
    bool ok[2];
    int bad = 0;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int c = lane + 32 * u;
        p[u] = c < T ? par[base + c] : -2;
        k[u] = c < T ? tok[base + c] : 0;
        ok[u] = c < T && (c == 0 ? p[u] == -1 : (p[u] >= 0 && p[u] < c));
        if (c < T && !ok[u]) bad = MLA_STATUS_BAD_PARENT;
        if (c < T) an[base + c] = ks[base + c] = nt[base + c] = -1;
    }
    __syncwarp();
    int cur = 0, n = 0;
    if (lane == 0) ks[base] = loc[base];
    for (int step = 0; step < T; ++step) {
        const int want = tgt[base + cur];
        const unsigned m0 = __ballot_sync(0xffffffffu, lane > 0 && ok[0] && p[0] == cur && k[0] == want);
        const unsigned m1 = __ballot_sync(0xffffffffu, ok[1] && p[1] == cur && k[1] == want);
        int nxt;
        if (m0)
            nxt = __ffs(m0) - 1;
        else if (m1)
            nxt = 32 + __ffs(m1) - 1;
        else
            break;
        if (lane == 0) {
            an[base + n] = nxt;
            nt[base + n] = tok[base + nxt];
            ks[base + n + 1] = loc[base + nxt];
        }
        ++n;
        cur = nxt;
    }
    if (lane == 0) {
        nt[base + n] = tgt[base + cur];
        commit[b] = n + 1;
    }
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (lane == 0) status_or(status, bad);
}

// ---------------------------------------------------------------- KV relocation
constexpr int kRelocRowsPerCta = 64;
constexpr int kRelocWarps = 8;
constexpr int kRowVec = kDqk * 2 / 16;  // 72 sixteen-byte pieces per 1152-byte row
constexpr int kRelocInFlight = 4;       // rows per warp whose loads are in flight together

__global__ void __launch_bounds__(kRelocWarps * 32)
kv_relocate_kernel(uint4* __restrict__ kv, int64_t pool_slots, int32_t* __restrict__ r2t,
                   int64_t stride, const int32_t* __restrict__ rpi, const int32_t* __restrict__ L,
                   const int32_t* __restrict__ dst, const int32_t* __restrict__ progress, int budget,
                   int32_t* status) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    const int b = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t len = L[b], j0 = progress[b];
    if (len < 0 || j0 < 0 || j0 > len) {
        if (threadIdx.x == 0 && blockIdx.x == 0) status_or(status, MLA_STATUS_BAD_PREFIX);
        return;
    }
    const int n = min(budget, len - j0);
    int32_t* row = r2t + (int64_t)rpi[b] * stride;
    const int r_end = min(n, (int)(blockIdx.x + 1) * kRelocRowsPerCta);
    int bad = 0;
    // Each warp moves kRelocInFlight rows per step: all their loads are in
    // flight before any of them is stored.
    for (int r0 = blockIdx.x * kRelocRowsPerCta + warp; r0 < r_end;
         r0 += kRelocInFlight * kRelocWarps) {
        int64_t s[kRelocInFlight], d[kRelocInFlight];
        bool mv[kRelocInFlight];
#pragma unroll
        for (int e = 0; e < kRelocInFlight; ++e) {
            const int r = r0 + e * kRelocWarps;
            mv[e] = false;
            s[e] = d[e] = -1;
            if (r < r_end) {
                const int j = j0 + r;
                s[e] = row[j];
                d[e] = (int64_t)dst[b] + j;
                if (s[e] < 0 || s[e] >= pool_slots || d[e] < 0 || d[e] >= pool_slots)
                    bad = MLA_STATUS_BAD_SLOT;
                else
                    mv[e] = s[e] != d[e];
            }
        }
        uint4 v[kRelocInFlight][3];
#pragma unroll
        for (int e = 0; e < kRelocInFlight; ++e)
#pragma unroll
            for (int u = 0; u < 3; ++u)
                if (mv[e] && lane + 32 * u < kRowVec) v[e][u] = __ldg(kv + s[e] * kRowVec + lane + 32 * u);
#pragma unroll
        for (int e = 0; e < kRelocInFlight; ++e)
#pragma unroll
            for (int u = 0; u < 3; ++u)
                if (mv[e] && lane + 32 * u < kRowVec) kv[d[e] * kRowVec + lane + 32 * u] = v[e][u];
        __syncwarp();
        if (lane == 0) {
#pragma unroll
            for (int e = 0; e < kRelocInFlight; ++e) {
                const int r = r0 + e * kRelocWarps;
                if (r < r_end && s[e] >= 0 && s[e] < pool_slots && d[e] >= 0 && d[e] < pool_slots)
                    row[j0 + r] = (int32_t)d[e];
            }
        }
    }
    if (lane == 0) status_or(status, bad);
}

__global__ void kv_relocate_progress_kernel(int32_t* progress, const int32_t* L, int batch,
                                            int budget) {
    pdl_launch_dependents();
    pdl_wait();  // after the copies have read the counters
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < batch) {
        const int32_t len = L[b], j0 = progress[b];
        if (len >= 0 && j0 >= 0 && j0 <= len) progress[b] = j0 + min(budget, len - j0);
    }
}

}  // namespace

cudaError_t launch_tree_accept(const int32_t* par, const int32_t* tok, const int32_t* tgt,
                               const int32_t* loc, int batch, int T, int32_t* commit, int32_t* an,
                               int32_t* ks, int32_t* nt, int32_t* status, cudaStream_t stream) {
    return launch_pdl(tree_accept_kernel, dim3(batch), dim3(32), 0, stream, par, tok, tgt, loc, T, commit,
                      an, ks, nt, status);
}

cudaError_t launch_kv_relocate(void* kv, int64_t pool_slots, int32_t* r2t, int64_t stride,
                               const int32_t* rpi, const int32_t* L, const int32_t* dst,
                               int32_t* progress, int batch, int budget, int32_t* status,
                               cudaStream_t stream) {
    dim3 grid((budget + kRelocRowsPerCta - 1) / kRelocRowsPerCta, batch);
    const cudaError_t e = launch_pdl(kv_relocate_kernel, grid, dim3(kRelocWarps * 32), 0, stream,
                                     static_cast<uint4*>(kv), pool_slots, r2t, stride, rpi, L, dst,
                                     static_cast<const int32_t*>(progress), budget, status);
    if (e != cudaSuccess) return e;
    return launch_pdl(kv_relocate_progress_kernel, dim3((batch + 127) / 128), dim3(128), 0, stream,
                      progress, L, batch, budget);
}

}  // namespace mlav
