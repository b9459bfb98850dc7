// Shared definitions of the MLA tree-verify attention library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "mla_verify.h"
#include "partition.h"

#define MLAV_API extern "C" __attribute__((visibility("default")))

namespace mlav {

constexpr int kDqk = 576;  // 512 latent + 64 RoPE dims
constexpr int kDv = 512;   // V = first 512 dims of the latent row
constexpr size_t kWsHeader = 256;  // status word + padding
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__host__ __device__ constexpr size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace layout: [header 256 B | lse_part fp32 [rows*nsplit] padded to
// 256 B | o_part fp32 [rows*nsplit][512]].
struct WsLayout {
    size_t lse_off;
    size_t o_off;
    size_t total;
};

__host__ __device__ inline WsLayout ws_layout(int batch, int T, int H, int nsplit) {
    const size_t parts = (size_t)batch * T * H * nsplit;
    WsLayout w;
    w.lse_off = kWsHeader;
    w.o_off = w.lse_off + round_up(parts * sizeof(float), 256);
    w.total = w.o_off + parts * kDv * sizeof(float);
    return w;
}


// Programmatic dependent launch. The verify path's kernels are launched
// with the programmatic stream-serialization attribute, so each may start
// (and set up its shared memory, TMEM and barriers) while the kernel before
// it on the stream is still running. pdl_wait() blocks until that kernel has
// completed and its writes are visible: every kernel calls it before its
// first global memory access, which by induction orders it after all
// earlier work on the stream. pdl_launch_dependents() lets the next kernel
// start early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Host: launches `kernel` with the programmatic stream-serialization attribute.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ void status_or(int32_t* st, int bits) {
    if (st != nullptr && bits != 0) atomicOr(st, bits);
}

// Ancestor-or-self masks of one request's tree, built in shared memory from
// parent links (parents precede children). A node whose parent is invalid is
// treated as a root and flagged. Called by one thread.
__device__ inline int build_anc_serial(const int32_t* par, int T, uint64_t* anc) {
    int bad = 0;
    for (int t = 0; t < T; ++t) {
        const int p = par[t];
        const bool ok = (t == 0) ? (p == -1) : (p >= 0 && p < t);
        if (!ok) bad = MLA_STATUS_BAD_PARENT;
        anc[t] = ((t > 0 && ok) ? anc[p] : 0ull) | (1ull << t);
    }
    return bad;
}

// The same sets built by one full warp by pointer jumping: each node t
// starts from {t} and its parent as pointer; round r ORs in the set of the
// node its pointer names and doubles the pointer's stride, so after six
// rounds every set spans the whole root path (depth <= 63). An invalid parent
// ends the path at the node itself, as in build_anc_serial. `ptr` is warp-
// private shared scratch of MLA_MAX_TREE entries. Returns the status bits
// (on every lane).
__device__ inline int build_anc_warp(const int32_t* par, int T, uint64_t* anc, int* ptr) {
    const int lane = threadIdx.x & 31;
    int bad = 0;
    for (int t = lane; t < MLA_MAX_TREE; t += 32) {
        int p = -1;
        if (t < T) {
            p = par[t];
            const bool ok = (t == 0) ? (p == -1) : (p >= 0 && p < t);
            if (!ok) {
                bad = MLA_STATUS_BAD_PARENT;
                p = -1;
            }
        }
        ptr[t] = p;
        anc[t] = t < T ? (1ull << t) : 0ull;
    }
    __syncwarp();
#pragma unroll 1
    for (int r = 0; r < 6; ++r) {
        uint64_t add[2] = {0ull, 0ull};
        int nxt[2] = {-1, -1};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int t = lane + 32 * u, q = ptr[t];
            if (q >= 0) {
                add[u] = anc[q];
                nxt[u] = ptr[q];
            }
        }
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int t = lane + 32 * u;
            anc[t] |= add[u];
            ptr[t] = nxt[u];
        }
        __syncwarp();
    }
    return __reduce_or_sync(0xffffffffu, bad);
}

// Visibility bits of 32 consecutive keys of a request, the first of which has
// tree index u0 (key L_b + u0): keys with a negative tree index are prefix
// keys, always visible; tree key u is visible iff bit u of `anc`, the row's
// ancestor-or-self mask with no bit at or above T, is set.
__device__ __forceinline__ uint32_t tree_keep_word(uint64_t anc, int u0) {
    if (u0 >= 64) return 0u;
    if (u0 >= 0) return (uint32_t)(anc >> u0);
    if (u0 <= -32) return 0xffffffffu;
    return (uint32_t)(anc << (-u0)) | ((1u << (-u0)) - 1u);
}
// Pairs of fp32 values in one 64-bit register (packed two-lane arithmetic,
// one instruction for two keys) and a three-input maximum.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Maximum of 128 scores in eight independent chains of three-input maxima.
__device__ __forceinline__ float max128(const float (&sc)[128]) {
    float m8[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) m8[j] = fmaxf(sc[j], sc[8 + j]);
#pragma unroll
    for (int c = 16; c < 128; c += 16)
#pragma unroll
        for (int j = 0; j < 8; ++j) m8[j] = fmax3(m8[j], sc[c + j], sc[c + 8 + j]);
    return fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
}

// The bits below T of a 64-bit mask.
__device__ __forceinline__ uint64_t tree_bits(int T) { return T >= 64 ? ~0ull : ((1ull << T) - 1ull); }

struct PartialArgs;

// Internal launchers (defined in the kernel translation units).
struct PartialArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* kv;
    const int32_t* kv_indices;
    const int32_t* kv_indptr;
    const int32_t* prefix_lens;
    const int32_t* tree_parent;  // exactly one of tree_parent / anc_mask
    const uint64_t* anc_mask;
    float* lse_part;
    float* o_part;
    int32_t* status;
    int batch, T, H, nsplit;
    int64_t pool_slots;
    float scale_log2;  // softmax_scale * log2(e)
    int wave_full;     // first item of the last, partial wave (split_range_waves)
    int parts;         // > 0: the two-SM kernel's split over this many partitions,
                       // all in one wave (split_range_one_wave); 0: wave-shaped
    // Paged form (kv_indices == nullptr): request b's keys are its table row
    // req_to_token[req_pool_indices[b]][0, L_b) followed by its T draft slots
    // out_cache_loc[b*T, b*T + T), read where the combined list would be.
    const int32_t* req_to_token;
    int64_t r2t_stride, r2t_rows;
    const int32_t* req_pool_indices;
    const int32_t* out_cache_loc;
};

// Prefix length and key count of request b, made consistent: a negative
// prefix counts as 0, and the key count is clamped to [0, L_b + T] (surplus
// keys are ignored, missing ones are absent). Returns the status bits.
__device__ inline int request_keys(const PartialArgs& a, int b, int& Lb, int& K) {
    int bad = 0;
    if (a.kv_indices == nullptr) {  // paged form: the builder's clamping, K = L_b + T
        Lb = a.prefix_lens[b];
        const int32_t r = a.req_pool_indices[b];
        if (r < 0 || r >= a.r2t_rows) {
            bad |= MLA_STATUS_BAD_PREFIX;
            Lb = 0;
        } else if (Lb < 0) {
            bad |= MLA_STATUS_BAD_PREFIX;
            Lb = 0;
        } else if (Lb > a.r2t_stride) {
            bad |= MLA_STATUS_BAD_PREFIX;
            Lb = (int)a.r2t_stride;
        }
        K = Lb + a.T;
        return bad;
    }
    Lb = a.prefix_lens[b];
    if (Lb < 0) {
        Lb = 0;
        bad |= MLA_STATUS_BAD_INDPTR;
    }
    K = a.kv_indptr[b + 1] - a.kv_indptr[b];
    if (K != Lb + a.T) bad |= MLA_STATUS_BAD_INDPTR;
    K = max(0, min(K, Lb + a.T));
    return bad;
}

// Where request b's keys start: its offset in the combined list, or, in the
// paged form, its table row's offset (0 for a row out of range, whose prefix
// request_keys has cut to nothing).
__device__ __forceinline__ int64_t key_base(const PartialArgs& a, int b) {
    if (a.kv_indices != nullptr) return a.kv_indptr[b];
    const int32_t r = a.req_pool_indices[b];
    return (r >= 0 && r < a.r2t_rows) ? (int64_t)r * a.r2t_stride : 0;
}

// Warms L2 with the slot entries of keys [j0, j1) of request b, one 128-byte
// line (32 entries) per lane step, so that the row staging of the tiles to
// come finds them there (the paged form reads the table, which no kernel
// has just written).
__device__ __forceinline__ void key_prefetch(const PartialArgs& a, int b, int64_t base, int Lb, int j0,
                                             int j1, int lane) {
    for (int j = j0 + 32 * lane; j < j1; j += 32 * 32) {
        const int32_t* p = a.kv_indices != nullptr ? a.kv_indices + base + j
                           : j < Lb ? a.req_to_token + base + j
                                    : a.out_cache_loc + (int64_t)b * a.T + (j - Lb);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
    }
}

// Pool rows of one tile of kTile keys starting at key j0 (and, for the
// softmax, their validity bits).
// Returns MLA_STATUS_BAD_SLOT if a slot was out of range (that key is masked).
// The source is chosen once per tile (one base for all the lanes' loads, as for
// the combined list): the table row while the tile is in the prefix, the
// draft slots after it; the one tile that straddles L_b takes its draft
// keys in a second pass.
template <int kTile>
__device__ __forceinline__ int stage_rows(const PartialArgs& a, int b, int64_t kbase, int Lb, int j0,
                                          int ke, int lane, int32_t* rows, uint32_t* valid) {
    int bad = 0;
    constexpr int kQ = kTile / 32;
    int32_t v[kQ];
    const bool paged = a.kv_indices == nullptr;
    const int32_t* src;
    int lim = ke;
    if (!paged) {
        src = a.kv_indices + kbase;
    } else if (j0 < Lb) {
        src = a.req_to_token + kbase;
        lim = min(ke, Lb);
    } else {
        src = a.out_cache_loc + ((int64_t)b * a.T - Lb);
    }
#pragma unroll
    for (int q = 0; q < kQ; ++q) {  // all the loads in flight together
        const int j = j0 + 32 * q + lane;
        v[q] = j < lim ? __ldg(src + j) : -1;
    }
    if (paged && j0 < Lb && j0 + kTile > Lb) {  // through shared memory: each lane its own entries
        const int32_t* dsrc = a.out_cache_loc + ((int64_t)b * a.T - Lb);
#pragma unroll
        for (int q = 0; q < kQ; ++q) rows[32 * q + lane] = v[q];
#pragma unroll 1
        for (int q = 0; q < kQ; ++q) {
            const int j = j0 + 32 * q + lane;
            if (j >= Lb && j < ke) rows[32 * q + lane] = __ldg(dsrc + j);
        }
#pragma unroll
        for (int q = 0; q < kQ; ++q) v[q] = rows[32 * q + lane];
    }
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
        if (v[q] < -1 || (v[q] >= 0 && (int64_t)v[q] >= a.pool_slots) ||
            (v[q] == -1 && j0 + 32 * q + lane < ke)) {
            bad |= MLA_STATUS_BAD_SLOT;
            v[q] = -1;
        }
        rows[32 * q + lane] = v[q];
        if (valid != nullptr) {
            const uint32_t w = __ballot_sync(0xffffffffu, v[q] >= 0);
            if (lane == q) valid[q] = w;
        }
    }
    return bad;
}

// Host-side checks of mla_verify_attention's arguments (api.cu); the
// library's per-device set-up on the current device, run lazily outside
// stream capture (MLA_ERR_NOT_INITIALIZED inside it); the allocation-free
// entry point's per-device scratch look-up (noalloc.cu), run by that set-up.
int check_attention_args(const void* q, const void* kv_pool, const int32_t* kv_indices,
                         const int32_t* kv_indptr, const int32_t* prefix_lens,
                         const int32_t* tree_parent, int T, int nsplit, const void* workspace,
                         const void* out, const float* lse, int batch, int num_heads,
                         int64_t pool_slots, float softmax_scale, size_t workspace_bytes);
int ensure_device_ready(cudaStream_t stream);
cudaError_t setup_noalloc(int device);

// `live_hint`: the number of splits with keys a row is expected to have
// (it only sets how the combine spreads a row's splits over threads).
cudaError_t launch_combine(const float* lse_part, const float* o_part, int rows, int nsplit,
                           int live_hint, __nv_bfloat16* out, float* lse, int32_t* status,
                           cudaStream_t stream);

cudaError_t launch_build_meta(const int32_t* req_to_token, int64_t stride, int64_t rows,
                              const int32_t* req_pool_indices, const int32_t* prefix_lens,
                              const int32_t* out_cache_loc, const int32_t* tree_parent,
                              int batch, int T, int64_t capacity, int32_t* kv_indptr,
                              int32_t* kv_indices, uint64_t* anc, int32_t* status,
                              cudaStream_t stream);

// Decode steps beside the verify attention (decode_steps.cu, fp8_indexer.cu).
cudaError_t launch_tree_accept(const int32_t* par, const int32_t* tok, const int32_t* tgt,
                               const int32_t* loc, int batch, int T, int32_t* commit, int32_t* an,
                               int32_t* ks, int32_t* nt, int32_t* status, cudaStream_t stream);
cudaError_t launch_kv_relocate(void* kv, int64_t pool_slots, int32_t* r2t, int64_t stride,
                               const int32_t* rpi, const int32_t* L, const int32_t* dst,
                               int32_t* progress, int batch, int budget, int32_t* status,
                               cudaStream_t stream);
cudaError_t setup_fp8_indexer();
cudaError_t launch_fp8_indexer(const void* q, const float* w, const void* kv, int64_t nblocks,
                               const int32_t* bt, const int32_t* lens, int batch, int H, int P,
                               float* out, int32_t* status, int grid, cudaStream_t stream);

}  // namespace mlav
