// Host-side TMA tensor-map encoding (driver entry point fetched through the
// runtime, so the library does not link libcuda directly).
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tmap.cuh"

namespace mlav {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

void load_entry() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

}  // namespace

bool make_kv_gather_map(CUtensorMap* map, const void* kv_pool, int64_t pool_slots) {
    std::call_once(g_once, load_entry);
    if (g_encode == nullptr || pool_slots < 1 || pool_slots > 0x7fffffffLL) return false;
    const cuuint64_t dims[2] = {576, (cuuint64_t)pool_slots};
    const cuuint64_t strides[1] = {576 * 2};
    const cuuint32_t box[2] = {64, 1};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(kv_pool),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_fp8_block_map(CUtensorMap* map, const void* kv_blocks, int64_t nblocks) {
    std::call_once(g_once, load_entry);
    if (g_encode == nullptr || nblocks > 0x7fffffffLL) return false;
    // [nblocks][8448] bytes viewed as [nblocks][64 rows][128 bytes] (the
    // scales after each block's 64 rows are skipped by the stride).
    const cuuint64_t dims[3] = {128, 64, (cuuint64_t)(nblocks > 0 ? nblocks : 1)};
    const cuuint64_t strides[2] = {128, 8448};
    const cuuint32_t box[3] = {128, 64, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(kv_blocks),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_fp8_scale_map(CUtensorMap* map, const void* kv_blocks, int64_t nblocks) {
    std::call_once(g_once, load_entry);
    if (g_encode == nullptr || nblocks > 0x7fffffffLL) return false;
    // The same blocks viewed as [block][66 rows][128 bytes]: rows 64-65 hold
    // the 64 fp32 scales; a box is those two rows, unswizzled (256 bytes).
    const cuuint64_t dims[3] = {128, 66, (cuuint64_t)(nblocks > 0 ? nblocks : 1)};
    const cuuint64_t strides[2] = {128, 8448};
    const cuuint32_t box[3] = {128, 2, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(kv_blocks),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_fp8_query_map(CUtensorMap* map, const void* q, int batch, int num_heads) {
    std::call_once(g_once, load_entry);
    if (g_encode == nullptr || batch < 1 || num_heads < 1 || num_heads > 256) return false;
    const cuuint64_t dims[3] = {128, (cuuint64_t)num_heads, (cuuint64_t)batch};
    const cuuint64_t strides[2] = {128, (cuuint64_t)num_heads * 128};
    const cuuint32_t box[3] = {128, (cuuint32_t)num_heads, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(q), dims,
                                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace mlav
