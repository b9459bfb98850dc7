// Host-side TMA tensor-map encoding for the latent KV pool.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace mlav {

// 2-D map over kv_pool bf16 [pool_slots][576]: a box of 64 columns x 1 row,
// 128-byte swizzle, zero fill outside the tensor (for tile::gather4 loads).
// Returns false if the driver entry point is unavailable or encoding fails.
bool make_kv_gather_map(CUtensorMap* map, const void* kv_pool, int64_t pool_slots);

// 3-D map over the fp8 indexer cache kv_blocks [nblocks][8448] bytes as
// [block][64 rows][128 bytes]: a box is one block's 64 key rows (8 KB),
// 128-byte swizzle. The 256 scale bytes of each block are not covered.
bool make_fp8_block_map(CUtensorMap* map, const void* kv_blocks, int64_t nblocks);

// The same cache viewed as [block][66 rows][128 bytes]: a box is rows 64-65,
// the block's 64 fp32 scales (256 bytes), unswizzled.
bool make_fp8_scale_map(CUtensorMap* map, const void* kv_blocks, int64_t nblocks);

// 3-D map over fp8 queries [batch][num_heads][128] bytes: a box is one
// request's num_heads rows, 128-byte swizzle.
bool make_fp8_query_map(CUtensorMap* map, const void* q, int batch, int num_heads);

}  // namespace mlav
