// Host-side TMA tensor-map encoding for the latent KV pool.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace mlav {

// 2-D map over kv_pool bf16 [pool_slots][576]: a box of 64 columns x 1 row,
// 128-byte swizzle, zero fill outside the tensor (for tile::gather4 loads).
// Returns false if the driver entry point is unavailable or encoding fails.
bool make_kv_gather_map(CUtensorMap* map, const void* kv_pool, int64_t pool_slots);

}  // namespace mlav
