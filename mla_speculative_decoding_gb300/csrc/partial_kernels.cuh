// Tensor-core (tcgen05 / TMEM) split-KV partial attention kernels: interface.
#pragma once

#include "common.cuh"

namespace mlav {

// Split-role pair kernel (two SMs per 128-row block): the default for
// requests of at most 128 rows.
cudaError_t launch_partial_pair(const PartialArgs& a, cudaStream_t stream);
cudaError_t setup_partial_pair();
// Partitions per query row that hold keys in the two-SM kernel's split on
// the current device for this shape, at most (a hint for the combine).
int pair_expected_parts(int batch, int T, int H, int nsplit);

// Two-pair kernel (four SMs per 256-row block, 2-SM MMAs): the default for
// requests with more than 128 rows.
cudaError_t launch_partial_quad(const PartialArgs& a, cudaStream_t stream);
cudaError_t setup_partial_quad();
// Partitions per query row the four-SM kernel's balanced plan is expected to
// fill on the current device for this shape (a hint for the combine).
int quad_expected_parts(int batch, int T, int H, int nsplit);

}  // namespace mlav
