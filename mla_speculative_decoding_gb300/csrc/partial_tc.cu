// Tensor-core (tcgen05 / TMEM) split-KV partial attention.
#include "partial_tc.cuh"

namespace mlav {

bool partial_tc_supported(const PartialArgs&) { return false; }

cudaError_t launch_partial_tc(const PartialArgs&, int, cudaStream_t) {
    return cudaErrorNotSupported;
}

cudaError_t setup_partial_tc() { return cudaSuccess; }

}  // namespace mlav
