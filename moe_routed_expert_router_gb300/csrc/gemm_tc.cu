// Tensor-core (tcgen05) grouped expert GEMMs.
#include "moe_internal.cuh"

namespace moe {

bool tc_supported(const Plan &) { return false; }
cudaError_t configure_tc(const Plan &) { return cudaSuccess; }
cudaError_t launch_ffn_tc(const Plan &, const void *, int, const ExpertPtrs &, const ExpertPtrs *, int, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace moe
