// Tensor-core (tcgen05) grouped GEMMs for large batches (prefill).
#include "common.cuh"

namespace moe {

cudaError_t launch_prefill(const PrefillArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace moe
