// Tensor-core (tcgen05 / TMEM / TMA) forward: not yet present in this build.
#include "common.cuh"
#include "kernels.h"

namespace vlf {
bool tc_forward_supported(const Params &) { return false; }
cudaError_t tc_forward(const Params &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace vlf
