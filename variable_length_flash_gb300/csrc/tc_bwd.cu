// Tensor-core (tcgen05 / TMEM / TMA) backward: not yet present in this build.
#include "common.cuh"
#include "kernels.h"

namespace vlf {
bool tc_backward_supported(const Params &) { return false; }
cudaError_t tc_backward(const Params &, cudaStream_t, const cudaEvent_t *) {
  return cudaErrorNotSupported;
}
size_t tc_backward_workspace(int total_q, int h_q, int d_qk) {
  return (size_t)total_q * (size_t)h_q * (size_t)d_qk * sizeof(float);
}
}  // namespace vlf
