// Host-side entry points of the kernel translation units (internal to libvlf.so).
#pragma once

#include <cuda_runtime.h>

namespace vlf {

struct Params;

// SIMT fp32-FMA kernels (simt.cu): every dtype and head width up to 256.
cudaError_t simt_forward(const Params &p, cudaStream_t st);
// Backward pre-pass: rowdot[h, row] = sum_c dO[row, h, c] * O[row, h, c] (simt.cu).
cudaError_t rowdot_forward(const Params &p, cudaStream_t st);
// ev: NULL or VLF_BWD_STAGES + 1 events recorded before the first and after each stage.
cudaError_t simt_backward(const Params &p, cudaStream_t st, const cudaEvent_t *ev);

// Tensor-core kernels (tc_fwd.cu / tc_bwd.cu).  `supported` says whether the shape has one.
bool tc_forward_supported(const Params &p);
cudaError_t tc_forward(const Params &p, cudaStream_t st);
// Split-KV forward (p.kv_splits > 1, p.o_part / p.lse_part set): the parts, then their combine.
// Only shapes with one query tile per CTA split (tc_forward_splittable).
bool tc_forward_splittable(const Params &p);
cudaError_t tc_forward_split(const Params &p, cudaStream_t st);
// The number of parts the library would cut each CTA's KV band into (1: no split), from the
// problem's launch shape and the device's SM count.
int fwd_num_splits(int num_seqs, int max_q, int max_kv, int h_q, int h_kv, int d_qk, int d_v,
                   int dtype, unsigned flags, int num_sms);
// fp32 inputs on the tensor cores, products in three tf32 passes (tc_fwd32.cu): head widths 32
// and 64.
bool tc_forward32_supported(const Params &p);
cudaError_t tc_forward32(const Params &p, cudaStream_t st);
bool tc_backward_supported(const Params &p);
// fp32 backward on the tensor cores, three tf32 passes (tc_bwd32.cu): head widths 32 and 64.
bool tc_backward32_supported(const Params &p);
cudaError_t tc_backward32(const Params &p, cudaStream_t st, const cudaEvent_t *ev);
cudaError_t tc_backward(const Params &p, cudaStream_t st, const cudaEvent_t *ev);
size_t tc_backward_workspace(int total_q, int h_q, int d_qk);

// Bias bands (bias_bands.cu): the buffer size, and the pass that fills it from p.bias.
size_t bias_bands_bytes(int total_q, int bias_heads);
cudaError_t bias_bands(const Params &p, void *bands, cudaStream_t st);

// Host-side count of successful kernel launches (api.cu).
void count_launch(int n = 1);
// cudaFuncSetAttribute(kern, MaxDynamicSharedMemorySize, bytes), made once per (kernel, device)
// and raised only when a launch needs more: the runtime call costs microseconds of host time,
// which small problems would pay on every launch.
cudaError_t set_smem_once(const void *kern, int bytes);

// Records ev[i] on st when ev is not NULL.
inline cudaError_t mark(const cudaEvent_t *ev, int i, cudaStream_t st) {
  return ev ? cudaEventRecord(ev[i], st) : cudaSuccess;
}

}  // namespace vlf
