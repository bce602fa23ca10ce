// Backward entry point that allocates nothing (declared in include/vlf.h as
// vlf_attn_varlen_bwd_noalloc).
//
// The regular backward asks its caller for a device workspace (the row dot products
// D = rowsum(dO o O), fp32 [h_q, total_q]).  Some callers cannot provide one at call time: a
// plugin whose enqueue hook is not allowed to allocate, a service that reserves its whole memory
// budget up front, or code that must avoid the implicit device-wide synchronisation cudaMalloc
// and cudaFree can cause.  For them this file keeps the workspace in a fixed-size array in the
// library's own device memory, so the call needs no allocation from anyone.
//
// Costs and limits:
//   * Every GPU that loads the library holds kNoAllocScratchBytes (32 MiB) for this array until
//     the process exits.
//   * Problems whose workspace exceeds the array (h_q * total_q > 8,388,608) are refused with
//     VLF_ERR_UNSUPPORTED before anything is enqueued.
//   * The array is shared by every call on a device and keeps the last call's contents.  Nothing
//     in it has to start at zero: the backward's first kernel writes every element the later ones
//     read.  Two calls whose work overlaps on the GPU (different streams, no ordering between
//     them) race on the array and give wrong gradients; order them on one stream or with events.
//   * The first call on each device looks up the array's device address (cudaGetSymbolAddress
//     with that device current); make that first call before any stream capture begins.
//   * That address is kept for the life of the process.  It is not valid after the device is
//     reset (cudaDeviceReset): a process that resets a device must not call this entry point on
//     it afterwards.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocScratchFloats = size_t(8) << 20;  // 8,388,608 floats
constexpr size_t kNoAllocScratchBytes = kNoAllocScratchFloats * sizeof(float);

// The workspace of vlf_attn_varlen_bwd_noalloc.  In host code this name is only a host-side
// stand-in for the symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once per device.
// Returns nullptr if the lookup fails.
void *noalloc_scratch_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return nullptr;
    g_noalloc_ptr[dev] = ptr;
  }
  return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" {

size_t vlf_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int vlf_attn_varlen_bwd_noalloc(const void *q, const void *k, const void *v, const void *out,
                                const float *lse, const void *dout, const int32_t *cu_seqlens_q,
                                const int32_t *cu_seqlens_kv, int num_seqs, int total_q,
                                int total_kv, int max_seqlen_q, int max_seqlen_kv, int h_q,
                                int h_kv, int d_qk, int d_v, int dtype, float scale, int causal,
                                int window, const float *bias, int bias_heads, void *dq, void *dk,
                                void *dv, vlf_stream_t stream) {
  const size_t need =
      vlf_attn_varlen_bwd_workspace_size(total_q, total_kv, h_q, h_kv, d_qk, d_v, dtype);
  if (need > kNoAllocScratchBytes) return VLF_ERR_UNSUPPORTED;
  void *scratch = noalloc_scratch_ptr();
  if (!scratch) return VLF_ERR_LAUNCH;
  return vlf_attn_varlen_bwd_ex(q, k, v, out, lse, dout, cu_seqlens_q, cu_seqlens_kv, num_seqs,
                                total_q, total_kv, max_seqlen_q, max_seqlen_kv, h_q, h_kv, d_qk,
                                d_v, dtype, scale, causal, window, bias, bias_heads, dq, dk, dv,
                                scratch, kNoAllocScratchBytes, stream, 0u, nullptr, 0, nullptr);
}

}  // extern "C"
