// C ABI of libvlf.so (declared in include/vlf.h): argument checks, dispatch to the kernels,
// and the per-device error word that the kernels write instead of trapping.
#include <math.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

// One error word per device (module-scope __device__ variable; each device that loads the
// library holds its own copy).  Kernels get its address through Params::err.  The address is
// looked up once per device and kept for the life of the process; it is not valid after a
// cudaDeviceReset of that device.
__device__ int g_vlf_error_word = 0;

namespace vlf {
static std::atomic<uint64_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

cudaError_t set_smem_once(const void *kern, int bytes) {
  struct Entry {
    const void *kern;
    int dev, bytes;
  };
  // per host thread (no lock on the launch path): a thread that has not set a kernel's limit
  // itself sets it once more, which is harmless
  thread_local Entry table[256];
  thread_local int n_entries = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < n_entries; ++i)
    if (table[i].kern == kern && table[i].dev == dev) {
      if (bytes <= table[i].bytes) return cudaSuccess;
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e == cudaSuccess) table[i].bytes = bytes;
      return e;
    }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && n_entries < 256) table[n_entries++] = Entry{kern, dev, bytes};
  return e;
}
}  // namespace vlf

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int *g_err_ptr[kMaxDevices] = {nullptr};

int *error_word_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  // the last device's address, per host thread, skips the lock on repeated calls
  thread_local int t_dev = -1;
  thread_local int *t_ptr = nullptr;
  if (dev == t_dev) return t_ptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_err_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_vlf_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int *>(ptr);
  }
  t_dev = dev;
  t_ptr = g_err_ptr[dev];
  return t_ptr;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared argument checks of the forward and backward.  Returns VLF_OK or a negative status.
int check_common(const void *q, const void *k, const void *v, const int32_t *cu_q,
                 const int32_t *cu_kv, int num_seqs, int total_q, int total_kv, int max_q,
                 int max_kv, int h_q, int h_kv, int d_qk, int d_v, int dtype, const float *bias,
                 int bias_heads) {
  if (num_seqs < 0 || total_q < 0 || total_kv < 0 || max_q < 0 || max_kv < 0) return VLF_ERR_INVALID;
  if (h_q < 1 || h_kv < 1 || h_q % h_kv != 0) return VLF_ERR_INVALID;
  if (d_qk < 1 || d_v < 1) return VLF_ERR_INVALID;
  if (dtype != VLF_F16 && dtype != VLF_BF16 && dtype != VLF_F32) return VLF_ERR_INVALID;
  if (num_seqs == 0 && (total_q != 0 || total_kv != 0)) return VLF_ERR_INVALID;
  if (num_seqs > 0 && (!cu_q || !cu_kv)) return VLF_ERR_INVALID;
  if ((total_q > 0 && !q) || (total_kv > 0 && (!k || !v))) return VLF_ERR_INVALID;
  if (bias && bias_heads != 1 && bias_heads != h_q) return VLF_ERR_INVALID;
  if (d_qk > 256 || d_v > 256) return VLF_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || h_q > 65535) return VLF_ERR_UNSUPPORTED;
  // row strides of 16-bit data must keep 16-byte alignment for vector / TMA access
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(cu_q) || !aligned16(cu_kv) ||
      !aligned16(bias))
    return VLF_ERR_ALIGN;
  return VLF_OK;
}

void fill_common(vlf::Params &p, const void *q, const void *k, const void *v, const int32_t *cu_q,
                 const int32_t *cu_kv, int num_seqs, int total_q, int total_kv, int max_q,
                 int max_kv, int h_q, int h_kv, int d_qk, int d_v, int dtype, float scale,
                 int causal, int window, const float *bias, int bias_heads, unsigned flags) {
  p = vlf::Params{};
  p.q = q; p.k = k; p.v = v; p.cu_q = cu_q; p.cu_kv = cu_kv;
  p.num_seqs = num_seqs; p.total_q = total_q; p.total_kv = total_kv;
  p.max_q = max_q; p.max_kv = max_kv;
  p.h_q = h_q; p.h_kv = h_kv; p.d_qk = d_qk; p.d_v = d_v; p.group = h_q / h_kv;
  p.dtype = dtype;
  p.scale = scale > 0.f ? scale : (float)(1.0 / sqrt((double)d_qk));
  p.scale_log2 = (float)((double)p.scale * 1.4426950408889634);
  p.causal = causal ? 1 : 0;
  p.window = window > 0 ? window : 0;
  p.bias = bias; p.bias_heads = bias ? bias_heads : 0;
  p.flags = flags;
}

// The bias bands' two tables in the caller's buffer (vlf_bias_bands): rows, then blocks.
void attach_bands(vlf::Params &p, const void *bands) {
  if (!bands || !p.bias || p.total_q <= 0) return;
  p.bias_rows = static_cast<const int4 *>(bands);
  p.bias_blocks = p.bias_rows + (size_t)p.total_q * (size_t)p.bias_heads;
}

size_t workspace_bytes_for(int total_q, int h_q, int d_qk, int dtype) {
  if (total_q < 0 || h_q < 1 || d_qk < 1) return 0;
  size_t rowdot = (size_t)h_q * (size_t)total_q * sizeof(float);
  rowdot = (rowdot + 255) & ~(size_t)255;
  if (dtype == VLF_F32) return rowdot;
  return rowdot + vlf::tc_backward_workspace(total_q, h_q, d_qk);
}

// Checks shared by the split-operand latent entry points (beyond check_common on the nope
// tensors): the rope tensors, rope_heads, and the one head shape with a kernel.
int check_latent(const void *q_rope, const void *k_rope, int total_q, int total_kv, int h_kv,
                 int rope_heads, int d_nope, int d_rope, int d_v, int dtype, unsigned flags) {
  if ((total_q > 0 && !q_rope) || (total_kv > 0 && !k_rope)) return VLF_ERR_INVALID;
  if (rope_heads != 1 && rope_heads != h_kv) return VLF_ERR_INVALID;
  if (!aligned16(q_rope) || !aligned16(k_rope)) return VLF_ERR_ALIGN;
  if (d_nope != 128 || d_rope != 64 || d_v != 128) return VLF_ERR_UNSUPPORTED;
  if ((dtype != VLF_F16 && dtype != VLF_BF16) || (flags & VLF_FLAG_FORCE_SIMT)) return VLF_ERR_UNSUPPORTED;
  return VLF_OK;
}

size_t latent_rope_part_bytes(int total_kv, int h_kv, int rope_heads) {
  if (rope_heads != 1 || h_kv <= 1 || total_kv <= 0) return 0;
  return ((size_t)h_kv * (size_t)total_kv * 64 * sizeof(float) + 255) & ~(size_t)255;
}

__global__ void fill_f32_kernel(float *p, size_t n, float v) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = v;
}

// The unsplit forward: the 16-bit tensor-core kernels, the fp32 three-pass tf32 kernel, or the
// SIMT fp32-FMA kernels (forced by VLF_FLAG_FORCE_SIMT, and for shapes without a tensor-core one).
cudaError_t forward_dispatch(const vlf::Params &p, cudaStream_t cs) {
  if (!(p.flags & VLF_FLAG_FORCE_SIMT)) {
    if (vlf::tc_forward_supported(p)) return vlf::tc_forward(p, cs);
    if (vlf::tc_forward32_supported(p)) return vlf::tc_forward32(p, cs);
  }
  return vlf::simt_forward(p, cs);
}

cudaError_t zero16(void *p, size_t elems, cudaStream_t st) {
  return elems && p ? cudaMemsetAsync(p, 0, elems * 2, st) : cudaSuccess;
}

}  // namespace

extern "C" {

int vlf_version(void) { return 100; }

uint64_t vlf_launch_count(void) { return vlf::g_launches.load(std::memory_order_relaxed); }

static vlf::Params shape_params(int h_q, int h_kv, int d_qk, int d_v, int dtype, int bias_heads,
                                unsigned flags) {
  vlf::Params p{};
  p.h_q = h_q; p.h_kv = h_kv; p.d_qk = d_qk; p.d_v = d_v; p.dtype = dtype;
  p.group = h_kv > 0 ? h_q / h_kv : 0;
  p.bias_heads = bias_heads;
  p.flags = flags;
  return p;
}

int vlf_fwd_path(int h_q, int h_kv, int d_qk, int d_v, int dtype, int bias_heads, unsigned flags) {
  if (h_q < 1 || h_kv < 1 || h_q % h_kv || d_qk < 1 || d_v < 1 || dtype < 0 || dtype > 2)
    return VLF_ERR_INVALID;
  if (d_qk > 256 || d_v > 256) return VLF_ERR_UNSUPPORTED;
  vlf::Params p = shape_params(h_q, h_kv, d_qk, d_v, dtype, bias_heads, flags);
  return (!(flags & VLF_FLAG_FORCE_SIMT) &&
          (vlf::tc_forward_supported(p) || vlf::tc_forward32_supported(p))) ? 1 : 0;
}

int vlf_bwd_path(int h_q, int h_kv, int d_qk, int d_v, int dtype, int bias_heads, unsigned flags) {
  if (h_q < 1 || h_kv < 1 || h_q % h_kv || d_qk < 1 || d_v < 1 || dtype < 0 || dtype > 2)
    return VLF_ERR_INVALID;
  if (d_qk > 256 || d_v > 256) return VLF_ERR_UNSUPPORTED;
  vlf::Params p = shape_params(h_q, h_kv, d_qk, d_v, dtype, bias_heads, flags);
  return (!(flags & VLF_FLAG_FORCE_SIMT) &&
          (vlf::tc_backward_supported(p) || vlf::tc_backward32_supported(p))) ? 1 : 0;
}

const char *vlf_status_string(int status) {
  switch (status) {
    case VLF_OK: return "ok";
    case VLF_ERR_INVALID: return "invalid argument";
    case VLF_ERR_UNSUPPORTED: return "unsupported problem (dtype / head width / size)";
    case VLF_ERR_ALIGN: return "pointer not 16-byte aligned";
    case VLF_ERR_LAUNCH: return "CUDA launch or runtime error";
    case VLF_ERR_TIMEOUT: return "device pipeline wait timed out";
    case VLF_ERR_BAD_SEQLENS: return "bad cu_seqlens (out of range, decreasing, or longer than max_seqlen)";
    case VLF_ERR_WORKSPACE: return "backward workspace missing or too small";
    default: return "unknown status";
  }
}

int vlf_sched_kv_band(int r0, int r1, int q_len, int kv_len, int causal, int window, int *lo,
                      int *hi) {
  if (!lo || !hi || q_len < 0 || kv_len < 0 || r0 < 0 || r1 <= r0 || r1 > q_len) return VLF_ERR_INVALID;
  vlf::kv_band(r0, r1, q_len, kv_len, causal, window, *lo, *hi);
  return VLF_OK;
}

int vlf_sched_q_band(int j0, int j1, int q_len, int kv_len, int causal, int window, int *lo,
                     int *hi) {
  if (!lo || !hi || q_len < 0 || kv_len < 0 || j0 < 0 || j1 <= j0 || j1 > kv_len) return VLF_ERR_INVALID;
  vlf::q_band(j0, j1, q_len, kv_len, causal, window, *lo, *hi);
  return VLF_OK;
}

int vlf_attn_varlen_fwd_ex(const void *q, const void *k, const void *v,
                           const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_kv, int num_seqs,
                           int total_q, int total_kv, int max_seqlen_q, int max_seqlen_kv,
                           int h_q, int h_kv, int d_qk, int d_v, int dtype, float scale,
                           int causal, int window, const float *bias, int bias_heads, void *out,
                           float *lse, vlf_stream_t stream, unsigned flags,
                           const void *bias_bands) {
  int st = check_common(q, k, v, cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q, total_kv,
                        max_seqlen_q, max_seqlen_kv, h_q, h_kv, d_qk, d_v, dtype, bias, bias_heads);
  if (st != VLF_OK) return st;
  if (total_q > 0 && !out) return VLF_ERR_INVALID;
  if (!aligned16(out) || !aligned16(lse)) return VLF_ERR_ALIGN;
  if (num_seqs == 0 || max_seqlen_q == 0) return VLF_OK;
  vlf::Params p;
  fill_common(p, q, k, v, cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q, total_kv, max_seqlen_q,
              max_seqlen_kv, h_q, h_kv, d_qk, d_v, dtype, scale, causal, window, bias, bias_heads,
              flags);
  p.out = out;
  p.lse = lse;
  if (!aligned16(bias_bands)) return VLF_ERR_ALIGN;
  attach_bands(p, bias_bands);
  p.err = error_word_ptr();
  if (!p.err) return VLF_ERR_LAUNCH;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = forward_dispatch(p, cs);
  return e == cudaSuccess ? VLF_OK : VLF_ERR_LAUNCH;
}

int vlf_attn_varlen_fwd(const void *q, const void *k, const void *v, const int32_t *cu_seqlens_q,
                        const int32_t *cu_seqlens_kv, int num_seqs, int total_q, int total_kv,
                        int max_seqlen_q, int max_seqlen_kv, int h_q, int h_kv, int d_qk, int d_v,
                        int dtype, float scale, int causal, int window, const float *bias,
                        int bias_heads, void *out, float *lse, vlf_stream_t stream) {
  return vlf_attn_varlen_fwd_ex(q, k, v, cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q, total_kv,
                                max_seqlen_q, max_seqlen_kv, h_q, h_kv, d_qk, d_v, dtype, scale,
                                causal, window, bias, bias_heads, out, lse, stream, 0u, nullptr);
}

int vlf_fwd_num_splits(int num_seqs, int max_seqlen_q, int max_seqlen_kv, int h_q, int h_kv,
                       int d_qk, int d_v, int dtype, unsigned flags, int num_sms) {
  if (num_sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 1;
  }
  return vlf::fwd_num_splits(num_seqs, max_seqlen_q, max_seqlen_kv, h_q, h_kv, d_qk, d_v, dtype,
                             flags, num_sms);
}

size_t vlf_attn_varlen_fwd_split_workspace_size(int total_q, int h_q, int d_v, int num_splits) {
  if (total_q < 0 || h_q < 1 || d_v < 1 || num_splits < 2) return 0;
  const size_t rows = (size_t)num_splits * (size_t)total_q * (size_t)h_q;
  const size_t o = (rows * (size_t)d_v * sizeof(float) + 255) & ~(size_t)255;
  return o + ((rows * sizeof(float) + 255) & ~(size_t)255);
}

int vlf_attn_varlen_fwd_split(const void *q, const void *k, const void *v,
                              const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_kv,
                              int num_seqs, int total_q, int total_kv, int max_seqlen_q,
                              int max_seqlen_kv, int h_q, int h_kv, int d_qk, int d_v, int dtype,
                              float scale, int causal, int window, const float *bias,
                              int bias_heads, void *out, float *lse, int num_splits,
                              void *workspace, size_t workspace_bytes, vlf_stream_t stream,
                              unsigned flags, const void *bias_bands) {
  int st = check_common(q, k, v, cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q, total_kv,
                        max_seqlen_q, max_seqlen_kv, h_q, h_kv, d_qk, d_v, dtype, bias, bias_heads);
  if (st != VLF_OK) return st;
  if (num_splits < 0) return VLF_ERR_INVALID;
  if (total_q > 0 && !out) return VLF_ERR_INVALID;
  if (!aligned16(out) || !aligned16(lse) || !aligned16(workspace) || !aligned16(bias_bands))
    return VLF_ERR_ALIGN;
  if (num_seqs == 0 || max_seqlen_q == 0) return VLF_OK;
  vlf::Params p;
  fill_common(p, q, k, v, cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q, total_kv, max_seqlen_q,
              max_seqlen_kv, h_q, h_kv, d_qk, d_v, dtype, scale, causal, window, bias, bias_heads,
              flags);
  p.out = out;
  p.lse = lse;
  attach_bands(p, bias_bands);
  p.err = error_word_ptr();
  if (!p.err) return VLF_ERR_LAUNCH;
  if (num_splits == 0)
    num_splits = vlf_fwd_num_splits(num_seqs, max_seqlen_q, max_seqlen_kv, h_q, h_kv, d_qk, d_v,
                                    dtype, flags, 0);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (num_splits >= 2 && !(flags & VLF_FLAG_FORCE_SIMT) && vlf::tc_forward_splittable(p)) {
    if (num_splits > 64 || (long long)num_splits * num_seqs > 65535) return VLF_ERR_UNSUPPORTED;
    const size_t need = vlf_attn_varlen_fwd_split_workspace_size(total_q, h_q, d_v, num_splits);
    if (!workspace || workspace_bytes < need) return VLF_ERR_WORKSPACE;
    const size_t rows = (size_t)num_splits * (size_t)total_q * (size_t)h_q;
    p.kv_splits = num_splits;
    p.o_part = static_cast<float *>(workspace);
    p.lse_part = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                           ((rows * (size_t)d_v * sizeof(float) + 255) & ~(size_t)255));
    e = vlf::tc_forward_split(p, cs);
  } else {
    e = forward_dispatch(p, cs);
  }
  return e == cudaSuccess ? VLF_OK : VLF_ERR_LAUNCH;
}

size_t vlf_attn_varlen_bwd_workspace_size(int total_q, int total_kv, int h_q, int h_kv, int d_qk,
                                          int d_v, int dtype) {
  (void)total_kv; (void)h_kv; (void)d_v;
  return workspace_bytes_for(total_q, h_q, d_qk, dtype);
}

int vlf_attn_varlen_bwd_ex(const void *q, const void *k, const void *v, const void *out,
                           const float *lse, const void *dout, const int32_t *cu_seqlens_q,
                           const int32_t *cu_seqlens_kv, int num_seqs, int total_q, int total_kv,
                           int max_seqlen_q, int max_seqlen_kv, int h_q, int h_kv, int d_qk,
                           int d_v, int dtype, float scale, int causal, int window,
                           const float *bias, int bias_heads, void *dq, void *dk, void *dv,
                           void *workspace, size_t workspace_bytes, vlf_stream_t stream,
                           unsigned flags, void *const *stage_events, int n_stage_events,
                           const void *bias_bands) {
  if (stage_events && n_stage_events < VLF_BWD_STAGES + 1) return VLF_ERR_INVALID;
  int st = check_common(q, k, v, cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q, total_kv,
                        max_seqlen_q, max_seqlen_kv, h_q, h_kv, d_qk, d_v, dtype, bias, bias_heads);
  if (st != VLF_OK) return st;
  if (total_q > 0 && (!out || !lse || !dout || !dq)) return VLF_ERR_INVALID;
  if (total_kv > 0 && (!dk || !dv)) return VLF_ERR_INVALID;
  if (!aligned16(out) || !aligned16(lse) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) ||
      !aligned16(dv) || !aligned16(workspace) || !aligned16(bias_bands))
    return VLF_ERR_ALIGN;
  const size_t need = workspace_bytes_for(total_q, h_q, d_qk, dtype);
  if (need > 0 && (!workspace || workspace_bytes < need)) return VLF_ERR_WORKSPACE;
  if (num_seqs == 0) return VLF_OK;
  vlf::Params p;
  fill_common(p, q, k, v, cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q, total_kv, max_seqlen_q,
              max_seqlen_kv, h_q, h_kv, d_qk, d_v, dtype, scale, causal, window, bias, bias_heads,
              flags);
  const cudaEvent_t *ev = reinterpret_cast<const cudaEvent_t *>(stage_events);
  p.out = const_cast<void *>(out);
  p.lse = const_cast<float *>(lse);
  p.dout = dout;
  p.dq = dq; p.dk = dk; p.dv = dv;
  p.rowdot = static_cast<float *>(workspace);
  p.dq_acc = nullptr;
  attach_bands(p, bias_bands);
  p.err = error_word_ptr();
  if (!p.err) return VLF_ERR_LAUNCH;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (!(flags & VLF_FLAG_FORCE_SIMT) && vlf::tc_backward_supported(p))
    e = vlf::tc_backward(p, cs, ev);
  else if (!(flags & VLF_FLAG_FORCE_SIMT) && vlf::tc_backward32_supported(p))
    e = vlf::tc_backward32(p, cs, ev);
  else
    e = vlf::simt_backward(p, cs, ev);
  return e == cudaSuccess ? VLF_OK : VLF_ERR_LAUNCH;
}

int vlf_attn_varlen_bwd(const void *q, const void *k, const void *v, const void *out,
                        const float *lse, const void *dout, const int32_t *cu_seqlens_q,
                        const int32_t *cu_seqlens_kv, int num_seqs, int total_q, int total_kv,
                        int max_seqlen_q, int max_seqlen_kv, int h_q, int h_kv, int d_qk, int d_v,
                        int dtype, float scale, int causal, int window, const float *bias,
                        int bias_heads, void *dq, void *dk, void *dv, void *workspace,
                        size_t workspace_bytes, vlf_stream_t stream) {
  return vlf_attn_varlen_bwd_ex(q, k, v, out, lse, dout, cu_seqlens_q, cu_seqlens_kv, num_seqs,
                                total_q, total_kv, max_seqlen_q, max_seqlen_kv, h_q, h_kv, d_qk,
                                d_v, dtype, scale, causal, window, bias, bias_heads, dq, dk, dv,
                                workspace, workspace_bytes, stream, 0u, nullptr, 0, nullptr);
}

int vlf_attn_varlen_fwd_latent(const void *q_nope, const void *q_rope, const void *k_nope,
                               const void *k_rope, const void *v, const int32_t *cu_seqlens_q,
                               const int32_t *cu_seqlens_kv, int num_seqs, int total_q,
                               int total_kv, int max_seqlen_q, int max_seqlen_kv, int h_q,
                               int h_kv, int rope_heads, int d_nope, int d_rope, int d_v,
                               int dtype, float scale, int causal, int window, const float *bias,
                               int bias_heads, void *out, float *lse, vlf_stream_t stream,
                               unsigned flags) {
  int st = check_common(q_nope, k_nope, v, cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q,
                        total_kv, max_seqlen_q, max_seqlen_kv, h_q, h_kv, d_nope + d_rope, d_v,
                        dtype, bias, bias_heads);
  if (st != VLF_OK) return st;
  st = check_latent(q_rope, k_rope, total_q, total_kv, h_kv, rope_heads, d_nope, d_rope, d_v, dtype, flags);
  if (st != VLF_OK) return st;
  if (total_q > 0 && !out) return VLF_ERR_INVALID;
  if (!aligned16(out) || !aligned16(lse)) return VLF_ERR_ALIGN;
  if (num_seqs == 0 || max_seqlen_q == 0 || total_q == 0) return VLF_OK;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (total_kv == 0) {  // no keys anywhere: O = 0, LSE = -inf
    e = zero16(out, (size_t)total_q * h_q * d_v, cs);
    if (e == cudaSuccess && lse) {
      const size_t n = (size_t)total_q * h_q;
      fill_f32_kernel<<<(unsigned)((n + 255) / 256), 256, 0, cs>>>(lse, n, -INFINITY);
      e = cudaGetLastError();
      if (e == cudaSuccess) vlf::count_launch();
    }
    return e == cudaSuccess ? VLF_OK : VLF_ERR_LAUNCH;
  }
  vlf::Params p;
  fill_common(p, q_nope, k_nope, v, cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q, total_kv,
              max_seqlen_q, max_seqlen_kv, h_q, h_kv, d_nope + d_rope, d_v, dtype, scale, causal,
              window, bias, bias_heads, flags);
  p.latent = 1;
  p.q_rope = q_rope;
  p.k_rope = k_rope;
  p.rope_heads = rope_heads;
  p.out = out;
  p.lse = lse;
  p.err = error_word_ptr();
  if (!p.err) return VLF_ERR_LAUNCH;
  e = vlf::tc_forward(p, cs);
  return e == cudaSuccess ? VLF_OK : VLF_ERR_LAUNCH;
}

size_t vlf_attn_varlen_bwd_latent_workspace_size(int total_q, int total_kv, int h_q, int h_kv,
                                                 int rope_heads, int dtype) {
  if (total_q < 0 || total_kv < 0 || h_q < 1 || h_kv < 1) return 0;
  return workspace_bytes_for(total_q, h_q, 192, dtype) +
         latent_rope_part_bytes(total_kv, h_kv, rope_heads);
}

int vlf_attn_varlen_bwd_latent(const void *q_nope, const void *q_rope, const void *k_nope,
                               const void *k_rope, const void *v, const void *out,
                               const float *lse, const void *dout, const int32_t *cu_seqlens_q,
                               const int32_t *cu_seqlens_kv, int num_seqs, int total_q,
                               int total_kv, int max_seqlen_q, int max_seqlen_kv, int h_q,
                               int h_kv, int rope_heads, int d_nope, int d_rope, int d_v,
                               int dtype, float scale, int causal, int window, const float *bias,
                               int bias_heads, void *dq_nope, void *dq_rope, void *dk_nope,
                               void *dk_rope, void *dv, void *workspace, size_t workspace_bytes,
                               vlf_stream_t stream, unsigned flags, void *const *stage_events,
                               int n_stage_events) {
  if (stage_events && n_stage_events < VLF_BWD_STAGES + 1) return VLF_ERR_INVALID;
  int st = check_common(q_nope, k_nope, v, cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q,
                        total_kv, max_seqlen_q, max_seqlen_kv, h_q, h_kv, d_nope + d_rope, d_v,
                        dtype, bias, bias_heads);
  if (st != VLF_OK) return st;
  st = check_latent(q_rope, k_rope, total_q, total_kv, h_kv, rope_heads, d_nope, d_rope, d_v, dtype, flags);
  if (st != VLF_OK) return st;
  if (total_q > 0 && (!out || !lse || !dout || !dq_nope || !dq_rope)) return VLF_ERR_INVALID;
  if (total_kv > 0 && (!dk_nope || !dk_rope || !dv)) return VLF_ERR_INVALID;
  if (!aligned16(out) || !aligned16(lse) || !aligned16(dout) || !aligned16(dq_nope) ||
      !aligned16(dq_rope) || !aligned16(dk_nope) || !aligned16(dk_rope) || !aligned16(dv) ||
      !aligned16(workspace))
    return VLF_ERR_ALIGN;
  const size_t rowdot_bytes = workspace_bytes_for(total_q, h_q, 192, dtype);
  const size_t need = rowdot_bytes + latent_rope_part_bytes(total_kv, h_kv, rope_heads);
  if (need > 0 && (!workspace || workspace_bytes < need)) return VLF_ERR_WORKSPACE;
  if (num_seqs == 0) return VLF_OK;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (total_q == 0 || total_kv == 0) {  // nothing attends: every gradient is zero
    cudaError_t e = zero16(dq_nope, (size_t)total_q * h_q * d_nope, cs);
    if (e == cudaSuccess) e = zero16(dq_rope, (size_t)total_q * h_q * d_rope, cs);
    if (e == cudaSuccess) e = zero16(dk_nope, (size_t)total_kv * h_kv * d_nope, cs);
    if (e == cudaSuccess) e = zero16(dk_rope, (size_t)total_kv * rope_heads * d_rope, cs);
    if (e == cudaSuccess) e = zero16(dv, (size_t)total_kv * h_kv * d_v, cs);
    return e == cudaSuccess ? VLF_OK : VLF_ERR_LAUNCH;
  }
  vlf::Params p;
  fill_common(p, q_nope, k_nope, v, cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q, total_kv,
              max_seqlen_q, max_seqlen_kv, h_q, h_kv, d_nope + d_rope, d_v, dtype, scale, causal,
              window, bias, bias_heads, flags);
  p.latent = 1;
  p.q_rope = q_rope;
  p.k_rope = k_rope;
  p.rope_heads = rope_heads;
  p.out = const_cast<void *>(out);
  p.lse = const_cast<float *>(lse);
  p.dout = dout;
  p.dq = dq_nope; p.dk = dk_nope; p.dv = dv;
  p.dq_rope = dq_rope; p.dk_rope = dk_rope;
  p.rowdot = static_cast<float *>(workspace);
  if (latent_rope_part_bytes(total_kv, h_kv, rope_heads) > 0)
    p.dk_rope_part = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + rowdot_bytes);
  p.err = error_word_ptr();
  if (!p.err) return VLF_ERR_LAUNCH;
  cudaError_t e = vlf::tc_backward(p, cs, reinterpret_cast<const cudaEvent_t *>(stage_events));
  return e == cudaSuccess ? VLF_OK : VLF_ERR_LAUNCH;
}

size_t vlf_bias_bands_size(int total_q, int bias_heads) {
  return vlf::bias_bands_bytes(total_q, bias_heads);
}

int vlf_bias_bands(const float *bias, int bias_heads, const int32_t *cu_seqlens_q,
                   const int32_t *cu_seqlens_kv, int num_seqs, int total_q, int max_seqlen_kv,
                   void *bands, size_t bands_bytes, vlf_stream_t stream) {
  if (num_seqs < 0 || total_q < 0 || max_seqlen_kv < 0 || bias_heads < 1) return VLF_ERR_INVALID;
  if (num_seqs > 65535) return VLF_ERR_UNSUPPORTED;
  if (total_q == 0) return VLF_OK;
  if (!bias || num_seqs == 0 || !cu_seqlens_q || !cu_seqlens_kv) return VLF_ERR_INVALID;
  if (!aligned16(bias) || !aligned16(bands) || !aligned16(cu_seqlens_q) || !aligned16(cu_seqlens_kv))
    return VLF_ERR_ALIGN;
  if (!bands || bands_bytes < vlf::bias_bands_bytes(total_q, bias_heads)) return VLF_ERR_WORKSPACE;
  vlf::Params p{};
  p.bias = bias;
  p.bias_heads = bias_heads;
  p.cu_q = cu_seqlens_q;
  p.cu_kv = cu_seqlens_kv;
  p.num_seqs = num_seqs;
  p.total_q = total_q;
  p.max_kv = max_seqlen_kv;
  const cudaError_t e = vlf::bias_bands(p, bands, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? VLF_OK : VLF_ERR_LAUNCH;
}

int vlf_check_error(vlf_stream_t stream) {
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(cs) != cudaSuccess) return VLF_ERR_LAUNCH;
  int *ptr = error_word_ptr();
  if (!ptr) return VLF_ERR_LAUNCH;
  int word = 0;
  if (cudaMemcpy(&word, ptr, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return VLF_ERR_LAUNCH;
  if (word != 0) {
    const int zero = 0;
    if (cudaMemcpy(ptr, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return VLF_ERR_LAUNCH;
  }
  if (cudaGetLastError() != cudaSuccess) return VLF_ERR_LAUNCH;
  return word;
}

}  // extern "C"
