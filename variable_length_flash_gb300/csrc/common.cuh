// Internal definitions shared by the kernels of libvlf.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/vlf.h"

namespace vlf {

// Everything a kernel needs, passed by value (kernel parameter space).
struct Params {
  const void *q, *k, *v;
  const int32_t *cu_q, *cu_kv;
  int num_seqs, total_q, total_kv, max_q, max_kv;
  int h_q, h_kv, d_qk, d_v, group;  // group = h_q / h_kv
  int dtype;
  float scale;       // softmax scale (natural-log domain)
  float scale_log2;  // scale * log2(e)
  int causal, window;
  const float *bias;
  int bias_heads;
  void *out;
  float *lse;  // [h_q, total_q]
  // backward
  const void *dout;
  void *dq, *dk, *dv;
  float *rowdot;  // [h_q, total_q]  D_i = sum_c dO_ic O_ic
  float *dq_acc;  // [total_q, h_q, d_qk] fp32 (tensor-core backward)
  int *err;       // per-device error word
  unsigned flags;
  // set by a launcher: grid x enumerates heads (y the row blocks), so that the CTAs reading the
  // same tiles of a head-broadcast bias run together and share them through L2
  int heads_fast = 0;
  // split-KV forward: kv_splits > 1 cuts each CTA's KV band into kv_splits contiguous parts
  // (grid z = sequence * kv_splits + part); each part writes its normalised fp32 result and its
  // log-sum-exp, which a combine kernel merges into out / lse
  int kv_splits = 1;
  float *o_part = nullptr;    // [kv_splits, total_q, h_q, d_v]
  float *lse_part = nullptr;  // [kv_splits, h_q, total_q]
  // latent head with split operands (QK width 192 = 128 "nope" + 64 "rope", V width 128): q and
  // k point to q_nope [total_q, h_q, 128] and k_nope [total_kv, h_kv, 128]; the last 64 columns
  // of each Q / K tile come from q_rope [total_q, h_q, 64] and k_rope [total_kv, rope_heads, 64]
  // (rope_heads 1: one rope key shared by every head).  The backward writes dq / dk as their
  // nope parts and dq_rope / dk_rope; a shared rope key's gradient goes per kv head to
  // dk_rope_part [h_kv, total_kv, 64] fp32 and is summed over heads afterwards.
  int latent = 0;
  const void *q_rope = nullptr, *k_rope = nullptr;
  int rope_heads = 0;
  void *dq_rope = nullptr, *dk_rope = nullptr;
  float *dk_rope_part = nullptr;
  // bias bands (bias_bands.cu), nullptr when not computed: bias_rows[hb * total_q + r] =
  // {lo, hi, pure, 0}, the keys [lo, hi) from the first to the last finite bias value of global
  // query row r and bias head hb, pure = the bias is exactly 0 throughout them (it is then that
  // interval mask alone); bias_blocks[hb * total_q + q0 + 64 b] = {lo, hi, ilo, ihi} for the
  // 64-row block b of the sequence starting at row q0: the union of the rows' intervals and, when
  // all are pure, their intersection (else ilo = ihi = -1).
  const int4 *bias_rows = nullptr, *bias_blocks = nullptr;
};

// ---------------------------------------------------------------- element access
template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// ---------------------------------------------------------------- errors
__device__ __forceinline__ void set_error(int *err, int code) {
  if (err) atomicCAS(err, 0, code);  // keep the first error
}

// ---------------------------------------------------------------- sequences
struct Seq {
  int q0, q_len, k0, kv_len;
};

// Reads and validates sequence s; on bad cu_seqlens records VLF_ERR_BAD_SEQLENS and returns false.
// (seq_from: the same from the four values cu_q[s], cu_q[s+1], cu_kv[s], cu_kv[s+1] already
// loaded, so that a kernel can issue the loads first and overlap their latency with its setup)
__device__ __forceinline__ bool seq_from(const Params &p, int a, int b, int c, int d, Seq &sq) {
  bool ok = (a >= 0) && (a <= b) && (b <= p.total_q) && (c >= 0) && (c <= d) &&
            (d <= p.total_kv) && (b - a <= p.max_q) && (d - c <= p.max_kv);
  if (!ok) {
    set_error(p.err, VLF_ERR_BAD_SEQLENS);
    return false;
  }
  sq.q0 = a;
  sq.q_len = b - a;
  sq.k0 = c;
  sq.kv_len = d - c;
  return true;
}

__device__ __forceinline__ bool load_seq(const Params &p, int s, Seq &sq) {
  return seq_from(p, __ldg(p.cu_q + s), __ldg(p.cu_q + s + 1), __ldg(p.cu_kv + s),
                  __ldg(p.cu_kv + s + 1), sq);
}

// ---------------------------------------------------------------- tile scheduler (band math)
// Diagonal of sequence-local row i is i + (kv_len - q_len) (end-aligned causal).
// Keys [lo, hi) that rows [r0, r1) may see: causal caps at the last row's diagonal, the window
// starts at the first row's band start.  Empty range -> lo == hi.
__host__ __device__ __forceinline__ void kv_band(int r0, int r1, int q_len, int kv_len,
                                                 int causal, int window, int &lo, int &hi) {
  const int off = kv_len - q_len;
  lo = 0;
  hi = kv_len;
  if (causal) {
    long long h = (long long)(r1 - 1) + off + 1;
    hi = h < 0 ? 0 : (h > kv_len ? kv_len : (int)h);
  }
  if (window > 0) {
    long long l = (long long)r0 + off - window + 1;
    lo = l < 0 ? 0 : (l > kv_len ? kv_len : (int)l);
  }
  if (hi < lo) hi = lo;
}

// Rows [lo, hi) that may see any key of [j0, j1).
__host__ __device__ __forceinline__ void q_band(int j0, int j1, int q_len, int kv_len, int causal,
                                                int window, int &lo, int &hi) {
  const int off = kv_len - q_len;
  lo = 0;
  hi = q_len;
  if (causal) {
    long long l = (long long)j0 - off;
    lo = l < 0 ? 0 : (l > q_len ? q_len : (int)l);
  }
  if (window > 0) {
    long long h = (long long)j1 - off + window - 1;
    hi = h < 0 ? 0 : (h > q_len ? q_len : (int)h);
  }
  if (hi < lo) hi = lo;
}

// Per-pair visibility (the per-element mask of a partially covered tile).
__device__ __forceinline__ bool pair_visible(int i, int j, int off, int kv_len, int causal,
                                             int window) {
  if (j < 0 || j >= kv_len) return false;
  const int diag = i + off;
  if (causal && j > diag) return false;
  if (window > 0 && j < diag - window + 1) return false;
  return true;
}

// The keys pair_visible accepts for row i form one interval: pair_visible(i, j, ...) holds
// exactly when lo <= j < hi (hi <= lo: the row sees nothing).
__device__ __forceinline__ void visible_range(int i, int off, int kv_len, int causal, int window,
                                              int &lo, int &hi) {
  const long long diag = (long long)i + off;
  lo = window > 0 ? (int)max(0ll, min((long long)kv_len, diag - window + 1)) : 0;
  hi = causal ? (int)max(0ll, min((long long)kv_len, diag + 1)) : kv_len;
}
// The same for a key j: the query rows i with pair_visible(i, j, ...) are exactly lo <= i < hi
// (for 0 <= j < kv_len).
__device__ __forceinline__ void visible_rows(int j, int off, int q_len, int causal, int window,
                                             int &lo, int &hi) {
  const long long first = (long long)j - off;  // the first row whose diagonal reaches j
  lo = causal ? (int)max(0ll, min((long long)q_len, first)) : 0;
  hi = window > 0 ? (int)max(0ll, min((long long)q_len, first + window)) : q_len;
}

// Bias element (row = global query row, column = sequence-local key), 64-bit offsets.
__device__ __forceinline__ float bias_at(const Params &p, int grow, int h, int j) {
  const int bh = p.bias_heads == 1 ? 0 : h;
  const size_t off = ((size_t)grow * (size_t)p.bias_heads + (size_t)bh) * (size_t)p.max_kv + (size_t)j;
  return __ldg(p.bias + off);
}

}  // namespace vlf
