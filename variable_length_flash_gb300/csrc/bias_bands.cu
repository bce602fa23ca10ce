// Bias bands: which keys of each query row an additive bias leaves visible.
//
// The additive bias of mtlattn 0.3.0 ("Use": attn_bias [total_q, H or 1, max_kv], -inf masks a
// pair; a boolean mask becomes 0 / -inf) often masks whole stretches of a row -- a prefix-LM
// mask hides every key past the prefix and the diagonal.  This pass records, per (bias head,
// query row), the keys from the first to the last finite bias value and whether every value in
// between is exactly 0 (the bias is then the interval mask alone).  The attention kernels use
// it to skip KV tiles that a CTA's rows cannot see (exact: those pairs contribute zero), and,
// where all of a CTA's rows are pure intervals, to mask by interval without reading the bias.
//
// Layout of the caller's buffer (vlf_bias_bands_size bytes): two int4 tables of
// [bias_heads][total_q] entries {lo, hi, pure, 0}:
//   rows   entry (hb, r): keys [lo, hi) of global query row r (lo = hi = 0 when no key is finite)
//   blocks entry (hb, q0 + 64 b) for each sequence (first row q0) and block b of 64 of its rows:
//          the union of those rows' intervals and the AND of their pure flags (other entries
//          unused).
#include "common.cuh"
#include "kernels.h"

namespace vlf {
namespace {

// The sequence that global query row r belongs to (cu_q[s] <= r < cu_q[s + 1]); -1 if none.
__device__ __forceinline__ int seq_of_row(const Params &p, int r) {
  int a = 0, b = p.num_seqs;  // invariant: cu_q[a] <= r < cu_q[b] when r is in range
  if (r < __ldg(p.cu_q) || r >= __ldg(p.cu_q + b)) return -1;
  while (b - a > 1) {
    const int m = (a + b) >> 1;
    if (__ldg(p.cu_q + m) <= r) a = m;
    else b = m;
  }
  return a;
}

// One warp per (bias head, query row): the finite range of the row's first kv_len values and
// whether they are all 0 there.
__global__ void __launch_bounds__(256) bias_row_bands_kernel(const Params p, int4 *rows) {
  const long long wid = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (wid >= (long long)p.total_q * p.bias_heads) return;
  const int lane = threadIdx.x & 31;
  const int hb = (int)(wid / p.total_q), r = (int)(wid % p.total_q);
  const int s = seq_of_row(p, r);
  int kv_len = 0;
  if (s >= 0) kv_len = min(max(__ldg(p.cu_kv + s + 1) - __ldg(p.cu_kv + s), 0), p.max_kv);
  const float *row = p.bias + ((size_t)r * (size_t)p.bias_heads + (size_t)hb) * (size_t)p.max_kv;
  // last finite value: scan back 128 values at a time (four coalesced 32-value loads per lane)
  int hi = 0;
  for (int j0 = kv_len; j0 > 0 && hi == 0; j0 -= 128) {
    unsigned found = 0u;
    int base = j0 - 128;
#pragma unroll
    for (int u = 3; u >= 0; --u) {
      const int j = base + 32 * u + lane;
      const bool fin = j >= 0 && j < j0 && __ldg(row + j) != -INFINITY;
      const unsigned m = __ballot_sync(0xffffffffu, fin);
      if (!found && m) found = 1u, hi = base + 32 * u + (31 - __clz((int)m)) + 1;
    }
  }
  // first finite value
  int lo = 0;
  if (hi > 0) {
    lo = -1;
    for (int j0 = 0; j0 < hi && lo < 0; j0 += 128) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + 32 * u + lane;
        const bool fin = j < hi && __ldg(row + j) != -INFINITY;
        const unsigned m = __ballot_sync(0xffffffffu, fin);
        if (lo < 0 && m) lo = j0 + 32 * u + (__ffs((int)m) - 1);
      }
    }
  }
  // pure: every value in [lo, hi) is exactly 0 (-inf holes, other values or NaN: not pure)
  int pure = 1;
  for (int j0 = lo; j0 < hi && pure; j0 += 128) {
    bool bad = false;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + 32 * u + lane;
      if (j < hi) bad |= !(__ldg(row + j) == 0.f);
    }
    if (__any_sync(0xffffffffu, bad)) pure = 0;
  }
  if (lane == 0) rows[(size_t)hb * p.total_q + r] = make_int4(lo, hi, pure, 0);
}

// One thread per (bias head, query row); the rows that start a 64-row block of their sequence
// combine that block's row entries.
__global__ void __launch_bounds__(256) bias_block_bands_kernel(const Params p, const int4 *rows,
                                                              int4 *blocks) {
  const long long t = (long long)blockIdx.x * 256 + threadIdx.x;
  if (t >= (long long)p.total_q * p.bias_heads) return;
  const int hb = (int)(t / p.total_q), r = (int)(t % p.total_q);
  const int s = seq_of_row(p, r);
  if (s < 0) return;
  const int q0 = __ldg(p.cu_q + s), q1 = __ldg(p.cu_q + s + 1);
  if ((r - q0) % 64 != 0) return;
  int lo = 0x7fffffff, hi = 0, pure = 1;
  for (int i = r; i < min(r + 64, q1); ++i) {
    const int4 e = rows[(size_t)hb * p.total_q + i];
    if (e.y > e.x) { lo = min(lo, e.x); hi = max(hi, e.y); }
    pure &= e.z;
  }
  if (hi == 0) lo = 0;
  blocks[(size_t)hb * p.total_q + r] = make_int4(lo, hi, pure, 0);
}

}  // namespace

size_t bias_bands_bytes(int total_q, int bias_heads) {
  if (total_q <= 0 || bias_heads <= 0) return 0;
  return 2 * (size_t)total_q * (size_t)bias_heads * sizeof(int4);
}

cudaError_t bias_bands(const Params &p, void *bands, cudaStream_t st) {
  const size_t n = (size_t)p.total_q * (size_t)p.bias_heads;
  if (n == 0) return cudaSuccess;
  int4 *rows = static_cast<int4 *>(bands), *blocks = rows + n;
  bias_row_bands_kernel<<<(unsigned)((n + 7) / 8), 256, 0, st>>>(p, rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  count_launch();
  bias_block_bands_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(p, rows, blocks);
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace vlf
