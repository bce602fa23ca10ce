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
// [bias_heads][total_q] entries:
//   rows   entry (hb, r) = {lo, hi, pure, 0}: keys [lo, hi) of global query row r (lo = hi = 0
//          when no key is finite), pure 1 when the bias is 0 throughout them
//   blocks entry (hb, q0 + 64 b) for each sequence (first row q0) and block b of 64 of its rows =
//          {lo, hi, ilo, ihi}: the union [lo, hi) of those rows' intervals and, when every row is
//          pure, their intersection [ilo, ihi) (keys every row of the block sees; empty if a row
//          sees none); ilo = ihi = -1 when some row is not pure (other entries unused).
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
// whether they are all 0 there.  The scans read 512 values (2 KB) per warp step, four 16-byte
// loads per lane in flight, when the row is 16-byte aligned (max_kv a multiple of 4); 128
// values per step with scalar loads otherwise.
__global__ void __launch_bounds__(256) bias_row_bands_kernel(const Params p, int4 *rows) {
  const long long wid = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (wid >= (long long)p.total_q * p.bias_heads) return;
  const int lane = threadIdx.x & 31;
  const int hb = (int)(wid / p.total_q), r = (int)(wid % p.total_q);
  const int s = seq_of_row(p, r);
  int kv_len = 0;
  if (s >= 0) kv_len = min(max(__ldg(p.cu_kv + s + 1) - __ldg(p.cu_kv + s), 0), p.max_kv);
  const float *row = p.bias + ((size_t)r * (size_t)p.bias_heads + (size_t)hb) * (size_t)p.max_kv;
  const bool vec = (p.max_kv & 3) == 0;
  const float4 *row4 = reinterpret_cast<const float4 *>(row);
  // the value at j, or -inf past the row's keys (j >= kv_len)
  auto fin4 = [&](int c4, float4 &v) {  // 16-byte chunk c4 (values 4 c4 .. 4 c4 + 3)
    v = 4 * c4 < kv_len ? __ldg(row4 + c4) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  };
  // last finite value: scan back from the end
  int hi = 0;
  if (vec) {
    const int n4 = (kv_len + 3) / 4;  // chunks holding the row's keys
    for (int c0 = n4; c0 > 0 && hi == 0; c0 -= 128) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c4 = c0 - 128 + 32 * u + lane;
        if (c4 >= 0 && c4 < c0) fin4(c4, v[u]);
        else v[u] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
      int best = -1;  // this lane's highest finite index in the step
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j0 = 4 * (c0 - 128 + 32 * u + lane);
        const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (e[q] != -INFINITY && j0 + q < kv_len) best = max(best, j0 + q);
      }
      best = __reduce_max_sync(0xffffffffu, best);
      if (best >= 0) hi = best + 1;
    }
  } else {
    for (int j0 = kv_len; j0 > 0 && hi == 0; j0 -= 128) {
      int best = -1;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 - 128 + 32 * u + lane;
        if (j >= 0 && j < j0 && __ldg(row + j) != -INFINITY) best = max(best, j);
      }
      best = __reduce_max_sync(0xffffffffu, best);
      if (best >= 0) hi = best + 1;
    }
  }
  // first finite value (below hi there is one)
  int lo = 0;
  if (hi > 0) {
    lo = -1;
    for (int j0 = 0; j0 < hi && lo < 0; j0 += vec ? 512 : 128) {
      int first = 0x7fffffff;
      if (vec) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c4 = j0 / 4 + 32 * u + lane;
          float4 v;
          fin4(c4, v);
          const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (e[q] != -INFINITY && 4 * c4 + q < hi) first = min(first, 4 * c4 + q);
        }
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + 32 * u + lane;
          if (j < hi && __ldg(row + j) != -INFINITY) first = min(first, j);
        }
      }
      first = __reduce_min_sync(0xffffffffu, first);
      if (first != 0x7fffffff) lo = first;
    }
  }
  // pure: every value in [lo, hi) is exactly 0 (-inf holes, other values or NaN: not pure)
  int pure = 1;
  for (int j0 = vec ? (lo & ~3) : lo; j0 < hi && pure; j0 += vec ? 512 : 128) {
    bool bad = false;
    if (vec) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c4 = j0 / 4 + 32 * u + lane;
        float4 v;
        fin4(c4, v);
        const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int j = 4 * c4 + q;
          if (j >= lo && j < hi) bad |= !(e[q] == 0.f);
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + 32 * u + lane;
        if (j < hi) bad |= !(__ldg(row + j) == 0.f);
      }
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
  int lo = 0x7fffffff, hi = 0, pure = 1, ilo = 0, ihi = 0x7fffffff;
  for (int i = r; i < min(r + 64, q1); ++i) {
    const int4 e = rows[(size_t)hb * p.total_q + i];
    if (e.y > e.x) { lo = min(lo, e.x); hi = max(hi, e.y); }
    ilo = max(ilo, e.x);
    ihi = min(ihi, e.y);
    pure &= e.z;
  }
  if (hi == 0) lo = 0;
  if (ihi < ilo) ihi = ilo;  // (empty intersection)
  blocks[(size_t)hb * p.total_q + r] = pure ? make_int4(lo, hi, ilo, ihi) : make_int4(lo, hi, -1, -1);
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
