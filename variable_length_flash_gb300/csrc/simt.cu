// SIMT (fp32 FMA) kernels: forward, backward row-dot pre-pass, dQ, dK/dV.
//
// These carry every feature of the operation (varlen packing, end-aligned causal, sliding
// window, GQA/MQA, additive bias, asymmetric head widths up to 256) with plain IEEE fp32
// products, so fp32 inputs are never rounded to tf32 (the tf32-vs-ieee gap of triton-msl
// part 1, "Portability, measured").  They are the path for fp32 data and for head widths the
// tensor-core kernels do not cover, and a second, independent GPU implementation for tests.
//
// Tiling: a block of 128 threads owns 16 query rows (forward, dQ) or 16 keys (dK/dV) of one
// (sequence, head); thread t works on row t/8 and on every 8th column.  KV tiles are 32 keys
// and start at multiples of 32, so skipping fully masked tiles changes no bit of the result
// (the online-softmax state is untouched by an all-masked tile).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace vlf {
namespace {

constexpr int kRows = 16;     // query rows (fwd, dQ) or keys (dK/dV) per block
constexpr int kTile = 32;     // keys per KV tile (fwd, dQ) / query rows per Q tile (dK/dV)
constexpr int kThreads = 128;

__device__ __forceinline__ float warp8_max(float x) {
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp8_sum(float x) {
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Stage rows [row0, row0 + n) (n <= cap) of one head of a packed [T, H, D] tensor into smem as
// fp32 with row stride `ld`; rows >= n are zero.
template <typename T>
__device__ __forceinline__ void stage_rows(float *dst, int ld, const T *src, int row0, int n,
                                           int cap, int heads, int head, int d) {
  for (int idx = threadIdx.x; idx < cap * d; idx += kThreads) {
    const int r = idx / d, c = idx - r * d;
    float x = 0.f;
    if (r < n) x = to_f32<T>(src[((size_t)(row0 + r) * heads + head) * d + c]);
    dst[r * ld + c] = x;
  }
}

// ------------------------------------------------------------------------------ forward
template <typename T, int DVPT>
__global__ void __launch_bounds__(kThreads) simt_fwd_kernel(const Params p) {
  extern __shared__ float smem[];
  const int s = blockIdx.z, h = blockIdx.y, hk = h / p.group;
  Seq sq;
  if (!load_seq(p, s, sq)) return;
  if (s == 0 && (__ldg(p.cu_q) != 0 || __ldg(p.cu_kv) != 0)) set_error(p.err, VLF_ERR_BAD_SEQLENS);
  if (s == p.num_seqs - 1 && (sq.q0 + sq.q_len != p.total_q || sq.k0 + sq.kv_len != p.total_kv))
    set_error(p.err, VLF_ERR_BAD_SEQLENS);
  const int r0 = blockIdx.x * kRows;
  if (r0 >= sq.q_len) return;
  const int r1 = min(r0 + kRows, sq.q_len);
  const int dq = p.d_qk, dv = p.d_v;
  const int ldq = dq + 1, ldv = dv;
  float *Qs = smem;                    // [kRows][ldq]
  float *Ks = Qs + kRows * ldq;        // [kTile][ldq]
  float *Vs = Ks + kTile * ldq;        // [kTile][ldv]
  float *Ps = Vs + kTile * ldv;        // [kRows][kTile + 1]
  const T *q = static_cast<const T *>(p.q), *k = static_cast<const T *>(p.k);
  const T *v = static_cast<const T *>(p.v);

  const int t = threadIdx.x, r = t >> 3, sub = t & 7;
  const int i = r0 + r;  // sequence-local row of this thread
  const bool row_ok = i < r1;
  const int off = sq.kv_len - sq.q_len;

  int lo, hi;
  kv_band(r0, r1, sq.q_len, sq.kv_len, p.causal, p.window, lo, hi);
  if (p.flags & VLF_FLAG_NO_SKIP) { lo = 0; hi = sq.kv_len; }
  lo = (lo / kTile) * kTile;

  stage_rows<T>(Qs, ldq, q, sq.q0 + r0, r1 - r0, kRows, p.h_q, h, dq);

  float m = -INFINITY, l = 0.f;
  float o[DVPT];
#pragma unroll
  for (int u = 0; u < DVPT; ++u) o[u] = 0.f;

#pragma unroll 1
  for (int kt = lo; kt < hi; kt += kTile) {
    const int nk = min(kTile, sq.kv_len - kt);
    __syncthreads();  // previous tile fully consumed
    stage_rows<T>(Ks, ldq, k, sq.k0 + kt, nk, kTile, p.h_kv, hk, dq);
    stage_rows<T>(Vs, ldv, v, sq.k0 + kt, nk, kTile, p.h_kv, hk, dv);
    __syncthreads();
    float sc[4];
    float tmax = -INFINITY;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int jj = sub + 8 * a, j = kt + jj;
      float x = -INFINITY;
      if (row_ok && pair_visible(i, j, off, sq.kv_len, p.causal, p.window)) {
        float acc = 0.f;
        for (int c = 0; c < dq; ++c) acc = fmaf(Qs[r * ldq + c], Ks[jj * ldq + c], acc);
        x = p.scale * acc;
        if (p.bias) x += bias_at(p, sq.q0 + i, h, j);
      }
      sc[a] = x;
      tmax = fmaxf(tmax, x);
    }
    tmax = warp8_max(tmax);
    const float m_new = fmaxf(m, tmax);
    float alpha = 1.f, psum = 0.f;
    if (m_new != -INFINITY) {
      alpha = expf(m - m_new);  // m == -inf -> 0
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const float e = expf(sc[a] - m_new);  // masked -> 0
        sc[a] = e;
        psum += e;
      }
    } else {
#pragma unroll
      for (int a = 0; a < 4; ++a) sc[a] = 0.f;
    }
    psum = warp8_sum(psum);
    l = l * alpha + psum;
    m = m_new;
#pragma unroll
    for (int a = 0; a < 4; ++a) Ps[r * (kTile + 1) + sub + 8 * a] = sc[a];
    __syncthreads();
#pragma unroll
    for (int u = 0; u < DVPT; ++u) o[u] *= alpha;
#pragma unroll 2
    for (int jj = 0; jj < kTile; ++jj) {
      const float pj = Ps[r * (kTile + 1) + jj];
      const float *vrow = Vs + jj * ldv;
#pragma unroll
      for (int u = 0; u < DVPT; ++u) {
        const int c = sub + 8 * u;
        if (c < dv) o[u] = fmaf(pj, vrow[c], o[u]);
      }
    }
  }
  if (!row_ok) return;
  const size_t grow = (size_t)sq.q0 + i;
  T *out = static_cast<T *>(p.out) + (grow * p.h_q + h) * dv;
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int u = 0; u < DVPT; ++u) {
    const int c = sub + 8 * u;
    if (c < dv) out[c] = from_f32<T>(o[u] * inv);
  }
  if (p.lse && sub == 0) p.lse[(size_t)h * p.total_q + grow] = l > 0.f ? m + logf(l) : -INFINITY;
}

// ------------------------------------------------------------------------------ backward pre-pass
// rowdot[h, row] = sum_c dO[row, h, c] * O[row, h, c]  (one warp per (row, head)).
template <typename T>
__global__ void __launch_bounds__(256) rowdot_kernel(const Params p) {
  const long long pair = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (pair >= (long long)p.total_q * p.h_q) return;
  const long long row = pair / p.h_q;
  const int h = (int)(pair - row * p.h_q);
  const T *o = static_cast<const T *>(p.out) + ((size_t)row * p.h_q + h) * p.d_v;
  const T *d = static_cast<const T *>(p.dout) + ((size_t)row * p.h_q + h) * p.d_v;
  float acc = 0.f;
  for (int c = lane; c < p.d_v; c += 32) acc = fmaf(to_f32<T>(o[c]), to_f32<T>(d[c]), acc);
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (lane == 0) p.rowdot[(size_t)h * p.total_q + row] = acc;
}

// The same for 16-bit tensors whose width is 8 G L (G threads per pair, a power of two, each
// taking L 16-byte loads of O and of dO): (row, head) pairs are contiguous d_v-element segments,
// and the group sums by shuffles.  Many wide loads in flight keep HBM busy.
template <typename T, int G, int L>
__global__ void __launch_bounds__(256) rowdot16_kernel(const Params p) {
  const long long gtid = (long long)blockIdx.x * 256 + threadIdx.x;
  const long long pair = gtid / G;
  const int part = (int)(gtid % G);
  const long long pairs = (long long)p.total_q * p.h_q;
  float acc = 0.f;
  if (pair < pairs) {
    const uint4 *o4 = reinterpret_cast<const uint4 *>(static_cast<const T *>(p.out) + pair * (8 * G * L));
    const uint4 *d4 = reinterpret_cast<const uint4 *>(static_cast<const T *>(p.dout) + pair * (8 * G * L));
#pragma unroll
    for (int l = 0; l < L; ++l) {
      const uint4 o = __ldg(o4 + part * L + l), d = __ldg(d4 + part * L + l);
      const T *oe = reinterpret_cast<const T *>(&o), *de = reinterpret_cast<const T *>(&d);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc = fmaf(to_f32<T>(oe[e]), to_f32<T>(de[e]), acc);
    }
  }
#pragma unroll
  for (int s = G / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (pair < pairs && part == 0) {
    const long long row = pair / p.h_q;
    const int h = (int)(pair - row * p.h_q);
    p.rowdot[(size_t)h * p.total_q + row] = acc;
  }
}

// ------------------------------------------------------------------------------ dQ
template <typename T, int DQPT>
__global__ void __launch_bounds__(kThreads) simt_dq_kernel(const Params p) {
  extern __shared__ float smem[];
  const int s = blockIdx.z, h = blockIdx.y, hk = h / p.group;
  Seq sq;
  if (!load_seq(p, s, sq)) return;
  const int r0 = blockIdx.x * kRows;
  if (r0 >= sq.q_len) return;
  const int r1 = min(r0 + kRows, sq.q_len);
  const int dq = p.d_qk, dv = p.d_v;
  const int ldq = dq + 1, ldv = dv + 1;
  float *Qs = smem;                  // [kRows][ldq]
  float *DOs = Qs + kRows * ldq;     // [kRows][ldv]
  float *Ks = DOs + kRows * ldv;     // [kTile][ldq]
  float *Vs = Ks + kTile * ldq;      // [kTile][ldv]
  float *Ss = Vs + kTile * ldv;      // [kRows][kTile + 1]  dS
  const T *q = static_cast<const T *>(p.q), *k = static_cast<const T *>(p.k);
  const T *v = static_cast<const T *>(p.v), *dout = static_cast<const T *>(p.dout);
  const int t = threadIdx.x, r = t >> 3, sub = t & 7;
  const int i = r0 + r;
  const bool row_ok = i < r1;
  const int off = sq.kv_len - sq.q_len;
  const size_t grow = (size_t)sq.q0 + (row_ok ? i : r0);
  const float lse = row_ok ? p.lse[(size_t)h * p.total_q + grow] : -INFINITY;
  const float Di = row_ok ? p.rowdot[(size_t)h * p.total_q + grow] : 0.f;

  int lo, hi;
  kv_band(r0, r1, sq.q_len, sq.kv_len, p.causal, p.window, lo, hi);
  if (p.flags & VLF_FLAG_NO_SKIP) { lo = 0; hi = sq.kv_len; }
  lo = (lo / kTile) * kTile;

  stage_rows<T>(Qs, ldq, q, sq.q0 + r0, r1 - r0, kRows, p.h_q, h, dq);
  stage_rows<T>(DOs, ldv, dout, sq.q0 + r0, r1 - r0, kRows, p.h_q, h, dv);

  float acc[DQPT];
#pragma unroll
  for (int u = 0; u < DQPT; ++u) acc[u] = 0.f;

#pragma unroll 1
  for (int kt = lo; kt < hi; kt += kTile) {
    const int nk = min(kTile, sq.kv_len - kt);
    __syncthreads();
    stage_rows<T>(Ks, ldq, k, sq.k0 + kt, nk, kTile, p.h_kv, hk, dq);
    stage_rows<T>(Vs, ldv, v, sq.k0 + kt, nk, kTile, p.h_kv, hk, dv);
    __syncthreads();
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int jj = sub + 8 * a, j = kt + jj;
      float ds = 0.f;
      if (row_ok && lse != -INFINITY && pair_visible(i, j, off, sq.kv_len, p.causal, p.window)) {
        float sdot = 0.f, pdot = 0.f;
        for (int c = 0; c < dq; ++c) sdot = fmaf(Qs[r * ldq + c], Ks[jj * ldq + c], sdot);
        for (int c = 0; c < dv; ++c) pdot = fmaf(DOs[r * ldv + c], Vs[jj * ldv + c], pdot);
        float x = p.scale * sdot;
        if (p.bias) x += bias_at(p, (int)grow, h, j);
        const float pr = expf(x - lse);
        ds = pr * (pdot - Di);
      }
      Ss[r * (kTile + 1) + jj] = ds;
    }
    __syncthreads();
#pragma unroll 2
    for (int jj = 0; jj < kTile; ++jj) {
      const float dsj = Ss[r * (kTile + 1) + jj];
      const float *krow = Ks + jj * ldq;
#pragma unroll
      for (int u = 0; u < DQPT; ++u) {
        const int c = sub + 8 * u;
        if (c < dq) acc[u] = fmaf(dsj, krow[c], acc[u]);
      }
    }
  }
  if (!row_ok) return;
  T *dqp = static_cast<T *>(p.dq) + (grow * p.h_q + h) * dq;
#pragma unroll
  for (int u = 0; u < DQPT; ++u) {
    const int c = sub + 8 * u;
    if (c < dq) dqp[c] = from_f32<T>(acc[u] * p.scale);
  }
}

// ------------------------------------------------------------------------------ dK / dV
// Block: 16 keys of one (sequence, kv head); loops over the group's query heads and the query
// rows that can see those keys, in tiles of 32 rows.  No atomics: one block owns its keys.
template <typename T, int DPT>
__global__ void __launch_bounds__(kThreads) simt_dkdv_kernel(const Params p) {
  extern __shared__ float smem[];
  const int s = blockIdx.z, hk = blockIdx.y;
  Seq sq;
  if (!load_seq(p, s, sq)) return;
  const int j0 = blockIdx.x * kRows;
  if (j0 >= sq.kv_len) return;
  const int j1 = min(j0 + kRows, sq.kv_len);
  const int dq = p.d_qk, dv = p.d_v;
  const int ldq = dq + 1, ldv = dv + 1;
  float *Ks = smem;                  // [kRows][ldq]
  float *Vs = Ks + kRows * ldq;      // [kRows][ldv]
  float *Qs = Vs + kRows * ldv;      // [kTile][ldq]
  float *DOs = Qs + kTile * ldq;     // [kTile][ldv]
  float *Ps = DOs + kTile * ldv;     // [kRows][kTile + 1]
  float *Ss = Ps + kRows * (kTile + 1);  // [kRows][kTile + 1]
  float *Ls = Ss + kRows * (kTile + 1);  // [kTile] lse
  float *Ds = Ls + kTile;                // [kTile] rowdot
  const T *q = static_cast<const T *>(p.q), *k = static_cast<const T *>(p.k);
  const T *v = static_cast<const T *>(p.v), *dout = static_cast<const T *>(p.dout);
  const int t = threadIdx.x, kr = t >> 3, sub = t & 7;
  const int j = j0 + kr;
  const bool key_ok = j < j1;
  const int off = sq.kv_len - sq.q_len;

  stage_rows<T>(Ks, ldq, k, sq.k0 + j0, j1 - j0, kRows, p.h_kv, hk, dq);
  stage_rows<T>(Vs, ldv, v, sq.k0 + j0, j1 - j0, kRows, p.h_kv, hk, dv);

  float ak[DPT], av[DPT];
#pragma unroll
  for (int u = 0; u < DPT; ++u) ak[u] = av[u] = 0.f;

  int qlo, qhi;
  q_band(j0, j1, sq.q_len, sq.kv_len, p.causal, p.window, qlo, qhi);
  if (p.flags & VLF_FLAG_NO_SKIP) { qlo = 0; qhi = sq.q_len; }
  qlo = (qlo / kTile) * kTile;

  for (int g = 0; g < p.group; ++g) {
    const int h = hk * p.group + g;
    for (int it = qlo; it < qhi; it += kTile) {
      const int nq = min(kTile, sq.q_len - it);
      __syncthreads();
      stage_rows<T>(Qs, ldq, q, sq.q0 + it, nq, kTile, p.h_q, h, dq);
      stage_rows<T>(DOs, ldv, dout, sq.q0 + it, nq, kTile, p.h_q, h, dv);
      if (t < kTile) {
        const bool ok = t < nq;
        Ls[t] = ok ? p.lse[(size_t)h * p.total_q + sq.q0 + it + t] : -INFINITY;
        Ds[t] = ok ? p.rowdot[(size_t)h * p.total_q + sq.q0 + it + t] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int ii = sub + 8 * a, i = it + ii;
        float pr = 0.f, ds = 0.f;
        if (key_ok && i < sq.q_len && Ls[ii] != -INFINITY &&
            pair_visible(i, j, off, sq.kv_len, p.causal, p.window)) {
          float sdot = 0.f, pdot = 0.f;
          for (int c = 0; c < dq; ++c) sdot = fmaf(Ks[kr * ldq + c], Qs[ii * ldq + c], sdot);
          for (int c = 0; c < dv; ++c) pdot = fmaf(Vs[kr * ldv + c], DOs[ii * ldv + c], pdot);
          float x = p.scale * sdot;
          if (p.bias) x += bias_at(p, sq.q0 + i, h, j);
          pr = expf(x - Ls[ii]);
          ds = pr * (pdot - Ds[ii]);
        }
        Ps[kr * (kTile + 1) + ii] = pr;
        Ss[kr * (kTile + 1) + ii] = ds;
      }
      __syncthreads();
#pragma unroll 2
      for (int ii = 0; ii < kTile; ++ii) {
        const float pi = Ps[kr * (kTile + 1) + ii], dsi = Ss[kr * (kTile + 1) + ii];
        const float *dorow = DOs + ii * ldv, *qrow = Qs + ii * ldq;
#pragma unroll
        for (int u = 0; u < DPT; ++u) {
          const int c = sub + 8 * u;
          if (c < dv) av[u] = fmaf(pi, dorow[c], av[u]);
          if (c < dq) ak[u] = fmaf(dsi, qrow[c], ak[u]);
        }
      }
    }
  }
  if (!key_ok) return;
  const size_t gk = (size_t)sq.k0 + j;
  T *dkp = static_cast<T *>(p.dk) + (gk * p.h_kv + hk) * dq;
  T *dvp = static_cast<T *>(p.dv) + (gk * p.h_kv + hk) * dv;
#pragma unroll
  for (int u = 0; u < DPT; ++u) {
    const int c = sub + 8 * u;
    if (c < dq) dkp[c] = from_f32<T>(ak[u] * p.scale);
    if (c < dv) dvp[c] = from_f32<T>(av[u]);
  }
}

template <typename Kern>
cudaError_t launch(Kern kern, dim3 grid, size_t smem, cudaStream_t st, const Params &p) {
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, st>>>(p);
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

template <typename T>
cudaError_t fwd_t(const Params &p, cudaStream_t st) {
  const dim3 grid((p.max_q + kRows - 1) / kRows, p.h_q, p.num_seqs);
  const size_t smem = sizeof(float) * ((size_t)kRows * (p.d_qk + 1) + (size_t)kTile * (p.d_qk + 1) +
                                       (size_t)kTile * p.d_v + (size_t)kRows * (kTile + 1));
  if (p.d_v <= 64) return launch(simt_fwd_kernel<T, 8>, grid, smem, st, p);
  if (p.d_v <= 128) return launch(simt_fwd_kernel<T, 16>, grid, smem, st, p);
  return launch(simt_fwd_kernel<T, 32>, grid, smem, st, p);
}

template <typename T>
cudaError_t bwd_t(const Params &p, cudaStream_t st, const cudaEvent_t *ev) {
  cudaError_t e = mark(ev, 0, st);
  if (e != cudaSuccess) return e;
  if (p.total_q > 0) {
    const long long pairs = (long long)p.total_q * p.h_q;
    rowdot_kernel<T><<<(unsigned)((pairs + 7) / 8), 256, 0, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launch();
  }
  if ((e = mark(ev, 1, st)) != cudaSuccess) return e;
  {
    // dK/dV (stage 1)
    const dim3 grid((p.max_kv + kRows - 1) / kRows, p.h_kv, p.num_seqs);
    const size_t smem = sizeof(float) * ((size_t)kRows * (p.d_qk + 1) + (size_t)kRows * (p.d_v + 1) +
                                         (size_t)kTile * (p.d_qk + 1) + (size_t)kTile * (p.d_v + 1) +
                                         2 * (size_t)kRows * (kTile + 1) + 2 * (size_t)kTile);
    const int dmax = p.d_qk > p.d_v ? p.d_qk : p.d_v;
    if (dmax <= 64) e = launch(simt_dkdv_kernel<T, 8>, grid, smem, st, p);
    else if (dmax <= 128) e = launch(simt_dkdv_kernel<T, 16>, grid, smem, st, p);
    else e = launch(simt_dkdv_kernel<T, 32>, grid, smem, st, p);
    if (e != cudaSuccess) return e;
  }
  if ((e = mark(ev, 2, st)) != cudaSuccess) return e;
  {
    // dQ (stage 2)
    const dim3 grid((p.max_q + kRows - 1) / kRows, p.h_q, p.num_seqs);
    const size_t smem = sizeof(float) * ((size_t)kRows * (p.d_qk + 1) + (size_t)kRows * (p.d_v + 1) +
                                         (size_t)kTile * (p.d_qk + 1) + (size_t)kTile * (p.d_v + 1) +
                                         (size_t)kRows * (kTile + 1));
    if (p.d_qk <= 64) e = launch(simt_dq_kernel<T, 8>, grid, smem, st, p);
    else if (p.d_qk <= 128) e = launch(simt_dq_kernel<T, 16>, grid, smem, st, p);
    else e = launch(simt_dq_kernel<T, 32>, grid, smem, st, p);
    if (e != cudaSuccess) return e;
  }
  return mark(ev, 3, st);
}

}  // namespace

cudaError_t simt_forward(const Params &p, cudaStream_t st) {
  if (p.max_q == 0 || p.num_seqs == 0) return cudaSuccess;
  switch (p.dtype) {
    case VLF_F16: return fwd_t<__half>(p, st);
    case VLF_BF16: return fwd_t<__nv_bfloat16>(p, st);
    default: return fwd_t<float>(p, st);
  }
}

cudaError_t rowdot_forward(const Params &p, cudaStream_t st) {
  if (p.total_q == 0) return cudaSuccess;
  const long long pairs = (long long)p.total_q * p.h_q;
  if (p.dtype != VLF_F32 && (p.d_v == 64 || p.d_v == 96 || p.d_v == 128 || p.d_v == 256)) {
    // (16-byte loads: the API requires 16-byte aligned tensors, and every segment starts at a
    // multiple of d_v elements, itself a multiple of 8)
    const int g = p.d_v == 96 ? 4 : (p.d_v == 256 ? 16 : p.d_v / 8);
    const unsigned blocks = (unsigned)((pairs * g + 255) / 256);
    const bool f16 = p.dtype == VLF_F16;
    if (p.d_v == 64) {
      if (f16) rowdot16_kernel<__half, 8, 1><<<blocks, 256, 0, st>>>(p);
      else rowdot16_kernel<__nv_bfloat16, 8, 1><<<blocks, 256, 0, st>>>(p);
    } else if (p.d_v == 96) {
      if (f16) rowdot16_kernel<__half, 4, 3><<<blocks, 256, 0, st>>>(p);
      else rowdot16_kernel<__nv_bfloat16, 4, 3><<<blocks, 256, 0, st>>>(p);
    } else if (p.d_v == 256) {
      if (f16) rowdot16_kernel<__half, 16, 2><<<blocks, 256, 0, st>>>(p);
      else rowdot16_kernel<__nv_bfloat16, 16, 2><<<blocks, 256, 0, st>>>(p);
    } else {
      if (f16) rowdot16_kernel<__half, 16, 1><<<blocks, 256, 0, st>>>(p);
      else rowdot16_kernel<__nv_bfloat16, 16, 1><<<blocks, 256, 0, st>>>(p);
    }
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launch();
    return e;
  }
  const unsigned blocks = (unsigned)((pairs + 7) / 8);
  switch (p.dtype) {
    case VLF_F16: rowdot_kernel<__half><<<blocks, 256, 0, st>>>(p); break;
    case VLF_BF16: rowdot_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(p); break;
    default: rowdot_kernel<float><<<blocks, 256, 0, st>>>(p); break;
  }
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

cudaError_t simt_backward(const Params &p, cudaStream_t st, const cudaEvent_t *ev) {
  switch (p.dtype) {
    case VLF_F16: return bwd_t<__half>(p, st, ev);
    case VLF_BF16: return bwd_t<__nv_bfloat16>(p, st, ev);
    default: return bwd_t<float>(p, st, ev);
  }
}

}  // namespace vlf
