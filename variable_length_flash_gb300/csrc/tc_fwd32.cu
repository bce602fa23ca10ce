// Tensor-core forward for fp32 inputs (sm_103a): the products in three tf32 passes.
//
// tf32 keeps 10 of fp32's 23 mantissa bits, so a single tf32 product loses accuracy that fp32
// data is expected to keep (triton-msl part 1, "Portability, measured": the tf32 matmul is the
// fast one and the inaccurate one).  Each fp32 operand x is split into x_hi = x rounded to tf32
// and x_lo = (x - x_hi) rounded to tf32 (the subtraction is exact); a product a b is then taken
// as a_hi b_lo + a_lo b_hi + a_hi b_hi with fp32 accumulation, which drops only a_lo b_lo and the
// rounding of the low parts (relative error about 2^-21 per product instead of 2^-11).
//
// The loop is the forward of tc_fwd.cu (FlashAttention-2: Q staged once, then per 64-key tile
// S = Q K^T, online softmax with a lazily moved reference max, O += P V), one 128-row query tile
// per CTA, with these differences:
//  * 384 threads: warp 0 issues TMA loads, warp 1 the S products, warp 2 the P.V products,
//    warps 4-7 run the softmax (one thread per query row), warps 8-11 split operands.  The
//    splitting warps round the Q tile and each K tile to tf32 in place and write their low
//    parts beside them (same swizzled layout); each V tile lands in a staging ring and is
//    written out transposed (keys along the row, K-major, the layout both tf32 operands of
//    the P.V product take) as its high and low parts.
//  * TMEM: O at column 0; S buffer b (64 fp32 columns) at 128 + 128 b, where the softmax writes
//    P's high parts over S, and P's low parts at 192 + 128 b.  P.V takes both from TMEM.
//  * fp32 output; O is normalised by the fp32 row sum of P.
// Every wait is bounded (tc_common.cuh); a timeout records VLF_ERR_TIMEOUT, the CTA drains its
// copies and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace vlf {

bool make_tmap_f32(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols,
                   uint64_t pitch_elems, uint32_t box_rows);

namespace {

using namespace tc;

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kBN = 64;                    // keys per KV tile

struct Fwd32Maps {
  CUtensorMap q, k, v;
};

// D: head width (32 or 64, Q/K and V alike).  NK: K ring slots; NVR: V staging slots; NV:
// transposed-V ring slots.
template <int D, int NK, int NVR, int NV>
struct F32Cfg {
  static constexpr int KB = D / 32;             // 32-column (128-byte) swizzle blocks per row
  static constexpr int QBLK = 128 * 128;        // 128 rows x 128 bytes
  static constexpr int KVBLK = kBN * 128;       // 64 rows x 128 bytes
  static constexpr int VTBLK = D * 128;         // transposed V: D rows x 32 keys x 4 bytes
  static constexpr int Q_BYTES = KB * QBLK, KV_BYTES = KB * KVBLK;
  static constexpr int OFF_Q = 0, OFF_QL = Q_BYTES;
  static constexpr int OFF_K = 2 * Q_BYTES, OFF_KL = OFF_K + NK * KV_BYTES;
  static constexpr int OFF_VR = OFF_KL + NK * KV_BYTES;           // V as loaded
  static constexpr int OFF_VT = OFF_VR + NVR * KV_BYTES;          // per slot: high, then low
  static constexpr int OFF_BAR = OFF_VT + NV * 2 * KV_BYTES;
  // barriers: q_full, qc_full (Q split), k_full[NK], kc_full[NK] (K split), k_empty[NK],
  // vr_full[NVR], vr_empty[NVR] (V staging read), vt_full[NV], vt_empty[NV], then per S buffer
  // s_full[2], p_full[2], o_done[2]; drain[2]
  static constexpr int B_Q = 0, B_QC = 1, B_KF = 2, B_KC = B_KF + NK, B_KE = B_KC + NK;
  static constexpr int B_VRF = B_KE + NK, B_VRE = B_VRF + NVR, B_VTF = B_VRE + NVR;
  static constexpr int B_VTE = B_VTF + NV, B_S = B_VTE + NV, B_P = B_S + 2, B_O = B_P + 2;
  static constexpr int B_DRAIN = B_O + 2, NBAR = B_DRAIN + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16;
  static constexpr int THREADS = 384;
  static constexpr uint32_t TMEM_COLS = 512, S_COL = 128, PL_OFF = 64;
  static_assert(D == 32 || D == 64, "head widths with an fp32 tensor-core forward");
  static_assert(NK >= 2 && NVR >= 1 && NV >= 2, "ring depths");
  static_assert(SMEM <= 232448, "shared memory");
};

// hi = x rounded to tf32, lo = (x - hi) rounded to tf32, as bit patterns
__device__ __forceinline__ void split_tf32(uint32_t x, uint32_t &hi, uint32_t &lo) {
  const float f = __uint_as_float(x);
  const float h = tf32_round(f);
  hi = __float_as_uint(h);
  lo = __float_as_uint(tf32_round(__fsub_rn(f, h)));
}

// Splits `bytes` of fp32 data at src in place into its tf32 high parts and writes the low parts
// at the same offsets from dst; thread t of n takes 16-byte chunks t, t + n, ...
__device__ __forceinline__ void split_block(uint32_t src, uint32_t dst, int bytes, int t, int n) {
  for (int c = t; c < bytes / 16; c += n) {
    uint32_t x0, x1, x2, x3, h0, h1, h2, h3, l0, l1, l2, l3;
    lds_v4(src + 16 * c, x0, x1, x2, x3);
    split_tf32(x0, h0, l0);
    split_tf32(x1, h1, l1);
    split_tf32(x2, h2, l2);
    split_tf32(x3, h3, l3);
    sts_v4(src + 16 * c, h0, h1, h2, h3);
    sts_v4(dst + 16 * c, l0, l1, l2, l3);
  }
}

__device__ __forceinline__ void sts_u32(uint32_t a, uint32_t x) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(x) : "memory");
}

template <int D, int NK, int NVR, int NV, int BIAS>
__global__ void __launch_bounds__(384, 1)
tc_fwd32_kernel(const __grid_constant__ Fwd32Maps maps, const Params p) {
  using C = F32Cfg<D, NK, NVR, NV>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int s = (int)blockIdx.z;
  Seq sq;
  if (!load_seq(p, s, sq)) return;
  if (s == 0 && (__ldg(p.cu_q) != 0 || __ldg(p.cu_kv) != 0)) set_error(p.err, VLF_ERR_BAD_SEQLENS);
  if (s == p.num_seqs - 1 && (sq.q0 + sq.q_len != p.total_q || sq.k0 + sq.kv_len != p.total_kv))
    set_error(p.err, VLF_ERR_BAD_SEQLENS);
  // heavy (late, long-band) row blocks first under causal masking
  const int bx = p.causal ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x;
  const int head = (int)blockIdx.y, hk = head / p.group;
  const int row0 = bx * 128;
  if (row0 >= sq.q_len) return;  // whole CTA beyond this sequence
  int lo = 0, hi = 0;           // the KV tiles of the band
  if (sq.kv_len > 0) {
    int klo, khi;
    kv_band(row0, min(row0 + 128, sq.q_len), sq.q_len, sq.kv_len, p.causal, p.window, klo, khi);
    if (p.flags & VLF_FLAG_NO_SKIP) { klo = 0; khi = sq.kv_len; }
    if (khi > klo) { lo = klo / kBN; hi = (khi + kBN - 1) / kBN; }
  }

  // no static shared memory: the dynamic window starts 1024-byte aligned, as the swizzle atoms
  // of the TMA tiles and the MMA descriptors require; refuse otherwise
  const uint32_t base = smem_u32(smem_raw);
  if (base & 1023u) {
    if (threadIdx.x == 0) set_error(p.err, VLF_ERR_ALIGN);
    return;
  }
  const uint32_t sQ = base + C::OFF_Q, sQL = base + C::OFF_QL, sK = base + C::OFF_K;
  const uint32_t sKL = base + C::OFF_KL, sVR = base + C::OFF_VR, sVT = base + C::OFF_VT;
  const uint32_t bar0 = base + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem_raw + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem_raw + C::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_Q), 1);
    mbar_init(bar(C::B_QC), 128);
    for (int i = 0; i < NK; ++i) {
      mbar_init(bar(C::B_KF + i), 1);
      mbar_init(bar(C::B_KC + i), 128);
      mbar_init(bar(C::B_KE + i), 1);
    }
    for (int i = 0; i < NVR; ++i) { mbar_init(bar(C::B_VRF + i), 1); mbar_init(bar(C::B_VRE + i), 128); }
    for (int i = 0; i < NV; ++i) { mbar_init(bar(C::B_VTF + i), 128); mbar_init(bar(C::B_VTE + i), 1); }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::B_S + b), 1);
      mbar_init(bar(C::B_P + b), 128);
      mbar_init(bar(C::B_O + b), 1);
      mbar_init(bar(C::B_DRAIN + b), 1);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
    tmem_relinquish();
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && hi > lo) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      mbar_expect_tx(bar(C::B_Q), C::Q_BYTES);
      for (int c = 0; c < C::KB; ++c)
        tma_load_2d(sQ + c * C::QBLK, &maps.q, head * D + 32 * c, sq.q0 + row0, bar(C::B_Q));
      int k_issued[NK] = {0}, v_issued[NVR] = {0};
      bool ok = true;
      // K tile j + 1 is issued before V tile j: a K load never queues behind a V slot
      for (int j = lo; j < hi + 1 && ok; ++j) {
        const int kj = j, vj = j - 1;
        if (kj < hi) {
          const int it = kj - lo, ks = it % NK;
          if (it >= NK) ok = mbar_wait(bar(C::B_KE + ks), ((it / NK) - 1) & 1, abort_flag, p.err);
          if (!ok) break;
          mbar_expect_tx(bar(C::B_KF + ks), C::KV_BYTES);
          for (int c = 0; c < C::KB; ++c)
            tma_load_2d(sK + ks * C::KV_BYTES + c * C::KVBLK, &maps.k, hk * D + 32 * c,
                        sq.k0 + kj * kBN, bar(C::B_KF + ks));
          ++k_issued[ks];
        }
        if (vj >= lo) {
          const int it = vj - lo, vs = it % NVR;
          if (it >= NVR) ok = mbar_wait(bar(C::B_VRE + vs), ((it / NVR) - 1) & 1, abort_flag, p.err);
          if (!ok) break;
          mbar_expect_tx(bar(C::B_VRF + vs), C::KV_BYTES);
          for (int c = 0; c < C::KB; ++c)
            tma_load_2d(sVR + vs * C::KV_BYTES + c * C::KVBLK, &maps.v, hk * D + 32 * c,
                        sq.k0 + vj * kBN, bar(C::B_VRF + vs));
          ++v_issued[vs];
        }
      }
      // no copy may still be landing in shared memory when the CTA leaves
      drain_wait(bar(C::B_Q), 0);
      for (int i = 0; i < NK; ++i)
        if (k_issued[i]) drain_wait(bar(C::B_KF + i), (k_issued[i] - 1) & 1);
      for (int i = 0; i < NVR; ++i)
        if (v_issued[i]) drain_wait(bar(C::B_VRF + i), (v_issued[i] - 1) & 1);
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------------ MMA issuers
    // warp 1: S(n) = Q K^T as Q_hi K_lo + Q_lo K_hi + Q_hi K_hi into S buffer n mod 2, once the
    // K tile is split and the P.V that read the buffer two tiles ago has completed;
    // warp 2: O += P_lo V_hi + P_hi V_lo + P_hi V_hi once the softmax has written P(n) and the
    // transposed V tile is ready.  Small products first: the large one is added last.
    const bool is_s = warp == 1;
    if (hi > lo) {
      bool ok = true;
      auto wait_all = [&](int b, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar(b), parity, abort_flag, p.err));
      };
      if (is_s) {
        const uint32_t id = idesc_tf32(128, kBN);
        const uint64_t dq = sdesc_sw128(sQ, 16, 1024), dql = sdesc_sw128(sQL, 16, 1024);
        ok = wait_all(C::B_Q, 0) && wait_all(C::B_QC, 0);
        for (int j = lo; j < hi && ok; ++j) {
          const int n = j - lo, ks = n % NK, b = n & 1;
          ok = wait_all(C::B_KF + ks, (n / NK) & 1) && wait_all(C::B_KC + ks, (n / NK) & 1);
          if (ok && n >= 2) ok = wait_all(C::B_O + b, ((n - 2) >> 1) & 1);
          if (!ok) break;
          fence_after();
          const uint64_t dk = sdesc_sw128(sK + ks * C::KV_BYTES, 16, 1024);
          const uint64_t dkl = sdesc_sw128(sKL + ks * C::KV_BYTES, 16, 1024);
          const uint32_t d_s = tmem + C::S_COL + 128 * b;
#pragma unroll
          for (int part = 0; part < 3; ++part) {
            const uint64_t a = part == 1 ? dql : dq, bb = part == 0 ? dkl : dk;
#pragma unroll
            for (int kk = 0; kk < D / 8; ++kk) {
              // a K step of 8 fp32 adds its byte offset / 16 to the start-address field
              const uint64_t oq = (uint64_t)(((kk >> 2) * C::QBLK + (kk & 3) * 32) >> 4);
              const uint64_t ok_ = (uint64_t)(((kk >> 2) * C::KVBLK + (kk & 3) * 32) >> 4);
              mma_ss_tf32_w(d_s, a + oq, bb + ok_, id, (part > 0 || kk > 0) ? 1u : 0u);
            }
          }
          mma_commit_w(bar(C::B_S + b));
          mma_commit_w(bar(C::B_KE + ks));  // the K slot (high and low parts) may be refilled
        }
      } else {
        const uint32_t id = idesc_tf32(128, D);
        for (int j = lo; j < hi && ok; ++j) {
          const int n = j - lo, vs = n % NV, b = n & 1;
          ok = wait_all(C::B_VTF + vs, (n / NV) & 1) && wait_all(C::B_P + b, (n >> 1) & 1);
          if (!ok) break;
          fence_after();
          const uint32_t vt = sVT + vs * 2 * C::KV_BYTES;
          const uint64_t dvh = sdesc_sw128(vt, 16, 1024), dvl = sdesc_sw128(vt + C::KV_BYTES, 16, 1024);
          const uint32_t ph = tmem + C::S_COL + 128 * b, pl = ph + C::PL_OFF;
#pragma unroll
          for (int part = 0; part < 3; ++part) {
            const uint32_t a = part == 0 ? pl : ph;
            const uint64_t bb = part == 1 ? dvl : dvh;
#pragma unroll
            for (int kk = 0; kk < kBN / 8; ++kk) {
              const uint64_t ov = (uint64_t)(((kk >> 2) * C::VTBLK + (kk & 3) * 32) >> 4);
              mma_ts_tf32_w(tmem, a + 8 * kk, bb + ov, id, (n > 0 || part > 0 || kk > 0) ? 1u : 0u);
            }
          }
          mma_commit_w(bar(C::B_O + b));
          mma_commit_w(bar(C::B_VTE + vs));  // the transposed V slot may be rewritten
        }
      }
      // drain: every MMA this warp issued has completed before TMEM is released
      const int drain = C::B_DRAIN + (is_s ? 0 : 1);
      mma_commit_w(bar(drain));
      drain_wait(bar(drain), 0);
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------------ operand splitting
    const int t = threadIdx.x - 256;
    if (hi > lo) {
      bool ok = mbar_wait(bar(C::B_Q), 0, abort_flag, p.err);
      if (ok) {
        split_block(sQ, sQL, C::Q_BYTES, t, 128);
        fence_proxy_async_smem();  // generic-proxy writes, read next by the tensor core
        mbar_arrive(bar(C::B_QC));
      }
      const int wl = t >> 5;  // this warp's share of the V transposition
      for (int j = lo; j < hi && ok; ++j) {
        const int n = j - lo;
        const int ks = n % NK;
        ok = mbar_wait(bar(C::B_KF + ks), (n / NK) & 1, abort_flag, p.err);
        if (!ok) break;
        split_block(sK + ks * C::KV_BYTES, sKL + ks * C::KV_BYTES, C::KV_BYTES, t, 128);
        fence_proxy_async_smem();
        mbar_arrive(bar(C::B_KC + ks));
        // V(n): staged [64 keys][D] (swizzled rows of 32 values) -> transposed high and low
        // parts [D][64 keys] in two K-major blocks of 32 keys.  Lane = key within a 32-key half;
        // for a fixed column the 32 lanes write one 128-byte row (no bank conflicts).
        const int vr = n % NVR, vs = n % NV;
        ok = mbar_wait(bar(C::B_VRF + vr), (n / NVR) & 1, abort_flag, p.err);
        if (ok && n >= NV) ok = mbar_wait(bar(C::B_VTE + vs), ((n / NV) - 1) & 1, abort_flag, p.err);
        if (!ok) break;
        const uint32_t src = sVR + vr * C::KV_BYTES, dh = sVT + vs * 2 * C::KV_BYTES, dl = dh + C::KV_BYTES;
        // (kh, column chunk cc of 4 values): 2 x D/4 items over 4 warps
        for (int item = wl; item < 2 * (D / 4); item += 4) {
          const int kh = item / (D / 4), cc = item % (D / 4);
          const int key = 32 * kh + lane;
          const uint32_t a = src + (cc >> 3) * C::KVBLK + key * 128 + (((cc & 7) ^ (key & 7)) << 4);
          uint32_t x[4];
          lds_v4(a, x[0], x[1], x[2], x[3]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int d = 4 * cc + e;
            uint32_t h, l;
            split_tf32(x[e], h, l);
            const uint32_t o = kh * C::VTBLK + d * 128 + ((((lane >> 2) ^ (d & 7))) << 4) + (lane & 3) * 4;
            sts_u32(dh + o, h);
            sts_u32(dl + o, l);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(C::B_VRE + vr));  // the staging slot may be refilled
        mbar_arrive(bar(C::B_VTF + vs));
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax / epilogue
    const int quarter = warp & 3;
    const int r = 32 * quarter + lane;
    const int i = row0 + r;  // sequence-local query row
    const bool row_ok = i < sq.q_len;
    const int off = sq.kv_len - sq.q_len;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16);
    const float sl2 = p.scale_log2;
    const float *brow = nullptr;
    if (BIAS && row_ok) {
      const int bh = p.bias_heads == 1 ? 0 : head;
      brow = p.bias + ((size_t)(sq.q0 + i) * (size_t)p.bias_heads + (size_t)bh) * (size_t)p.max_kv;
    }
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = lo; j < hi; ++j) {
      const int n = j - lo, b = n & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_S + b), (n >> 1) & 1, abort_flag, p.err));
      if (!ok) break;
      fence_after();
      const uint32_t sb = lane_addr + C::S_COL + 128 * b;
      const int kb = j * kBN;
      const bool plain = !BIAS && row_ok && (kb + kBN - 1 < sq.kv_len) &&
                         (!p.causal || kb + kBN - 1 <= i + off) &&
                         (p.window <= 0 || kb >= i + off - p.window + 1);
      uint32_t v[kBN];
      __syncwarp();
      tmem_ld32_at(sb + 0, v, 0);
      tmem_ld32_at(sb + 32, v, 32);
      tmem_ld_wait();
      // row max of the base-2 logits; plain tiles keep raw q.k in v (the scale goes into the
      // exponent FMA), others get v = scale*log2e*q.k + log2e*bias, or -inf where masked
      float mx = -INFINITY;
      if (plain) {
#pragma unroll
        for (int e = 0; e < kBN; ++e) mx = fmaxf(mx, __uint_as_float(v[e]));
        mx *= sl2;
      } else {
        int vlo, vhi;
        visible_range(i, off, sq.kv_len, p.causal, p.window, vlo, vhi);
        if (!row_ok) vhi = vlo;
        const int elo = vlo - kb, ehi = vhi - kb;
#pragma unroll
        for (int e = 0; e < kBN; ++e) {
          float x = __uint_as_float(v[e]) * sl2;
          if (BIAS && brow) x = fmaf(__ldg(brow + min(kb + e, sq.kv_len - 1)), kLog2e, x);
          x = (e >= elo && e < ehi) ? x : -INFINITY;
          v[e] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      }
      // move the reference max only when the row max exceeds it by more than the threshold
      const float m_new = fmaxf(m_ref, mx);
      float alpha = 1.f;
      bool move = false;
      if (m_new != -INFINITY && m_new > m_ref + kRescaleThreshold) {
        alpha = ex2(m_ref - m_new);  // m_ref == -inf -> 0
        move = true;
      }
      const bool need = move && n > 0 && l > 0.f;
      if (__any_sync(0xffffffffu, need)) {
        // rescale O once the previous P.V (and so every earlier one) has completed
        const int np = n - 1;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_O + (np & 1)), (np >> 1) & 1, abort_flag, p.err));
        if (!ok) break;
        fence_after();
        const float a = need ? alpha : 1.f;
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(lane_addr + ch * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
          tmem_st32(lane_addr + ch * 32, o);
        }
      }
      if (move) {
        l *= alpha;
        m_ref = m_new;
      }
      // P = 2^(logit2 - m_ref) in fp32 (a row still without a visible key has every logit at
      // -inf and m_ref = -inf: offset 0, P = 0); its tf32 high parts over S, low parts beside
      const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
      const float sc = plain ? sl2 : 1.f;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int ch = 0; ch < kBN / 32; ++ch) {
        uint32_t ph[32], pl[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float pe = ex2(fmaf(__uint_as_float(v[32 * ch + e]), sc, neg_m));
          if (e & 1) s1 += pe; else s0 += pe;
          split_tf32(__float_as_uint(pe), ph[e], pl[e]);
        }
        __syncwarp();
        tmem_st32(sb + 32 * ch, ph);
        tmem_st32(sb + C::PL_OFF + 32 * ch, pl);
      }
      l += s0 + s1;
      __syncwarp();
      tmem_st_wait();
      fence_before();
      mbar_arrive(bar(C::B_P + b));
    }
    // epilogue: O / l (fp32), LSE in natural log
    const int nt = hi - lo;
    if (ok && nt > 0) {
      const int np = nt - 1;
      ok = mbar_wait(bar(C::B_O + (np & 1)), (np >> 1) & 1, abort_flag, p.err);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const size_t grow = (size_t)sq.q0 + (size_t)(row_ok ? i : 0);
      float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + (grow * p.h_q + head) * D);
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        if (nt > 0) {
          __syncwarp();
          tmem_ld32(lane_addr + ch * 32, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (row_ok) {
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            dst[ch * 8 + q4] = make_float4(__uint_as_float(o[4 * q4]) * inv, __uint_as_float(o[4 * q4 + 1]) * inv,
                                           __uint_as_float(o[4 * q4 + 2]) * inv, __uint_as_float(o[4 * q4 + 3]) * inv);
        }
      }
      if (row_ok && p.lse)
        p.lse[(size_t)head * p.total_q + grow] = l > 0.f ? (m_ref + lg2(l)) * kLn2 : -INFINITY;
    }
  }

  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, int NK, int NVR, int NV>
cudaError_t launch_fwd32(const Params &p, cudaStream_t st) {
  using C = F32Cfg<D, NK, NVR, NV>;
  Fwd32Maps maps;
  if (!make_tmap_f32(&maps.q, p.q, p.total_q, (uint64_t)p.h_q * D, (uint64_t)p.h_q * D, 128) ||
      !make_tmap_f32(&maps.k, p.k, p.total_kv, (uint64_t)p.h_kv * D, (uint64_t)p.h_kv * D, kBN) ||
      !make_tmap_f32(&maps.v, p.v, p.total_kv, (uint64_t)p.h_kv * D, (uint64_t)p.h_kv * D, kBN))
    return cudaErrorInvalidValue;
  const unsigned blocks = (unsigned)((p.max_q + 127) / 128);
  if (blocks == 0) return cudaSuccess;
  const dim3 grid(blocks, (unsigned)p.h_q, (unsigned)p.num_seqs);
  void (*kern)(const Fwd32Maps, const Params) =
      p.bias ? tc_fwd32_kernel<D, NK, NVR, NV, 1> : tc_fwd32_kernel<D, NK, NVR, NV, 0>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, C::THREADS, C::SMEM, st>>>(maps, p);
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace

bool tc_forward32_supported(const Params &p) {
  return p.dtype == VLF_F32 && p.d_qk == p.d_v && (p.d_qk == 32 || p.d_qk == 64);
}

cudaError_t tc_forward32(const Params &p, cudaStream_t st) {
  if (p.total_q == 0 || p.total_kv == 0) return simt_forward(p, st);  // nothing to stage
  if (p.d_qk == 32) return launch_fwd32<32, 3, 2, 3>(p, st);
  return launch_fwd32<64, 2, 2, 2>(p, st);
}

}  // namespace vlf
