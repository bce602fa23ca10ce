// Tensor-core backward for fp32 inputs (sm_103a): the products in three tf32 passes.
//
// The FlashAttention-2 backward of tc_bwd.cu (triton-msl part 2, "Beyond softmax": S recomputed
// per tile, P = exp(S - LSE), dV += P^T dO, dP = dO V^T, dS = P o (dP - D), dK += dS^T Q,
// dQ += dS K; a dK/dV kernel and a dQ kernel, no atomics) for fp32 data, every product taken as
// a_hi b_lo + a_lo b_hi + a_hi b_hi in tf32 with fp32 accumulation (x_hi = x rounded to tf32,
// x_lo = (x - x_hi) rounded to tf32; see tc_fwd32.cu).  One body serves both kernels:
//   dK/dV (KEYS): a CTA owns 128 keys of one kv head; K and V stay resident as the A operands of
//          S^T = K Q^T and dP^T = V dO^T (high parts in TMEM, low parts in shared memory); it
//          walks the 32-row query items of every query head of its GQA group in the key tile's
//          query band.
//   dQ:    a CTA owns 128 query rows of one head; Q and dO (both parts) stay in TMEM as the A
//          operands of S = Q K^T and dP = dO V^T; it walks the 32-key items of its KV band.
// The accumulations take the large product (hi hi) into one accumulator and the two small ones
// into a second, added once at the end: the tensor core rounds its fp32 accumulator at every
// step, and over a long chain (hundreds of steps for dV / dK) those roundings add up -- with a
// single accumulator a 600-row GQA case missed the fp32 gate on dV by half again; with the
// large terms alone in the long chain it is a third as long.
// 320 threads: warp 0 TMA (outer tile once, items through a ring, with the items' -LSE / -D
// pairs for dK/dV); warp 1 all MMAs (and the TMEM allocation); warps 2-5 split operands (the
// outer tile into TMEM once; per item the natural high / low parts in shared memory, K-major along
// the head dimension, and the transposed ones, K-major along the item's rows, that the
// accumulations take as B); warps 6-9 form P and dS (thread = TMEM lane = outer row), writing
// their high parts over S / dP in TMEM and their low parts beside them.  S / dP are single
// buffered: the products of item n + 1 wait for the accumulations of item n.
// Every wait is bounded (tc_common.cuh); on a timeout the CTA records VLF_ERR_TIMEOUT, drains
// and returns.
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

constexpr int kIR = 32;  // inner rows per item (query rows for dK/dV, keys for dQ)

struct Bwd32Maps {
  CUtensorMap outer0, outer1, inner0, inner1;
};

// D: head width (32 or 64).  NS: item ring slots.
template <bool KEYS, int D, int NS>
struct B32Cfg {
  static constexpr int KB = D / 32;                 // 32-column (128-byte) blocks per row
  static constexpr int OBLK = 128 * 128;             // outer tile block: 128 rows x 128 bytes
  static constexpr int IBLK = kIR * 128;             // item block: 32 rows x 128 bytes
  static constexpr int O_BYTES = KB * OBLK;          // one outer tensor's tile
  static constexpr int I_BYTES = KB * IBLK;          // one inner tensor's item (natural layout)
  static constexpr int T_BYTES = D * 128;            // its transpose: D rows x 32 values
  // per slot: inner0 high (landed raw, split in place), inner0 low, inner0^T high / low,
  // inner1 high (in place), inner1 low; dK/dV also inner1^T high / low (dV takes dO^T; dQ takes
  // no V^T)
  static constexpr int N_T = KEYS ? 4 : 2;
  static constexpr int SLOT = 4 * I_BYTES + N_T * T_BYTES;
  static constexpr int OFF_I0 = 0, OFF_I0L = I_BYTES, OFF_I1 = 2 * I_BYTES, OFF_I1L = 3 * I_BYTES;
  static constexpr int OFF_I0T = 4 * I_BYTES, OFF_I1T = OFF_I0T + 2 * T_BYTES;
  static constexpr int OFF_OUT = 0;                         // outer tiles (landed raw)
  static constexpr int OFF_RING = 2 * O_BYTES;
  static constexpr int OFF_LD = OFF_RING + NS * SLOT;       // dK/dV: per slot 32 x {-LSE2, -D}
  static constexpr int OFF_BAR = OFF_LD + NS * kIR * 8;
  // barriers: out_full, outc (outer tile in TMEM), in_full[NS], inc[NS] (item split),
  // in_empty[NS], s_full, p_ready, acc_done, drain
  static constexpr int B_OUT = 0, B_OUTC = 1, B_IF = 2, B_IC = B_IF + NS, B_IE = B_IC + NS;
  static constexpr int B_S = B_IE + NS, B_P = B_S + 1, B_ACC = B_P + 1, B_DRAIN = B_ACC + 1;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16;
  static constexpr int THREADS = 320;
  // TMEM columns.  dK/dV: K high, V high (A operands; their low parts stay in shared memory
  // where TMA left the tiles), dV, dK, their small-product accumulators; dQ: Q high / low, dO
  // high / low, dQ, its small-product accumulator.  Then S (P high over it), P low, dP (dS high
  // over it), dS low (dQ: S holds dS high).
  static constexpr uint32_t O0H = 0, O1H = KEYS ? D : 2 * D;
  static constexpr uint32_t O0L = KEYS ? 0 : D, O1L = KEYS ? 0 : 3 * D;  // (dQ only)
  static constexpr uint32_t ACC0 = KEYS ? 2 * D : 4 * D, ACC1 = ACC0 + D;  // dV, dK or dQ
  static constexpr uint32_t ACC0S = KEYS ? 4 * D : 5 * D, ACC1S = ACC0S + D;
  static constexpr uint32_t SC = 6 * D;
  static constexpr uint32_t PL = SC + kIR, DP = SC + 2 * kIR, DSL = SC + 3 * kIR;
  static_assert(D == 32 || D == 64, "head widths with an fp32 tensor-core backward");
  static_assert(DSL + kIR <= 512, "TMEM columns");
  static_assert(SMEM <= 232448, "shared memory");
};

__device__ __forceinline__ void split_tf32(uint32_t x, uint32_t &hi, uint32_t &lo) {
  const float f = __uint_as_float(x);
  const float h = tf32_round(f);
  hi = __float_as_uint(h);
  lo = __float_as_uint(tf32_round(__fsub_rn(f, h)));
}
__device__ __forceinline__ void sts_u32(uint32_t a, uint32_t x) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(x) : "memory");
}

// The item at `src` ([32 rows][D], swizzled 32-column blocks as TMA left it): split in place
// into its high parts, the low parts at `lo` (same layout), and -- with TRANSPOSE -- the
// transposed high / low parts at th / tl ([D][32 rows], one 128-byte swizzled row per column).
// 128 threads; thread t takes row t mod 32 and the column chunks t / 32, t / 32 + 4, ...
template <int D, bool TRANSPOSE>
__device__ __forceinline__ void split_item(uint32_t src, uint32_t lo, uint32_t th, uint32_t tl, int t) {
  constexpr int IBLK = kIR * 128;
  const int row = t & 31;
#pragma unroll
  for (int cc = t >> 5; cc < D / 4; cc += 4) {  // 16-byte chunk cc: columns 4 cc .. 4 cc + 3
    const uint32_t off = (cc >> 3) * IBLK + row * 128 + (((cc & 7) ^ (row & 7)) << 4);
    uint32_t x[4], h[4], l[4];
    lds_v4(src + off, x[0], x[1], x[2], x[3]);
#pragma unroll
    for (int e = 0; e < 4; ++e) split_tf32(x[e], h[e], l[e]);
    sts_v4(src + off, h[0], h[1], h[2], h[3]);
    sts_v4(lo + off, l[0], l[1], l[2], l[3]);
    if (TRANSPOSE) {
      // column d = 4 cc + e, value `row`: one 128-byte row per column, 16-byte chunk row / 4
      // swizzled by d mod 8 (the 32 lanes of a warp write one row: no bank conflicts)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int d = 4 * cc + e;
        const uint32_t o = d * 128 + ((((row >> 2) ^ (d & 7))) << 4) + (row & 3) * 4;
        sts_u32(th + o, h[e]);
        sts_u32(tl + o, l[e]);
      }
    }
  }
}

template <bool KEYS, int D, int NS, int BIAS>
__global__ void __launch_bounds__(320, 1)
tc_bwd32_kernel(const __grid_constant__ Bwd32Maps maps, const Params p) {
  using C = B32Cfg<KEYS, D, NS>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Seq sq;
  if (!load_seq(p, (int)blockIdx.z, sq)) return;
  const int off = sq.kv_len - sq.q_len;
  int tile0, head_outer, hk, n_items, lo = 0, nq_tiles = 0;
  if (KEYS) {
    tile0 = (int)blockIdx.x * 128;
    hk = head_outer = (int)blockIdx.y;
    if (tile0 >= sq.kv_len) return;
    int qlo = 0, qhi = 0;
    if (sq.q_len > 0) {
      q_band(tile0, min(tile0 + 128, sq.kv_len), sq.q_len, sq.kv_len, p.causal, p.window, qlo, qhi);
      if (p.flags & VLF_FLAG_NO_SKIP) { qlo = 0; qhi = sq.q_len; }
    }
    lo = (qlo / kIR) * kIR;
    nq_tiles = qhi > qlo ? (qhi - lo + kIR - 1) / kIR : 0;
    n_items = nq_tiles * p.group;
  } else {
    const int bx = p.causal ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x;
    tile0 = bx * 128;
    head_outer = (int)blockIdx.y;
    hk = head_outer / p.group;
    if (tile0 >= sq.q_len) return;
    int klo = 0, khi = 0;
    if (sq.kv_len > 0) {
      kv_band(tile0, min(tile0 + 128, sq.q_len), sq.q_len, sq.kv_len, p.causal, p.window, klo, khi);
      if (p.flags & VLF_FLAG_NO_SKIP) { klo = 0; khi = sq.kv_len; }
    }
    lo = (klo / kIR) * kIR;
    n_items = khi > klo ? (khi - lo + kIR - 1) / kIR : 0;
  }
  // item n: (query head, first inner row); inner rows are query rows (dK/dV) or keys (dQ)
  auto item_head = [&](int n) { return KEYS ? hk * p.group + n / nq_tiles : head_outer; };
  auto item_row = [&](int n) { return KEYS ? lo + (n % nq_tiles) * kIR : lo + n * kIR; };

  const uint32_t base = smem_u32(smem_raw);
  if (base & 1023u) {
    if (threadIdx.x == 0) set_error(p.err, VLF_ERR_ALIGN);
    return;
  }
  const uint32_t sOut = base + C::OFF_OUT, sRing = base + C::OFF_RING;
  float2 *ldbuf = reinterpret_cast<float2 *>(smem_raw + C::OFF_LD);  // [slot][32 rows]
  const uint32_t bar0 = base + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem_raw + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem_raw + C::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_OUT), 1);
    mbar_init(bar(C::B_OUTC), 128);
    for (int i = 0; i < NS; ++i) {
      mbar_init(bar(C::B_IF + i), 33);  // lane 0's expect_tx + every producer lane's LSE / D
      mbar_init(bar(C::B_IC + i), 128);
      mbar_init(bar(C::B_IE + i), 1);
    }
    mbar_init(bar(C::B_S), 1);
    mbar_init(bar(C::B_P), 128);
    mbar_init(bar(C::B_ACC), 1);
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_holder;
  auto slot = [&](int n) { return sRing + (n % NS) * C::SLOT; };

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (n_items > 0) {
      if (lane == 0) {
        tma_prefetch_desc(&maps.outer0);
        tma_prefetch_desc(&maps.outer1);
        tma_prefetch_desc(&maps.inner0);
        tma_prefetch_desc(&maps.inner1);
        const int orow = (KEYS ? sq.k0 : sq.q0) + tile0;
        const int oh = KEYS ? hk : head_outer;
        mbar_expect_tx(bar(C::B_OUT), 2 * C::O_BYTES);
        for (int c = 0; c < C::KB; ++c) {
          tma_load_2d(sOut + c * C::OBLK, &maps.outer0, oh * D + 32 * c, orow, bar(C::B_OUT));
          tma_load_2d(sOut + C::O_BYTES + c * C::OBLK, &maps.outer1, oh * D + 32 * c, orow, bar(C::B_OUT));
        }
      }
      int issued[NS] = {0};
      for (int n = 0; n < n_items; ++n) {
        const int st = n % NS;
        bool w = true;
        if (lane == 0 && n >= NS) w = mbar_wait(bar(C::B_IE + st), ((n / NS) - 1) & 1, abort_flag, p.err);
        if (!__shfl_sync(0xffffffffu, (int)w, 0)) break;
        const int h = item_head(n), ir = item_row(n);
        if (KEYS) {
          // -LSE (base 2; -inf for rows past the sequence or seeing nothing: P = 0) and -D of
          // the item's rows, one per lane
          const int qi = ir + lane;
          float nl = -INFINITY, nd = 0.f;
          if (qi < sq.q_len) {
            const size_t gi = (size_t)h * p.total_q + sq.q0 + qi;
            const float L = __ldg(p.lse + gi);
            nl = L == -INFINITY ? -INFINITY : -L * kLog2e;
            nd = -__ldg(p.rowdot + gi);
          }
          ldbuf[st * kIR + lane] = make_float2(nl, nd);
        }
        if (lane == 0) {
          const int ih = KEYS ? h : hk;  // head inside the inner tensors
          const int irow = (KEYS ? sq.q0 : sq.k0) + ir;
          const uint32_t sl = slot(n);
          mbar_expect_tx(bar(C::B_IF + st), 2 * C::I_BYTES);
          for (int c = 0; c < C::KB; ++c) {
            tma_load_2d(sl + C::OFF_I0 + c * C::IBLK, &maps.inner0, ih * D + 32 * c, irow, bar(C::B_IF + st));
            tma_load_2d(sl + C::OFF_I1 + c * C::IBLK, &maps.inner1, ih * D + 32 * c, irow, bar(C::B_IF + st));
          }
          ++issued[st];
        }
        mbar_arrive(bar(C::B_IF + st));
      }
      if (lane == 0) {
        drain_wait(bar(C::B_OUT), 0);
        for (int i = 0; i < NS; ++i)
          if (issued[i]) drain_wait(bar(C::B_IF + i), (issued[i] - 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (n_items > 0) {
      auto wait_all = [&](int b, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar(b), parity, abort_flag, p.err));
      };
      const uint32_t id_sp = idesc_tf32(128, kIR), id_acc = idesc_tf32(128, D);
      bool ok = wait_all(C::B_OUTC, 0);
      for (int n = 0; n < n_items && ok; ++n) {
        const int st = n % NS;
        ok = wait_all(C::B_IC + st, (n / NS) & 1);
        // S / dP of this item overwrite the P / dS the previous item's accumulations read
        if (ok && n > 0) ok = wait_all(C::B_ACC, (n - 1) & 1);
        if (!ok) break;
        fence_after();
        const uint32_t sl = slot(n);
        // S (dK/dV: S^T) = outer0 inner0^T and dP (dP^T) = outer1 inner1^T, A from TMEM
        const uint64_t d_i0h = sdesc_sw128(sl + C::OFF_I0, 16, 1024), d_i0l = sdesc_sw128(sl + C::OFF_I0L, 16, 1024);
        const uint64_t d_i1h = sdesc_sw128(sl + C::OFF_I1, 16, 1024), d_i1l = sdesc_sw128(sl + C::OFF_I1L, 16, 1024);
        // (dK/dV: the outer tiles' low parts are A operands in shared memory)
        const uint64_t d_o0l = sdesc_sw128(sOut, 16, 1024), d_o1l = sdesc_sw128(sOut + C::O_BYTES, 16, 1024);
#pragma unroll
        for (int part = 0; part < 3; ++part) {
          const uint64_t b0 = part == 0 ? d_i0l : d_i0h, b1 = part == 0 ? d_i1l : d_i1h;
#pragma unroll
          for (int kk = 0; kk < D / 8; ++kk) {
            const uint64_t o = (uint64_t)(((kk >> 2) * C::IBLK + (kk & 3) * 32) >> 4);
            const uint32_t acc = (part > 0 || kk > 0) ? 1u : 0u;
            if (KEYS && part == 1) {
              const uint64_t oa = (uint64_t)(((kk >> 2) * C::OBLK + (kk & 3) * 32) >> 4);
              mma_ss_tf32_w(tmem + C::SC, d_o0l + oa, b0 + o, id_sp, acc);
              mma_ss_tf32_w(tmem + C::DP, d_o1l + oa, b1 + o, id_sp, acc);
            } else {
              const uint32_t a0 = tmem + (part == 1 ? C::O0L : C::O0H), a1 = tmem + (part == 1 ? C::O1L : C::O1H);
              mma_ts_tf32_w(tmem + C::SC, a0 + 8 * kk, b0 + o, id_sp, acc);
              mma_ts_tf32_w(tmem + C::DP, a1 + 8 * kk, b1 + o, id_sp, acc);
            }
          }
        }
        mma_commit_w(bar(C::B_S));
        ok = wait_all(C::B_P, n & 1);
        if (!ok) break;
        fence_after();
        // accumulations, A from TMEM (P / dS high and low parts), B the transposed items:
        // dK/dV: dV += P^T dO, dK += dS^T Q; dQ: dQ += dS K
        const uint64_t d_t0h = sdesc_sw128(sl + C::OFF_I0T, 16, 1024);
        const uint64_t d_t0l = sdesc_sw128(sl + C::OFF_I0T + C::T_BYTES, 16, 1024);
        const uint64_t d_t1h = sdesc_sw128(sl + C::OFF_I1T, 16, 1024);
        const uint64_t d_t1l = sdesc_sw128(sl + C::OFF_I1T + C::T_BYTES, 16, 1024);
        const uint32_t dsh = KEYS ? C::DP : C::SC;  // where dS's high parts are
        // part 0: lo hi and part 1: hi lo into the small-product accumulators, part 2: hi hi
#pragma unroll
        for (int part = 0; part < 3; ++part) {
#pragma unroll
          for (int kk = 0; kk < kIR / 8; ++kk) {
            const uint64_t o = (uint64_t)(((kk & 3) * 32) >> 4);
            const uint32_t acc = (n > 0 || part == 1 || kk > 0) ? 1u : 0u;
            if (KEYS) {
              const uint32_t ap = tmem + (part == 0 ? C::PL : C::SC) + 8 * kk;
              mma_ts_tf32_w(tmem + (part == 2 ? C::ACC0 : C::ACC0S), ap, (part == 1 ? d_t1l : d_t1h) + o,
                            id_acc, acc);
            }
            const uint32_t as = tmem + (part == 0 ? C::DSL : dsh) + 8 * kk;
            const uint32_t ad = KEYS ? (part == 2 ? C::ACC1 : C::ACC1S) : (part == 2 ? C::ACC0 : C::ACC0S);
            mma_ts_tf32_w(tmem + ad, as, (part == 1 ? d_t0l : d_t0h) + o, id_acc, acc);
          }
        }
        mma_commit_w(bar(C::B_ACC));
        mma_commit_w(bar(C::B_IE + st));  // the item's slot may be refilled
      }
      mma_commit_w(bar(C::B_DRAIN));
      drain_wait(bar(C::B_DRAIN), 0);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------------ operand splitting
    const int t = threadIdx.x - 64;          // 0 .. 127
    const int r = 32 * (warp & 3) + lane;    // TMEM lane = outer row
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    if (n_items > 0) {
      bool ok = mbar_wait(bar(C::B_OUT), 0, abort_flag, p.err);
      if (ok) {
        // this thread's row of both outer tiles -> high / low parts in TMEM (A operands)
#pragma unroll
        for (int o = 0; o < 2; ++o) {
#pragma unroll
          for (int half = 0; half < D / 32; ++half) {
            uint32_t h[32], l[32];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint32_t a = sOut + o * C::O_BYTES + half * C::OBLK + r * 128 + ((q ^ (r & 7)) << 4);
              uint32_t x[4];
              lds_v4(a, x[0], x[1], x[2], x[3]);
#pragma unroll
              for (int e = 0; e < 4; ++e) split_tf32(x[e], h[4 * q + e], l[4 * q + e]);
            }
            __syncwarp();
            tmem_st32(lane_addr + (o ? C::O1H : C::O0H) + 32 * half, h);
            if (KEYS) {
              // the low parts go back where the row was, as the shared-memory A operand
#pragma unroll
              for (int q = 0; q < 8; ++q)
                sts_v4(sOut + o * C::O_BYTES + half * C::OBLK + r * 128 + ((q ^ (r & 7)) << 4), l[4 * q],
                       l[4 * q + 1], l[4 * q + 2], l[4 * q + 3]);
            } else {
              tmem_st32(lane_addr + (o ? C::O1L : C::O0L) + 32 * half, l);
            }
          }
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        fence_before();
        mbar_arrive(bar(C::B_OUTC));
      }
      for (int n = 0; n < n_items && ok; ++n) {
        const int st = n % NS;
        ok = mbar_wait(bar(C::B_IF + st), (n / NS) & 1, abort_flag, p.err);
        if (!ok) break;
        const uint32_t sl = slot(n);
        // inner0 (Q, dK/dV; K, dQ) natural and transposed; inner1 (dO; V) natural, and
        // transposed for dK/dV
        split_item<D, true>(sl + C::OFF_I0, sl + C::OFF_I0L, sl + C::OFF_I0T,
                            sl + C::OFF_I0T + C::T_BYTES, t);
        split_item<D, KEYS>(sl + C::OFF_I1, sl + C::OFF_I1L, sl + C::OFF_I1T,
                            sl + C::OFF_I1T + C::T_BYTES, t);
        fence_proxy_async_smem();  // generic-proxy writes, read next by the tensor core
        mbar_arrive(bar(C::B_IC + st));
      }
    }
  } else {
    // ------------------------------------------------------------------ P, dS and the epilogue
    const int r = 32 * (warp & 3) + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const float sl2 = p.scale_log2;
    const int orow = tile0 + r;
    const bool orow_ok = KEYS ? orow < sq.kv_len : orow < sq.q_len;
    int vis_lo, vis_hi;  // the columns this row may see: query rows (dK/dV) or keys (dQ)
    if (KEYS) visible_rows(orow, off, sq.q_len, p.causal, p.window, vis_lo, vis_hi);
    else visible_range(orow, off, sq.kv_len, p.causal, p.window, vis_lo, vis_hi);
    if (!orow_ok) vis_hi = vis_lo;
    float row_nl = -INFINITY, row_nd = 0.f;
    const float *brow = nullptr;
    if (!KEYS && orow_ok) {
      const size_t gi = (size_t)head_outer * p.total_q + sq.q0 + orow;
      const float L = p.lse[gi];
      row_nl = L == -INFINITY ? -INFINITY : -L * kLog2e;
      row_nd = -p.rowdot[gi];
      if (BIAS) {
        const int bh = p.bias_heads == 1 ? 0 : head_outer;
        brow = p.bias + ((size_t)(sq.q0 + orow) * p.bias_heads + bh) * (size_t)p.max_kv;
      }
    }
    bool ok = true;
    for (int n = 0; n < n_items && ok; ++n) {
      const int st = n % NS, h = item_head(n), i0 = item_row(n);
      bool w = mbar_wait(bar(C::B_S), n & 1, abort_flag, p.err);
      // the LSE / D pairs were written by the producer lanes before their arrive on in_full
      if (KEYS && w) w = mbar_wait(bar(C::B_IF + st), (n / NS) & 1, abort_flag, p.err);
      ok = __all_sync(0xffffffffu, w);
      if (!ok) break;
      fence_after();
      uint32_t sv[kIR], dv[kIR];
      __syncwarp();
      tmem_ld32(lane_addr + C::SC, sv);
      tmem_ld32(lane_addr + C::DP, dv);
      tmem_ld_wait();
      if (KEYS && BIAS && orow_ok) {
        const int bh = p.bias_heads == 1 ? 0 : h;
        brow = p.bias + (size_t)bh * p.max_kv + orow;  // + (q0 + i) * bias_heads * max_kv per row
      }
      // 16 columns at a time (register pressure): P and dS, their high / low parts to TMEM
#pragma unroll
      for (int hc = 0; hc < kIR / 16; ++hc) {
        uint32_t ph[16], pl[16], dh[16], dl[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c = 16 * hc + e;
          const int cc = i0 + c;  // sequence-local column: query row (dK/dV) or key (dQ)
          float nl, nd;
          if (KEYS) {
            const float2 q = ldbuf[st * kIR + c];
            nl = q.x;
            nd = q.y;
          } else {
            nl = row_nl;
            nd = row_nd;
          }
          float x = __uint_as_float(sv[c]) * sl2;
          if (BIAS && brow) {
            // clamped into the sequence so that masked columns read a valid address
            const float bv = KEYS ? __ldg(brow + (size_t)(sq.q0 + min(cc, sq.q_len - 1)) * p.bias_heads * (size_t)p.max_kv)
                                  : __ldg(brow + min(cc, sq.kv_len - 1));
            x = fmaf(bv, kLog2e, x);
          }
          x = (cc >= vis_lo && cc < vis_hi) ? x : -INFINITY;
          const float pe = ex2(x + nl);  // masked (-inf) and rows without keys (nl = -inf): 0
          const float ds = pe * (__uint_as_float(dv[c]) + nd);
          split_tf32(__float_as_uint(pe), ph[e], pl[e]);
          split_tf32(__float_as_uint(ds), dh[e], dl[e]);
        }
        __syncwarp();
        if (KEYS) {
          tmem_st16(lane_addr + C::SC + 16 * hc, ph);
          tmem_st16(lane_addr + C::PL + 16 * hc, pl);
          tmem_st16(lane_addr + C::DP + 16 * hc, dh);
          tmem_st16(lane_addr + C::DSL + 16 * hc, dl);
        } else {
          tmem_st16(lane_addr + C::SC + 16 * hc, dh);  // dQ: dS high over S, its low parts at DSL
          tmem_st16(lane_addr + C::DSL + 16 * hc, dl);
        }
      }
      tmem_st_wait();
      fence_before();
      mbar_arrive(bar(C::B_P));
    }
    // epilogue: the last item's accumulations complete every MMA of the CTA
    if (ok && n_items > 0) ok = mbar_wait(bar(C::B_ACC), (n_items - 1) & 1, abort_flag, p.err);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      fence_after();
      const size_t g = (size_t)((KEYS ? sq.k0 : sq.q0) + (orow_ok ? orow : 0));
      // the large-product accumulator plus the small-product one, times mul
      auto store = [&](uint32_t col, uint32_t col_s, float *dst, float mul) {
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t v[32], w[32];
          if (n_items > 0) {  // (every lane of the warp loads; rows past the sequence store nothing)
            __syncwarp();
            tmem_ld32(lane_addr + col + 32 * ch, v);
            tmem_ld32(lane_addr + col_s + 32 * ch, w);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) + __uint_as_float(w[e]));
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          }
          if (!orow_ok) continue;
          float4 *d4 = reinterpret_cast<float4 *>(dst + 32 * ch);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            d4[q] = make_float4(__uint_as_float(v[4 * q]) * mul, __uint_as_float(v[4 * q + 1]) * mul,
                                __uint_as_float(v[4 * q + 2]) * mul, __uint_as_float(v[4 * q + 3]) * mul);
        }
      };
      if (KEYS) {
        store(C::ACC0, C::ACC0S, static_cast<float *>(p.dv) + (g * p.h_kv + hk) * D, 1.f);
        store(C::ACC1, C::ACC1S, static_cast<float *>(p.dk) + (g * p.h_kv + hk) * D, p.scale);
      } else {
        store(C::ACC0, C::ACC0S, static_cast<float *>(p.dq) + (g * p.h_q + head_outer) * D, p.scale);
      }
    }
  }

  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool KEYS, int D, int NS>
cudaError_t launch_bwd32(const Params &p, cudaStream_t st) {
  using C = B32Cfg<KEYS, D, NS>;
  Bwd32Maps m;
  const uint64_t qc = (uint64_t)p.h_q * D, kc = (uint64_t)p.h_kv * D;
  bool ok;
  if (KEYS)
    ok = make_tmap_f32(&m.outer0, p.k, p.total_kv, kc, kc, 128) &&
         make_tmap_f32(&m.outer1, p.v, p.total_kv, kc, kc, 128) &&
         make_tmap_f32(&m.inner0, p.q, p.total_q, qc, qc, kIR) &&
         make_tmap_f32(&m.inner1, p.dout, p.total_q, qc, qc, kIR);
  else
    ok = make_tmap_f32(&m.outer0, p.q, p.total_q, qc, qc, 128) &&
         make_tmap_f32(&m.outer1, p.dout, p.total_q, qc, qc, 128) &&
         make_tmap_f32(&m.inner0, p.k, p.total_kv, kc, kc, kIR) &&
         make_tmap_f32(&m.inner1, p.v, p.total_kv, kc, kc, kIR);
  if (!ok) return cudaErrorInvalidValue;
  const unsigned tiles = KEYS ? (p.max_kv + 127) / 128 : (p.max_q + 127) / 128;
  if (tiles == 0) return cudaSuccess;
  const dim3 grid(tiles, KEYS ? p.h_kv : p.h_q, p.num_seqs);
  void (*kern)(const Bwd32Maps, const Params) =
      p.bias ? tc_bwd32_kernel<KEYS, D, NS, 1> : tc_bwd32_kernel<KEYS, D, NS, 0>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, C::THREADS, C::SMEM, st>>>(m, p);
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

template <int D>
cudaError_t bwd32_shape(const Params &p, cudaStream_t st, const cudaEvent_t *ev) {
  cudaError_t e;
  if ((e = mark(ev, 0, st)) != cudaSuccess) return e;
  if ((e = rowdot_forward(p, st)) != cudaSuccess) return e;
  if ((e = mark(ev, 1, st)) != cudaSuccess) return e;
  if ((e = launch_bwd32<true, D, 2>(p, st)) != cudaSuccess) return e;
  if ((e = mark(ev, 2, st)) != cudaSuccess) return e;
  if ((e = launch_bwd32<false, D, 2>(p, st)) != cudaSuccess) return e;
  return mark(ev, 3, st);
}

}  // namespace

bool tc_backward32_supported(const Params &p) {
  return p.dtype == VLF_F32 && p.d_qk == p.d_v && (p.d_qk == 32 || p.d_qk == 64);
}

cudaError_t tc_backward32(const Params &p, cudaStream_t st, const cudaEvent_t *ev) {
  if (p.total_q == 0 || p.total_kv == 0) return simt_backward(p, st, ev);
  if (p.d_qk == 32) return bwd32_shape<32>(p, st, ev);
  return bwd32_shape<64>(p, st, ev);
}

}  // namespace vlf
