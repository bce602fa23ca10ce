// Tensor-core backward (sm_103a): the FlashAttention-2 backward that triton-msl part 2
// ("Beyond softmax") describes -- recompute S per tile, P = exp(S - LSE), dV += P^T dO,
// dP = dO V^T, dS = P o (dP - D) with D = rowsum(dO o O), dK += dS^T Q, dQ += dS K -- split into
// a dK/dV kernel and a dQ kernel so that no output is accumulated with atomics (results are
// deterministic), with tcgen05 MMAs accumulating in TMEM and TMA-staged tiles.
//
// One kernel body serves both (MODE):
//   dK/dV: a CTA owns 128 keys of one kv head (K, V tiles stay in shared memory) and walks the
//          64-row Q / dO tiles of every query head of its GQA group that can see those keys.
//          S^T = K Q^T and dP^T = V dO^T land in TMEM (lanes = keys); the compute warpgroup
//          turns them into 16-bit P^T and dS^T in TMEM; dV += P^T dO and dK += dS^T Q take
//          their A operand from TMEM.  LSE and D of the 64 query columns come through smem.
//   dQ:    a CTA owns 128 query rows of one head (Q, dO stay in shared memory) and walks the
//          64-key K / V tiles of its band: S = Q K^T, dP = dO V^T, dS in TMEM, dQ += dS K.
// Warp roles (192 threads): warp 0 TMA, warp 1 TMEM allocation + MMA issue, warps 2-5 compute
// (one thread per TMEM lane).  S/dP buffers are double-buffered in TMEM where columns allow so
// the next tile's products overlap this tile's elementwise pass.  Tiles outside the causal /
// window band are skipped (they contribute exact zeros).  Every wait is bounded.
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace vlf {

bool make_tmap_16bit(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols,
                     uint64_t pitch_elems, uint32_t box_rows, int is_bf16);

namespace {

using namespace tc;

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kDkdv = 0, kDq = 1;

struct BwdMaps {
  CUtensorMap outer0, outer1, inner0, inner1;
};

// outer0/outer1: K, V (dK/dV) or Q, dO (dQ), 128 rows.  inner0/inner1: Q, dO (dK/dV) or K, V
// (dQ), 64 rows per item.
template <int MODE, int DQK, int DV, int NBUF, int NSTAGE>
struct BwdCfg {
  static constexpr int KB0 = DQK / 64, KB1 = DV / 64;  // 64-col blocks of tensors 0 / 1
  static constexpr int OBLK = 128 * 128, IBLK = 64 * 128;  // bytes per 64-col block
  static constexpr int O0_BYTES = KB0 * OBLK, O1_BYTES = KB1 * OBLK;
  static constexpr int I0_BYTES = KB0 * IBLK, I1_BYTES = KB1 * IBLK;
  static constexpr int STAGE_BYTES = I0_BYTES + I1_BYTES;
  static constexpr int OFF_O0 = 0, OFF_O1 = O0_BYTES, OFF_IN = O0_BYTES + O1_BYTES;
  static constexpr int OFF_LD = OFF_IN + NSTAGE * STAGE_BYTES;  // per-warp LSE / D columns
  static constexpr int OFF_BAR = OFF_LD + 4 * 128 * 4;
  // barriers: outer_full, in_full[NSTAGE], in_empty[NSTAGE], s_full[NBUF], p_ready[NBUF],
  // item_done[NBUF], drain
  static constexpr int B_OUT = 0, B_IF = 1, B_IE = B_IF + NSTAGE, B_S = B_IE + NSTAGE;
  static constexpr int B_P = B_S + NBUF, B_D = B_P + NBUF, B_DRAIN = B_D + NBUF;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  // TMEM: accumulators first, then NBUF x (S 64 cols, dP 64 cols)
  static constexpr uint32_t ACC0 = 0;                           // dV (dK/dV) or dQ (dQ)
  static constexpr uint32_t ACC1 = 128;                         // dK (dK/dV)
  static constexpr uint32_t BUF = MODE == kDkdv ? 128 + DQK : 256;
  static_assert(BUF + NBUF * 128 <= 512, "TMEM columns");
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(DV <= 128 && DQK <= 256 && DQK % 64 == 0 && DV % 64 == 0, "head widths");
};

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > 200000000ull) break;
  }
}

template <int MODE, int DQK, int DV, int NBUF, int NSTAGE>
__global__ void __launch_bounds__(192, 1)
tc_bwd_kernel(const __grid_constant__ BwdMaps maps, const Params p) {
  using C = BwdCfg<MODE, DQK, DV, NBUF, NSTAGE>;
  extern __shared__ uint8_t smem_raw[];
  const int s = blockIdx.z;
  Seq sq;
  if (!load_seq(p, s, sq)) return;
  const int off = sq.kv_len - sq.q_len;
  // the CTA's outer tile and its item range
  int tile0, head_outer, hk, n_items, lo64 = 0, nq_tiles = 0;
  if (MODE == kDkdv) {
    tile0 = blockIdx.x * 128;  // first key
    hk = blockIdx.y;
    head_outer = hk;
    if (tile0 >= sq.kv_len) return;
    int qlo = 0, qhi = 0;
    if (sq.q_len > 0) {
      q_band(tile0, min(tile0 + 128, sq.kv_len), sq.q_len, sq.kv_len, p.causal, p.window, qlo, qhi);
      if (p.flags & VLF_FLAG_NO_SKIP) { qlo = 0; qhi = sq.q_len; }
    }
    lo64 = (qlo / 64) * 64;
    nq_tiles = qhi > qlo ? (qhi - lo64 + 63) / 64 : 0;
    n_items = nq_tiles * p.group;
  } else {
    const int bx = p.causal ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
    tile0 = bx * 128;  // first query row
    head_outer = blockIdx.y;
    hk = head_outer / p.group;
    if (tile0 >= sq.q_len) return;
    int klo = 0, khi = 0;
    if (sq.kv_len > 0) {
      kv_band(tile0, min(tile0 + 128, sq.q_len), sq.q_len, sq.kv_len, p.causal, p.window, klo, khi);
      if (p.flags & VLF_FLAG_NO_SKIP) { klo = 0; khi = sq.kv_len; }
    }
    lo64 = (klo / 64) * 64;
    n_items = khi > klo ? (khi - lo64 + 63) / 64 : 0;
  }

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - raw);
  const uint32_t sO0 = base + C::OFF_O0, sO1 = base + C::OFF_O1, sIn = base + C::OFF_IN;
  float *ldbuf = reinterpret_cast<float *>(gbase + C::OFF_LD);  // [warp][LSE 64 | D 64]
  const uint32_t bar0 = base + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(gbase + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + C::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_OUT), 1);
    for (int i = 0; i < NSTAGE; ++i) { mbar_init(bar(C::B_IF + i), 1); mbar_init(bar(C::B_IE + i), 1); }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(bar(C::B_S + b), 1);
      mbar_init(bar(C::B_P + b), 128);
      mbar_init(bar(C::B_D + b), 1);
    }
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
  const int is_bf16 = p.dtype == VLF_BF16;

  // item n -> (query head, first inner row) ; inner rows are queries (dK/dV) or keys (dQ)
  auto item_head = [&](int n) { return MODE == kDkdv ? hk * p.group + n / nq_tiles : head_outer; };
  auto item_row = [&](int n) { return MODE == kDkdv ? lo64 + (n % nq_tiles) * 64 : lo64 + n * 64; };

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && n_items > 0) {
      tma_prefetch_desc(&maps.outer0);
      tma_prefetch_desc(&maps.outer1);
      tma_prefetch_desc(&maps.inner0);
      tma_prefetch_desc(&maps.inner1);
      const int orow = (MODE == kDkdv ? sq.k0 : sq.q0) + tile0;
      const int oh = MODE == kDkdv ? hk : head_outer;  // head index inside the outer tensors
      mbar_expect_tx(bar(C::B_OUT), C::O0_BYTES + C::O1_BYTES);
      for (int c = 0; c < C::KB0; ++c)
        tma_load_2d(sO0 + c * C::OBLK, &maps.outer0, oh * DQK + 64 * c, orow, bar(C::B_OUT));
      for (int c = 0; c < C::KB1; ++c)
        tma_load_2d(sO1 + c * C::OBLK, &maps.outer1, oh * DV + 64 * c, orow, bar(C::B_OUT));
      int issued[NSTAGE] = {0};
      bool ok = true;
      for (int n = 0; n < n_items && ok; ++n) {
        const int st = n % NSTAGE;
        if (n >= NSTAGE) ok = mbar_wait(bar(C::B_IE + st), ((n / NSTAGE) - 1) & 1, abort_flag, p.err);
        if (!ok) break;
        const int ih = MODE == kDkdv ? item_head(n) : hk;  // head inside the inner tensors
        const int irow = (MODE == kDkdv ? sq.q0 : sq.k0) + item_row(n);
        const uint32_t dst = sIn + st * C::STAGE_BYTES;
        mbar_expect_tx(bar(C::B_IF + st), C::STAGE_BYTES);
        for (int c = 0; c < C::KB0; ++c)
          tma_load_2d(dst + c * C::IBLK, &maps.inner0, ih * DQK + 64 * c, irow, bar(C::B_IF + st));
        for (int c = 0; c < C::KB1; ++c)
          tma_load_2d(dst + C::I0_BYTES + c * C::IBLK, &maps.inner1, ih * DV + 64 * c, irow,
                      bar(C::B_IF + st));
        ++issued[st];
      }
      drain_wait(bar(C::B_OUT), 0);
      for (int i = 0; i < NSTAGE; ++i)
        if (issued[i]) drain_wait(bar(C::B_IF + i), (issued[i] - 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_items > 0) {
      // S / dP: M = 128 outer rows, N = 64 inner rows, both operands K-major
      const uint32_t id_sp = idesc_f16(is_bf16, 128, 64, 0, 0);
      // accumulations: A from TMEM (K = 64 inner rows), B = inner tile MN-major
      const uint32_t id_a0 = idesc_f16(is_bf16, 128, MODE == kDkdv ? DV : DQK, 0, 1);
      const uint32_t id_a1 = idesc_f16(is_bf16, 128, DQK, 0, 1);
      auto issue_sp = [&](int n) {
        const int b = n % NBUF, st = n % NSTAGE;
        const uint32_t in0 = sIn + st * C::STAGE_BYTES, in1 = in0 + C::I0_BYTES;
        const uint32_t s_col = tmem + C::BUF + 128 * b, dp_col = s_col + 64;
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint32_t oa = (kk >> 2) * C::OBLK + (kk & 3) * 32, ia = (kk >> 2) * C::IBLK + (kk & 3) * 32;
          mma_ss(s_col, sdesc_sw128(sO0 + oa, 16, 1024), sdesc_sw128(in0 + ia, 16, 1024), id_sp, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk) {
          const uint32_t oa = (kk >> 2) * C::OBLK + (kk & 3) * 32, ia = (kk >> 2) * C::IBLK + (kk & 3) * 32;
          mma_ss(dp_col, sdesc_sw128(sO1 + oa, 16, 1024), sdesc_sw128(in1 + ia, 16, 1024), id_sp, kk > 0);
        }
        mma_commit(bar(C::B_S + b));
      };
      auto issue_acc = [&](int n) {
        const int b = n % NBUF, st = n % NSTAGE;
        const uint32_t in0 = sIn + st * C::STAGE_BYTES, in1 = in0 + C::I0_BYTES;
        const uint32_t s_col = tmem + C::BUF + 128 * b, dp_col = s_col + 64;
        if (MODE == kDkdv) {
          // dV += P^T dO   (P^T over the first half of S^T; dO MN-major, 64-column blocks 8 KB apart)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + C::ACC0, s_col + kk * 8, sdesc_sw128(in1 + kk * 2048, C::IBLK, 1024), id_a0,
                   (n > 0 || kk > 0) ? 1u : 0u);
          // dK += dS^T Q
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + C::ACC1, dp_col + kk * 8, sdesc_sw128(in0 + kk * 2048, C::IBLK, 1024), id_a1,
                   (n > 0 || kk > 0) ? 1u : 0u);
        } else {
          // dQ += dS K   (K tile MN-major)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + C::ACC0, dp_col + kk * 8, sdesc_sw128(in0 + kk * 2048, C::IBLK, 1024), id_a0,
                   (n > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(C::B_D + b));
        mma_commit(bar(C::B_IE + st));
      };
      bool ok = mbar_wait(bar(C::B_OUT), 0, abort_flag, p.err);
      for (int n = 0; n < NBUF && n < n_items && ok; ++n) {
        ok = mbar_wait(bar(C::B_IF + n % NSTAGE), (n / NSTAGE) & 1, abort_flag, p.err);
        if (!ok) break;
        fence_after();
        issue_sp(n);
      }
      for (int n = 0; n < n_items && ok; ++n) {
        const int b = n % NBUF;
        ok = mbar_wait(bar(C::B_P + b), (n / NBUF) & 1, abort_flag, p.err);
        if (!ok) break;
        fence_after();
        issue_acc(n);
        const int m = n + NBUF;
        if (m < n_items) {
          // the products of item m reuse buffer b: wait until item n's accumulations read it
          ok = mbar_wait(bar(C::B_D + b), (n / NBUF) & 1, abort_flag, p.err) &&
               mbar_wait(bar(C::B_IF + m % NSTAGE), (m / NSTAGE) & 1, abort_flag, p.err);
          if (!ok) break;
          fence_after();
          issue_sp(m);
        }
      }
      mma_commit(bar(C::B_DRAIN));
      drain_wait(bar(C::B_DRAIN), 0);
    }
  } else {
    // ------------------------------------------------------------------ elementwise + epilogue
    const int quarter = warp & 3;
    const int r = 32 * quarter + lane;  // TMEM lane = outer row (key for dK/dV, query for dQ)
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16);
    const float sl2 = p.scale_log2;
    // this thread's outer row
    const int orow = tile0 + r;
    const bool orow_ok = MODE == kDkdv ? orow < sq.kv_len : orow < sq.q_len;
    float row_lse2 = INFINITY, row_d = 0.f;  // dQ: this row's LSE (base 2) and D
    const float *brow_dq = nullptr;
    if (MODE == kDq && orow_ok) {
      const size_t gi = (size_t)head_outer * p.total_q + sq.q0 + orow;
      const float L = p.lse[gi];
      row_lse2 = L == -INFINITY ? INFINITY : L * kLog2e;
      row_d = p.rowdot[gi];
      if (p.bias) {
        const int bh = p.bias_heads == 1 ? 0 : head_outer;
        brow_dq = p.bias + ((size_t)(sq.q0 + orow) * p.bias_heads + bh) * (size_t)p.max_kv;
      }
    }
    bool ok = true;
    for (int n = 0; n < n_items; ++n) {
      const int b = n % NBUF;
      const int h = item_head(n);
      const int i0 = item_row(n);  // first inner row of the item
      float *lsb = ldbuf + quarter * 128;
      if (MODE == kDkdv) {
        // LSE (base 2; +inf for rows that see nothing or lie past the sequence) and D of the
        // item's 64 query columns; each warp keeps its own copy (warp-local sync only)
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int qi = i0 + lane + 32 * u;
          float L2 = INFINITY, Dv = 0.f;
          if (qi < sq.q_len) {
            const size_t gi = (size_t)h * p.total_q + sq.q0 + qi;
            const float L = p.lse[gi];
            L2 = L == -INFINITY ? INFINITY : L * kLog2e;
            Dv = p.rowdot[gi];
          }
          lsb[lane + 32 * u] = L2;
          lsb[64 + lane + 32 * u] = Dv;
        }
        __syncwarp();
      }
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_S + b), (n / NBUF) & 1, abort_flag, p.err));
      if (!ok) break;
      fence_after();
      const uint32_t s_addr = lane_addr + C::BUF + 128 * b, dp_addr = s_addr + 64;
      const float *brow = brow_dq;
      if (MODE == kDkdv && p.bias && orow_ok) {
        const int bh = p.bias_heads == 1 ? 0 : h;
        brow = p.bias + (size_t)bh * p.max_kv + orow;  // + (q0 + i) * bias_heads * max_kv per column
      }
      // is every element of this thread's row of the item visible (no per-element mask)?
      bool plain;
      if (MODE == kDkdv) {
        const int j = orow, ilast = i0 + 63;
        plain = orow_ok && ilast < sq.q_len && (!p.causal || j <= i0 + off) &&
                (p.window <= 0 || j >= ilast + off - p.window + 1);
      } else {
        const int i = orow, jlast = i0 + 63;
        plain = orow_ok && jlast < sq.kv_len && (!p.causal || jlast <= i + off) &&
                (p.window <= 0 || i0 >= i + off - p.window + 1);
      }
      plain = plain && p.bias == nullptr;
#pragma unroll 1
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t sv[32], dv[32];
        __syncwarp();
        tmem_ld32(s_addr + ch * 32, sv);
        tmem_ld32(dp_addr + ch * 32, dv);
        tmem_ld_wait();
        float pr[32], ds[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int col = ch * 32 + e;
          float lse2, dcol;
          if (MODE == kDkdv) { lse2 = lsb[col]; dcol = lsb[64 + col]; }
          else { lse2 = row_lse2; dcol = row_d; }
          float x;
          if (plain) {
            x = __uint_as_float(sv[e]) * sl2;
          } else {
            const int i = MODE == kDkdv ? i0 + col : orow;
            const int j = MODE == kDkdv ? orow : i0 + col;
            x = -INFINITY;
            if (orow_ok && i < sq.q_len && pair_visible(i, j, off, sq.kv_len, p.causal, p.window)) {
              x = __uint_as_float(sv[e]) * sl2;
              if (brow) {
                const float bv = MODE == kDkdv
                                     ? __ldg(brow + (size_t)(sq.q0 + i) * p.bias_heads * (size_t)p.max_kv)
                                     : __ldg(brow + j);
                x = fmaf(bv, kLog2e, x);
              }
            }
          }
          pr[e] = ex2(x - lse2);  // masked (-inf) or dead row (lse2 = +inf) -> 0
          ds[e] = pr[e] * (__uint_as_float(dv[e]) - dcol);
        }
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          pk[e] = pack2(pr[2 * e], pr[2 * e + 1], is_bf16);
          dk[e] = pack2(ds[2 * e], ds[2 * e + 1], is_bf16);
        }
        __syncwarp();
        if (MODE == kDkdv) tmem_st16(s_addr + ch * 16, pk);
        tmem_st16(dp_addr + ch * 16, dk);
      }
      __syncwarp();
      tmem_st_wait();
      fence_before();
      mbar_arrive(bar(C::B_P + b));
    }
    // epilogue
    if (ok && n_items > 0)
      ok = mbar_wait(bar(C::B_D + (n_items - 1) % NBUF), ((n_items - 1) / NBUF) & 1, abort_flag, p.err);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      fence_after();
      auto store_acc = [&](uint32_t col, int width, void *dst_base, int heads, int head, float mul) {
        uint4 *dst = nullptr;
        if (orow_ok) {
          const size_t g = (size_t)((MODE == kDkdv ? sq.k0 : sq.q0) + orow);
          dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(dst_base) +
                                          ((g * heads + head) * (size_t)width) * 2);
        }
#pragma unroll 1
        for (int ch = 0; ch < width / 32; ++ch) {
          uint32_t v[32];
          if (n_items > 0) {
            __syncwarp();
            tmem_ld32(lane_addr + col + ch * 32, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          }
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul, is_bf16);
          if (dst) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              dst[ch * 4 + q4] = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
          }
        }
      };
      if (MODE == kDkdv) {
        store_acc(C::ACC0, DV, p.dv, p.h_kv, hk, 1.f);
        store_acc(C::ACC1, DQK, p.dk, p.h_kv, hk, p.scale);
      } else {
        store_acc(C::ACC0, DQK, p.dq, p.h_q, head_outer, p.scale);
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

template <int MODE, int DQK, int DV, int NBUF, int NSTAGE>
cudaError_t launch_bwd(const Params &p, cudaStream_t st) {
  using C = BwdCfg<MODE, DQK, DV, NBUF, NSTAGE>;
  const int bf = p.dtype == VLF_BF16;
  BwdMaps m;
  const uint64_t tq = p.total_q, tk = p.total_kv;
  bool ok;
  if (MODE == kDkdv) {
    ok = make_tmap_16bit(&m.outer0, p.k, tk, (uint64_t)p.h_kv * DQK, (uint64_t)p.h_kv * DQK, 128, bf) &&
         make_tmap_16bit(&m.outer1, p.v, tk, (uint64_t)p.h_kv * DV, (uint64_t)p.h_kv * DV, 128, bf) &&
         make_tmap_16bit(&m.inner0, p.q, tq, (uint64_t)p.h_q * DQK, (uint64_t)p.h_q * DQK, 64, bf) &&
         make_tmap_16bit(&m.inner1, p.dout, tq, (uint64_t)p.h_q * DV, (uint64_t)p.h_q * DV, 64, bf);
  } else {
    ok = make_tmap_16bit(&m.outer0, p.q, tq, (uint64_t)p.h_q * DQK, (uint64_t)p.h_q * DQK, 128, bf) &&
         make_tmap_16bit(&m.outer1, p.dout, tq, (uint64_t)p.h_q * DV, (uint64_t)p.h_q * DV, 128, bf) &&
         make_tmap_16bit(&m.inner0, p.k, tk, (uint64_t)p.h_kv * DQK, (uint64_t)p.h_kv * DQK, 64, bf) &&
         make_tmap_16bit(&m.inner1, p.v, tk, (uint64_t)p.h_kv * DV, (uint64_t)p.h_kv * DV, 64, bf);
  }
  if (!ok) return cudaErrorInvalidValue;
  const dim3 grid(MODE == kDkdv ? (p.max_kv + 127) / 128 : (p.max_q + 127) / 128,
                  MODE == kDkdv ? p.h_kv : p.h_q, p.num_seqs);
  if (grid.x == 0) return cudaSuccess;
  auto kern = tc_bwd_kernel<MODE, DQK, DV, NBUF, NSTAGE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, 192, C::SMEM, st>>>(m, p);
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

template <int DQK, int DV, int NBUF_KV>
cudaError_t bwd_shape(const Params &p, cudaStream_t st, const cudaEvent_t *ev) {
  cudaError_t e;
  if ((e = mark(ev, 0, st)) != cudaSuccess) return e;
  if ((e = rowdot_forward(p, st)) != cudaSuccess) return e;
  if ((e = mark(ev, 1, st)) != cudaSuccess) return e;
  if ((e = launch_bwd<kDkdv, DQK, DV, NBUF_KV, 3>(p, st)) != cudaSuccess) return e;
  if ((e = mark(ev, 2, st)) != cudaSuccess) return e;
  if ((e = launch_bwd<kDq, DQK, DV, 2, 3>(p, st)) != cudaSuccess) return e;
  return mark(ev, 3, st);
}

}  // namespace

bool tc_backward_supported(const Params &p) {
  if (p.dtype != VLF_F16 && p.dtype != VLF_BF16) return false;
  return (p.d_qk == 64 && p.d_v == 64) || (p.d_qk == 128 && p.d_v == 128) ||
         (p.d_qk == 192 && p.d_v == 128);
}

cudaError_t tc_backward(const Params &p, cudaStream_t st, const cudaEvent_t *ev) {
  if (p.total_q == 0 || p.total_kv == 0) return simt_backward(p, st, ev);
  if (p.d_qk == 64) return bwd_shape<64, 64, 2>(p, st, ev);
  if (p.d_qk == 128) return bwd_shape<128, 128, 2>(p, st, ev);
  return bwd_shape<192, 128, 1>(p, st, ev);
}

// The tensor-core backward writes dQ directly (no fp32 accumulator); only the row dot
// products D = rowsum(dO o O) live in the workspace.
size_t tc_backward_workspace(int, int, int) { return 0; }

}  // namespace vlf
