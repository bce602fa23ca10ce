// Tensor-core forward (sm_103a): tcgen05 MMAs accumulating in TMEM, TMA-staged Q/K/V tiles.
//
// The loop is the FlashAttention-2 one that triton-msl part 1 ("What works") describes -- Q
// staged once, then for each K/V tile: S = Q K^T, online softmax (running max and sum with a
// rescale), O += P V -- re-laid out for Blackwell:
//
//  * A CTA owns NT 128-row query tiles of one sequence.  NT = 1 (head widths 64 and 128): 256
//    threads, 256 TMEM columns and under half the SM's shared memory, so two CTAs share an SM
//    and one's prologue (Q load, first tile) and epilogue overlap the other's main loop -- this
//    measured faster than sharing K/V between two tiles.  NT = 2 (QK width 192, whose tiles do
//    not fit twice): consecutive row blocks of one head, or, when a kv head serves an even
//    number of query heads (GQA), the same rows of two query heads that share K/V; each 64-key
//    K/V tile brought into shared memory feeds both.
//  * Warp roles.  NT = 2 (416 threads): warp 0 issues TMA loads (Q once, then K and V tiles
//    into rings); four warps issue the MMAs, one per SM sub-partition (S and P.V of each query
//    tile); warps 2-9 run the softmax, 2-5 for tile 0 and 6-9 for tile 1.  NT = 1 (256
//    threads): warp 0 TMA, warp 1 S MMAs, warp 2 P.V MMAs, warps 4-7 softmax.  One thread per
//    query row (TMEM lane = row); the S-issuing warp of tile 0 owns the TMEM allocation.
//  * TMEM: query tile t owns two 64-column S buffers at 128 t and 128 t + 64 and its O
//    accumulator at 128 NT + 128 t.  KV tile n of a query tile lands in S buffer n mod 2, so
//    S(n+1) is computed while the softmax of S(n) runs and the softmax warps go from one tile
//    to the next without waiting for the tensor core.  P(n) (16-bit) is written over the first
//    32 columns of its S buffer and fed to the P.V MMA straight from TMEM; S(n+2) reuses the
//    buffer once that P.V has completed.
//  * Tile scheduler (mtlattn 0.3.0, "Use"): each query tile visits only the KV tiles of its
//    causal / window band; the per-element mask is applied only in the tiles the band cuts.
//    Tiles start at multiples of 64 keys, so skipping changes no bit of the result.
//  * Online softmax in base 2 with the scale folded into one FMA; the running max used for the
//    exponent is only moved (and O rescaled) when the row max grows by more than 8 (P <= 256),
//    which leaves the result mathematically unchanged.  A rescale waits for the previous P.V
//    (the only time the softmax waits on the tensor core).  O is normalised by the sum of the
//    16-bit P values the MMA actually multiplies (a one-hot row returns its V row unchanged);
//    LSE uses the fp32 sum.
//  * Every wait is bounded (see tc_common.cuh); a timeout records VLF_ERR_TIMEOUT and the CTA
//    drains its in-flight copies and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace vlf {
namespace {

using namespace tc;

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kBN = 64;                    // keys per KV tile

struct FwdMaps {
  CUtensorMap q, k, v;
  CUtensorMap q3;    // PACK: Q as [tokens][heads][D_qk], box {64, G heads, 128 / G tokens}
  CUtensorMap bias;  // bias through TMA: [total_q][bias_heads x max_kv] fp32, box {32, 128}
  CUtensorMap q_rope, k_rope;  // latent head with split operands: the rope tensors (64 columns)
};
// The kernels that need none of the extra maps take only Q, K, V: a smaller parameter block to
// copy per launch (host time a small problem pays on every call).
struct FwdMapsPlain {
  CUtensorMap q, k, v;
};
template <int DQK, bool PACK, int BIAS>
struct FwdMapsFor {
  using type = typename std::conditional<(PACK || BIAS == 2 || DQK == 192), FwdMaps, FwdMapsPlain>::type;
};
__device__ __forceinline__ const CUtensorMap *q3_of(const FwdMaps &m) { return &m.q3; }
__device__ __forceinline__ const CUtensorMap *q3_of(const FwdMapsPlain &m) { return &m.q; }
__device__ __forceinline__ const CUtensorMap *bias_of(const FwdMaps &m) { return &m.bias; }
__device__ __forceinline__ const CUtensorMap *bias_of(const FwdMapsPlain &m) { return &m.q; }
__device__ __forceinline__ const CUtensorMap *qrope_of(const FwdMaps &m) { return &m.q_rope; }
__device__ __forceinline__ const CUtensorMap *qrope_of(const FwdMapsPlain &m) { return &m.q; }
__device__ __forceinline__ const CUtensorMap *krope_of(const FwdMaps &m) { return &m.k_rope; }
__device__ __forceinline__ const CUtensorMap *krope_of(const FwdMapsPlain &m) { return &m.k; }

// NT: query tiles per CTA.  NT = 2: 416 threads and all 512 TMEM columns, one CTA per SM.
// NT = 1: 256 threads, 256 TMEM columns and at most half the SM's shared memory, so two CTAs
// share an SM and one's prologue / epilogue overlaps the other's main loop.
// NBS: stages of the bias ring (0: no bias through TMA).
template <int DQK, int DV, int NK, int NV, int NT, int NBS = 0>
struct FwdCfg {
  // 64-column (128-byte) swizzle blocks per row.  A width that is not a multiple of 64 (96) is
  // padded to whole blocks: the extra columns hold the next head's values (or the tensor's zero
  // fill); the QK^T products step only over the real width, the P.V product runs at the padded
  // N and its extra O columns are never stored.
  static constexpr int KBQ = (DQK + 63) / 64, KBV = (DV + 63) / 64;
  static constexpr int NV_PAD = KBV * 64;  // N of the P.V product
  static constexpr int QBLK = 128 * 128;               // one 128-row x 64-col block of Q
  static constexpr int KVBLK = kBN * 128;              // one 64-row x 64-col block of K or V
  static constexpr int Q_BYTES = KBQ * QBLK, K_BYTES = KBQ * KVBLK, V_BYTES = KBV * KVBLK;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NT * Q_BYTES;
  static constexpr int OFF_V = OFF_K + NK * K_BYTES;
  // bias tile of a 128-row query tile and a 64-key KV tile: two 32-column boxes (128-byte rows)
  static constexpr int BIAS_BOX = 128 * 128, BIAS_STAGE = 2 * BIAS_BOX;
  static constexpr int NBS_ = NBS > 0 ? NBS : 1;  // (a nonzero divisor where there is no ring)
  static constexpr int OFF_B = OFF_V + NV * V_BYTES;
  static constexpr int OFF_BAR = OFF_B + NBS * BIAS_STAGE;
  // barriers: q_full, k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], then per query tile t
  // and S buffer b (index 2 t + b): s_full, p_full, o_done (the P.V that read buffer b); drain
  // (one per MMA-issuing warp)
  static constexpr int B_Q = 0, B_KF = 1, B_KE = B_KF + NK, B_VF = B_KE + NK, B_VE = B_VF + NV;
  static constexpr int B_S = B_VE + NV, B_P = B_S + 2 * NT, B_O = B_P + 2 * NT;
  static constexpr int B_DRAIN = B_O + 2 * NT;
  static constexpr int B_BF = B_DRAIN + 2 * NT, B_BE = B_BF + NBS;  // bias full / empty
  static constexpr int NBAR = B_BE + NBS;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // (no alignment slack: the dynamic shared window starts 1024-byte aligned, checked in-kernel)
  static constexpr int SMEM = OFF_MISC + 16;
  static constexpr int THREADS = NT == 2 ? 416 : 256;
  // TMEM: query tile t's two 64-column S buffers at 128 t, its O at O_COL + 128 t.  WIDE
  // (width 256, NT = 1): O takes 256 columns and the CTA the whole TMEM -- one CTA per SM, as its
  // shared memory (a 64 KB Q tile, 32 KB K / V slots) already is.
  static constexpr bool WIDE = NV_PAD > 128;
  static constexpr uint32_t TMEM_COLS = WIDE ? 512 : 256 * NT, O_COL = 128 * NT;
  static constexpr int MIN_BLOCKS = NT == 1 && !WIDE ? 2 : 1;  // CTAs resident per SM
  // The producer issues K(j + LEAD) before V(j).  A K or V tile waits for its ring slot; with
  // one query tile a K load must not queue behind a V slot that frees late, so K leads by one.
  static constexpr int LEAD = NT == 1 ? 1 : 0;
  static_assert(NT == 1 || NT == 2, "query tiles per CTA");
  static_assert(NV >= 2 && NK >= 2, "ring depth");
  static_assert(DQK % 32 == 0 && DV % 32 == 0 && NV_PAD <= (NT == 1 ? 256 : 128), "tile shapes");
  static_assert(SMEM <= (MIN_BLOCKS == 1 || NBS > 0 ? 232448 : 115712), "shared memory");
};


struct TileInfo {
  // row0: first sequence-local query row; head: query head (PACK: the kv head)
  int row0[2], head[2];
  int jlo[2], jhi[2];  // KV tile range of each query tile (empty: jlo == jhi)
  int lo, hi;          // union
};

// Query tiles of CTA (bx, by): NT = 2 takes two row blocks of one head, or the same rows of two
// heads sharing a kv head (pair_heads); NT = 1 one row block.  Tile 1 of an NT = 1 CTA is empty.
// PACK (NT = 1): the tile's 128 rows are 128 / G query rows x the G query heads of kv head by
// (row r = query row r / G of head by G + r mod G), so each K/V tile serves the whole group.
template <int NT, bool PACK>
__device__ __forceinline__ void tile_info(const Params &p, const Seq &sq, int bx, int by,
                                          bool pair_heads, TileInfo &ti) {
  const int rows = PACK ? 128 / p.group : 128;  // query rows per tile
  for (int t = 0; t < 2; ++t) {
    ti.row0[t] = NT == 1 ? (t == 0 ? bx * rows : sq.q_len) : (pair_heads ? bx * 128 : bx * 256 + 128 * t);
    ti.head[t] = NT == 1 ? by : (pair_heads ? 2 * by + t : by);
    int jl = 0, jh = 0;
    if (ti.row0[t] < sq.q_len && sq.kv_len > 0) {
      int klo, khi;
      kv_band(ti.row0[t], min(ti.row0[t] + rows, sq.q_len), sq.q_len, sq.kv_len, p.causal,
              p.window, klo, khi);
      if (p.flags & VLF_FLAG_NO_SKIP) { klo = 0; khi = sq.kv_len; }
      if (khi > klo) { jl = klo / kBN; jh = (khi + kBN - 1) / kBN; }
    }
    ti.jlo[t] = jl;
    ti.jhi[t] = jh;
  }
  const bool e0 = ti.jhi[0] <= ti.jlo[0], e1 = ti.jhi[1] <= ti.jlo[1];
  if (e0 && e1) { ti.lo = ti.hi = 0; }
  else if (e0) { ti.lo = ti.jlo[1]; ti.hi = ti.jhi[1]; }
  else if (e1) { ti.lo = ti.jlo[0]; ti.hi = ti.jhi[0]; }
  else { ti.lo = min(ti.jlo[0], ti.jlo[1]); ti.hi = max(ti.jhi[0], ti.jhi[1]); }
}

// Barrier phases.  Each (tile, buffer) barrier completes once per use of that buffer, and a use
// n + 2 never starts before use n has been consumed (S(n+2) is issued after P.V(n) completed;
// P.V(n+2) after the softmax of S(n+2)), so every waiter is at most one phase behind and the
// parity (n >> 1) & 1 is unambiguous.  tcgen05.commit arrives when every MMA the committing
// thread issued before it has completed; the P.V MMAs of a query tile come from one warp, so the
// o_done of P.V(n) also covers P.V(n-1).

// BF16: element type of Q/K/V/O (bf16, else fp16), fixed at compile time so the per-element
// conversions carry no runtime branch.
// BIAS: 0 no bias, 1 bias rows read from global memory, 2 bias tiles staged through TMA (NT = 1,
// not PACK); separate instantiations, so that kernels without a bias carry none of its code or
// registers.
// PACK (NT = 1 only): the G query heads of a kv head share each tile (decode-sized problems).
// SPLIT (NT = 1, BIAS 0 or 1): split-KV part kernel -- the CTA takes part blockIdx.z mod
// p.kv_splits of its KV band and writes fp32 partial results (a separate instantiation, so that
// the unsplit kernels carry none of its code or registers).
template <int DQK, int DV, int NK, int NV, int NT, bool BF16, int BIAS, bool PACK, bool SPLIT>
__global__ void __launch_bounds__(FwdCfg<DQK, DV, NK, NV, NT>::THREADS, FwdCfg<DQK, DV, NK, NV, NT>::MIN_BLOCKS)
tc_fwd_kernel(const __grid_constant__ typename FwdMapsFor<DQK, PACK, BIAS>::type maps, const Params p) {
  constexpr int NBS = BIAS == 2 ? 2 : 0;
  static_assert(BIAS != 2 || (NT == 1 && !PACK), "bias tiles through TMA: one unpacked tile");
  static_assert(!SPLIT || (NT == 1 && BIAS != 2), "split-KV parts: one tile, no bias ring");
  using C = FwdCfg<DQK, DV, NK, NV, NT, NBS>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // launched with programmatic stream serialization (small problems, launch_kernel below): let
  // the next kernel be launched now, and read nothing global before the previous one is done
  pdl_trigger();
  pdl_wait();
  const bool pair_heads = NT == 2 && (p.group % 2 == 0);
  // (split-KV: the part index is recomputed where it is needed, so that it is not held in a
  // register through the main loop)
  const int s = SPLIT ? (int)blockIdx.z / p.kv_splits : (int)blockIdx.z;
  Seq sq;
  if (!load_seq(p, s, sq)) return;
  if (s == 0 && (__ldg(p.cu_q) != 0 || __ldg(p.cu_kv) != 0)) set_error(p.err, VLF_ERR_BAD_SEQLENS);
  if (s == p.num_seqs - 1 && (sq.q0 + sq.q_len != p.total_q || sq.k0 + sq.kv_len != p.total_kv))
    set_error(p.err, VLF_ERR_BAD_SEQLENS);
  // heavy (late, long-band) row blocks first under causal masking; heads_fast swaps the grid's
  // x and y so that the heads of one row block run together
  const int bxr = p.heads_fast ? (int)blockIdx.y : (int)blockIdx.x;
  const int gx = p.heads_fast ? (int)gridDim.y : (int)gridDim.x;
  const int bx = p.causal ? gx - 1 - bxr : bxr;
  const int by = p.heads_fast ? (int)blockIdx.x : (int)blockIdx.y;
  TileInfo ti;
  static_assert(!PACK || NT == 1, "packed heads use one query tile per CTA");
  tile_info<NT, PACK>(p, sq, bx, by, pair_heads, ti);
  if (ti.row0[0] >= sq.q_len) return;  // whole CTA beyond this sequence
  if (SPLIT) {
    // this part's share of the band, in whole KV tiles (possibly none: it then writes O = 0
    // and LSE = -inf, which the combine weighs by zero)
    const int part = (int)blockIdx.z % p.kv_splits;
    const int per = (ti.hi - ti.lo + p.kv_splits - 1) / p.kv_splits;
    const int a = min(ti.hi, ti.lo + part * per), b = min(ti.hi, a + per);
    ti.jlo[0] = ti.lo = a;
    ti.jhi[0] = ti.hi = b;
  }
  // Bias bands: the KV tiles in which some row of the tile has a finite bias value (the others
  // hold only masked pairs: skipping them is exact); cta_pure: every row's bias is 0 over its
  // finite interval, so the tile is masked by those intervals and the bias is not read.
  bool cta_pure = false;
  if constexpr (BIAS != 0 && NT == 1 && !PACK && !SPLIT) {
    if (p.bias_blocks && ti.hi > ti.lo) {
      const int hb = p.bias_heads == 1 ? 0 : ti.head[0];
      const int4 *bb = p.bias_blocks + (size_t)hb * p.total_q + sq.q0 + ti.row0[0];
      const int4 e0 = __ldg(bb);
      int blo = e0.x, bhi = e0.y, pure = e0.z >= 0;
      if (ti.row0[0] + 64 < sq.q_len) {
        const int4 e1 = __ldg(bb + 64);
        if (e1.y > e1.x) {
          blo = bhi > blo ? min(blo, e1.x) : e1.x;
          bhi = max(bhi, e1.y);
        }
        pure &= e1.z >= 0;
      }
      int jl = ti.lo, jh = ti.hi;
      if (bhi > blo) {
        jl = max(jl, blo / kBN);
        jh = min(jh, (bhi + kBN - 1) / kBN);
      }
      if (bhi <= blo || jh <= jl) jl = jh = 0;
      ti.jlo[0] = ti.lo = jl;
      ti.jhi[0] = ti.hi = jh;
      cta_pure = pure != 0;
    }
  }

  // The kernel has no static shared memory, so the dynamic window starts 1024-byte aligned, as
  // the 128-byte swizzle atoms of the TMA tiles and MMA descriptors require; refuse otherwise.
  const uint32_t base = smem_u32(smem_raw);
  if (base & 1023u) {
    if (threadIdx.x == 0) set_error(p.err, VLF_ERR_ALIGN);
    return;
  }
  uint8_t *gbase = smem_raw;
  const uint32_t sQ = base + C::OFF_Q, sK = base + C::OFF_K, sV = base + C::OFF_V;
  const uint32_t sB = base + C::OFF_B;
  const uint32_t bar0 = base + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(gbase + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_Q), 1);
    // a K or V slot is free once both query tiles' issuers have released it
    for (int i = 0; i < NK; ++i) { mbar_init(bar(C::B_KF + i), 1); mbar_init(bar(C::B_KE + i), NT); }
    for (int i = 0; i < NV; ++i) { mbar_init(bar(C::B_VF + i), 1); mbar_init(bar(C::B_VE + i), NT); }
    for (int i = 0; i < 2 * NT; ++i) {
      mbar_init(bar(C::B_S + i), 1);
      mbar_init(bar(C::B_P + i), 128);
      mbar_init(bar(C::B_O + i), 1);
      mbar_init(bar(C::B_DRAIN + i), 1);
    }
    for (int i = 0; i < NBS; ++i) { mbar_init(bar(C::B_BF + i), 1); mbar_init(bar(C::B_BE + i), 128); }
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
  const int hk = PACK ? ti.head[0] : ti.head[0] / p.group;  // both query tiles read one kv head
  constexpr int is_bf16 = BF16 ? 1 : 0;
  const int lo = ti.lo, hi = ti.hi;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && hi > lo) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      // a latent head given as split operands (QK width 192 only): the first two 64-column
      // blocks of each Q / K tile come from the nope tensors (row width 128 per head), the third
      // from the rope tensors
      const bool lat = DQK == 192 && p.latent;
      const int qw = lat ? 128 : DQK;
      const int rh = lat && p.rope_heads == 1 ? 0 : hk;  // the kv head's rope key
      if (lat) {
        tma_prefetch_desc(qrope_of(maps));
        tma_prefetch_desc(krope_of(maps));
      }
      int nq = 0;
      for (int t = 0; t < 2; ++t) nq += ti.row0[t] < sq.q_len ? 1 : 0;
      // (VLF_FLAG_TEST_TIMEOUT: no query tile, so that the waits on it run out)
      const bool drop_q = (p.flags & VLF_FLAG_TEST_TIMEOUT) != 0;
      if (!drop_q) mbar_expect_tx(bar(C::B_Q), nq * C::Q_BYTES);
      for (int t = 0; t < 2 && !drop_q; ++t) {
        if (ti.row0[t] >= sq.q_len) continue;
        for (int c = 0; c < C::KBQ; ++c) {
          if (PACK)  // rows (token, head of the group): one 3-D box
            tma_load_3d(sQ + t * C::Q_BYTES + c * C::QBLK, q3_of(maps), 64 * c, hk * p.group,
                        sq.q0 + ti.row0[t], bar(C::B_Q));
          else if (lat && c == 2)
            tma_load_2d(sQ + t * C::Q_BYTES + c * C::QBLK, qrope_of(maps), ti.head[t] * 64,
                        sq.q0 + ti.row0[t], bar(C::B_Q));
          else
            tma_load_2d(sQ + t * C::Q_BYTES + c * C::QBLK, &maps.q, ti.head[t] * qw + 64 * c,
                        sq.q0 + ti.row0[t], bar(C::B_Q));
        }
      }
      int k_issued[NK] = {0}, v_issued[NV] = {0}, b_issued[NBS > 0 ? NBS : 1] = {0};
      if (BIAS == 2) tma_prefetch_desc(bias_of(maps));
      const int bcol = BIAS == 2 ? (p.bias_heads == 1 ? 0 : ti.head[0]) * p.max_kv : 0;
      bool ok = true;
      for (int j = lo; j < hi + C::LEAD && ok; ++j) {
        const int kj = j, vj = j - C::LEAD;  // K tile issued ahead of V by LEAD
        if (BIAS == 2 && kj < hi && !cta_pure) {
          // the query tile's bias columns of KV tile kj: rows row0 .. row0 + 127
          const int it = kj - lo, bs = it % C::NBS_;
          if (it >= C::NBS_) ok = mbar_wait(bar(C::B_BE + bs), ((it / C::NBS_) - 1) & 1, abort_flag, p.err);
          if (!ok) break;
          mbar_expect_tx(bar(C::B_BF + bs), C::BIAS_STAGE);
          for (int c = 0; c < 2; ++c)
            tma_load_2d(sB + bs * C::BIAS_STAGE + c * C::BIAS_BOX, bias_of(maps), bcol + kj * kBN + 32 * c,
                        sq.q0 + ti.row0[0], bar(C::B_BF + bs));
          ++b_issued[bs];
        }
        if (kj < hi) {
          const int it = kj - lo, ks = it % NK;
          if (it >= NK) ok = mbar_wait(bar(C::B_KE + ks), ((it / NK) - 1) & 1, abort_flag, p.err);
          if (!ok) break;
          mbar_expect_tx(bar(C::B_KF + ks), C::K_BYTES);
          for (int c = 0; c < C::KBQ; ++c) {
            if (lat && c == 2)
              tma_load_2d(sK + ks * C::K_BYTES + c * C::KVBLK, krope_of(maps), rh * 64,
                          sq.k0 + kj * kBN, bar(C::B_KF + ks));
            else
              tma_load_2d(sK + ks * C::K_BYTES + c * C::KVBLK, &maps.k, hk * qw + 64 * c,
                          sq.k0 + kj * kBN, bar(C::B_KF + ks));
          }
          ++k_issued[ks];
        }
        if (vj >= lo) {
          const int it = vj - lo, vs = it % NV;
          if (it >= NV) ok = mbar_wait(bar(C::B_VE + vs), ((it / NV) - 1) & 1, abort_flag, p.err);
          if (!ok) break;
          mbar_expect_tx(bar(C::B_VF + vs), C::V_BYTES);
          for (int c = 0; c < C::KBV; ++c)
            tma_load_2d(sV + vs * C::V_BYTES + c * C::KVBLK, &maps.v, hk * DV + 64 * c,
                        sq.k0 + vj * kBN, bar(C::B_VF + vs));
          ++v_issued[vs];
        }
      }
      // make sure no copy is still landing in shared memory when the CTA leaves
      drain_wait(bar(C::B_Q), 0);
      for (int i = 0; i < NK; ++i)
        if (k_issued[i]) drain_wait(bar(C::B_KF + i), (k_issued[i] - 1) & 1);
      for (int i = 0; i < NV; ++i)
        if (v_issued[i]) drain_wait(bar(C::B_VF + i), (v_issued[i] - 1) & 1);
      for (int i = 0; i < NBS; ++i)
        if (b_issued[i]) drain_wait(bar(C::B_BF + i), (b_issued[i] - 1) & 1);
    }
  } else if (NT == 2 ? (warp == 1 || warp >= 10) : (warp == 1 || warp == 2)) {
    // ------------------------------------------------------------------ MMA issuers
    // Four warps issue MMAs, one per SM sub-partition: S = Q K^T of query tile 0 (warp 1) and
    // tile 1 (warp 11), O += P V of tile 0 (warp 12) and tile 1 (warp 10).  An MMA issue returns
    // only once the tensor pipe accepts it, so an issuer that waits (for a P, or for a P.V to
    // free an S buffer) would leave the pipe idle if it were the only one; and a warp blocked in
    // MMA issue slows the other warps of its sub-partition, so the issue load is spread evenly
    // over the softmax warps.  Each issuer walks every KV tile of the CTA's range (to release
    // its share of the K or V ring slot) and issues the MMAs of its own query tile; it runs its
    // loop as a whole warp (uniform operands) and elect.sync picks the issuing lane.
    // NT = 1: warp 1 issues S, warp 2 P.V
    const bool is_s = NT == 2 ? (warp == 1 || warp == 11) : warp == 1;
    const int t = NT == 2 ? ((warp == 1 || warp == 12) ? 0 : 1) : 0;
    const int drain = C::B_DRAIN + (NT == 2 ? (warp == 1 ? 0 : warp - 9) : warp - 1);
    if (hi > lo) {
      const int jlo = ti.jlo[t], jhi = ti.jhi[t];
      bool ok = true;
      if (is_s) {
        const uint32_t id_s = idesc_f16(is_bf16, 128, kBN, 0, 0);  // both operands K-major
        const uint64_t dq = sdesc_sw128(sQ + t * C::Q_BYTES, 16, 1024);
        const uint64_t dk0 = sdesc_sw128(sK, 16, 1024);
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_Q), 0, abort_flag, p.err));
        for (int j = lo; j < hi && ok; ++j) {
          const int it = j - lo;
          // every issuer waits for each K tile, used or not: its release of the slot then never
          // runs a full ring ahead of the other tile's, which keeps the two-arrival phases apart
          ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_KF + it % NK), (it / NK) & 1, abort_flag, p.err));
          if (!ok) break;
          if (j >= jlo && j < jhi) {
            const int n = j - jlo, b = n & 1;
            if (n >= 2) {
              // S(n) overwrites the buffer P(n-2) was read from: wait for that P.V
              const int np = n - 2;
              ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_O + 2 * t + b), (np >> 1) & 1, abort_flag, p.err));
              if (!ok) break;
            }
            fence_after();
            const uint64_t dk = dk0 + (uint64_t)(((it % NK) * C::K_BYTES) >> 4);
#pragma unroll
            for (int kk = 0; kk < DQK / 16; ++kk) {
              // a K step adds its byte offset / 16 to the descriptor's start-address field
              const uint64_t oq = (uint64_t)(((kk >> 2) * C::QBLK + (kk & 3) * 32) >> 4);
              const uint64_t okk = (uint64_t)(((kk >> 2) * C::KVBLK + (kk & 3) * 32) >> 4);
              mma_ss_w(tmem + 128 * t + 64 * b, dq + oq, dk + okk, id_s, kk > 0);
            }
            mma_commit_w(bar(C::B_S + 2 * t + b));
          }
          // this tile's share of releasing the K slot (arrives once its S MMAs have read it)
          mma_commit_w(bar(C::B_KE + it % NK));
        }
      } else {
        const uint32_t id_o = idesc_f16(is_bf16, 128, C::NV_PAD, 0, 1);  // V is MN-major
        const uint64_t dv0 = sdesc_sw128(sV, C::KVBLK, 1024);
        for (int j = lo; j < hi && ok; ++j) {
          const int it = j - lo;
          ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_VF + it % NV), (it / NV) & 1, abort_flag, p.err));
          if (!ok) break;
          if (j >= jlo && j < jhi) {
            const int n = j - jlo, b = n & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_P + 2 * t + b), (n >> 1) & 1, abort_flag, p.err));
            if (!ok) break;
            fence_after();
            const uint64_t dv = dv0 + (uint64_t)(((it % NV) * C::V_BYTES) >> 4);
            const uint32_t pcol = tmem + 128 * t + 64 * b;
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              mma_ts_w(tmem + C::O_COL + 128 * t, pcol + kk * 8, dv + (uint64_t)((kk * 2048) >> 4), id_o,
                       (n > 0 || kk > 0) ? 1u : 0u);
            mma_commit_w(bar(C::B_O + 2 * t + b));
          }
          mma_commit_w(bar(C::B_VE + it % NV));
        }
      }
      // drain: every MMA this warp issued has completed before TMEM is released
      mma_commit_w(bar(drain));
      drain_wait(bar(drain), 0);
    }
  } else if (NT == 2 || warp >= 4) {
    // ------------------------------------------------------------------ softmax / epilogue
    // (NT = 2: warps 2-9; NT = 1: warps 4-7, warp 3 has no role)
    const int t = NT == 2 ? (warp - 2) >> 2 : 0;
    const int quarter = warp & 3;
    const int r = 32 * quarter + lane;
    const int i = ti.row0[t] + (PACK ? r / p.group : r);  // sequence-local query row
    const bool row_ok = i < sq.q_len;
    const int off = sq.kv_len - sq.q_len;
    const int head = PACK ? hk * p.group + r % p.group : ti.head[t];  // this row's query head
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16);
    const uint32_t s_addr = lane_addr + 128 * t, o_addr = lane_addr + C::O_COL + 128 * t;
    const float sl2 = p.scale_log2;
    const float *brow = nullptr;
    if (BIAS && row_ok && !cta_pure) {
      const int bh = p.bias_heads == 1 ? 0 : head;
      brow = p.bias + ((size_t)(sq.q0 + i) * (size_t)p.bias_heads + (size_t)bh) * (size_t)p.max_kv;
    }
    // a pure CTA: this row's finite-bias interval, intersected with its causal / window range
    int rlo = 0, rhi = sq.kv_len;
    if (BIAS && cta_pure && row_ok) {
      const int bh = p.bias_heads == 1 ? 0 : head;
      const int4 e = __ldg(p.bias_rows + (size_t)bh * p.total_q + sq.q0 + i);
      rlo = e.x;
      rhi = e.y;
    }
    const bool bias_vals = BIAS && !cta_pure;  // bias values are added to the logits
    // l: sum of the rounded P the MMA multiplies (normalises O); lf: the fp32 sum (for LSE)
    float m_ref = -INFINITY, l = 0.f, lf = 0.f;
    const int jlo = ti.jlo[t], jhi = ti.jhi[t];
    bool ok = true;
    for (int j = jlo; j < jhi; ++j) {
      const int n = j - jlo, b = n & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_S + 2 * t + b), (n >> 1) & 1, abort_flag, p.err));
      if (!ok) break;
      fence_after();
      const uint32_t sb = s_addr + 64 * b;
      const int kb = j * kBN;
      const bool full = row_ok && (kb + kBN - 1 < sq.kv_len) && (!p.causal || kb + kBN - 1 <= i + off) &&
                        (p.window <= 0 || kb >= i + off - p.window + 1) && kb >= rlo && kb + kBN <= rhi;
      const bool plain = full && !bias_vals;
      // the whole S row (64 fp32) in registers: two TMEM loads, one wait
      uint32_t v[kBN];
      __syncwarp();
      tmem_ld32_at(sb + 0, v, 0);
      tmem_ld32_at(sb + 32, v, 32);
      tmem_ld_wait();
      // P = 2^(logit2 - m_ref) two at a time (packed FMA), written in 16-bit over the first 32
      // columns of the S buffer, 16 pairs at a time; with the fp32 row sum and the sum of the
      // rounded P the MMA consumes (so the weights that multiply V are normalised exactly: a
      // one-hot row returns its V row unchanged).  Two accumulators each keep the dependent add
      // chains short.
      float sumr = 0.f, lsum = 0.f;
      auto exp_pass = [&](float scale, float neg_m) {
        const uint64_t scale2 = f2pack(scale, scale), negm2 = f2pack(neg_m, neg_m);
        uint64_t sf0 = f2pack(0.f, 0.f), sf1 = sf0;
        float sr0 = 0.f, sr1 = 0.f;
#pragma unroll
        for (int ch = 0; ch < kBN / 32; ++ch) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c = 32 * ch + 2 * e;
            const float2 x = f2unpack(fma2(f2pack(__uint_as_float(v[c]), __uint_as_float(v[c + 1])),
                                           scale2, negm2));
            const float pa = ex2(x.x), pb = ex2(x.y);
            pk[e] = pack2(pa, pb, is_bf16);
            if (e & 1) {
              sf1 = add2(sf1, f2pack(pa, pb));
              sr1 = add_halves(sr1, pk[e], is_bf16);
            } else {
              sf0 = add2(sf0, f2pack(pa, pb));
              sr0 = add_halves(sr0, pk[e], is_bf16);
            }
          }
          __syncwarp();
          tmem_st16(sb + ch * 16, pk);
        }
        const float2 f0 = f2unpack(sf0), f1 = f2unpack(sf1);
        lsum = (f0.x + f0.y) + (f1.x + f1.y);
        sumr = sr0 + sr1;
      };
      // Speculative pass: when every row of the warp is an unmasked tile that already has a
      // reference max, P is computed with that reference while the row max is found alongside
      // (no dependency between the two).  Only a row max beyond the threshold sends the warp
      // through the general pass below, which recomputes P; otherwise the reference stays put
      // and the result is exactly what the general pass gives.
      bool done = false;
      if (__all_sync(0xffffffffu, plain && m_ref != -INFINITY)) {
        exp_pass(sl2, -m_ref);
        float m8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float *f = reinterpret_cast<const float *>(v) + 8 * q;
          m8[q] = fmax3(fmax3(f[0], f[1], f[2]), fmax3(f[3], f[4], f[5]), fmaxf(f[6], f[7]));
        }
        const float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) * sl2;
        done = !__any_sync(0xffffffffu, mx > m_ref + kRescaleThreshold);
        // the general pass rewrites P: let the speculative stores land first
        if (!done) tmem_st_wait();
      }
      if (!done) {
        // row max of the base-2 logits.  plain rows keep raw q.k in v (the scale goes into the
        // exponent FMA); other rows get v = scale*log2e*q.k + log2e*bias, or -inf where masked.
        float mx;
        if (plain) {
          float m8[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float *f = reinterpret_cast<const float *>(v) + 8 * q;
            m8[q] = fmax3(fmax3(f[0], f[1], f[2]), fmax3(f[3], f[4], f[5]), fmaxf(f[6], f[7]));
          }
          mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) * sl2;
        } else {
          // the visible keys of this row are one interval: mask by two compares per element
          int vlo, vhi;
          visible_range(i, off, sq.kv_len, p.causal, p.window, vlo, vhi);
          vlo = max(vlo, rlo);
          vhi = min(vhi, rhi);
          if (!row_ok) vhi = vlo;
          const int elo = vlo - kb, ehi = vhi - kb;
          // logits in base 2; the bias row is read 16 bytes at a time when its address allows
          // and the tile lies inside it, else element by element (the column clamped into the
          // row: masked elements read a valid address)
          if (!bias_vals) {
#pragma unroll
            for (int e = 0; e < kBN; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * sl2);
          } else if (BIAS == 2) {
            // the tile's bias, staged by the producer: this row of the two 32-column boxes
            // (128-byte swizzle: 16-byte chunk q of row r sits at chunk q ^ (r mod 8))
            const int it = j - jlo, bs = it % C::NBS_;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_BF + bs), (it / C::NBS_) & 1, abort_flag, p.err));
            if (!ok) break;
            const uint32_t rowb = sB + bs * C::BIAS_STAGE + r * 128;
#pragma unroll
            for (int q = 0; q < kBN / 4; ++q) {
              const uint32_t a = rowb + (q >> 3) * C::BIAS_BOX + (((q & 7) ^ (r & 7)) << 4);
              const float4 bq = lds_f32x4(a);
              v[4 * q + 0] = __float_as_uint(fmaf(bq.x, kLog2e, __uint_as_float(v[4 * q + 0]) * sl2));
              v[4 * q + 1] = __float_as_uint(fmaf(bq.y, kLog2e, __uint_as_float(v[4 * q + 1]) * sl2));
              v[4 * q + 2] = __float_as_uint(fmaf(bq.z, kLog2e, __uint_as_float(v[4 * q + 2]) * sl2));
              v[4 * q + 3] = __float_as_uint(fmaf(bq.w, kLog2e, __uint_as_float(v[4 * q + 3]) * sl2));
            }
            mbar_arrive(bar(C::B_BE + bs));  // the slot may be refilled
          } else if (BIAS && brow && (reinterpret_cast<uintptr_t>(brow) & 15u) == 0 && kb + kBN <= p.max_kv) {
            const float4 *b4 = reinterpret_cast<const float4 *>(brow + kb);
#pragma unroll
            for (int q = 0; q < kBN / 4; ++q) {
              const float4 bq = __ldg(b4 + q);
              v[4 * q + 0] = __float_as_uint(fmaf(bq.x, kLog2e, __uint_as_float(v[4 * q + 0]) * sl2));
              v[4 * q + 1] = __float_as_uint(fmaf(bq.y, kLog2e, __uint_as_float(v[4 * q + 1]) * sl2));
              v[4 * q + 2] = __float_as_uint(fmaf(bq.z, kLog2e, __uint_as_float(v[4 * q + 2]) * sl2));
              v[4 * q + 3] = __float_as_uint(fmaf(bq.w, kLog2e, __uint_as_float(v[4 * q + 3]) * sl2));
            }
          } else {
#pragma unroll
            for (int e = 0; e < kBN; ++e) {
              float x = __uint_as_float(v[e]) * sl2;
              if (BIAS && brow) x = fmaf(__ldg(brow + min(kb + e, sq.kv_len - 1)), kLog2e, x);
              v[e] = __float_as_uint(x);
            }
          }
          mx = -INFINITY;
#pragma unroll
          for (int e = 0; e < kBN; ++e) {
            const float x = (e >= elo && e < ehi) ? __uint_as_float(v[e]) : -INFINITY;
            v[e] = __float_as_uint(x);
            mx = fmaxf(mx, x);
          }
        }
        // move the reference max only when it grows by more than the threshold
        const float m_new = fmaxf(m_ref, mx);
        float alpha = 1.f;
        bool move = false;
        if (m_new != -INFINITY && m_new > m_ref + kRescaleThreshold) {
          alpha = ex2(m_ref - m_new);  // m_ref == -inf -> 0
          move = true;
        }
        // rows whose reference moved and that have accumulated something rescale O_t, once the
        // P.V of the previous KV tile (and so every earlier one) has completed
        const bool need = move && n > 0 && l > 0.f;
        if (__any_sync(0xffffffffu, need)) {
          const int np = n - 1;
          ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_O + 2 * t + (np & 1)), (np >> 1) & 1, abort_flag, p.err));
          if (!ok) break;
          fence_after();
          const float a = need ? alpha : 1.f;
#pragma unroll 1
          for (int ch = 0; ch < DV / 32; ++ch) {
            uint32_t o[32];
            tmem_ld32(o_addr + ch * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
            tmem_st32(o_addr + ch * 32, o);
          }
        }
        if (move) {
          l *= alpha;
          lf *= alpha;
          m_ref = m_new;
        }
        // a row still without any visible key has every logit at -inf: its exponent offset is
        // taken as 0 so that P = 0
        exp_pass(plain ? sl2 : 1.f, m_ref == -INFINITY ? 0.f : -m_ref);
      }
      l += sumr;
      lf += lsum;
      __syncwarp();
      tmem_st_wait();
      fence_before();
      mbar_arrive(bar(C::B_P + 2 * t + b));
    }
    // epilogue: O / l in the output dtype, LSE in natural log
    const int nt = jhi - jlo;
    if (ok && nt > 0) {
      const int np = nt - 1;
      ok = mbar_wait(bar(C::B_O + 2 * t + (np & 1)), (np >> 1) & 1, abort_flag, p.err);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (SPLIT && ok) {
      // a part's result for the combine: fp32 O / l and the part's log-sum-exp
      fence_after();
      const int part = (int)blockIdx.z % p.kv_splits;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const size_t grow = (size_t)sq.q0 + (size_t)(row_ok ? i : 0);
      float4 *dst = reinterpret_cast<float4 *>(p.o_part + (((size_t)part * p.total_q + grow) * p.h_q + head) * DV);
#pragma unroll 1
      for (int ch = 0; ch < DV / 32; ++ch) {
        uint32_t v[32];
        if (nt > 0) {
          __syncwarp();
          tmem_ld32(o_addr + ch * 32, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        if (row_ok) {
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            dst[ch * 8 + q4] = make_float4(__uint_as_float(v[4 * q4]) * inv, __uint_as_float(v[4 * q4 + 1]) * inv,
                                           __uint_as_float(v[4 * q4 + 2]) * inv, __uint_as_float(v[4 * q4 + 3]) * inv);
        }
      }
      if (row_ok)
        p.lse_part[((size_t)part * p.h_q + head) * p.total_q + grow] =
            lf > 0.f ? (m_ref + lg2(lf)) * kLn2 : -INFINITY;
    } else if (!SPLIT && ok) {
      fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const size_t grow = (size_t)sq.q0 + (size_t)(row_ok ? i : 0);
      uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.out) +
                                             ((grow * p.h_q + head) * DV) * 2);
#pragma unroll 1
      for (int ch = 0; ch < DV / 32; ++ch) {
        uint32_t v[32];
        if (nt > 0) {
          __syncwarp();
          tmem_ld32(o_addr + ch * 32, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack2(__uint_as_float(v[2 * e]) * inv, __uint_as_float(v[2 * e + 1]) * inv, is_bf16);
        if (row_ok) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            dst[ch * 4 + q4] = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
        }
      }
      if (row_ok && p.lse)
        p.lse[(size_t)head * p.total_q + grow] = lf > 0.f ? (m_ref + lg2(lf)) * kLn2 : -INFINITY;
    }
  }

  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Merges the parts of a split-KV forward.  With L_s the parts' log-sum-exps and O_s their
// normalised results: LSE = log sum_s exp(L_s), O = sum_s exp(L_s - LSE) O_s (a part that saw no
// key has L_s = -inf and weight 0; a row no part saw gets O = 0, LSE = -inf).  One warp per
// (query row, head); lane c reads columns c, c + 32, ... of every part (coalesced rows).
template <int DV, bool BF16>
__global__ void __launch_bounds__(256) split_combine_kernel(const Params p) {
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  const long long w = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (w >= (long long)p.total_q * p.h_q) return;
  const int lane = threadIdx.x & 31;
  const int row = (int)(w / p.h_q), head = (int)(w % p.h_q);
  const int S = p.kv_splits;
  auto part_lse = [&](int sp) { return p.lse_part[((size_t)sp * p.h_q + head) * p.total_q + row]; };
  float m = -INFINITY;
  for (int sp = lane; sp < S; sp += 32) m = fmaxf(m, part_lse(sp));
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float sum = 0.f;
  if (m != -INFINITY)
    for (int sp = lane; sp < S; sp += 32) sum += expf(part_lse(sp) - m);
#pragma unroll
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float lse = m == -INFINITY ? -INFINITY : m + logf(sum);
  constexpr int NC = DV / 32;
  float acc[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) acc[c] = 0.f;
  if (lse != -INFINITY) {
    for (int sp = 0; sp < S; ++sp) {
      const float wgt = expf(part_lse(sp) - lse);
      const float *src = p.o_part + (((size_t)sp * p.total_q + row) * p.h_q + head) * DV;
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[c] = fmaf(wgt, src[lane + 32 * c], acc[c]);
    }
  }
  T *dst = static_cast<T *>(p.out) + ((size_t)row * p.h_q + head) * DV;
#pragma unroll
  for (int c = 0; c < NC; ++c) dst[lane + 32 * c] = from_f32<T>(acc[c]);
  if (lane == 0 && p.lse) p.lse[(size_t)head * p.total_q + row] = lse;
}

template <int DV>
cudaError_t launch_combine(const Params &p, cudaStream_t st) {
  const long long pairs = (long long)p.total_q * p.h_q;
  if (pairs == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((pairs + 7) / 8);
  if (p.dtype == VLF_BF16) split_combine_kernel<DV, true><<<blocks, 256, 0, st>>>(p);
  else split_combine_kernel<DV, false><<<blocks, 256, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

// Launches kern with programmatic stream serialization when the grid is small (fewer CTAs than
// SMs): its CTAs may then be made resident while the kernel ahead of them in the stream runs and
// start the moment it finishes (the kernels wait for it before any global read), instead of
// paying the launch latency after it -- microseconds that a small problem's whole kernel is made
// of.  Larger grids launch normally (their first wave could only wait on busy SMs).
cudaError_t launch_kernel(const void *kern, dim3 grid, int threads, int smem, cudaStream_t st,
                          void **args) {
  static int num_sms = [] {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    return n;
  }();
  const long long ctas = (long long)grid.x * grid.y * grid.z;
  if (num_sms <= 0 || ctas >= num_sms) {
    const cudaError_t e = cudaLaunchKernel(kern, grid, dim3(threads), args, (size_t)smem, st);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, kern, args);
}

PFN_cuTensorMapEncodeTiled_v12000 driver_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

// Every argument of one encode, zero-padded so that two keys compare with memcmp.
struct TmapKey {
  void *base;
  cuuint64_t dims[3], strides[2];
  cuuint32_t box[3], es[3];
  uint32_t dtype, rank, interleave, swizzle, l2, oob;
};
struct TmapEntry {
  CUtensorMap map;
  TmapKey key;
  bool valid;
};
// Encoded maps of recent calls, per host thread (no locking): a call that repeats a tensor's
// address, shape and box -- every training or decode step -- copies its map instead of encoding
// it again (host time per call matters for small problems, whose kernels take microseconds).
thread_local TmapEntry t_tmap_cache[64];

CUresult CUDAAPI cached_encode(CUtensorMap *m, CUtensorMapDataType dt, cuuint32_t rank, void *base,
                               const cuuint64_t *dims, const cuuint64_t *strides,
                               const cuuint32_t *box, const cuuint32_t *es,
                               CUtensorMapInterleave il, CUtensorMapSwizzle sw,
                               CUtensorMapL2promotion l2, CUtensorMapFloatOOBfill oob) {
  if (rank < 1 || rank > 3) return driver_encode_fn()(m, dt, rank, base, dims, strides, box, es, il, sw, l2, oob);
  TmapKey k;
  memset(&k, 0, sizeof(k));
  k.base = base;
  for (cuuint32_t i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
    k.es[i] = es[i];
    if (i + 1 < rank) k.strides[i] = strides[i];
  }
  k.dtype = (uint32_t)dt; k.rank = rank; k.interleave = (uint32_t)il; k.swizzle = (uint32_t)sw;
  k.l2 = (uint32_t)l2; k.oob = (uint32_t)oob;
  uint64_t h = reinterpret_cast<uint64_t>(base) >> 4;
  for (cuuint32_t i = 0; i < rank; ++i) h = h * 0x9E3779B97F4A7C15ull + dims[i] * 131 + box[i];
  TmapEntry &e = t_tmap_cache[(h ^ (h >> 29)) & 63];
  if (e.valid && memcmp(&e.key, &k, sizeof(k)) == 0) {
    *m = e.map;
    return CUDA_SUCCESS;
  }
  const CUresult r = driver_encode_fn()(m, dt, rank, base, dims, strides, box, es, il, sw, l2, oob);
  if (r == CUDA_SUCCESS) {
    e.map = *m;
    e.key = k;
    e.valid = true;
  }
  return r;
}

// The encoder the map builders below use: the driver's cuTensorMapEncodeTiled behind the cache.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() { return driver_encode_fn() ? cached_encode : nullptr; }

}  // namespace

// 2-D map over a [rows, cols] row-major 16-bit matrix with row pitch `pitch_elems`; box of 64
// columns x box_rows rows, 128-byte swizzle (the layout the MMA descriptors above expect).
bool make_tmap_16bit(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols,
                     uint64_t pitch_elems, uint32_t box_rows, int is_bf16) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc || rows == 0 || cols == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_elems * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   2, const_cast<void *>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D map over a [rows, cols] row-major fp32 matrix with row pitch `pitch_elems`; box of 32
// columns (128 bytes) x box_rows rows, 128-byte swizzle (the K-major tf32 operand layout).
bool make_tmap_f32(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols,
                   uint64_t pitch_elems, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc || rows == 0 || cols == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_elems * 4};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D map over the bias as [total_q][bias_heads x max_kv] fp32: box {32 columns, box_rows rows}
// (128-byte rows), optionally 128-byte swizzled (threads that read along a row then take chunk
// c at c ^ (row mod 8)).
bool make_tmap_bias(CUtensorMap *m, const float *base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows, bool swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc || rows == 0 || cols == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool tc_forward_supported(const Params &p) {
  if (p.dtype != VLF_F16 && p.dtype != VLF_BF16) return false;
  const bool shape = (p.d_qk == 64 && p.d_v == 64) || (p.d_qk == 96 && p.d_v == 96) ||
                     (p.d_qk == 128 && p.d_v == 128) || (p.d_qk == 192 && p.d_v == 128) ||
                     (p.d_qk == 256 && p.d_v == 256);
  return shape;
}

namespace {
// 3-D map over Q as [tokens][heads][D] (16-bit): box {64 columns, box_heads, box_tokens},
// 128-byte swizzle -- 128 dense 128-byte rows (token-major, head-minor) as a 2-D box gives.
bool make_tmap_q3(CUtensorMap *m, const void *base, uint64_t tokens, uint64_t heads, uint64_t d,
                  uint32_t box_heads, uint32_t box_tokens, int is_bf16) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc || tokens == 0 || heads == 0 || d == 0) return false;
  cuuint64_t dims[3] = {d, heads, tokens};
  cuuint64_t strides[2] = {d * 2, heads * d * 2};
  cuuint32_t box[3] = {64, box_heads, box_tokens};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   3, const_cast<void *>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The kernel instantiation for a dtype and bias kind (0 none, 1 rows from global memory, 2 TMA
// tiles: unpacked, unsplit, one tile per CTA only).
// The chosen kernel and whether it takes the full map set (FwdMaps) or Q, K, V alone.
struct FwdPick {
  const void *kern;
  bool full;
};
template <int DQK, int DV, int NK, int NV, int NT, bool BF16, int BIAS, bool PACK, bool SPLIT>
FwdPick fwd_pick_one() {
  return {reinterpret_cast<const void *>(tc_fwd_kernel<DQK, DV, NK, NV, NT, BF16, BIAS, PACK, SPLIT>),
          std::is_same<typename FwdMapsFor<DQK, PACK, BIAS>::type, FwdMaps>::value};
}
template <int DQK, int DV, int NK, int NV, int NT, bool PACK, bool SPLIT>
FwdPick pick_fwd(bool bf, int bias_kind) {
  if constexpr (NT == 1 && !PACK && !SPLIT && DV <= 128) {
    if (bias_kind == 2)
      return bf ? fwd_pick_one<DQK, DV, NK, NV, NT, true, 2, false, false>()
                : fwd_pick_one<DQK, DV, NK, NV, NT, false, 2, false, false>();
  }
  if (bias_kind != 0)
    return bf ? fwd_pick_one<DQK, DV, NK, NV, NT, true, 1, PACK, SPLIT>()
              : fwd_pick_one<DQK, DV, NK, NV, NT, false, 1, PACK, SPLIT>();
  return bf ? fwd_pick_one<DQK, DV, NK, NV, NT, true, 0, PACK, SPLIT>()
            : fwd_pick_one<DQK, DV, NK, NV, NT, false, 0, PACK, SPLIT>();
}

template <int DQK, int DV, int NK, int NV, int NT>
cudaError_t launch_fwd(const Params &p, cudaStream_t st) {
  using C = FwdCfg<DQK, DV, NK, NV, NT>;
  FwdMaps maps;
  const int bf = p.dtype == VLF_BF16;
  if (p.total_q == 0 || p.total_kv == 0) return simt_forward(p, st);  // nothing to stage
  // Decode-sized problems (every sequence's query rows fit one tile per kv head) pack the G
  // query heads of a kv head into one tile, so each K/V tile is read once for the group.
  const bool pack = NT == 1 && p.group >= 2 && 128 % p.group == 0 && p.max_q * p.group <= 128 &&
                    !(p.flags & VLF_FLAG_NO_PACK);
  // a latent head with split operands: q / k hold the 128-wide nope parts
  const bool lat = DQK == 192 && p.latent;
  const uint64_t qw = lat ? 128 : DQK;
  if (lat && (!make_tmap_16bit(&maps.q_rope, p.q_rope, p.total_q, (uint64_t)p.h_q * 64, (uint64_t)p.h_q * 64, 128, bf) ||
              !make_tmap_16bit(&maps.k_rope, p.k_rope, p.total_kv, (uint64_t)p.rope_heads * 64,
                               (uint64_t)p.rope_heads * 64, kBN, bf)))
    return cudaErrorInvalidValue;
  if (!make_tmap_16bit(&maps.q, p.q, p.total_q, (uint64_t)p.h_q * qw, (uint64_t)p.h_q * qw, 128, bf) ||
      !make_tmap_16bit(&maps.k, p.k, p.total_kv, (uint64_t)p.h_kv * qw, (uint64_t)p.h_kv * qw, kBN, bf) ||
      !make_tmap_16bit(&maps.v, p.v, p.total_kv, (uint64_t)p.h_kv * DV, (uint64_t)p.h_kv * DV, kBN, bf))
    return cudaErrorInvalidValue;
  if (pack && !make_tmap_q3(&maps.q3, p.q, p.total_q, p.h_q, DQK, p.group, 128 / p.group, bf))
    return cudaErrorInvalidValue;
  if (!pack) maps.q3 = maps.q;
  if (!lat) { maps.q_rope = maps.q; maps.k_rope = maps.k; }
  const bool pair_heads = NT == 2 && (p.group % 2 == 0);
  const int rows_per_cta = pack ? 128 / p.group : (NT == 1 || pair_heads ? 128 : 256);
  const unsigned blocks = (unsigned)((p.max_q + rows_per_cta - 1) / rows_per_cta);
  const unsigned heads = pack ? p.h_kv : (pair_heads ? p.h_q / 2 : p.h_q);
  if (blocks == 0) return cudaSuccess;
  // split-KV parts (NT = 1): grid z enumerates (sequence, part); their bias rows are read with
  // per-thread loads (the parts keep two CTAs per SM)
  const bool split = NT == 1 && p.kv_splits > 1;
  // A bias whose rows are 16-byte aligned goes through TMA tiles (one unpacked tile per CTA; the
  // ring takes the room of a second CTA per SM); others are read row by row.
  const bool bias_tma = NT == 1 && DV <= 128 && !pack && !split && p.bias != nullptr && p.max_kv % 4 == 0 &&
                        (reinterpret_cast<uintptr_t>(p.bias) & 15u) == 0;
  if (bias_tma && !make_tmap_bias(&maps.bias, p.bias, p.total_q, (uint64_t)p.bias_heads * p.max_kv, 128, true))
    return cudaErrorInvalidValue;
  if (!bias_tma) maps.bias = maps.q;
  // a head-broadcast bias: the heads of one row block run together and share its tiles in L2
  Params pl = p;
  pl.heads_fast = p.bias != nullptr && p.bias_heads == 1 && !pack;
  const unsigned zdim = (unsigned)p.num_seqs * (split ? (unsigned)p.kv_splits : 1u);
  if (zdim > 65535u) return cudaErrorInvalidValue;
  const dim3 grid = pl.heads_fast ? dim3(heads, blocks, zdim) : dim3(blocks, heads, zdim);
  FwdPick kern;
  int smem = C::SMEM;
  const int bias_kind = p.bias ? (bias_tma ? 2 : 1) : 0;
  if constexpr (NT == 1) {
    if (split)
      kern = pack ? pick_fwd<DQK, DV, NK, NV, NT, true, true>(bf, bias_kind)
                  : pick_fwd<DQK, DV, NK, NV, NT, false, true>(bf, bias_kind);
    else
      kern = pack ? pick_fwd<DQK, DV, NK, NV, NT, true, false>(bf, bias_kind)
                  : pick_fwd<DQK, DV, NK, NV, NT, false, false>(bf, bias_kind);
    if constexpr (DV <= 128)
      if (bias_tma) smem = FwdCfg<DQK, DV, NK, NV, NT, 2>::SMEM;
  } else {
    if (pack || split || bias_tma) return cudaErrorInvalidValue;
    kern = pick_fwd<DQK, DV, NK, NV, NT, false, false>(bf, bias_kind);
  }
  cudaError_t e = set_smem_once(kern.kern, smem);
  if (e != cudaSuccess) return e;
  FwdMapsPlain plain{maps.q, maps.k, maps.v};
  void *args[2] = {kern.full ? static_cast<void *>(&maps) : static_cast<void *>(&plain), &pl};
  e = launch_kernel(kern.kern, grid, C::THREADS, smem, st, args);
  if (e == cudaSuccess) count_launch();
  return e;
}
}  // namespace

bool tc_forward_splittable(const Params &p) {
  return tc_forward_supported(p) && p.d_qk == p.d_v;  // one query tile per CTA
}

cudaError_t tc_forward_split(const Params &p, cudaStream_t st) {
  if (!tc_forward_splittable(p) || p.kv_splits < 2 || !p.o_part || !p.lse_part) return cudaErrorInvalidValue;
  cudaError_t e = tc_forward(p, st);
  if (e != cudaSuccess || p.total_q == 0 || p.total_kv == 0) return e;  // (empty: plain path ran)
  if (p.d_v == 64) return launch_combine<64>(p, st);
  if (p.d_v == 96) return launch_combine<96>(p, st);
  if (p.d_v == 256) return launch_combine<256>(p, st);
  return launch_combine<128>(p, st);
}

// Parts per CTA band: split when the unsplit grid leaves SMs idle (fewer CTAs than resident
// slots: two one-tile CTAs per SM, one at width 256), into as many parts as keep the grid within
// one such wave,
// each part at least four KV tiles long (a part costs a prologue, an fp32 partial write and a
// read in the combine).  Between one and three waves, a grid whose last wave is partly empty
// (under 95% wave efficiency) is cut into 2 or 3 parts, whichever fills its waves better (the
// fewer on a tie), each part at least 16 KV tiles: shorter CTAs shorten the partly occupied
// tail (measured on decode rows x 8 kv heads against 4096-16384 keys: 5-28% faster).
int fwd_num_splits(int num_seqs, int max_q, int max_kv, int h_q, int h_kv, int d_qk, int d_v,
                   int dtype, unsigned flags, int num_sms) {
  if ((dtype != VLF_F16 && dtype != VLF_BF16) || (flags & VLF_FLAG_FORCE_SIMT)) return 1;
  if (d_qk != d_v || (d_qk != 64 && d_qk != 96 && d_qk != 128 && d_qk != 256)) return 1;
  if (num_seqs < 1 || max_q < 1 || max_kv < 1 || h_kv < 1 || h_q % h_kv != 0 || num_sms < 1) return 1;
  const int group = h_q / h_kv;
  const bool pack = group >= 2 && 128 % group == 0 && (long long)max_q * group <= 128 &&
                    !(flags & VLF_FLAG_NO_PACK);
  const long long rows = pack ? 128 / group : 128;
  const long long ctas = (max_q + rows - 1) / rows * (pack ? h_kv : h_q) * (long long)num_seqs;
  const long long slots = (d_v == 256 ? 1LL : 2LL) * num_sms;  // CTAs resident per SM
  const long long tiles = ((long long)max_kv + kBN - 1) / kBN;
  if (ctas >= slots) {
    if (ctas >= 3 * slots) return 1;
    // wave efficiency of sp parts: ctas * sp / (slots * waves), compared by cross-multiplying
    auto waves = [&](long long sp) { return (ctas * sp + slots - 1) / slots; };
    if (ctas * 100 >= 95 * slots * waves(1)) return 1;
    int best = 1;
    for (int sp = 2; sp <= 3; ++sp) {
      if (tiles < 16 * sp || (long long)sp * num_seqs > 65535) break;
      if (best == 1 || ctas * sp * waves(best) > ctas * best * waves(sp)) best = sp;
    }
    return best;
  }
  const long long by_grid = slots / ctas;
  const long long by_len = tiles / 4;
  long long sp = by_grid < by_len ? by_grid : by_len;
  if (sp > 64) sp = 64;
  if (sp * num_seqs > 65535) sp = 65535 / num_seqs;
  return sp < 2 ? 1 : (int)sp;
}

cudaError_t tc_forward(const Params &p, cudaStream_t st) {
  if (p.d_qk == 64) return launch_fwd<64, 64, 3, 3, 1>(p, st);
  if (p.d_qk == 96) return launch_fwd<96, 96, 3, 2, 1>(p, st);
  if (p.d_qk == 128) return launch_fwd<128, 128, 3, 2, 1>(p, st);
  if (p.d_qk == 256) return launch_fwd<256, 256, 3, 2, 1>(p, st);
  return launch_fwd<192, 128, 3, 3, 2>(p, st);
}

}  // namespace vlf
