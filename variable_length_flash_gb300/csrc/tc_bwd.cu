// Tensor-core backward (sm_103a): the FlashAttention-2 backward that triton-msl part 2
// ("Beyond softmax") describes -- recompute S per tile, P = exp(S - LSE), dV += P^T dO,
// dP = dO V^T, dS = P o (dP - D) with D = rowsum(dO o O), dK += dS^T Q, dQ += dS K -- split into
// a dK/dV kernel and a dQ kernel so that no output is accumulated with atomics (results are
// deterministic), with tcgen05 MMAs accumulating in TMEM and TMA-staged tiles.
//
// One kernel body serves both (MODE):
//   dK/dV: a CTA owns 128 keys of one kv head (K, V tiles stay in shared memory) and walks the
//          IR-row Q / dO tiles ("items") of every query head of its GQA group that can see those
//          keys.  S^T = K Q^T and dP^T = V dO^T land in TMEM (lanes = keys); the compute warps
//          turn them into 16-bit P^T and dS^T in TMEM; dV += P^T dO and dK += dS^T Q take their A
//          operand from TMEM.  LSE and D of the item's query columns come through smem.
//   dQ:    a CTA owns 128 query rows of one head (Q, dO stay in shared memory) and walks the
//          IR-key K / V items of its band: S = Q K^T, dP = dO V^T, dS in TMEM, dQ += dS K.
// Item width IR: an MMA of 128 x N x 16 with both operands in shared memory runs at full rate
// only for N >= 128 (at N = 64 it is limited by shared-memory bandwidth), but 128-row items
// leave TMEM room for one S/dP buffer only.  Measured, the dK/dV kernel runs two buffers of
// 64-row items (the next item's products overlap this item's elementwise pass; the latent head,
// QK width 192, whose dK accumulator leaves room for one buffer, runs one); the plain dQ kernel
// runs 128-key items with dS written over S (two S buffers, one dP buffer: mode kDqS), and
// 64-key items where a bias or the latent head takes the TMEM columns (kDq).  Width 256 splits
// the key-tile work into a dV pass and a dK pass (kDv, kDk).
// Warp roles (384 threads): warp 0 stages tiles with TMA and, with all its lanes, the item's LSE
// and D columns into the same shared-memory stage; warps 1, 11 and 10 issue the S, dP and
// accumulation MMAs (warp 1 also owns the TMEM allocation); warps 2-9 are two compute
// warpgroups, each owning half of the item's columns (one thread per TMEM lane).  Each warpgroup
// writes its 16-bit P / dS over its own S / dP columns.
// MMA order: after item n's P / dS are ready its accumulations are issued; the products of the
// item that next uses n's columns (n + NBUF) follow as soon as those columns are released: S
// once accumulation 0 (dK/dV: dV += P^T dO) has read P^T (dQ: once the compute warps have read
// S), dP once the last accumulation has read dS.  With one 32-column chunk per compute thread
// (all but the 128-key dQ items) S and dP complete on separate barriers: the compute warps form
// P from S while dP still runs, then wait for dP to form dS; in the dK/dV kernel P^T goes to the
// dV accumulation before dS^T is formed.
// Tiles outside the causal / window band are skipped (they contribute exact zeros).  Every wait
// is bounded.
#include <cudaTypedefs.h>
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace vlf {

bool make_tmap_16bit(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols,
                     uint64_t pitch_elems, uint32_t box_rows, int is_bf16);
bool make_tmap_bias(CUtensorMap *m, const float *base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows, bool swizzle);

namespace {

using namespace tc;

// kDq keeps dS in the dP columns and double-buffers S and dP; kDqS writes dS over the S columns
// instead, so the single dP buffer is free as soon as the compute warps have loaded it and the
// next item's dP can run during this item's elementwise pass (S stays double-buffered).
constexpr int kDkdv = 0, kDq = 1, kDqS = 2;
// Width 256: the dK and dV accumulators (256 columns each) fill TMEM, so the key-tile work runs
// as two kernels -- kDv (S^T, P^T, dV += P^T dO) and kDk (S^T, dP^T, dS^T, dK += dS^T Q) --
// each with room for its product buffers (one S recompute more than kDkdv).
constexpr int kDv = 3, kDk = 4;

struct BwdMaps {
  CUtensorMap outer0, outer1, inner0, inner1, bias;
  // latent head with split operands: the rope tensors behind outer0 / inner0 (64 columns)
  CUtensorMap outer0_rope, inner0_rope;
  // outputs stored by TMA boxes {64 columns, 128 rows}: dV, dK (dK/dV); dV (kDv); dK (kDk); dQ
  CUtensorMap out0, out1;
};

// outer0/outer1: K, V (dK/dV) or Q, dO (dQ), 128 rows.  inner0/inner1: Q, dO (dK/dV) or K, V
// (dQ), IR rows per item.  NBS: stages of the bias ring (0: no bias through TMA).
template <int MODE, int DQK, int DV, int IR, int NBUF, int NSTAGE, int NSTAGE1, int NBS = 0>
struct BwdCfg {
  // key-tile CTAs (outer tiles K / V, inner items Q / dO) and which products / accumulations run
  static constexpr bool KEYS = MODE == kDkdv || MODE == kDv || MODE == kDk;
  static constexpr bool HAS_DP = MODE != kDv;              // dP (dK/dV: dP^T) product
  static constexpr bool HAS_DV = MODE == kDkdv || MODE == kDv;  // dV += P^T dO
  static constexpr bool HAS_LAST = MODE != kDv;            // dK or dQ accumulation
  // 64-col blocks of tensors 0 / 1; a width that is not a multiple of 64 (96) is padded to
  // whole blocks (next head's values or zero fill): products step over the real width along K,
  // accumulations run at the padded N and the extra accumulator columns are never stored
  static constexpr int KB0 = (DQK + 63) / 64, KB1 = (DV + 63) / 64;
  static constexpr int NQ_PAD = KB0 * 64, NV_PAD = KB1 * 64;
  static constexpr int OBLK = 128 * 128, IBLK = IR * 128;  // bytes per 64-col block
  // OT (the width-256 passes): the outer tile that is a product's A operand goes to TMEM (columns
  // OTA on) -- K for the dV pass's S^T (OT_K), V for the dK pass's dP^T (OT_V) -- so that product
  // reads only its inner tile from shared memory.  In the dK pass an item's S^T and dP^T share
  // one 64-column region (SR): dP^T overwrites S^T once the compute warps have loaded it, dS^T
  // overwrites dP^T, and the next item of the region waits for dK to have read dS^T; two regions
  // fit beside the 256-column dK accumulator and V.  The tile lands in
  // ring-0 slots 1 .. (its 64 KB), the compute warps copy their rows into TMEM, and those slots
  // then take Q items: the rings get the tile's shared memory.
  static constexpr bool OT_K = MODE == kDv && DQK == 256, OT_V = MODE == kDk;
  static constexpr bool OT = OT_K || OT_V;
  static constexpr int OT_KB = OT_K ? KB0 : KB1;  // 64-column blocks of the tile
  static constexpr int O0_BYTES = OT_K ? 0 : KB0 * OBLK;
  static constexpr int O1_BYTES = MODE == kDv || OT_V ? 0 : KB1 * OBLK;  // kDv: no V
  static constexpr int I0_BYTES = KB0 * IBLK, I1_BYTES = KB1 * IBLK;
  // two rings of inner tiles: ring 0 (Q for dK/dV, K for dQ; NSTAGE slots) and ring 1 (dO for
  // dK/dV, V for dQ; NSTAGE1 slots), each slot released as soon as its last reader is done
  static constexpr int OFF_O0 = 0, OFF_O1 = O0_BYTES, OFF_IN0 = O0_BYTES + O1_BYTES;
  static constexpr int OFF_IN1 = OFF_IN0 + NSTAGE * I0_BYTES;
  // per ring-0 slot: the item's IR columns as IR/2 pairs {-LSE2_c, -LSE2_c+1, -D_c, -D_c+1}
  // (dK/dV only)
  static constexpr int PAIRS = KEYS ? IR / 2 : 0;
  static constexpr int OFF_LD = OFF_IN1 + NSTAGE1 * I1_BYTES;
  // dK/dV with TMA-staged bias: per ring-0 slot the item's rows' finite-bias intervals as IR/2
  // pairs {lo_c, hi_c, lo_c+1, hi_c+1} (bias bands; pure items are masked by them).  The bias
  // is staged through TMA at QK widths up to 128 only.
  static constexpr int BD_BYTES = KEYS && NQ_PAD <= 128 ? NSTAGE * PAIRS * 16 : 0;
  static constexpr int OFF_BD = OFF_LD + NSTAGE * PAIRS * 16;
  // dK/dV: per ring-0 slot the kept item's candidate index and flags (1: its rows are pure
  // 0 / -inf intervals, 2: every row sees every key of the tile) for the compute warps
  static constexpr int IS_BYTES = KEYS ? NSTAGE * 8 : 0;
  static constexpr int OFF_IS = OFF_BD + BD_BYTES;
  // bias ring: per item its 128 x IR fp32 tile as 32-column boxes.  dK/dV: 4 boxes {32 keys, IR
  // query rows}, unswizzled (the 32 keys of a warp read one 128-byte row at a time); dQ: IR / 32
  // boxes {32 keys, 128 query rows}, 128-byte swizzled (each thread reads along its own row).
  static constexpr int BIAS_BOX = KEYS ? 32 * IR * 4 : 32 * 128 * 4;
  static constexpr int BIAS_STAGE = 128 * IR * 4;
  static constexpr int NBS_ = NBS > 0 ? NBS : 1;  // (a nonzero divisor where there is no ring)
  // (swizzled boxes start 1024-byte aligned, unswizzled ones 128-byte aligned)
  static constexpr int B_ALIGN = KEYS ? 128 : 1024;
  static constexpr int OFF_B = (OFF_IS + IS_BYTES + B_ALIGN - 1) & ~(B_ALIGN - 1);
  static constexpr int OFF_BAR = OFF_B + NBS * BIAS_STAGE;
  // barriers: outer_full, in_full[NSTAGE], in_empty[NSTAGE] (ring 0), in1_full[NSTAGE1],
  // in1_empty[NSTAGE1] (ring 1), s_full[NBUF] (S done; and dP unless SPLIT: two arrivals),
  // p_ready[NBUF], acc0_done[NBUF] (dV), acc_done[NBUF] (dK or dQ: the item's last
  // accumulation), drain[3] (one per MMA-issuing warp), dp_free (kDqS)
  static constexpr int B_OUT = 0, B_IF = 1, B_IE = B_IF + NSTAGE, B_IF1 = B_IE + NSTAGE;
  static constexpr int B_IE1 = B_IF1 + NSTAGE1, B_S = B_IE1 + NSTAGE1;
  static constexpr int B_P = B_S + NBUF, B_D0 = B_P + NBUF, B_D = B_D0 + NBUF, B_DRAIN = B_D + NBUF;
  static constexpr int B_PF = B_DRAIN + 3;  // kDqS: the compute warps have loaded dP
  static constexpr int B_QT = B_PF + 1;     // QT, OT: the outer tiles' rows are in TMEM
  static constexpr int B_BF = B_QT + 1, B_BE = B_BF + NBS;  // bias full / empty
  // dp_full[NBUF] (SPLIT: dP done), ds_ready[NBUF] (P_EARLY: dS^T written; p_ready then means P^T)
  static constexpr int B_DP = B_BE + NBS, B_DS = B_DP + NBUF;
  // s_loaded[NBUF] (SR): the compute warps have loaded S from the region
  static constexpr int B_SL = B_DS + NBUF;
  static constexpr int NBAR = B_SL + NBUF;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // (no alignment slack: the dynamic shared window starts 1024-byte aligned, checked in-kernel)
  static constexpr int SMEM = OFF_MISC + 16;
  // TMEM: accumulators first, then NBUF x (S IR cols, dP IR cols); kDqS: NBUF S buffers, then
  // one dP buffer.  kDv / kDk: the one accumulator (dV / dK, up to 256 columns) at 0.
  static constexpr uint32_t ACC0 = 0;                       // dV (dK/dV, kDv) or dQ (dQ)
  static constexpr uint32_t ACC1 = MODE == kDk ? 0 : 128;   // dK (dK/dV, kDk)
  static constexpr uint32_t BUF = MODE == kDkdv ? 128 + NQ_PAD
                                  : (MODE == kDv ? NV_PAD : (MODE == kDk || MODE == kDqS ? NQ_PAD : 256));
  static constexpr bool SR = MODE == kDk;
  __host__ __device__ static constexpr uint32_t s_col(int b) {
    return MODE == kDqS || MODE == kDv || SR ? BUF + IR * b : BUF + 2 * IR * b;  // (kDv: no dP columns)
  }
  __host__ __device__ static constexpr uint32_t dp_col(int b) {
    return MODE == kDqS ? BUF + NBUF * IR : (SR ? BUF + IR * b : BUF + 2 * IR * b + IR);
  }
  // kDq: the outer Q (QT_Q, widths up to 128) and dO (QT_DO) tiles are copied once into the
  // TMEM columns between the accumulator and the S / dP buffers, 16-bit pairs along the row, and
  // are the A operands of S and dP from there: those products then read only their inner K / V
  // tile from shared memory (with both operands in shared memory a 64-key product is bound by
  // its reads).  QK width 192: the 192-column accumulator leaves room for dO only.  kDqS has no
  // free columns.
  static constexpr bool QT_Q = MODE == kDq && NQ_PAD <= 128 && NV_PAD <= 128;
  static constexpr uint32_t QA = 128, DOA = QT_Q ? 128 + NQ_PAD / 2 : NQ_PAD;
  static constexpr bool QT_DO = MODE == kDq && NV_PAD <= 128 && DOA + NV_PAD / 2 <= BUF;
  static constexpr bool QT = QT_Q || QT_DO;
  static_assert(!QT_Q || QT_DO, "TMEM columns of the A operands");
  // the A operands sit past the accumulator, [0, NQ_PAD), and end before the S / dP buffers
  static_assert(!QT_Q || (QA >= NQ_PAD && QA + NQ_PAD / 2 <= DOA), "TMEM columns of the Q operand");
  static_assert(!QT_DO || (DOA >= NQ_PAD && DOA + NV_PAD / 2 <= BUF), "TMEM columns of the dO operand");
  static constexpr int HALF = IR / 2;      // columns per compute warpgroup
  static constexpr int CHUNKS = HALF / 32;  // 32-column chunks per compute thread
  // SPLIT (one 32-column chunk per compute thread): S and dP complete on separate barriers, and
  // an item whose dP has not landed with S has its P formed first, its dP loaded after.  With two
  // chunks (128-column dQ items) S and dP are awaited and loaded together, chunk by chunk.
  // P_EARLY (dK/dV): P^T goes to the dV accumulation before dS^T is formed.
  static constexpr bool SPLIT = HAS_DP && CHUNKS == 1;
  static constexpr bool P_EARLY = HAS_DV && HAS_DP;
  static_assert(!P_EARLY || SPLIT, "P^T released early needs the split form");
  static_assert((MODE == kDqS ? BUF + (NBUF + 1) * IR : BUF + NBUF * (MODE == kDv || SR ? 1 : 2) * IR) <= 512,
                "TMEM columns");
  static constexpr uint32_t OTA = BUF + NBUF * (MODE == kDv || SR ? 1 : 2) * IR;  // OT: the tile's rows
  static_assert(!OT || (OTA + OT_KB * 32 <= 512 && (NSTAGE - 1) * I0_BYTES >= OT_KB * OBLK),
                "OT: TMEM columns of the tile, ring-0 slots that stage it");
  static_assert(SMEM <= 232448, "shared memory");
  static_assert((MODE != kDkdv || NV_PAD <= 128) && NV_PAD <= 256 && NQ_PAD <= 256 && DQK % 32 == 0 &&
                DV % 32 == 0, "head widths");
  static_assert(IR == 64 || IR == 128, "item rows");
  static_assert(NBUF == 1 || IR == 64 || MODE == kDqS, "double buffering only with 64-row items");
};


// BF16: element type of the 16-bit tensors (bf16, else fp16), fixed at compile time so the
// per-element conversions carry no runtime branch.
// BIAS: 0 none; 1 the compute threads load their bias values from global memory; 2 the producer
// stages each item's bias tile through the NBS-stage ring; 3 a bias whose rows (those this CTA
// works on) are all 0 / -inf intervals: masked by the bias bands, no bias value read (a separate
// instantiation each, so that kernels without a bias carry none of its code or registers).
template <int MODE, int DQK, int DV, int IR, int NBUF, int NSTAGE, int NSTAGE1, int NBS, bool BF16,
          int BIAS>
__device__ __forceinline__ void tc_bwd_body(const BwdMaps &maps, const Params &p) {
  using C = BwdCfg<MODE, DQK, DV, IR, NBUF, NSTAGE, NSTAGE1, NBS>;
  static_assert((BIAS == 2) == (NBS > 0), "the bias ring serves TMA-staged bias only");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int s = blockIdx.z;
  Seq sq;
  if (!load_seq(p, s, sq)) return;
  const int off = sq.kv_len - sq.q_len;
  // the CTA's outer tile and its item range (items start at multiples of IR)
  int tile0, head_outer, hk, n_items, lo = 0, nq_tiles = 0;
  bool cta_pure = false;  // dQ with bias bands: mask by the rows' intervals, bias not read
  // heads_fast (a head-broadcast bias): grid x enumerates heads, y the 128-row tiles, so that the
  // heads of one tile run together and share its bias tiles in L2
  const int bxr = p.heads_fast ? (int)blockIdx.y : (int)blockIdx.x;
  const int gx = p.heads_fast ? (int)gridDim.y : (int)gridDim.x;
  const int byh = p.heads_fast ? (int)blockIdx.x : (int)blockIdx.y;
  if (C::KEYS) {
    tile0 = bxr * 128;  // first key
    hk = byh;
    head_outer = hk;
    if (tile0 >= sq.kv_len) return;
    int qlo = 0, qhi = 0;
    if (sq.q_len > 0) {
      q_band(tile0, min(tile0 + 128, sq.kv_len), sq.q_len, sq.kv_len, p.causal, p.window, qlo, qhi);
      if (p.flags & VLF_FLAG_NO_SKIP) { qlo = 0; qhi = sq.q_len; }
    }
    lo = (qlo / IR) * IR;
    nq_tiles = qhi > qlo ? (qhi - lo + IR - 1) / IR : 0;
    n_items = nq_tiles * p.group;
  } else {
    const int bx = p.causal ? gx - 1 - bxr : bxr;
    tile0 = bx * 128;  // first query row
    head_outer = byh;
    hk = head_outer / p.group;
    if (tile0 >= sq.q_len) return;
    int klo = 0, khi = 0;
    if (sq.kv_len > 0) {
      kv_band(tile0, min(tile0 + 128, sq.q_len), sq.q_len, sq.kv_len, p.causal, p.window, klo, khi);
      if (p.flags & VLF_FLAG_NO_SKIP) { klo = 0; khi = sq.kv_len; }
    }
    // bias bands: only the keys some row of the tile has a finite bias value for (the others
    // hold masked pairs alone); cta_pure: every row's bias is 0 over its finite interval
    if (BIAS != 0 && p.bias_blocks && khi > klo) {
      const int hb = p.bias_heads == 1 ? 0 : head_outer;
      const int4 *bb = p.bias_blocks + (size_t)hb * p.total_q + sq.q0 + tile0;
      const int4 e0 = __ldg(bb);
      int blo = e0.x, bhi = e0.y, pure = e0.z >= 0;
      if (tile0 + 64 < sq.q_len) {
        const int4 e1 = __ldg(bb + 64);
        if (e1.y > e1.x) {
          blo = bhi > blo ? min(blo, e1.x) : e1.x;
          bhi = max(bhi, e1.y);
        }
        pure &= e1.z >= 0;
      }
      if (bhi > blo) {
        klo = max(klo, blo);
        khi = min(khi, bhi);
      }
      if (bhi <= blo || khi <= klo) khi = klo;
      cta_pure = (BIAS == 2 || BIAS == 3) && pure != 0;
    }
    lo = (klo / IR) * IR;
    n_items = khi > klo ? (khi - lo + IR - 1) / IR : 0;
  }

  // dK/dV with bias bands: the items (query head, 64-row block) whose rows have a finite bias
  // value among this tile's keys; the others hold masked pairs alone and are skipped (exact).
  // Every role walks the candidates in order and counts the kept ones, which index the rings
  // and buffers; n_kept replaces n_items as the length of the pipeline.
  const int4 *item_bands = (C::KEYS && BIAS != 0) ? p.bias_blocks : nullptr;
  auto item_band = [&](int n) -> int4 {
    const int hb = p.bias_heads == 1 ? 0 : hk * p.group + n / nq_tiles;
    return __ldg(item_bands + (size_t)hb * p.total_q + sq.q0 + lo + (n % nq_tiles) * IR);
  };
  auto item_kept = [&](const int4 &e) { return e.y > e.x && e.x < tile0 + 128 && e.y > tile0; };
  // a kept item's flags: 1 its rows are pure 0 / -inf intervals (masked by them, no bias value
  // read), 2 besides, every one of its rows sees every key of this tile (no mask from the bias)
  auto item_flags = [&](const int4 &e) {
    // (pure items are masked by their rows' intervals, staged per ring slot: BD_BYTES > 0)
    if ((BIAS != 2 && BIAS != 3) || C::BD_BYTES == 0 || !p.bias_rows || e.z < 0) return 0;
    return 1 | ((e.z <= tile0 && e.w >= min(tile0 + 128, sq.kv_len)) ? 2 : 0);
  };
  int n_kept = n_items;
  if (item_bands) {
    n_kept = 0;
    for (int b0 = 0; b0 < n_items; b0 += (int)blockDim.x) {
      const int n = b0 + (int)threadIdx.x;
      n_kept += __syncthreads_count(n < n_items && item_kept(item_band(n)));
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
  const uint32_t sO0 = base + C::OFF_O0, sO1 = base + C::OFF_O1;
  const uint32_t sIn0 = base + C::OFF_IN0, sIn1 = base + C::OFF_IN1, sBias = base + C::OFF_B;
  float4 *ldbuf = reinterpret_cast<float4 *>(gbase + C::OFF_LD);  // [stage][IR/2 column pairs]
  int4 *bdbuf = reinterpret_cast<int4 *>(gbase + C::OFF_BD);      // [stage][IR/2 column pairs]
  int2 *islot = reinterpret_cast<int2 *>(gbase + C::OFF_IS);      // [stage] {candidate, flags}
  const uint32_t bar0 = base + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(gbase + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + C::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_OUT), 1);
    // in_full: the TMA bytes plus 33 arrivals (lane 0's expect_tx and every producer lane after
    // writing its LSE / D pairs); p_ready: all 256 compute threads
    for (int i = 0; i < NSTAGE; ++i) { mbar_init(bar(C::B_IF + i), 33); mbar_init(bar(C::B_IE + i), 1); }
    for (int i = 0; i < NSTAGE1; ++i) { mbar_init(bar(C::B_IF1 + i), 1); mbar_init(bar(C::B_IE1 + i), 1); }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(bar(C::B_S + b), C::HAS_DP && !C::SPLIT ? 2 : 1);  // S (and dP) done
      mbar_init(bar(C::B_P + b), 256);
      mbar_init(bar(C::B_D + b), 1);
      mbar_init(bar(C::B_D0 + b), 1);
    }
    for (int i = 0; i < 3; ++i) mbar_init(bar(C::B_DRAIN + i), 1);
    mbar_init(bar(C::B_PF), 256);
    mbar_init(bar(C::B_QT), 256);
    for (int b = 0; b < NBUF; ++b) mbar_init(bar(C::B_SL + b), 256);
    for (int i = 0; i < NBS; ++i) { mbar_init(bar(C::B_BF + i), 1); mbar_init(bar(C::B_BE + i), 256); }
    for (int b = 0; b < NBUF; ++b) { mbar_init(bar(C::B_DP + b), 1); mbar_init(bar(C::B_DS + b), 256); }
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
  constexpr int is_bf16 = BF16 ? 1 : 0;

  // item n -> (query head, first inner row) ; inner rows are queries (dK/dV) or keys (dQ)
  auto item_head = [&](int n) { return C::KEYS ? hk * p.group + n / nq_tiles : head_outer; };
  auto item_row = [&](int n) { return C::KEYS ? lo + (n % nq_tiles) * IR : lo + n * IR; };

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    // a latent head given as split operands (QK width 192 only): blocks 0-1 of each Q / K tile
    // come from the nope tensors (row width 128 per head), block 2 from the rope tensors
    const bool lat = DQK == 192 && p.latent;
    const int qw = lat ? 128 : DQK;
    const int rh = lat && p.rope_heads == 1 ? 0 : hk;  // the kv head's rope key
    if (n_kept > 0) {
      if (lane == 0) {
        tma_prefetch_desc(&maps.outer0);
        tma_prefetch_desc(&maps.outer1);
        tma_prefetch_desc(&maps.inner0);
        tma_prefetch_desc(&maps.inner1);
        if (BIAS == 2) tma_prefetch_desc(&maps.bias);
        if (lat) {
          tma_prefetch_desc(&maps.outer0_rope);
          tma_prefetch_desc(&maps.inner0_rope);
        }
        const int orow = (C::KEYS ? sq.k0 : sq.q0) + tile0;
        const int oh = C::KEYS ? hk : head_outer;  // head index inside the outer tensors
        mbar_expect_tx(bar(C::B_OUT), C::O0_BYTES + C::O1_BYTES + (C::OT ? C::OT_KB * C::OBLK : 0));
        const uint32_t sOT = sIn0 + C::I0_BYTES;  // OT: ring-0 slots 1 ..
        for (int c = 0; c < C::KB0; ++c) {
          const uint32_t dst = (C::OT_K ? sOT : sO0) + c * C::OBLK;
          if (lat && c == 2)  // the rope block: K's from the (possibly shared) rope key, or Q's
            tma_load_2d(dst, &maps.outer0_rope, (C::KEYS ? rh : oh) * 64, orow, bar(C::B_OUT));
          else
            tma_load_2d(dst, &maps.outer0, oh * qw + 64 * c, orow, bar(C::B_OUT));
        }
        for (int c = 0; c < (C::O1_BYTES > 0 || C::OT_V ? C::KB1 : 0); ++c)  // (kDv reads no V)
          tma_load_2d((C::OT_V ? sOT : sO1) + c * C::OBLK, &maps.outer1, oh * DV + 64 * c, orow, bar(C::B_OUT));
      }
      int issued0[NSTAGE] = {0}, issued1[NSTAGE1] = {0}, issuedb[C::NBS_] = {0};
      // dK/dV: -LSE (base 2; -inf for rows that see nothing or lie past the sequence, so P = 0)
      // and -D of item n's column pairs lane, lane + 32, ..., loaded one item ahead into
      // registers so that their global-load latency is off the producer's per-item path
      // (the raw values are kept: no instruction uses them, so nothing waits, until the write)
      constexpr int PPL = C::PAIRS > 0 ? C::PAIRS / 32 : 1;
      float rl[PPL][2], rd[PPL][2];
      // (dK/dV with bias bands and TMA-staged bias: the rows' finite-bias intervals as well)
      const bool stage_bands = (BIAS == 2 || BIAS == 3) && C::BD_BYTES > 0 && p.bias_rows != nullptr;
      int rbl[PPL][2], rbh[PPL][2];
      auto load_pairs = [&](int n) {
        const int h = item_head(n), i0 = item_row(n);
        const int hb = p.bias_heads == 1 ? 0 : h;
#pragma unroll
        for (int pp = 0; pp < PPL; ++pp) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int qi = i0 + 2 * (lane + 32 * pp) + u;
            rl[pp][u] = -INFINITY;
            rd[pp][u] = 0.f;
            rbl[pp][u] = rbh[pp][u] = 0;
            if (qi < sq.q_len) {
              const size_t gi = (size_t)h * p.total_q + sq.q0 + qi;
              rl[pp][u] = __ldg(p.lse + gi);
              rd[pp][u] = __ldg(p.rowdot + gi);
              if (stage_bands) {
                const int4 e = __ldg(p.bias_rows + (size_t)hb * p.total_q + sq.q0 + qi);
                rbl[pp][u] = e.x;
                rbh[pp][u] = e.y;
              }
            }
          }
        }
      };
      // the next kept candidate item at or after n (every candidate without bias bands)
      auto next_kept = [&](int n) {
        if (item_bands)
          while (n < n_items && !item_kept(item_band(n))) ++n;
        return n;
      };
      const int4 none = make_int4(0, 0, -1, -1);
      int n = next_kept(0);
      int4 e_n = item_bands && n < n_items ? item_band(n) : none;  // its block band
      if (C::KEYS && n < n_items) load_pairs(n);
      for (int k = 0; n < n_items; ++k) {
        const int st = k % NSTAGE, st1 = k % NSTAGE1;
        // the next candidate's band, loaded here so that its latency passes during this item's
        // waits; the walk to the next kept candidate follows below
        int n_next = n + 1;
        int4 e_next = item_bands && n_next < n_items ? item_band(n_next) : none;
        const int flags_n = item_bands ? item_flags(e_n) : 0;
        if (BIAS == 2 && !cta_pure) {
          // the item's bias tile (needed last, by the compute warps; its slot frees earliest);
          // an item whose rows' bias is 0 over their intervals (pure) needs no tile: its slot
          // is passed along without a copy
          const bool pure_item = (flags_n & 1) != 0;
          const int bs = k % C::NBS_;
          bool wb = true;
          if (lane == 0) {
            if (k >= C::NBS_) wb = mbar_wait(bar(C::B_BE + bs), ((k / C::NBS_) - 1) & 1, abort_flag, p.err);
            if (wb && pure_item) {
              mbar_arrive(bar(C::B_BF + bs));
              ++issuedb[bs];
            } else if (wb) {
              const uint32_t dst = sBias + bs * C::BIAS_STAGE;
              mbar_expect_tx(bar(C::B_BF + bs), C::BIAS_STAGE);
              // bias columns: bias head * max_seqlen_kv + sequence-local key; rows: global query
              // rows.  Boxes past the tensor are zero-filled; columns past the sequence's keys
              // and rows past its queries are masked by the compute threads.
              if (C::KEYS) {
                const int x = (p.bias_heads == 1 ? 0 : item_head(n)) * p.max_kv + tile0;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                  tma_load_2d(dst + c * C::BIAS_BOX, &maps.bias, x + 32 * c, sq.q0 + item_row(n), bar(C::B_BF + bs));
              } else {
                const int x = (p.bias_heads == 1 ? 0 : head_outer) * p.max_kv + item_row(n);
#pragma unroll
                for (int c = 0; c < IR / 32; ++c)
                  tma_load_2d(dst + c * C::BIAS_BOX, &maps.bias, x + 32 * c, sq.q0 + tile0, bar(C::B_BF + bs));
              }
              ++issuedb[bs];
            }
          }
          if (!__shfl_sync(0xffffffffu, (int)wb, 0)) break;
        }
        if (k >= NSTAGE || (C::OT && k == 1)) {
          // (OT: slots 1 .. held the outer tile until the compute warps copied it into TMEM)
          bool w = true;
          if (lane == 0)
            w = k >= NSTAGE ? mbar_wait(bar(C::B_IE + st), ((k / NSTAGE) - 1) & 1, abort_flag, p.err)
                            : mbar_wait(bar(C::B_QT), 0, abort_flag, p.err);
          if (!__shfl_sync(0xffffffffu, (int)w, 0)) break;
        }
        if (C::KEYS) {
          if (item_bands)
            while (n_next < n_items && !item_kept(e_next)) {
              ++n_next;
              if (n_next < n_items) e_next = item_band(n_next);
            }
#pragma unroll
          for (int pp = 0; pp < PPL; ++pp) {
            float nl[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) nl[u] = rl[pp][u] == -INFINITY ? -INFINITY : -rl[pp][u] * kLog2e;
            ldbuf[st * C::PAIRS + lane + 32 * pp] = make_float4(nl[0], nl[1], -rd[pp][0], -rd[pp][1]);
            if (stage_bands)
              bdbuf[st * C::PAIRS + lane + 32 * pp] = make_int4(rbl[pp][0], rbh[pp][0], rbl[pp][1], rbh[pp][1]);
          }
          if (lane == 0) islot[st] = make_int2(n, flags_n);
          if (n_next < n_items) load_pairs(n_next);  // (consumed next iteration)
        }
        const int ih = C::KEYS ? item_head(n) : hk;  // head inside the inner tensors
        const int irow = (C::KEYS ? sq.q0 : sq.k0) + item_row(n);
        if (lane == 0) {
          mbar_expect_tx(bar(C::B_IF + st), C::I0_BYTES);
          for (int c = 0; c < C::KB0; ++c) {
            if (lat && c == 2)
              tma_load_2d(sIn0 + st * C::I0_BYTES + c * C::IBLK, &maps.inner0_rope,
                          (C::KEYS ? ih : rh) * 64, irow, bar(C::B_IF + st));
            else
              tma_load_2d(sIn0 + st * C::I0_BYTES + c * C::IBLK, &maps.inner0, ih * qw + 64 * c, irow,
                          bar(C::B_IF + st));
          }
          ++issued0[st];
        }
        mbar_arrive(bar(C::B_IF + st));
        bool w1 = true;
        if (lane == 0) {
          if (k >= NSTAGE1) w1 = mbar_wait(bar(C::B_IE1 + st1), ((k / NSTAGE1) - 1) & 1, abort_flag, p.err);
          if (w1) {
            mbar_expect_tx(bar(C::B_IF1 + st1), C::I1_BYTES);
            for (int c = 0; c < C::KB1; ++c)
              tma_load_2d(sIn1 + st1 * C::I1_BYTES + c * C::IBLK, &maps.inner1, ih * DV + 64 * c, irow,
                          bar(C::B_IF1 + st1));
            ++issued1[st1];
          }
        }
        if (!__shfl_sync(0xffffffffu, (int)w1, 0)) break;
        n = n_next;
        e_n = e_next;
      }
      if (lane == 0) {
        drain_wait(bar(C::B_OUT), 0);
        for (int i = 0; i < NSTAGE; ++i)
          if (issued0[i]) drain_wait(bar(C::B_IF + i), (issued0[i] - 1) & 1);
        for (int i = 0; i < NSTAGE1; ++i)
          if (issued1[i]) drain_wait(bar(C::B_IF1 + i), (issued1[i] - 1) & 1);
        for (int i = 0; i < NBS; ++i)
          if (issuedb[i]) drain_wait(bar(C::B_BF + i), (issuedb[i] - 1) & 1);
      }
    }
  } else if (warp == 1 || warp >= 10) {
    // ------------------------------------------------------------------ MMA issuers
    // Three warps on three SM sub-partitions: warp 1 issues S (dK/dV: S^T), warp 11 dP (dP^T),
    // warp 10 the two accumulations that take their A operand from TMEM.  An MMA issue returns
    // only once the tensor pipe accepts it, so one issuer waiting on a completion would leave
    // the pipe idle; split, each waits only for what its own products need.  Each runs its
    // loop as a whole converged warp (uniform operands) and elect.sync picks the issuing lane.
    const int role = warp == 1 ? 0 : (warp == 11 ? 1 : 2);  // 0: S, 1: dP, 2: accumulations
    if (n_kept > 0 && (C::HAS_DP || role != 1)) {  // (kDv: no dP products)
      // S / dP: M = 128 outer rows, N = IR inner rows, both operands K-major
      const uint32_t id_sp = idesc_f16(is_bf16, 128, IR, 0, 0);
      // accumulations: A from TMEM (K = IR inner rows), B = inner tile MN-major
      const uint32_t id_a0 = idesc_f16(is_bf16, 128, C::KEYS ? C::NV_PAD : C::NQ_PAD, 0, 1);
      const uint32_t id_a1 = idesc_f16(is_bf16, 128, C::NQ_PAD, 0, 1);
      // descriptors are built once; a K step adds its byte offset / 16 to the start-address
      // field (shared addresses stay far below the field's 2^18-byte range, so nothing carries)
      const uint64_t d_o0 = sdesc_sw128(sO0, 16, 1024), d_o1 = sdesc_sw128(sO1, 16, 1024);
      auto s_cols = [&](int n) { return tmem + C::s_col(n % NBUF); };
      auto dp_cols = [&](int n) { return tmem + C::dp_col(n % NBUF); };
      auto issue_s = [&](int n) {  // S (dK/dV: S^T) of item n
        const uint64_t d_i0 = sdesc_sw128(sIn0 + (n % NSTAGE) * C::I0_BYTES, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint32_t oa = (kk >> 2) * C::OBLK + (kk & 3) * 32, ia = (kk >> 2) * C::IBLK + (kk & 3) * 32;
          if (C::QT_Q || C::OT_K)
            mma_ts_w(s_cols(n), tmem + (C::OT_K ? C::OTA : C::QA) + 8 * kk, d_i0 + (ia >> 4), id_sp, kk > 0);
          else mma_ss_w(s_cols(n), d_o0 + (oa >> 4), d_i0 + (ia >> 4), id_sp, kk > 0);
        }
      };
      auto issue_dp = [&](int n) {  // dP (dK/dV: dP^T) of item n
        const uint64_t d_i1 = sdesc_sw128(sIn1 + (n % NSTAGE1) * C::I1_BYTES, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk) {
          const uint32_t oa = (kk >> 2) * C::OBLK + (kk & 3) * 32, ia = (kk >> 2) * C::IBLK + (kk & 3) * 32;
          if (C::QT_DO || C::OT_V)
            mma_ts_w(dp_cols(n), tmem + (C::OT_V ? C::OTA : C::DOA) + 8 * kk, d_i1 + (ia >> 4), id_sp, kk > 0);
          else mma_ss_w(dp_cols(n), d_o1 + (oa >> 4), d_i1 + (ia >> 4), id_sp, kk > 0);
        }
      };
      // the 16-bit A operand of K step kk (16 inner rows) sits in the first half of the 32-column
      // chunk its compute thread loaded: column 32 * (kk / 2) + 8 * (kk % 2)
      auto a_col = [](int kk) { return (uint32_t)(32 * (kk >> 1) + 8 * (kk & 1)); };
      // accumulation 0 (dV += P^T dO) -- dK/dV and kDv
      auto issue_acc0 = [&](int n) {
        const uint64_t d_i1 = sdesc_sw128(sIn1 + (n % NSTAGE1) * C::I1_BYTES, C::IBLK, 1024);
#pragma unroll
        for (int kk = 0; kk < IR / 16; ++kk)
          mma_ts_w(tmem + C::ACC0, s_cols(n) + a_col(kk), d_i1 + (uint64_t)((kk * 2048) >> 4), id_a0,
                   (n > 0 || kk > 0) ? 1u : 0u);
      };
      // last accumulation: dK += dS^T Q (dK/dV) or dQ += dS K (dQ)
      auto issue_acc1 = [&](int n) {
        const uint64_t d_i0 = sdesc_sw128(sIn0 + (n % NSTAGE) * C::I0_BYTES, C::IBLK, 1024);
        const uint32_t acc = C::KEYS ? C::ACC1 : C::ACC0;
        const uint32_t id = C::KEYS ? id_a1 : id_a0;
#pragma unroll
        for (int kk = 0; kk < IR / 16; ++kk)
          mma_ts_w(tmem + acc, (MODE == kDqS ? s_cols(n) : dp_cols(n)) + a_col(kk),
                   d_i0 + (uint64_t)((kk * 2048) >> 4), id, (n > 0 || kk > 0) ? 1u : 0u);
      };
      auto wait_all = [&](int b, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar(b), parity, abort_flag, p.err));
      };
      bool ok = true;
      if (role < 2) {
        // products of item m, once its inner tile has landed and its TMEM columns are free
        // (QT: once the compute warps have copied the outer rows into TMEM)
        ok = wait_all(C::QT || (role == 0 ? C::OT_K : C::OT_V) ? C::B_QT : C::B_OUT, 0);
        for (int m = 0; m < n_kept && ok; ++m) {
          const int b = m % NBUF;
          // S reads ring 0 (Q or K), dP reads ring 1 (dO or V)
          ok = role == 0 ? wait_all(C::B_IF + m % NSTAGE, (m / NSTAGE) & 1)
                         : wait_all(C::B_IF1 + m % NSTAGE1, (m / NSTAGE1) & 1);
          // P_EARLY: P^T(m) may go to the dV accumulation before dP(m) has been issued, so S(m)
          // waits for the item's dO tile too (dV reads it)
          if (C::P_EARLY && role == 0 && ok) ok = wait_all(C::B_IF1 + m % NSTAGE1, (m / NSTAGE1) & 1);
          if (!ok) break;
          if (MODE == kDqS && role == 1) {
            // the single dP buffer is free once the compute warps have loaded item m-1's dP
            if (m >= 1) ok = wait_all(C::B_PF, (m - 1) & 1);
          } else if (C::SR && role == 1) {
            // dP(m) overwrites S(m) in the item's region once the compute warps have loaded it
            ok = wait_all(C::B_SL + b, (m / NBUF) & 1);
          } else if (m >= NBUF) {
            const int n = m - NBUF;  // the item that used these columns before
            const uint32_t par = (n / NBUF) & 1;
            if (role == 0) {
              // S(m) overwrites the columns accumulation 0 (dK/dV, kDv) read P^T from; kDq, kDk:
              // they are free as soon as the compute warps have loaded them; kDqS: once the dQ
              // accumulation has read the dS written there
              // (SR: the region is free once dK has read the dS written there)
              ok = C::HAS_DV ? wait_all(C::B_D0 + b, par)
                             : C::SR ? wait_all(C::B_D + b, par)
                             : (MODE == kDq || MODE == kDk ? wait_all(C::B_P + b, par)
                                                           : wait_all(C::B_D + b, par));
            } else {
              // dP(m) overwrites the dS the last accumulation reads
              ok = wait_all(C::B_D + b, par);
            }
          }
          if (!ok) break;
          fence_after();
          if (role == 0) issue_s(m);
          else issue_dp(m);
          mma_commit_w(bar((C::SPLIT && role == 1 ? C::B_DP : C::B_S) + b));
          // dQ, kDk: V / dO (ring 1) has no reader after dP
          if (!C::HAS_DV && role == 1) mma_commit_w(bar(C::B_IE1 + m % NSTAGE1));
        }
      } else {
        for (int n = 0; n < n_kept && ok; ++n) {
          const int b = n % NBUF;
          ok = wait_all(C::B_P + b, (n / NBUF) & 1);
          if (!ok) break;
          fence_after();
          if (C::HAS_DV) {
            // kDv: no dP product has waited for this item's dO tile; wait for it here (dK/dV:
            // the S issuer has, before S)
            if (MODE == kDv) {
              ok = wait_all(C::B_IF1 + n % NSTAGE1, (n / NSTAGE1) & 1);
              if (!ok) break;
              fence_after();
            }
            issue_acc0(n);
            mma_commit_w(bar(C::B_D0 + b));
            if (!C::P_EARLY) mma_commit_w(bar(C::B_IE1 + n % NSTAGE1));  // dO (ring 1): no reader after dV
          }
          if (C::P_EARLY) {
            // dK once dS^T is written; dO's other reader, dP(n), completed before the compute
            // warps loaded it, so the dO slot frees with this item's accumulations
            ok = wait_all(C::B_DS + b, (n / NBUF) & 1);
            if (!ok) break;
            fence_after();
          }
          if (C::HAS_LAST) issue_acc1(n);
          if (C::P_EARLY) mma_commit_w(bar(C::B_IE1 + n % NSTAGE1));
          mma_commit_w(bar(C::B_D + b));  // (the item's last accumulation)
          mma_commit_w(bar(C::B_IE + n % NSTAGE));
        }
      }
      const int drain = C::B_DRAIN + role;
      mma_commit_w(bar(drain));
      drain_wait(bar(drain), 0);
    }
  } else {
    // ------------------------------------------------------------------ elementwise + epilogue
    const int half = (warp - 2) >> 2;  // which half of the item's columns
    const int quarter = warp & 3;
    const int r = 32 * quarter + lane;  // TMEM lane = outer row (key for dK/dV, query for dQ)
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16);
    const float sl2 = p.scale_log2;
    const int orow = tile0 + r;  // this thread's outer row
    const bool orow_ok = C::KEYS ? orow < sq.kv_len : orow < sq.q_len;
    // the columns this row may see form one interval (query rows for dK/dV, keys for dQ)
    int vis_lo, vis_hi;
    if (C::KEYS) visible_rows(orow, off, sq.q_len, p.causal, p.window, vis_lo, vis_hi);
    else visible_range(orow, off, sq.kv_len, p.causal, p.window, vis_lo, vis_hi);
    if (!C::KEYS && cta_pure && orow_ok) {
      // dQ over rows whose bias is 0 on its finite interval: that interval masks the keys
      const int hb = p.bias_heads == 1 ? 0 : head_outer;
      const int4 e = __ldg(p.bias_rows + (size_t)hb * p.total_q + sq.q0 + orow);
      vis_lo = max(vis_lo, e.x);
      vis_hi = min(vis_hi, e.y);
    }
    if (!orow_ok || vis_hi < vis_lo) vis_hi = vis_lo;
    float row_nl = -INFINITY, row_nd = 0.f;  // dQ: this row's -LSE (base 2) and -D
    const float *brow_dq = nullptr;
    if (!C::KEYS && orow_ok) {
      const size_t gi = (size_t)head_outer * p.total_q + sq.q0 + orow;
      const float L = p.lse[gi];
      row_nl = L == -INFINITY ? -INFINITY : -L * kLog2e;
      row_nd = -p.rowdot[gi];
      if (BIAS == 1) {
        const int bh = p.bias_heads == 1 ? 0 : head_outer;
        brow_dq = p.bias + ((size_t)(sq.q0 + orow) * p.bias_heads + bh) * (size_t)p.max_kv;
      }
    }
    bool ok = true;
    if (C::QT && n_kept > 0) {
      // this thread's row of the outer Q (first half of the compute warps) or dO tile (second
      // half), 16 bytes at a time from its 128-byte-swizzled blocks, into the A-operand columns
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_OUT), 0, abort_flag, p.err));
      if (ok && (half == 0 ? C::QT_Q : C::QT_DO)) {
        const uint32_t src = (half == 0 ? sO0 : sO1) + r * 128;
        const uint32_t dst = lane_addr + (half == 0 ? C::QA : C::DOA);
        const int nb = half == 0 ? C::KB0 : C::KB1;
#pragma unroll 1
        for (int c = 0; c < nb; ++c) {
          uint32_t v[32];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            lds_v4(src + c * C::OBLK + ((q ^ (r & 7)) << 4), v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          __syncwarp();
          tmem_st32(dst + 32 * c, v);
        }
        tmem_st_wait();
      }
      fence_before();
      mbar_arrive(bar(C::B_QT));
    }
    if (C::OT && n_kept > 0) {
      // this thread's row of the outer tile (the two halves take half of its 64-column blocks
      // each) from ring-0 slots 1 .. into TMEM columns OTA on; the slots then take Q items
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_OUT), 0, abort_flag, p.err));
      if (ok) {
        const uint32_t src = sIn0 + C::I0_BYTES + r * 128;
        constexpr int nbh = (C::OT_KB + 1) / 2;
#pragma unroll 1
        for (int c = half * nbh; c < min(C::OT_KB, (half + 1) * nbh); ++c) {
          uint32_t v[32];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            lds_v4(src + c * C::OBLK + ((q ^ (r & 7)) << 4), v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          __syncwarp();
          tmem_st32(lane_addr + C::OTA + 32 * c, v);
        }
        tmem_st_wait();
      }
      // (these reads precede the TMA writes of Q items into the slots)
      fence_proxy_async_smem();
      fence_before();
      mbar_arrive(bar(C::B_QT));
    }
    for (int it = 0; it < n_kept && ok; ++it) {
      // it: the item's place in the pipeline (rings, buffers, barrier phases); n: which item it
      // is (query head and rows, dK/dV, from the producer's slot record; keys, dQ)
      const int b = it % NBUF, st = it % NSTAGE;
      bool w = mbar_wait(bar(C::B_S + b), (it / NBUF) & 1, abort_flag, p.err);
      // the LSE / D pairs were written by the producer lanes before their arrive on in_full:
      // acquire that barrier too before reading them
      if (C::KEYS && w) w = mbar_wait(bar(C::B_IF + st), (it / NSTAGE) & 1, abort_flag, p.err);
      if (BIAS == 2 && !cta_pure && w)
        w = mbar_wait(bar(C::B_BF + it % C::NBS_), (it / C::NBS_) & 1, abort_flag, p.err);
      ok = __all_sync(0xffffffffu, w);
      if (!ok) break;
      int n = it, iflags = 0;
      if (C::KEYS) {
        const int2 rec = islot[st];
        n = rec.x;
        iflags = rec.y;
      }
      const bool ipure = (iflags & 1) != 0, iinterior = (iflags & 2) != 0;
      // bias values enter the logits (TMA-staged or read row by row), unless this item's or
      // this CTA's rows are all pure intervals
      const bool use_vals = BIAS == 1 || (BIAS == 2 && !ipure && !cta_pure);
      const int h = item_head(n);
      // SPLIT: has dP landed too (then it is loaded with S)?  (Observed before the fence that
      // orders this thread's TMEM loads after it.)
      const bool dp_now = C::SPLIT && __all_sync(0xffffffffu, mbar_test(bar(C::B_DP + b), (it / NBUF) & 1));
      fence_after();
      const float *brow = brow_dq;
      if (C::KEYS && BIAS == 1 && orow_ok) {
        const int bh = p.bias_heads == 1 ? 0 : h;
        brow = p.bias + (size_t)bh * p.max_kv + orow;  // + (q0 + i) * bias_heads * max_kv per column
      }
      const bool with_dp = C::HAS_DP && (!C::SPLIT || dp_now);
#pragma unroll 1
      for (int ch = 0; ch < C::CHUNKS; ++ch) {
        const int col0 = C::HALF * half + 32 * ch;  // this chunk's first column in the item
        const int i0 = item_row(n) + col0;          // its first inner row
        const uint32_t s_addr = lane_addr + C::s_col(b) + col0, dp_addr = lane_addr + C::dp_col(b) + col0;
        uint32_t sv[32], dv[32];
        __syncwarp();
        tmem_ld32(s_addr, sv);
        if (with_dp) tmem_ld32(dp_addr, dv);
        // is every element of this thread's 32 columns visible (no per-element mask)?
        bool plain;
        if (C::KEYS) {
          const int j = orow, ilast = i0 + 31;
          plain = orow_ok && ilast < sq.q_len && (!p.causal || j <= i0 + off) &&
                  (p.window <= 0 || j >= ilast + off - p.window + 1);
        } else {
          const int i = orow, jlast = i0 + 31;
          plain = orow_ok && jlast < sq.kv_len && (!p.causal || jlast <= i + off) &&
                  (p.window <= 0 || i0 >= i + off - p.window + 1);
        }
        plain = plain && BIAS != 1;
        // dK/dV, a pure item: the columns (query rows) whose finite-bias interval holds this key
        unsigned bmask = 0xffffffffu;
        if (C::BD_BYTES > 0 && ipure && !iinterior) {
          const int4 *bp = bdbuf + st * C::PAIRS + col0 / 2;
          bmask = 0u;
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int4 bb = bp[e];
            bmask |= (unsigned)(bb.x <= orow && orow < bb.y) << (2 * e);
            bmask |= (unsigned)(bb.z <= orow && orow < bb.w) << (2 * e + 1);
          }
          plain = plain && bmask == 0xffffffffu;
        }
        // dQ over pure rows: the chunk's keys must all lie in this row's interval
        if (!C::KEYS && cta_pure) plain = plain && i0 >= vis_lo && i0 + 31 < vis_hi;
        const float4 *lp = ldbuf + st * C::PAIRS + col0 / 2;  // this chunk's 16 pairs (dK/dV)
        // TMA-staged bias: the chunk's 32 values of this thread -- dQ: along its row, from the
        // chunk's swizzled box; dK/dV: down its key's column, one 128-byte box row per query row
        float bq4[32];
        if (BIAS == 2 && use_vals) {
          const uint32_t bstage = sBias + (it % C::NBS_) * C::BIAS_STAGE;
          if (C::KEYS) {
            const uint32_t bcol = bstage + quarter * C::BIAS_BOX + lane * 4 + col0 * 128;
#pragma unroll
            for (int k = 0; k < 32; ++k) bq4[k] = lds_f32(bcol + k * 128);
          } else {
            const uint32_t rowb = bstage + (col0 / 32) * C::BIAS_BOX + r * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 b = lds_f32x4(rowb + ((q ^ (r & 7)) << 4));
              bq4[4 * q] = b.x; bq4[4 * q + 1] = b.y; bq4[4 * q + 2] = b.z; bq4[4 * q + 3] = b.w;
            }
          }
        }
        tmem_ld_wait();
        if (C::SR) {
          // S is in registers: dP may overwrite its columns
          fence_before();
          mbar_arrive(bar(C::B_SL + b));
        }
        if (MODE == kDqS && with_dp && ch == C::CHUNKS - 1) {
          // every dP column of the item is in registers: the next dP may overwrite them
          fence_before();
          mbar_arrive(bar(C::B_PF));
        }
        uint32_t pk[16];
        float pf[32];  // P
        if (plain) {
          // every pair visible: P = 2^(S log2e scale - LSE2 [+ bias log2e])
          // (packed f32x2 arithmetic: the same per-lane rounding as the scalar forms)
          const uint64_t sl22 = f2pack(sl2, sl2), lg22 = f2pack(kLog2e, kLog2e);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c = 2 * e;
            const float2 nl = C::KEYS ? make_float2(lp[e].x, lp[e].y) : make_float2(row_nl, row_nl);
            uint64_t x2 = fma2(f2pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl22,
                               f2pack(nl.x, nl.y));
            if (BIAS == 2 && use_vals) x2 = fma2(f2pack(bq4[c], bq4[c + 1]), lg22, x2);
            const float2 x = f2unpack(x2);
            pf[c] = ex2(x.x);
            pf[c + 1] = ex2(x.y);
            pk[e] = pack2(pf[c], pf[c + 1], is_bf16);
          }
        } else {
          // dQ with a bias from global memory: the chunk's 32 bias values of this row, 16 bytes
          // at a time when the row address is 16-byte aligned and the chunk lies inside the row
          const bool bvec = BIAS == 1 && !C::KEYS && brow != nullptr &&
                            (reinterpret_cast<uintptr_t>(brow + i0) & 15u) == 0 && i0 + 32 <= p.max_kv;
          if (bvec) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 b = __ldg(reinterpret_cast<const float4 *>(brow + i0) + q);
              bq4[4 * q] = b.x; bq4[4 * q + 1] = b.y; bq4[4 * q + 2] = b.z; bq4[4 * q + 3] = b.w;
            }
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c = 2 * e;
            const float2 nl = C::KEYS ? make_float2(lp[e].x, lp[e].y) : make_float2(row_nl, row_nl);
            float xs[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int cc = i0 + c + u;  // sequence-local column: query row (dK/dV) or key (dQ)
              float x = __uint_as_float(sv[c + u]) * sl2;
              if (BIAS == 2) {
                if (use_vals) x = fmaf(bq4[c + u], kLog2e, x);
              } else if (BIAS == 1 && brow) {
                // element by element unless the chunk was loaded 16 bytes at a time (bq4),
                // clamped into the sequence so that masked columns read a valid address
                const float bv = C::KEYS
                                     ? __ldg(brow + (size_t)(sq.q0 + min(cc, sq.q_len - 1)) * p.bias_heads * (size_t)p.max_kv)
                                     : (bvec ? bq4[c + u] : __ldg(brow + min(cc, sq.kv_len - 1)));
                x = fmaf(bv, kLog2e, x);
              }
              xs[u] = (cc >= vis_lo && cc < vis_hi && ((bmask >> (c + u)) & 1u)) ? x : -INFINITY;
            }
            // masked logits (-inf) and rows without keys (-LSE2 = -inf) give P = 0
            const float2 x = f2unpack(add2(f2pack(xs[0], xs[1]), f2pack(nl.x, nl.y)));
            pf[c] = ex2(x.x);
            pf[c + 1] = ex2(x.y);
            pk[e] = pack2(pf[c], pf[c + 1], is_bf16);
          }
        }
        if (C::HAS_DV) {
          __syncwarp();
          tmem_st16(s_addr, pk);  // P^T for dV
        }
        if (C::P_EARLY) {
          // P^T to the dV accumulation now, before dS^T
          tmem_st_wait();
          fence_before();
          mbar_arrive(bar(C::B_P + b));
        }
        if (C::SPLIT && !dp_now) {
          // dP ran while P was formed
          ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_DP + b), (it / NBUF) & 1, abort_flag, p.err));
          if (!ok) break;
          fence_after();
          __syncwarp();
          tmem_ld32(dp_addr, dv);
          tmem_ld_wait();
          if (MODE == kDqS) {
            fence_before();
            mbar_arrive(bar(C::B_PF));
          }
        }
        if (C::HAS_DP) {
          // dS = P (dP - D)
          uint32_t dk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c = 2 * e;
            const float2 nd = C::KEYS ? make_float2(lp[e].z, lp[e].w) : make_float2(row_nd, row_nd);
            const uint64_t t2 = add2(f2pack(__uint_as_float(dv[c]), __uint_as_float(dv[c + 1])),
                                     f2pack(nd.x, nd.y));
            const float2 d = f2unpack(mul2(f2pack(pf[c], pf[c + 1]), t2));
            dk[e] = pack2(d.x, d.y, is_bf16);
          }
          __syncwarp();
          tmem_st16(MODE == kDqS ? s_addr : dp_addr, dk);  // dS (dK/dV: dS^T)
        }
      }
      if (!ok) break;
      if (BIAS == 2 && !cta_pure) mbar_arrive(bar(C::B_BE + it % C::NBS_));  // the slot may be refilled
      tmem_st_wait();
      fence_before();
      mbar_arrive(bar((C::P_EARLY ? C::B_DS : C::B_P) + b));
    }
    // epilogue: the last item's last accumulation completes every MMA of the CTA
    if (ok && n_kept > 0)
      ok = mbar_wait(bar(C::B_D + (n_kept - 1) % NBUF), ((n_kept - 1) / NBUF) & 1, abort_flag, p.err);
    ok = __all_sync(0xffffffffu, ok);
    // Outputs of a full 128-row tile whose widths are whole 64-column blocks leave through TMA:
    // each thread writes its row into the idle outer-tile shared memory in the 128-byte-swizzled
    // box layout and one thread stores whole boxes (per-thread row stores land 32 rows of
    // another head apart and cost a store transaction per 16 bytes).  Other tiles store rows.
    const bool lat_out = DQK == 192 && p.latent;
    const bool tma_out =
        !lat_out && (C::KEYS ? sq.kv_len : sq.q_len) - tile0 >= 128 &&
        (MODE == kDkdv ? DV % 64 == 0 && DQK % 64 == 0 : (MODE == kDv ? DV % 64 == 0 : DQK % 64 == 0));
    if (ok) {
      fence_after();
      // TMEM columns [tcol, tcol + ncols) of this row, times mul, into the staging boxes from
      // output column col0 on (64 columns per box, 16 KB each, at the outer tiles' offset)
      auto stage_acc = [&](uint32_t tcol, int ncols, int col0, float mul) {
#pragma unroll 1
        for (int ch = 0; ch < ncols / 32; ++ch) {
          uint32_t v[32];
          if (n_kept > 0) {
            __syncwarp();
            tmem_ld32(lane_addr + tcol + ch * 32, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          }
          uint32_t o16[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            o16[e] = pack2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul, is_bf16);
          const int col = col0 + 32 * ch, c16 = (col % 64) / 8;
          const uint32_t rowa = base + C::OFF_O0 + (col / 64) * C::OBLK + r * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            sts_v4(rowa + (((c16 + q) ^ (r & 7)) << 4), o16[4 * q], o16[4 * q + 1], o16[4 * q + 2], o16[4 * q + 3]);
        }
      };
      if (tma_out) {
        if (MODE == kDkdv) {
          if (half == 0) stage_acc(C::ACC0, DV, 0, 1.f);                 // dV: boxes 0 .. KB1-1
          else stage_acc(C::ACC1, DQK, C::KB1 * 64, p.scale);            // dK: the boxes after
        } else {
          constexpr int W = MODE == kDv ? DV : DQK, first = 32 * ((W / 32 + 1) / 2);
          const uint32_t acc = MODE == kDv ? C::ACC0 : (MODE == kDk ? C::ACC1 : C::ACC0);
          const float mul = MODE == kDv ? 1.f : p.scale;
          if (half == 0) stage_acc(acc, first, 0, mul);
          else if (W > first) stage_acc(acc + first, W - first, first, mul);
        }
      }
      // TMEM columns [tcol, tcol + ncols) of this thread's row, times mul, to dst_base + off
      // (elements): 16-bit, or fp32 when f32
      const size_t g = (size_t)((C::KEYS ? sq.k0 : sq.q0) + (orow_ok ? orow : 0));
      auto store_acc = [&](uint32_t tcol, int ncols, void *dst_base, size_t off, float mul, bool f32) {
#pragma unroll 1
        for (int ch = 0; ch < ncols / 32; ++ch) {
          uint32_t v[32];
          if (n_kept > 0) {
            __syncwarp();
            tmem_ld32(lane_addr + tcol + ch * 32, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          }
          if (!orow_ok) continue;
          if (f32) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(dst_base) + off + 32 * ch);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              dst[q4] = make_float4(__uint_as_float(v[4 * q4]) * mul, __uint_as_float(v[4 * q4 + 1]) * mul,
                                    __uint_as_float(v[4 * q4 + 2]) * mul, __uint_as_float(v[4 * q4 + 3]) * mul);
          } else {
            uint32_t o16[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              o16[e] = pack2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul, is_bf16);
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(dst_base) + off + 32 * ch);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              dst[q4] = make_uint4(o16[4 * q4], o16[4 * q4 + 1], o16[4 * q4 + 2], o16[4 * q4 + 3]);
          }
        }
      };
      // a latent head given as split operands: the nope and rope parts of dK / dQ go to separate
      // tensors; a rope key shared by the kv heads gets its per-head part in fp32, summed later
      const bool lat = lat_out;
      if (tma_out) {
        // (staged above)
      } else if (MODE == kDv || MODE == kDk) {
        // the pass's one accumulator, its columns split between the two halves
        constexpr int W = MODE == kDv ? DV : DQK, first = 32 * ((W / 32 + 1) / 2);
        void *dst = MODE == kDv ? p.dv : p.dk;
        const uint32_t acc = MODE == kDv ? C::ACC0 : C::ACC1;
        const float mul = MODE == kDv ? 1.f : p.scale;
        if (half == 0) store_acc(acc, first, dst, (g * p.h_kv + hk) * W, mul, false);
        else if (W > first) store_acc(acc + first, W - first, dst, (g * p.h_kv + hk) * W + first, mul, false);
      } else if (MODE == kDkdv) {
        if (half == 0) {
          store_acc(C::ACC0, DV, p.dv, (g * p.h_kv + hk) * DV, 1.f, false);
        } else if (!lat) {
          store_acc(C::ACC1, DQK, p.dk, (g * p.h_kv + hk) * DQK, p.scale, false);
        } else {
          store_acc(C::ACC1, 128, p.dk, (g * p.h_kv + hk) * 128, p.scale, false);
          if (p.dk_rope_part)
            store_acc(C::ACC1 + 128, 64, p.dk_rope_part, ((size_t)hk * p.total_kv + g) * 64, p.scale, true);
          else
            store_acc(C::ACC1 + 128, 64, p.dk_rope, (g * p.rope_heads + (p.rope_heads == 1 ? 0 : hk)) * 64,
                      p.scale, false);
        }
      } else {
        const size_t row = g * p.h_q + head_outer;
        if (lat) {
          if (half == 0) store_acc(C::ACC0, 128, p.dq, row * 128, p.scale, false);
          else store_acc(C::ACC0 + 128, 64, p.dq_rope, row * 64, p.scale, false);
        } else {
          // the two halves split dQ's 32-column chunks (an odd count: the first takes one more)
          constexpr int nch = DQK / 32, first = (nch + 1) / 2;
          if (half == 0) store_acc(C::ACC0, 32 * first, p.dq, row * DQK, p.scale, false);
          else if (nch > first)
            store_acc(C::ACC0 + 32 * first, 32 * (nch - first), p.dq, row * DQK + 32 * first, p.scale, false);
        }
      }
    }
    if (tma_out) {
      // every compute thread has staged its rows (a warp that aborted staged nothing; the error
      // word reports that): make the writes visible to TMA, then one thread stores the boxes and
      // waits until they have been read out of shared memory
      fence_proxy_async_smem();
      named_sync(1, 256);
      if (warp == 2 && lane == 0 && ok) {
        const int y = (C::KEYS ? sq.k0 : sq.q0) + tile0;
        const uint32_t stage0 = base + C::OFF_O0;
        if (MODE == kDkdv) {
          for (int j = 0; j < C::KB1; ++j) tma_store_2d(&maps.out0, stage0 + j * C::OBLK, hk * DV + 64 * j, y);
          for (int j = 0; j < C::KB0; ++j)
            tma_store_2d(&maps.out1, stage0 + (C::KB1 + j) * C::OBLK, hk * DQK + 64 * j, y);
        } else if (MODE == kDv) {
          for (int j = 0; j < C::KB1; ++j) tma_store_2d(&maps.out0, stage0 + j * C::OBLK, hk * DV + 64 * j, y);
        } else {
          const int oh = MODE == kDk ? hk : head_outer;
          for (int j = 0; j < C::KB0; ++j) tma_store_2d(&maps.out0, stage0 + j * C::OBLK, oh * DQK + 64 * j, y);
        }
        bulk_commit();
        bulk_wait_read();
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

// Whether every row this CTA works on has a bias that is 0 over its finite interval (bias
// bands): dQ -- the CTA's 128 query rows; dK/dV -- the rows of every query item it keeps.  The
// tile and item walk are those of tc_bwd_body.  Every thread of the CTA calls it.
template <bool KEYS, int IR>
__device__ __forceinline__ bool bwd_cta_all_pure(const Params &p) {
  if (!p.bias_blocks) return false;
  Seq sq;
  if (!load_seq(p, (int)blockIdx.z, sq)) return false;
  const int bxr = p.heads_fast ? (int)blockIdx.y : (int)blockIdx.x;
  const int gx = p.heads_fast ? (int)gridDim.y : (int)gridDim.x;
  const int byh = p.heads_fast ? (int)blockIdx.x : (int)blockIdx.y;
  if (KEYS) {
    const int tile0 = bxr * 128, hk = byh;
    if (tile0 >= sq.kv_len) return false;
    int qlo = 0, qhi = 0;
    if (sq.q_len > 0) {
      q_band(tile0, min(tile0 + 128, sq.kv_len), sq.q_len, sq.kv_len, p.causal, p.window, qlo, qhi);
      if (p.flags & VLF_FLAG_NO_SKIP) { qlo = 0; qhi = sq.q_len; }
    }
    const int lo = (qlo / IR) * IR;
    const int nq_tiles = qhi > qlo ? (qhi - lo + IR - 1) / IR : 0;
    const int n_items = nq_tiles * p.group;
    bool all = true;
    for (int b0 = 0; b0 < n_items; b0 += (int)blockDim.x) {
      const int n = b0 + (int)threadIdx.x;
      bool pure = true;
      if (n < n_items) {
        const int hb = p.bias_heads == 1 ? 0 : hk * p.group + n / nq_tiles;
        const int4 e = __ldg(p.bias_blocks + (size_t)hb * p.total_q + sq.q0 + lo + (n % nq_tiles) * IR);
        if (e.y > e.x && e.x < tile0 + 128 && e.y > tile0) pure = e.z >= 0;
      }
      all = __syncthreads_and(pure) && all;
    }
    return all;
  }
  const int bx = p.causal ? gx - 1 - bxr : bxr;
  const int tile0 = bx * 128, hb = p.bias_heads == 1 ? 0 : byh;
  if (tile0 >= sq.q_len) return false;
  const int4 *bb = p.bias_blocks + (size_t)hb * p.total_q + sq.q0 + tile0;
  int pure = __ldg(bb).z >= 0;
  if (tile0 + 64 < sq.q_len) pure &= __ldg(bb + 64).z >= 0;
  return pure != 0;
}

// The backward kernel.  With a TMA-staged bias (BIAS 2) and PST > 0, a CTA whose rows are all
// 0 / -inf intervals runs the body without a bias ring instead (BIAS 3): its rings take the
// shared memory of the bias tiles (PST / PST1 slots), as deep as the kernel without a bias.
//
// The backward kernels are launched with programmatic stream serialization (launch_bwd).  The
// first key-tile kernel after the row-dot pass (dK/dV, or the width-256 dV pass) reads D, so it
// waits for the kernel ahead before reading anything global; every backward kernel then lets the
// next one be launched.  The kernels after it (the dK pass, dQ) read only the inputs and D -- no
// output of the kernel just ahead -- so their CTAs start on the SMs the previous kernel's last
// CTAs leave (D was complete before any CTA of that kernel allowed them to launch), and they wait
// for it only at their end, so that their completion still implies its completion.
template <int MODE, int DQK, int DV, int IR, int NBUF, int NSTAGE, int NSTAGE1, int NBS, bool BF16,
          int BIAS, int PST = 0, int PST1 = 0>
__global__ void __launch_bounds__(384, 1)
tc_bwd_kernel(const __grid_constant__ BwdMaps maps, const Params p) {
  constexpr bool first = MODE == kDkdv || MODE == kDv;
  if (first) pdl_wait();
  pdl_trigger();
  bool done = false;
  if constexpr (BIAS == 2 && PST > 0) {
    if (bwd_cta_all_pure<BwdCfg<MODE, DQK, DV, IR, NBUF, NSTAGE, NSTAGE1, NBS>::KEYS, IR>(p)) {
      tc_bwd_body<MODE, DQK, DV, IR, NBUF, PST, PST1, 0, BF16, 3>(maps, p);
      done = true;
    }
  }
  if (!done) tc_bwd_body<MODE, DQK, DV, IR, NBUF, NSTAGE, NSTAGE1, NBS, BF16, BIAS>(maps, p);
  if (!first) pdl_wait();
}

// NBS > 0: the problem's bias is staged through TMA (the caller checked that it can be); PST /
// PST1: the ring depths of its CTAs over pure 0 / -inf interval rows (0: none).
template <int MODE, int DQK, int DV, int IR, int NBUF, int NSTAGE, int NSTAGE1, int NBS, int PST = 0,
          int PST1 = 0>
cudaError_t launch_bwd(const Params &p, cudaStream_t st) {
  using C = BwdCfg<MODE, DQK, DV, IR, NBUF, NSTAGE, NSTAGE1, NBS>;
  const int bf = p.dtype == VLF_BF16;
  BwdMaps m;
  const uint64_t tq = p.total_q, tk = p.total_kv;
  bool ok;
  // a latent head with split operands: q / k hold the 128-wide nope parts, q_rope / k_rope the
  // 64-wide rope parts
  const bool lat = DQK == 192 && p.latent;
  const uint64_t qw = lat ? 128 : DQK;
  const uint64_t qc = (uint64_t)p.h_q * qw, kc = (uint64_t)p.h_kv * qw;
  const uint64_t qrc = (uint64_t)p.h_q * 64, krc = (uint64_t)(lat ? p.rope_heads : 1) * 64;
  if (C::KEYS) {
    ok = make_tmap_16bit(&m.outer0, p.k, tk, kc, kc, 128, bf) &&
         make_tmap_16bit(&m.outer1, p.v, tk, (uint64_t)p.h_kv * DV, (uint64_t)p.h_kv * DV, 128, bf) &&
         make_tmap_16bit(&m.inner0, p.q, tq, qc, qc, IR, bf) &&
         make_tmap_16bit(&m.inner1, p.dout, tq, (uint64_t)p.h_q * DV, (uint64_t)p.h_q * DV, IR, bf);
    if (lat)
      ok = ok && make_tmap_16bit(&m.outer0_rope, p.k_rope, tk, krc, krc, 128, bf) &&
           make_tmap_16bit(&m.inner0_rope, p.q_rope, tq, qrc, qrc, IR, bf);
  } else {
    ok = make_tmap_16bit(&m.outer0, p.q, tq, qc, qc, 128, bf) &&
         make_tmap_16bit(&m.outer1, p.dout, tq, (uint64_t)p.h_q * DV, (uint64_t)p.h_q * DV, 128, bf) &&
         make_tmap_16bit(&m.inner0, p.k, tk, kc, kc, IR, bf) &&
         make_tmap_16bit(&m.inner1, p.v, tk, (uint64_t)p.h_kv * DV, (uint64_t)p.h_kv * DV, IR, bf);
    if (lat)
      ok = ok && make_tmap_16bit(&m.outer0_rope, p.q_rope, tq, qrc, qrc, 128, bf) &&
           make_tmap_16bit(&m.inner0_rope, p.k_rope, tk, krc, krc, IR, bf);
  }
  if (!lat) { m.outer0_rope = m.outer0; m.inner0_rope = m.inner0; }  // (unused)
  // the outputs, for the TMA epilogue of full tiles (dk / dq row widths as the nope parts' for a
  // split latent head, which stores rows instead)
  const uint64_t dvc = (uint64_t)p.h_kv * DV;
  if (MODE == kDkdv)
    ok = ok && make_tmap_16bit(&m.out0, p.dv, tk, dvc, dvc, 128, bf) &&
         make_tmap_16bit(&m.out1, p.dk, tk, kc, kc, 128, bf);
  else if (MODE == kDv)
    ok = ok && make_tmap_16bit(&m.out0, p.dv, tk, dvc, dvc, 128, bf);
  else if (MODE == kDk)
    ok = ok && make_tmap_16bit(&m.out0, p.dk, tk, kc, kc, 128, bf);
  else
    ok = ok && make_tmap_16bit(&m.out0, p.dq, tq, qc, qc, 128, bf);
  if (MODE != kDkdv) m.out1 = m.out0;  // (unused)
  if (NBS > 0)
    ok = ok && make_tmap_bias(&m.bias, p.bias, tq, (uint64_t)p.bias_heads * p.max_kv,
                              C::KEYS ? IR : 128, !C::KEYS);
  else
    m.bias = m.inner0;  // (unused)
  if (!ok) return cudaErrorInvalidValue;
  const unsigned tiles = C::KEYS ? (p.max_kv + 127) / 128 : (p.max_q + 127) / 128;
  const unsigned heads = C::KEYS ? p.h_kv : p.h_q;
  if (tiles == 0) return cudaSuccess;
  Params pl = p;
  pl.heads_fast = p.bias != nullptr && p.bias_heads == 1;
  const dim3 grid = pl.heads_fast ? dim3(heads, tiles, p.num_seqs) : dim3(tiles, heads, p.num_seqs);
  void (*kern)(const BwdMaps, const Params);
  int smem = C::SMEM;
  if constexpr (NBS > 0) {
    kern = bf ? tc_bwd_kernel<MODE, DQK, DV, IR, NBUF, NSTAGE, NSTAGE1, NBS, true, 2, PST, PST1>
              : tc_bwd_kernel<MODE, DQK, DV, IR, NBUF, NSTAGE, NSTAGE1, NBS, false, 2, PST, PST1>;
    if constexpr (PST > 0) smem = max(smem, BwdCfg<MODE, DQK, DV, IR, NBUF, PST, PST1, 0>::SMEM);
  } else {
    kern = p.bias ? (bf ? tc_bwd_kernel<MODE, DQK, DV, IR, NBUF, NSTAGE, NSTAGE1, 0, true, 1>
                        : tc_bwd_kernel<MODE, DQK, DV, IR, NBUF, NSTAGE, NSTAGE1, 0, false, 1>)
                  : (bf ? tc_bwd_kernel<MODE, DQK, DV, IR, NBUF, NSTAGE, NSTAGE1, 0, true, 0>
                        : tc_bwd_kernel<MODE, DQK, DV, IR, NBUF, NSTAGE, NSTAGE1, 0, false, 0>);
  }
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(384);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void *args[] = {&m, &pl};
  e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(kern), args);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

// The gradient of a rope key shared by the kv heads of a split-operand latent head: the dK/dV
// kernel left each kv head's part in fp32 [h_kv, total_kv, 64]; sum them in head order
// (deterministic) into dk_rope [total_kv, 1, 64].
template <bool BF16>
__global__ void __launch_bounds__(256) rope_grad_sum_kernel(const Params p) {
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  const size_t n = (size_t)p.total_kv * 64;
  const size_t i = (size_t)blockIdx.x * 256 + threadIdx.x;
  if (i >= n) return;
  float acc = 0.f;
  for (int h = 0; h < p.h_kv; ++h) acc += p.dk_rope_part[(size_t)h * n + i];
  static_cast<T *>(p.dk_rope)[i] = from_f32<T>(acc);
}

cudaError_t rope_grad_sum(const Params &p, cudaStream_t st) {
  const size_t n = (size_t)p.total_kv * 64;
  if (n == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((n + 255) / 256);
  if (p.dtype == VLF_BF16) rope_grad_sum_kernel<true><<<blocks, 256, 0, st>>>(p);
  else rope_grad_sum_kernel<false><<<blocks, 256, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

// Per head width: item rows, buffers, ring-0 / ring-1 stages and bias stages of the dK/dV kernel
// (IR_KV, NBUF_KV, NST_KV, NST1_KV, NBS_KV) and the mode, item rows, buffers, ring stages and
// bias stages of the dQ kernel (MODE_Q, IR_Q, NBUF_Q, NST_Q, NST1_Q, NBS_Q).  A ring slot is
// refilled only after its item's last product has read it, so the rings are as deep as shared
// memory allows.  With a TMA-staged bias, PST* are the ring depths of the CTAs whose rows are
// all 0 / -inf intervals (the bias tiles' shared memory goes to the rings).
template <int DQK, int DV, int IR_KV, int NBUF_KV, int NST_KV, int NST1_KV, int NBS_KV, int MODE_Q,
          int IR_Q, int NBUF_Q, int NST_Q, int NST1_Q, int NBS_Q, int PST_KV = 0, int PST1_KV = 0,
          int PST_Q = 0, int PST1_Q = 0>
cudaError_t bwd_shape(const Params &p, cudaStream_t st, const cudaEvent_t *ev) {
  cudaError_t e;
  if ((e = mark(ev, 0, st)) != cudaSuccess) return e;
  if ((e = rowdot_forward(p, st)) != cudaSuccess) return e;
  if ((e = mark(ev, 1, st)) != cudaSuccess) return e;
  if ((e = launch_bwd<kDkdv, DQK, DV, IR_KV, NBUF_KV, NST_KV, NST1_KV, NBS_KV, PST_KV, PST1_KV>(p, st)) != cudaSuccess)
    return e;
  if (DQK == 192 && p.latent && p.dk_rope_part && (e = rope_grad_sum(p, st)) != cudaSuccess) return e;
  if ((e = mark(ev, 2, st)) != cudaSuccess) return e;
  if ((e = launch_bwd<MODE_Q, DQK, DV, IR_Q, NBUF_Q, NST_Q, NST1_Q, NBS_Q, PST_Q, PST1_Q>(p, st)) != cudaSuccess)
    return e;
  return mark(ev, 3, st);
}

// Width 256: the row-dot, the dV pass and the dK pass (together the dK/dV stage), then dQ (dS
// over S, 64-key items).  Rings as deep as shared memory allows: 64 KB outer tiles, 32 KB items.
cudaError_t bwd_shape256(const Params &p, cudaStream_t st, const cudaEvent_t *ev) {
  cudaError_t e;
  if ((e = mark(ev, 0, st)) != cudaSuccess) return e;
  if ((e = rowdot_forward(p, st)) != cudaSuccess) return e;
  if ((e = mark(ev, 1, st)) != cudaSuccess) return e;
  if ((e = launch_bwd<kDv, 256, 256, 64, 2, 5, 2, 0>(p, st)) != cudaSuccess) return e;
  if ((e = launch_bwd<kDk, 256, 256, 64, 2, 3, 2, 0>(p, st)) != cudaSuccess) return e;
  if ((e = mark(ev, 2, st)) != cudaSuccess) return e;
  if ((e = launch_bwd<kDqS, 256, 256, 64, 2, 2, 1, 0>(p, st)) != cudaSuccess) return e;
  return mark(ev, 3, st);
}

}  // namespace

bool tc_backward_supported(const Params &p) {
  if (p.dtype != VLF_F16 && p.dtype != VLF_BF16) return false;
  return (p.d_qk == 64 && p.d_v == 64) || (p.d_qk == 96 && p.d_v == 96) ||
         (p.d_qk == 128 && p.d_v == 128) || (p.d_qk == 192 && p.d_v == 128) ||
         (p.d_qk == 256 && p.d_v == 256);
}

cudaError_t tc_backward(const Params &p, cudaStream_t st, const cudaEvent_t *ev) {
  if (p.total_q == 0 || p.total_kv == 0) return simt_backward(p, st, ev);
  // A bias whose rows start 16-byte aligned streams through TMA in 64-row items (bias tiles take
  // a third of shared memory: the Q / dO and K / V rings are shallower); other bias shapes load
  // their values from global memory in the compute threads.  (Read into registers one item ahead
  // instead, the dK/dV kernel's bias was slower: 40.2 against 35.8 ms on the per-head bias.)
  const bool bias_tma = p.bias != nullptr && p.max_kv % 4 == 0 &&
                        (reinterpret_cast<uintptr_t>(p.bias) & 15u) == 0 && p.d_qk <= 128;
  if (bias_tma) {
    if (p.d_qk == 64) return bwd_shape<64, 64, 64, 2, 4, 4, 3, kDq, 64, 2, 4, 4, 3, 6, 6, 6, 6>(p, st, ev);
    if (p.d_qk == 96) return bwd_shape<96, 96, 64, 2, 2, 2, 3, kDq, 64, 2, 2, 2, 3, 5, 4, 5, 4>(p, st, ev);
    return bwd_shape<128, 128, 64, 2, 2, 2, 3, kDq, 64, 2, 2, 2, 3, 5, 4, 5, 4>(p, st, ev);
  }
  if (p.d_qk == 64) return bwd_shape<64, 64, 64, 2, 6, 6, 0, kDqS, 128, 2, 3, 3, 0>(p, st, ev);
  if (p.d_qk == 96) return bwd_shape<96, 96, 64, 2, 5, 4, 0, kDqS, 128, 2, 3, 2, 0>(p, st, ev);
  if (p.d_qk == 128) return bwd_shape<128, 128, 64, 2, 5, 4, 0, kDqS, 128, 2, 3, 2, 0>(p, st, ev);
  if (p.d_qk == 256) return bwd_shape256(p, st, ev);
  return bwd_shape<192, 128, 64, 1, 3, 3, 0, kDq, 64, 2, 3, 3, 0>(p, st, ev);
}

// The tensor-core backward writes dQ directly (no fp32 accumulator); only the row dot
// products D = rowsum(dO o O) live in the workspace.
size_t tc_backward_workspace(int, int, int) { return 0; }

}  // namespace vlf
