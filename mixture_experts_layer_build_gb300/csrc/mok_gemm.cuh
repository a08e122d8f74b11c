// mok_gemm.cuh -- the grouped expert GEMMs of the layer on the 5th-generation tensor cores.
//
// One persistent, warp-specialised kernel template serves all six contractions of the layer
// ("Cursor Open-Sources Mixture-of-Kittens (MoK) ...", English summary: SwiGLU experts, forward
// and backward, router-weight gradient inside the SwiGLU backward):
//   FWD_GATEUP  [g|u] = Xg Wg_e^T | Xg Wu_e^T, epilogue a = silu(g) u          (K = H)
//   FWD_DOWN    y = a Wd_e^T                                                   (K = I)
//   DGRAD1      dA' = dYg Wd_e, epilogue: dS partials, SwiGLU backward, s*a     (K = H, B MN-major)
//   DGRAD2      dXg = [dg|du] [Wg_e;Wu_e]                                       (K = 2I, B MN-major)
//   WGRAD_GU    [dWg;dWu]_e = [dg|du]_e^T Xg_e                                  (K = rows of e, A,B MN-major)
//   WGRAD_D     dWd_e = dYg_e^T (s a)_e                                         (K = rows of e, A,B MN-major)
//
// Row-tiled BF16 tiles may run on CTA pairs (chosen by shape, use_pairs; a cluster of two CTAs,
// tcgen05.mma.cta_group::2, M = 256): the
// pair shares one B tile, each CTA loading half of it, so a CTA receives 32 KB per K block of a
// 128 x 256 accumulator instead of 48 KB and keeps six K blocks in flight instead of four.  The
// row-tiled variants pair two consecutive 128-row blocks of a minibatch tile (the second CTA of a
// tile's last pair may have no rows: it loads its half of B, and skips its epilogue); the weight
// gradients stay on single CTAs (bound by their fp32 dW writes, they lose to the pairing).  The
// first CTA of the pair issues the MMAs; every CTA's epilogue drains its own TMEM rows.
//
// Roles: warp 0 lane 0 issues TMA tile loads into a ring of shared-memory stages; warp 1 owns the
// tensor memory and its lane 0 issues tcgen05.mma (M = 128, N = BN, K = 16) into one of two TMEM
// accumulators (MXFP8: the four K-major contractions run natively on E4M3 operands with
// kind::mxf8f6f4.block_scale, K = 32, their E8M0 scale atoms copied shared -> TMEM per stage); four epilogue warps (one per TMEM lane quarter) drain the other accumulator
// (tcgen05.ld), apply the epilogue math and write through swizzled shared tiles with TMA tile
// stores.  Every output element is produced by
// exactly one CTA with a fixed K order, so results are bitwise independent of the grid size and of
// the tile order.
#pragma once
#include <cstdint>
#include <cuda.h>

#include "mok_internal.cuh"
#include "mok_once.h"
#include "mok_ptx.cuh"

namespace mok {

enum GemmVariant : int {
  V_FWD_GATEUP = 0,
  V_FWD_DOWN = 1,
  V_DGRAD1 = 2,
  V_DGRAD2 = 3,
  V_WGRAD_GU = 4,
  V_WGRAD_D = 5,
};

constexpr int kBM = 128;      // MMA M (rows of the accumulator = TMEM lanes)
constexpr int kBK = 64;       // bf16 elements per K block: one 128-byte swizzle row
constexpr int kUmmaK = 16;    // K of one tcgen05.mma.kind::f16

struct GemmArgs {
  // work enumeration
  const int32_t* mblocks;  // row-tiled variants: 128-row blocks {expert, first row, valid, tile}
  const int32_t* tiles;    // minibatch tiles {expert, first row, valid, macro}
  const int32_t* meta;     // meta[2] = number of 128-row blocks
  const int32_t* poff;     // weight-gradient variants: padded expert offsets
  const int32_t* counts;   // BF16 weight gradients: routed rows per expert (the K loop stops at the
                           // last 64-row block holding one; the rest of the padding adds only zeros)
  int32_t E, I, H;
  int32_t n_tiles;         // N / BN
  int32_t m_tiles;         // weight-gradient variants: M / 128
  int32_t k_blocks;        // row-tiled variants: K / 64
  int32_t kb_split;        // DGRAD2: K blocks read from Wg before switching to Wu (I / 64; MX: I / 128)
  // epilogue operands
  void* out0;
  void* out1;
  void* out2;
  const void* in0;
  const void* in1;
  const float* row_weight;
  uint32_t* status;
  // MXFP8 variants: atom-tiled E8M0 scales (512-byte atoms of 128 rows x 4 k-groups, see
  // sf_atom_offset) of A (k_blocks atoms per 128-row tile) and of B (sfb_kq atoms per tile; sfb2
  // for DGRAD2's Wu half), and the scales the GATEUP / DGRAD1 epilogues write for the next GEMM.
  const uint8_t* sfa;
  const uint8_t* sfb;
  const uint8_t* sfb2;
  int32_t sfb_kq;
  int32_t out_kq;
  uint8_t* out_sf;
  // MXFP8 weight gradients: operands quantised along the routed rows, stored transposed [features,
  // rcap] (K-major for the MMA); sf_kq = 128-row K atoms of the routed-row capacity.  DGRAD1 writes their scales: out_sf2 ([dg | du],
  // A operand), out_sf3 (s * a, B operand in groups of sa_groups atoms).
  int32_t sf_kq;
  int32_t sa_groups;
  uint8_t* out_sf2;
  uint8_t* out_sf3;
  // CTA-pair row-tiled variants: pairs of 128-row blocks {expert, first row, tile, tile's first pair}
  const int4* pairs;
  // single-CTA tiles: 1 = the grid holds one CTA per unit and running CTAs take over the units of
  // CTAs that have not started (cluster launch control); 0 = static persistent round robin
  int32_t clc;
};

// Units of a CTA under cluster launch control travel from the producer thread, which asks for
// them, to the MMA thread and the epilogue warps through a ring in shared memory.
constexpr int kUnitRing = 8;


// A stage holds one K block of A and B as rows of 128 bytes (64 bf16 or 128 e4m3 along K) and, with
// MX, the K block's scale atoms: one for A's 128 rows, BN / 128 for B's rows.
//   bf16, and MX with BN = 128: two TMEM accumulators (the epilogue of one tile overlaps the
//     main loop of the next), four epilogue warps (eight, two per lane quarter with 64 columns
//     each, for the block-scaled DGRAD1 with SPLIT).  MX puts stage s's scale words in TMEM
//     columns 256 + 8 s ...
//   MX with BN = 256 ("wide"): two 256-column accumulators would fill TMEM and leave no room for
//     the scale words, so there is one; eight epilogue warps (two per lane quarter, 128 columns
//     each) copy it to registers and release it at once, then finish the tile's epilogue while
//     the next tile's MMAs run.  Stage s's scale words sit in columns 256 + 12 s ...  To fit four
//     stages, each epilogue warp stages its stores through a single 2 KB tile.
// The scale atoms of stage s live in a ring of their own after the A/B stages.
template <int VAR, int BN, bool MX, bool PAIR = false, bool SPLIT = false>
struct GemmCfg {
  static_assert(!MX || BN == 128 || BN == 256, "block-scaled tiles are 128 x 128 or 128 x 256");
  // block-scaled tiles run on single CTAs, except the weight gradients of long experts
  static_assert(!(MX && PAIR) || VAR == V_WGRAD_GU || VAR == V_WGRAD_D, "block-scaled pairs: weight gradients");
  static constexpr bool kWide = MX && BN == 256;
  // SPLIT (block-scaled DGRAD1 only): eight epilogue warps, two per lane quarter, 64 columns each
  static_assert(!SPLIT || (MX && VAR == V_DGRAD1 && BN == 128), "split epilogue: block-scaled DGRAD1");
  static constexpr bool kSplitEpi = SPLIT;
  static constexpr bool kDg1Mx = MX && VAR == V_DGRAD1;
  static constexpr int kAccBufs = kWide ? 1 : 2;
  static constexpr int kStages = MX ? (kWide ? (PAIR ? 6 : 4) : 5) : PAIR ? (BN == 256 ? 6 : 8) : (BN == 256 ? 4 : 6);
  static constexpr int kEpiWarps = kWide || kSplitEpi ? 8 : 4;  // warp w accesses TMEM lane quarter w % 4
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr uint32_t kABytes = kBM * 128;
  static constexpr uint32_t kBBytes = (PAIR ? BN / 2 : BN) * 128;  // the B rows this CTA holds
  static constexpr uint32_t kSfBytes = MX ? 512 + BN * 4 : 0;  // A atom, then B's BN / 128 atoms
  // bytes landing per stage (a pair counts both CTAs' loads, scale atoms included, on the first
  // CTA's barrier)
  static constexpr uint32_t kTxBytes = (PAIR ? 2 : 1) * (kABytes + kBBytes + kSfBytes);
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;           // multiple of 1024: swizzle atoms
  static constexpr uint32_t kTmemCols = MX ? 512 : 2 * BN;
  static constexpr uint32_t kSfCol0 = kAccBufs * BN;
  static constexpr uint32_t kSfCols = 4 + BN / 32;  // scale-word columns per stage (A, then B)
  static constexpr int kStageBufs = kWide ? 1 : 2;  // staging tiles per epilogue warp
  // (block-scaled DGRAD1 stores 1 KB tiles only: 32 rows x 32 E4M3 codes)
  static constexpr uint32_t kStageBufBytes = kWide ? 2048 : kDg1Mx ? 1024 : 4096;
  static constexpr uint32_t kStagingBytes = kEpiWarps * kStageBufs * kStageBufBytes;
  static constexpr uint32_t kSfRing = static_cast<uint32_t>(kStages) * kStageBytes;  // offset of the atom ring
  static constexpr uint32_t kStagingOff = kSfRing + static_cast<uint32_t>(kStages) * kSfBytes;
  // MXFP8 dgrad1: a 32 x 36 fp32 transpose scratch per epilogue warp (quantisation along the rows)
  static constexpr uint32_t kScratchWarp = 32u * 36u * 4u;
  static constexpr uint32_t kScratchBytes = kDg1Mx ? kEpiWarps * kScratchWarp : 0u;
  static constexpr uint32_t kScratchOff = kStagingOff + kStagingBytes;
  static constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(kScratchOff) + kScratchBytes + 512;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(!MX || kSfCol0 + kStages * kSfCols <= kTmemCols, "scale words fit in TMEM");
};

struct Unit {
  int e, row0, nt, mt, kblocks;
  bool peer_rows;  // CTA pair: the other CTA of the pair has rows too
};

// Units of work: one per CTA, or (PAIR) one per CTA pair.
template <int VAR, bool PAIR>
__device__ __forceinline__ int gemm_num_units(const GemmArgs& a) {
  if constexpr (VAR == V_WGRAD_GU || VAR == V_WGRAD_D) return a.E * (PAIR ? a.m_tiles / 2 : a.m_tiles) * a.n_tiles;
  else return (PAIR ? a.meta[3] : a.meta[2]) * a.n_tiles;
}

// Row-tiled variants: all units of one minibatch tile are consecutive, N tile outer and 128-row
// block inner, so a weight tile is reused by the tile's blocks while it sits in L2.
// CTA pairs (row-tiled variants; rank = this CTA's place in the pair): the same enumeration over
// pairs of row blocks (N tiles outer, pairs inner, within each minibatch tile).  A CTA without rows
// gets row0 = -1.
template <int VAR, bool MX, bool PAIR = false, int BN = 256>
__device__ __forceinline__ Unit gemm_decode(const GemmArgs& a, int u, int rank = 0) {
  Unit w;
  w.peer_rows = true;
  if constexpr (VAR == V_WGRAD_GU || VAR == V_WGRAD_D) {
    // CTA pairs (block-scaled, long experts): a unit is two consecutive M tiles, one per CTA
    const int mts = PAIR ? a.m_tiles / 2 : a.m_tiles;
    const int per_e = mts * a.n_tiles;
    w.e = u / per_e;
    const int r = u - w.e * per_e;
    if (MX && a.m_tiles * kBM <= a.n_tiles * BN) {
      // the smaller operand's tiles fastest: the tiles running together sweep all of its slices,
      // which then stay in L2 while the larger operand streams through once (with the larger one
      // fastest, a long expert's slices of it were re-read from DRAM for every group of tiles)
      w.nt = r / mts;
      w.mt = r - w.nt * mts;
    } else {
      w.mt = r / a.n_tiles;
      w.nt = r - w.mt * a.n_tiles;
    }
    if constexpr (PAIR) w.mt = 2 * w.mt + rank;
    const int p0 = __ldg(a.poff + w.e), p1 = __ldg(a.poff + w.e + 1);
    w.row0 = p0;
    if constexpr (MX) w.kblocks = (p1 - p0) / 128;  // block-scaled K blocks are the 128-row padding unit
    else w.kblocks = (__ldg(a.counts + w.e) + kBK - 1) / kBK;
  } else if constexpr (PAIR) {
    const int4 pe = __ldg(a.pairs + u / a.n_tiles);
    const int4 tl = __ldg(reinterpret_cast<const int4*>(a.tiles) + pe.z);
    const int nmb = (tl.z + kBM - 1) / kBM;
    const int npb = (nmb + 1) >> 1;
    const int local = u - pe.w * a.n_tiles;
    w.nt = local / npb;
    const int blk = 2 * (local - w.nt * npb) + rank;
    w.row0 = blk < nmb ? tl.y + blk * kBM : -1;
    w.peer_rows = (blk ^ 1) < nmb;
    w.e = pe.x;
    w.mt = 0;
    w.kblocks = a.k_blocks;
  } else {
    const int bq = u / a.n_tiles;
    const int4 mbk = __ldg(reinterpret_cast<const int4*>(a.mblocks) + bq);
    const int4 tl = __ldg(reinterpret_cast<const int4*>(a.tiles) + mbk.w);
    const int mb0 = tl.y / kBM;
    const int nmb = (tl.z + kBM - 1) / kBM;
    const int local = u - mb0 * a.n_tiles;
    w.nt = local / nmb;
    w.row0 = (mb0 + (local - w.nt * nmb)) * kBM;
    w.e = mbk.x;
    w.mt = 0;
    w.kblocks = a.k_blocks;
  }
  return w;
}

// Issue the loads of one K block into stage (sa, sb[, sf]), all completing on barrier `bar`.  MX
// (E4M3, K-major A and B, 128 K values per block): A rows of the routed operand, B rows of the
// caller's weight copy quantised along this GEMM's K ([E*I, H] Wg|Wu, [E*H, I] Wd, [E*I, H] Wd^T,
// [E*H, I] Wg^T|Wu^T), plus the block's scale atoms by untiled bulk copies: A's atom, and B's
// BN / 128 atoms, which the per-call re-tiling stores next to each other.  GATEUP's B tile (BN =
// 256) is 128 gate rows then the same 128 up rows; its atom pair is the gate atom, then the up.
template <int VAR, int BN, bool MX>
__device__ __forceinline__ void gemm_load(const GemmArgs& a, const Unit& w, int kb, uint32_t sa, uint32_t sb,
                                          uint32_t sf, uint32_t bar, const CUtensorMap* tA, const CUtensorMap* tB,
                                          const CUtensorMap* tB2) {
  if constexpr (MX && (VAR == V_WGRAD_GU || VAR == V_WGRAD_D)) {
    // weight gradients: A [M features, rows] and B [N features, rows], K-major with K = the
    // expert's routed rows; scale atoms indexed by the global 128-row block of the rows
    constexpr uint32_t kSfb = BN * 4;
    const int k0 = w.row0 + kb * 128;
    tma_load_2d(sa, tA, bar, k0, w.mt * kBM);
    tma_load_2d(sb, tB, bar, k0, w.nt * BN);
    bulk_load(sf, a.sfa + (static_cast<int64_t>(w.mt) * a.sf_kq + (k0 >> 7)) * 512, 512, bar);
    bulk_load(sf + 512, a.sfb + (static_cast<int64_t>(w.nt) * a.sf_kq + (k0 >> 7)) * kSfb, kSfb, bar);
    return;
  } else if constexpr (MX) {
    constexpr uint32_t kSfb = BN * 4;  // bytes of B scale atoms per K block; sf: A atom, then B's
    const int k0 = kb * 128;
    tma_load_2d(sa, tA, bar, k0, w.row0);
    bulk_load(sf, a.sfa + (static_cast<int64_t>(w.row0 >> 7) * a.k_blocks + kb) * 512, 512, bar);
    if constexpr (VAR == V_FWD_GATEUP) {
      static_assert(BN == 256, "MX gate/up tiles pair 128 gate and 128 up columns");
      const int n0 = w.e * a.I + w.nt * 128;
      tma_load_2d(sb, tB, bar, k0, n0);
      tma_load_2d(sb + 128 * 128, tB2, bar, k0, n0);
      bulk_load(sf + 512, a.sfb + (static_cast<int64_t>(n0 >> 7) * a.sfb_kq + kb) * kSfb, kSfb, bar);
    } else if constexpr (VAR == V_DGRAD2) {
      const bool first = kb < a.kb_split;
      const int kq = first ? kb : kb - a.kb_split;
      const int n0 = w.e * a.H + w.nt * BN;
      tma_load_2d(sb, first ? tB : tB2, bar, kq * 128, n0);
      bulk_load(sf + 512, (first ? a.sfb : a.sfb2) + (static_cast<int64_t>(n0 / BN) * a.sfb_kq + kq) * kSfb, kSfb,
                bar);
    } else {  // FWD_DOWN: B rows e*H + n; DGRAD1: B rows e*I + n
      const int n0 = w.e * (VAR == V_FWD_DOWN ? a.H : a.I) + w.nt * BN;
      tma_load_2d(sb, tB, bar, k0, n0);
      bulk_load(sf + 512, a.sfb + (static_cast<int64_t>(n0 / BN) * a.sfb_kq + kb) * kSfb, kSfb, bar);
    }
    return;
  }
  const int k0 = kb * kBK;
  if constexpr (VAR == V_FWD_GATEUP) {
    tma_load_2d(sa, tA, bar, k0, w.row0);
    const int n0 = w.e * a.I + w.nt * (BN / 2);
    tma_load_2d(sb, tB, bar, k0, n0);
    tma_load_2d(sb + (BN / 2) * 128, tB2, bar, k0, n0);
  } else if constexpr (VAR == V_FWD_DOWN) {
    tma_load_2d(sa, tA, bar, k0, w.row0);
    tma_load_2d(sb, tB, bar, k0, w.e * a.H + w.nt * BN);
  } else if constexpr (VAR == V_DGRAD1) {
    tma_load_2d(sa, tA, bar, k0, w.row0);
#pragma unroll
    for (int j = 0; j < BN / 64; ++j) tma_load_2d(sb + j * 8192, tB, bar, w.nt * BN + j * 64, w.e * a.H + k0);
  } else if constexpr (VAR == V_DGRAD2) {
    tma_load_2d(sa, tA, bar, k0, w.row0);
    const bool first = kb < a.kb_split;
    const CUtensorMap* tm = first ? tB : tB2;
    const int krow = w.e * a.I + (first ? k0 : k0 - a.kb_split * kBK);
#pragma unroll
    for (int j = 0; j < BN / 64; ++j) tma_load_2d(sb + j * 8192, tm, bar, w.nt * BN + j * 64, krow);
  } else {  // weight gradients: both operands MN-major, K runs over the expert's rows
    const int krow = w.row0 + k0;
#pragma unroll
    for (int j = 0; j < 2; ++j) tma_load_2d(sa + j * 8192, tA, bar, w.mt * kBM + j * 64, krow);
#pragma unroll
    for (int j = 0; j < BN / 64; ++j) tma_load_2d(sb + j * 8192, tB, bar, w.nt * BN + j * 64, krow);
  }
}

// CTA pair (BF16, row-tiled): the loads of this CTA's half of one K block, completing on the first
// CTA's barrier `bar` (shared::cluster address).  A: this CTA's 128 rows (none when row0 < 0); B:
// columns [rank * BN / 2, (rank + 1) * BN / 2) of the pair's N tile -- for GATEUP the first CTA
// holds the 128 gate rows, the second the same 128 up rows.
template <int VAR, int BN>
__device__ __forceinline__ void gemm_load_pair(const GemmArgs& a, const Unit& w, int kb, uint32_t sa, uint32_t sb,
                                               uint32_t bar, const CUtensorMap* tA, const CUtensorMap* tB,
                                               const CUtensorMap* tB2, int rank) {
  constexpr int HB = BN / 2;
  const int k0 = kb * kBK;
  if (w.row0 >= 0) tma_load_2d_pair(sa, tA, bar, k0, w.row0);
  if constexpr (VAR == V_FWD_GATEUP) {
    tma_load_2d_pair(sb, rank ? tB2 : tB, bar, k0, w.e * a.I + w.nt * HB);
  } else if constexpr (VAR == V_FWD_DOWN) {
    tma_load_2d_pair(sb, tB, bar, k0, w.e * a.H + w.nt * BN + rank * HB);
  } else if constexpr (VAR == V_DGRAD1) {
#pragma unroll
    for (int j = 0; j < HB / 64; ++j)
      tma_load_2d_pair(sb + j * 8192, tB, bar, w.nt * BN + rank * HB + j * 64, w.e * a.H + k0);
  } else {
    static_assert(VAR == V_DGRAD2, "row-tiled variants only");
    const bool first = kb < a.kb_split;
    const CUtensorMap* tm = first ? tB : tB2;
    const int krow = w.e * a.I + (first ? k0 : k0 - a.kb_split * kBK);
#pragma unroll
    for (int j = 0; j < HB / 64; ++j) tma_load_2d_pair(sb + j * 8192, tm, bar, w.nt * BN + rank * HB + j * 64, krow);
  }
}

// CTA pair, block-scaled weight gradients: this CTA's loads of one K block (128 routed rows), all
// completing on the first CTA's barrier `bar` (shared::cluster address): A = its own 128 M rows, B =
// its half of the pair's N tile, then the scale atoms -- its A rows' atom, and the atoms of all N
// rows of B (each CTA's TMEM must hold all of them) -- through pair-form loads over [atoms x 4, 128
// bytes] views of the atom arrays (tSfa: one atom per box; tSfb: BN / 128 atoms per box).
template <int BN>
__device__ __forceinline__ void gemm_load_pair_mx(const GemmArgs& a, const Unit& w, int kb, uint32_t sa, uint32_t sb,
                                                  uint32_t sf, uint32_t bar, const CUtensorMap* tA,
                                                  const CUtensorMap* tB, const CUtensorMap* tSfa,
                                                  const CUtensorMap* tSfb, int rank) {
  const int k0 = w.row0 + kb * 128;
  tma_load_2d_pair(sa, tA, bar, k0, w.mt * kBM);
  tma_load_2d_pair(sb, tB, bar, k0, w.nt * BN + rank * (BN / 2));
  tma_load_2d_pair(sf, tSfa, bar, 0, (w.mt * a.sf_kq + (k0 >> 7)) * 4);
  tma_load_2d_pair(sf + 512, tSfb, bar, 0, (w.nt * a.sf_kq + (k0 >> 7)) * 4 * (BN / 128));
}

// SwiGLU pieces in fp32 with the fast approximate division (about 2 ulp; the results are rounded to
// bf16 next, 2^-9).
__device__ __forceinline__ float sigmoid_f(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ uint4 ldg_v4(const uint16_t* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

// Per-warp output stager: NBUF shared-memory tiles (4 KB apart) of 32 rows x ROW bytes in the TMA
// swizzle layout of that row size -- 128-byte rows: 16-byte chunk j of row r sits at chunk
// j ^ (r & 7); 64-byte rows: at j ^ ((r >> 1) & 3); 32-byte rows: at j ^ ((r >> 2) & 1).  All keep
// the 32 lanes' row writes free of bank conflicts.  Each filled tile leaves as one asynchronous
// TMA tile store; a tile is refilled only after its previous store has finished reading it, so up
// to NBUF stores are in flight.
template <int NBUF, uint32_t BUFBYTES>
struct Stager {
  uint32_t buf0;
  int cur;
  int lane;
  __device__ __forceinline__ uint32_t acquire() {
    if (lane == 0) bulk_wait_read<NBUF - 1>();
    __syncwarp();
    const uint32_t b = buf0 + static_cast<uint32_t>(cur) * BUFBYTES;
    cur = cur + 1 == NBUF ? 0 : cur + 1;
    return b;
  }
  // Lane r writes its row (ROW / 16 chunks of 16 bytes) and the warp stores the tile at (c0, c1).
  template <int ROW>
  __device__ __forceinline__ void put(const uint4* ch, const CUtensorMap* tm, int c0, int c1, bool ef = false) {
    static_assert(ROW == 128 || ROW == 64 || ROW == 32, "row size with a TMA swizzle mode");
    static_assert(32 * ROW <= BUFBYTES, "tile fits the staging buffer");
    const uint32_t b = acquire();
    const uint32_t row = b + static_cast<uint32_t>(lane) * ROW;
    const int sw = ROW == 128 ? (lane & 7) : ROW == 64 ? ((lane >> 1) & 3) : ((lane >> 2) & 1);
#pragma unroll
    for (int j = 0; j < ROW / 16; ++j) st_shared_v4(row + (static_cast<uint32_t>(j ^ sw) << 4), ch[j]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (ef) tma_store_2d_evict_first(tm, b, c0, c1);
      else tma_store_2d(tm, b, c0, c1);
      bulk_commit();
    }
  }
  __device__ __forceinline__ void drain() {
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
};

// Output stager shared by the four epilogue warps: two 16 KB tiles of 128 rows x 128 bytes (the
// 128-byte swizzle) in the staging area.  Warp q writes rows q * 32 + lane; after a group barrier
// (an mbarrier of 128 arrivals, bounded wait) one thread stores the tile with a single TMA store,
// a quarter of the stores of per-warp 32-row tiles.  A tile is refilled only after its previous
// store has read it.  Returns false after an abort.
struct GroupStager {
  uint32_t base;  // 32 KB: tile 0, then tile 1
  uint32_t bar;
  uint32_t phase;
  int cur;
  int row;        // this thread's row in the tile (q * 32 + lane)
  bool leader;
  __device__ __forceinline__ bool sync(volatile int* abort, uint32_t* status) {
    mbar_arrive(bar);
    if (!mbar_wait(bar, phase, abort, status)) return false;
    phase ^= 1u;
    return true;
  }
  __device__ __forceinline__ bool put(const uint4 (&ch)[8], const CUtensorMap* tm, int c0, int row0,
                                      volatile int* abort, uint32_t* status, bool ef = false) {
    const uint32_t tile = base + static_cast<uint32_t>(cur) * 16384u;
    const uint32_t r = tile + static_cast<uint32_t>(row) * 128u;
#pragma unroll
    for (int j = 0; j < 8; ++j) st_shared_v4(r + (static_cast<uint32_t>(j ^ (row & 7)) << 4), ch[j]);
    fence_proxy_async_smem();
    if (!sync(abort, status)) return false;  // all 128 rows are in the tile
    if (leader) {
      if (ef) tma_store_2d_evict_first(tm, tile, c0, row0);
      else tma_store_2d(tm, tile, c0, row0);
      bulk_commit();
      bulk_wait_read<1>();  // the other tile's store has read it
    }
    cur ^= 1;
    return sync(abort, status);
  }
};

template <int N>
__device__ __forceinline__ void pack_bf16(const float* v, uint4* ch) {
#pragma unroll
  for (int j = 0; j < N / 8; ++j)
    ch[j] = make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                       pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r0[32], r1[32];
  tmem_ld_32x32b_x32(taddr, r0);
  tmem_ld_32x32b_x32(taddr + 32, r1);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = __uint_as_float(r0[i]);
    v[32 + i] = __uint_as_float(r1[i]);
  }
}

__device__ __forceinline__ void unpack8(uint4 x, float* v) {
  v[0] = bf16_lo(x.x); v[1] = bf16_hi(x.x); v[2] = bf16_lo(x.y); v[3] = bf16_hi(x.y);
  v[4] = bf16_lo(x.z); v[5] = bf16_hi(x.z); v[6] = bf16_lo(x.w); v[7] = bf16_hi(x.w);
}

// Hand the accumulator back to the MMA warp once this thread has read its last TMEM column.  PAIR:
// `tempty` is the shared::cluster address of the first CTA's barrier.
template <bool PAIR = false>
__device__ __forceinline__ void release_acc(uint32_t tempty) {
  tc_fence_before();
  if constexpr (PAIR) mbar_arrive_cluster(tempty);
  else mbar_arrive(tempty);
}

// The forward context's g, u, a for one 32-column chunk of one row (DGRAD1 epilogue operand).
struct Dg1Chunk {
  uint4 g[4], u[4], a[4];
};
__device__ __forceinline__ void dgrad1_fetch(const GemmArgs& a, const Unit& w, int q, int lane, int c, Dg1Chunk& d) {
  const int64_t row = w.row0 + q * 32 + lane;
  const int64_t I = a.I;
  const uint16_t* gu = static_cast<const uint16_t*>(a.in0) + row * 2 * I + c;
  const uint16_t* av = static_cast<const uint16_t*>(a.in1) + row * I + c;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    d.g[j] = ldg_v4(gu + 8 * j);
    d.u[j] = ldg_v4(gu + I + 8 * j);
    d.a[j] = ldg_v4(av + 8 * j);
  }
}

// MX quantisation of one 32 x 32 block along the rows: lane = row, v[j] = column j (feature f0 + j).
// The block is transposed through the warp's fp32 scratch (element (r, c) at r * 36 + c: each lane
// writes its row with eight 16-byte stores, the 8 lanes of a quarter warp in 8 different bank
// groups; the column reads of the 32 lanes hit 32 different banks; every address is a per-lane base
// plus a constant, so no table of addresses stays live), lane j then quantises column j
// over the 32 rows as one MX block, and its 32 codes leave as row j of a byte tile stored at
// (row rowc, feature f0) of the transposed [features, rows] copy; lane j writes column j's scale
// into the atom-tiled array (groups of 2^gl atoms, kq atoms along K).
template <class Stg>
__device__ __forceinline__ void quant_rows_store(const float (&v)[32], uint32_t scratch, Stg& stg,
                                                 const CUtensorMap* tm, uint8_t* sf, int rowc, int f0, int kq, int gl,
                                                 int lane) {
  const uint32_t row = scratch + static_cast<uint32_t>(lane) * 144;
#pragma unroll
  for (int c = 0; c < 32; c += 4)
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(row + 4u * c), "f"(v[c]), "f"(v[c + 1]),
                 "f"(v[c + 2]), "f"(v[c + 3])
                 : "memory");
  __syncwarp();
  float col[32];
  const uint32_t colp = scratch + static_cast<uint32_t>(lane) * 4;
#pragma unroll
  for (int r = 0; r < 32; ++r) asm volatile("ld.shared.f32 %0, [%1];" : "=f"(col[r]) : "r"(colp + 144u * r) : "memory");
  __syncwarp();
  uint32_t codes[8];
  const uint32_t sb = mx_quant32<false>(col, codes);
  const uint4 ch[2] = {make_uint4(codes[0], codes[1], codes[2], codes[3]),
                       make_uint4(codes[4], codes[5], codes[6], codes[7])};
  stg.template put<32>(ch, tm, rowc, f0, true);  // read by the weight gradients, after the next GEMM
  sf[sf_atom_offset_p2(f0 + lane, rowc >> 5, kq, gl)] = static_cast<uint8_t>(sb);
}

// Epilogue of one unit for the warp's 32 accumulator rows (slab `q`); lane = row in the slab; `h`
// = the warp's column half in the wide (8-warp) configuration.  tO0 / tO1 / tO2 are the output
// tensor maps of the variant; `tempty` is released as soon as the last accumulator column has been
// read.  `pre` holds DGRAD1's first prefetched context chunk.
template <int VAR, int BN, bool MX, bool PAIR, bool SPLIT, class Stg>
__device__ __forceinline__ void gemm_epilogue(const GemmArgs& a, const Unit& w, int q, int h, int lane,
                                              uint32_t taddr, Stg& stg, uint32_t scratch, const CUtensorMap* tO0,
                                              const CUtensorMap* tO1, const CUtensorMap* tO2, uint32_t tempty,
                                              Dg1Chunk& pre, GroupStager& gs, uint32_t epi_bar,
                                              uint32_t& epi_phase, volatile int* abort_flag) {
  if constexpr (VAR == V_FWD_GATEUP && MX) {
    // accumulator columns [0, 128) are gate, [128, 256) up, for I columns nt*128 ...; this warp
    // takes 64 of them (half h).  g and u leave in fp32 (the backward re-quantises dg, du from
    // them); a = silu(g) u leaves MX-quantised along I: its dequantised values in bf16 for the
    // backward, its E4M3 codes and scales for the down projection.
    const int i0 = w.nt * 128 + 64 * h;
    const int rowc = w.row0 + q * 32;
    const int64_t row = rowc + lane;
    uint32_t gr[64], ur[64];
    tmem_ld_32x32b_x32(taddr + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(gr));
    tmem_ld_32x32b_x32(taddr + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(gr + 32));
    tmem_ld_32x32b_x32(taddr + 128 + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(ur));
    tmem_ld_32x32b_x32(taddr + 128 + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(ur + 32));
    tmem_ld_wait();
    release_acc<PAIR>(tempty);
#pragma unroll
    for (int c = 0; c < 64; c += 32) {
      uint4 ch[4];
#pragma unroll
      for (int c16 = 0; c16 < 32; c16 += 16) {  // fp32 g, u in 16-column (64-byte) tiles
#pragma unroll
        for (int j = 0; j < 4; ++j)
          ch[j] = make_uint4(gr[c + c16 + 4 * j], gr[c + c16 + 4 * j + 1], gr[c + c16 + 4 * j + 2],
                             gr[c + c16 + 4 * j + 3]);
        stg.template put<64>(ch, tO0, i0 + c + c16, rowc, true);  // context: read in the backward
#pragma unroll
        for (int j = 0; j < 4; ++j)
          ch[j] = make_uint4(ur[c + c16 + 4 * j], ur[c + c16 + 4 * j + 1], ur[c + c16 + 4 * j + 2],
                             ur[c + c16 + 4 * j + 3]);
        stg.template put<64>(ch, tO0, a.I + i0 + c + c16, rowc, true);
      }
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = silu_f(__uint_as_float(gr[c + i])) * __uint_as_float(ur[c + i]);
      uint32_t codes[8];
      const uint32_t sbyte = mx_quant32(v, codes);
      pack_bf16<32>(v, ch);
      stg.template put<64>(ch, tO1, i0 + c, rowc);
      ch[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
      ch[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
      stg.template put<32>(ch, tO2, i0 + c, rowc);
      a.out_sf[sf_atom_offset(row, (i0 + c) >> 5, a.out_kq)] = static_cast<uint8_t>(sbyte);
    }
  } else if constexpr ((VAR == V_FWD_DOWN || VAR == V_DGRAD2) && MX && BN == 256) {
    // wide tile: this warp's 128 columns go to registers, the accumulator is released, then the
    // bf16 rows leave in four 32-column (64-byte) tiles
    const int rowc = w.row0 + q * 32;
    uint32_t r[128];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      tmem_ld_32x32b_x32(taddr + 128 * h + 32 * j, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * j));
    tmem_ld_wait();
    release_acc<PAIR>(tempty);
#pragma unroll
    for (int c = 0; c < 128; c += 32) {
      uint4 ch[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ch[j] = make_uint4(pack_bf16x2(__uint_as_float(r[c + 8 * j]), __uint_as_float(r[c + 8 * j + 1])),
                           pack_bf16x2(__uint_as_float(r[c + 8 * j + 2]), __uint_as_float(r[c + 8 * j + 3])),
                           pack_bf16x2(__uint_as_float(r[c + 8 * j + 4]), __uint_as_float(r[c + 8 * j + 5])),
                           pack_bf16x2(__uint_as_float(r[c + 8 * j + 6]), __uint_as_float(r[c + 8 * j + 7])));
      stg.template put<64>(ch, tO0, w.nt * BN + 128 * h + c, rowc);
    }
  } else if constexpr (VAR == V_FWD_GATEUP) {
    // columns [0, BN/2) of the accumulator are gate, [BN/2, BN) up, for I columns i0 ...
    const int i0 = w.nt * (BN / 2);
#pragma unroll 1
    for (int c = 0; c < BN / 2; c += 64) {
      float g[64], u[64];
      tmem_ld64(taddr + c, g);
      tmem_ld64(taddr + BN / 2 + c, u);
      if (c + 64 >= BN / 2) release_acc<PAIR>(tempty);
      uint4 ch[8];
      pack_bf16<64>(g, ch);  // g, u: the context, read in the backward
      if (!gs.put(ch, tO0, i0 + c, w.row0, abort_flag, a.status, true)) return;
      pack_bf16<64>(u, ch);
      if (!gs.put(ch, tO0, a.I + i0 + c, w.row0, abort_flag, a.status, true)) return;
#pragma unroll
      for (int i = 0; i < 64; ++i) g[i] = silu_f(g[i]) * u[i];
      pack_bf16<64>(g, ch);
      if (!gs.put(ch, tO1, i0 + c, w.row0, abort_flag, a.status)) return;
    }
  } else if constexpr (VAR == V_FWD_DOWN || VAR == V_DGRAD2) {
#pragma unroll 1
    for (int c = 0; c < BN; c += 64) {
      float v[64];
      tmem_ld64(taddr + c, v);
      if (c + 64 >= BN) release_acc<PAIR>(tempty);
      uint4 ch[8];
      pack_bf16<64>(v, ch);
      if (!gs.put(ch, tO0, w.nt * BN + c, w.row0, abort_flag, a.status)) return;
    }
  } else if constexpr (VAR == V_DGRAD1 && MX) {
    // MXFP8: dA' = dYq Wd^T (block-scaled), the SwiGLU backward from the forward's fp32 g, u, and
    // per 32-column chunk:
    //   dS partial from a's quantisation along I (the context);
    //   dg, du quantised along I (row-major codes + A atoms) for the second data-gradient GEMM;
    //   dg, du and s * a quantised along this warp's 32 routed rows, for the weight-gradient GEMMs.
    // SPLIT (eight warps): this one takes columns [64 h, 64 h + 64) of the tile, and its dS
    // partial has a slot of its own (two per N tile and row).
    const int64_t row = w.row0 + q * 32 + lane;
    const int64_t I = a.I;
    const int i0 = w.nt * BN;
    const float* gu = static_cast<const float*>(a.in0) + row * 2 * I;
    const uint16_t* av = static_cast<const uint16_t*>(a.in1) + row * I;
    const float s = __ldg(a.row_weight + row);
    const int rowc = w.row0 + q * 32;
    float part = 0.0f;
    const int c_beg = SPLIT ? 64 * h : 0, c_end = SPLIT ? 64 * h + 64 : BN;
    const int sa_gl = a.sa_groups == 2 ? 1 : 0;  // s * a's scales: groups of 1 or 2 atoms
#pragma unroll 1
    for (int c = c_beg; c < c_end; c += 32) {
      // g and u of 32 columns; s * a first (it needs no accumulator), then dA' from TMEM, and dg,
      // du computed in place of u, g: at most four 32-value arrays are live at once
      float g[32], u[32];
      {
        const float4* gp = reinterpret_cast<const float4*>(gu + i0 + c);
        const float4* up = reinterpret_cast<const float4*>(gu + I + i0 + c);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 x = __ldg(gp + j), y = __ldg(up + j);
          g[4 * j] = x.x, g[4 * j + 1] = x.y, g[4 * j + 2] = x.z, g[4 * j + 3] = x.w;
          u[4 * j] = y.x, u[4 * j + 1] = y.y, u[4 * j + 2] = y.z, u[4 * j + 3] = y.w;
        }
      }
      // the products below run two lanes of fp32 per instruction (mul / fma .f32x2)
      float sg[32];
      {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) sg[i] = sigmoid_f(g[i]);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {  // s * (g * sigmoid(g) * u)
          float t0, t1;
          mul_f32x2(t0, t1, g[i], g[i + 1], sg[i], sg[i + 1]);
          mul_f32x2(t0, t1, t0, t1, u[i], u[i + 1]);
          mul_f32x2(v[i], v[i + 1], s, s, t0, t1);
        }
        quant_rows_store(v, scratch, stg, tO1, a.out_sf3, rowc, i0 + c, a.sf_kq, sa_gl, lane);
      }
      {
        uint32_t rv[32];
        tmem_ld_32x32b_x32(taddr + c, rv);
        tmem_ld_wait();
        if (c + 32 >= c_end) release_acc<PAIR>(tempty);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float a8[8];
          unpack8(ldg_v4(av + i0 + c + 8 * j), a8);
#pragma unroll
          for (int k = 0; k < 8; ++k) part = fmaf(__uint_as_float(rv[8 * j + k]), a8[k], part);
        }
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          // da = s dA'; x = da sigmoid(g); du = x g; dg = x u (1 + g (1 - sigmoid(g)))
          float da0, da1, x0, x1, w0, w1, y0, y1;
          mul_f32x2(da0, da1, s, s, __uint_as_float(rv[i]), __uint_as_float(rv[i + 1]));
          mul_f32x2(x0, x1, da0, da1, sg[i], sg[i + 1]);
          fma_f32x2(w0, w1, sg[i], sg[i + 1], -1.0f, -1.0f, 1.0f, 1.0f);
          fma_f32x2(w0, w1, g[i], g[i + 1], w0, w1, 1.0f, 1.0f);
          mul_f32x2(y0, y1, x0, x1, u[i], u[i + 1]);
          mul_f32x2(g[i], g[i + 1], x0, x1, g[i], g[i + 1]);  // du
          mul_f32x2(u[i], u[i + 1], y0, y1, w0, w1);          // dg
        }
      }
      uint4 ch[2];
      uint32_t codes[8];
      quant_rows_store(u, scratch, stg, tO0, a.out_sf2, rowc, i0 + c, a.sf_kq, 0, lane);
      uint32_t sb = mx_quant32<false>(u, codes);
      ch[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
      ch[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
      stg.template put<32>(ch, tO2, i0 + c, rowc);
      a.out_sf[sf_atom_offset(row, (i0 + c) >> 5, a.out_kq)] = static_cast<uint8_t>(sb);
      quant_rows_store(g, scratch, stg, tO0, a.out_sf2, rowc, a.I + i0 + c, a.sf_kq, 0, lane);
      sb = mx_quant32<false>(g, codes);
      ch[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
      ch[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
      stg.template put<32>(ch, tO2, a.I + i0 + c, rowc);
      a.out_sf[sf_atom_offset(row, (a.I + i0 + c) >> 5, a.out_kq)] = static_cast<uint8_t>(sb);
    }
    if constexpr (SPLIT) static_cast<float*>(a.out2)[(row * a.n_tiles + w.nt) * 2 + h] = part;
    else static_cast<float*>(a.out2)[row * a.n_tiles + w.nt] = part;
  } else if constexpr (VAR == V_DGRAD1) {
    // dA' = dY Wd (this tile's BN columns of I); the forward's g, u, a come from the context,
    // fetched one 32-column chunk ahead.  dg, du and s*a leave as 32 x 64-byte tiles.
    const int64_t row = w.row0 + q * 32 + lane;
    const int i0 = w.nt * BN;
    const float s = __ldg(a.row_weight + row);
    const int rowc = w.row0 + q * 32;
    float part = 0.0f;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      const Dg1Chunk cur = pre;
      if (c + 32 < BN) dgrad1_fetch(a, w, q, lane, i0 + c + 32, pre);
      uint32_t rv[32];
      tmem_ld_32x32b_x32(taddr + c, rv);
      tmem_ld_wait();
      if (c + 32 >= BN) release_acc<PAIR>(tempty);
      uint4 cdg[4], cdu[4], csa[4];
      {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float g8[8], u8[8], a8[8], dg[8], du[8], sa[8];
          unpack8(cur.g[j], g8);
          unpack8(cur.u[j], u8);
          unpack8(cur.a[j], a8);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float dap = __uint_as_float(rv[8 * j + k]);
            part = fmaf(dap, a8[k], part);
            const float da = s * dap;
            const float sg = sigmoid_f(g8[k]);
            dg[k] = da * u8[k] * sg * (1.0f + g8[k] * (1.0f - sg));
            du[k] = da * g8[k] * sg;
            sa[k] = s * a8[k];
          }
          pack_bf16<8>(dg, cdg + j);
          pack_bf16<8>(du, cdu + j);
          pack_bf16<8>(sa, csa + j);
        }
      }
      stg.template put<64>(cdg, tO0, i0 + c, rowc);
      stg.template put<64>(cdu, tO0, a.I + i0 + c, rowc);
      stg.template put<64>(csa, tO1, i0 + c, rowc);
    }
    static_cast<float*>(a.out2)[row * a.n_tiles + w.nt] = part;
  } else if constexpr ((VAR == V_WGRAD_GU || VAR == V_WGRAD_D) && MX && BN == 256) {
    // wide MXFP8 weight-gradient tile: this warp's 128 fp32 columns go to registers, the accumulator
    // is released, then the rows leave in 16-column (64-byte) tiles of the warp's own 32 rows
    // (measured: 128-row tiles shared by four warps, single-buffered in the wide configuration's
    // staging, were up to 15 % slower here).  Experts without rows: zeros.
    const bool empty = w.kblocks == 0;
    const int m0 = w.mt * kBM + q * 32;
    const CUtensorMap* tm;
    int r0;
    if constexpr (VAR == V_WGRAD_GU) {
      tm = m0 < a.I ? tO0 : tO1;
      r0 = w.e * a.I + (m0 < a.I ? m0 : m0 - a.I);
    } else {
      tm = tO0;
      r0 = w.e * a.H + m0;
    }
    uint32_t r[128];
    if (!empty) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        tmem_ld_32x32b_x32(taddr + 128 * h + 32 * j, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * j));
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int i = 0; i < 128; ++i) r[i] = 0u;
    }
    release_acc<PAIR>(tempty);
#pragma unroll
    for (int c = 0; c < 128; c += 16) {
      uint4 ch[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ch[j] = make_uint4(r[c + 4 * j], r[c + 4 * j + 1], r[c + 4 * j + 2], r[c + 4 * j + 3]);
      stg.template put<64>(ch, tm, w.nt * BN + 128 * h + c, r0, true);  // dW: not read again
    }
  } else {
    // weight gradients, fp32 out in 128-row x 32-column tiles of the group stager (a quarter of the
    // TMA stores of per-warp 32-row tiles: 5 % (384 rows per expert) to 17 % (64 rows per expert)
    // faster).  Experts without rows get zeros.
    const bool empty = w.kblocks == 0;
    const int mt0 = w.mt * kBM;
    const CUtensorMap* tm;
    int rt;
    if constexpr (VAR == V_WGRAD_GU) {
      tm = mt0 < a.I ? tO0 : tO1;
      rt = w.e * a.I + (mt0 < a.I ? mt0 : mt0 - a.I);
    } else {
      tm = tO0;
      rt = w.e * a.H + mt0;
    }
    if (empty) release_acc<PAIR>(tempty);
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t rv[32];
      if (!empty) {
        tmem_ld_32x32b_x32(taddr + c, rv);
        tmem_ld_wait();
        if (c + 32 >= BN) release_acc<PAIR>(tempty);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) rv[i] = 0u;
      }
      uint4 ch[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) ch[j] = make_uint4(rv[4 * j], rv[4 * j + 1], rv[4 * j + 2], rv[4 * j + 3]);
      if (!gs.put(ch, tm, w.nt * BN + c, rt, abort_flag, a.status, true)) return;  // dW: not read again
    }
  }
}

// Bounded wait that ignores the abort flag: used only while winding down.
__device__ __forceinline__ bool mbar_wait_final(uint32_t bar, uint32_t parity, uint32_t* status) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs / 4) {
      record_status(status, MOK_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

template <int VAR, int BN, bool MX, bool PAIR, bool SPLIT>
__global__ void __launch_bounds__(GemmCfg<VAR, BN, MX, PAIR, SPLIT>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmO0,
                const __grid_constant__ CUtensorMap tmO1, const __grid_constant__ CUtensorMap tmO2,
                const GemmArgs args) {
  using C = GemmCfg<VAR, BN, MX, PAIR, SPLIT>;
  constexpr bool kAmn = (VAR == V_WGRAD_GU || VAR == V_WGRAD_D) && !MX;
  constexpr bool kBmn = (VAR >= V_DGRAD1) && !MX;
  constexpr uint32_t kIdesc = idesc_bf16(PAIR ? 2 * kBM : kBM, BN, kAmn, kBmn);
  constexpr int S = C::kStages;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms need 1024-byte alignment
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sf_ring = base + C::kSfRing;
  const uint32_t staging = base + C::kStagingOff;
  const uint32_t scratch0 = base + C::kScratchOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + C::kScratchOff + C::kScratchBytes);
  // bars[0..S) full, [S..2S) empty, [2S, 2S+2) accumulator full, [2S+2, 2S+4) accumulator empty,
  // [2S+4] drain, [2S+5, 2S+7) epilogue group barriers.  A pair uses the first CTA's full and accumulator-empty barriers (both CTAs'
  // loads and epilogues count there) and each CTA's own empty, accumulator-full and drain
  // barriers (the first CTA's commits arrive on both).
  // [2S+7, +8) unit ring full, [2S+15, +8) unit ring empty, [2S+23] cluster-launch-control answer;
  // then the 16-byte answer, the ring's units, the TMEM address and the abort flag
  const uint32_t uq_full0 = smem_u32(bars + 2 * S + 7), uq_empty0 = smem_u32(bars + 2 * S + 15);
  const uint32_t clc_bar = smem_u32(bars + 2 * S + 23);
  const uint32_t clc_resp = smem_u32(bars + 2 * S + 24);
  volatile int* unit_q = reinterpret_cast<volatile int*>(bars + 2 * S + 26);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 30);
  // group barriers of four epilogue warps (the wide MX tiles' column half h uses epi_bar + 8 h)
  const uint32_t epi_bar = smem_u32(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const int unit0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int unit_step = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), (PAIR ? 2 : 1) * 32 * C::kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    mbar_init(epi_bar, 128);
    mbar_init(epi_bar + 8, 128);
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(uq_full0 + 8u * i, 1);
      mbar_init(uq_empty0 + 8u * i, 1 + C::kEpiWarps);
    }
    mbar_init(clc_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmB2);
    tma_prefetch_desc(&tmO0);
    tma_prefetch_desc(&tmO1);
    tma_prefetch_desc(&tmO2);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR) cluster_sync();  // the peer's barriers are initialised before any remote arrive
  else __syncthreads();
  // the set-up above touches no global memory; from here on the producers' results are needed
  pdl_wait();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_units = gemm_num_units<VAR, PAIR>(args);
  const bool clc = !PAIR && args.clc != 0;
  // consumers' side of the unit ring: the next unit, -1 at the end (or after an abort)
  auto unit_pop = [&](int& qi, uint32_t& qph, bool one_per_warp) -> int {
    int v = -1;
    if (!one_per_warp || lane == 0) {
      if (mbar_wait(uq_full0 + 8u * qi, qph, abort_flag, args.status)) v = unit_q[qi];
      mbar_arrive(uq_empty0 + 8u * qi);
    }
    if (one_per_warp) v = __shfl_sync(0xffffffffu, v, 0);
    if (++qi == kUnitRing) {
      qi = 0;
      qph ^= 1u;
    }
    return v;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      int last_parity[S];
      for (int s = 0; s < S; ++s) last_parity[s] = -1;
      bool ok = true;
      int qi = 0;
      uint32_t qph = 0, clc_phase = 0;
      bool clc_pending = false;
      for (int u = unit0; ok;) {
        if (clc) {  // hand the unit to the other roles, ask for the next one while it runs
          const int uu = u < num_units ? u : -1;
          if (!mbar_wait(uq_empty0 + 8u * qi, qph ^ 1u, abort_flag, args.status)) break;
          unit_q[qi] = uu;
          mbar_arrive(uq_full0 + 8u * qi);
          if (++qi == kUnitRing) {
            qi = 0;
            qph ^= 1u;
          }
          if (uu < 0) break;
          mbar_arrive_expect_tx(clc_bar, 16);
          clc_try_cancel(clc_resp, clc_bar);
          clc_pending = true;
        } else if (u >= num_units) {
          break;
        }
        const Unit w = gemm_decode<VAR, MX, PAIR, BN>(args, u, rank);
        for (int kb = 0; kb < w.kblocks; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * C::kStageBytes;
          if constexpr (PAIR && MX) {  // block-scaled weight gradients (the scale maps ride in B2 and O2)
            if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), C::kTxBytes);
            gemm_load_pair_mx<BN>(args, w, kb, sa, sa + C::kABytes, sf_ring + stage * C::kSfBytes,
                                  mapa_shared(full_bar(stage), 0), &tmA, &tmB, &tmB2, &tmO2, rank);
          } else if constexpr (PAIR) {
            if (rank == 0)
              mbar_arrive_expect_tx(full_bar(stage), w.peer_rows ? C::kTxBytes : C::kTxBytes - C::kABytes);
            gemm_load_pair<VAR, BN>(args, w, kb, sa, sa + C::kABytes, mapa_shared(full_bar(stage), 0), &tmA, &tmB,
                                    &tmB2, rank);
          } else {
            mbar_arrive_expect_tx(full_bar(stage), C::kTxBytes);
            gemm_load<VAR, BN, MX>(args, w, kb, sa, sa + C::kABytes, sf_ring + stage * C::kSfBytes, full_bar(stage),
                                   &tmA, &tmB, &tmB2);
          }
          last_parity[stage] = static_cast<int>(phase);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (clc) {
          // the next unit: the CTA the answer cancelled; CTAs past the last unit (row-tiled grids
          // are sized for the most units a schedule can have) are cancelled and dropped here, so
          // they never start; nothing cancelled: the next round ends the ring
          int nx = num_units;
          while (ok) {
            if (!mbar_wait(clc_bar, clc_phase, abort_flag, args.status)) {
              ok = false;
              break;
            }
            clc_phase ^= 1u;
            clc_pending = false;
            nx = clc_cancelled_x(clc_resp);
            if (nx < num_units) break;
            mbar_arrive_expect_tx(clc_bar, 16);
            clc_try_cancel(clc_resp, clc_bar);
            clc_pending = true;
          }
          if (!ok) break;
          u = nx < 0 ? num_units : nx;
        } else {
          u += unit_step;
        }
      }
      if (clc_pending) mbar_wait_final(clc_bar, clc_phase, args.status);  // the answer lands before exit
      // wind down: let the copies already issued land before the CTA exits (a pair's second CTA
      // counts its copies on the first CTA's barriers, which that CTA waits for)
      if (!ok && rank == 0) {
        for (int s = 0; s < S; ++s)
          if (last_parity[s] >= 0) mbar_wait_final(full_bar(s), static_cast<uint32_t>(last_parity[s]), args.status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (the first CTA of a pair) ----------------
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      int qi = 0;
      uint32_t qph = 0;
      for (int u = unit0; ok; u += unit_step) {
        if (clc) {
          u = unit_pop(qi, qph, false);
          if (u < 0) break;
        } else if (u >= num_units) {
          break;
        }
        const Unit w = gemm_decode<VAR, MX, PAIR, BN>(args, u, rank);
        if (!mbar_wait<PAIR>(tempty_bar(acc), acc_phase ^ 1u, abort_flag, args.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < w.kblocks; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + stage * C::kStageBytes, sb = sa + C::kABytes;
          if constexpr (MX) {
            // this stage's scale atoms -> its own 8 TMEM columns (A words, then B words); the copies
            // and the MMAs that read them execute in issue order
            const uint32_t sf = sf_ring + stage * C::kSfBytes;
            const uint32_t tsf = tmem_base + C::kSfCol0 + static_cast<uint32_t>(stage) * C::kSfCols;
            if constexpr (PAIR) {  // both CTAs' atoms, each into its own TMEM
              tmem_cp_sf_atom_pair(tsf, sdesc_plain(sf));
#pragma unroll
              for (int j = 0; j < BN / 128; ++j) tmem_cp_sf_atom_pair(tsf + 4 + 4 * j, sdesc_plain(sf + 512 + 512 * j));
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                umma_mxf8_pair(d_tmem, sdesc_sw128(sa + ks * 32, 16, 1024), sdesc_sw128(sb + ks * 32, 16, 1024),
                               idesc_mx(2 * kBM, BN, static_cast<uint32_t>(ks)), (kb | ks) != 0 ? 1u : 0u, tsf,
                               tsf + 4);
            } else {
              tmem_cp_sf_atom(tsf, sdesc_plain(sf));
#pragma unroll
              for (int j = 0; j < BN / 128; ++j)  // B row n's word lands in column n / 32
                tmem_cp_sf_atom(tsf + 4 + 4 * j, sdesc_plain(sf + 512 + 512 * j));
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)  // K = 32 e4m3 (32 bytes) per instruction; k-group ks
                umma_mxf8(d_tmem, sdesc_sw128(sa + ks * 32, 16, 1024), sdesc_sw128(sb + ks * 32, 16, 1024),
                          idesc_mx(kBM, BN, static_cast<uint32_t>(ks)), (kb | ks) != 0 ? 1u : 0u, tsf, tsf + 4);
            }
          } else {
#pragma unroll
            for (int ks = 0; ks < kBK / kUmmaK; ++ks) {
              const uint64_t ad =
                  kAmn ? sdesc_sw128(sa + ks * 2048, 8192, 1024) : sdesc_sw128(sa + ks * 32, 16, 1024);
              const uint64_t bd =
                  kBmn ? sdesc_sw128(sb + ks * 2048, 8192, 1024) : sdesc_sw128(sb + ks * 32, 16, 1024);
              if constexpr (PAIR) umma_bf16_pair(d_tmem, ad, bd, kIdesc, (kb | ks) != 0 ? 1u : 0u);
              else umma_bf16(d_tmem, ad, bd, kIdesc, (kb | ks) != 0 ? 1u : 0u);
            }
          }
          if constexpr (PAIR) umma_commit_pair(empty_bar(stage));
          else umma_commit(empty_bar(stage));
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (PAIR) umma_commit_pair(tfull_bar(acc));
        else umma_commit(tfull_bar(acc));
        if (++acc == C::kAccBufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // every MMA issued by this thread has completed before TMEM is released (in both CTAs)
      if constexpr (PAIR) umma_commit_pair(drain_bar);
      else umma_commit(drain_bar);
      mbar_wait_final(drain_bar, 0, args.status);
    } else if (PAIR && lane == 0) {
      mbar_wait_final(drain_bar, 0, args.status);  // the first CTA's MMAs into this CTA's TMEM
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps 2..5 ----------------
    const int q = warp & 3;         // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;  // column half (wide configuration only)
    Stager<C::kStageBufs, C::kStageBufBytes> stg{
        staging + static_cast<uint32_t>(warp - 2) * (C::kStageBufs * C::kStageBufBytes), 0, lane};
    int acc = 0;
    uint32_t acc_phase = 0, epi_phase = 0;
    // non-wide tiles: the four warps' staging (2 x 4 x 4 KB) serves as the group stager's two tiles
    GroupStager gs{staging, epi_bar, 0u, 0, q * 32 + lane, q == 2 && lane == 0};
    int qi = 0;
    uint32_t qph = 0;
    for (int u = unit0;; u += unit_step) {
      if (clc) {
        u = unit_pop(qi, qph, true);
        if (u < 0) break;
      } else if (u >= num_units) {
        break;
      }
      const Unit w = gemm_decode<VAR, MX, PAIR, BN>(args, u, rank);
      const uint32_t tempty = PAIR ? mapa_shared(tempty_bar(acc), 0) : tempty_bar(acc);
      Dg1Chunk pre;
      if constexpr (VAR == V_DGRAD1 && !MX) {  // before the wait
        if (!PAIR || w.row0 >= 0) dgrad1_fetch(args, w, q, lane, w.nt * BN, pre);
      }
      int ok = 0;
      if (lane == 0) ok = mbar_wait(tfull_bar(acc), acc_phase, abort_flag, args.status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      if (!PAIR || w.row0 >= 0) {
        const uint32_t taddr =
            tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
        gemm_epilogue<VAR, BN, MX, PAIR, SPLIT>(args, w, q, h, lane, taddr, stg,
                                         scratch0 + static_cast<uint32_t>(warp - 2) * C::kScratchWarp, &tmO0, &tmO1, &tmO2,
                                         tempty, pre, gs, epi_bar, epi_phase, abort_flag);
      } else {
        release_acc<PAIR>(tempty);  // a pair's CTA without rows: nothing to store
      }
      if (++acc == C::kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    stg.drain();
  }
  if constexpr (PAIR) {
    if (*abort_flag) {  // failure path: copies or arrivals of the peer may still be in flight
      const uint64_t t0 = global_timer_ns();
      while (global_timer_ns() - t0 < kWaitLimitNs / 100) {
      }
    }
    __syncwarp();
  }
  tc_fence_before();
  if constexpr (PAIR) cluster_sync();  // neither CTA leaves while the other may still address it
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                    uint32_t box_outer);
bool make_tmap_bf16_sw64(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                         uint32_t box_outer);
bool make_tmap_f32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                   uint32_t box_outer);
bool make_tmap_f32_sw64(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                        uint32_t box_outer);
// bytes (E4M3 codes); swizzle_bytes 128, 64, 32, or 0 for none
bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                  uint32_t box_outer, int swizzle_bytes);

// CTAs to launch: one per unit under cluster launch control (single-CTA tiles; the running CTAs
// take over the units of those that have not started), else the persistent grid of num_ctas
// (CTA pairs: two CTAs per unit), never more CTAs than units.  Sets args.clc to match.
inline int gemm_grid(const Sizes& z, int num_ctas, int64_t units, bool pair, GemmArgs& a) {
  a.clc = (!pair && !z.mx && z.clc) ? 1 : 0;
  if (a.clc) return static_cast<int>(units < 0x7fffffff ? units : 0x7fffffff);
  const int64_t cap = pair ? 2 * units : units;
  return static_cast<int>(cap < num_ctas ? cap : num_ctas);
}

// Row-tiled BF16 GEMMs run on CTA pairs when most pairs of 128-row blocks are full: minibatch
// tiles of at least two blocks (pairs never cross a tile) and at least `rows` routed rows per
// expert on average.  (Measured on GB300: gate/up, down and dgrad2 gain 2 to 8 % from two blocks
// per expert on; dgrad1, whose epilogue dominates, only from four; with one block per expert every
// pair is half empty and single CTAs are faster.)
inline bool use_pairs(const Sizes& z, int rows) {
  return z.mb >= 2 * kRowTile && z.R >= static_cast<int64_t>(rows) * z.E;
}

template <int VAR, int BN, bool MX = false, bool PAIR = false, bool SPLIT = false>
int launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2, const CUtensorMap& o0,
                const CUtensorMap& o1, const CUtensorMap& o2, const GemmArgs& args, int grid, cudaStream_t stream) {
  using C = GemmCfg<VAR, BN, MX, PAIR, SPLIT>;
  static DeviceOnce once;  // the shared-memory limit is set on each device that launches the kernel
  const int se = once.run([](int* d) { return static_cast<int>(cudaGetDevice(d)); },
                          [] {
                            return static_cast<int>(cudaFuncSetAttribute(gemm_kernel<VAR, BN, MX, PAIR, SPLIT>,
                                                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                                         static_cast<int>(C::kSmemBytes)));
                          },
                          static_cast<int>(cudaErrorInvalidDevice));
  if (se) return se;
  if (grid <= 0) return 0;
  if (PAIR) grid = grid < 2 ? 2 : grid & ~1;  // whole pairs
  constexpr int kKind = VAR == V_FWD_GATEUP  ? K_GEMM_FWD_GATEUP
                        : VAR == V_FWD_DOWN  ? K_GEMM_FWD_DOWN
                        : VAR == V_DGRAD1    ? K_GEMM_DGRAD1
                        : VAR == V_DGRAD2    ? K_GEMM_DGRAD2
                        : VAR == V_WGRAD_GU  ? K_GEMM_WGRAD_GU
                                             : K_GEMM_WGRAD_D;
  trace_begin(stream, kKind);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // the kernel calls pdl_wait()
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = PAIR ? 2 : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = PAIR ? 2 : 1;
  const cudaError_t le = cudaLaunchKernelEx(&cfg, gemm_kernel<VAR, BN, MX, PAIR, SPLIT>, a, b, b2, o0, o1, o2, args);
  trace_end(stream);
  return le != cudaSuccess ? static_cast<int>(le) : static_cast<int>(cudaGetLastError());
}

}  // namespace mok
