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
// Roles: warp 0 lane 0 issues TMA tile loads into a ring of shared-memory stages; warp 1 owns the
// tensor memory and its lane 0 issues tcgen05.mma (M = 128, N = BN, K = 16) into one of two TMEM
// accumulators; four epilogue warps (one per TMEM lane quarter) drain the other accumulator
// (tcgen05.ld), apply the epilogue math and write through swizzled shared tiles with TMA tile
// stores.  Every output element is produced by
// exactly one CTA with a fixed K order, so results are bitwise independent of the grid size and of
// the tile order.
#pragma once
#include <cstdint>
#include <cuda.h>

#include "mok_internal.cuh"
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
  int32_t E, I, H;
  int32_t n_tiles;         // N / BN
  int32_t m_tiles;         // weight-gradient variants: M / 128
  int32_t k_blocks;        // row-tiled variants: K / 64
  int32_t kb_split;        // DGRAD2: K blocks read from Wg before switching to Wu (I / 64)
  // epilogue operands
  void* out0;
  void* out1;
  void* out2;
  const void* in0;
  const void* in1;
  const float* row_weight;
  uint32_t* status;
};

template <int VAR, int BN>
struct GemmCfg {
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr int kStageBufs = 2;  // staging tiles per epilogue warp
  static constexpr int kEpiWarps = 4;   // one warp per TMEM lane quarter
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr uint32_t kABytes = kBM * kBK * 2;
  static constexpr uint32_t kBBytes = BN * kBK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = 2 * BN;
  static constexpr uint32_t kStagingBytes = kEpiWarps * kStageBufs * 4096;  // per warp: tiles of 4 KB
  static constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(kStages) * kStageBytes + kStagingBytes + 256;
};

struct Unit {
  int e, row0, nt, mt, kblocks;
};

template <int VAR>
__device__ __forceinline__ int gemm_num_units(const GemmArgs& a) {
  if constexpr (VAR == V_WGRAD_GU || VAR == V_WGRAD_D) return a.E * a.m_tiles * a.n_tiles;
  else return a.meta[2] * a.n_tiles;
}

// Row-tiled variants: all units of one minibatch tile are consecutive, N tile outer and 128-row
// block inner, so a weight tile is reused by the tile's blocks while it sits in L2.
template <int VAR>
__device__ __forceinline__ Unit gemm_decode(const GemmArgs& a, int u) {
  Unit w;
  if constexpr (VAR == V_WGRAD_GU || VAR == V_WGRAD_D) {
    const int per_e = a.m_tiles * a.n_tiles;
    w.e = u / per_e;
    const int r = u - w.e * per_e;
    w.mt = r / a.n_tiles;
    w.nt = r - w.mt * a.n_tiles;
    const int p0 = __ldg(a.poff + w.e), p1 = __ldg(a.poff + w.e + 1);
    w.row0 = p0;
    w.kblocks = (p1 - p0) / kBK;
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

// Issue the TMA loads of one K block into stage (sa, sb), all completing on barrier `bar`.  With MX
// the dgrad variants read B from K-major transposed weight copies ([E*I, H] for dgrad1, [E*H, I]
// for dgrad2) instead of the MN-major forward layout.
template <int VAR, int BN, bool MX>
__device__ __forceinline__ void gemm_load(const GemmArgs& a, const Unit& w, int kb, uint32_t sa, uint32_t sb,
                                          uint32_t bar, const CUtensorMap* tA, const CUtensorMap* tB,
                                          const CUtensorMap* tB2) {
  const int k0 = kb * kBK;
  if constexpr (MX && VAR == V_DGRAD1) {
    tma_load_2d(sa, tA, bar, k0, w.row0);
    tma_load_2d(sb, tB, bar, k0, w.e * a.I + w.nt * BN);
    return;
  }
  if constexpr (MX && VAR == V_DGRAD2) {
    tma_load_2d(sa, tA, bar, k0, w.row0);
    const bool first = kb < a.kb_split;
    tma_load_2d(sb, first ? tB : tB2, bar, first ? k0 : k0 - a.kb_split * kBK, w.e * a.H + w.nt * BN);
    return;
  }
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

// SwiGLU pieces in fp32 with the fast approximate division (about 2 ulp; the results are rounded to
// bf16 next, 2^-9).
__device__ __forceinline__ float sigmoid_f(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ uint4 ldg_v4(const uint16_t* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

// Per-warp output stager: NBUF shared-memory tiles (4 KB apart) of 32 rows x ROW bytes in the TMA
// swizzle layout of that row size -- 128-byte rows: 16-byte chunk j of row r sits at chunk
// j ^ (r & 7); 64-byte rows: at j ^ ((r >> 1) & 3).  Both keep the 32 lanes' row writes free of
// bank conflicts.  Each filled tile leaves as one asynchronous TMA tile store; a tile is refilled
// only after its previous store has finished reading it, so up to NBUF stores are in flight.
template <int ROW, int NBUF>
struct Stager {
  static constexpr int kChunks = ROW / 16;
  uint32_t buf0;
  int cur;
  int lane;
  __device__ __forceinline__ uint32_t acquire() {
    if (lane == 0) bulk_wait_read<NBUF - 1>();
    __syncwarp();
    const uint32_t b = buf0 + (static_cast<uint32_t>(cur) << 12);
    cur = cur + 1 == NBUF ? 0 : cur + 1;
    return b;
  }
  // Lane r writes its row (kChunks chunks of 16 bytes) and the warp stores the tile at (c0, c1).
  __device__ __forceinline__ void put_and_store(const uint4* ch, const CUtensorMap* tm, int c0, int c1) {
    const uint32_t b = acquire();
    const uint32_t row = b + static_cast<uint32_t>(lane) * ROW;
    const int sw = ROW == 128 ? (lane & 7) : ((lane >> 1) & 3);
#pragma unroll
    for (int j = 0; j < kChunks; ++j) st_shared_v4(row + (static_cast<uint32_t>(j ^ sw) << 4), ch[j]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tm, b, c0, c1);
      bulk_commit();
    }
  }
  __device__ __forceinline__ void drain() {
    if (lane == 0) bulk_wait_all();
    __syncwarp();
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

// Hand the accumulator back to the MMA warp once this thread has read its last TMEM column.
__device__ __forceinline__ void release_acc(uint32_t tempty) {
  tc_fence_before();
  mbar_arrive(tempty);
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

template <int VAR>
constexpr int epi_row_bytes() { return VAR == V_DGRAD1 ? 64 : 128; }

// Epilogue of one unit for the warp's 32 accumulator rows (slab `q`); lane = row in the slab.
// tO0 / tO1 are the output tensor maps of the variant; `tempty` is released as soon as the last
// accumulator column has been read.  `pre` holds DGRAD1's first prefetched context chunk.
template <int VAR, int BN, bool MX, class Stg>
__device__ __forceinline__ void gemm_epilogue(const GemmArgs& a, const Unit& w, int q, int lane, uint32_t taddr,
                                              Stg& stg, const CUtensorMap* tO0, const CUtensorMap* tO1,
                                              uint32_t tempty, Dg1Chunk& pre) {
  if constexpr (VAR == V_FWD_GATEUP) {
    // columns [0, BN/2) of the accumulator are gate, [BN/2, BN) up, for I columns i0 ...
    const int i0 = w.nt * (BN / 2);
    const int rowc = w.row0 + q * 32;
#pragma unroll 1
    for (int c = 0; c < BN / 2; c += 64) {
      float g[64], u[64];
      tmem_ld64(taddr + c, g);
      tmem_ld64(taddr + BN / 2 + c, u);
      if (c + 64 >= BN / 2) release_acc(tempty);
      uint4 ch[8];
      if constexpr (MX) {  // g, u kept in fp32 for the backward's re-quantisation of dg, du
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            ch[j] = make_uint4(__float_as_uint(g[32 * h + 4 * j]), __float_as_uint(g[32 * h + 4 * j + 1]),
                               __float_as_uint(g[32 * h + 4 * j + 2]), __float_as_uint(g[32 * h + 4 * j + 3]));
          stg.put_and_store(ch, tO0, i0 + c + 32 * h, rowc);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            ch[j] = make_uint4(__float_as_uint(u[32 * h + 4 * j]), __float_as_uint(u[32 * h + 4 * j + 1]),
                               __float_as_uint(u[32 * h + 4 * j + 2]), __float_as_uint(u[32 * h + 4 * j + 3]));
          stg.put_and_store(ch, tO0, a.I + i0 + c + 32 * h, rowc);
        }
      } else {
        pack_bf16<64>(g, ch);
        stg.put_and_store(ch, tO0, i0 + c, rowc);
        pack_bf16<64>(u, ch);
        stg.put_and_store(ch, tO0, a.I + i0 + c, rowc);
      }
#pragma unroll
      for (int i = 0; i < 64; ++i) g[i] = silu_f(g[i]) * u[i];
      if constexpr (MX) {  // a leaves MX-quantised along I (two blocks of 32)
        mx_fakequant32(g);
        mx_fakequant32(g + 32);
      }
      pack_bf16<64>(g, ch);
      stg.put_and_store(ch, tO1, i0 + c, rowc);
    }
  } else if constexpr (VAR == V_FWD_DOWN || VAR == V_DGRAD2) {
    const int rowc = w.row0 + q * 32;
#pragma unroll 1
    for (int c = 0; c < BN; c += 64) {
      float v[64];
      tmem_ld64(taddr + c, v);
      if (c + 64 >= BN) release_acc(tempty);
      uint4 ch[8];
      pack_bf16<64>(v, ch);
      stg.put_and_store(ch, tO0, w.nt * BN + c, rowc);
    }
  } else if constexpr (VAR == V_DGRAD1 && MX) {
    // MXFP8: as below, with g, u read in fp32 and dg, du quantise-dequantised per block of 32.
    const int64_t row = w.row0 + q * 32 + lane;
    const int64_t I = a.I;
    const int i0 = w.nt * BN;
    const float* gu = static_cast<const float*>(a.in0) + row * 2 * I;
    const uint16_t* av = static_cast<const uint16_t*>(a.in1) + row * I;
    const float s = __ldg(a.row_weight + row);
    const int rowc = w.row0 + q * 32;
    float part = 0.0f;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      float4 g4[8], u4[8];
      const float4* gp = reinterpret_cast<const float4*>(gu + i0 + c);
      const float4* up = reinterpret_cast<const float4*>(gu + I + i0 + c);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        g4[j] = __ldg(gp + j);
        u4[j] = __ldg(up + j);
      }
      uint32_t rv[32];
      tmem_ld_32x32b_x32(taddr + c, rv);
      tmem_ld_wait();
      if (c + 32 >= BN) release_acc(tempty);
      const float* g = reinterpret_cast<const float*>(g4);
      const float* u = reinterpret_cast<const float*>(u4);
      float dg[32], du[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float da = s * __uint_as_float(rv[i]);
        const float sg = sigmoid_f(g[i]);
        dg[i] = da * u[i] * sg * (1.0f + g[i] * (1.0f - sg));
        du[i] = da * g[i] * sg;
      }
      mx_fakequant32(dg);
      mx_fakequant32(du);
      uint4 ch[4];
      pack_bf16<32>(dg, ch);
      stg.put_and_store(ch, tO0, i0 + c, rowc);
      pack_bf16<32>(du, ch);
      stg.put_and_store(ch, tO0, a.I + i0 + c, rowc);
      float sa[32];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float a8[8];
        unpack8(ldg_v4(av + i0 + c + 8 * j), a8);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          part = fmaf(__uint_as_float(rv[8 * j + k]), a8[k], part);
          sa[8 * j + k] = s * a8[k];
        }
      }
      pack_bf16<32>(sa, ch);
      stg.put_and_store(ch, tO1, i0 + c, rowc);
    }
    static_cast<float*>(a.out2)[row * a.n_tiles + w.nt] = part;
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
      if (c + 32 >= BN) release_acc(tempty);
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
      stg.put_and_store(cdg, tO0, i0 + c, rowc);
      stg.put_and_store(cdu, tO0, a.I + i0 + c, rowc);
      stg.put_and_store(csa, tO1, i0 + c, rowc);
    }
    static_cast<float*>(a.out2)[row * a.n_tiles + w.nt] = part;
  } else {  // weight gradients, fp32 out, 32-column tiles
    const bool empty = w.kblocks == 0;
    const int m0 = w.mt * kBM + q * 32;  // first of this warp's 32 output rows
    const CUtensorMap* tm;
    int r0;
    if constexpr (VAR == V_WGRAD_GU) {
      tm = m0 < a.I ? tO0 : tO1;
      r0 = w.e * a.I + (m0 < a.I ? m0 : m0 - a.I);
    } else {
      tm = tO0;
      r0 = w.e * a.H + m0;
    }
    if (empty) release_acc(tempty);
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t rv[32];
      if (!empty) {
        tmem_ld_32x32b_x32(taddr + c, rv);
        tmem_ld_wait();
        if (c + 32 >= BN) release_acc(tempty);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) rv[i] = 0u;
      }
      uint4 ch[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) ch[j] = make_uint4(rv[4 * j], rv[4 * j + 1], rv[4 * j + 2], rv[4 * j + 3]);
      stg.put_and_store(ch, tm, w.nt * BN + c, r0);
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

template <int VAR, int BN, bool MX>
__global__ void __launch_bounds__(GemmCfg<VAR, BN>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmO0,
                const __grid_constant__ CUtensorMap tmO1, const GemmArgs args) {
  using C = GemmCfg<VAR, BN>;
  constexpr bool kAmn = (VAR == V_WGRAD_GU || VAR == V_WGRAD_D);
  constexpr bool kBmn = (VAR >= V_DGRAD1) && !(MX && (VAR == V_DGRAD1 || VAR == V_DGRAD2));
  constexpr uint32_t kIdesc = idesc_bf16(kBM, BN, kAmn, kBmn);
  constexpr int S = C::kStages;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms need 1024-byte alignment
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t staging = base + S * C::kStageBytes;  // 1024-byte aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + S * C::kStageBytes + C::kStagingBytes);
  // bars[0..S) full, [S..2S) empty, [2S, 2S+2) accumulator full, [2S+2, 2S+4) accumulator empty,
  // [2S+4] drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 32 * C::kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmB2);
    tma_prefetch_desc(&tmO0);
    tma_prefetch_desc(&tmO1);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_units = gemm_num_units<VAR>(args);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      int last_parity[S];
      for (int s = 0; s < S; ++s) last_parity[s] = -1;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
        const Unit w = gemm_decode<VAR>(args, u);
        for (int kb = 0; kb < w.kblocks; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), C::kStageBytes);
          const uint32_t sa = base + stage * C::kStageBytes;
          gemm_load<VAR, BN, MX>(args, w, kb, sa, sa + C::kABytes, full_bar(stage), &tmA, &tmB, &tmB2);
          last_parity[stage] = static_cast<int>(phase);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {  // wind down: let the copies already issued land before the CTA exits
        for (int s = 0; s < S; ++s)
          if (last_parity[s] >= 0) mbar_wait_final(full_bar(s), static_cast<uint32_t>(last_parity[s]), args.status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
        const Unit w = gemm_decode<VAR>(args, u);
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, args.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < w.kblocks; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + stage * C::kStageBytes, sb = sa + C::kABytes;
#pragma unroll
          for (int ks = 0; ks < kBK / kUmmaK; ++ks) {
            const uint64_t ad = kAmn ? sdesc_sw128(sa + ks * 2048, 8192, 1024) : sdesc_sw128(sa + ks * 32, 16, 1024);
            const uint64_t bd = kBmn ? sdesc_sw128(sb + ks * 2048, 8192, 1024) : sdesc_sw128(sb + ks * 32, 16, 1024);
            umma_bf16(d_tmem, ad, bd, kIdesc, (kb | ks) != 0 ? 1u : 0u);
          }
          umma_commit(empty_bar(stage));
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // every MMA issued by this thread has completed before TMEM is released
      umma_commit(drain_bar);
      mbar_wait_final(drain_bar, 0, args.status);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps 2..5 ----------------
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    Stager<epi_row_bytes<VAR>(), C::kStageBufs> stg{
        staging + static_cast<uint32_t>(warp - 2) * (C::kStageBufs * 4096u), 0, lane};
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
      const Unit w = gemm_decode<VAR>(args, u);
      Dg1Chunk pre;
      if constexpr (VAR == V_DGRAD1 && !MX) dgrad1_fetch(args, w, q, lane, w.nt * BN, pre);  // before the wait
      int ok = 0;
      if (lane == 0) ok = mbar_wait(tfull_bar(acc), acc_phase, abort_flag, args.status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      gemm_epilogue<VAR, BN, MX>(args, w, q, lane, taddr, stg, &tmO0, &tmO1, tempty_bar(acc), pre);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    stg.drain();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
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

template <int VAR, int BN, bool MX = false>
int launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2, const CUtensorMap& o0,
                const CUtensorMap& o1, const GemmArgs& args, int grid, cudaStream_t stream) {
  using C = GemmCfg<VAR, BN>;
  static bool configured = false;  // per process; the attribute is per function, set once
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<VAR, BN, MX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kSmemBytes));
    if (e != cudaSuccess) return static_cast<int>(e);
    configured = true;
  }
  if (grid <= 0) return 0;
  constexpr int kKind = VAR == V_FWD_GATEUP  ? K_GEMM_FWD_GATEUP
                        : VAR == V_FWD_DOWN  ? K_GEMM_FWD_DOWN
                        : VAR == V_DGRAD1    ? K_GEMM_DGRAD1
                        : VAR == V_DGRAD2    ? K_GEMM_DGRAD2
                        : VAR == V_WGRAD_GU  ? K_GEMM_WGRAD_GU
                                             : K_GEMM_WGRAD_D;
  trace_begin(stream, kKind);
  gemm_kernel<VAR, BN, MX><<<grid, C::kThreads, C::kSmemBytes, stream>>>(a, b, b2, o0, o1, args);
  trace_end(stream);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace mok
