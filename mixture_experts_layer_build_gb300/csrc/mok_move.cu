// mok_move.cu -- the HBM-bound steps: dispatch gather, fixed-order weighted combine / dX reduce,
// router-gradient reduce, and MXFP8 quantisation.
//
// Dispatch and combine are the one-GPU form of the pages' pull dispatch and push combine
// ("Mixture-of-Kittens(MoK)란? ..." (alltoptrend), section 4 (1)): token rows are gathered into the
// expert-grouped layout, and each token's K expert outputs are summed back in ascending k in fp32
// and rounded once to bf16, so the result does not depend on any scheduling order.
#include "mok_internal.cuh"
#include "mok_once.h"
#include "mok_ptx.cuh"

namespace mok {
namespace {

constexpr int kMoveThreads = 256;

// Token t's row in the token buffers: one plain buffer, or (expert parallelism) the buffer of the
// rank holding t, at its row t % rows_per -- a peer's memory when the ranks are separate GPUs.
// (Token and slot indices fit in 32 bits -- the schedule's tables are int32 -- so the rank is a
// 32-bit division, not the much longer 64-bit one.)
__device__ __forceinline__ const uint16_t* token_row(const RowSrc& src, int64_t t, int64_t H) {
  if (src.n == 0) return src.p[0] + t * H;
  const uint32_t per = static_cast<uint32_t>(src.rows_per);
  const uint32_t r = static_cast<uint32_t>(t) / per;
  return pick_rank(src.p, r) + (static_cast<uint32_t>(t) - r * per) * H;
}

// The dispatch gather in token order: token t's row is read once and written to the rows of its
// K slots (row inv[t*K+k]; a slot with inv < 0 -- an invalid id, or an expert another rank owns --
// is skipped), then every padding row (row_token < 0, row < Rpad = meta[0]) is zeroed.  A warp's
// work item is one chunk of 32 * U 16-byte vectors of one token row (chunks fastest, so warps
// running together read whole rows), lanes striding along it: U loads per lane, then the K stores
// of each.  Walking the rows in expert order instead re-reads each token row K times from wherever
// L2 has let it go; in token order HBM sees one read of the token rows and one write of the
// gathered ones, and both streams are marked evict-first.  Padding rows are dealt out to the
// warps by a row stride (padding sits in runs at the end of each expert's rows): each lane looks
// up one of the warp's next 32 rows, and the warp zeroes the ones that are padding.  With expert
// parallelism this is the pull dispatch of the pages: the rank owning the experts reads, from the
// ranks holding them, the rows of the tokens with a slot on one of its experts.
template <int U>
__global__ void __launch_bounds__(kMoveThreads) gather_tokens_kernel(const RowSrc src,
                                                                    const int32_t* __restrict__ inv,
                                                                    const int32_t* __restrict__ row_token,
                                                                    const int32_t* __restrict__ meta, int64_t T,
                                                                    int K, int64_t vecs, uint4* __restrict__ dst) {
  pdl_wait();
  constexpr int64_t kChunk = 32 * U;
  const int lane = threadIdx.x & 31;
  const int64_t warp = static_cast<int64_t>(blockIdx.x) * (kMoveThreads / 32) + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kMoveThreads / 32);
  const int64_t chunks = (vecs + kChunk - 1) / kChunk;
  // every loop bound and branch condition below is the same on all 32 lanes, so each
  // __ballot_sync / __shfl_sync is reached by the whole warp
  for (int64_t item = warp; item < T * chunks; item += nwarps) {
    const int64_t t = item / chunks;
    const int64_t c0 = (item - t * chunks) * kChunk;
    const uint4* s = reinterpret_cast<const uint4*>(token_row(src, t, vecs * 8));
    for (int k0 = 0; k0 < K; k0 += 32) {
      const int row = k0 + lane < K ? __ldg(inv + t * K + k0 + lane) : -1;
      const unsigned live = __ballot_sync(0xffffffffu, row >= 0);
      if (!live) continue;
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t c = c0 + 32 * u + lane;
        v[u] = c < vecs ? __ldcs(s + c) : make_uint4(0, 0, 0, 0);
      }
      for (unsigned m = live; m; m &= m - 1) {
        const int64_t r = __shfl_sync(0xffffffffu, row, __ffs(m) - 1);
        uint4* d = dst + r * vecs;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t c = c0 + 32 * u + lane;
          if (c < vecs) __stcs(d + c, v[u]);
        }
      }
    }
  }
  const int64_t rpad = meta[0];
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int64_t r0 = warp; r0 < rpad; r0 += 32 * nwarps) {  // rows r0 + j * nwarps, j = 0..31
    const int64_t r = r0 + lane * nwarps;
    const bool pad = r < rpad && __ldg(row_token + r) < 0;
    for (unsigned m = __ballot_sync(0xffffffffu, pad); m; m &= m - 1) {
      uint4* d = dst + (r0 + static_cast<int64_t>(__ffs(m) - 1) * nwarps) * vecs;
      for (int64_t c = lane; c < vecs; c += 32) __stcs(d + c, z);
    }
  }
}

// out[t] = bf16( sum_{k = 0..K-1 ascending} w[t,k] * y[inv[t*K+k]] ), fp32 accumulation; w == nullptr
// means weight 1 (the dX reduction).  Slots with inv < 0 (invalid ids) contribute nothing.  With
// inv == nullptr the rows are per slot (row t*K+k: the token owner's receive buffer under expert
// parallelism) and a slot counts when its id lies in [0, e_total).  Each
// lane keeps eight 16-byte row loads in flight: U column vectors x (8 / U) of the K rows, issued
// together before the fixed-order FMA chains (U = 8 for top-1 ... U = 1 for K >= 8).  Rows are
// read once and written once: both streams are marked evict-first.
template <int U, bool ONE>
__global__ void __launch_bounds__(kMoveThreads, 4) combine_kernel(const uint4* __restrict__ y,
                                                              const int32_t* __restrict__ inv,
                                                              const int32_t* __restrict__ ids, int e_total,
                                                              const float* __restrict__ w, int64_t T, int K,
                                                              int64_t vecs, uint4* __restrict__ out) {
  pdl_wait();
  constexpr int kBatch = 8 / U;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kMoveThreads / 32);
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (kMoveThreads / 32) + (threadIdx.x >> 5); t < T;
       t += nwarps) {
    for (int64_t c0 = lane; c0 < vecs; c0 += 32 * U) {
      if constexpr (ONE) {
        // all K slots in one batch (K <= 8 / U): each column vector is reduced and stored as soon
        // as its loads land, so no U x 8 accumulator array stays live across a runtime k loop (the
        // top-1 instance: 95 -> 62 registers, four blocks per SM instead of two, enough warps to
        // cover the HBM latency).  Same fused multiply-adds in the same ascending k order as the
        // general path.
        uint4 v[U][kBatch];
        float wk[kBatch];
        int row[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          if (b >= K) {
            row[b] = -1;
          } else if (inv) {
            row[b] = __ldg(inv + t * K + b);
          } else {
            const int g = __ldg(ids + t * K + b);
            row[b] = (g >= 0 && g < e_total) ? static_cast<int>(t * K + b) : -1;
          }
          wk[b] = (row[b] >= 0 && w) ? __ldg(w + t * K + b) : 1.0f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int64_t c = c0 + 32 * u;
            v[u][b] = (row[b] >= 0 && c < vecs) ? __ldcs(y + static_cast<int64_t>(row[b]) * vecs + c)
                                                : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          float acc[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            if (row[b] < 0) continue;
            const uint32_t p[4] = {v[u][b].x, v[u][b].y, v[u][b].z, v[u][b].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              acc[2 * i] = fmaf(wk[b], bf16_lo(p[i]), acc[2 * i]);
              acc[2 * i + 1] = fmaf(wk[b], bf16_hi(p[i]), acc[2 * i + 1]);
            }
          }
          const int64_t c = c0 + 32 * u;
          if (c < vecs)
            __stcs(out + t * vecs + c, make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                                  pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
        }
        continue;
      }
      float acc[U][8];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;
      for (int k0 = 0; k0 < K; k0 += kBatch) {
        uint4 v[U][kBatch];
        float wk[kBatch];
        int row[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int k = k0 + b;
          if (k >= K) {
            row[b] = -1;
          } else if (inv) {
            row[b] = __ldg(inv + t * K + k);
          } else {
            const int g = __ldg(ids + t * K + k);
            row[b] = (g >= 0 && g < e_total) ? static_cast<int>(t * K + k) : -1;
          }
          wk[b] = (row[b] >= 0 && w) ? __ldg(w + t * K + k) : 1.0f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int64_t c = c0 + 32 * u;
            v[u][b] = (row[b] >= 0 && c < vecs) ? __ldcs(y + static_cast<int64_t>(row[b]) * vecs + c)
                                                : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          if (row[b] < 0) continue;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const uint32_t p[4] = {v[u][b].x, v[u][b].y, v[u][b].z, v[u][b].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              acc[u][2 * i] = fmaf(wk[b], bf16_lo(p[i]), acc[u][2 * i]);
              acc[u][2 * i + 1] = fmaf(wk[b], bf16_hi(p[i]), acc[u][2 * i + 1]);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t c = c0 + 32 * u;
        if (c < vecs)
          __stcs(out + t * vecs + c,
                 make_uint4(pack_bf16x2(acc[u][0], acc[u][1]), pack_bf16x2(acc[u][2], acc[u][3]),
                            pack_bf16x2(acc[u][4], acc[u][5]), pack_bf16x2(acc[u][6], acc[u][7])));
      }
    }
  }
}

// ds[j] = sum over N tiles (ascending) of part[inv[j], :]; 0 for skipped slots.
__global__ void __launch_bounds__(kMoveThreads) ds_reduce_kernel(const float* __restrict__ part,
                                                                const int32_t* __restrict__ inv, int64_t R,
                                                                int n_tiles, float* __restrict__ ds) {
  pdl_wait();
  const int64_t j = static_cast<int64_t>(blockIdx.x) * kMoveThreads + threadIdx.x;
  if (j >= R) return;
  const int row = inv[j];
  float acc = 0.0f;
  if (row >= 0) {
    const float* p = part + static_cast<int64_t>(row) * n_tiles;
    for (int n = 0; n < n_tiles; ++n) acc += p[n];
  }
  ds[j] = acc;
}

// Expert parallelism: the dS of this rank's slots, sum over N tiles (ascending) of part[inv[j], :],
// pushed to the token owner's [slots_per] buffer; this rank's own tokens' invalid slots get 0 (no
// expert owns them).  Every slot of the group is written by exactly one rank.
__global__ void __launch_bounds__(kMoveThreads) ds_push_kernel(const float* __restrict__ part,
                                                              const int32_t* __restrict__ inv, int64_t R,
                                                              int n_tiles, const RowDst dst, int rank) {
  pdl_wait();
  const int64_t j = static_cast<int64_t>(blockIdx.x) * kMoveThreads + threadIdx.x;
  if (j >= R) return;
  const int row = inv[j];
  const int64_t r = static_cast<uint32_t>(j) / static_cast<uint32_t>(dst.slots_per);
  if (row >= 0) {
    const float* p = part + static_cast<int64_t>(row) * n_tiles;
    float acc = 0.0f;
    for (int n = 0; n < n_tiles; ++n) acc += p[n];
    static_cast<float*>(pick_rank(dst.p, r))[j - r * dst.slots_per] = acc;
  } else if (row == kSlotInvalid && r == rank) {
    static_cast<float*>(pick_rank(dst.p, r))[j - r * dst.slots_per] = 0.0f;
  }
}

// Expert parallelism, the push combine of the pages: row r of the expert-grouped rows (r < Rpad),
// holding slot j = perm[r], goes to the rank holding slot j, at its row j % slots_per.  One warp per
// row, 16-byte vectors; both streams single-use (evict-first).
__global__ void __launch_bounds__(kMoveThreads) push_rows_kernel(const uint4* __restrict__ src,
                                                                const int32_t* __restrict__ perm,
                                                                const int32_t* __restrict__ meta, int64_t vecs,
                                                                const RowDst dst) {
  pdl_wait();
  const int64_t rpad = meta[0];
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kMoveThreads / 32);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (kMoveThreads / 32) + (threadIdx.x >> 5); row < rpad;
       row += nwarps) {
    const int64_t j = perm[row];
    if (j < 0) continue;  // padding row
    const int64_t r = static_cast<uint32_t>(j) / static_cast<uint32_t>(dst.slots_per);
    const uint4* s = src + row * vecs;
    uint4* d = static_cast<uint4*>(pick_rank(dst.p, r)) + (j - r * dst.slots_per) * vecs;
    int64_t c = lane;
    for (; c + 96 < vecs; c += 128) {
      const uint4 v0 = __ldcs(s + c), v1 = __ldcs(s + c + 32), v2 = __ldcs(s + c + 64), v3 = __ldcs(s + c + 96);
      __stcs(d + c, v0);
      __stcs(d + c + 32, v1);
      __stcs(d + c + 64, v2);
      __stcs(d + c + 96, v3);
    }
    for (; c < vecs; c += 32) __stcs(d + c, __ldcs(s + c));
  }
}

// ---------------------------------------------------------------------------------------------
// MXFP8: E4M3 elements with one E8M0 scale per 32 consecutive values ("Mixture-of-Kittens (MoK)"
// project card, "Key concepts": ops.mxfp8_quantize).  Per block: amax = max |v|; shared =
// floor(log2 amax) - 8 (8 = the exponent of E4M3's largest normal), clamped below at -127; each
// element is v * 2^-shared rounded to nearest even on the E4M3 grid, saturating at 448; a block
// holding Inf or NaN gets scale byte 0xFF and every code 0x7F.
// ---------------------------------------------------------------------------------------------

// Packed bf16 arithmetic: two values per 32-bit word, one instruction each.
// absmax: per 16-bit half the larger magnitude, NaN if either operand is NaN; the sign bits of the
// result (the XOR of the operands') mean nothing and are masked off at the end.
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Per half, a value times a power of two.  Exact while the product is a normal bf16; a product
// below that is under half of E4M3's smallest subnormal and encodes as a zero of its sign.
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Per-half magnitude maxima of N packed words (a pairwise tree), sign bits cleared.
template <int N>
__device__ __forceinline__ uint32_t bf16x2_absmax_words(const uint32_t (&w)[N]) {
  static_assert(N >= 2 && (N & (N - 1)) == 0, "power of two");
  uint32_t m[N / 2];
#pragma unroll
  for (int i = 0; i < N / 2; ++i) m[i] = bf16x2_absmax(w[i], w[i + N / 2]);
#pragma unroll
  for (int s = N / 4; s >= 1; s >>= 1) {
#pragma unroll
    for (int i = 0; i < s; ++i) m[i] = bf16x2_absmax(m[i], m[i + s]);
  }
  return m[0] & 0x7FFF7FFFu;
}
// The shared exponent of a block from its 15-bit bf16 magnitude maximum (finite): floor(log2 amax)
// - 8, clamped below at -127 (zero and subnormal maxima give -127).  Its bf16 multiplier 2^-shared
// is the exponent field 127 - shared in [8, 254]: always a normal number.
__device__ __forceinline__ int gmx_shared(uint32_t amax) {
  const int s = static_cast<int>(amax >> 7) - 135;
  return s < -127 ? -127 : s;
}
__device__ __forceinline__ uint32_t gmx_mult(int shared) { return static_cast<uint32_t>(127 - shared) << 7; }
// E4M3 codes of the two bf16 halves of word w (low half in the low byte).
__device__ __forceinline__ uint32_t e4m3x2_of_bf16x2(uint32_t w) {
  uint16_t q;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(q) : "f"(__uint_as_float(w & 0xFFFF0000u)),
      "f"(__uint_as_float(w << 16)));
  return q;
}
// Same, for the low halves (COL 0) or the high halves (COL 1) of two words: value of w0, then w1.
template <int COL>
__device__ __forceinline__ uint32_t e4m3x2_of_halves(uint32_t w0, uint32_t w1) {
  uint16_t q;
  if constexpr (COL == 0)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(q) : "f"(__uint_as_float(w1 << 16)),
        "f"(__uint_as_float(w0 << 16)));
  else
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(q) : "f"(__uint_as_float(w1 & 0xFFFF0000u)),
        "f"(__uint_as_float(w0 & 0xFFFF0000u)));
  return q;
}
// 32 bytes to global memory in one instruction (p 32-byte aligned), with an L2 evict-first policy:
// the codes are read by later kernels from DRAM anyway, and the gathered x rows (read K times)
// should be the lines L2 keeps.  Measured against plain streaming stores (.cs): 0.205 -> 0.202 ms
// per gather on sweep_zipf1_mx.
__device__ __forceinline__ void st_ef_32B(void* p, const uint32_t (&c)[8]) {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  asm volatile("st.global.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(p), "r"(c[0]),
               "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4]), "r"(c[5]), "r"(c[6]), "r"(c[7]), "l"(pol)
               : "memory");
}

// One 32-value block along a row, held as 16 packed words (values 2i, 2i + 1 = low, high half of
// w[i]); w is scaled in place.  Returns the scale byte.  The codes and the byte are those of
// mx_quant32 on the same values: a bf16 magnitude's bits order like the value, its exponent field is
// the fp32 one, and scaling by a power of two is exact (see bf16x2_mul).
__device__ __forceinline__ uint32_t gmx_quant_row(uint32_t (&w)[16], uint32_t (&codes)[8]) {
  uint32_t m = bf16x2_absmax_words(w);
  m = bf16x2_absmax(m, m >> 16) & 0x7FFFu;
  if (m >= 0x7F80u) {  // an Inf or NaN in the block
#pragma unroll
    for (int i = 0; i < 8; ++i) codes[i] = 0x7F7F7F7Fu;
    return 0xFFu;
  }
  const int shared = gmx_shared(m);
  const uint32_t dn2 = gmx_mult(shared) * 0x10001u;
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = bf16x2_mul(w[i], dn2);
#pragma unroll
  for (int i = 0; i < 8; ++i) codes[i] = e4m3x2_of_bf16x2(w[2 * i]) | (e4m3x2_of_bf16x2(w[2 * i + 1]) << 16);
  return static_cast<uint32_t>(shared + 127);
}

// One thread per 32-element block; 64 bytes read, 32 + 1 bytes written.
__global__ void __launch_bounds__(kMoveThreads) mxfp8_quantize_kernel(const uint4* __restrict__ in,
                                                                     int64_t nblocks, uint4* __restrict__ q,
                                                                     uint8_t* __restrict__ sc) {
  pdl_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kMoveThreads;
  for (int64_t b = static_cast<int64_t>(blockIdx.x) * kMoveThreads + threadIdx.x; b < nblocks; b += stride) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(in + b * 4 + i);
      w[4 * i] = v.x, w[4 * i + 1] = v.y, w[4 * i + 2] = v.z, w[4 * i + 3] = v.w;
    }
    uint32_t codes[8];
    sc[b] = static_cast<uint8_t>(gmx_quant_row(w, codes));
    __stcs(q + b * 2, make_uint4(codes[0], codes[1], codes[2], codes[3]));
    __stcs(q + b * 2 + 1, make_uint4(codes[4], codes[5], codes[6], codes[7]));
  }
}

// MX gather, one CTA per (32-row block of the expert-grouped layout, 128 columns), 64 threads.
// The 32 gathered rows are staged in shared memory as bf16 (zero for padding rows); then
//   along H: each thread quantises two 32-column blocks of rows -- row-major E4M3 codes for the
//     forward / data-gradient GEMMs, A-operand atoms;
//   along the routed rows: each thread quantises two adjacent columns over the 32-row block
//     (reading both as one 32-bit word per row) -- 32 consecutive bytes per column of the
//     transposed copy [H, rcap] the weight-gradient GEMM reads K-major, atoms grouped gT at a time.
// Both passes keep the values as packed bf16 pairs: the block maxima and the power-of-two scaling
// take one instruction per two values, and only the final E4M3 conversion widens them to fp32.
// The scale bytes are collected in shared memory and leave as one 32-bit word per row (its four
// 32-column blocks) and one byte per column (its 32-row block).  Small blocks put twenty CTAs on
// an SM, so more of them are between their row loads and their quantisation at any time
// (measured per gather on sweep_zipf1_mx: 128 rows and 256 threads 0.220 ms, 64 rows 0.210, 32
// rows 0.205).
// The rounding is bit-exact with mxfp8_quantize_kernel (shared exponent from amax, E4M3
// round-to-nearest-even, saturating).  Row blocks never straddle two experts: segments start at
// multiples of 128.
constexpr int kGmxStride = 128 * 2 + 16;  // bytes per staged bf16 row (the pad spreads banks)

// 32-row blocks, 64 threads, twenty CTAs per SM (48 registers, no spills).
constexpr int kGmxRows = 32;
__global__ void __launch_bounds__(64, 20) gather_rows_mx_kernel(const RowSrc src,
                                                            const int32_t* __restrict__ row_token,
                                                            const int32_t* __restrict__ meta, int32_t H,
                                                            uint8_t* __restrict__ dst_q, uint8_t* __restrict__ dst_sf,
                                                            uint8_t* __restrict__ dstR_q,
                                                            uint8_t* __restrict__ dstR_sf, int64_t rcap, int gT) {
  pdl_wait();
  __shared__ __align__(16) uint8_t tile[kGmxRows * kGmxStride];
  __shared__ __align__(4) uint8_t sc_row[kGmxRows * 4];  // [row][32-column block]
  __shared__ __align__(4) uint8_t sc_col[128];           // [column]
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kGmxRows;
  if (r0 >= meta[0]) return;
  const int c0 = static_cast<int>(blockIdx.x) * 128;
  const int t = threadIdx.x;
  {
    uint4 val[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // thread t: 16-byte vector t % 16 of rows t / 16 + 4 i
      const int r = t / 16 + 4 * i;
      const int tok = __ldg(row_token + r0 + r);
      val[i] = tok >= 0 ? __ldg(reinterpret_cast<const uint4*>(token_row(src, tok, H) + c0) + t % 16)
                        : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
      *reinterpret_cast<uint4*>(tile + (t / 16 + 4 * i) * kGmxStride + (t % 16) * 16) = val[i];
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    // along H: a warp takes 8 rows x the 4 blocks of 32 columns, the 8 lanes of a quarter warp 8
    // rows of one block (their 16-byte reads fall in 8 different bank groups)
    const int it = t + 64 * k, r = 8 * (it >> 5) + (it & 7), b = (it & 31) >> 3;
    uint32_t wr[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = *reinterpret_cast<const uint4*>(tile + r * kGmxStride + b * 64 + 16 * i);
      wr[4 * i] = v.x, wr[4 * i + 1] = v.y, wr[4 * i + 2] = v.z, wr[4 * i + 3] = v.w;
    }
    uint32_t codes[8];
    sc_row[4 * r + b] = static_cast<uint8_t>(gmx_quant_row(wr, codes));
    st_ef_32B(dst_q + (r0 + r) * H + c0 + 32 * b, codes);
  }
  {  // along the rows: columns c0 + 2 (t % 64) and the next one (the low and high halves of each
     // staged word), row block t / 64; both columns' maxima and scaling share the packed words
    const int cp = t, rb = 0;
    uint32_t w2[32];
#pragma unroll
    for (int r = 0; r < 32; ++r)
      w2[r] = *reinterpret_cast<const uint32_t*>(tile + (32 * rb + r) * kGmxStride + 4 * cp);
    const uint32_t m = bf16x2_absmax_words(w2);
    const uint32_t m0 = m & 0xFFFFu, m1 = m >> 16;
    const int s0 = gmx_shared(m0), s1 = gmx_shared(m1);
    const uint32_t dn2 = gmx_mult(s0) | (gmx_mult(s1) << 16);
#pragma unroll
    for (int r = 0; r < 32; ++r) w2[r] = bf16x2_mul(w2[r], dn2);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t codes[8];
      const bool bad = (j ? m1 : m0) >= 0x7F80u;  // an Inf or NaN in this column's block
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t lo = j ? e4m3x2_of_halves<1>(w2[4 * i], w2[4 * i + 1])
                              : e4m3x2_of_halves<0>(w2[4 * i], w2[4 * i + 1]);
        const uint32_t hi = j ? e4m3x2_of_halves<1>(w2[4 * i + 2], w2[4 * i + 3])
                              : e4m3x2_of_halves<0>(w2[4 * i + 2], w2[4 * i + 3]);
        codes[i] = bad ? 0x7F7F7F7Fu : lo | (hi << 16);
      }
      sc_col[2 * cp + j] = static_cast<uint8_t>(bad ? 0xFFu : (j ? s1 : s0) + 127);
      st_ef_32B(dstR_q + static_cast<int64_t>(c0 + 2 * cp + j) * rcap + r0 + 32 * rb, codes);
    }
  }
  __syncthreads();
  // k-groups c0 / 32 ... + 3 of row r0 + t (t < 32: a 32-bit word); row group r0 / 32 of columns
  // c0 + t and c0 + 64 + t (one byte each)
  if (t < kGmxRows) {
    *reinterpret_cast<uint32_t*>(dst_sf + sf_atom_offset(r0 + t, c0 >> 5, H / 128)) =
        *reinterpret_cast<const uint32_t*>(sc_row + 4 * t);
  }
  dstR_sf[sf_atom_offset_g(c0 + t, r0 >> 5, rcap / 128, gT)] = sc_col[t];
  dstR_sf[sf_atom_offset_g(c0 + 64 + t, r0 >> 5, rcap / 128, gT)] = sc_col[64 + t];
}

// Scale atoms.  One block per 128-row slab of a source scale matrix (group g, atom j of the group):
// the slab's rows (kq 32-bit words each: four k-groups per word) are read with coalesced 4-byte
// loads into shared memory, then its kq atoms leave as 32 lines of 16 bytes each -- line l of atom
// q holds word q of rows l, l+32, l+64, l+96, the order tcgen05.cp's 32x128b.warpx4 shape expects.
// (Reading the four words of a line straight from global memory took 4 bytes from each of 32 rows
// per load instruction.)  The staged rows are an odd number of words apart, so the column reads of
// the 32 lanes fall in 32 different banks.  blockIdx.y selects the job.
struct ScaleJobs {
  ScaleJob j[3];
};
__global__ void __launch_bounds__(kMoveThreads) mx_scale_atoms_kernel(const ScaleJobs jobs) {
  pdl_wait();
  extern __shared__ uint32_t slab_words[];
  const ScaleJob jb = jobs.j[blockIdx.y];
  const int64_t slab = blockIdx.x;
  if (slab >= jb.groups * jb.atoms) return;
  const int64_t g = slab / jb.atoms;
  const int j = static_cast<int>(slab - g * jb.atoms);
  const int kq = jb.kq;
  const int stride = kq % 2 == 0 ? kq + 1 : kq;
  const uint8_t* srcp = (jb.two_src && j) ? jb.src1 : jb.src0;
  const int64_t row0 = jb.two_src ? g * 128 : slab * 128;
  const uint32_t* rows = reinterpret_cast<const uint32_t*>(srcp + row0 * 4 * kq);
  for (int w = threadIdx.x; w < 128 * kq; w += kMoveThreads) {
    const int r = w / kq;
    slab_words[r * stride + (w - r * kq)] = __ldg(rows + w);
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(jb.dst);
  for (int x = threadIdx.x; x < 32 * kq; x += kMoveThreads) {
    const int q = x >> 5, l = x & 31;
    const int64_t atom = (g * kq + q) * jb.atoms + j;
    dst[atom * 32 + l] = make_uint4(slab_words[l * stride + q], slab_words[(l + 32) * stride + q],
                                    slab_words[(l + 64) * stride + q], slab_words[(l + 96) * stride + q]);
  }
}

int grid_for(int64_t items, int per_block) {
  const int64_t want = (items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
  return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

int launch_gather_rows(const RowSrc& src, const int32_t* inv, const int32_t* row_token, const int32_t* meta,
                       int64_t T, int32_t K, int64_t rpad_max, int32_t H, uint16_t* dst, int kind,
                       cudaStream_t stream) {
  if (rpad_max <= 0) return 0;
  const int64_t vecs = H / 8;
  const int grid = grid_for(T * ((vecs + 127) / 128) + rpad_max / 32, kMoveThreads / 32);
  trace_begin(stream, kind);
  uint4* d = reinterpret_cast<uint4*>(dst);
  if (vecs >= 32 * 4)
    launch_pdl(gather_tokens_kernel<4>, dim3(grid), dim3(kMoveThreads), 0, stream, src, inv, row_token, meta, T, K, vecs, d);
  else
    launch_pdl(gather_tokens_kernel<1>, dim3(grid), dim3(kMoveThreads), 0, stream, src, inv, row_token, meta, T, K, vecs, d);
  trace_end(stream);
  return static_cast<int>(cudaGetLastError());
}

int launch_gather_rows_mx(const RowSrc& src, const int32_t* row_token, const int32_t* meta, int64_t rpad_max,
                          int32_t H, uint8_t* dst_q, uint8_t* dst_sf, uint8_t* dstR_q, uint8_t* dstR_sf,
                          int64_t rcap, int gT, int kind, cudaStream_t stream) {
  if (rpad_max <= 0) return 0;
  // column tiles fastest: blocks running together read whole source rows, not 256-byte pieces of
  // 128 scattered rows
  if ((rpad_max + kGmxRows - 1) / kGmxRows > 65535) return static_cast<int>(cudaErrorInvalidValue);
  const dim3 grid(static_cast<unsigned>(H / 128), static_cast<unsigned>((rpad_max + kGmxRows - 1) / kGmxRows));
  trace_begin(stream, kind);
  launch_pdl(gather_rows_mx_kernel, dim3(grid), dim3(64), 0, stream, src, row_token, meta, H, dst_q, dst_sf, dstR_q, dstR_sf, rcap, gT);
  trace_end(stream);
  return static_cast<int>(cudaGetLastError());
}

int launch_mx_scale_atoms(const ScaleJob* jobs, int njobs, cudaStream_t stream) {
  if (njobs <= 0 || njobs > 3) return static_cast<int>(cudaErrorInvalidValue);
  static DeviceOnce once;  // slabs of wide scale rows need more than the default 48 KB, on each device
  const int se = once.run([](int* d) { return static_cast<int>(cudaGetDevice(d)); },
                          [] {
                            return static_cast<int>(cudaFuncSetAttribute(
                                mx_scale_atoms_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024));
                          },
                          static_cast<int>(cudaErrorInvalidDevice));
  if (se) return se;
  ScaleJobs p{};
  int64_t slabs = 0;
  int kq = 0;
  for (int i = 0; i < njobs; ++i) {
    p.j[i] = jobs[i];
    const int64_t n = jobs[i].groups * jobs[i].atoms;
    slabs = n > slabs ? n : slabs;
    kq = jobs[i].kq > kq ? jobs[i].kq : kq;
  }
  if (slabs <= 0 || kq <= 0) return 0;
  const size_t smem = sizeof(uint32_t) * 128 * static_cast<size_t>(kq + 1);
  if (smem > 227 * 1024 || slabs > 0x7fffffff) return static_cast<int>(cudaErrorInvalidValue);
  const dim3 grid(static_cast<unsigned>(slabs), static_cast<unsigned>(njobs));
  trace_begin(stream, K_MX_SCALE_ATOMS);
  launch_pdl(mx_scale_atoms_kernel, dim3(grid), dim3(kMoveThreads), smem, stream, p);
  trace_end(stream);
  return static_cast<int>(cudaGetLastError());
}

static int combine_any(const uint16_t* y, const int32_t* inv, const int32_t* ids, int32_t e_total, const float* s,
                       int64_t T, int32_t K, int32_t H, uint16_t* out, int kind, cudaStream_t stream) {
  if (T <= 0) return 0;
  const int grid = grid_for(T, kMoveThreads / 32);
  trace_begin(stream, kind);
  const uint4* yv = reinterpret_cast<const uint4*>(y);
  uint4* ov = reinterpret_cast<uint4*>(out);
  if (K == 1)
    launch_pdl(combine_kernel<8, true>, dim3(grid), dim3(kMoveThreads), 0, stream, yv, inv, ids, e_total, s, T, K, H / 8, ov);
  else if (K == 2)
    launch_pdl(combine_kernel<4, true>, dim3(grid), dim3(kMoveThreads), 0, stream, yv, inv, ids, e_total, s, T, K, H / 8, ov);
  else if (K <= 4)
    launch_pdl(combine_kernel<2, true>, dim3(grid), dim3(kMoveThreads), 0, stream, yv, inv, ids, e_total, s, T, K, H / 8, ov);
  else  // one column vector, up to eight rows per batch (64 registers as it is)
    launch_pdl(combine_kernel<1, false>, dim3(grid), dim3(kMoveThreads), 0, stream, yv, inv, ids, e_total, s, T, K, H / 8, ov);
  trace_end(stream);
  return static_cast<int>(cudaGetLastError());
}

int launch_combine(const uint16_t* y, const int32_t* inv, const float* s, int64_t T, int32_t K, int32_t H,
                   uint16_t* out, int kind, cudaStream_t stream) {
  return combine_any(y, inv, nullptr, 0, s, T, K, H, out, kind, stream);
}

int launch_combine_slots(const uint16_t* rows, const int32_t* ids, int32_t e_total, const float* s, int64_t T,
                         int32_t K, int32_t H, uint16_t* out, int kind, cudaStream_t stream) {
  return combine_any(rows, nullptr, ids, e_total, s, T, K, H, out, kind, stream);
}

int launch_push_rows(const uint16_t* src, const int32_t* perm, const int32_t* meta, int64_t rpad_max, int32_t H,
                     const RowDst& dst, int kind, cudaStream_t stream) {
  if (rpad_max <= 0) return 0;
  const int grid = grid_for(rpad_max, kMoveThreads / 32);
  trace_begin(stream, kind);
  launch_pdl(push_rows_kernel, dim3(grid), dim3(kMoveThreads), 0, stream, reinterpret_cast<const uint4*>(src), perm, meta, H / 8, dst);
  trace_end(stream);
  return static_cast<int>(cudaGetLastError());
}

int launch_ds_push(const float* part, const int32_t* inv, int64_t R, int32_t n_tiles, const RowDst& dst, int32_t rank,
                   cudaStream_t stream) {
  if (R <= 0) return 0;
  const int grid = static_cast<int>((R + kMoveThreads - 1) / kMoveThreads);
  trace_begin(stream, K_DS_PUSH);
  launch_pdl(ds_push_kernel, dim3(grid), dim3(kMoveThreads), 0, stream, part, inv, R, n_tiles, dst, rank);
  trace_end(stream);
  return static_cast<int>(cudaGetLastError());
}

int launch_ds_reduce(const float* part, const int32_t* inv, int64_t R, int32_t n_tiles, float* ds,
                     cudaStream_t stream) {
  if (R <= 0) return 0;
  const int grid = static_cast<int>((R + kMoveThreads - 1) / kMoveThreads);
  trace_begin(stream, K_DS_REDUCE);
  launch_pdl(ds_reduce_kernel, dim3(grid), dim3(kMoveThreads), 0, stream, part, inv, R, n_tiles, ds);
  trace_end(stream);
  return static_cast<int>(cudaGetLastError());
}

int launch_mxfp8_quantize(const uint16_t* in, int64_t rows, int64_t cols, uint8_t* q, uint8_t* sc,
                          cudaStream_t stream) {
  const int64_t nblocks = rows * (cols / 32);
  if (nblocks <= 0) return 0;
  const int grid = grid_for(nblocks, kMoveThreads);
  trace_begin(stream, K_MXFP8_QUANTIZE);
  launch_pdl(mxfp8_quantize_kernel, dim3(grid), dim3(kMoveThreads), 0, stream, reinterpret_cast<const uint4*>(in), nblocks,
                                                           reinterpret_cast<uint4*>(q), sc);
  trace_end(stream);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace mok
