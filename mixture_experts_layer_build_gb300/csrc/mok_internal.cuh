// mok_internal.cuh -- declarations shared by the library's translation units (not part of the ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "mok.h"

namespace mok {

constexpr int kRowTile = 128;       // GEMM row tile: each expert's segment is padded to it
constexpr int kSchedChunk = 512;    // slots per warp in the schedule histogram / scatter
constexpr int kSchedWarps = 8;      // warps per CTA in the schedule kernels

// Expert parallelism: buffers of the group's ranks, read (or written) through tables of device
// pointers.  Token t of the group's global order lives on rank t / rows_per at row t % rows_per;
// slot j = t * K + k likewise at j % (rows_per * K).  n == 0: one plain buffer, p[0].
constexpr int kEpMax = 8;
struct RouteSrc {             // the routing the schedule reads
  const int32_t* ids[kEpMax];
  const float* w[kEpMax];
  int64_t slots_per;          // slots per rank (tokens per rank * K)
  int32_t n;                  // ranks, 0 = plain
  int32_t e0;                 // first global expert of this rank: local id = global id - e0
  int32_t e_total;            // experts of the group: global ids outside [0, e_total) are invalid
};
struct RowSrc {               // token rows the gathers read
  const uint16_t* p[kEpMax];
  int64_t rows_per;
  int32_t n;
};
struct RowDst {               // per-slot rows / values the pushes write ([rows_per * K] per rank)
  void* p[kEpMax];
  int64_t slots_per;
  int32_t n;
};
#ifdef __CUDACC__
// Entry r of a per-rank table held in a kernel parameter, chosen by an unrolled select: indexing the
// parameter array with a run-time r makes the compiler copy the whole struct to local memory in
// every thread.
template <class P>
__device__ __forceinline__ P pick_rank(const P (&tab)[kEpMax], int64_t r) {
  P v = tab[0];
#pragma unroll
  for (int i = 1; i < kEpMax; ++i) v = r == i ? tab[i] : v;
  return v;
}
#endif
// Slot codes of the schedule's inv[] besides a row index: a slot whose expert another rank owns
// (expert parallelism), and a slot whose id is invalid (outside [0, E) or the group's experts).
constexpr int32_t kSlotForeign = -1;
constexpr int32_t kSlotInvalid = -2;

// Derived sizes of one (shape, config) pair.
struct Sizes {
  int64_t T, R, rpad_max, tiles_max, mblocks_max, nchunks;
  int32_t H, I, E, K, mb, MB;
  bool mx;  // MXFP8 mode
  bool clc;  // single-CTA GEMM tiles scheduled by cluster launch control (else static round robin)
  // MXFP8 tile width (N) of the GEMMs whose N runs over H (or I): 256 when the size allows it
  int32_t mx_bn_h() const { return H % 256 == 0 ? 256 : 128; }
  int32_t mx_bn_i() const { return I % 256 == 0 ? 256 : 128; }
  // block-scaled first data-gradient GEMM: eight epilogue warps (two column halves, two dS
  // partials per 128-column tile) while K = H is short enough that the epilogue bounds the tile
  bool mx_dg1_split() const { return mx && H <= 4096; }
  // MXFP8 weight gradients: routed-row capacity in 128-row K atoms, and in rows
  int64_t kq_rows() const { return (rpad_max + kRowTile - 1) / kRowTile; }
  int64_t rcap() const { return kq_rows() * kRowTile; }
};
bool make_sizes(const mok_config* cfg, const mok_shape* shape, Sizes* s);

// Staging buffers inside the workspace (after the schedule tables) and the forward context.
struct Staging {
  uint16_t* ybuf;    // [rpad_max, H] bf16: expert outputs y (forward), then dX per row (backward)
  // BF16 mode only
  uint16_t* dyg;     // [rpad_max, H] bf16: gathered upstream gradient rows
  uint16_t* dgdu;    // [rpad_max, 2I] bf16: [dg | du]
  uint16_t* as;      // [rpad_max, I] bf16: s * a
  float* dspart;     // [rpad_max, I/128] fp32: router-gradient partial sums per N tile
  // BF16 GEMMs run by CTA pairs: per pair of consecutive 128-row blocks of one minibatch tile
  // {expert, first row, tile index, index of the tile's first pair}; meta[3] pairs
  int4* pairs;       // [mblocks_max]
  int32_t* chunk_hist;  // [nchunks, E+1]
  // MXFP8 mode only: E4M3 operands of the block-scaled GEMMs and their E8M0 scales, the scales
  // atom-tiled (sf_atom_offset: 512 bytes per 128 rows x 4 k-groups)
  uint8_t* xq;       // [rpad_max, H]  gathered x, quantised along H
  uint8_t* xs;       //   scales: rtiles x H/128 atoms
  uint8_t* aq;       // [rpad_max, I]  a, quantised along I
  uint8_t* as_sf;    //   scales: rtiles x I/128 atoms
  uint8_t* dyq;      // [rpad_max, H]  gathered dY, quantised along H
  uint8_t* dys;      //   scales: rtiles x H/128 atoms
  uint8_t* dgq;      // [rpad_max, 2I] [dg | du], quantised along I
  uint8_t* dgs;      //   scales: rtiles x 2I/128 atoms
  // weight-gradient operands, quantised along the routed rows (32-row blocks of the padded layout),
  // transposed [features, rcap] (K-major operands of the wgrad GEMMs); scales in sf_atom_offset_g
  // layout (row f = feature, k-group = row / 32, kq_rows atoms along K)
  uint8_t* dyr;      // [H, rcap]  dY          scales dyrs: A operand (G = 1)
  uint8_t* dyrs;
  uint8_t* dgr;      // [2I, rcap] [dg | du]   scales dgrs: A operand (G = 1)
  uint8_t* dgrs;
  uint8_t* sar;      // [I, rcap]  s * a       scales sars: B operand (G = mx_bn_i / 128)
  uint8_t* sars;
  // the caller's weight scales re-tiled into atom groups matching the B tiles (per call)
  uint8_t* sw_gu;    // s_gate, s_up: per 128 rows of I, the gate atom then the up atom
  uint8_t* sw_d;     // s_down: groups of BN_down / 128 atoms
  uint8_t* swt_d;    // st_down: single atoms (128-row tiles)
  uint8_t* swt_g;    // st_gate: groups of BN_dgrad2 / 128 atoms
  uint8_t* swt_u;    // st_up: same
};
struct Ctx {
  uint16_t* xg;      // BF16 mode: [rpad_max, H] bf16 gathered x rows (zero on padding rows)
  uint8_t* xr;       // MXFP8 mode: [H, rcap] x quantised along the routed rows, transposed
  uint8_t* xrs;      //   scales: B operand of the gate/up weight gradient (G = mx_bn_h / 128)
  void* gu;          // [rpad_max, 2I]: [g | u], bf16 (BF16 mode) or fp32 (MXFP8 mode, whose
                     // backward re-quantises dg, du and s * a and needs g, u unrounded)
  uint16_t* a;       // [rpad_max, I] bf16: silu(g) * u (MXFP8: its quantisation along I)
};
size_t carve_workspace(const Sizes& z, char* base, mok_schedule* sched, Staging* st);  // returns bytes
size_t carve_ctx(const Sizes& z, char* base, Ctx* ctx);

int sm_count();

// Kernel kinds reported through mok_trace.
enum KernelKind : int {
  K_SCHED_HIST = 0,
  K_SCHED_SCAN,
  K_SCHED_SCATTER,
  K_GATHER_X,
  K_GEMM_FWD_GATEUP,
  K_GEMM_FWD_DOWN,
  K_COMBINE,
  K_GATHER_DY,
  K_GEMM_DGRAD1,
  K_DS_REDUCE,
  K_GEMM_DGRAD2,
  K_DX_REDUCE,
  K_GEMM_WGRAD_GU,
  K_GEMM_WGRAD_D,
  K_MXFP8_QUANTIZE,
  K_MX_SCALE_ATOMS,
  K_ROUTER_LOGITS,
  K_ROUTER_TOPK,
  K_ROUTER_TRANSPOSE,
  K_ROUTER_DX,
  K_ROUTER_DW,
  K_SELFTEST_WAIT,
  K_PUSH_Y,
  K_PUSH_DX,
  K_EP_COMBINE,
  K_EP_DX_REDUCE,
  K_DS_PUSH,
  K_NUM_KINDS
};
void trace_begin(cudaStream_t s, int kind);  // no-ops unless a trace is set
void trace_end(cudaStream_t s);

// A kernel launch with programmatic stream serialisation: the grid may start launching as the
// previous kernel's last CTAs exit.  Only for kernels that begin with pdl_wait() (mok_ptx.cuh), so
// nothing they read or write is touched before their producer has completed.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// launchers (return a cudaError_t as int)
int launch_schedule(const Sizes& z, const RouteSrc& route, const mok_schedule& s, const Staging& st,
                    cudaStream_t stream);
inline RouteSrc plain_route(const int32_t* ids, const float* w) {
  RouteSrc r{};
  r.ids[0] = ids;
  r.w[0] = w;
  return r;
}
inline RowSrc plain_rows(const void* p) {
  RowSrc r{};
  r.p[0] = static_cast<const uint16_t*>(p);
  return r;
}
int launch_gather_rows(const RowSrc& src, const int32_t* inv, const int32_t* row_token, const int32_t* meta,
                       int64_t T, int32_t K, int64_t rpad_max, int32_t H, uint16_t* dst, int kind,
                       cudaStream_t stream);
// MX gather of 32-row blocks: dst_q / dst_sf = rows quantised along H (row-major, A-operand atoms);
// dstR_q / dstR_sf = the same rows quantised along the rows, transposed [H, rcap] (atoms grouped gT
// at a time).
int launch_gather_rows_mx(const RowSrc& src, const int32_t* row_token, const int32_t* meta, int64_t rpad_max,
                          int32_t H, uint8_t* dst_q, uint8_t* dst_sf, uint8_t* dstR_q, uint8_t* dstR_sf,
                          int64_t rcap, int gT, int kind, cudaStream_t stream);
// Re-tile row-major E8M0 scales [rows, 4 kq] into groups of `atoms` 512-byte atoms (up to three
// jobs per launch): group g, K atom q holds `atoms` consecutive atoms at ((g * kq + q) * atoms + j)
// * 512.  One source: atom j covers rows (g * atoms + j) * 128 ...; two sources (atoms = 2): atom
// j covers rows g * 128 ... of source j.
struct ScaleJob {
  const uint8_t* src0;
  const uint8_t* src1;  // two-source jobs only
  uint8_t* dst;
  int64_t groups;
  int32_t kq;           // K atoms = k-groups / 4
  int32_t atoms;        // atoms per group: 1 or 2
  int32_t two_src;
};
int launch_mx_scale_atoms(const ScaleJob* jobs, int njobs, cudaStream_t stream);
int launch_combine(const uint16_t* y, const int32_t* inv, const float* s, int64_t T, int32_t K, int32_t H,
                   uint16_t* out, int kind, cudaStream_t stream);
// Expert parallelism, the token owner's combine: out[t] = sum over k ascending of s[t,k] * rows[t*K+k]
// (s == nullptr: weight 1), over the slots whose global id lies in [0, e_total).
int launch_combine_slots(const uint16_t* rows, const int32_t* ids, int32_t e_total, const float* s, int64_t T,
                         int32_t K, int32_t H, uint16_t* out, int kind, cudaStream_t stream);
int launch_ds_reduce(const float* part, const int32_t* inv, int64_t R, int32_t n_tiles, float* ds,
                     cudaStream_t stream);
// Expert parallelism: dS of this rank's slots into the token owners' [slots_per] buffers; this
// rank also writes 0 for its own tokens' invalid slots (rank = own index in dst).
int launch_ds_push(const float* part, const int32_t* inv, int64_t R, int32_t n_tiles, const RowDst& dst, int32_t rank,
                   cudaStream_t stream);
// Expert parallelism: row r of src ([Rpad, H] bf16, r < meta[0]) holding slot j = perm[r] goes to
// the slot's owner, dst.p[j / slots_per] + (j % slots_per) * H.
int launch_push_rows(const uint16_t* src, const int32_t* perm, const int32_t* meta, int64_t rpad_max, int32_t H,
                     const RowDst& dst, int kind, cudaStream_t stream);
int launch_mxfp8_quantize(const uint16_t* in, int64_t rows, int64_t cols, uint8_t* q, uint8_t* sc,
                          cudaStream_t stream);

// GEMM phases
int launch_fwd_gemms(const Sizes& z, const mok_schedule& s, const Ctx& ctx, const Staging& st, const mok_weights& w,
                     int num_ctas, cudaStream_t stream);
int launch_dgrad_gemms(const Sizes& z, const mok_schedule& s, const Ctx& ctx, const Staging& st,
                       const mok_weights& w, int num_ctas, int phase, cudaStream_t stream);
int launch_wgrad_gemms(const Sizes& z, const mok_schedule& s, const Ctx& ctx, const Staging& st,
                       const mok_grads& g, int num_ctas, cudaStream_t stream);

}  // namespace mok
