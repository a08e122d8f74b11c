// mok_gemm_fwd.cu -- forward expert GEMMs: gate/up with the fused SwiGLU epilogue, then down.
// "Cursor Open-Sources Mixture-of-Kittens (MoK) ...", English summary: SwiGLU experts, BF16 mode.
#include "mok_gemm.cuh"

namespace mok {

static GemmArgs common_args(const Sizes& z, const mok_schedule& s) {
  GemmArgs a{};
  a.mblocks = s.mblocks;
  a.tiles = s.tiles;
  a.meta = s.meta;
  a.poff = s.poff;
  a.E = z.E;
  a.I = z.I;
  a.H = z.H;
  a.row_weight = s.row_weight;
  a.status = s.status;
  return a;
}

static int clamp_grid(int num_ctas, int64_t units) {
  return static_cast<int>(units < num_ctas ? units : num_ctas);
}

int launch_fwd_gemms(const Sizes& z, const mok_schedule& s, const Ctx& ctx, const Staging& st, const mok_weights& w,
                     int num_ctas, cudaStream_t stream) {
  CUtensorMap tA, tB, tB2, tO0, tO1;
  GemmArgs a = common_args(z, s);
  // [g | u] = Xg [Wg_e | Wu_e]^T : 128 gate columns and the same 128 up columns per tile
  if (!make_tmap_bf16(&tA, ctx.xg, z.H, z.rpad_max, 64, 128)) return -1;
  // MXFP8 mode: the exact bf16 decodes of the pre-quantised copies, same layouts
  const void* wg = z.mx ? static_cast<const void*>(st.wg_f) : w.w_gate;
  const void* wu = z.mx ? static_cast<const void*>(st.wu_f) : w.w_up;
  const void* wd = z.mx ? static_cast<const void*>(st.wd_f) : w.w_down;
  if (!make_tmap_bf16(&tB, wg, z.H, static_cast<uint64_t>(z.E) * z.I, 64, 128)) return -1;
  if (!make_tmap_bf16(&tB2, wu, z.H, static_cast<uint64_t>(z.E) * z.I, 64, 128)) return -1;
  a.n_tiles = z.I / 128;
  a.k_blocks = z.H / kBK;
  a.out0 = ctx.gu;
  a.out1 = ctx.a;
  if (z.mx) {  // g, u saved in fp32: 32-column tiles of 128-byte rows
    if (!make_tmap_f32(&tO0, ctx.gu, 2 * static_cast<uint64_t>(z.I), z.rpad_max, 32, 32)) return -1;
  } else if (!make_tmap_bf16(&tO0, ctx.gu, 2 * static_cast<uint64_t>(z.I), z.rpad_max, 64, 32)) {
    return -1;
  }
  if (!make_tmap_bf16(&tO1, ctx.a, z.I, z.rpad_max, 64, 32)) return -1;
  const int grid1 = clamp_grid(num_ctas, z.mblocks_max * a.n_tiles);
  int rc = z.mx ? launch_gemm<V_FWD_GATEUP, 256, true>(tA, tB, tB2, tO0, tO1, a, grid1, stream)
                : launch_gemm<V_FWD_GATEUP, 256>(tA, tB, tB2, tO0, tO1, a, grid1, stream);
  if (rc) return rc;
  // y = a Wd_e^T
  const int BN = z.H % 256 == 0 ? 256 : 128;
  if (!make_tmap_bf16(&tA, ctx.a, z.I, z.rpad_max, 64, 128)) return -1;
  if (!make_tmap_bf16(&tB, wd, z.I, static_cast<uint64_t>(z.E) * z.H, 64, BN)) return -1;
  a.n_tiles = z.H / BN;
  a.k_blocks = z.I / kBK;
  a.out0 = st.ybuf;
  a.out1 = nullptr;
  if (!make_tmap_bf16(&tO0, st.ybuf, z.H, z.rpad_max, 64, 32)) return -1;
  const int grid = clamp_grid(num_ctas, z.mblocks_max * a.n_tiles);
  return BN == 256 ? launch_gemm<V_FWD_DOWN, 256>(tA, tB, tB, tO0, tO0, a, grid, stream)
                   : launch_gemm<V_FWD_DOWN, 128>(tA, tB, tB, tO0, tO0, a, grid, stream);
}

}  // namespace mok
