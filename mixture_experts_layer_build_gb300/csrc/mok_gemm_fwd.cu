// mok_gemm_fwd.cu -- forward expert GEMMs: gate/up with the fused SwiGLU epilogue, then down.
// "Cursor Open-Sources Mixture-of-Kittens (MoK) ...", English summary: SwiGLU experts, BF16 and
// MXFP8 modes.
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

// MXFP8: both GEMMs block-scaled on E4M3 operands, 128 x 256 tiles (128 x 128 for the down
// projection when H is not a multiple of 256).
static int launch_fwd_gemms_mx(const Sizes& z, const mok_schedule& s, const Ctx& ctx, const Staging& st,
                               const mok_weights& w, int num_ctas, cudaStream_t stream) {
  CUtensorMap tA, tB, tB2, tO0, tO1, tO2;
  GemmArgs a = common_args(z, s);
  const uint64_t EI = static_cast<uint64_t>(z.E) * z.I, EH = static_cast<uint64_t>(z.E) * z.H;
  // [g | u] = Xq [Wg_e | Wu_e]^T: 128 gate columns and the same 128 up columns per tile
  if (!make_tmap_u8(&tA, st.xq, z.H, z.rpad_max, 128, 128, 128)) return -1;
  if (!make_tmap_u8(&tB, w.q_gate, z.H, EI, 128, 128, 128)) return -1;
  if (!make_tmap_u8(&tB2, w.q_up, z.H, EI, 128, 128, 128)) return -1;
  a.n_tiles = z.I / 128;
  a.k_blocks = z.H / 128;
  a.sfa = st.xs;
  a.sfb = st.sw_gu;
  a.sfb_kq = z.H / 128;
  a.out0 = ctx.gu;
  a.out1 = ctx.a;
  a.out_sf = st.as_sf;
  a.out_kq = z.I / 128;
  // wide-tile epilogue stores: 2 KB tiles (16 fp32 / 32 bf16 / 32 e4m3 columns x 32 rows)
  if (!make_tmap_f32_sw64(&tO0, ctx.gu, 2 * static_cast<uint64_t>(z.I), z.rpad_max, 16, 32)) return -1;
  if (!make_tmap_bf16_sw64(&tO1, ctx.a, z.I, z.rpad_max, 32, 32)) return -1;
  if (!make_tmap_u8(&tO2, st.aq, z.I, z.rpad_max, 32, 32, 32)) return -1;
  const int grid1 = gemm_grid(z, num_ctas, z.mblocks_max * a.n_tiles, false, a);
  int rc = launch_gemm<V_FWD_GATEUP, 256, true>(tA, tB, tB2, tO0, tO1, tO2, a, grid1, stream);
  if (rc) return rc;
  // y = aq Wd_e^T
  const int BN = z.mx_bn_h();
  if (!make_tmap_u8(&tA, st.aq, z.I, z.rpad_max, 128, 128, 128)) return -1;
  if (!make_tmap_u8(&tB, w.q_down, z.I, EH, 128, BN, 128)) return -1;
  a.n_tiles = z.H / BN;
  a.k_blocks = z.I / 128;
  a.sfa = st.as_sf;
  a.sfb = st.sw_d;
  a.sfb_kq = z.I / 128;
  a.out0 = st.ybuf;
  a.out1 = nullptr;
  a.out_sf = nullptr;
  if (!(BN == 256 ? make_tmap_bf16_sw64(&tO0, st.ybuf, z.H, z.rpad_max, 32, 32)
                  : make_tmap_bf16(&tO0, st.ybuf, z.H, z.rpad_max, 64, 128)))
    return -1;
  const int grid = gemm_grid(z, num_ctas, z.mblocks_max * a.n_tiles, false, a);
  return BN == 256 ? launch_gemm<V_FWD_DOWN, 256, true>(tA, tB, tB, tO0, tO0, tO0, a, grid, stream)
                   : launch_gemm<V_FWD_DOWN, 128, true>(tA, tB, tB, tO0, tO0, tO0, a, grid, stream);
}

int launch_fwd_gemms(const Sizes& z, const mok_schedule& s, const Ctx& ctx, const Staging& st, const mok_weights& w,
                     int num_ctas, cudaStream_t stream) {
  if (z.mx) return launch_fwd_gemms_mx(z, s, ctx, st, w, num_ctas, stream);
  CUtensorMap tA, tB, tB2, tO0, tO1;
  GemmArgs a = common_args(z, s);
  a.pairs = st.pairs;
  const bool pair = use_pairs(z, 256);
  // [g | u] = Xg [Wg_e | Wu_e]^T : 128 gate columns and the same 128 up columns per tile (on a CTA
  // pair, the first CTA holds the gate rows of Wg, the second the up rows of Wu)
  if (!make_tmap_bf16(&tA, ctx.xg, z.H, z.rpad_max, 64, 128)) return -1;
  if (!make_tmap_bf16(&tB, w.w_gate, z.H, static_cast<uint64_t>(z.E) * z.I, 64, 128)) return -1;
  if (!make_tmap_bf16(&tB2, w.w_up, z.H, static_cast<uint64_t>(z.E) * z.I, 64, 128)) return -1;
  a.n_tiles = z.I / 128;
  a.k_blocks = z.H / kBK;
  a.out0 = ctx.gu;
  a.out1 = ctx.a;
  if (!make_tmap_bf16(&tO0, ctx.gu, 2 * static_cast<uint64_t>(z.I), z.rpad_max, 64, 128)) return -1;
  if (!make_tmap_bf16(&tO1, ctx.a, z.I, z.rpad_max, 64, 128)) return -1;
  const int grid1 = gemm_grid(z, num_ctas, z.mblocks_max * a.n_tiles, pair, a);
  int rc = pair ? launch_gemm<V_FWD_GATEUP, 256, false, true>(tA, tB, tB2, tO0, tO1, tO0, a, grid1, stream)
                : launch_gemm<V_FWD_GATEUP, 256>(tA, tB, tB2, tO0, tO1, tO0, a, grid1, stream);
  if (rc) return rc;
  // y = a Wd_e^T (each CTA of a pair loads BN / 2 rows of Wd)
  const int BN = z.H % 256 == 0 ? 256 : 128;
  if (!make_tmap_bf16(&tA, ctx.a, z.I, z.rpad_max, 64, 128)) return -1;
  if (!make_tmap_bf16(&tB, w.w_down, z.I, static_cast<uint64_t>(z.E) * z.H, 64, pair ? BN / 2 : BN)) return -1;
  a.n_tiles = z.H / BN;
  a.k_blocks = z.I / kBK;
  a.out0 = st.ybuf;
  a.out1 = nullptr;
  if (!make_tmap_bf16(&tO0, st.ybuf, z.H, z.rpad_max, 64, 128)) return -1;
  const int grid = gemm_grid(z, num_ctas, z.mblocks_max * a.n_tiles, pair, a);
  if (pair)
    return BN == 256 ? launch_gemm<V_FWD_DOWN, 256, false, true>(tA, tB, tB, tO0, tO0, tO0, a, grid, stream)
                     : launch_gemm<V_FWD_DOWN, 128, false, true>(tA, tB, tB, tO0, tO0, tO0, a, grid, stream);
  return BN == 256 ? launch_gemm<V_FWD_DOWN, 256>(tA, tB, tB, tO0, tO0, tO0, a, grid, stream)
                   : launch_gemm<V_FWD_DOWN, 128>(tA, tB, tB, tO0, tO0, tO0, a, grid, stream);
}

}  // namespace mok
