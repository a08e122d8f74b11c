// mok_gemm_dgrad.cu -- backward data-gradient expert GEMMs.
//   phase 1: dA' = dYg Wd_e with the SwiGLU backward and the router-weight gradient partials fused
//            into the epilogue ("Cursor Open-Sources Mixture-of-Kittens (MoK) ...", English summary:
//            SonicMoE-style router-weight gradient inside the SwiGLU backward);
//   phase 2: dXg = [dg | du] [Wg_e ; Wu_e].
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

// MXFP8: both GEMMs block-scaled on E4M3 operands.  B is the K-major transposed weight copy
// quantised along this GEMM's K: Wd^T [E*I, H] for phase 1 (128 x 128 tiles: its epilogue keeps
// two accumulators), Wg^T | Wu^T [E*H, I] for phase 2 (128 x 256 tiles when H allows).
static int launch_dgrad_gemms_mx(const Sizes& z, const mok_schedule& s, const Ctx& ctx, const Staging& st,
                                 const mok_weights& w, int num_ctas, int phase, cudaStream_t stream) {
  CUtensorMap tA, tB, tB2, tO0, tO1, tO2;
  GemmArgs a = common_args(z, s);
  const uint64_t EI = static_cast<uint64_t>(z.E) * z.I, EH = static_cast<uint64_t>(z.E) * z.H;
  if (phase == 1) {
    if (!make_tmap_u8(&tA, st.dyq, z.H, z.rpad_max, 128, 128, 128)) return -1;
    if (!make_tmap_u8(&tB, w.qt_down, z.H, EI, 128, 128, 128)) return -1;
    a.n_tiles = z.I / 128;
    a.k_blocks = z.H / 128;
    a.sfa = st.dys;
    a.sfb = st.swt_d;
    a.sfb_kq = z.H / 128;
    a.in0 = ctx.gu;
    a.in1 = ctx.a;
    a.out2 = st.dspart;
    a.out_sf = st.dgs;
    a.out_kq = 2 * z.I / 128;
    a.sf_kq = static_cast<int32_t>(z.kq_rows());
    a.sa_groups = z.mx_bn_i() / 128;
    a.out_sf2 = st.dgrs;
    a.out_sf3 = st.sars;
    // 32 x 32 byte tiles of the row-quantised [dg | du] and s a, transposed [features, rcap]
    const uint64_t rcap = static_cast<uint64_t>(z.rcap());
    if (!make_tmap_u8(&tO0, st.dgr, rcap, 2 * static_cast<uint64_t>(z.I), 32, 32, 32)) return -1;
    if (!make_tmap_u8(&tO1, st.sar, rcap, z.I, 32, 32, 32)) return -1;
    if (!make_tmap_u8(&tO2, st.dgq, 2 * static_cast<uint64_t>(z.I), z.rpad_max, 32, 32, 32)) return -1;
    const int grid = gemm_grid(z, num_ctas, z.mblocks_max * a.n_tiles, false, a);
    // The tile's epilogue (dg, du and s a, each quantised along both axes) is about as long as
    // its MMAs over K = H = 4096: up to there eight epilogue warps pay; beyond, the operand feed
    // bounds the tile and four warps are as fast.
    if (z.mx_dg1_split()) return launch_gemm<V_DGRAD1, 128, true, false, true>(tA, tB, tB, tO0, tO1, tO2, a, grid, stream);
    return launch_gemm<V_DGRAD1, 128, true>(tA, tB, tB, tO0, tO1, tO2, a, grid, stream);
  }
  const int BN = z.mx_bn_h();
  if (!make_tmap_u8(&tA, st.dgq, 2 * static_cast<uint64_t>(z.I), z.rpad_max, 128, 128, 128)) return -1;
  if (!make_tmap_u8(&tB, w.qt_gate, z.I, EH, 128, BN, 128)) return -1;
  if (!make_tmap_u8(&tB2, w.qt_up, z.I, EH, 128, BN, 128)) return -1;
  a.n_tiles = z.H / BN;
  a.k_blocks = 2 * z.I / 128;
  a.kb_split = z.I / 128;
  a.sfa = st.dgs;
  a.sfb = st.swt_g;
  a.sfb2 = st.swt_u;
  a.sfb_kq = z.I / 128;
  a.out0 = st.ybuf;
  if (!(BN == 256 ? make_tmap_bf16_sw64(&tO0, st.ybuf, z.H, z.rpad_max, 32, 32)
                  : make_tmap_bf16(&tO0, st.ybuf, z.H, z.rpad_max, 64, 128)))
    return -1;
  const int grid = gemm_grid(z, num_ctas, z.mblocks_max * a.n_tiles, false, a);
  return BN == 256 ? launch_gemm<V_DGRAD2, 256, true>(tA, tB, tB2, tO0, tO0, tO0, a, grid, stream)
                   : launch_gemm<V_DGRAD2, 128, true>(tA, tB, tB2, tO0, tO0, tO0, a, grid, stream);
}

int launch_dgrad_gemms(const Sizes& z, const mok_schedule& s, const Ctx& ctx, const Staging& st,
                       const mok_weights& w, int num_ctas, int phase, cudaStream_t stream) {
  if (z.mx) return launch_dgrad_gemms_mx(z, s, ctx, st, w, num_ctas, phase, stream);
  CUtensorMap tA, tB, tB2, tO0, tO1;
  GemmArgs a = common_args(z, s);
  a.pairs = st.pairs;  // on a CTA pair each CTA loads BN / 2 columns of B
  if (phase == 1) {
    const bool pair = use_pairs(z, 512);
    const int BN = z.I % 256 == 0 ? 256 : 128;
    if (!make_tmap_bf16(&tA, st.dyg, z.H, z.rpad_max, 64, 128)) return -1;
    if (!make_tmap_bf16(&tB, w.w_down, z.I, static_cast<uint64_t>(z.E) * z.H, 64, 64)) return -1;
    a.n_tiles = z.I / BN;
    a.k_blocks = z.H / kBK;
    a.in0 = ctx.gu;
    a.in1 = ctx.a;
    a.out0 = st.dgdu;
    a.out1 = st.as;
    a.out2 = st.dspart;
    if (!make_tmap_bf16_sw64(&tO0, st.dgdu, 2 * static_cast<uint64_t>(z.I), z.rpad_max, 32, 32)) return -1;
    if (!make_tmap_bf16_sw64(&tO1, st.as, z.I, z.rpad_max, 32, 32)) return -1;
    const int grid = gemm_grid(z, num_ctas, z.mblocks_max * a.n_tiles, pair, a);
    if (pair)
      return BN == 256 ? launch_gemm<V_DGRAD1, 256, false, true>(tA, tB, tB, tO0, tO1, tO0, a, grid, stream)
                       : launch_gemm<V_DGRAD1, 128, false, true>(tA, tB, tB, tO0, tO1, tO0, a, grid, stream);
    return BN == 256 ? launch_gemm<V_DGRAD1, 256>(tA, tB, tB, tO0, tO1, tO0, a, grid, stream)
                     : launch_gemm<V_DGRAD1, 128>(tA, tB, tB, tO0, tO1, tO0, a, grid, stream);
  }
  const bool pair = use_pairs(z, 256);
  const int BN = z.H % 256 == 0 ? 256 : 128;
  if (!make_tmap_bf16(&tA, st.dgdu, 2 * static_cast<uint64_t>(z.I), z.rpad_max, 64, 128)) return -1;
  if (!make_tmap_bf16(&tB, w.w_gate, z.H, static_cast<uint64_t>(z.E) * z.I, 64, 64)) return -1;
  if (!make_tmap_bf16(&tB2, w.w_up, z.H, static_cast<uint64_t>(z.E) * z.I, 64, 64)) return -1;
  a.n_tiles = z.H / BN;
  a.k_blocks = 2 * z.I / kBK;
  a.kb_split = z.I / kBK;
  a.out0 = st.ybuf;
  if (!make_tmap_bf16(&tO0, st.ybuf, z.H, z.rpad_max, 64, 128)) return -1;
  const int grid = gemm_grid(z, num_ctas, z.mblocks_max * a.n_tiles, pair, a);
  if (pair)
    return BN == 256 ? launch_gemm<V_DGRAD2, 256, false, true>(tA, tB, tB2, tO0, tO0, tO0, a, grid, stream)
                     : launch_gemm<V_DGRAD2, 128, false, true>(tA, tB, tB2, tO0, tO0, tO0, a, grid, stream);
  return BN == 256 ? launch_gemm<V_DGRAD2, 256>(tA, tB, tB2, tO0, tO0, tO0, a, grid, stream)
                   : launch_gemm<V_DGRAD2, 128>(tA, tB, tB2, tO0, tO0, tO0, a, grid, stream);
}

}  // namespace mok
