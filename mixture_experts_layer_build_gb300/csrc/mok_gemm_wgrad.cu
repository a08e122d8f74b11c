// mok_gemm_wgrad.cu -- weight-gradient expert GEMMs (BF16, and block-scaled E4M3 in MXFP8 mode).  Each output tile of dW is reduced by one CTA
// over its expert's rows in ascending row order (K = the expert's padded rows; padding rows are
// zero), so the reduction order is fixed and no atomics are used.  Experts without rows get zeros.
#include "mok_gemm.cuh"

namespace mok {

// MXFP8: block-scaled E4M3 on operands quantised along the routed rows (K), read K-major from their
// transposed copies: [dWg ; dWu]_e = [dg | du]_e^T x_e and dWd_e = dY_e^T (s a)_e over e's padded rows.
// Block-scaled weight gradients run on CTA pairs (M = 256, each CTA holding half of the B tile)
// when the experts are long: the pair moves a third fewer shared-memory bytes per flop, and with K
// of 16 or more 128-row blocks per tile its single accumulator's drain is a small share of a tile.
// The scale atoms of a pair are loaded by tensor maps over the atom arrays seen as 128-byte rows.
static bool mx_wgrad_pairs(const Sizes& z) { return z.R >= static_cast<int64_t>(2048) * z.E; }

static int launch_wgrad_gemms_mx(const Sizes& z, const mok_schedule& s, const Ctx& ctx, const Staging& st,
                                 const mok_grads& g, int num_ctas, cudaStream_t stream) {
  CUtensorMap tA, tB, tO0, tO1, tSa, tSb;
  GemmArgs a{};
  a.poff = s.poff;
  a.E = z.E;
  a.I = z.I;
  a.H = z.H;
  a.status = s.status;
  a.sf_kq = static_cast<int32_t>(z.kq_rows());
  const uint64_t rcap = static_cast<uint64_t>(z.rcap());
  const uint64_t kq = static_cast<uint64_t>(z.kq_rows());
  // fp32 dW tiles: 32 rows x 16 columns per warp (wide tiles) or 128 rows x 32 columns per group
  // of four epilogue warps
  auto out_map = [&](CUtensorMap* m, float* p, uint64_t inner, uint64_t outer, int bn) {
    return bn == 256 ? make_tmap_f32_sw64(m, p, inner, outer, 16, 32) : make_tmap_f32(m, p, inner, outer, 32, 128);
  };
  // scale atoms as rows of 128 bytes: A's one atom per (M tile, K block), B's BN / 128 per (N tile,
  // K block)
  auto scale_maps = [&](const uint8_t* sfa, const uint8_t* sfb, int bn) {
    return make_tmap_u8(&tSa, sfa, 128, static_cast<uint64_t>(a.m_tiles) * kq * 4, 128, 4, 0) &&
           make_tmap_u8(&tSb, sfb, 128, static_cast<uint64_t>(a.n_tiles) * kq * (bn / 128) * 4, 128,
                        4 * (bn / 128), 0);
  };
  {  // [dWg ; dWu]_e: M = 2I (A = [dg | du]^T), N = H (B = x^T)
    const int BN = z.mx_bn_h();
    a.m_tiles = 2 * z.I / kBM;
    a.n_tiles = z.H / BN;
    const bool pair = mx_wgrad_pairs(z) && a.m_tiles % 2 == 0;
    if (!make_tmap_u8(&tA, st.dgr, rcap, 2 * static_cast<uint64_t>(z.I), 128, 128, 128)) return -1;
    if (!make_tmap_u8(&tB, ctx.xr, rcap, z.H, 128, pair ? BN / 2 : BN, 128)) return -1;
    a.sfa = st.dgrs;
    a.sfb = ctx.xrs;
    a.out0 = g.dw_gate;
    a.out1 = g.dw_up;
    if (!out_map(&tO0, g.dw_gate, z.H, static_cast<uint64_t>(z.E) * z.I, BN)) return -1;
    if (!out_map(&tO1, g.dw_up, z.H, static_cast<uint64_t>(z.E) * z.I, BN)) return -1;
    const int64_t units = static_cast<int64_t>(z.E) * (pair ? a.m_tiles / 2 : a.m_tiles) * a.n_tiles;
    const int grid = gemm_grid(z, num_ctas, units, pair, a);
    int rc;
    if (pair) {
      if (!scale_maps(st.dgrs, ctx.xrs, BN)) return -1;
      rc = BN == 256 ? launch_gemm<V_WGRAD_GU, 256, true, true>(tA, tB, tSa, tO0, tO1, tSb, a, grid, stream)
                     : launch_gemm<V_WGRAD_GU, 128, true, true>(tA, tB, tSa, tO0, tO1, tSb, a, grid, stream);
    } else {
      rc = BN == 256 ? launch_gemm<V_WGRAD_GU, 256, true>(tA, tB, tB, tO0, tO1, tO0, a, grid, stream)
                     : launch_gemm<V_WGRAD_GU, 128, true>(tA, tB, tB, tO0, tO1, tO0, a, grid, stream);
    }
    if (rc) return rc;
  }
  {  // dWd_e: M = H (A = dY^T), N = I (B = (s a)^T)
    const int BN = z.mx_bn_i();
    a.m_tiles = z.H / kBM;
    a.n_tiles = z.I / BN;
    const bool pair = mx_wgrad_pairs(z) && a.m_tiles % 2 == 0;
    if (!make_tmap_u8(&tA, st.dyr, rcap, z.H, 128, 128, 128)) return -1;
    if (!make_tmap_u8(&tB, st.sar, rcap, z.I, 128, pair ? BN / 2 : BN, 128)) return -1;
    a.sfa = st.dyrs;
    a.sfb = st.sars;
    a.out0 = g.dw_down;
    a.out1 = nullptr;
    if (!out_map(&tO0, g.dw_down, z.I, static_cast<uint64_t>(z.E) * z.H, BN)) return -1;
    const int64_t units = static_cast<int64_t>(z.E) * (pair ? a.m_tiles / 2 : a.m_tiles) * a.n_tiles;
    const int grid = gemm_grid(z, num_ctas, units, pair, a);
    if (pair) {
      if (!scale_maps(st.dyrs, st.sars, BN)) return -1;
      return BN == 256 ? launch_gemm<V_WGRAD_D, 256, true, true>(tA, tB, tSa, tO0, tO0, tSb, a, grid, stream)
                       : launch_gemm<V_WGRAD_D, 128, true, true>(tA, tB, tSa, tO0, tO0, tSb, a, grid, stream);
    }
    return BN == 256 ? launch_gemm<V_WGRAD_D, 256, true>(tA, tB, tB, tO0, tO0, tO0, a, grid, stream)
                     : launch_gemm<V_WGRAD_D, 128, true>(tA, tB, tB, tO0, tO0, tO0, a, grid, stream);
  }
}

int launch_wgrad_gemms(const Sizes& z, const mok_schedule& s, const Ctx& ctx, const Staging& st,
                       const mok_grads& g, int num_ctas, cudaStream_t stream) {
  if (z.mx) return launch_wgrad_gemms_mx(z, s, ctx, st, g, num_ctas, stream);
  CUtensorMap tA, tB, tO0, tO1;
  GemmArgs a{};
  a.poff = s.poff;
  a.counts = s.counts;
  a.E = z.E;
  a.I = z.I;
  a.H = z.H;
  a.status = s.status;
  // fp32 dW leaves in 128-row x 32-column tiles
  constexpr uint32_t orows = 128;
  // [dWg ; dWu]_e = [dg | du]_e^T Xg_e   (M = 2I, N = H)
  {
    const int BN = z.H % 256 == 0 ? 256 : 128;
    if (!make_tmap_bf16(&tA, st.dgdu, 2 * static_cast<uint64_t>(z.I), z.rpad_max, 64, 64)) return -1;
    if (!make_tmap_bf16(&tB, ctx.xg, z.H, z.rpad_max, 64, 64)) return -1;
    a.m_tiles = 2 * z.I / kBM;
    a.n_tiles = z.H / BN;
    a.out0 = g.dw_gate;
    a.out1 = g.dw_up;
    if (!make_tmap_f32(&tO0, g.dw_gate, z.H, static_cast<uint64_t>(z.E) * z.I, 32, orows)) return -1;
    if (!make_tmap_f32(&tO1, g.dw_up, z.H, static_cast<uint64_t>(z.E) * z.I, 32, orows)) return -1;
    const int64_t units = static_cast<int64_t>(z.E) * a.m_tiles * a.n_tiles;
    const int grid = gemm_grid(z, num_ctas, units, false, a);
    const int rc = BN == 256 ? launch_gemm<V_WGRAD_GU, 256>(tA, tB, tB, tO0, tO1, tO0, a, grid, stream)
                             : launch_gemm<V_WGRAD_GU, 128>(tA, tB, tB, tO0, tO1, tO0, a, grid, stream);
    if (rc) return rc;
  }
  // dWd_e = dYg_e^T (s a)_e   (M = H, N = I)
  {
    const int BN = z.I % 256 == 0 ? 256 : 128;
    if (!make_tmap_bf16(&tA, st.dyg, z.H, z.rpad_max, 64, 64)) return -1;
    if (!make_tmap_bf16(&tB, st.as, z.I, z.rpad_max, 64, 64)) return -1;
    a.m_tiles = z.H / kBM;
    a.n_tiles = z.I / BN;
    a.out0 = g.dw_down;
    a.out1 = nullptr;
    if (!make_tmap_f32(&tO0, g.dw_down, z.I, static_cast<uint64_t>(z.E) * z.H, 32, orows)) return -1;
    const int64_t units = static_cast<int64_t>(z.E) * a.m_tiles * a.n_tiles;
    const int grid = gemm_grid(z, num_ctas, units, false, a);
    return BN == 256 ? launch_gemm<V_WGRAD_D, 256>(tA, tB, tB, tO0, tO0, tO0, a, grid, stream)
                     : launch_gemm<V_WGRAD_D, 128>(tA, tB, tB, tO0, tO0, tO0, a, grid, stream);
  }
}

}  // namespace mok
