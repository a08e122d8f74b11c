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

static int clamp_grid(int num_ctas, int64_t units) {
  return static_cast<int>(units < num_ctas ? units : num_ctas);
}

int launch_dgrad_gemms(const Sizes& z, const mok_schedule& s, const Ctx& ctx, const Staging& st,
                       const mok_weights& w, int num_ctas, int phase, cudaStream_t stream) {
  CUtensorMap tA, tB, tB2, tO0, tO1;
  GemmArgs a = common_args(z, s);
  if (phase == 1) {
    const int BN = z.I % 256 == 0 ? 256 : 128;
    if (!make_tmap_bf16(&tA, st.dyg, z.H, z.rpad_max, 64, 128)) return -1;
    if (z.mx) {  // K-major B: Wd^T decoded from the copy quantised along H, [E*I, H]
      if (!make_tmap_bf16(&tB, st.wd_b, z.H, static_cast<uint64_t>(z.E) * z.I, 64, BN)) return -1;
    } else if (!make_tmap_bf16(&tB, w.w_down, z.I, static_cast<uint64_t>(z.E) * z.H, 64, 64)) {
      return -1;
    }
    a.n_tiles = z.I / BN;
    a.k_blocks = z.H / kBK;
    a.in0 = ctx.gu;
    a.in1 = ctx.a;
    a.out0 = st.dgdu;
    a.out1 = st.as;
    a.out2 = st.dspart;
    if (!make_tmap_bf16_sw64(&tO0, st.dgdu, 2 * static_cast<uint64_t>(z.I), z.rpad_max, 32, 32)) return -1;
    if (!make_tmap_bf16_sw64(&tO1, st.as, z.I, z.rpad_max, 32, 32)) return -1;
    const int grid = clamp_grid(num_ctas, z.mblocks_max * a.n_tiles);
    if (z.mx)
      return BN == 256 ? launch_gemm<V_DGRAD1, 256, true>(tA, tB, tB, tO0, tO1, a, grid, stream)
                       : launch_gemm<V_DGRAD1, 128, true>(tA, tB, tB, tO0, tO1, a, grid, stream);
    return BN == 256 ? launch_gemm<V_DGRAD1, 256>(tA, tB, tB, tO0, tO1, a, grid, stream)
                     : launch_gemm<V_DGRAD1, 128>(tA, tB, tB, tO0, tO1, a, grid, stream);
  }
  const int BN = z.H % 256 == 0 ? 256 : 128;
  if (!make_tmap_bf16(&tA, st.dgdu, 2 * static_cast<uint64_t>(z.I), z.rpad_max, 64, 128)) return -1;
  if (z.mx) {  // K-major B: Wg^T, Wu^T decoded from the copies quantised along I, [E*H, I]
    if (!make_tmap_bf16(&tB, st.wg_b, z.I, static_cast<uint64_t>(z.E) * z.H, 64, BN)) return -1;
    if (!make_tmap_bf16(&tB2, st.wu_b, z.I, static_cast<uint64_t>(z.E) * z.H, 64, BN)) return -1;
  } else {
    if (!make_tmap_bf16(&tB, w.w_gate, z.H, static_cast<uint64_t>(z.E) * z.I, 64, 64)) return -1;
    if (!make_tmap_bf16(&tB2, w.w_up, z.H, static_cast<uint64_t>(z.E) * z.I, 64, 64)) return -1;
  }
  a.n_tiles = z.H / BN;
  a.k_blocks = 2 * z.I / kBK;
  a.kb_split = z.I / kBK;
  a.out0 = st.ybuf;
  if (!make_tmap_bf16(&tO0, st.ybuf, z.H, z.rpad_max, 64, 32)) return -1;
  const int grid = clamp_grid(num_ctas, z.mblocks_max * a.n_tiles);
  if (z.mx)
    return BN == 256 ? launch_gemm<V_DGRAD2, 256, true>(tA, tB, tB2, tO0, tO0, a, grid, stream)
                     : launch_gemm<V_DGRAD2, 128, true>(tA, tB, tB2, tO0, tO0, a, grid, stream);
  return BN == 256 ? launch_gemm<V_DGRAD2, 256>(tA, tB, tB2, tO0, tO0, a, grid, stream)
                   : launch_gemm<V_DGRAD2, 128>(tA, tB, tB2, tO0, tO0, a, grid, stream);
}

}  // namespace mok
