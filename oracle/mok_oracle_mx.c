/*
 * mok_oracle_mx.c -- TEST INFRASTRUCTURE ONLY: the fp64 oracle of the layer's MXFP8 mode.
 *
 * Same status as mok_oracle.c: only tests/, __graft_entry__.smoke() and bench.py's CPU baseline may
 * load it; it shares nothing with the CUDA library.
 *
 * Source: "Cursor Open-Sources Mixture-of-Kittens (MoK) ..." (yifor-blog digest of MarkTechPost),
 * English summary (BF16 and MXFP8 precision modes, forward and backward); "Mixture-of-Kittens
 * (MoK)" project card, "Key concepts" (MXFP8 weights pre-quantised with ops.mxfp8_quantize).
 *
 * The pages do not say which tensors are quantised where.  Reading used here (both sides):
 *   forward   x quantised along H; Wg, Wu pre-quantised along H; a = silu(g) u computed from the
 *             fp64 g, u and quantised along I; Wd pre-quantised along I.
 *   dgrad     dY quantised along H with Wd pre-quantised along H (a copy of Wd^T quantised per
 *             row); dS = <dA', a_q>; dg, du (fp64, from the unquantised g, u) quantised along I
 *             with Wg, Wu pre-quantised along I (copies of Wg^T, Wu^T).
 *   wgrad     each operand quantised along the wgrad's own K, the routed rows: per expert, its
 *             rows in the expert-grouped order (ascending slot, padded with zero rows to a
 *             multiple of 128) are cut into blocks of 32 rows, and every column of a block is one
 *             MX block.  dWg = sum Qr(dg) Qr(x)^T, dWu likewise with du, dWd = sum Qr(dY)
 *             Qr(s a)^T, from the unquantised dg, du (fp64), x, dY (bf16) and a = silu(g) u
 *             (fp64, before its quantisation along I).
 * One MX block = 32 consecutive values along the quantised axis: shared = floor(log2 amax) - 8
 * clamped to [-127, 127], element = E4M3 RNE of v / 2^shared saturating to +-448, and the value
 * used is element * 2^shared.  All other arithmetic is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

double orc_bf16_value(uint16_t b);
double orc_e4m3_value(uint8_t c);
uint8_t orc_e4m3_encode(double v);

/* Pin switch for tests: 0 turns every MX quantise-dequantise into the identity, so the MX dataflow
 * can be compared with the BF16 oracle on inputs that are already on the MX grid. */
static int g_mx_quant = 1;
void orc_mx_set_quant(int on) { g_mx_quant = on; }

/* MX quantise-dequantise of n values in place, in blocks of 32 (n a multiple of 32). */
void orc_mx_fakequant(double *v, int64_t n) {
    if (!g_mx_quant) return;
    for (int64_t b = 0; b < n; b += 32) {
        double amax = 0.0;
        for (int i = 0; i < 32; ++i)
            if (fabs(v[b + i]) > amax) amax = fabs(v[b + i]);
        int shared = -127;
        if (amax > 0.0) {
            int ex;
            frexp(amax, &ex);
            shared = ex - 1 - 8;
            if (shared < -127) shared = -127;
            if (shared > 127) shared = 127;
        }
        for (int i = 0; i < 32; ++i)
            v[b + i] = ldexp(orc_e4m3_value(orc_e4m3_encode(ldexp(v[b + i], -shared))), shared);
    }
}

typedef struct {
    int64_t T;
    int32_t H, I, E, K;
    const int32_t *ids;
    const float *s;
    const uint16_t *x, *dY;
    /* pre-quantised weights: bytes [rows, cols] + scales [rows, cols/32] */
    const uint8_t *qg, *sg, *qu, *su; /* Wg, Wu as [E*I, H], along H */
    const uint8_t *qd, *sd;           /* Wd as [E*H, I], along I */
    const uint8_t *qgt, *sgt, *qut, *sut; /* Wg^T, Wu^T as [E*H, I], along I */
    const uint8_t *qdt, *sdt;             /* Wd^T as [E*I, H], along H */
    double e4[256], sc[256];
} mxl_t;

static void mxl_tables(mxl_t *M) {
    for (int c = 0; c < 256; ++c) {
        M->e4[c] = orc_e4m3_value((uint8_t)c);
        M->sc[c] = c == 255 ? NAN : ldexp(1.0, c - 127);
    }
}

/* decoded weight element (row, col) of a [rows, cols] MXFP8 matrix */
static inline double mxw(const mxl_t *M, const uint8_t *q, const uint8_t *s, int64_t row, int64_t col,
                         int64_t cols) {
    return M->e4[q[row * cols + col]] * M->sc[s[row * (cols / 32) + col / 32]];
}

/* x_q[t] (length H) */
static void xq_row(const mxl_t *M, const uint16_t *src, int64_t t, double *out) {
    for (int64_t h = 0; h < M->H; ++h) out[h] = orc_bf16_value(src[t * M->H + h]);
    orc_mx_fakequant(out, M->H);
}

static double sigm(double z) { return 1.0 / (1.0 + exp(-z)); }

/* one slot, columns [i0, i0 + n) of I: g, u, a (unquantised) from x_q */
static void mx_up_cols(const mxl_t *M, int32_t e, const double *xq, int64_t i0, int64_t n, double *g, double *u,
                       double *a) {
    const int64_t H = M->H, I = M->I;
    for (int64_t ii = 0; ii < n; ++ii) {
        const int64_t i = i0 + ii;
        double sg = 0.0, su = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            sg += mxw(M, M->qg, M->sg, (int64_t)e * I + i, h, H) * xq[h];
            su += mxw(M, M->qu, M->su, (int64_t)e * I + i, h, H) * xq[h];
        }
        g[ii] = sg;
        u[ii] = su;
        a[ii] = sg * sigm(sg) * su;
    }
}

/* dA'[i] for columns [i0, i0 + n): sum_h Wd_b[e, h, i] dY_q[h] */
static void mx_dap_cols(const mxl_t *M, int32_t e, const double *dyq, int64_t i0, int64_t n, double *dap) {
    const int64_t H = M->H, I = M->I;
    for (int64_t ii = 0; ii < n; ++ii) {
        const int64_t i = i0 + ii;
        double acc = 0.0;
        for (int64_t h = 0; h < H; ++h) acc += mxw(M, M->qdt, M->sdt, (int64_t)e * I + i, h, H) * dyq[h];
        dap[ii] = acc;
    }
}

/* per-slot quantities of one slot j */
typedef struct {
    double *g, *u, *a, *aq, *dap, *dg, *du, *dgq, *duq; /* length I */
    double *y;                                          /* length H */
} slotbuf_t;

static slotbuf_t slot_alloc(int64_t H, int64_t I) {
    slotbuf_t b;
    b.g = malloc(sizeof(double) * I);
    b.u = malloc(sizeof(double) * I);
    b.a = malloc(sizeof(double) * I);
    b.aq = malloc(sizeof(double) * I);
    b.dap = malloc(sizeof(double) * I);
    b.dg = malloc(sizeof(double) * I);
    b.du = malloc(sizeof(double) * I);
    b.dgq = malloc(sizeof(double) * I);
    b.duq = malloc(sizeof(double) * I);
    b.y = malloc(sizeof(double) * H);
    return b;
}
static void slot_free(slotbuf_t *b) {
    free(b->g); free(b->u); free(b->a); free(b->aq); free(b->dap); free(b->dg); free(b->du); free(b->dgq);
    free(b->duq); free(b->y);
}

/* forward of slot j: g, u, a_q, y */
static void mx_slot_fwd(const mxl_t *M, int64_t j, const double *xq, slotbuf_t *b) {
    const int64_t H = M->H, I = M->I;
    const int32_t e = M->ids[j];
    mx_up_cols(M, e, xq, 0, I, b->g, b->u, b->a);
    memcpy(b->aq, b->a, sizeof(double) * I);
    orc_mx_fakequant(b->aq, I);
    for (int64_t h = 0; h < H; ++h) {
        double acc = 0.0;
        for (int64_t i = 0; i < I; ++i) acc += mxw(M, M->qd, M->sd, (int64_t)e * H + h, i, I) * b->aq[i];
        b->y[h] = acc;
    }
}

/* backward quantities of slot j (after mx_slot_fwd): dA', dS, dg, du and their quantisations along I */
static double mx_slot_bwd(const mxl_t *M, int64_t j, const double *dyq, slotbuf_t *b) {
    const int64_t I = M->I;
    const int32_t e = M->ids[j];
    mx_dap_cols(M, e, dyq, 0, I, b->dap);
    double ds = 0.0;
    for (int64_t i = 0; i < I; ++i) ds += b->dap[i] * b->aq[i];
    const double sv = (double)M->s[j];
    for (int64_t i = 0; i < I; ++i) {
        const double sg = sigm(b->g[i]), da = sv * b->dap[i];
        b->dg[i] = da * b->u[i] * sg * (1.0 + b->g[i] * (1.0 - sg));
        b->du[i] = da * b->g[i] * sg;
    }
    memcpy(b->dgq, b->dg, sizeof(double) * I);
    memcpy(b->duq, b->du, sizeof(double) * I);
    orc_mx_fakequant(b->dgq, I);
    orc_mx_fakequant(b->duq, I);
    return ds;
}

/* MX quantise-dequantise along rows: every column of a row-major [nrows, ncols] matrix in blocks
 * of 32 consecutive rows (nrows a multiple of 32). */
static void fakequant_cols(double *m, int64_t nrows, int64_t ncols) {
    double blk[32];
    for (int64_t r0 = 0; r0 < nrows; r0 += 32)
        for (int64_t c = 0; c < ncols; ++c) {
            for (int i = 0; i < 32; ++i) blk[i] = m[(r0 + i) * ncols + c];
            orc_mx_fakequant(blk, 32);
            for (int i = 0; i < 32; ++i) m[(r0 + i) * ncols + c] = blk[i];
        }
}

/* The slots of expert e in ascending order; returns their count, *npad = the count rounded up to
 * the 128-row padding of the expert-grouped layout. */
static int64_t expert_slots(const int32_t *ids, int64_t R, int32_t e, int64_t *slots, int64_t *npad) {
    int64_t n = 0;
    for (int64_t j = 0; j < R; ++j)
        if (ids[j] == e) slots[n++] = j;
    *npad = (n + 127) / 128 * 128;
    return n;
}

static mxl_t make_mx(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const int32_t *ids, const float *s,
                     const uint16_t *x, const uint16_t *dY, const uint8_t *const *w) {
    mxl_t M;
    memset(&M, 0, sizeof M);
    M.T = T; M.H = H; M.I = I; M.E = E; M.K = K;
    M.ids = ids; M.s = s; M.x = x; M.dY = dY;
    M.qg = w[0]; M.sg = w[1]; M.qu = w[2]; M.su = w[3]; M.qd = w[4]; M.sd = w[5];
    M.qgt = w[6]; M.sgt = w[7]; M.qut = w[8]; M.sut = w[9]; M.qdt = w[10]; M.sdt = w[11];
    mxl_tables(&M);
    return M;
}

/* Full MXFP8 forward + backward (small shapes).  w = the 12 weight arrays in mxl_t order.
 * out [T,H]; dX [T,H]; dWg, dWu [E,I,H]; dWd [E,H,I]; dS [T,K]; optional a_q [R,I], and the
 * unquantised dg, du, a [R,I] (slot order). */
void orc_layer_mx(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const int32_t *ids, const float *s,
                  const uint16_t *x, const uint16_t *dY, const uint8_t *const *w, double *out, double *dX,
                  double *dWg, double *dWu, double *dWd, double *dS, double *aq_out, double *dg_out,
                  double *du_out, double *a_out) {
    mxl_t M = make_mx(T, H, I, E, K, ids, s, x, dY, w);
    const int64_t R = T * (int64_t)K;
    double *XQ = malloc(sizeof(double) * T * H), *DYQ = malloc(sizeof(double) * T * H);
    double *AQ = malloc(sizeof(double) * R * I), *DGQ = malloc(sizeof(double) * R * I);
    double *DUQ = malloc(sizeof(double) * R * I), *Y = malloc(sizeof(double) * R * H);
    double *A = malloc(sizeof(double) * R * I), *DG = malloc(sizeof(double) * R * I);
    double *DU = malloc(sizeof(double) * R * I);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        xq_row(&M, x, t, XQ + t * H);
        xq_row(&M, dY, t, DYQ + t * H);
    }
#pragma omp parallel
    {
        slotbuf_t b = slot_alloc(H, I);
#pragma omp for schedule(dynamic, 1)
        for (int64_t j = 0; j < R; ++j) {
            const int64_t t = j / K;
            mx_slot_fwd(&M, j, XQ + t * H, &b);
            dS[j] = mx_slot_bwd(&M, j, DYQ + t * H, &b);
            memcpy(AQ + j * I, b.aq, sizeof(double) * I);
            memcpy(DGQ + j * I, b.dgq, sizeof(double) * I);
            memcpy(DUQ + j * I, b.duq, sizeof(double) * I);
            memcpy(A + j * I, b.a, sizeof(double) * I);
            memcpy(DG + j * I, b.dg, sizeof(double) * I);
            memcpy(DU + j * I, b.du, sizeof(double) * I);
            memcpy(Y + j * H, b.y, sizeof(double) * H);
        }
        slot_free(&b);
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            out[t * H + h] = 0.0;
            dX[t * H + h] = 0.0;
        }
        for (int32_t k = 0; k < K; ++k) {
            const int64_t j = t * K + k;
            const int32_t e = ids[j];
            for (int64_t h = 0; h < H; ++h) out[t * H + h] += (double)s[j] * Y[j * H + h];
            for (int64_t h = 0; h < H; ++h) {
                double acc = 0.0;
                for (int64_t i = 0; i < I; ++i)
                    acc += mxw(&M, M.qgt, M.sgt, (int64_t)e * H + h, i, I) * DGQ[j * I + i] +
                           mxw(&M, M.qut, M.sut, (int64_t)e * H + h, i, I) * DUQ[j * I + i];
                dX[t * H + h] += acc;
            }
        }
    }
    /* weight gradients, operands quantised along the expert's padded rows */
    int64_t *slots = malloc(sizeof(int64_t) * (R ? R : 1));
    for (int32_t e = 0; e < E; ++e) {
        int64_t npad;
        const int64_t n = expert_slots(ids, R, e, slots, &npad);
        const int64_t np = npad ? npad : 1;
        double *qdg = calloc(np * I, sizeof(double)), *qdu = calloc(np * I, sizeof(double));
        double *qsa = calloc(np * I, sizeof(double)), *qx = calloc(np * H, sizeof(double));
        double *qdy = calloc(np * H, sizeof(double));
        for (int64_t r = 0; r < n; ++r) {
            const int64_t j = slots[r], t = j / K;
            for (int64_t i = 0; i < I; ++i) {
                qdg[r * I + i] = DG[j * I + i];
                qdu[r * I + i] = DU[j * I + i];
                qsa[r * I + i] = (double)s[j] * A[j * I + i];
            }
            for (int64_t h = 0; h < H; ++h) {
                qx[r * H + h] = orc_bf16_value(x[t * H + h]);
                qdy[r * H + h] = orc_bf16_value(dY[t * H + h]);
            }
        }
        fakequant_cols(qdg, npad, I);
        fakequant_cols(qdu, npad, I);
        fakequant_cols(qsa, npad, I);
        fakequant_cols(qx, npad, H);
        fakequant_cols(qdy, npad, H);
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t i = 0; i < I; ++i) {
            double *rg = dWg + ((int64_t)e * I + i) * H, *ru = dWu + ((int64_t)e * I + i) * H;
            for (int64_t h = 0; h < H; ++h) {
                double ag = 0.0, au = 0.0;
                for (int64_t r = 0; r < npad; ++r) {
                    ag += qdg[r * I + i] * qx[r * H + h];
                    au += qdu[r * I + i] * qx[r * H + h];
                }
                rg[h] = ag;
                ru[h] = au;
            }
        }
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t h = 0; h < H; ++h) {
            double *rd = dWd + ((int64_t)e * H + h) * I;
            for (int64_t i = 0; i < I; ++i) {
                double ad = 0.0;
                for (int64_t r = 0; r < npad; ++r) ad += qdy[r * H + h] * qsa[r * I + i];
                rd[i] = ad;
            }
        }
        free(qdg); free(qdu); free(qsa); free(qx); free(qdy);
    }
    free(slots);
    if (dg_out) memcpy(dg_out, DG, sizeof(double) * R * I);
    if (du_out) memcpy(du_out, DU, sizeof(double) * R * I);
    if (a_out) memcpy(a_out, A, sizeof(double) * R * I);
    if (aq_out) memcpy(aq_out, AQ, sizeof(double) * R * I);
    free(XQ); free(DYQ); free(AQ); free(DGQ); free(DUQ); free(Y); free(A); free(DG); free(DU);
}

/* Sampled tokens: out, dX [ntok, H] and dS [ntok, K]. */
void orc_tokens_mx(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const int32_t *ids, const float *s,
                   const uint16_t *x, const uint16_t *dY, const uint8_t *const *w, int64_t ntok, const int64_t *tok,
                   double *out, double *dX, double *dS) {
    mxl_t M = make_mx(T, H, I, E, K, ids, s, x, dY, w);
#pragma omp parallel
    {
        slotbuf_t b = slot_alloc(H, I);
        double *xq = malloc(sizeof(double) * H), *dyq = malloc(sizeof(double) * H);
#pragma omp for schedule(dynamic, 1)
        for (int64_t n = 0; n < ntok; ++n) {
            const int64_t t = tok[n];
            xq_row(&M, x, t, xq);
            xq_row(&M, dY, t, dyq);
            for (int64_t h = 0; h < H; ++h) {
                out[n * H + h] = 0.0;
                dX[n * H + h] = 0.0;
            }
            for (int32_t k = 0; k < K; ++k) {
                const int64_t j = t * K + k;
                const int32_t e = ids[j];
                mx_slot_fwd(&M, j, xq, &b);
                dS[n * K + k] = mx_slot_bwd(&M, j, dyq, &b);
                for (int64_t h = 0; h < H; ++h) {
                    out[n * H + h] += (double)s[j] * b.y[h];
                    double acc = 0.0;
                    for (int64_t i = 0; i < I; ++i)
                        acc += mxw(&M, M.qgt, M.sgt, (int64_t)e * H + h, i, I) * b.dgq[i] +
                               mxw(&M, M.qut, M.sut, (int64_t)e * H + h, i, I) * b.duq[i];
                    dX[n * H + h] += acc;
                }
            }
        }
        slot_free(&b);
        free(xq); free(dyq);
    }
}

/* One 32-column block [i0, i0+32) of I for expert e, against the nh sampled hidden columns hs:
 *   dwg[ii * nh + n] = dWg[e, i0+ii, hs[n]], dwu likewise, dwd[n * 32 + ii] = dWd[e, hs[n], i0+ii].
 * The operands of e's padded rows are quantised along the rows exactly as in orc_layer_mx; every
 * column's row blocks are independent, so the block's 32 columns of dg, du, s a and the sampled
 * columns of x and dY are all the sums need. */
void orc_dw_block_mx(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const int32_t *ids, const float *s,
                     const uint16_t *x, const uint16_t *dY, const uint8_t *const *w, int32_t e, int32_t i0,
                     int64_t nh, const int32_t *hs, double *dwg, double *dwu, double *dwd) {
    mxl_t M = make_mx(T, H, I, E, K, ids, s, x, dY, w);
    const int64_t R = T * (int64_t)K;
    int64_t *slots = malloc(sizeof(int64_t) * (R ? R : 1));
    int64_t npad;
    const int64_t nslots = expert_slots(ids, R, e, slots, &npad);
    const int64_t np = npad ? npad : 1;
    double *DG = calloc(np * 32, sizeof(double)), *DU = calloc(np * 32, sizeof(double));
    double *SA = calloc(np * 32, sizeof(double));
    double *XS = calloc(np * (nh ? nh : 1), sizeof(double)), *DYS = calloc(np * (nh ? nh : 1), sizeof(double));
#pragma omp parallel
    {
        double *xq = malloc(sizeof(double) * H), *dyq = malloc(sizeof(double) * H);
        double g[32], u[32], a[32], dap[32];
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nslots; ++r) {
            const int64_t j = slots[r], t = j / K;
            xq_row(&M, x, t, xq);
            xq_row(&M, dY, t, dyq);
            mx_up_cols(&M, e, xq, i0, 32, g, u, a);
            mx_dap_cols(&M, e, dyq, i0, 32, dap);
            const double sv = (double)s[j];
            for (int ii = 0; ii < 32; ++ii) {
                const double sg = sigm(g[ii]), da = sv * dap[ii];
                DG[r * 32 + ii] = da * u[ii] * sg * (1.0 + g[ii] * (1.0 - sg));
                DU[r * 32 + ii] = da * g[ii] * sg;
                SA[r * 32 + ii] = sv * a[ii];
            }
            for (int64_t n = 0; n < nh; ++n) {
                XS[r * nh + n] = orc_bf16_value(x[t * H + hs[n]]);
                DYS[r * nh + n] = orc_bf16_value(dY[t * H + hs[n]]);
            }
        }
        free(xq); free(dyq);
    }
    fakequant_cols(DG, npad, 32);
    fakequant_cols(DU, npad, 32);
    fakequant_cols(SA, npad, 32);
    fakequant_cols(XS, npad, nh);
    fakequant_cols(DYS, npad, nh);
    for (int ii = 0; ii < 32; ++ii)
        for (int64_t n = 0; n < nh; ++n) {
            double ag = 0.0, au = 0.0, ad = 0.0;
            for (int64_t r = 0; r < npad; ++r) {
                ag += DG[r * 32 + ii] * XS[r * nh + n];
                au += DU[r * 32 + ii] * XS[r * nh + n];
                ad += DYS[r * nh + n] * SA[r * 32 + ii];
            }
            dwg[ii * nh + n] = ag;
            dwu[ii * nh + n] = au;
            dwd[n * 32 + ii] = ad;
        }
    free(slots); free(DG); free(DU); free(SA); free(XS); free(DYS);
}
