/*
 * mok_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU oracle of the deterministic top-k routed SwiGLU expert layer
 * (Mixture-of-Kittens, collapsed to one GPU).  Only tests/, __graft_entry__.smoke() and
 * bench.py's CPU-baseline / reference arm may load this library; the CUDA product path never
 * does, and the two share no code, headers, tables or helpers.
 *
 * Sources followed (page title + section):
 *  [MTP]  "Cursor Open-Sources Mixture-of-Kittens (MoK): A Deterministic MoE Training Megakernel
 *          for GB300 NVL72 Racks" (yifor-blog digest of MarkTechPost), English summary:
 *          BF16 and MXFP8 modes, forward and backward, SwiGLU experts, router-weight gradient
 *          computed SonicMoE-style inside the SwiGLU backward, fully deterministic.
 *  [ATT]  "Mixture-of-Kittens(MoK)란? Cursor의 결정론적 MoE 메가커널 완전 정리" (alltoptrend),
 *          section 4 (1): one schedule table drives dispatch and combine, forward and backward;
 *          section 4 (3): no token is ever dropped, minibatch / macrobatch granularity.
 *  [ALH]  "Mixture-of-Kittens (MoK)" project card (agentlenshq), "Functional API" block
 *          (build_schedule takes the top-k expert ids) and "Key concepts" table (MoKConfig knobs:
 *          minibatch granularity, macrobatch size; MXFP8 weights pre-quantised by
 *          ops.mxfp8_quantize).
 *
 * The pages print no formula.  Where they leave a step open this file takes the plainest
 * standard reading (each reading is listed with the functions below):
 *   - SwiGLU expert: a = silu(g) * u, g = Wg x, u = Wu x, y = Wd a, no bias, no clamp.
 *   - combine: out[t] = sum over k ascending of s[t,k] * y(t,k); the weight is applied after the
 *     down projection.
 *   - router-weight gradient: dS[t,k] = <dY[t], y(t,k)> = <Wd^T dY[t], a(t,k)>.
 *   - schedule: counting sort of flat slots j = t*K + k by expert id, stable in j, experts in
 *     ascending id, each expert's segment padded to a multiple of the GEMM row tile Mt.
 *   - MXFP8: OCP MX E4M3 elements with one E8M0 scale per 32 consecutive values.
 *
 * All arithmetic is fp64; bf16 and E4M3 inputs enter as their exact values.  The layer loops
 * (expert_up .. orc_backward) take their arithmetic type from ORC_REAL (default double): a second
 * build with ORC_REAL=float serves only as the timed fp32 CPU baseline, never as a reference.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORC_REAL
#define ORC_REAL double
#endif
typedef ORC_REAL real;
/* exp in the arithmetic type of the layer loops */
static inline real real_exp(real z) { return sizeof(real) == sizeof(float) ? (real)expf((float)z) : (real)exp((double)z); }

/* ------------------------------------------------------------------------------------------ */
/* number formats                                                                              */
/* ------------------------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32; its value is exact in double. */
double orc_bf16_value(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3 ("fn"): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.
 * Exponent field 0 is subnormal: (m/8) * 2^-6.  Otherwise (1 + m/8) * 2^(E-7).
 * S.1111.111 is NaN; there is no infinity; the largest finite magnitude is 448 (0x7E). */
double orc_e4m3_value(uint8_t c) {
    int s = (c >> 7) & 1, E = (c >> 3) & 15, m = c & 7;
    double v;
    if (E == 15 && m == 7) return NAN;
    if (E == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, E - 7);
    return s ? -v : v;
}

/* Round-to-nearest-even onto the E4M3 grid, saturating to +-448 (satfinite reading).
 * The 127 non-negative finite codes 0x00..0x7E have increasing values; bisection finds the code c
 * with value(c) <= |v| < value(c + 1), then the nearer of the two wins, and on an exact tie the
 * code with the even mantissa (even code).  NaN maps to 0x7F. */
uint8_t orc_e4m3_encode(double v) {
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    int lo = 0, hi = 0x7E; /* value(lo) <= a < value(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (orc_e4m3_value((uint8_t)mid) <= a) lo = mid;
        else hi = mid;
    }
    double dlo = a - orc_e4m3_value((uint8_t)lo), dhi = orc_e4m3_value((uint8_t)hi) - a;
    int best = (dlo < dhi || (dlo == dhi && (lo & 1) == 0)) ? lo : hi;
    return (uint8_t)(sign | best);
}

/* E8M0 scale byte: the value is 2^(byte - 127); 0xFF is NaN. */
double orc_e8m0_value(uint8_t b) {
    if (b == 0xFF) return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* MXFP8 quantisation of a row-major bf16 matrix [rows, cols] into E4M3 bytes [rows, cols] and
 * E8M0 scales [rows, cols/32], one scale per 32 consecutive elements of a row ([ALH] Key
 * concepts, "MXFP8": ops.mxfp8_quantize; [MTP] English summary, MXFP8 mode).
 * Per block (reading of the OCP MX rule):
 *   amax = max |v|; shared = floor(log2(amax)) - 8 (8 = exponent of E4M3's largest normal),
 *   clamped to [-127, 127]; amax == 0 gives shared = -127 (scale byte 0).
 *   element = RNE(v / 2^shared) on the E4M3 grid, saturating to +-448.
 *   A block holding NaN or +-Inf gets scale 0xFF and every element 0x7F.
 * Returns 0, or 1 when cols is not a multiple of 32. */
int orc_mxfp8_quantize(const uint16_t *in, int64_t rows, int64_t cols, uint8_t *q, uint8_t *scale) {
    if (cols % 32 != 0) return 1;
    int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const uint16_t *blk = in + r * cols + b * 32;
            double amax = 0.0;
            int bad = 0;
            for (int i = 0; i < 32; ++i) {
                double v = orc_bf16_value(blk[i]);
                if (!isfinite(v)) bad = 1;
                else if (fabs(v) > amax) amax = fabs(v);
            }
            uint8_t *qo = q + r * cols + b * 32;
            if (bad) {
                scale[r * nb + b] = 0xFF;
                for (int i = 0; i < 32; ++i) qo[i] = 0x7F;
                continue;
            }
            int shared;
            if (amax == 0.0) {
                shared = -127;
            } else {
                int ex;
                frexp(amax, &ex); /* amax = f * 2^ex, f in [0.5, 1): floor(log2 amax) = ex - 1 */
                shared = (ex - 1) - 8;
                if (shared < -127) shared = -127;
                if (shared > 127) shared = 127;
            }
            scale[r * nb + b] = (uint8_t)(shared + 127);
            for (int i = 0; i < 32; ++i) qo[i] = orc_e4m3_encode(ldexp(orc_bf16_value(blk[i]), -shared));
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* schedule ([ATT] section 4 (1) and (3); [ALH] Functional API: build_schedule(topk_experts))  */
/* ------------------------------------------------------------------------------------------ */

/* Upper bound of the padded row count: every expert wastes at most Mt - 1 rows. */
int64_t orc_rpad_max(int64_t T, int32_t K, int32_t E, int32_t Mt) {
    return T * (int64_t)K + (int64_t)E * (Mt - 1);
}

/* The schedule of R = T*K routed slots (slot j = t*K + k carries expert ids[j]):
 *   counts[e]   = #{ j : ids[j] == e }
 *   offsets[e]  = sum_{e' < e} counts[e']                          (E+1 entries)
 *   poff[e]     = sum_{e' < e} ceil(counts[e'] / Mt) * Mt          (E+1 entries; Rpad = poff[E])
 *   perm[row]   = the q-th slot (ascending j) of expert e for row = poff[e] + q, q < counts[e];
 *                 -1 on the padding rows poff[e] + counts[e] .. poff[e+1]-1
 *   inv[j]      = the row with perm[row] == j
 *   tiles       = minibatch tiles {expert, first row, valid rows, macrobatch id}: per expert in
 *                 ascending id, its slots cut into runs of mb rows starting at poff[e]; the last
 *                 run may be short; tiles never cross experts; macro id = first row / MB.
 *   mblocks     = one entry per Mt-row block of the padded layout {expert, first row,
 *                 valid rows, index of the minibatch tile holding it}.
 * No slot is ever dropped.  Returns 0; 1 when an id is outside [0, E); 2 when a capacity given
 * by the caller is too small. */
int orc_schedule(int64_t T, int32_t K, int32_t E, const int32_t *ids, int32_t Mt, int32_t mb, int32_t MB,
                 int32_t *counts, int32_t *offsets, int32_t *poff, int32_t *perm, int64_t perm_cap,
                 int32_t *inv, int32_t *tiles, int64_t tiles_cap, int64_t *ntiles, int32_t *mblocks,
                 int64_t mblocks_cap, int64_t *nmblocks, int64_t *rpad) {
    int64_t R = T * (int64_t)K;
    for (int64_t j = 0; j < R; ++j)
        if (ids[j] < 0 || ids[j] >= E) return 1;
    for (int32_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t j = 0; j < R; ++j) counts[ids[j]] += 1;
    offsets[0] = 0;
    poff[0] = 0;
    for (int32_t e = 0; e < E; ++e) {
        offsets[e + 1] = offsets[e] + counts[e];
        int32_t padded = (counts[e] + Mt - 1) / Mt * Mt;
        poff[e + 1] = poff[e] + padded;
    }
    int64_t Rp = poff[E];
    if (Rp > perm_cap) return 2;
    *rpad = Rp;
    /* stable counting sort: for each expert, walk the slots in ascending j */
    for (int32_t e = 0; e < E; ++e) {
        int64_t row = poff[e];
        for (int64_t j = 0; j < R; ++j) {
            if (ids[j] == e) {
                perm[row] = (int32_t)j;
                inv[j] = (int32_t)row;
                ++row;
            }
        }
        for (; row < poff[e + 1]; ++row) perm[row] = -1;
    }
    /* minibatch tiles */
    int64_t nt = 0;
    for (int32_t e = 0; e < E; ++e) {
        for (int32_t q = 0; q < counts[e]; q += mb) {
            if (nt >= tiles_cap) return 2;
            int32_t first = poff[e] + q;
            int32_t valid = counts[e] - q < mb ? counts[e] - q : mb;
            tiles[4 * nt + 0] = e;
            tiles[4 * nt + 1] = first;
            tiles[4 * nt + 2] = valid;
            tiles[4 * nt + 3] = first / MB;
            ++nt;
        }
    }
    *ntiles = nt;
    /* Mt-row blocks of the padded layout */
    int64_t nb = Rp / Mt;
    if (nb > mblocks_cap) return 2;
    for (int64_t b = 0; b < nb; ++b) {
        int32_t first = (int32_t)(b * Mt);
        int32_t e = 0;
        while (!(poff[e] <= first && first < poff[e + 1])) ++e;
        int32_t within = first - poff[e];
        int32_t valid = counts[e] - within < Mt ? counts[e] - within : Mt;
        int32_t tile = -1;
        for (int64_t i = 0; i < nt; ++i) {
            int32_t t0 = tiles[4 * i + 1];
            int32_t span = (tiles[4 * i + 2] + Mt - 1) / Mt * Mt;
            if (tiles[4 * i + 0] == e && t0 <= first && first < t0 + span) {
                tile = (int32_t)i;
                break;
            }
        }
        mblocks[4 * b + 0] = e;
        mblocks[4 * b + 1] = first;
        mblocks[4 * b + 2] = valid;
        mblocks[4 * b + 3] = tile;
    }
    *nmblocks = nb;
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* the SwiGLU expert, one routed slot at a time ([MTP] English summary: SwiGLU experts)        */
/* ------------------------------------------------------------------------------------------ */

static real sigmoid_r(real z) { return (real)1 / ((real)1 + real_exp(-z)); }
/* a bf16 value in the arithmetic type (exact in either) */
static inline real bf16r(uint16_t b) { return (real)orc_bf16_value(b); }
static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

typedef struct {
    int64_t T;
    int32_t H, I, E, K;
    const int32_t *ids;   /* [T, K] */
    const float *s;       /* [T, K] renormalised top-k weights */
    const uint16_t *x;    /* [T, H] bf16 */
    const uint16_t *Wg;   /* [E, I, H] bf16 (PyTorch [out, in]) */
    const uint16_t *Wu;   /* [E, I, H] bf16 */
    const uint16_t *Wd;   /* [E, H, I] bf16 */
    const uint16_t *dY;   /* [T, H] bf16, may be NULL for forward only */
} layer_t;

/* g = Wg[e] x[t], u = Wu[e] x[t] (length I), a = silu(g) * u. */
static void expert_up(const layer_t *L, int32_t e, int64_t t, real *g, real *u, real *a) {
    const int64_t H = L->H, I = L->I;
    const uint16_t *xt = L->x + t * H;
    for (int64_t i = 0; i < I; ++i) {
        const uint16_t *wg = L->Wg + ((int64_t)e * I + i) * H;
        const uint16_t *wu = L->Wu + ((int64_t)e * I + i) * H;
        real sg = (real)0, su = (real)0;
        for (int64_t h = 0; h < H; ++h) {
            real xv = bf16r(xt[h]);
            sg += bf16r(wg[h]) * xv;
            su += bf16r(wu[h]) * xv;
        }
        g[i] = sg;
        u[i] = su;
        a[i] = sg * sigmoid_r(sg) * su;
    }
}

/* y = Wd[e] a (length H). */
static void expert_down(const layer_t *L, int32_t e, const real *a, real *y) {
    const int64_t H = L->H, I = L->I;
    for (int64_t h = 0; h < H; ++h) {
        const uint16_t *wd = L->Wd + ((int64_t)e * H + h) * I;
        real acc = (real)0;
        for (int64_t i = 0; i < I; ++i) acc += bf16r(wd[i]) * a[i];
        y[h] = acc;
    }
}

/* dA' = Wd[e]^T dY[t] (length I). */
static void expert_down_t(const layer_t *L, int32_t e, int64_t t, real *dap) {
    const int64_t H = L->H, I = L->I;
    const uint16_t *dy = L->dY + t * H;
    for (int64_t i = 0; i < I; ++i) dap[i] = (real)0;
    for (int64_t h = 0; h < H; ++h) {
        real d = bf16r(dy[h]);
        const uint16_t *wd = L->Wd + ((int64_t)e * H + h) * I;
        for (int64_t i = 0; i < I; ++i) dap[i] += bf16r(wd[i]) * d;
    }
}

/* SwiGLU backward for one slot with combine weight sv:
 *   dA = sv * dA';  dg = dA * u * sig(g) * (1 + g (1 - sig(g)));  du = dA * g * sig(g). */
static void swiglu_bwd(int64_t I, real sv, const real *g, const real *u, const real *dap, real *dg,
                       real *du) {
    for (int64_t i = 0; i < I; ++i) {
        real sg = sigmoid_r(g[i]);
        real da = sv * dap[i];
        dg[i] = da * u[i] * sg * ((real)1 + g[i] * ((real)1 - sg));
        du[i] = da * g[i] * sg;
    }
}

static layer_t make_layer(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const int32_t *ids, const float *s,
                          const uint16_t *x, const uint16_t *Wg, const uint16_t *Wu, const uint16_t *Wd,
                          const uint16_t *dY) {
    layer_t L = {T, H, I, E, K, ids, s, x, Wg, Wu, Wd, dY};
    return L;
}

/* Forward of the whole layer.
 *   out[t] = sum_{k = 0..K-1, ascending} s[t,k] * Wd[e] (silu(Wg[e] x[t]) * (Wu[e] x[t])),  e = ids[t,k]
 * Optional per-slot intermediates (slot order j = t*K + k): g, u, a [R, I]; y [R, H]; pass NULL
 * to skip.  [MTP] English summary (SwiGLU experts, forward); [ATT] section 4 (1) (combine). */
void orc_forward(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const int32_t *ids, const float *s,
                 const uint16_t *x, const uint16_t *Wg, const uint16_t *Wu, const uint16_t *Wd, real *out, real *g,
                 real *u, real *a, real *y) {
    layer_t L = make_layer(T, H, I, E, K, ids, s, x, Wg, Wu, Wd, NULL);
#pragma omp parallel
    {
        real *gb = malloc(sizeof(real) * I), *ub = malloc(sizeof(real) * I), *ab = malloc(sizeof(real) * I);
        real *yb = malloc(sizeof(real) * H);
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
            real *o = out + t * H;
            for (int64_t h = 0; h < H; ++h) o[h] = (real)0;
            for (int32_t k = 0; k < K; ++k) {
                int64_t j = t * K + k;
                int32_t e = ids[j];
                expert_up(&L, e, t, gb, ub, ab);
                expert_down(&L, e, ab, yb);
                real sv = (real)s[j];
                for (int64_t h = 0; h < H; ++h) o[h] += sv * yb[h];
                if (g) memcpy(g + j * I, gb, sizeof(real) * I);
                if (u) memcpy(u + j * I, ub, sizeof(real) * I);
                if (a) memcpy(a + j * I, ab, sizeof(real) * I);
                if (y) memcpy(y + j * H, yb, sizeof(real) * H);
            }
        }
        free(gb); free(ub); free(ab); free(yb);
    }
}

/* Backward of the whole layer for upstream gradient dY = dL/dout.
 *   dS[t,k]  = <Wd[e]^T dY[t], a>       (router-weight gradient inside the SwiGLU backward,
 *                                          [MTP] English summary "SonicMoE-style")
 *   dScheck  = <dY[t], Wd[e] a>          (the same number, computed the other way round)
 *   dX[t]    = sum_k (Wg[e]^T dg + Wu[e]^T du)
 *   dWg[e]   = sum over e's slots of dg (x)^T,  dWu[e] likewise with du,
 *   dWd[e]   = sum over e's slots of (s * dY[t]) a^T
 * with dA = s * Wd[e]^T dY[t], dg, du as in swiglu_bwd.  Experts with no slot get dW = 0.
 * dW sums run over each expert's slots in ascending slot order. */
void orc_backward(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const int32_t *ids, const float *s,
                  const uint16_t *x, const uint16_t *Wg, const uint16_t *Wu, const uint16_t *Wd, const uint16_t *dY,
                  real *dX, real *dWg, real *dWu, real *dWd, real *dS, real *dScheck) {
    layer_t L = make_layer(T, H, I, E, K, ids, s, x, Wg, Wu, Wd, dY);
    const int64_t R = T * (int64_t)K;
    real *G = malloc(sizeof(real) * R * I), *U = malloc(sizeof(real) * R * I);
    real *A = malloc(sizeof(real) * R * I), *DG = malloc(sizeof(real) * R * I);
    real *DU = malloc(sizeof(real) * R * I);
    /* per-slot quantities */
#pragma omp parallel
    {
        real *dap = malloc(sizeof(real) * I), *yb = malloc(sizeof(real) * H);
#pragma omp for schedule(dynamic, 1)
        for (int64_t j = 0; j < R; ++j) {
            int64_t t = j / K;
            int32_t e = ids[j];
            expert_up(&L, e, t, G + j * I, U + j * I, A + j * I);
            expert_down_t(&L, e, t, dap);
            real acc = (real)0;
            for (int64_t i = 0; i < I; ++i) acc += dap[i] * A[j * I + i];
            dS[j] = acc;
            if (dScheck) {
                expert_down(&L, e, A + j * I, yb);
                real c = (real)0;
                for (int64_t h = 0; h < H; ++h) c += bf16r(dY[t * H + h]) * yb[h];
                dScheck[j] = c;
            }
            swiglu_bwd(I, (real)s[j], G + j * I, U + j * I, dap, DG + j * I, DU + j * I);
        }
        free(dap); free(yb);
    }
    /* dX per token, k ascending */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        real *d = dX + t * H;
        for (int64_t h = 0; h < H; ++h) d[h] = (real)0;
        for (int32_t k = 0; k < K; ++k) {
            int64_t j = t * K + k;
            int32_t e = ids[j];
            for (int64_t i = 0; i < I; ++i) {
                const uint16_t *wg = Wg + ((int64_t)e * I + i) * H;
                const uint16_t *wu = Wu + ((int64_t)e * I + i) * H;
                real cg = DG[j * I + i], cu = DU[j * I + i];
                for (int64_t h = 0; h < H; ++h) d[h] += bf16r(wg[h]) * cg + bf16r(wu[h]) * cu;
            }
        }
    }
    /* dW per expert row, slots ascending */
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int32_t e = 0; e < E; ++e) {
        for (int64_t i = 0; i < I; ++i) {
            real *rg = dWg + ((int64_t)e * I + i) * H, *ru = dWu + ((int64_t)e * I + i) * H;
            for (int64_t h = 0; h < H; ++h) { rg[h] = (real)0; ru[h] = (real)0; }
            for (int64_t j = 0; j < R; ++j) {
                if (ids[j] != e) continue;
                const uint16_t *xt = x + (j / K) * H;
                real cg = DG[j * I + i], cu = DU[j * I + i];
                for (int64_t h = 0; h < H; ++h) {
                    real xv = bf16r(xt[h]);
                    rg[h] += cg * xv;
                    ru[h] += cu * xv;
                }
            }
        }
    }
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int32_t e = 0; e < E; ++e) {
        for (int64_t h = 0; h < H; ++h) {
            real *rd = dWd + ((int64_t)e * H + h) * I;
            for (int64_t i = 0; i < I; ++i) rd[i] = (real)0;
            for (int64_t j = 0; j < R; ++j) {
                if (ids[j] != e) continue;
                real c = (real)s[j] * bf16r(dY[(j / K) * H + h]);
                for (int64_t i = 0; i < I; ++i) rd[i] += c * A[j * I + i];
            }
        }
    }
    free(G); free(U); free(A); free(DG); free(DU);
}

#ifndef ORC_TIMING_ONLY
/* ------------------------------------------------------------------------------------------ */
/* sampled outputs for full-size checks: the same definitions, one output at a time             */
/* ------------------------------------------------------------------------------------------ */

/* out[tok[n]] for n < ntok (rows of H). */
void orc_forward_tokens(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const int32_t *ids, const float *s,
                        const uint16_t *x, const uint16_t *Wg, const uint16_t *Wu, const uint16_t *Wd, int64_t ntok,
                        const int64_t *tok, double *out) {
    layer_t L = make_layer(T, H, I, E, K, ids, s, x, Wg, Wu, Wd, NULL);
#pragma omp parallel
    {
        double *gb = malloc(sizeof(double) * I), *ub = malloc(sizeof(double) * I), *ab = malloc(sizeof(double) * I);
        double *yb = malloc(sizeof(double) * H);
#pragma omp for schedule(dynamic, 1)
        for (int64_t n = 0; n < ntok; ++n) {
            int64_t t = tok[n];
            double *o = out + n * H;
            for (int64_t h = 0; h < H; ++h) o[h] = 0.0;
            for (int32_t k = 0; k < K; ++k) {
                int32_t e = ids[t * K + k];
                expert_up(&L, e, t, gb, ub, ab);
                expert_down(&L, e, ab, yb);
                double sv = (double)s[t * K + k];
                for (int64_t h = 0; h < H; ++h) o[h] += sv * yb[h];
            }
        }
        free(gb); free(ub); free(ab); free(yb);
    }
}

/* dX[tok[n]] (rows of H) and dS[tok[n], :] (rows of K). */
void orc_backward_tokens(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const int32_t *ids, const float *s,
                         const uint16_t *x, const uint16_t *Wg, const uint16_t *Wu, const uint16_t *Wd,
                         const uint16_t *dY, int64_t ntok, const int64_t *tok, double *dX, double *dS) {
    layer_t L = make_layer(T, H, I, E, K, ids, s, x, Wg, Wu, Wd, dY);
#pragma omp parallel
    {
        double *gb = malloc(sizeof(double) * I), *ub = malloc(sizeof(double) * I), *ab = malloc(sizeof(double) * I);
        double *dap = malloc(sizeof(double) * I), *dg = malloc(sizeof(double) * I), *du = malloc(sizeof(double) * I);
#pragma omp for schedule(dynamic, 1)
        for (int64_t n = 0; n < ntok; ++n) {
            int64_t t = tok[n];
            double *d = dX + n * H;
            for (int64_t h = 0; h < H; ++h) d[h] = 0.0;
            for (int32_t k = 0; k < K; ++k) {
                int64_t j = t * K + k;
                int32_t e = ids[j];
                expert_up(&L, e, t, gb, ub, ab);
                expert_down_t(&L, e, t, dap);
                double acc = 0.0;
                for (int64_t i = 0; i < I; ++i) acc += dap[i] * ab[i];
                dS[n * K + k] = acc;
                swiglu_bwd(I, (double)s[j], gb, ub, dap, dg, du);
                for (int64_t i = 0; i < I; ++i) {
                    const uint16_t *wg = Wg + ((int64_t)e * I + i) * H;
                    const uint16_t *wu = Wu + ((int64_t)e * I + i) * H;
                    for (int64_t h = 0; h < H; ++h) d[h] += orc_bf16_value(wg[h]) * dg[i] + orc_bf16_value(wu[h]) * du[i];
                }
            }
        }
        free(gb); free(ub); free(ab); free(dap); free(dg); free(du);
    }
}

/* Single weight-gradient entries.  which[n] = 0: dWg[e][m][c] (m < I, c < H); 1: dWu[e][m][c];
 * 2: dWd[e][m][c] (m < H, c < I).  Each is the sum over e's slots in ascending slot order. */
void orc_dw_entries(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const int32_t *ids, const float *s,
                    const uint16_t *x, const uint16_t *Wg, const uint16_t *Wu, const uint16_t *Wd, const uint16_t *dY,
                    int64_t n_entries, const int32_t *which, const int32_t *ent_e, const int32_t *ent_m,
                    const int32_t *ent_c, double *val) {
    const int64_t R = T * (int64_t)K;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t n = 0; n < n_entries; ++n) {
        int32_t w = which[n], e = ent_e[n], m = ent_m[n], c = ent_c[n];
        int32_t icol = (w == 2) ? c : m; /* the intermediate column involved */
        double acc = 0.0;
        for (int64_t j = 0; j < R; ++j) {
            if (ids[j] != e) continue;
            int64_t t = j / K;
            /* g, u at column icol */
            const uint16_t *xt = x + t * H;
            const uint16_t *wg = Wg + ((int64_t)e * I + icol) * H;
            const uint16_t *wu = Wu + ((int64_t)e * I + icol) * H;
            double g = 0.0, u = 0.0;
            for (int64_t h = 0; h < H; ++h) {
                double xv = orc_bf16_value(xt[h]);
                g += orc_bf16_value(wg[h]) * xv;
                u += orc_bf16_value(wu[h]) * xv;
            }
            double sg = sigmoid(g);
            if (w == 2) {
                double a = g * sg * u;
                acc += (double)s[j] * orc_bf16_value(dY[t * H + m]) * a;
            } else {
                double dap = 0.0;
                for (int64_t h = 0; h < H; ++h)
                    dap += orc_bf16_value(Wd[((int64_t)e * H + h) * I + icol]) * orc_bf16_value(dY[t * H + h]);
                double da = (double)s[j] * dap;
                double d = (w == 0) ? da * u * sg * (1.0 + g * (1.0 - sg)) : da * g * sg;
                acc += d * orc_bf16_value(xt[c]);
            }
        }
        val[n] = acc;
    }
}

/* One 32-column block [i0, i0+32) of I for expert e, against the nh sampled hidden columns hs:
 *   dwg[ii * nh + n] = dWg[e, i0+ii, hs[n]], dwu likewise, dwd[n * 32 + ii] = dWd[e, hs[n], i0+ii].
 * The same sums as orc_backward ([MTP] English summary: backward of the SwiGLU experts), over the
 * expert's slots in ascending order; each slot's g, u and dA' are needed only on the block's 32
 * columns, so a block costs the expert's rows times 96 H multiply-adds however many hidden columns
 * are sampled. */
void orc_dw_block(int64_t T, int32_t H, int32_t I, int32_t E, int32_t K, const int32_t *ids, const float *s,
                  const uint16_t *x, const uint16_t *Wg, const uint16_t *Wu, const uint16_t *Wd, const uint16_t *dY,
                  int32_t e, int32_t i0, int64_t nh, const int32_t *hs, double *dwg, double *dwu, double *dwd) {
    (void)E;
    const int64_t R = T * (int64_t)K;
    int64_t *slots = malloc(sizeof(int64_t) * (R ? R : 1));
    int64_t n = 0;
    for (int64_t j = 0; j < R; ++j)
        if (ids[j] == e) slots[n++] = j;
    /* per slot: dg, du and s a on the block's 32 columns */
    double *DG = malloc(sizeof(double) * 32 * (n ? n : 1)), *DU = malloc(sizeof(double) * 32 * (n ? n : 1));
    double *SA = malloc(sizeof(double) * 32 * (n ? n : 1));
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < n; ++r) {
        const int64_t j = slots[r], t = j / K;
        const uint16_t *xt = x + t * H, *dy = dY + t * H;
        const double sv = (double)s[j];
        for (int ii = 0; ii < 32; ++ii) {
            const int64_t i = i0 + ii;
            const uint16_t *wg = Wg + ((int64_t)e * I + i) * H, *wu = Wu + ((int64_t)e * I + i) * H;
            double g = 0.0, u = 0.0, dap = 0.0;
            for (int64_t h = 0; h < H; ++h) {
                const double xv = orc_bf16_value(xt[h]);
                g += orc_bf16_value(wg[h]) * xv;
                u += orc_bf16_value(wu[h]) * xv;
                dap += orc_bf16_value(Wd[((int64_t)e * H + h) * I + i]) * orc_bf16_value(dy[h]);
            }
            const double sg = sigmoid(g), da = sv * dap;
            DG[r * 32 + ii] = da * u * sg * (1.0 + g * (1.0 - sg));
            DU[r * 32 + ii] = da * g * sg;
            SA[r * 32 + ii] = sv * g * sg * u;
        }
    }
    for (int ii = 0; ii < 32; ++ii)
        for (int64_t q = 0; q < nh; ++q) {
            double ag = 0.0, au = 0.0, ad = 0.0;
            for (int64_t r = 0; r < n; ++r) {
                const int64_t t = slots[r] / K;
                const double xv = orc_bf16_value(x[t * H + hs[q]]), dv = orc_bf16_value(dY[t * H + hs[q]]);
                ag += DG[r * 32 + ii] * xv;
                au += DU[r * 32 + ii] * xv;
                ad += dv * SA[r * 32 + ii];
            }
            dwg[ii * nh + q] = ag;
            dwu[ii * nh + q] = au;
            dwd[q * 32 + ii] = ad;
        }
    free(slots); free(DG); free(DU); free(SA);
}

#endif /* ORC_TIMING_ONLY */

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
