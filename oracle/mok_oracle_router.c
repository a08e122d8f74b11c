/*
 * mok_oracle_router.c -- TEST INFRASTRUCTURE ONLY.
 *
 * CPU oracle of the router step that precedes the expert layer: logits of a linear router, the
 * top-k experts of its softmax, the renormalised top-k weights, and the backward from the top-k
 * weight gradient to the logits, the router weight, its bias and the layer input.  Only tests/
 * may load it; the CUDA library never does, and the two share no code.
 *
 * Sources (page title + section):
 *  [ALH]  "Mixture-of-Kittens (MoK)" project card (agentlenshq), "Functional API": the layer's
 *         schedule takes the top-k expert ids (and weights) that the router produced.
 *  [MTP]  "Cursor Open-Sources Mixture-of-Kittens (MoK) ..." (yifor-blog digest), English summary:
 *         the router-weight gradient is part of the backward.
 *
 * The pages print no router formula.  Readings (the plainest form the rest supports):
 *   - logits[t,e] = sum_h x[t,h] W[h,e] + b[e], W [H,E], b optional;
 *   - p = softmax over all E experts; the K experts of largest p in descending order, equal p
 *     in ascending expert id; weights w_k = p_k / sum_j p_j over the K selected, which equals
 *     the softmax over the K selected logits (the full denominator cancels);
 *   - backward: with d_k = dL/dw_k, dL/dl_k = w_k (d_k - sum_j w_j d_j) on the selected logits
 *     and 0 on the others; dW[h,e] = sum_t x[t,h] dL/dl[t,e], db[e] = sum_t dL/dl[t,e],
 *     dx[t,h] = sum_e dL/dl[t,e] W[h,e].
 *
 * The top-k choice is an integer decision taken from floating point, so the oracle takes it in
 * the kernel's precision: logits in fp32, accumulated over h in ascending order with one fused
 * multiply-add per step (each step rounded once), the bias added last.  Everything after the
 * choice is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static float bf16f(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static double bf16d(uint16_t b) { return (double)bf16f(b); }

/* logits [T,E] fp32 (reading above: fp32 sequential fused multiply-add over h, then + b[e]). */
void orc_router_logits(const uint16_t *x, const uint16_t *w, const float *bias, int64_t T, int32_t H, int32_t E,
                       float *logits) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t e = 0; e < E; ++e) {
            float acc = 0.0f;
            for (int32_t h = 0; h < H; ++h) acc = fmaf(bf16f(x[t * H + h]), bf16f(w[(int64_t)h * E + e]), acc);
            if (bias) acc = acc + bias[e];
            logits[t * E + e] = acc;
        }
    }
}

/* Top-k by descending logit (softmax is increasing in the logit), equal logits in ascending id;
 * weights = softmax over the K selected logits, fp64. */
void orc_router_topk(const float *logits, int64_t T, int32_t E, int32_t K, int32_t *ids, double *weights) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        char *sel = calloc((size_t)E, 1);
        for (int32_t k = 0; k < K; ++k) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e)
                if (!sel[e] && (best < 0 || l[e] > l[best])) best = e;  /* strict: the lower id wins ties */
            sel[best] = 1;
            ids[t * K + k] = best;
        }
        free(sel);
        const double m = (double)l[ids[t * K]];
        double den = 0.0;
        for (int32_t k = 0; k < K; ++k) den += exp((double)l[ids[t * K + k]] - m);
        for (int32_t k = 0; k < K; ++k) weights[t * K + k] = exp((double)l[ids[t * K + k]] - m) / den;
    }
}

/* Backward (reading above).  weights and dtopk are the forward's fp32 weights and the layer's
 * fp32 top-k weight gradient; dw [H,E], dbias [E] (may be NULL), dx [T,H]: fp64. */
void orc_router_backward(const uint16_t *x, const uint16_t *w, int64_t T, int32_t H, int32_t E, int32_t K,
                         const int32_t *ids, const float *weights, const float *dtopk, double *dw, double *dbias,
                         double *dx) {
    double *g = malloc(sizeof(double) * (size_t)(T * K));
    for (int64_t t = 0; t < T; ++t) {
        double s = 0.0;
        for (int32_t k = 0; k < K; ++k) s += (double)weights[t * K + k] * (double)dtopk[t * K + k];
        for (int32_t k = 0; k < K; ++k)
            g[t * K + k] = (double)weights[t * K + k] * ((double)dtopk[t * K + k] - s);
    }
    memset(dw, 0, sizeof(double) * (size_t)H * (size_t)E);
    if (dbias) memset(dbias, 0, sizeof(double) * (size_t)E);
#pragma omp parallel for schedule(static)
    for (int32_t h = 0; h < H; ++h) {
        for (int64_t t = 0; t < T; ++t) {
            const double xv = bf16d(x[t * H + h]);
            for (int32_t k = 0; k < K; ++k) dw[(int64_t)h * E + ids[t * K + k]] += xv * g[t * K + k];
        }
    }
    if (dbias)
        for (int64_t t = 0; t < T; ++t)
            for (int32_t k = 0; k < K; ++k) dbias[ids[t * K + k]] += g[t * K + k];
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int32_t k = 0; k < K; ++k) acc += g[t * K + k] * bf16d(w[(int64_t)h * E + ids[t * K + k]]);
            dx[t * H + h] = acc;
        }
    }
    free(g);
}
