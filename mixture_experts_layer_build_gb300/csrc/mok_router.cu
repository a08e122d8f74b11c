// mok_router.cu -- the router step before the expert layer: logits of a linear router, the
// top-k experts of its softmax with renormalised weights, and the backward from the layer's
// top-k weight gradient to the router weight, its bias and the layer input.
//
// "Mixture-of-Kittens (MoK)" project card, "Functional API": the layer's schedule takes the
// top-k expert ids and weights that the router produced; "Cursor Open-Sources Mixture-of-Kittens
// (MoK) ...", English summary: the router-weight gradient is part of the backward.
//
// The top-k choice is an integer decision taken from floating point.  The logits are fp32, each
// accumulated over h in ascending order with one fused multiply-add per step and the bias added
// last, so the decision is reproducible (and the oracle takes it the same way).  Everything here
// is deterministic: no atomics, fixed reduction orders.
#include <cfloat>
#include <climits>

#include "mok_internal.cuh"
#include "mok_ptx.cuh"

namespace mok {
namespace {

// ---------------------------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------------------------
constexpr int kLgExperts = 64;  // experts per block
constexpr int kLgTokens = 32;   // tokens per block
constexpr int kLgChunk = 64;    // h values staged per step

// logits[t,e] = (sum over h ascending of x[t,h] W[h,e], fused multiply-add) + bias[e].  Block of
// 128 threads: 32 tokens x 64 experts; thread (te, tt) owns experts e0 + 4 te .. + 3 and tokens
// t0 + 4 tt .. + 3 (16 independent accumulation chains).  x and W chunks of 64 h are staged in
// shared memory as fp32: per h a thread reads its four W values as one 16-byte load and its four
// x values (shared by the warp's two token groups).  Chunk c + 1 is loaded into registers while
// chunk c is computed, in 16-byte loads: 64 h of compute is what covers a global load's latency
// (32 h did not).
__global__ void __launch_bounds__(128) router_logits_kernel(const uint16_t* __restrict__ x,
                                                            const uint16_t* __restrict__ w,
                                                            const float* __restrict__ bias, int64_t T, int H, int E,
                                                            float* __restrict__ logits) {
  pdl_wait();
  __shared__ __align__(16) float xs[kLgTokens][kLgChunk + 4];
  __shared__ __align__(16) float ws[kLgChunk][kLgExperts];
  const int tid = threadIdx.x;
  const int te = tid & 15, tt = tid >> 4;
  const int e0 = blockIdx.x * kLgExperts;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * kLgTokens;
  const bool wvec = (E & 7) == 0;  // W rows of 8 experts are 16-byte aligned
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  // x: token tid / 4, h (tid % 4) * 16 .. + 15 (two 16-byte loads).  W, 8-expert rows: row q / 8,
  // experts (q % 8) * 8 .. + 7 for q = tid + 128 j (four 16-byte loads); otherwise element q % 64 of
  // row q / 64 for q = tid + 128 j, j < 32, packed two per word.
  const int xr = tid >> 2, xc = (tid & 3) * 16;
  const int64_t xt = t0 + xr;
  uint4 xv[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
  uint4 wv[4];
  auto fetch = [&](int h0) {
    if (xt < T) {
      const uint4* p = reinterpret_cast<const uint4*>(x + xt * H + h0 + xc);
      xv[0] = __ldg(p);
      xv[1] = __ldg(p + 1);
    }
    if (wvec) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int q = tid + 128 * j, r = q >> 3, c = (q & 7) * 8;
        wv[j] = e0 + c < E ? __ldg(reinterpret_cast<const uint4*>(w + static_cast<int64_t>(h0 + r) * E + e0 + c))
                           : make_uint4(0, 0, 0, 0);
      }
    } else {
      uint32_t* pw = reinterpret_cast<uint32_t*>(wv);
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        uint32_t v2 = 0;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int q = tid + 128 * (j + k), r = q >> 6, c = q & 63;
          const uint32_t b = e0 + c < E ? __ldg(w + static_cast<int64_t>(h0 + r) * E + e0 + c) : 0u;
          v2 |= b << (16 * k);
        }
        pw[j >> 1] = v2;
      }
    }
  };
  fetch(0);
  for (int h0 = 0; h0 < H; h0 += kLgChunk) {
    __syncthreads();  // the previous chunk's reads of xs / ws are done
    {
      float4* d = reinterpret_cast<float4*>(&xs[xr][xc]);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        d[2 * i] = make_float4(bf16_lo(xv[i].x), bf16_hi(xv[i].x), bf16_lo(xv[i].y), bf16_hi(xv[i].y));
        d[2 * i + 1] = make_float4(bf16_lo(xv[i].z), bf16_hi(xv[i].z), bf16_lo(xv[i].w), bf16_hi(xv[i].w));
      }
    }
    if (wvec) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int q = tid + 128 * j, r = q >> 3, c = (q & 7) * 8;
        float4* d = reinterpret_cast<float4*>(&ws[r][c]);
        d[0] = make_float4(bf16_lo(wv[j].x), bf16_hi(wv[j].x), bf16_lo(wv[j].y), bf16_hi(wv[j].y));
        d[1] = make_float4(bf16_lo(wv[j].z), bf16_hi(wv[j].z), bf16_lo(wv[j].w), bf16_hi(wv[j].w));
      }
    } else {
      const uint32_t* pw = reinterpret_cast<const uint32_t*>(wv);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int q = tid + 128 * j;
        ws[q >> 6][q & 63] = (j & 1) ? bf16_hi(pw[j >> 1]) : bf16_lo(pw[j >> 1]);
      }
    }
    __syncthreads();
    if (h0 + kLgChunk < H) fetch(h0 + kLgChunk);
#pragma unroll 8
    for (int h = 0; h < kLgChunk; ++h) {
      const float4 wq = *reinterpret_cast<const float4*>(&ws[h][4 * te]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float xq = xs[4 * tt + i][h];
        acc[i][0] = __fmaf_rn(xq, wq.x, acc[i][0]);
        acc[i][1] = __fmaf_rn(xq, wq.y, acc[i][1]);
        acc[i][2] = __fmaf_rn(xq, wq.z, acc[i][2]);
        acc[i][3] = __fmaf_rn(xq, wq.w, acc[i][3]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t t = t0 + 4 * tt + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + 4 * te + j;
      if (e < E) logits[t * E + e] = bias ? __fadd_rn(acc[i][j], bias[e]) : acc[i][j];
    }
  }
}

// Top-K of each token's logits (warp per token): K rounds of a warp arg-max over the unselected
// experts, larger logit first and, on equal logits, the lower expert id; NaN logits are never
// chosen (a token with fewer than K non-NaN logits gets id -1, which the schedule reports).  The
// weights are the softmax over the K chosen logits (the full softmax renormalised to the top K).
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ logits, int64_t T, int E, int K,
                                                          int32_t* __restrict__ ids, float* __restrict__ wts) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (t >= T) return;  // whole warp
  const float* l = logits + t * E;
  uint32_t taken = 0;  // bit i: expert lane + 32 i chosen
  int my_id = -1;
  float my_l = 0.0f;
  for (int k = 0; k < K; ++k) {
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int i = 0, e = lane; e < E; ++i, e += 32) {
      if (taken & (1u << i)) continue;
      const float v = __ldg(l + e);
      if (v > bv || (v == bv && e < bi)) {
        bv = v;
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi == INT_MAX) bi = -1;
    if (bi >= 0 && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == k) {
      my_id = bi;
      my_l = bv;
    }
  }
  const float l0 = __shfl_sync(0xffffffffu, my_l, 0);
  const float ex = lane < K && my_id >= 0 ? expf(my_l - l0) : 0.0f;
  float den = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  if (lane < K) {
    ids[t * K + lane] = my_id;
    wts[t * K + lane] = my_id >= 0 ? ex / den : 0.0f;
  }
}

// ---------------------------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------------------------
// wt[e, h] = w[h, e] (32 x 32 tiles through shared memory).
__global__ void __launch_bounds__(256) router_transpose_kernel(const uint16_t* __restrict__ w, int H, int E,
                                                               uint16_t* __restrict__ wt) {
  pdl_wait();
  __shared__ uint16_t tile[32][33];
  const int e0 = blockIdx.x * 32, h0 = blockIdx.y * 32;
  for (int r = threadIdx.y; r < 32; r += 8) {
    const int h = h0 + r, e = e0 + threadIdx.x;
    tile[r][threadIdx.x] = (h < H && e < E) ? w[static_cast<int64_t>(h) * E + e] : 0;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += 8) {
    const int e = e0 + r, h = h0 + threadIdx.x;
    if (e < E && h < H) wt[static_cast<int64_t>(e) * H + h] = tile[threadIdx.x][r];
  }
}

// Warp per token: g_k = w_k (d_k - sum_j w_j d_j) (the gradient of the k-th chosen logit; the
// sum over the K lanes is a fixed butterfly), stored for the weight gradient, and
// dx[t, h] = (accumulate ? dx[t, h] : 0) + sum over k ascending of g_k wt[id_k, h], one bf16
// rounding.  Lanes take 8 consecutive h at a time.
__global__ void __launch_bounds__(256) router_dx_kernel(const int32_t* __restrict__ ids,
                                                        const float* __restrict__ wts,
                                                        const float* __restrict__ dtopk,
                                                        const uint16_t* __restrict__ wt, int64_t T, int H, int E,
                                                        int K, float* __restrict__ gbuf, uint16_t* __restrict__ dx,
                                                        int accumulate) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (t >= T) return;  // whole warp
  int id = -1;
  float wk = 0.0f, dk = 0.0f;
  if (lane < K) {
    id = __ldg(ids + t * K + lane);
    wk = __ldg(wts + t * K + lane);
    dk = __ldg(dtopk + t * K + lane);
  }
  const bool ok = id >= 0 && id < E;
  float s = ok ? wk * dk : 0.0f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  const float g = ok ? wk * (dk - s) : 0.0f;
  if (lane < K) gbuf[t * K + lane] = g;
  for (int h = lane * 8; h < H; h += 256) {
    float acc[8];
    if (accumulate) {
      const uint4 o = *reinterpret_cast<const uint4*>(dx + t * H + h);
      const uint32_t p[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = bf16_lo(p[i]);
        acc[2 * i + 1] = bf16_hi(p[i]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    }
    for (int k = 0; k < K; ++k) {
      const int ek = __shfl_sync(0xffffffffu, id, k);
      const float gk = __shfl_sync(0xffffffffu, g, k);
      if (ek < 0 || ek >= E) continue;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(wt + static_cast<int64_t>(ek) * H + h));
      const uint32_t p[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fmaf_rn(gk, bf16_lo(p[i]), acc[2 * i]);
        acc[2 * i + 1] = __fmaf_rn(gk, bf16_hi(p[i]), acc[2 * i + 1]);
      }
    }
    *reinterpret_cast<uint4*>(dx + t * H + h) =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                   pack_bf16x2(acc[6], acc[7]));
  }
}

// dW[h, e] = sum over expert e's routed rows (the schedule's expert-grouped layout) of
// x[token, h] g[slot]; db[e] likewise of g[slot].  Block (expert e, 512 h) of 256 P threads: the
// expert's rows are split into P parts; thread part p (tid / 256) sums part p in ascending row
// order for h0 + 2 (tid % 256) .. + 1, and the result is part 0 + part 1 (a fixed order).  The
// loop is bound by load latency, so P = 2 halves the time when the grid is too small to fill the
// GPU (fewer than two blocks per SM); otherwise P = 1 (every row in one ascending chain).  Each
// part's rows (token, g) come through shared memory 64 at a time.
constexpr int kDwRows = 64;
template <int P>
__global__ void __launch_bounds__(256 * P) router_dw_kernel(const uint16_t* __restrict__ x,
                                                        const float* __restrict__ gbuf,
                                                        const int32_t* __restrict__ counts,
                                                        const int32_t* __restrict__ poff,
                                                        const int32_t* __restrict__ perm, int H, int E, int K,
                                                        float* __restrict__ dw, float* __restrict__ db) {
  pdl_wait();
  static_assert(P == 1 || P == 2, "one or two row parts");
  __shared__ int64_t s_tok[P][kDwRows];
  __shared__ float s_g[P][kDwRows];
  __shared__ float2 s_part[256];
  __shared__ float s_db;
  const int e = blockIdx.x;
  const int p = P == 2 ? static_cast<int>(threadIdx.x >> 8) : 0, tl = threadIdx.x & 255;
  const int h = blockIdx.y * 512 + 2 * tl;
  const int n = __ldg(counts + e), nh = (n + P - 1) / P;
  const int r0 = __ldg(poff + e) + (p ? nh : 0), np = p ? n - nh : nh;  // this part's rows
  float a0 = 0.0f, a1 = 0.0f, ab = 0.0f;
  for (int c0 = 0; c0 < nh; c0 += kDwRows) {  // both parts take the same number of steps
    const int m = max(0, min(kDwRows, np - c0));
    __syncthreads();
    if (tl < m) {
      const int j = __ldg(perm + r0 + c0 + tl);
      s_tok[p][tl] = j < 0 ? -1 : j / K;
      s_g[p][tl] = j < 0 ? 0.0f : __ldg(gbuf + j);
    }
    __syncthreads();
    if (h < H) {
#pragma unroll 8
      for (int i = 0; i < m; ++i) {
        const int64_t t = s_tok[p][i];
        if (t < 0) continue;
        const float g = s_g[p][i];
        const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(x + t * H + h));
        a0 = __fmaf_rn(bf16_lo(v), g, a0);
        a1 = __fmaf_rn(bf16_hi(v), g, a1);
      }
    }
    if (tl == 0)
      for (int i = 0; i < m; ++i) ab += s_g[p][i];
  }
  if constexpr (P == 2) {
    if (p == 1) {
      s_part[tl] = make_float2(a0, a1);
      if (tl == 0) s_db = ab;
    }
    __syncthreads();
    if (p == 1) return;
    a0 = __fadd_rn(a0, s_part[tl].x);
    a1 = __fadd_rn(a1, s_part[tl].y);
    ab = __fadd_rn(ab, s_db);
  }
  if (h < H) {
    dw[static_cast<int64_t>(h) * E + e] = a0;
    dw[static_cast<int64_t>(h + 1) * E + e] = a1;
  }
  if (db && blockIdx.y == 0 && tl == 0) db[e] = ab;
}

bool router_shape_ok(int64_t T, int H, int E, int K) {
  return T >= 0 && H > 0 && H % 128 == 0 && E >= 1 && E <= 1024 && K >= 1 && K <= 32 && K <= E;
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

}  // namespace
}  // namespace mok

using namespace mok;

extern "C" MOK_API size_t mok_router_workspace_bytes(const mok_shape* s) {
  if (!s || !router_shape_ok(s->T, s->H, s->E, s->K)) return 0;
  return align256(static_cast<size_t>(s->E) * s->H * 2) + align256(static_cast<size_t>(s->T) * s->K * 4);
}

extern "C" MOK_API mok_status mok_router_forward(const mok_shape* s, const void* x, const void* w_router,
                                                 const float* bias, float* logits, int32_t* topk_ids,
                                                 float* topk_weights, void* stream) {
  if (!s || !router_shape_ok(s->T, s->H, s->E, s->K)) return MOK_ERR_INVALID_ARG;
  if (s->T == 0) return MOK_OK;
  if (!x || !w_router || !logits || !topk_ids || !topk_weights || (reinterpret_cast<uintptr_t>(x) & 15))
    return MOK_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const dim3 g1((s->E + kLgExperts - 1) / kLgExperts, static_cast<unsigned>((s->T + kLgTokens - 1) / kLgTokens));
  trace_begin(st, K_ROUTER_LOGITS);
  launch_pdl(router_logits_kernel, dim3(g1), dim3(128), 0, st, static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(w_router),
                                           bias, s->T, s->H, s->E, logits);
  trace_end(st);
  trace_begin(st, K_ROUTER_TOPK);
  launch_pdl(router_topk_kernel, dim3(static_cast<unsigned>((s->T + 7) / 8)), dim3(256), 0, st, logits, s->T, s->E,
             s->K, topk_ids, topk_weights);
  trace_end(st);
  return cudaGetLastError() == cudaSuccess ? MOK_OK : MOK_ERR_CUDA;
}

extern "C" MOK_API mok_status mok_router_backward(const mok_schedule* sched, const void* x, const void* w_router,
                                                  const int32_t* topk_ids, const float* topk_weights,
                                                  const float* d_topk_weights, float* dw_router, float* d_bias,
                                                  void* dx, int32_t accumulate_dx, void* ws, size_t ws_bytes,
                                                  void* stream) {
  if (!sched) return MOK_ERR_INVALID_ARG;
  const mok_shape& s = sched->shape;
  if (!router_shape_ok(s.T, s.H, s.E, s.K)) return MOK_ERR_INVALID_ARG;
  if (!w_router || !dw_router || !ws || ws_bytes < mok_router_workspace_bytes(&s)) return MOK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ws) % 256) return MOK_ERR_INVALID_ARG;
  if (s.T > 0 && (!x || !topk_ids || !topk_weights || !d_topk_weights || !dx ||
                  (reinterpret_cast<uintptr_t>(dx) & 15) || (reinterpret_cast<uintptr_t>(x) & 3)))
    return MOK_ERR_INVALID_ARG;
  if (!sched->counts || !sched->poff || !sched->perm) return MOK_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint16_t* wt = static_cast<uint16_t*>(ws);
  float* gbuf = reinterpret_cast<float*>(static_cast<char*>(ws) + align256(static_cast<size_t>(s.E) * s.H * 2));
  const dim3 gt((s.E + 31) / 32, (s.H + 31) / 32);
  trace_begin(st, K_ROUTER_TRANSPOSE);
  launch_pdl(router_transpose_kernel, dim3(gt), dim3(32, 8), 0, st, static_cast<const uint16_t*>(w_router), s.H, s.E, wt);
  trace_end(st);
  if (s.T > 0) {
    trace_begin(st, K_ROUTER_DX);
    launch_pdl(router_dx_kernel, dim3(static_cast<unsigned>((s.T + 7) / 8)), dim3(256), 0, st, topk_ids, topk_weights,
               d_topk_weights, wt, s.T, s.H, s.E, s.K, gbuf, static_cast<uint16_t*>(dx), accumulate_dx);
    trace_end(st);
  }
  const dim3 gw(s.E, (s.H + 511) / 512);
  trace_begin(st, K_ROUTER_DW);
  if (static_cast<int64_t>(gw.x) * gw.y < 2 * static_cast<int64_t>(sm_count()))  // small grid: two row parts
    launch_pdl(router_dw_kernel<2>, dim3(gw), dim3(512), 0, st, static_cast<const uint16_t*>(x), gbuf, sched->counts, sched->poff,
                                            sched->perm, s.H, s.E, s.K, dw_router, d_bias);
  else
    launch_pdl(router_dw_kernel<1>, dim3(gw), dim3(256), 0, st, static_cast<const uint16_t*>(x), gbuf, sched->counts, sched->poff,
                                            sched->perm, s.H, s.E, s.K, dw_router, d_bias);
  trace_end(st);
  return cudaGetLastError() == cudaSuccess ? MOK_OK : MOK_ERR_CUDA;
}
