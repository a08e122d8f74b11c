// mok_sched.cu -- the schedule: expert histogram, warp-scan prefix sums, stable permutation into the
// expert-grouped padded layout, minibatch tiles and 128-row blocks.
//
// "Mixture-of-Kittens(MoK)란? ..." (alltoptrend), section 4 (1): a single schedule table drives the
// forward and backward dispatch and combine; section 4 (3): no token is dropped and no CPU sizing
// step is needed (every size here is bounded on the host, nothing is read back).
//
// Three launches, all integer work, bit-exact by construction:
//   1. per-warp histograms of 512-slot chunks (shared-memory integer atomics: order-free), all of
//      a warp's id loads in flight together;
//   2. one CTA: a two-level scan -- 32 chunk groups x experts summed with loads coalesced across
//      experts, a per-expert scan over the groups, block-wide warp-shuffle scans over experts
//      (offsets, padded offsets, tile starts) -- then the tile and block tables, the padding rows,
//      and every chunk's absolute first row per expert written back;
//   3. per-warp stable scatter: a chunk walked in 32-slot pieces in order, equal experts ranked
//      by lane with __match_any_sync, so slots keep ascending order inside each expert.  Two warps
//      per CTA spread the scattered row writes over many SMs.
#include <climits>

#include "mok_internal.cuh"
#include "mok_once.h"
#include "mok_ptx.cuh"

namespace mok {
namespace {

constexpr int kHistWarps = 2;                    // warps per CTA of the histogram / scatter launches

// The local expert of slot j, or kSlotInvalid (an id outside the experts), or kSlotForeign (expert
// parallelism: an expert another rank owns).  Plain routing: ids in [0, E) are local.
__device__ __forceinline__ int route_id(const RouteSrc& r, int64_t j, int E) {
  if (r.n == 0) {
    const int e = __ldg(r.ids[0] + j);
    return (e < 0 || e >= E) ? kSlotInvalid : e;
  }
  const int64_t s = j / r.slots_per;
  const int g = __ldg(pick_rank(r.ids, s) + (j - s * r.slots_per));
  if (g < 0 || g >= r.e_total) return kSlotInvalid;
  const int e = g - r.e0;
  return (e < 0 || e >= E) ? kSlotForeign : e;
}
__device__ __forceinline__ float route_w(const RouteSrc& r, int64_t j) {
  if (r.n == 0) return __ldg(r.w[0] + j);
  const int64_t s = j / r.slots_per;
  return __ldg(pick_rank(r.w, s) + (j - s * r.slots_per));
}
constexpr int kPieces = kSchedChunk / 32;        // 32-slot pieces per chunk
constexpr int kBatch = 8;                        // pieces whose loads are in flight together

__global__ void __launch_bounds__(kHistWarps * 32) sched_hist_kernel(const RouteSrc route, int64_t R, int E,
                                                                    int64_t nchunks,
                                                                    int32_t* __restrict__ chunk_hist) {
  pdl_wait();
  extern __shared__ int32_t sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t chunk = static_cast<int64_t>(blockIdx.x) * kHistWarps + warp;
  int32_t* h = sh + warp * (E + 1);
  for (int e = lane; e <= E; e += 32) h[e] = 0;
  __syncwarp();
  if (chunk >= nchunks) return;
  const int64_t j0 = chunk * kSchedChunk;
  for (int p0 = 0; p0 < kPieces; p0 += kBatch) {
    int ev[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int64_t j = j0 + (p0 + b) * 32 + lane;
      ev[b] = j < R ? route_id(route, j, E) : INT32_MIN;
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (ev[b] == INT32_MIN || ev[b] == kSlotForeign) continue;  // another rank counts its slots
      const int e = ev[b] == kSlotInvalid ? E : ev[b];  // column E counts invalid ids
      atomicAdd(&h[e], 1);
    }
  }
  __syncwarp();
  for (int e = lane; e <= E; e += 32) chunk_hist[chunk * (E + 1) + e] = h[e];
}

// Inclusive warp scan.
__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += n;
  }
  return v;
}

// Exclusive block scan of three values (blockDim.x == 1024).  Returns totals through tot[3].
template <int N>
__device__ void block_excl_scan(int (&v)[N], int (&tot)[N]) {
  __shared__ int wsum[N][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl[N];
#pragma unroll
  for (int q = 0; q < N; ++q) {
    incl[q] = warp_incl_scan(v[q], lane);
    if (lane == 31) wsum[q][warp] = incl[q];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int q = 0; q < N; ++q) wsum[q][lane] = warp_incl_scan(wsum[q][lane], lane);
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < N; ++q) {
    const int before = warp > 0 ? wsum[q][warp - 1] : 0;
    const int ex = before + incl[q] - v[q];
    tot[q] = wsum[q][31];
    v[q] = ex;
  }
}

__global__ void __launch_bounds__(1024) sched_scan_kernel(int E, int64_t nchunks, int32_t* __restrict__ chunk_hist,
                                                         int mb, int MB, int64_t rpad_max, int64_t tiles_max,
                                                         int64_t mblocks_max, int32_t* __restrict__ counts,
                                                         int32_t* __restrict__ offsets, int32_t* __restrict__ poff,
                                                         int32_t* __restrict__ perm, int32_t* __restrict__ row_token,
                                                         float* __restrict__ row_weight, int32_t* __restrict__ tiles,
                                                         int32_t* __restrict__ mblocks, int32_t* __restrict__ meta,
                                                         int4* __restrict__ pairs) {
  pdl_wait();
  extern __shared__ int32_t part[];  // [32 chunk groups][E + 1]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int W = E + 1;
  const int64_t L = (nchunks + 31) / 32;  // chunks per group; group g = warp g
  const int64_t c0 = warp * L, c1 = min(nchunks, c0 + L);
  // level 1: per (group, expert) sums; lanes read consecutive experts of one chunk (coalesced),
  // eight chunks' loads in flight at a time
  for (int e = lane; e < W; e += 32) {
    int sum = 0;
    for (int64_t cb = c0; cb < c1; cb += 8) {
      int v8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v8[k] = cb + k < c1 ? chunk_hist[(cb + k) * W + e] : 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) sum += v8[k];
    }
    part[warp * W + e] = sum;
  }
  __syncthreads();
  // level 2: per expert, exclusive over the groups
  const int e = threadIdx.x;
  int cnt = 0;
  if (e < E) {
    for (int g = 0; g < 32; ++g) {
      const int v = part[g * W + e];
      part[g * W + e] = cnt;
      cnt += v;
    }
  }
  __shared__ int s_bad;
  __shared__ int2 s_pad[1024];  // per expert: [first padding row, end of its padded segment)
  if (threadIdx.x == 0) {
    int bad = 0;
    for (int g = 0; g < 32; ++g) bad += part[g * W + E];
    s_bad = bad;
  }
  const int padded = (cnt + kRowTile - 1) / kRowTile * kRowTile;
  const int ntile = (cnt + mb - 1) / mb;
  // pairs of consecutive 128-row blocks within each minibatch tile (the last one may be single)
  const int npair = ntile == 0 ? 0
                               : (ntile - 1) * ((mb / kRowTile + 1) / 2) +
                                     ((cnt - (ntile - 1) * mb + kRowTile - 1) / kRowTile + 1) / 2;
  int v[4] = {cnt, padded, ntile, npair}, tot[4];
  block_excl_scan<4>(v, tot);
  const int off = v[0], pof = v[1], tst = v[2], ppo = v[3];
  const bool overflow = (tot[1] > rpad_max) || (tot[2] > tiles_max) || (tot[1] / kRowTile > mblocks_max);
  if (e < E && !overflow) {
    counts[e] = cnt;
    offsets[e] = off;
    poff[e] = pof;
    for (int q = 0; q < ntile; ++q) {
      int32_t* t = tiles + 4 * static_cast<int64_t>(tst + q);
      const int first = pof + q * mb;
      t[0] = e;
      t[1] = first;
      t[2] = min(mb, cnt - q * mb);
      t[3] = first / MB;
    }
    for (int b = 0; b < padded / kRowTile; ++b) {
      int32_t* m = mblocks + 4 * static_cast<int64_t>(pof / kRowTile + b);
      m[0] = e;
      m[1] = pof + b * kRowTile;
      m[2] = min(kRowTile, cnt - b * kRowTile);
      m[3] = tst + (b * kRowTile) / mb;
    }
    if (pairs) {
      int p = ppo;
      for (int q = 0; q < ntile; ++q) {
        const int np = ((min(mb, cnt - q * mb) + kRowTile - 1) / kRowTile + 1) / 2;
        for (int j = 0; j < np; ++j) pairs[p + j] = make_int4(e, pof + q * mb + 2 * j * kRowTile, tst + q, p);
        p += np;
      }
    }
    s_pad[e] = make_int2(pof + cnt, pof + padded);
    for (int g = 0; g < 32; ++g) part[g * W + e] += pof;  // first row of group g's slots of e
  }
  if (e == 0) {
    offsets[E] = tot[0];
    poff[E] = overflow ? 0 : tot[1];
    meta[0] = overflow ? 0 : tot[1];
    meta[1] = overflow ? 0 : tot[2];
    meta[2] = overflow ? 0 : tot[1] / kRowTile;
    meta[3] = overflow || !pairs ? 0 : tot[3];
    uint32_t st = 0;
    if (s_bad) st |= 1u << MOK_ERR_BAD_EXPERT_ID;
    if (overflow) st |= 1u << MOK_ERR_CAPACITY;
    meta[15] = static_cast<int32_t>(st);  // the device status word; later kernels only OR into it
  }
  __syncthreads();
  if (overflow) return;
  // padding rows of every expert, spread over the whole block
  for (int idx = threadIdx.x; idx < E * kRowTile; idx += blockDim.x) {
    const int2 pr = s_pad[idx / kRowTile];
    const int r = pr.x + idx % kRowTile;
    if (r < pr.y) {
      perm[r] = -1;
      row_token[r] = -1;
      row_weight[r] = 0.0f;
    }
  }
  // every chunk's first row per expert, in place (eight chunks' loads in flight at a time)
  for (int ex = lane; ex < E; ex += 32) {
    int run = part[warp * W + ex];
    for (int64_t cb = c0; cb < c1; cb += 8) {
      int v8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v8[k] = cb + k < c1 ? chunk_hist[(cb + k) * W + ex] : 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (cb + k < c1) chunk_hist[(cb + k) * W + ex] = run;
        run += v8[k];
      }
    }
  }
}

__global__ void __launch_bounds__(kHistWarps * 32) sched_scatter_kernel(
    const RouteSrc route, int64_t R, int K, int E, int64_t nchunks,
    const int32_t* __restrict__ chunk_first, const int32_t* __restrict__ meta, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv, int32_t* __restrict__ row_token, float* __restrict__ row_weight) {
  pdl_wait();
  extern __shared__ int32_t sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t chunk = static_cast<int64_t>(blockIdx.x) * kHistWarps + warp;
  if (chunk >= nchunks) return;  // whole warp leaves together
  if (meta[15] & (1 << MOK_ERR_CAPACITY)) return;
  int32_t* run = sh + warp * E;
  for (int e = lane; e < E; e += 32) run[e] = chunk_first[chunk * (E + 1) + e];
  __syncwarp();
  const int64_t j0 = chunk * kSchedChunk;
  for (int p0 = 0; p0 < kPieces; p0 += kBatch) {
    int ev[kBatch];
    float wv[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int64_t j = j0 + (p0 + b) * 32 + lane;
      ev[b] = kSlotForeign;
      wv[b] = 0.0f;
      if (j < R) {
        ev[b] = route_id(route, j, E);
        wv[b] = route_w(route, j);
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int64_t j = j0 + (p0 + b) * 32 + lane;
      const int e = ev[b] >= 0 ? ev[b] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int base = (e >= 0) ? run[e] : 0;
      __syncwarp();
      if (e >= 0) {
        const int row = base + rank;
        perm[row] = static_cast<int32_t>(j);
        inv[j] = row;
        row_token[row] = static_cast<int32_t>(j / K);
        row_weight[row] = wv[b];
        if (lane == 31 - __clz(peers)) run[e] = base + __popc(peers);
      } else if (j < R) {
        // skipped: another rank's expert, or an invalid id (the status word says so; with
        // expert parallelism it is marked apart, since its token's owner zeroes its dS)
        inv[j] = (route.n != 0 && ev[b] == kSlotInvalid) ? kSlotInvalid : kSlotForeign;
      }
      __syncwarp();
    }
  }
}

}  // namespace

int launch_schedule(const Sizes& z, const RouteSrc& route, const mok_schedule& s, const Staging& st,
                    cudaStream_t stream) {
  static DeviceOnce once;  // the scan's group sums need up to 32 x 1025 int32 of shared memory, on each device
  const int se = once.run([](int* d) { return static_cast<int>(cudaGetDevice(d)); },
                          [] {
                            return static_cast<int>(cudaFuncSetAttribute(
                                sched_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(sizeof(int32_t) * 32 * 1025)));
                          },
                          static_cast<int>(cudaErrorInvalidDevice));
  if (se) return se;
  const int64_t nchunks = z.nchunks;
  const int blocks = static_cast<int>((nchunks + kHistWarps - 1) / kHistWarps);
  if (blocks > 0) {
    const size_t sh = sizeof(int32_t) * kHistWarps * (z.E + 1);
    trace_begin(stream, K_SCHED_HIST);
    launch_pdl(sched_hist_kernel, dim3(blocks), dim3(kHistWarps * 32), sh, stream, route, z.R, z.E, nchunks, st.chunk_hist);
    trace_end(stream);
  }
  trace_begin(stream, K_SCHED_SCAN);
  launch_pdl(sched_scan_kernel, dim3(1), dim3(1024), sizeof(int32_t) * 32 * (z.E + 1), stream, 
      z.E, nchunks, st.chunk_hist, z.mb, z.MB, z.rpad_max, z.tiles_max, z.mblocks_max, s.counts, s.offsets, s.poff,
      s.perm, s.row_token, s.row_weight, s.tiles, s.mblocks, s.meta, st.pairs);
  trace_end(stream);
  if (blocks > 0) {
    const size_t sh = sizeof(int32_t) * kHistWarps * z.E;
    trace_begin(stream, K_SCHED_SCATTER);
    launch_pdl(sched_scatter_kernel, dim3(blocks), dim3(kHistWarps * 32), sh, stream, route, z.R, z.K, z.E, nchunks, st.chunk_hist,
                                                                   s.meta, s.perm, s.inv, s.row_token, s.row_weight);
    trace_end(stream);
  }
  return static_cast<int>(cudaGetLastError());
}

}  // namespace mok
