// mok_sched.cu -- the schedule: expert histogram, warp-scan prefix sums, stable permutation into the
// expert-grouped padded layout, minibatch tiles and 128-row blocks.
//
// "Mixture-of-Kittens(MoK)란? ..." (alltoptrend), section 4 (1): a single schedule table drives the
// forward and backward dispatch and combine; section 4 (3): no token is dropped and no CPU sizing
// step is needed (every size here is bounded on the host, nothing is read back).
//
// Three launches, all integer work, bit-exact by construction:
//   1. per-warp histograms of 512-slot chunks (shared-memory integer atomics: order-free);
//   2. one CTA: per-expert exclusive scan over chunks, block-wide warp-shuffle scans over experts
//      (offsets, padded offsets, tile starts), the tile and block tables, padding rows;
//   3. per-warp stable scatter: chunks walked in 32-slot pieces in order, equal experts ranked
//      by lane with __match_any_sync, so slots keep ascending order inside each expert.
#include "mok_internal.cuh"
#include "mok_ptx.cuh"

namespace mok {
namespace {

__global__ void __launch_bounds__(kSchedWarps * 32) sched_hist_kernel(const int32_t* __restrict__ ids, int64_t R,
                                                                     int E, int64_t nchunks,
                                                                     int32_t* __restrict__ chunk_hist) {
  extern __shared__ int32_t sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t chunk = static_cast<int64_t>(blockIdx.x) * kSchedWarps + warp;
  int32_t* h = sh + warp * (E + 1);
  for (int e = lane; e <= E; e += 32) h[e] = 0;
  __syncwarp();
  if (chunk >= nchunks) return;
  const int64_t j0 = chunk * kSchedChunk;
  for (int i = lane; i < kSchedChunk; i += 32) {
    const int64_t j = j0 + i;
    if (j < R) {
      int e = ids[j];
      if (e < 0 || e >= E) e = E;  // column E counts invalid ids
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
__device__ void block_excl_scan3(int (&v)[3], int (&tot)[3]) {
  __shared__ int wsum[3][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl[3];
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    incl[q] = warp_incl_scan(v[q], lane);
    if (lane == 31) wsum[q][warp] = incl[q];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int q = 0; q < 3; ++q) wsum[q][lane] = warp_incl_scan(wsum[q][lane], lane);
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < 3; ++q) {
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
                                                         int32_t* __restrict__ mblocks, int32_t* __restrict__ meta) {
  const int e = threadIdx.x;
  int cnt = 0;
  if (e < E) {
    for (int64_t c = 0; c < nchunks; ++c) {
      int32_t* p = chunk_hist + c * (E + 1) + e;
      const int v = *p;
      *p = cnt;  // becomes the count of expert e in the chunks before c
      cnt += v;
    }
  }
  __shared__ int s_bad;
  if (threadIdx.x == 0) {
    int bad = 0;
    for (int64_t c = 0; c < nchunks; ++c) bad += chunk_hist[c * (E + 1) + E];
    s_bad = bad;
  }
  const int padded = (cnt + kRowTile - 1) / kRowTile * kRowTile;
  const int ntile = (cnt + mb - 1) / mb;
  int v[3] = {cnt, padded, ntile}, tot[3];
  block_excl_scan3(v, tot);
  const int off = v[0], pof = v[1], tst = v[2];
  bool overflow = (tot[1] > rpad_max) || (tot[2] > tiles_max) || (tot[1] / kRowTile > mblocks_max);
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
    for (int r = pof + cnt; r < pof + padded; ++r) {
      perm[r] = -1;
      row_token[r] = -1;
      row_weight[r] = 0.0f;
    }
  }
  if (e == 0) {
    offsets[E] = tot[0];
    poff[E] = overflow ? 0 : tot[1];
    meta[0] = overflow ? 0 : tot[1];
    meta[1] = overflow ? 0 : tot[2];
    meta[2] = overflow ? 0 : tot[1] / kRowTile;
    uint32_t st = 0;
    if (s_bad) st |= 1u << MOK_ERR_BAD_EXPERT_ID;
    if (overflow) st |= 1u << MOK_ERR_CAPACITY;
    meta[15] = static_cast<int32_t>(st);  // the device status word; later kernels only OR into it
  }
}

__global__ void __launch_bounds__(kSchedWarps * 32) sched_scatter_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ w, int64_t R, int K, int E, int64_t nchunks,
    const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ poff, const int32_t* __restrict__ meta,
    int32_t* __restrict__ perm, int32_t* __restrict__ inv, int32_t* __restrict__ row_token,
    float* __restrict__ row_weight) {
  extern __shared__ int32_t sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t chunk = static_cast<int64_t>(blockIdx.x) * kSchedWarps + warp;
  if (chunk >= nchunks) return;  // whole warp leaves together
  if (meta[15] & (1 << MOK_ERR_CAPACITY)) return;
  int32_t* run = sh + warp * E;
  for (int e = lane; e < E; e += 32) run[e] = poff[e] + chunk_base[chunk * (E + 1) + e];
  __syncwarp();
  const int64_t j0 = chunk * kSchedChunk;
  for (int p = 0; p < kSchedChunk / 32; ++p) {
    const int64_t j = j0 + p * 32 + lane;
    int e = -1;
    if (j < R) {
      e = ids[j];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int base = (e >= 0) ? run[e] : 0;
    __syncwarp();
    if (e >= 0) {
      const int row = base + rank;
      perm[row] = static_cast<int32_t>(j);
      inv[j] = row;
      row_token[row] = static_cast<int32_t>(j / K);
      row_weight[row] = w[j];
      if (lane == 31 - __clz(peers)) run[e] = base + __popc(peers);
    } else if (j < R) {
      inv[j] = -1;  // an invalid id: the slot is skipped (status word says so)
    }
    __syncwarp();
  }
}

}  // namespace

int launch_schedule(const Sizes& z, const int32_t* ids, const float* w, const mok_schedule& s, const Staging& st,
                    cudaStream_t stream) {
  const int64_t nchunks = z.nchunks;
  const int blocks = static_cast<int>((nchunks + kSchedWarps - 1) / kSchedWarps);
  if (blocks > 0) {
    const size_t sh = sizeof(int32_t) * kSchedWarps * (z.E + 1);
    trace_begin(stream, K_SCHED_HIST);
    sched_hist_kernel<<<blocks, kSchedWarps * 32, sh, stream>>>(ids, z.R, z.E, nchunks, st.chunk_hist);
    trace_end(stream);
  }
  trace_begin(stream, K_SCHED_SCAN);
  sched_scan_kernel<<<1, 1024, 0, stream>>>(z.E, nchunks, st.chunk_hist, z.mb, z.MB, z.rpad_max, z.tiles_max,
                                            z.mblocks_max, s.counts, s.offsets, s.poff, s.perm, s.row_token,
                                            s.row_weight, s.tiles, s.mblocks, s.meta);
  trace_end(stream);
  if (blocks > 0) {
    const size_t sh = sizeof(int32_t) * kSchedWarps * z.E;
    trace_begin(stream, K_SCHED_SCATTER);
    sched_scatter_kernel<<<blocks, kSchedWarps * 32, sh, stream>>>(ids, w, z.R, z.K, z.E, nchunks, st.chunk_hist,
                                                                    s.poff, s.meta, s.perm, s.inv, s.row_token,
                                                                    s.row_weight);
    trace_end(stream);
  }
  return static_cast<int>(cudaGetLastError());
}

}  // namespace mok
