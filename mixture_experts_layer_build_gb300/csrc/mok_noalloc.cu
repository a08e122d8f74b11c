// mok_noalloc.cu -- a schedule build that needs no device allocation at all.
//
// mok_build_schedule keeps its per-chunk expert histogram (scratch) in the caller's workspace.
// Callers that cannot allocate device memory -- code running where cudaMalloc is forbidden or
// unavailable, such as inside a memory-pool-managed runtime that hands out only fixed buffers, or
// a framework hook that may not allocate while it runs -- use mok_build_schedule_noalloc
// instead: the caller provides only the input ids/weights and the output tables, and the scratch
// lives in the fixed-size device array below, which every GPU that loads this library holds
// until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "mok_internal.cuh"

namespace mok {
namespace {

// Largest per-chunk histogram this entry point accepts: nchunks * (E + 1) int32 entries, with
// nchunks = ceil(T*K / 512).  2 MiB.
constexpr int64_t kNoallocHistEntries = int64_t(1) << 19;

static __device__ __align__(256) int32_t g_sched_scratch[kNoallocHistEntries];

// Device address of g_sched_scratch, looked up once per device with that device current.  In host
// code the symbol's name is only a host-side stand-in, never a device address.
int32_t* scratch_address(int dev) {
  static std::mutex mu;
  static int32_t* addr[64] = {nullptr};
  if (dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sched_scratch) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<int32_t*>(p);
  }
  return addr[dev];
}

}  // namespace
}  // namespace mok

using namespace mok;

extern "C" MOK_API mok_status mok_build_schedule_noalloc(const mok_config* cfg, const mok_shape* shape,
                                                         const int32_t* topk_ids, const float* topk_weights,
                                                         mok_schedule* sched, void* stream) {
  Sizes z;
  if (!sched || !make_sizes(cfg, shape, &z)) return MOK_ERR_INVALID_ARG;
  if (z.nchunks * (z.E + 1) > kNoallocHistEntries) return MOK_ERR_UNSUPPORTED;  // beyond the static scratch
  // the caller states the capacities of its tables; the kernels write up to the sizes this shape
  // and the resolved minibatch need, so a smaller buffer is refused before anything is enqueued
  if (sched->rpad_max < z.rpad_max || sched->tiles_max < z.tiles_max || sched->mblocks_max < z.mblocks_max)
    return MOK_ERR_WORKSPACE_TOO_SMALL;
  if (z.R > 0 && (!topk_ids || !topk_weights)) return MOK_ERR_INVALID_ARG;
  if (!sched->counts || !sched->offsets || !sched->poff || !sched->perm || !sched->inv || !sched->tiles ||
      !sched->mblocks || !sched->meta || !sched->row_weight || !sched->row_token)
    return MOK_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOK_ERR_CUDA;
  int32_t* scratch = scratch_address(dev);
  if (!scratch) return MOK_ERR_CUDA;
  sched->shape = *shape;
  sched->config = *cfg;
  sched->config.minibatch_rows = z.mb;  // automatic sizes resolved
  sched->config.macrobatch_rows = z.MB;
  sched->rpad_max = z.rpad_max;
  sched->tiles_max = z.tiles_max;
  sched->mblocks_max = z.mblocks_max;
  sched->status = reinterpret_cast<uint32_t*>(sched->meta + 15);
  sched->topk_weights = topk_weights;
  sched->ws = nullptr;
  sched->ws_bytes = 0;
  Staging st{};
  st.chunk_hist = scratch;  // every entry the schedule reads is written first: nothing to clear
  const int rc = launch_schedule(z, plain_route(topk_ids, topk_weights), *sched, st, static_cast<cudaStream_t>(stream));
  return rc ? MOK_ERR_CUDA : MOK_OK;
}
