// mok_api.cu -- the C ABI: host-side validation, workspace carving, TMA descriptors and the launch
// sequence of each call.  The calls follow the functional API of the "Mixture-of-Kittens (MoK)"
// project card (agentlenshq), "Functional API" block: get_workspace -> mok_workspace_bytes,
// build_schedule(topk_experts) -> mok_build_schedule, forward -> mok_forward, backward ->
// mok_backward, and ops.mxfp8_quantize -> mok_mxfp8_quantize.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <initializer_list>
#include <mutex>

#include "mok_gemm.cuh"
#include "mok_internal.cuh"

namespace mok {

namespace {
constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct Carver {
  char* base;
  size_t off = 0;
  template <class T>
  T* take(int64_t n) {
    off = align_up(off);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += static_cast<size_t>(n > 0 ? n : 0) * sizeof(T);
    return p;
  }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

mok_status from_cuda(int rc) { return rc == 0 ? MOK_OK : MOK_ERR_CUDA; }
}  // namespace

bool make_sizes(const mok_config* cfg, const mok_shape* shape, Sizes* s) {
  if (!cfg || !shape) return false;
  const mok_shape& p = *shape;
  if (p.T < 0 || p.H <= 0 || p.I <= 0 || p.K <= 0 || p.E <= 0) return false;
  if (p.H % 128 != 0 || p.I % 128 != 0) return false;
  if (p.K > p.E || p.E > 1024) return false;
  if (p.T * static_cast<int64_t>(p.K) >= (int64_t(1) << 31)) return false;
  // 0 = automatic granularity: a minibatch tile of about one expert's share of the routed rows (the
  // average rows per expert rounded up to 256 .. 2048 in powers of two; measured on GB300, every
  // size from 256 rows up ran within noise of the best, 128 rows 2 to 3 % slower), and a
  // macrobatch of at least four minibatches and 2048 rows
  int32_t mb = cfg->minibatch_rows, MB = cfg->macrobatch_rows;
  if (mb == 0) {
    const int64_t avg = (p.T * p.K + p.E - 1) / p.E;
    mb = 2 * kRowTile;
    while (mb < avg && mb < 2048) mb *= 2;
  }
  if (mb < kRowTile || mb % kRowTile != 0) return false;
  if (MB == 0) {
    const int32_t want = 4 * mb > 2048 ? 4 * mb : 2048;
    MB = (want + mb - 1) / mb * mb;
  }
  if (MB < mb || MB % mb != 0) return false;
  if (cfg->num_ctas < 0 || (cfg->debug_flags & ~MOK_FLAG_STATIC_TILES) != 0) return false;
  if (cfg->precision != MOK_BF16 && cfg->precision != MOK_MXFP8) return false;
  s->T = p.T;
  s->H = p.H;
  s->I = p.I;
  s->E = p.E;
  s->K = p.K;
  s->mb = mb;
  s->MB = MB;
  s->R = p.T * p.K;
  s->rpad_max = s->R + static_cast<int64_t>(p.E) * (kRowTile - 1);
  s->tiles_max = (s->R + s->mb - 1) / s->mb + p.E;
  s->mblocks_max = s->rpad_max / kRowTile;
  s->nchunks = (s->R + kSchedChunk - 1) / kSchedChunk;
  s->mx = cfg->precision == MOK_MXFP8;
  s->clc = (cfg->debug_flags & MOK_FLAG_STATIC_TILES) == 0;
  if (s->rpad_max >= (int64_t(1) << 31)) return false;
  return true;
}

size_t carve_workspace(const Sizes& z, char* base, mok_schedule* s, Staging* st) {
  Carver c{base};
  mok_schedule d{};
  d.counts = c.take<int32_t>(z.E);
  d.offsets = c.take<int32_t>(z.E + 1);
  d.poff = c.take<int32_t>(z.E + 1);
  d.perm = c.take<int32_t>(z.rpad_max);
  d.inv = c.take<int32_t>(z.R);
  d.tiles = c.take<int32_t>(4 * z.tiles_max);
  d.mblocks = c.take<int32_t>(4 * z.mblocks_max);
  d.meta = c.take<int32_t>(16);
  d.status = reinterpret_cast<uint32_t*>(d.meta ? d.meta + 15 : nullptr);
  d.row_weight = c.take<float>(z.rpad_max);
  d.row_token = c.take<int32_t>(z.rpad_max);
  Staging t{};
  t.chunk_hist = c.take<int32_t>(z.nchunks * (z.E + 1));
  t.ybuf = c.take<uint16_t>(z.rpad_max * z.H);
  if (!z.mx) {
    t.dyg = c.take<uint16_t>(z.rpad_max * z.H);
    t.dgdu = c.take<uint16_t>(z.rpad_max * 2 * z.I);
    t.as = c.take<uint16_t>(z.rpad_max * z.I);
  }
  t.dspart = c.take<float>(z.rpad_max * (z.I / 64));  // dS partials: at most two per 128 columns
  if (z.mx) {
    const int64_t rt = (z.rpad_max + kRowTile - 1) / kRowTile;  // 128-row tiles of the routed rows
    const int64_t EH = static_cast<int64_t>(z.E) * z.H, EI = static_cast<int64_t>(z.E) * z.I;
    t.xq = c.take<uint8_t>(z.rpad_max * z.H);
    t.xs = c.take<uint8_t>(rt * 128 * (z.H / 32));
    t.aq = c.take<uint8_t>(z.rpad_max * z.I);
    t.as_sf = c.take<uint8_t>(rt * 128 * (z.I / 32));
    t.dyq = c.take<uint8_t>(z.rpad_max * z.H);
    t.dys = c.take<uint8_t>(rt * 128 * (z.H / 32));
    t.dgq = c.take<uint8_t>(z.rpad_max * 2 * z.I);
    t.dgs = c.take<uint8_t>(rt * 128 * (2 * z.I / 32));
    const int64_t rcap = z.rcap();
    t.dyr = c.take<uint8_t>(z.H * rcap);
    t.dyrs = c.take<uint8_t>(z.H * rcap / 32);
    t.dgr = c.take<uint8_t>(2 * z.I * rcap);
    t.dgrs = c.take<uint8_t>(2 * z.I * rcap / 32);
    t.sar = c.take<uint8_t>(z.I * rcap);
    t.sars = c.take<uint8_t>(z.I * rcap / 32);
    t.sw_gu = c.take<uint8_t>(2 * EI * (z.H / 32));
    t.sw_d = c.take<uint8_t>(EH * (z.I / 32));
    t.swt_d = c.take<uint8_t>(EI * (z.H / 32));
    t.swt_g = c.take<uint8_t>(EH * (z.I / 32));
    t.swt_u = c.take<uint8_t>(EH * (z.I / 32));
  }
  t.pairs = reinterpret_cast<int4*>(c.take<int32_t>(4 * z.mblocks_max));
  if (s) {
    s->counts = d.counts;
    s->offsets = d.offsets;
    s->poff = d.poff;
    s->perm = d.perm;
    s->inv = d.inv;
    s->tiles = d.tiles;
    s->mblocks = d.mblocks;
    s->meta = d.meta;
    s->status = d.status;
    s->row_weight = d.row_weight;
    s->row_token = d.row_token;
  }
  if (st) *st = t;
  return align_up(c.off);
}

size_t carve_ctx(const Sizes& z, char* base, Ctx* ctx) {
  Carver c{base};
  Ctx x{};
  if (z.mx) {
    x.xr = c.take<uint8_t>(z.H * z.rcap());
    x.xrs = c.take<uint8_t>(z.H * z.rcap() / 32);
  } else {
    x.xg = c.take<uint16_t>(z.rpad_max * z.H);
  }
  x.gu = z.mx ? static_cast<void*>(c.take<float>(z.rpad_max * 2 * z.I))
              : static_cast<void*>(c.take<uint16_t>(z.rpad_max * 2 * z.I));
  x.a = c.take<uint16_t>(z.rpad_max * z.I);
  if (ctx) *ctx = x;
  return align_up(c.off);
}

// SM count of the current device, cached per device; 0 when it cannot be read (the caller's launch
// then fails and reports MOK_ERR_CUDA rather than running on a guessed grid).
int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link against libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D tensor [outer, inner] (inner contiguous), 128-byte swizzled boxes [box_outer, box_inner].
static bool make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, uint32_t esize, const void* base, uint64_t inner,
                         uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                         CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !base || !aligned16(base)) return false;
  if (outer == 0) outer = 1;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * esize};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                    uint32_t box_outer) {
  return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, outer, box_inner, box_outer);
}

bool make_tmap_bf16_sw64(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                         uint32_t box_outer) {
  return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, outer, box_inner, box_outer,
                      CU_TENSOR_MAP_SWIZZLE_64B);
}

bool make_tmap_f32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                   uint32_t box_outer) {
  return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, inner, outer, box_inner, box_outer);
}

bool make_tmap_f32_sw64(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                        uint32_t box_outer) {
  return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, inner, outer, box_inner, box_outer,
                      CU_TENSOR_MAP_SWIZZLE_64B);
}

bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                  uint32_t box_outer, int swizzle_bytes) {
  const CUtensorMapSwizzle sw = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                      : CU_TENSOR_MAP_SWIZZLE_NONE;
  return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, inner, outer, box_inner, box_outer, sw);
}

// One thread waits on an mbarrier that nothing completes, through the bounded wait every GEMM role
// uses: it must give up at the deadline, record MOK_ERR_TIMEOUT in *status and return.
__global__ void selftest_wait_kernel(uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(smem_u32(&bar), 1);
  fence_barrier_init();
  mbar_wait(smem_u32(&bar), 0u, reinterpret_cast<volatile int*>(&abort_flag), status);
}

static mok_trace* g_trace = nullptr;

void trace_begin(cudaStream_t s, int kind) {
  mok_trace* t = g_trace;
  if (!t || t->count >= t->capacity) return;
  t->kinds[t->count] = kind;
  cudaEventRecord(static_cast<cudaEvent_t>(t->events[2 * t->count]), s);
}

void trace_end(cudaStream_t s) {
  mok_trace* t = g_trace;
  if (!t || t->count >= t->capacity) return;
  cudaEventRecord(static_cast<cudaEvent_t>(t->events[2 * t->count + 1]), s);
  ++t->count;
}

}  // namespace mok

using namespace mok;

extern "C" {

const char* mok_version(void) { return "0.1.0"; }

const char* mok_status_string(mok_status s) {
  switch (s) {
    case MOK_OK: return "ok";
    case MOK_ERR_INVALID_ARG: return "invalid argument";
    case MOK_ERR_UNSUPPORTED: return "unsupported";
    case MOK_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOK_ERR_CUDA: return "CUDA error";
    case MOK_ERR_BAD_EXPERT_ID: return "expert id out of range";
    case MOK_ERR_CAPACITY: return "schedule capacity exceeded";
    case MOK_ERR_TIMEOUT: return "bounded device wait timed out";
  }
  return "unknown status";
}

size_t mok_workspace_bytes(const mok_config* cfg, const mok_shape* shape) {
  Sizes z;
  if (!make_sizes(cfg, shape, &z)) return 0;
  return carve_workspace(z, nullptr, nullptr, nullptr);
}

size_t mok_fwd_ctx_bytes(const mok_config* cfg, const mok_shape* shape) {
  Sizes z;
  if (!make_sizes(cfg, shape, &z)) return 0;
  return carve_ctx(z, nullptr, nullptr);
}

mok_status mok_mxfp8_quantize(const void* in_bf16, int64_t rows, int64_t cols, uint8_t* out_e4m3,
                              uint8_t* out_e8m0, void* stream) {
  if (rows < 0 || cols < 0 || cols % 32 != 0) return MOK_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return MOK_OK;
  if (!in_bf16 || !out_e4m3 || !out_e8m0) return MOK_ERR_INVALID_ARG;
  if (!aligned16(in_bf16) || !aligned16(out_e4m3)) return MOK_ERR_INVALID_ARG;
  return from_cuda(launch_mxfp8_quantize(static_cast<const uint16_t*>(in_bf16), rows, cols, out_e4m3, out_e8m0,
                                         as_stream(stream)));
}

mok_status mok_build_schedule(const mok_config* cfg, const mok_shape* shape, const int32_t* topk_ids,
                              const float* topk_weights, void* ws, size_t ws_bytes, mok_schedule* out,
                              void* stream) {
  Sizes z;
  if (!out || !make_sizes(cfg, shape, &z)) return MOK_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return MOK_ERR_INVALID_ARG;
  if (z.R > 0 && (!topk_ids || !topk_weights)) return MOK_ERR_INVALID_ARG;
  Staging st;
  mok_schedule s{};
  const size_t need = carve_workspace(z, static_cast<char*>(ws), &s, &st);
  if (ws_bytes < need) return MOK_ERR_WORKSPACE_TOO_SMALL;
  s.shape = *shape;
  s.config = *cfg;
  s.config.minibatch_rows = z.mb;  // automatic sizes resolved
  s.config.macrobatch_rows = z.MB;
  s.rpad_max = z.rpad_max;
  s.tiles_max = z.tiles_max;
  s.mblocks_max = z.mblocks_max;
  s.topk_weights = topk_weights;
  s.ws = ws;
  s.ws_bytes = ws_bytes;
  const int rc = launch_schedule(z, plain_route(topk_ids, topk_weights), s, st, as_stream(stream));
  if (rc) return MOK_ERR_CUDA;
  *out = s;
  return MOK_OK;
}

static mok_status check_sched(const mok_schedule* s, Sizes* z, Staging* st) {
  if (!s || !s->ws) return MOK_ERR_INVALID_ARG;
  if (!make_sizes(&s->config, &s->shape, z)) return MOK_ERR_INVALID_ARG;
  mok_schedule again{};
  const size_t need = carve_workspace(*z, static_cast<char*>(s->ws), &again, st);
  if (s->ws_bytes < need || again.meta != s->meta) return MOK_ERR_INVALID_ARG;
  return MOK_OK;
}

static int grid_of(const mok_schedule* s) {
  const int n = s->config.num_ctas;
  return n > 0 ? n : sm_count();
}

static bool all16(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (!p || !aligned16(p)) return false;
  return true;
}

static bool all4(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (!p || (reinterpret_cast<uintptr_t>(p) & 3u) != 0) return false;
  return true;
}

}  // extern "C"

namespace mok {
namespace {

// Where a pass's per-slot results go: the plain layer combines them itself; expert parallelism
// pushes them to the ranks holding the tokens, which combine them afterwards.
struct SlotOut {
  const RowDst* rows;  // expert parallelism: y (forward) or dX rows (backward) per slot
  const RowDst* ds;    // expert parallelism: d_topk_weights per slot (backward)
  int32_t rank;
};

// The forward through the down projection (or the combine, plain layer): gather (dispatch), the
// gate/up and down GEMMs, then the combine into out (plain) or the push of each y row (EP).
mok_status forward_impl(const mok_schedule* sched, const RowSrc& x, const mok_weights* w, void* out, void* fwd_ctx,
                        size_t fwd_ctx_bytes, const SlotOut* ep, void* stream) {
  Sizes z;
  Staging st;
  mok_status rc = check_sched(sched, &z, &st);
  if (rc != MOK_OK) return rc;
  if (!w || !fwd_ctx) return MOK_ERR_INVALID_ARG;
  Ctx ctx;
  if (fwd_ctx_bytes < carve_ctx(z, static_cast<char*>(fwd_ctx), &ctx)) return MOK_ERR_WORKSPACE_TOO_SMALL;
  if (reinterpret_cast<uintptr_t>(fwd_ctx) % kAlign) return MOK_ERR_INVALID_ARG;
  for (int r = 0; r < (x.n ? x.n : 1); ++r)
    if (z.T > 0 && (!x.p[r] || !aligned16(x.p[r]))) return MOK_ERR_INVALID_ARG;
  if (!ep && z.T > 0 && (!out || !aligned16(out))) return MOK_ERR_INVALID_ARG;
  if (z.mx) {
    if (!all16({w->q_gate, w->q_up, w->q_down}) || !all4({w->s_gate, w->s_up, w->s_down})) return MOK_ERR_INVALID_ARG;
  } else if (!all16({w->w_gate, w->w_up, w->w_down})) {
    return MOK_ERR_INVALID_ARG;
  }
  cudaStream_t s = as_stream(stream);
  if (z.mx) {  // weight scales into atoms, then x quantised on the gather
    const int64_t EI = static_cast<int64_t>(z.E) * z.I, EH = static_cast<int64_t>(z.E) * z.H;
    const int ad = z.mx_bn_h() / 128;  // atoms per B tile of the down projection
    const ScaleJob jobs[2] = {{w->s_gate, w->s_up, st.sw_gu, EI / 128, z.H / 128, 2, 1},
                              {w->s_down, nullptr, st.sw_d, EH / (128 * ad), z.I / 128, ad, 0}};
    if (launch_mx_scale_atoms(jobs, 2, s)) return MOK_ERR_CUDA;
    if (launch_gather_rows_mx(x, sched->row_token, sched->meta, z.rpad_max, z.H, st.xq, st.xs, ctx.xr, ctx.xrs,
                              z.rcap(), z.mx_bn_h() / 128, K_GATHER_X, s))
      return MOK_ERR_CUDA;
  } else if (launch_gather_rows(x, sched->inv, sched->row_token, sched->meta, z.T, z.K, z.rpad_max, z.H,
                                     ctx.xg, K_GATHER_X, s)) {
    return MOK_ERR_CUDA;
  }
  const int g = grid_of(sched);
  if (g <= 0) return MOK_ERR_CUDA;
  int e = launch_fwd_gemms(z, *sched, ctx, st, *w, g, s);
  if (e < 0) return MOK_ERR_INVALID_ARG;
  if (e) return MOK_ERR_CUDA;
  if (ep) return from_cuda(launch_push_rows(st.ybuf, sched->perm, sched->meta, z.rpad_max, z.H, *ep->rows, K_PUSH_Y, s));
  return from_cuda(launch_combine(st.ybuf, sched->inv, sched->topk_weights, z.T, z.K, z.H,
                                  static_cast<uint16_t*>(out), K_COMBINE, s));
}

// The backward: gather dY, the first data-gradient GEMM (SwiGLU backward, dS partials), the dS
// reduction, the second data-gradient GEMM, the dX reduction (plain) or the push of each dX row (EP),
// and the weight gradients.
mok_status backward_impl(const mok_schedule* sched, const void* fwd_ctx, const RowSrc& dy, const mok_weights* w,
                         const mok_grads* g, const SlotOut* ep, void* stream) {
  Sizes z;
  Staging st;
  mok_status rc = check_sched(sched, &z, &st);
  if (rc != MOK_OK) return rc;
  if (!w || !g || !fwd_ctx || (reinterpret_cast<uintptr_t>(fwd_ctx) % kAlign)) return MOK_ERR_INVALID_ARG;
  if (!all16({g->dw_gate, g->dw_up, g->dw_down})) return MOK_ERR_INVALID_ARG;
  for (int r = 0; r < (dy.n ? dy.n : 1); ++r)
    if (z.T > 0 && (!dy.p[r] || !aligned16(dy.p[r]))) return MOK_ERR_INVALID_ARG;
  if (!ep && z.T > 0 && (!g->dx || !g->d_topk_weights || !aligned16(g->dx))) return MOK_ERR_INVALID_ARG;
  if (z.mx) {
    if (!all16({w->qt_gate, w->qt_up, w->qt_down}) || !all4({w->st_gate, w->st_up, w->st_down}))
      return MOK_ERR_INVALID_ARG;
  } else if (!all16({w->w_gate, w->w_up, w->w_down})) {
    return MOK_ERR_INVALID_ARG;
  }
  Ctx ctx;
  carve_ctx(z, static_cast<char*>(const_cast<void*>(fwd_ctx)), &ctx);
  cudaStream_t s = as_stream(stream);
  const int grid = grid_of(sched);
  if (grid <= 0) return MOK_ERR_CUDA;
  if (z.mx) {  // weight scales into atoms, then dY quantised on the gather
    const int64_t EI = static_cast<int64_t>(z.E) * z.I, EH = static_cast<int64_t>(z.E) * z.H;
    const int ag = z.mx_bn_h() / 128;  // atoms per B tile of the second data-gradient GEMM
    const ScaleJob jobs[3] = {{w->st_down, nullptr, st.swt_d, EI / 128, z.H / 128, 1, 0},
                              {w->st_gate, nullptr, st.swt_g, EH / (128 * ag), z.I / 128, ag, 0},
                              {w->st_up, nullptr, st.swt_u, EH / (128 * ag), z.I / 128, ag, 0}};
    if (launch_mx_scale_atoms(jobs, 3, s)) return MOK_ERR_CUDA;
    if (launch_gather_rows_mx(dy, sched->row_token, sched->meta, z.rpad_max, z.H, st.dyq, st.dys, st.dyr, st.dyrs,
                              z.rcap(), 1, K_GATHER_DY, s))
      return MOK_ERR_CUDA;
  } else if (launch_gather_rows(dy, sched->inv, sched->row_token, sched->meta, z.T, z.K, z.rpad_max, z.H,
                                     st.dyg, K_GATHER_DY, s)) {
    return MOK_ERR_CUDA;
  }
  int e = launch_dgrad_gemms(z, *sched, ctx, st, *w, grid, 1, s);
  if (e) return e < 0 ? MOK_ERR_INVALID_ARG : MOK_ERR_CUDA;
  // dS partials per row: one per N tile of the first data-gradient GEMM (two per 128-column tile
  // when the block-scaled one splits its columns between two warps)
  const int n_tiles1 = z.mx ? z.I / (z.mx_dg1_split() ? 64 : 128) : z.I / (z.I % 256 == 0 ? 256 : 128);
  if (ep ? launch_ds_push(st.dspart, sched->inv, z.R, n_tiles1, *ep->ds, ep->rank, s)
         : launch_ds_reduce(st.dspart, sched->inv, z.R, n_tiles1, g->d_topk_weights, s))
    return MOK_ERR_CUDA;
  e = launch_dgrad_gemms(z, *sched, ctx, st, *w, grid, 2, s);
  if (e) return e < 0 ? MOK_ERR_INVALID_ARG : MOK_ERR_CUDA;
  if (ep ? launch_push_rows(st.ybuf, sched->perm, sched->meta, z.rpad_max, z.H, *ep->rows, K_PUSH_DX, s)
         : launch_combine(st.ybuf, sched->inv, nullptr, z.T, z.K, z.H, static_cast<uint16_t*>(g->dx), K_DX_REDUCE, s))
    return MOK_ERR_CUDA;
  e = launch_wgrad_gemms(z, *sched, ctx, st, *g, grid, s);
  if (e) return e < 0 ? MOK_ERR_INVALID_ARG : MOK_ERR_CUDA;
  return MOK_OK;
}

// Expert-parallel group description -> tables; false when the description is unusable.
bool ep_ok(const mok_ep_group* ep) {
  return ep && ep->world >= 1 && ep->world <= MOK_EP_MAX_RANKS && ep->rank >= 0 && ep->rank < ep->world &&
         ep->tokens_per_rank >= 0;
}

// Copy a host table of `world` per-rank device pointers; every entry must be set when `need`.
template <class D, class S>
bool fill_table(const S* src, int world, bool need, D* out) {
  for (int r = 0; r < MOK_EP_MAX_RANKS; ++r) out[r] = nullptr;
  if (!src) return !need;
  for (int r = 0; r < world; ++r) {
    out[r] = (D)(src[r]);
    if (need && !out[r]) return false;
  }
  return true;
}

}  // namespace
}  // namespace mok

extern "C" {

mok_status mok_forward(const mok_schedule* sched, const void* x, const mok_weights* w, void* out, void* fwd_ctx,
                       size_t fwd_ctx_bytes, void* stream) {
  return forward_impl(sched, plain_rows(x), w, out, fwd_ctx, fwd_ctx_bytes, nullptr, stream);
}

mok_status mok_backward(const mok_schedule* sched, const void* fwd_ctx, const void* dy, const mok_weights* w,
                        const mok_grads* g, void* stream) {
  return backward_impl(sched, fwd_ctx, plain_rows(dy), w, g, nullptr, stream);
}

mok_status mok_ep_build_schedule(const mok_config* cfg, const mok_shape* shape, const mok_ep_group* ep,
                                 const int32_t* const* topk_ids, const float* const* topk_weights, void* ws,
                                 size_t ws_bytes, mok_schedule* out, void* stream) {
  Sizes z;
  if (!out || !ep_ok(ep) || !make_sizes(cfg, shape, &z)) return MOK_ERR_INVALID_ARG;
  if (z.T != static_cast<int64_t>(ep->world) * ep->tokens_per_rank) return MOK_ERR_INVALID_ARG;
  if (static_cast<int64_t>(z.E) * ep->world > 1 << 30) return MOK_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return MOK_ERR_INVALID_ARG;
  RouteSrc route{};
  if (!fill_table(topk_ids, ep->world, z.R > 0, route.ids) || !fill_table(topk_weights, ep->world, z.R > 0, route.w))
    return MOK_ERR_INVALID_ARG;
  route.n = ep->world;
  route.slots_per = ep->tokens_per_rank * z.K;
  route.e0 = ep->rank * z.E;
  route.e_total = ep->world * z.E;
  if (route.slots_per == 0) route.slots_per = 1;
  Staging st;
  mok_schedule s{};
  const size_t need = carve_workspace(z, static_cast<char*>(ws), &s, &st);
  if (ws_bytes < need) return MOK_ERR_WORKSPACE_TOO_SMALL;
  s.shape = *shape;
  s.config = *cfg;
  s.config.minibatch_rows = z.mb;
  s.config.macrobatch_rows = z.MB;
  s.rpad_max = z.rpad_max;
  s.tiles_max = z.tiles_max;
  s.mblocks_max = z.mblocks_max;
  s.topk_weights = nullptr;  // the weights stay with the token owners; the rows carry them
  s.ws = ws;
  s.ws_bytes = ws_bytes;
  if (launch_schedule(z, route, s, st, as_stream(stream))) return MOK_ERR_CUDA;
  *out = s;
  return MOK_OK;
}

mok_status mok_ep_forward(const mok_schedule* sched, const mok_ep_group* ep, const void* const* x,
                          const mok_weights* w, void* const* y_recv, void* fwd_ctx, size_t fwd_ctx_bytes,
                          void* stream) {
  if (!sched || !ep_ok(ep) || sched->shape.T != static_cast<int64_t>(ep->world) * ep->tokens_per_rank)
    return MOK_ERR_INVALID_ARG;
  const bool any = sched->shape.T > 0;
  RowSrc src{};
  if (!fill_table(x, ep->world, any, src.p))
    return MOK_ERR_INVALID_ARG;
  src.n = ep->world;
  src.rows_per = ep->tokens_per_rank > 0 ? ep->tokens_per_rank : 1;
  RowDst dst{};
  if (!fill_table(y_recv, ep->world, any, dst.p)) return MOK_ERR_INVALID_ARG;
  for (int r = 0; r < ep->world; ++r)
    if (dst.p[r] && !aligned16(dst.p[r])) return MOK_ERR_INVALID_ARG;
  dst.n = ep->world;
  dst.slots_per = src.rows_per * sched->shape.K;
  const SlotOut so{&dst, nullptr, ep->rank};
  return forward_impl(sched, src, w, nullptr, fwd_ctx, fwd_ctx_bytes, &so, stream);
}

mok_status mok_ep_backward(const mok_schedule* sched, const mok_ep_group* ep, const void* fwd_ctx,
                           const void* const* dy, const mok_weights* w, float* dw_gate, float* dw_up, float* dw_down,
                           void* const* dx_recv, float* const* d_topk_weights, void* stream) {
  if (!sched || !ep_ok(ep) || sched->shape.T != static_cast<int64_t>(ep->world) * ep->tokens_per_rank)
    return MOK_ERR_INVALID_ARG;
  const bool any = sched->shape.T > 0;
  RowSrc src{};
  if (!fill_table(dy, ep->world, any, src.p))
    return MOK_ERR_INVALID_ARG;
  src.n = ep->world;
  src.rows_per = ep->tokens_per_rank > 0 ? ep->tokens_per_rank : 1;
  RowDst rows{}, ds{};
  if (!fill_table(dx_recv, ep->world, any, rows.p) || !fill_table(d_topk_weights, ep->world, any, ds.p))
    return MOK_ERR_INVALID_ARG;
  for (int r = 0; r < ep->world; ++r)
    if (rows.p[r] && !aligned16(rows.p[r])) return MOK_ERR_INVALID_ARG;
  rows.n = ds.n = ep->world;
  rows.slots_per = ds.slots_per = src.rows_per * sched->shape.K;
  const SlotOut so{&rows, &ds, ep->rank};
  mok_grads g{};
  g.dw_gate = dw_gate;
  g.dw_up = dw_up;
  g.dw_down = dw_down;
  return backward_impl(sched, fwd_ctx, src, w, &g, &so, stream);
}

mok_status mok_ep_combine(const mok_shape* shape, const mok_ep_group* ep, const int32_t* topk_ids,
                          const float* topk_weights, const void* recv, void* out, void* stream) {
  if (!shape || !ep_ok(ep) || shape->K <= 0 || shape->H <= 0 || shape->H % 8 != 0 || shape->E <= 0)
    return MOK_ERR_INVALID_ARG;
  const int64_t Tl = ep->tokens_per_rank;
  if (Tl == 0) return MOK_OK;
  if (!topk_ids || !recv || !out || !aligned16(recv) || !aligned16(out)) return MOK_ERR_INVALID_ARG;
  return from_cuda(launch_combine_slots(static_cast<const uint16_t*>(recv), topk_ids, ep->world * shape->E,
                                       topk_weights, Tl, shape->K, shape->H, static_cast<uint16_t*>(out),
                                       topk_weights ? K_EP_COMBINE : K_EP_DX_REDUCE, as_stream(stream)));
}

mok_status mok_set_trace(mok_trace* trace) {
  if (trace && (!trace->events || !trace->kinds || trace->capacity < 0 || trace->count < 0))
    return MOK_ERR_INVALID_ARG;
  g_trace = trace;
  return MOK_OK;
}

const char* mok_kernel_name(int32_t kind) {
  static const char* names[K_NUM_KINDS] = {
      "sched_hist",      "sched_scan",    "sched_scatter", "gather_x",       "gemm_fwd_gateup",
      "gemm_fwd_down",   "combine",       "gather_dy",     "gemm_dgrad1",    "ds_reduce",
      "gemm_dgrad2",     "dx_reduce",     "gemm_wgrad_gu", "gemm_wgrad_d",   "mxfp8_quantize",
      "mx_scale_atoms",  "router_logits", "router_topk",   "router_transpose", "router_dx",
      "router_dw",       "selftest_wait", "push_y",        "push_dx",        "ep_combine",
      "ep_dx_reduce",    "ds_push"};
  return (kind >= 0 && kind < K_NUM_KINDS) ? names[kind] : "?";
}

mok_status mok_mx_operands_of(const mok_schedule* sched, const void* fwd_ctx, mok_mx_operands* out) {
  Sizes z;
  Staging st;
  if (!out || !fwd_ctx || check_sched(sched, &z, &st) != MOK_OK || !z.mx) return MOK_ERR_INVALID_ARG;
  Ctx ctx;
  carve_ctx(z, static_cast<char*>(const_cast<void*>(fwd_ctx)), &ctx);
  out->xq = st.xq;
  out->xs = st.xs;
  out->aq = st.aq;
  out->as = st.as_sf;
  out->dyq = st.dyq;
  out->dys = st.dys;
  out->dgq = st.dgq;
  out->dgs = st.dgs;
  out->xr = ctx.xr;
  out->xrs = ctx.xrs;
  out->dyr = st.dyr;
  out->dyrs = st.dyrs;
  out->dgr = st.dgr;
  out->dgrs = st.dgrs;
  out->sar = st.sar;
  out->sars = st.sars;
  out->rows = z.rpad_max;
  out->rcap = z.rcap();
  out->xr_groups = z.mx_bn_h() / 128;
  out->sar_groups = z.mx_bn_i() / 128;
  return MOK_OK;
}

mok_status mok_selftest_wait_timeout(uint32_t* status, void* stream) {
  if (!status) return MOK_ERR_INVALID_ARG;
  trace_begin(as_stream(stream), K_SELFTEST_WAIT);
  selftest_wait_kernel<<<1, 32, 0, as_stream(stream)>>>(status);
  trace_end(as_stream(stream));
  return cudaGetLastError() == cudaSuccess ? MOK_OK : MOK_ERR_CUDA;
}

mok_status mok_read_device_status(const mok_schedule* sched, uint32_t* out, void* stream) {
  if (!sched || !sched->status || !out) return MOK_ERR_INVALID_ARG;
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, sched->status, sizeof v, cudaMemcpyDeviceToHost, as_stream(stream)) != cudaSuccess)
    return MOK_ERR_CUDA;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return MOK_ERR_CUDA;
  *out = v;
  return MOK_OK;
}

}  // extern "C"
