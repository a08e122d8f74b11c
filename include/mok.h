/*
 * mok.h -- C ABI of libmok: the deterministic top-k routed SwiGLU expert layer (Mixture-of-Kittens
 * style), forward and backward, on one GB300 GPU (sm_103a).
 *
 * The calls follow the functional API the project card describes ("Mixture-of-Kittens (MoK)"
 * project card, agentlenshq: "Functional API" block -- get_workspace, build_schedule(topk_experts),
 * forward, backward -- and "Key concepts" table -- ops.mxfp8_quantize, the MoKConfig knobs).
 * With one GPU the expert-parallel dispatch and combine of the pages become on-device gathers and
 * a fixed-order weighted reduction.
 *
 * Conventions shared by every call
 *  - Pointers are DEVICE pointers unless a comment says otherwise.  bf16 tensors are row-major
 *    arrays of 16-bit patterns; fp32 is IEEE binary32; E4M3 / E8M0 are bytes.
 *  - Ownership: the caller allocates and frees every buffer (inputs, outputs, the workspace and
 *    the forward context).  The library never allocates device memory and keeps no state
 *    between calls beyond per-device caches (the SM count, which kernels have had their
 *    shared-memory limit raised on that device) and one driver entry point.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).  Every
 *    call only enqueues work on it and returns; none synchronises, except
 *    mok_read_device_status.  Inputs must stay valid until the enqueued work has run.
 *  - CUDA graphs: mok_build_schedule, mok_forward and mok_backward allocate nothing and read
 *    nothing back, and their grids and tensor maps depend only on the shape and the buffer
 *    addresses.  A step made of them may be captured once (stream capture) and replayed; each
 *    replay rebuilds the schedule on the device from the routing the captured buffers then hold.
 *    Call each entry point once outside capture first on each device, so that its one-time
 *    kernel attribute setup for that device is done.
 *  - Errors: argument, shape, alignment and size problems are detected on the host and returned
 *    before anything is enqueued.  Data-dependent problems found on the device (an expert id
 *    outside [0, E), a bounded wait that timed out) set bits (1 << code) in the schedule's device
 *    status word; the kernels skip the offending work and return normally.  Read the word with
 *    mok_read_device_status.
 *  - Determinism: for the same inputs every output is bitwise identical from run to run, for any
 *    num_ctas, minibatch or macrobatch setting; no floating-point atomics are used.
 *  - Re-entrancy: calls on distinct workspaces may run concurrently.
 */
#ifndef MOK_H
#define MOK_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOK_API __attribute__((visibility("default")))
#else
#define MOK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOK_OK = 0,
  MOK_ERR_INVALID_ARG = 1,          /* null pointer, bad shape, misaligned pointer */
  MOK_ERR_UNSUPPORTED = 2,          /* a shape or mode this build does not implement */
  MOK_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace or forward context smaller than required */
  MOK_ERR_CUDA = 4,                 /* a CUDA runtime / driver call failed */
  MOK_ERR_BAD_EXPERT_ID = 5,        /* device status: a top-k id outside [0, E); that slot is skipped */
  MOK_ERR_CAPACITY = 6,             /* device status: a schedule table overflowed (cannot happen
                                       with a workspace of mok_workspace_bytes) */
  MOK_ERR_TIMEOUT = 7               /* device status: a bounded in-kernel wait gave up */
} mok_status;

typedef enum { MOK_BF16 = 0, MOK_MXFP8 = 1 } mok_precision;

/* Layer knobs (the project card's MoKConfig: minibatch granularity and macrobatch size; the
 * communication-SM count has no meaning on one GPU).
 *  minibatch_rows  rows of one minibatch tile of the schedule; a multiple of 128, >= 128.  Tiles
 *                  never cross experts.  It sets the order in which GEMM tiles are visited (all
 *                  tiles of one minibatch are visited together, weights then stay in L2) and
 *                  whether row tiles pair up on CTA pairs (tiles of 256 rows and more); it never
 *                  changes a result.  0 = automatic: the average routed rows per expert,
 *                  ceil(T*K/E), rounded up to a power of two times 128 in [256, 2048].
 *  macrobatch_rows a multiple of minibatch_rows; each tile records first_row / macrobatch_rows.
 *                  0 = automatic: the smallest multiple of minibatch_rows that is at least
 *                  4 * minibatch_rows and 2048.  A schedule holds the resolved sizes in its copy
 *                  of the config.
 *  num_ctas        persistent grid size of the statically scheduled GEMM kernels (CTA pairs, and
 *                  every kernel under MOK_FLAG_STATIC_TILES); 0 = one CTA per SM.
 *  precision       mok_precision.
 *  debug_flags     0, or MOK_FLAG_STATIC_TILES.  By default the single-CTA GEMM kernels launch one
 *                  CTA per tile and the running CTAs take over the tiles of CTAs that have not
 *                  started (cluster launch control, "Cursor Open-Sources Mixture-of-Kittens (MoK)
 *                  ...", English summary: Cluster Launch Control scheduling); with the flag every
 *                  GEMM walks its tiles in a static round robin over a persistent grid.  Either
 *                  way each tile is computed by one CTA in a fixed K order: the same bits. */
#define MOK_FLAG_STATIC_TILES 1u
typedef struct {
  int32_t minibatch_rows;
  int32_t macrobatch_rows;
  int32_t num_ctas;
  int32_t precision;
  uint32_t debug_flags;
} mok_config;

/* T tokens, hidden size H, expert intermediate size I, E experts, top-K.
 * Supported: T >= 0; H and I multiples of 128; 1 <= K <= E <= 1024; T * K < 2^31. */
typedef struct {
  int64_t T;
  int32_t H, I, E, K;
} mok_shape;

/* Filled by mok_build_schedule: device pointers into the caller's workspace (all int32 unless
 * noted).  R = T*K routed slots, slot j = t*K + k; rows are positions in the expert-grouped
 * layout, each expert's segment padded to a multiple of 128 rows.
 *   counts[E]            slots routed to each expert
 *   offsets[E+1]         exclusive prefix sum of counts
 *   poff[E+1]            exclusive prefix sum of counts rounded up to 128 (poff[E] = Rpad)
 *   perm[rpad_max]       slot held by each row, -1 on padding rows (valid for row < Rpad)
 *   inv[R]               row holding each slot
 *   tiles[tiles_max][4]  minibatch tiles {expert, first row, valid rows, first row / MB}
 *   mblocks[mblocks_max][4]  128-row blocks {expert, first row, valid rows, tile index}
 *   meta[16]             meta[0] = Rpad, meta[1] = number of tiles, meta[2] = number of blocks,
 *                        meta[3] = number of block pairs (two consecutive 128-row blocks of one
 *                        tile, or a tile's last single block) used by the library's GEMMs
 *   row_weight[rpad_max] fp32 combine weight of each row (0 on padding rows)
 *   row_token[rpad_max]  token of each row (-1 on padding rows)
 *   status               device status word (bit (1 << mok_status code) per problem seen) */
typedef struct {
  mok_shape shape;
  mok_config config;
  int64_t rpad_max, tiles_max, mblocks_max;
  int32_t* counts;
  int32_t* offsets;
  int32_t* poff;
  int32_t* perm;
  int32_t* inv;
  int32_t* tiles;
  int32_t* mblocks;
  int32_t* meta;
  float* row_weight;
  int32_t* row_token;
  uint32_t* status;
  const float* topk_weights; /* the caller's [T, K] fp32 weights, read by the combine */
  void* ws;                  /* the workspace the schedule lives in (start of the carve) */
  size_t ws_bytes;
} mok_schedule;

/* Expert weights in the PyTorch [out, in] convention.
 * BF16 mode: w_gate, w_up [E, I, H] bf16; w_down [E, H, I] bf16.
 * MXFP8 mode (precision == MOK_MXFP8) reads only pre-quantised copies made with mok_mxfp8_quantize
 * (the project card, "Key concepts": weights are pre-quantised with ops.mxfp8_quantize), each
 * quantised along the K axis of the GEMM that consumes it:
 *   forward   q_gate, q_up [E*I, H] E4M3 + s_gate, s_up [E*I, H/32] E8M0   (Wg, Wu along H)
 *             q_down [E*H, I] + s_down [E*H, I/32]                         (Wd along I)
 *   backward  qt_gate, qt_up [E*H, I] + st_gate, st_up [E*H, I/32]          (Wg^T, Wu^T along I)
 *             qt_down [E*I, H] + st_down [E*I, H/32]                        (Wd^T along H)
 * Fields a mode does not read may be NULL. */
typedef struct {
  const void* w_gate;
  const void* w_up;
  const void* w_down;
  const uint8_t* q_gate;
  const uint8_t* s_gate;
  const uint8_t* q_up;
  const uint8_t* s_up;
  const uint8_t* q_down;
  const uint8_t* s_down;
  const uint8_t* qt_gate;
  const uint8_t* st_gate;
  const uint8_t* qt_up;
  const uint8_t* st_up;
  const uint8_t* qt_down;
  const uint8_t* st_down;
} mok_weights;

/* Gradients, overwritten (not accumulated):
 *   dx [T, H] bf16; dw_gate, dw_up [E, I, H] fp32; dw_down [E, H, I] fp32 (experts that received
 *   no slot get exact zeros); d_topk_weights [T, K] fp32 = dL/ds for the renormalised weights. */
typedef struct {
  void* dx;
  float* dw_gate;
  float* dw_up;
  float* dw_down;
  float* d_topk_weights;
} mok_grads;

/* Library version string (the project card's `mok.__version__`).  Host pointer, static. */
MOK_API const char* mok_version(void);

/* Human-readable name of a status code.  Host pointer, static. */
MOK_API const char* mok_status_string(mok_status s);

/* Bytes of device workspace needed by mok_build_schedule / mok_forward / mok_backward for this
 * shape and config (the project card's get_workspace).  0 when the arguments are invalid. */
MOK_API size_t mok_workspace_bytes(const mok_config* cfg, const mok_shape* shape);

/* Bytes of the forward context (activations saved by mok_forward for mok_backward). */
MOK_API size_t mok_fwd_ctx_bytes(const mok_config* cfg, const mok_shape* shape);

/* MXFP8 quantisation (the project card's ops.mxfp8_quantize; MXFP8 mode of "Cursor Open-Sources
 * Mixture-of-Kittens (MoK) ...", English summary).  in_bf16 [rows, cols] row-major, cols a
 * multiple of 32; out_e4m3 [rows, cols]; out_e8m0 [rows, cols/32].  Per 32 consecutive elements of
 * a row: shared = floor(log2(amax)) - 8 clamped to [-127, 127] (amax = 0 gives -127), scale byte =
 * shared + 127, element = E4M3 round-to-nearest-even of v / 2^shared saturating to +-448.  A block
 * holding NaN or Inf gets scale 0xFF and elements 0x7F.  All three pointers 16-byte aligned. */
MOK_API mok_status mok_mxfp8_quantize(const void* in_bf16, int64_t rows, int64_t cols, uint8_t* out_e4m3,
                              uint8_t* out_e8m0, void* stream);

/* Build the schedule ("Mixture-of-Kittens(MoK)란? ..." (alltoptrend), section 4 (1): one schedule
 * table drives dispatch and combine of both passes; section 4 (3): no token is dropped).
 * topk_ids [T, K] int32, topk_weights [T, K] fp32 (both device, kept by reference in *sched_out
 * and read by later calls).  ws: device workspace of at least mok_workspace_bytes bytes, 256-byte
 * aligned.  sched_out: HOST struct, filled here.  The schedule is a stable counting sort of the
 * slots by expert (ascending slot index within an expert), padded per expert to 128 rows,
 * cut into minibatch tiles. */
MOK_API mok_status mok_build_schedule(const mok_config* cfg, const mok_shape* shape, const int32_t* topk_ids,
                              const float* topk_weights, void* ws, size_t ws_bytes, mok_schedule* sched_out,
                              void* stream);

/* Forward: out[t] = sum over k ascending of s[t,k] * Wd[e] (silu(Wg[e] x[t]) * (Wu[e] x[t])),
 * e = ids[t,k], computed in fp32 on the tensor cores and rounded once to bf16 ("Cursor
 * Open-Sources Mixture-of-Kittens (MoK) ...", English summary: SwiGLU experts, BF16 / MXFP8).
 * x [T, H] bf16; out [T, H] bf16; fwd_ctx: device buffer of mok_fwd_ctx_bytes bytes that
 * mok_backward reads (gathered x, gate/up pre-activations, SwiGLU output). */
MOK_API mok_status mok_forward(const mok_schedule* sched, const void* x, const mok_weights* w, void* out, void* fwd_ctx,
                       size_t fwd_ctx_bytes, void* stream);

/* Backward for upstream gradient dy [T, H] bf16 = dL/dout.  Writes every field of *g.  The
 * router-weight gradient d_topk_weights[t,k] = <Wd[e]^T dy[t], a(t,k)> is formed inside the
 * SwiGLU backward ("Cursor Open-Sources ...", English summary: SonicMoE-style router-weight
 * gradient fused into the SwiGLU backward).  fwd_ctx must hold the matching mok_forward's
 * context; sched must be the schedule both calls used. */
MOK_API mok_status mok_backward(const mok_schedule* sched, const void* fwd_ctx, const void* dy, const mok_weights* w,
                        const mok_grads* g, void* stream);

/* Kernel-level tracing for profiling.  Every kernel the library launches while a trace is set
 * is bracketed by two cudaEventRecord calls on its stream, into caller-created events:
 *   events    HOST array of 2 * capacity cudaEvent_t handles (as void*), created by the caller
 *             (timing enabled); launch i uses events[2i] (before) and events[2i+1] (after).
 *   kinds     HOST array of capacity int32: the kernel kind of launch i (mok_kernel_name).
 *   count     launches recorded so far; the library increments it and stops at capacity.
 * Pass NULL to stop tracing.  The trace is process-wide and not thread-safe: set it only around
 * single-threaded profiling runs.  Event records add a stream operation per launch boundary. */
typedef struct {
  void** events;
  int32_t* kinds;
  int32_t capacity;
  int32_t count;
} mok_trace;

MOK_API mok_status mok_set_trace(mok_trace* trace);

/* Name of a kernel kind recorded in mok_trace.kinds (static host string; "?" when unknown). */
MOK_API const char* mok_kernel_name(int32_t kind);

/* Schedule build for callers that cannot allocate device memory.  The pages have no counterpart
 * to this call: it exists for code that may not call cudaMalloc (or any allocating routine) while
 * it runs, e.g. a runtime that only hands out fixed, pre-sized buffers.  It computes exactly the
 * tables of mok_build_schedule (for either precision: the tables do not depend on it), but its
 * scratch (the per-chunk expert histogram) lives in a fixed array inside the library: 2 MiB of
 * device memory per GPU that loads the library, held until the process exits.
 *   sched   HOST struct.  On entry the caller sets these DEVICE pointers to its own buffers:
 *           counts [E], offsets [E+1], poff [E+1], perm [rpad_max], inv [T*K], tiles
 *           [tiles_max*4], mblocks [mblocks_max*4], meta [16], row_weight [rpad_max] (fp32),
 *           row_token [rpad_max]; and rpad_max, tiles_max, mblocks_max to the capacities of those
 *           buffers.  The shape needs rpad_max >= T*K + 127*E, tiles_max >= ceil(T*K / mb) + E and
 *           mblocks_max >= floor((T*K + 127*E) / 128), mb the minibatch rows; with minibatch_rows
 *           = 0 (automatic) mb is at least 256, so tiles_max = ceil(T*K / 256) + E always
 *           suffices.  A smaller capacity gives MOK_ERR_WORKSPACE_TOO_SMALL before any work is
 *           enqueued.  The call sets the capacity fields to the sizes the shape needs and fills the
 *           remaining fields (config holds the resolved minibatch and macrobatch; status points at
 *           meta[15]; ws is NULL).  Such a schedule holds no workspace, so it serves inspection and
 *           the caller's own kernels, not mok_forward / mok_backward.
 * Limit: ceil(T*K / 512) * (E + 1) <= 524288, else MOK_ERR_UNSUPPORTED is returned before any
 * work is enqueued.  The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  All calls share the one
 * array, so calls whose work overlaps on the GPU (different streams, or different host threads)
 * race; serialise them.  Nothing needs clearing between calls: every scratch entry a call reads,
 * it has written first. */
MOK_API mok_status mok_build_schedule_noalloc(const mok_config* cfg, const mok_shape* shape,
                                              const int32_t* topk_ids, const float* topk_weights,
                                              mok_schedule* sched, void* stream);

/* The MXFP8 operand copies that mok_forward / mok_backward write, for inspection (tests,
 * debugging); the layer itself needs no call of this.  DEVICE pointers into sched->ws or fwd_ctx
 * (xr, xrs), valid while those are.  Row r of the expert-grouped layout is routed slot perm[r];
 * padding rows hold zero codes and scale byte 0.  rows = sched->rpad_max; rcap = rows rounded up
 * to a multiple of 128.
 * Quantised along each GEMM's K, row-major (forward and data-gradient GEMMs):
 *   xq  [rows, H]  E4M3 of the gathered x (blocks of 32 along H)      xs  its E8M0 scales
 *   aq  [rows, I]  E4M3 of a = silu(g) u (blocks of 32 along I)         as  its scales
 *   dyq [rows, H]  E4M3 of the gathered dY                            dys its scales
 *   dgq [rows, 2I] E4M3 of [dg | du] (blocks of 32 along I)           dgs its scales
 * Quantised along the routed rows (every column in blocks of 32 rows of the padded layout; the
 * weight-gradient GEMMs' K), stored transposed [features, rcap]:
 *   xr [H, rcap] x, dyr [H, rcap] dY, dgr [2I, rcap] [dg | du], sar [I, rcap] s * a
 * Scales are atom-tiled for the block-scaled MMA.  Row-major copies (kq = row length / 128): the
 * scale of row r, k-group g (elements 32g .. 32g+31) sits at byte
 *   ((r / 128) * kq + g / 4) * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4 + g % 4.
 * Copies quantised along the rows (column f, row block g = r / 32, kq = rcap / 128, G atoms per
 * group: 1 for dyrs and dgrs, xr_groups for xrs, sar_groups for sars):
 *   (((f / (128 G)) * kq + g / 4) * G + (f / 128) % G) * 512 + (f % 32) * 16 + ((f / 32) % 4) * 4
 *   + g % 4.
 * Returns MOK_ERR_INVALID_ARG unless sched holds a workspace built with precision MOK_MXFP8.
 * The copies hold the values of the last mok_forward (xq, aq, xr) / mok_backward (the rest). */
typedef struct {
  const uint8_t* xq;
  const uint8_t* xs;
  const uint8_t* aq;
  const uint8_t* as;
  const uint8_t* dyq;
  const uint8_t* dys;
  const uint8_t* dgq;
  const uint8_t* dgs;
  const uint8_t* xr;
  const uint8_t* xrs;
  const uint8_t* dyr;
  const uint8_t* dyrs;
  const uint8_t* dgr;
  const uint8_t* dgrs;
  const uint8_t* sar;
  const uint8_t* sars;
  int64_t rows;
  int64_t rcap;
  int32_t xr_groups;
  int32_t sar_groups;
} mok_mx_operands;

MOK_API mok_status mok_mx_operands_of(const mok_schedule* sched, const void* fwd_ctx, mok_mx_operands* out);

/* ---------------------------------------------------------------------------------------------
 * Router step (before the layer; its outputs are mok_build_schedule's inputs).  "Mixture-of-
 * Kittens (MoK)" project card, "Functional API": the schedule takes the router's top-k expert ids
 * and weights; "Cursor Open-Sources ...", English summary: the router-weight gradient is part of
 * the backward.  A linear router: logits = x W + b, W [H,E] bf16 row-major, b [E] fp32 optional.
 * Shapes: H a multiple of 128, 1 <= K <= 32, K <= E <= 1024.
 * ------------------------------------------------------------------------------------------- */

/* Bytes of device workspace mok_router_backward needs (256-byte aligned): W transposed (E*H bf16)
 * and the gradient of the chosen logits (T*K fp32).  0 for an unsupported shape. */
MOK_API size_t mok_router_workspace_bytes(const mok_shape* shape);

/* logits [T,E] fp32: logits[t,e] = (sum over h = 0 .. H-1 in ascending order of x[t,h] W[h,e],
 * one fused multiply-add per step in fp32) + b[e] (one fp32 add; bias may be NULL).  topk_ids
 * [T,K] int32: the K largest logits of each token in descending order, equal logits in ascending
 * expert id (NaN logits are never chosen; a token with fewer than K non-NaN logits gets id -1).
 * topk_weights [T,K] fp32: the softmax over the K chosen logits, which is the softmax over all E
 * renormalised to the chosen K.  x [T,H] bf16 (16-byte aligned) and W device pointers; all
 * outputs device, written in full. */
MOK_API mok_status mok_router_forward(const mok_shape* shape, const void* x, const void* w_router, const float* bias,
                                      float* logits, int32_t* topk_ids, float* topk_weights, void* stream);

/* Router backward from d_topk_weights [T,K] fp32 (mok_backward's router-weight gradient).  With
 * the forward's ids and weights: g[t,k] = w[t,k] (d[t,k] - sum_j w[t,j] d[t,j]) is the gradient of
 * the chosen logit (the others get 0).  Writes dw_router [H,E] fp32, dw[h,e] = sum over the rows
 * of expert e in the schedule's ascending order of x[token,h] g; d_bias [E] fp32 (may be NULL)
 * likewise of g; dx [T,H] bf16: dx[t,h] = (accumulate_dx ? dx[t,h] : 0) + sum over k ascending of
 * g[t,k] W[h, ids[t,k]], fp32, rounded once (accumulate_dx adds the router's share to the layer's
 * dX in place).  sched: the schedule mok_build_schedule built from these ids (its shape gives T,
 * H, E, K).  ws: device workspace of mok_router_workspace_bytes bytes, 256-byte aligned.  x 4-byte
 * and dx 16-byte aligned. */
MOK_API mok_status mok_router_backward(const mok_schedule* sched, const void* x, const void* w_router,
                                       const int32_t* topk_ids, const float* topk_weights,
                                       const float* d_topk_weights, float* dw_router, float* d_bias, void* dx,
                                       int32_t accumulate_dx, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Expert parallelism ("Mixture-of-Kittens(MoK)란? ..." (alltoptrend), section 4 (1): destination
 * ranks pull the token rows of their experts, expert outputs are pushed back to the ranks holding
 * the tokens, and the backward runs the opposite directions, all driven by one schedule table).
 * A group of `world` ranks: rank r holds tokens_per_rank tokens (the group's token t lives on rank
 * t / tokens_per_rank) and owns experts [r * E, (r + 1) * E), E = the shape's expert count per
 * rank.  Each call takes per-rank buffer tables (arrays of `world` DEVICE pointers, host arrays):
 * on one GPU every entry is local memory; across GPUs the entries for other ranks must be
 * addresses this GPU can load from and store to (peer-mapped memory).  Rows move with plain loads
 * and stores, no multicast.  Results are bitwise those of the single-rank layer on the
 * concatenated tokens and experts.  Order: every rank's mok_ep_forward, then (after all of them
 * have completed: stream order on one GPU, a group barrier across GPUs) every rank's
 * mok_ep_combine of its y rows; the same for mok_ep_backward and the dX combine.
 * ------------------------------------------------------------------------------------------- */
#define MOK_EP_MAX_RANKS 8
typedef struct {
  int32_t world;            /* ranks in the group, 1 .. MOK_EP_MAX_RANKS */
  int32_t rank;             /* this rank */
  int64_t tokens_per_rank;  /* tokens on every rank; the group's T = world * tokens_per_rank */
} mok_ep_group;

/* This rank's schedule over the group's slots (slot j = t * K + k of the group's token t).  It
 * reads every rank's routing -- topk_ids[r], topk_weights[r]: rank r's [tokens_per_rank, K] int32
 * global expert ids and fp32 weights -- and keeps the slots of its own experts; slots of other
 * ranks' experts are skipped silently, ids outside [0, world * E) set MOK_ERR_BAD_EXPERT_ID.
 * shape: T = world * tokens_per_rank, E = experts per rank.  ws as for mok_build_schedule (size
 * mok_workspace_bytes of the same shape). */
MOK_API mok_status mok_ep_build_schedule(const mok_config* cfg, const mok_shape* shape, const mok_ep_group* ep,
                                         const int32_t* const* topk_ids, const float* const* topk_weights, void* ws,
                                         size_t ws_bytes, mok_schedule* sched_out, void* stream);

/* This rank's forward: pulls the token rows of its experts from x[r] (rank r's [tokens_per_rank,
 * H] bf16), runs its experts (w: its E experts' weights, as for mok_forward), and pushes each
 * expert output row y(t, k) to the token's rank: y_recv[r] is rank r's [tokens_per_rank * K, H]
 * bf16 receive buffer, row t_local * K + k.  fwd_ctx as for mok_forward (mok_fwd_ctx_bytes). */
MOK_API mok_status mok_ep_forward(const mok_schedule* sched, const mok_ep_group* ep, const void* const* x,
                                  const mok_weights* w, void* const* y_recv, void* fwd_ctx, size_t fwd_ctx_bytes,
                                  void* stream);

/* This rank's backward: pulls dY rows of its experts' slots from dy[r] ([tokens_per_rank, H] bf16
 * per rank), writes the weight gradients of its E experts (dw_gate, dw_up [E, I, H], dw_down [E, H,
 * I] fp32, overwritten), and pushes per slot the dX row to dx_recv[r] ([tokens_per_rank * K, H] bf16,
 * row t_local * K + k) and the router-weight gradient to d_topk_weights[r] ([tokens_per_rank, K]
 * fp32).  Slots with an invalid id get dS = 0 from their token's own rank. */
MOK_API mok_status mok_ep_backward(const mok_schedule* sched, const mok_ep_group* ep, const void* fwd_ctx,
                                   const void* const* dy, const mok_weights* w, float* dw_gate, float* dw_up,
                                   float* dw_down, void* const* dx_recv, float* const* d_topk_weights,
                                   void* stream);

/* The token owner's fixed-order combine of the rows pushed to it: out[t] = sum over k ascending of
 * topk_weights[t,k] * recv[t * K + k] in fp32, rounded once to bf16, over the slots whose id lies
 * in [0, world * E) (topk_weights NULL: weight 1, the dX reduction).  topk_ids, topk_weights: this
 * rank's [tokens_per_rank, K]; recv [tokens_per_rank * K, H]; out [tokens_per_rank, H] bf16.  Only
 * shape->H, K and E are read. */
MOK_API mok_status mok_ep_combine(const mok_shape* shape, const mok_ep_group* ep, const int32_t* topk_ids,
                                  const float* topk_weights, const void* recv, void* out, void* stream);

/* Copy the schedule's device status word to *out (host pointer) after synchronising the stream.
 * The only call that blocks. */
MOK_API mok_status mok_read_device_status(const mok_schedule* sched, uint32_t* out, void* stream);

/* Failure-path self test.  Enqueues one single-thread kernel that waits, through the library's
 * bounded mbarrier wait (the one every GEMM role uses), on a barrier that nothing completes.  The
 * wait gives up at the library's deadline (2 s), ORs (1 << MOK_ERR_TIMEOUT) into *status (a device
 * word the caller owns) and the kernel returns normally, leaving the context usable.  No GPU
 * fault, trap or unbounded wait is involved. */
MOK_API mok_status mok_selftest_wait_timeout(uint32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOK_H */
