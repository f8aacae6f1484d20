// api.cu -- host implementation of include/mhc_boundary.h.
//
// Call structure ([GLM] AllReduceMhcBoundary.__call__ / join): on the
// caller's stream, the MoE fold kernel (finalize_moe) or the owner-reduce
// kernel (MHC_FLAG_OWNER_REDUCE), then the stage kernel and the finish
// kernel, both programmatic dependent launches; the finish kernel also
// computes post and the Sinkhorn mix.  With MHC_FLAG_STATIC_WEIGHT the stage
// kernel stages and splits the prenorm weight before it waits for the
// kernel ahead of it.  With MHC_FLAG_SIDE_MIXES the post / Sinkhorn
// kernel runs instead on a library side stream after an event; the next call
// (or join) waits for its completion event.  With MHC_FLAG_SYNC_MIXES that
// kernel runs on the caller's stream.  Every argument is validated before the
// first launch and a failing call leaves the handle unchanged ([DSV]
// AllReduceMHC._consumer).
//
// Pages: [GLM] vllm.models.glm5next.nvidia.specialized_decode.all_reduce_mhc,
//        [DSV] vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc.
#include <algorithm>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "launch.cuh"
#include "mhc_boundary.h"
#include "mhc_boundary_test.h"

using namespace mhc;

// mhc_boundary_run_host splits a call into up to HOST_CHUNKS_MAX token
// chunks of at least HOST_CHUNK_MIN tokens (multiples of 128, so that each
// chunk's MXFP8 scales are one contiguous run of the swizzled layout).
constexpr int HOST_CHUNKS_MAX = 8;
constexpr int HOST_CHUNK_MIN = 256;

struct mhc_boundary {
  mhc_boundary_config_t cfg;
  int device = 0;
  int slices = 0;
  int sm_count = 0;
  cudaStream_t side = nullptr;
  cudaEvent_t main_ready = nullptr;
  cudaEvent_t side_done = nullptr;
  bool side_pending = false;
  // capture id of the stream capture side_done was last recorded in (0: none);
  // a call inside a capture waits only for side kernels of the same capture
  unsigned long long side_capture = 0;
  float *mixes = nullptr;        // [cap][24] raw mixes read by the side kernel
  float *part = nullptr;         // [cap][part_row_floats(slices)] stage-kernel partial sums
  uint16_t *fold = nullptr;      // [cap][H] bf16 stage-1 sum of MoE calls (top_k > 0) or owner sums
  unsigned int *err = nullptr;   // device-detected argument errors
  // the one-kernel path for a few tokens (k_small.cu): CTAs a cluster (0: not
  // available at this shape) and clusters that run at once
  int small_cs = 0;
  int small_clusters = 0;
  unsigned char *staging = nullptr;
  size_t staging_bytes = 0;
  // mhc_boundary_run_host's pipeline: copy streams in each direction and the
  // events that hand each token chunk from copy to compute to copy
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t host_start = nullptr, host_end = nullptr;
  cudaEvent_t in_done[HOST_CHUNKS_MAX] = {}, run_done[HOST_CHUNKS_MAX] = {};
  // profiling: 6 events per recorded call (stage, finish, mixes: start/end)
  std::vector<cudaEvent_t> prof_events;
  int prof_capacity = 0;
  int prof_calls = 0;
  std::string last_error;
};

namespace {

thread_local std::string g_create_error;

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int device) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != device) cudaSetDevice(device);
  }
  ~DeviceGuard() {
    int now = -1;
    if (prev >= 0 && cudaGetDevice(&now) == cudaSuccess && now != prev) cudaSetDevice(prev);
  }
};

mhc_status_t fail(std::string &slot, mhc_status_t status, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  slot = buf;
  return status;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t scale_bytes(int32_t m, int32_t hidden) {
  if (m < 1 || hidden < 32 || hidden % 32) return 0;
  return size_t((m + 127) / 128) * 128 * size_t((hidden / 32 + 3) / 4 * 4);
}

// Checks of one call; fills msg and returns non-OK on the first problem.
mhc_status_t validate(const mhc_boundary *b, const mhc_run_args_t *a, bool moe, std::string &msg) {
  const mhc_boundary_config_t &c = b->cfg;
  if (!a) return fail(msg, MHC_ERR_INVALID_ARG, "args is NULL");
  if (a->m < 1 || a->m > c.max_num_tokens)
    return fail(msg, MHC_ERR_CAPACITY, "M=%d is outside [1, %d]", a->m, c.max_num_tokens);
  struct Need { const void *p; const char *name; size_t align; };
  const Need required[] = {
      {a->residual, "residual", 16}, {a->post, "post", 16}, {a->comb, "comb", 16},
      {a->scale, "scale", 4}, {a->base, "base", 4},
      {a->norm_weight, "norm_weight", 16}, {a->residual_out, "residual_out", 16},
      {a->layer_input, "layer_input", 16}, {a->post_out, "post_out", 4},
      {a->comb_out, "comb_out", 4}};
  for (const Need &n : required) {
    if (!n.p) return fail(msg, MHC_ERR_INVALID_ARG, "%s is NULL", n.name);
    if (!aligned(n.p, n.align))
      return fail(msg, MHC_ERR_INVALID_ARG, "%s is not %zu-byte aligned", n.name, n.align);
  }
  if ((a->hc_fn == nullptr) == (a->hc_fn_bf16 == nullptr))
    return fail(msg, MHC_ERR_INVALID_ARG, "exactly one of hc_fn and hc_fn_bf16 is required");
  if (!aligned(a->hc_fn ? static_cast<const void *>(a->hc_fn) : a->hc_fn_bf16, 16))
    return fail(msg, MHC_ERR_INVALID_ARG, "the prenorm weight is not 16-byte aligned");
  if (a->hc_fn_bf16 && !moe && c.tp > TP_TMA_MAX)
    return fail(msg, MHC_ERR_UNSUPPORTED, "hc_fn_bf16 needs tp <= %d", TP_TMA_MAX);
  if (moe) {
    if (a->partials) return fail(msg, MHC_ERR_INVALID_ARG, "partials must be NULL for finalize_moe");
  } else {
    if (!a->partials) return fail(msg, MHC_ERR_INVALID_ARG, "partials is NULL");
    if (!aligned(a->partials, 16)) return fail(msg, MHC_ERR_INVALID_ARG, "partials is not 16-byte aligned");
  }
  const Need optional[] = {{a->pre_out, "pre_out", 4}, {a->mixes_out, "mixes_out", 4},
                           {a->reduced_out, "reduced_out", 16}, {a->mxfp8_values, "mxfp8_values", 16},
                           {a->mxfp8_scales, "mxfp8_scales", 16}};
  for (const Need &n : optional)
    if (n.p && !aligned(n.p, n.align))
      return fail(msg, MHC_ERR_INVALID_ARG, "%s is not %zu-byte aligned", n.name, n.align);
  if ((a->mxfp8_values == nullptr) != (a->mxfp8_scales == nullptr))
    return fail(msg, MHC_ERR_INVALID_ARG, "mxfp8_values and mxfp8_scales are both given or both NULL");
  if (a->mxfp8_values && !(c.flags & MHC_FLAG_MXFP8))
    return fail(msg, MHC_ERR_UNSUPPORTED, "created without MHC_FLAG_MXFP8");
  return MHC_OK;
}

mhc_status_t validate_moe(const mhc_boundary *b, const mhc_moe_args_t *a, std::string &msg) {
  if (!a) return fail(msg, MHC_ERR_INVALID_ARG, "args is NULL");
  if (b->cfg.top_k < 1) return fail(msg, MHC_ERR_UNSUPPORTED, "created with top_k = 0");
  mhc_status_t s = validate(b, &a->run, true, msg);
  if (s != MHC_OK) return s;
  if (a->rows_per_rank < 1) return fail(msg, MHC_ERR_INVALID_ARG, "rows_per_rank must be >= 1");
  if (!a->routed || !a->idx || !a->weights || !a->shared)
    return fail(msg, MHC_ERR_INVALID_ARG, "routed, idx, weights and shared are required");
  if (!aligned(a->routed, 16) || !aligned(a->shared, 16))
    return fail(msg, MHC_ERR_INVALID_ARG, "routed and shared must be 16-byte aligned");
  if (!aligned(a->idx, 4) || !aligned(a->weights, 4))
    return fail(msg, MHC_ERR_INVALID_ARG, "idx and weights must be 4-byte aligned");
  return MHC_OK;
}

// Checks of one delayed-mHC consumer call.
mhc_status_t validate_consume(const mhc_boundary *b, const mhc_consume_args_t *a, std::string &msg) {
  const mhc_boundary_config_t &c = b->cfg;
  if (!a) return fail(msg, MHC_ERR_INVALID_ARG, "args is NULL");
  if (a->m < 1 || a->m > c.max_num_tokens)
    return fail(msg, MHC_ERR_CAPACITY, "M=%d is outside [1, %d]", a->m, c.max_num_tokens);
  struct Need { const void *p; const char *name; size_t align; };
  const Need required[] = {{a->residual, "residual", 16}, {a->post, "post", 16}, {a->comb, "comb", 16},
                           {a->residual_out, "residual_out", 16}};
  for (const Need &n : required) {
    if (!n.p) return fail(msg, MHC_ERR_INVALID_ARG, "%s is NULL", n.name);
    if (!aligned(n.p, n.align))
      return fail(msg, MHC_ERR_INVALID_ARG, "%s is not %zu-byte aligned", n.name, n.align);
  }
  if (a->partials) {
    if (!aligned(a->partials, 16)) return fail(msg, MHC_ERR_INVALID_ARG, "partials is not 16-byte aligned");
    if (c.tp > TP_TMA_MAX) return fail(msg, MHC_ERR_UNSUPPORTED, "the consumer needs tp <= %d", TP_TMA_MAX);
  } else {
    if (c.top_k < 1) return fail(msg, MHC_ERR_UNSUPPORTED, "no partials and created with top_k = 0");
    if (a->rows_per_rank < 1) return fail(msg, MHC_ERR_INVALID_ARG, "rows_per_rank must be >= 1");
    if (!a->routed || !a->idx || !a->weights || !a->shared)
      return fail(msg, MHC_ERR_INVALID_ARG, "the MoE fold needs routed, idx, weights and shared");
    if (!aligned(a->routed, 16) || !aligned(a->shared, 16))
      return fail(msg, MHC_ERR_INVALID_ARG, "routed and shared must be 16-byte aligned");
    if (!aligned(a->idx, 4) || !aligned(a->weights, 4))
      return fail(msg, MHC_ERR_INVALID_ARG, "idx and weights must be 4-byte aligned");
  }
  if (a->reduced_out && !aligned(a->reduced_out, 16))
    return fail(msg, MHC_ERR_INVALID_ARG, "reduced_out is not 16-byte aligned");
  if ((a->mxfp8_values == nullptr) != (a->mxfp8_scales == nullptr))
    return fail(msg, MHC_ERR_INVALID_ARG, "mxfp8_values and mxfp8_scales are both given or both NULL");
  if (!a->pre) {
    if (a->norm_weight || a->layer_input)
      return fail(msg, MHC_ERR_INVALID_ARG, "residual only (pre NULL) takes no norm_weight or layer_input");
    if (a->mxfp8_values)
      return fail(msg, MHC_ERR_INVALID_ARG, "a residual-only consumer has no layer input to quantize");
  } else {
    if (!a->norm_weight || !a->layer_input)
      return fail(msg, MHC_ERR_INVALID_ARG, "a carried pre needs norm_weight and layer_input");
    if (!aligned(a->pre, 4) || !aligned(a->norm_weight, 16) || !aligned(a->layer_input, 16))
      return fail(msg, MHC_ERR_INVALID_ARG, "pre, norm_weight or layer_input is misaligned");
    if (a->mxfp8_values && !(c.flags & MHC_FLAG_MXFP8))
      return fail(msg, MHC_ERR_UNSUPPORTED, "created without MHC_FLAG_MXFP8");
    if (a->mxfp8_values && (!aligned(a->mxfp8_values, 16) || !aligned(a->mxfp8_scales, 16)))
      return fail(msg, MHC_ERR_INVALID_ARG, "mxfp8 buffers must be 16-byte aligned");
  }
  return MHC_OK;
}

// The id of the capture `stream` is recording into, 0 when it is not capturing.
cudaError_t capture_id(cudaStream_t stream, unsigned long long *id) {
  cudaStreamCaptureStatus status = cudaStreamCaptureStatusNone;
  *id = 0;
  const cudaError_t e = cudaStreamGetCaptureInfo(stream, &status, id);
  if (status != cudaStreamCaptureStatusActive) *id = 0;
  return e;
}

// Whether work on a stream in capture `capture` (0: none) must wait for the
// last side kernel: always outside a capture, unless that kernel was itself
// captured (a graph orders its own side branch); inside a capture only when
// it was recorded in the same capture (an earlier eager call must have been
// joined before the capture began).
bool side_join_needed(const mhc_boundary *b, unsigned long long capture) {
  if (!b->side_pending) return false;
  return capture == 0 ? b->side_capture == 0 : b->side_capture == capture;
}

// Clusters the one-kernel path runs a call of m tokens on (with `tp`
// partials a token after any fold or owner reduce), or 0 for the stage and
// finish kernels: every token's cluster share within the tokens a cluster
// takes at this shape, all clusters running at once.
int small_clusters_for(const mhc_boundary *b, int m, int tp) {
  if (b->small_cs == 0 || m > SMALL_M_MAX) return 0;
  const int b_max = small_tokens_max(b->cfg.hidden, tp, b->small_cs);
  // a token a cluster up to four tokens, then two a cluster: from five
  // tokens on, fewer clusters leave the next call room to start beside this
  // one (measured at eight tokens: 9.4 us a call against 9.9 us with a token
  // a cluster, and against 9.9 us for the stage and finish kernels; at 12
  // tokens six clusters take 9.3 us)
  int clusters = m <= 4 ? m : (m + 1) / 2;
  if (clusters > b->small_clusters) clusters = b->small_clusters;
  if (b_max < 1 || clusters < 1 || (m + clusters - 1) / clusters > b_max) return 0;
  return clusters;
}

mhc_status_t launch_call(mhc_boundary *b, const mhc_run_args_t *a, const mhc_moe_args_t *moe,
                         cudaStream_t stream) {
  const mhc_boundary_config_t &c = b->cfg;
  unsigned long long capture = 0;
  cudaError_t e = capture_id(stream, &capture);
  if (e == cudaSuccess && side_join_needed(b, capture)) e = cudaStreamWaitEvent(stream, b->side_done, 0);
  if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "join: %s", cudaGetErrorString(e));
  cudaEvent_t *ev = nullptr;   // 6 events of this call when profiling (never inside a capture)
  if (capture == 0 && b->prof_calls < b->prof_capacity) ev = &b->prof_events[size_t(b->prof_calls) * 6];
  const bool sync_mixes = (c.flags & MHC_FLAG_SYNC_MIXES) != 0;
  if (ev) cudaEventRecord(ev[0], stream);

  StageParams sp = {};
  sp.m = a->m;
  sp.hidden = c.hidden;
  sp.tp = c.tp;
  sp.partials = static_cast<const uint16_t *>(a->partials);
  if (moe) {
    // stage 1 of a MoE call: the fold kernel writes y, which the
    // tensor-core stage kernel then takes as its single partial
    FoldParams fo = {};
    fo.m = a->m;
    fo.hidden = c.hidden;
    fo.tp = c.tp;
    fo.top_k = c.top_k;
    fo.rows_per_rank = moe->rows_per_rank;
    fo.routed = static_cast<const uint16_t *>(moe->routed);
    fo.idx = moe->idx;
    fo.weights = moe->weights;
    fo.shared = static_cast<const uint16_t *>(moe->shared);
    fo.y = b->fold;
    fo.err = b->err;
    e = launch_moe_fold(fo, b->sm_count, stream);
    if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "MoE fold kernel: %s", cudaGetErrorString(e));
    sp.tp = 1;
    sp.partials = b->fold;
  } else if (c.flags & MHC_FLAG_OWNER_REDUCE) {
    // two-shot reduction: the owners' sums, then the stage kernel takes
    // them as its single partial
    const OwnerParams op = {a->m, c.hidden, c.tp, static_cast<const uint16_t *>(a->partials), b->fold};
    e = launch_owner_reduce(op, b->sm_count * 16, stream);
    if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "owner reduce kernel: %s", cudaGetErrorString(e));
    sp.tp = 1;
    sp.partials = b->fold;
  }
  // post / Sinkhorn: in the boundary's own kernels (default), or a separate
  // kernel on the side stream ([GLM] design) or on the caller's stream
  const bool separate = (c.flags & (MHC_FLAG_SIDE_MIXES | MHC_FLAG_SYNC_MIXES)) != 0;
  const bool on_side = separate && !sync_mixes;
  // a few tokens: the whole boundary in one kernel of CTA clusters
  const int clusters = small_clusters_for(b, a->m, sp.tp);
  if (clusters > 0) {
    SmallParams q = {};
    q.m = a->m;
    q.hidden = c.hidden;
    q.tp = sp.tp;
    q.cs = b->small_cs;
    q.cols_max = small_cols_max(c.hidden, b->small_cs);
    q.partials = sp.partials;
    q.residual = static_cast<const uint16_t *>(a->residual);
    q.post = a->post;
    q.comb = a->comb;
    q.hc_fn = a->hc_fn;
    q.hc_fn_bf16 = static_cast<const uint16_t *>(a->hc_fn_bf16);
    q.scale = a->scale;
    q.base = a->base;
    q.gamma = static_cast<const uint16_t *>(a->norm_weight);
    q.early_weight = (c.flags & MHC_FLAG_STATIC_WEIGHT) != 0;
    q.rms_eps = c.rms_eps;
    q.hc_eps = c.hc_eps;
    q.norm_eps = c.norm_eps;
    q.post_mult = c.post_mult;
    q.repeat = c.sinkhorn_repeat;
    q.residual_out = static_cast<uint16_t *>(a->residual_out);
    q.reduced_out = static_cast<uint16_t *>(a->reduced_out);
    q.layer_input = static_cast<uint16_t *>(a->layer_input);
    q.mixes = separate ? b->mixes : nullptr;
    q.mixes_out = a->mixes_out;
    q.pre_out = a->pre_out;
    q.post_out = separate ? nullptr : a->post_out;
    q.comb_out = separate ? nullptr : a->comb_out;
    q.mx_values = a->mxfp8_values;
    q.mx_scales = a->mxfp8_scales;
    q.err = b->err;
    e = launch_small(q, clusters, stream);
    if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "boundary kernel: %s", cudaGetErrorString(e));
    if (ev) {
      cudaEventRecord(ev[1], stream);
      cudaEventRecord(ev[2], stream);
      cudaEventRecord(ev[3], stream);
    }
  } else {
    // partial-sum groups: 64-column slices (CUDA-core kernel) or 128-column
    // groups (tensor-core kernel); the scratch holds the larger count
    const bool tc_path = sp.tp <= TP_TMA_MAX;
    int stage_grid = 0;   // CTAs of the tensor-core stage kernel
    sp.slices = tc_path ? (c.hidden + TC_GROUP_COLS - 1) / TC_GROUP_COLS : b->slices;
    sp.residual = static_cast<const uint16_t *>(a->residual);
    sp.post = a->post;
    sp.comb = a->comb;
    sp.hc_fn = a->hc_fn;
    sp.hc_fn_bf16 = static_cast<const uint16_t *>(a->hc_fn_bf16);
    sp.fn_terms = a->hc_fn_bf16 ? 1 : 3;
    sp.early_weight = (c.flags & MHC_FLAG_STATIC_WEIGHT) != 0;
    sp.residual_out = static_cast<uint16_t *>(a->residual_out);
    sp.reduced_out = static_cast<uint16_t *>(a->reduced_out);
    sp.part = b->part;
    sp.part_stride = part_row_floats(sp.slices);
    sp.err = b->err;
    e = tc_path ? launch_stage_tc(sp, b->sm_count, stream, &stage_grid) : launch_stage(sp, stream);
    if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "stage kernel: %s", cudaGetErrorString(e));
    if (ev) {
      cudaEventRecord(ev[1], stream);
      cudaEventRecord(ev[2], stream);
    }

    FinishParams fp = {};
    fp.m = a->m;
    fp.hidden = c.hidden;
    fp.slices = sp.slices;
    fp.part = b->part;
    fp.part_stride = sp.part_stride;
    fp.err = b->err;
    fp.scale = a->scale;
    fp.base = a->base;
    fp.gamma = static_cast<const uint16_t *>(a->norm_weight);
    fp.streams = static_cast<const uint16_t *>(a->residual_out);
    fp.rms_eps = c.rms_eps;
    fp.hc_eps = c.hc_eps;
    fp.norm_eps = c.norm_eps;
    fp.mixes = separate ? b->mixes : nullptr;
    fp.mixes_out = a->mixes_out;
    fp.pre_out = a->pre_out;
    fp.post_out = separate ? nullptr : a->post_out;
    fp.comb_out = separate ? nullptr : a->comb_out;
    fp.post_mult = c.post_mult;
    fp.repeat = c.sinkhorn_repeat;
    fp.layer_input = static_cast<uint16_t *>(a->layer_input);
    fp.mx_values = a->mxfp8_values;
    fp.mx_scales = a->mxfp8_scales;
    e = launch_finish(fp, b->sm_count, stream, ev == nullptr, stage_grid);
    if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "finish kernel: %s", cudaGetErrorString(e));
    if (ev) cudaEventRecord(ev[3], stream);
  }

  if (separate) {
    MixesParams mp = {};
    mp.m = a->m;
    mp.repeat = c.sinkhorn_repeat;
    mp.mixes = b->mixes;
    mp.scale = a->scale;
    mp.base = a->base;
    mp.post_mult = c.post_mult;
    mp.eps = c.hc_eps;
    mp.post_out = a->post_out;
    mp.comb_out = a->comb_out;
    cudaStream_t mix_stream = on_side ? b->side : stream;
    if (on_side) {
      e = cudaEventRecord(b->main_ready, stream);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(b->side, b->main_ready, 0);
    }
    if (e == cudaSuccess && ev) e = cudaEventRecord(ev[4], mix_stream);
    if (e == cudaSuccess) e = launch_mixes(mp, mix_stream);
    if (e == cudaSuccess && ev) e = cudaEventRecord(ev[5], mix_stream);
    if (e == cudaSuccess && on_side) e = cudaEventRecord(b->side_done, mix_stream);
    if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "mixes kernel: %s", cudaGetErrorString(e));
  } else if (ev) {
    // no separate mixes kernel: its profiled time is zero
    cudaEventRecord(ev[4], stream);
    cudaEventRecord(ev[5], stream);
  }
  if (ev) ++b->prof_calls;
  if (on_side) {
    b->side_pending = true;
    b->side_capture = capture;
  }
  b->last_error.clear();
  return MHC_OK;
}

// One delayed-mHC consumer call: the optional MoE fold, the stage kernel
// without its GEMV, and (unless residual only) the finish kernel with the
// carried pre-mix, all on `stream`.
mhc_status_t consume_call(mhc_boundary *b, const mhc_consume_args_t *a, cudaStream_t stream) {
  const mhc_boundary_config_t &c = b->cfg;
  unsigned long long capture = 0;
  cudaError_t e = capture_id(stream, &capture);
  if (e == cudaSuccess && side_join_needed(b, capture)) e = cudaStreamWaitEvent(stream, b->side_done, 0);
  if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "join: %s", cudaGetErrorString(e));
  StageParams sp = {};
  sp.m = a->m;
  sp.hidden = c.hidden;
  sp.tp = c.tp;
  sp.partials = static_cast<const uint16_t *>(a->partials);
  if (!a->partials) {
    FoldParams fo = {};
    fo.m = a->m;
    fo.hidden = c.hidden;
    fo.tp = c.tp;
    fo.top_k = c.top_k;
    fo.rows_per_rank = a->rows_per_rank;
    fo.routed = static_cast<const uint16_t *>(a->routed);
    fo.idx = a->idx;
    fo.weights = a->weights;
    fo.shared = static_cast<const uint16_t *>(a->shared);
    fo.y = b->fold;
    fo.err = b->err;
    e = launch_moe_fold(fo, b->sm_count, stream);
    if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "MoE fold kernel: %s", cudaGetErrorString(e));
    sp.tp = 1;
    sp.partials = b->fold;
  } else if (c.flags & MHC_FLAG_OWNER_REDUCE) {
    const OwnerParams op = {a->m, c.hidden, c.tp, static_cast<const uint16_t *>(a->partials), b->fold};
    e = launch_owner_reduce(op, b->sm_count * 16, stream);
    if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "owner reduce kernel: %s", cudaGetErrorString(e));
    sp.tp = 1;
    sp.partials = b->fold;
  }
  // a few tokens: the consumer in one kernel of CTA clusters.  Without a
  // carried pre (the streams only) the stage kernel alone is the lighter
  // path from eight tokens on (H = 6144 tp = 8, graph replay: 3.4 us a call
  // against 4.1 at eight tokens, 3.5 against 4.4 at twelve; the one kernel
  // is faster by 0.4-0.7 us up to four tokens); with a carried pre the one
  // kernel is faster by 0.8-3 us up to twelve tokens
  const int clusters = a->pre || a->m <= 4 ? small_clusters_for(b, a->m, sp.tp) : 0;
  if (clusters > 0) {
    SmallParams q = {};
    q.m = a->m;
    q.hidden = c.hidden;
    q.tp = sp.tp;
    q.cs = b->small_cs;
    q.cols_max = small_cols_max(c.hidden, b->small_cs);
    q.partials = sp.partials;
    q.residual = static_cast<const uint16_t *>(a->residual);
    q.post = a->post;
    q.comb = a->comb;
    q.consume = 1;
    q.pre_in = a->pre;
    q.gamma = static_cast<const uint16_t *>(a->norm_weight);
    q.rms_eps = c.rms_eps;
    q.hc_eps = c.hc_eps;
    q.norm_eps = c.norm_eps;
    q.post_mult = c.post_mult;
    q.repeat = c.sinkhorn_repeat;
    q.residual_out = static_cast<uint16_t *>(a->residual_out);
    q.reduced_out = static_cast<uint16_t *>(a->reduced_out);
    q.layer_input = a->pre ? static_cast<uint16_t *>(a->layer_input) : nullptr;
    q.mx_values = a->pre ? a->mxfp8_values : nullptr;
    q.mx_scales = a->pre ? a->mxfp8_scales : nullptr;
    q.err = b->err;
    e = launch_small(q, clusters, stream);
    if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "consumer kernel: %s", cudaGetErrorString(e));
    b->last_error.clear();
    return MHC_OK;
  }
  sp.slices = (c.hidden + TC_GROUP_COLS - 1) / TC_GROUP_COLS;
  sp.residual = static_cast<const uint16_t *>(a->residual);
  sp.post = a->post;
  sp.comb = a->comb;
  sp.fn_terms = 0;   // no GEMV
  sp.residual_out = static_cast<uint16_t *>(a->residual_out);
  sp.reduced_out = static_cast<uint16_t *>(a->reduced_out);
  sp.part = b->part;
  sp.part_stride = part_row_floats(sp.slices);
  sp.err = b->err;
  int stage_grid = 0;
  e = launch_stage_tc(sp, b->sm_count, stream, &stage_grid);
  if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "stage kernel: %s", cudaGetErrorString(e));
  if (a->pre) {
    FinishParams fp = {};
    fp.m = a->m;
    fp.hidden = c.hidden;
    fp.slices = 0;
    fp.part_stride = 0;
    fp.gamma = static_cast<const uint16_t *>(a->norm_weight);
    fp.streams = static_cast<const uint16_t *>(a->residual_out);
    fp.norm_eps = c.norm_eps;
    fp.pre_in = a->pre;
    fp.layer_input = static_cast<uint16_t *>(a->layer_input);
    fp.mx_values = a->mxfp8_values;
    fp.mx_scales = a->mxfp8_scales;
    fp.err = b->err;
    e = launch_finish(fp, b->sm_count, stream, true, stage_grid);
    if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "finish kernel: %s", cudaGetErrorString(e));
  }
  b->last_error.clear();
  return MHC_OK;
}

// Staging layout for mhc_boundary_run_host: every tensor at 256-byte offsets.
struct Staging {
  size_t partials, residual, post, comb, hc_fn, scale, base, gamma;
  size_t residual_out, layer_input, post_out, comb_out, pre_out, mixes_out, reduced_out;
  size_t mx_values, mx_scales, total;
};

Staging staging_layout(const mhc_boundary_config_t &c) {
  const size_t cap = size_t(c.max_num_tokens), H = size_t(c.hidden);
  Staging s = {};
  size_t off = 0;
  auto take = [&off](size_t bytes) {
    const size_t at = off;
    off += (bytes + 255) / 256 * 256;
    return at;
  };
  s.partials = take(size_t(c.tp) * cap * H * 2);
  s.residual = take(cap * HC * H * 2);
  s.post = take(cap * HC * 4);
  s.comb = take(cap * HC * HC * 4);
  s.hc_fn = take(HC * H * MIX * 4);
  s.scale = take(3 * 4);
  s.base = take(MIX * 4);
  s.gamma = take(H * 2);
  s.residual_out = take(cap * HC * H * 2);
  s.layer_input = take(cap * H * 2);
  s.post_out = take(cap * HC * 4);
  s.comb_out = take(cap * HC * HC * 4);
  s.pre_out = take(cap * HC * 4);
  s.mixes_out = take(cap * MIX * 4);
  s.reduced_out = take(cap * H * 2);
  const bool mx = (c.flags & MHC_FLAG_MXFP8) != 0;
  s.mx_values = take(mx ? cap * H : 0);
  s.mx_scales = take(mx ? scale_bytes(c.max_num_tokens, c.hidden) : 0);
  s.total = off;
  return s;
}

void destroy_profile_events(mhc_boundary *b) {
  for (cudaEvent_t ev : b->prof_events)
    if (ev) cudaEventDestroy(ev);
  b->prof_events.clear();
  b->prof_capacity = 0;
  b->prof_calls = 0;
}

void release(mhc_boundary *b) {
  if (b->side) cudaStreamSynchronize(b->side);
  destroy_profile_events(b);
  if (b->staging) cudaFree(b->staging);
  for (int k = 0; k < HOST_CHUNKS_MAX; ++k) {
    if (b->in_done[k]) cudaEventDestroy(b->in_done[k]);
    if (b->run_done[k]) cudaEventDestroy(b->run_done[k]);
  }
  if (b->host_start) cudaEventDestroy(b->host_start);
  if (b->host_end) cudaEventDestroy(b->host_end);
  if (b->h2d) cudaStreamDestroy(b->h2d);
  if (b->d2h) cudaStreamDestroy(b->d2h);
  if (b->mixes) cudaFree(b->mixes);
  if (b->part) cudaFree(b->part);
  if (b->fold) cudaFree(b->fold);
  if (b->err) cudaFree(b->err);
  if (b->main_ready) cudaEventDestroy(b->main_ready);
  if (b->side_done) cudaEventDestroy(b->side_done);
  if (b->side) cudaStreamDestroy(b->side);
}

}  // namespace

extern "C" {

mhc_status_t mhc_boundary_create(const mhc_boundary_config_t *config, int device, mhc_boundary_t **out) {
  g_create_error.clear();
  if (!config || !out) return fail(g_create_error, MHC_ERR_INVALID_ARG, "config and out are required");
  const mhc_boundary_config_t &c = *config;
  if (c.hc_mult != HC) return fail(g_create_error, MHC_ERR_UNSUPPORTED, "hc_mult must be 4 (24 mixes = 2*hc + hc*hc)");
  if (c.hidden <= 0 || c.hidden % VEC)
    return fail(g_create_error, MHC_ERR_INVALID_ARG, "hidden must be a positive multiple of 8");
  if (c.hidden > MAX_HIDDEN) return fail(g_create_error, MHC_ERR_UNSUPPORTED, "hidden > %d", MAX_HIDDEN);
  if (c.tp < 1 || c.tp > 32) return fail(g_create_error, MHC_ERR_INVALID_ARG, "tp must be in [1, 32]");
  if (c.max_num_tokens < 1 || c.max_num_tokens > (1 << 20))
    return fail(g_create_error, MHC_ERR_INVALID_ARG, "max_num_tokens must be in [1, 2^20]");
  if (c.sinkhorn_repeat < 1 || c.sinkhorn_repeat > 10000)
    return fail(g_create_error, MHC_ERR_INVALID_ARG, "sinkhorn_repeat must be in [1, 10000]");
  if (c.top_k < 0 || c.top_k > 64) return fail(g_create_error, MHC_ERR_INVALID_ARG, "top_k must be in [0, 64]");
  if ((c.flags & MHC_FLAG_MXFP8) && c.hidden % 128)
    return fail(g_create_error, MHC_ERR_INVALID_ARG, "MXFP8 output needs hidden %% 128 == 0");
  if (c.flags & ~uint32_t(MHC_FLAG_MXFP8 | MHC_FLAG_SYNC_MIXES | MHC_FLAG_HOST_STAGING | MHC_FLAG_SIDE_MIXES |
                          MHC_FLAG_STATIC_WEIGHT | MHC_FLAG_OWNER_REDUCE))
    return fail(g_create_error, MHC_ERR_INVALID_ARG, "unknown flag bits 0x%x", c.flags);
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || device < 0 || device >= count)
    return fail(g_create_error, MHC_ERR_CUDA, "device %d is not available", device);

  DeviceGuard guard(device);
  mhc_boundary *b = new (std::nothrow) mhc_boundary();
  if (!b) return fail(g_create_error, MHC_ERR_OOM, "host allocation failed");
  b->cfg = c;
  b->device = device;
  b->slices = (c.hidden + SLICE - 1) / SLICE;
  const size_t cap = size_t(c.max_num_tokens);
  cudaError_t e = stage_set_attributes();
  if (e == cudaSuccess) e = stage_tc_set_attributes();
  if (e == cudaSuccess) e = finish_set_attributes();
  if (e == cudaSuccess) e = small_set_attributes();
  if (e == cudaSuccess) e = moe_fold_set_attributes();
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&b->sm_count, cudaDevAttrMultiProcessorCount, device);
  if (e == cudaSuccess) {
    // the one-kernel path: 16-CTA clusters where they fit at this shape, else 8
    for (int cs : {16, 8}) {
      const int b_max = small_tokens_max(c.hidden, c.tp, cs);
      if (b_max < 1) continue;
      const int n = small_active_clusters(cs, small_smem_bytes(c.hidden, c.tp, cs, b_max));
      if (n >= 1) {
        b->small_cs = cs;
        b->small_clusters = n;
        break;
      }
    }
  }
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&b->side, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&b->main_ready, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&b->side_done, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    release(b);
    delete b;
    return fail(g_create_error, MHC_ERR_CUDA, "create: %s", cudaGetErrorString(e));
  }
  e = cudaMalloc(&b->mixes, cap * MIX * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&b->part, cap * part_row_floats(b->slices) * sizeof(float));
  if (e == cudaSuccess && (c.top_k > 0 || (c.flags & MHC_FLAG_OWNER_REDUCE)))
    e = cudaMalloc(&b->fold, cap * size_t(c.hidden) * 2);
  if (e == cudaSuccess) e = cudaMalloc(&b->err, sizeof(unsigned int));
  if (e == cudaSuccess) e = cudaMemset(b->err, 0, sizeof(unsigned int));
  if (e == cudaSuccess && (c.flags & MHC_FLAG_HOST_STAGING)) {
    b->staging_bytes = staging_layout(c).total;
    e = cudaMalloc(&b->staging, b->staging_bytes);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&b->h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&b->d2h, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&b->host_start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&b->host_end, cudaEventDisableTiming);
    for (int k = 0; k < HOST_CHUNKS_MAX && e == cudaSuccess; ++k) {
      e = cudaEventCreateWithFlags(&b->in_done[k], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&b->run_done[k], cudaEventDisableTiming);
    }
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    const mhc_status_t s = e == cudaErrorMemoryAllocation ? MHC_ERR_OOM : MHC_ERR_CUDA;
    cudaGetLastError();
    release(b);
    delete b;
    return fail(g_create_error, s, "create: %s", cudaGetErrorString(e));
  }
  *out = b;
  return MHC_OK;
}

mhc_status_t mhc_boundary_run(mhc_boundary_t *b, const mhc_run_args_t *args, mhc_stream_t stream) {
  if (!b) return MHC_ERR_INVALID_ARG;
  std::string msg;
  const mhc_status_t s = validate(b, args, false, msg);
  if (s != MHC_OK) {
    b->last_error = msg;
    return s;
  }
  DeviceGuard guard(b->device);
  return launch_call(b, args, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

mhc_status_t mhc_boundary_finalize_moe(mhc_boundary_t *b, const mhc_moe_args_t *args, mhc_stream_t stream) {
  if (!b) return MHC_ERR_INVALID_ARG;
  std::string msg;
  const mhc_status_t s = validate_moe(b, args, msg);
  if (s != MHC_OK) {
    b->last_error = msg;
    return s;
  }
  DeviceGuard guard(b->device);
  return launch_call(b, &args->run, args, reinterpret_cast<cudaStream_t>(stream));
}

mhc_status_t mhc_boundary_consume(mhc_boundary_t *b, const mhc_consume_args_t *args, mhc_stream_t stream) {
  if (!b) return MHC_ERR_INVALID_ARG;
  std::string msg;
  const mhc_status_t s = validate_consume(b, args, msg);
  if (s != MHC_OK) {
    b->last_error = msg;
    return s;
  }
  DeviceGuard guard(b->device);
  return consume_call(b, args, reinterpret_cast<cudaStream_t>(stream));
}

mhc_status_t mhc_boundary_join(mhc_boundary_t *b, mhc_stream_t stream) {
  if (!b) return MHC_ERR_INVALID_ARG;
  if (!b->side_pending) return MHC_OK;
  DeviceGuard guard(b->device);
  unsigned long long capture = 0;
  cudaError_t e = capture_id(reinterpret_cast<cudaStream_t>(stream), &capture);
  if (e == cudaSuccess && side_join_needed(b, capture))
    e = cudaStreamWaitEvent(reinterpret_cast<cudaStream_t>(stream), b->side_done, 0);
  if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "join: %s", cudaGetErrorString(e));
  return MHC_OK;
}

mhc_status_t mhc_boundary_run_host(mhc_boundary_t *b, const mhc_run_args_t *host, mhc_stream_t stream_) {
  if (!b) return MHC_ERR_INVALID_ARG;
  if (!b->staging)
    return fail(b->last_error, MHC_ERR_UNSUPPORTED, "created without MHC_FLAG_HOST_STAGING");
  if (!host) return fail(b->last_error, MHC_ERR_INVALID_ARG, "args is NULL");
  const mhc_boundary_config_t &c = b->cfg;
  const Staging L = staging_layout(c);
  unsigned char *base = b->staging;
  const int m = host->m;
  const size_t M = size_t(m), H = size_t(c.hidden);
  // the device view of the call: staging buffers wherever the caller asked
  mhc_run_args_t d = {};
  d.m = m;
  d.partials = host->partials ? base + L.partials : nullptr;
  d.residual = host->residual ? base + L.residual : nullptr;
  d.post = host->post ? reinterpret_cast<float *>(base + L.post) : nullptr;
  d.comb = host->comb ? reinterpret_cast<float *>(base + L.comb) : nullptr;
  d.hc_fn = host->hc_fn ? reinterpret_cast<float *>(base + L.hc_fn) : nullptr;
  d.hc_fn_bf16 = host->hc_fn_bf16 ? static_cast<const void *>(base + L.hc_fn) : nullptr;
  d.scale = host->scale ? reinterpret_cast<float *>(base + L.scale) : nullptr;
  d.base = host->base ? reinterpret_cast<float *>(base + L.base) : nullptr;
  d.norm_weight = host->norm_weight ? base + L.gamma : nullptr;
  d.residual_out = host->residual_out ? base + L.residual_out : nullptr;
  d.layer_input = host->layer_input ? base + L.layer_input : nullptr;
  d.post_out = host->post_out ? reinterpret_cast<float *>(base + L.post_out) : nullptr;
  d.comb_out = host->comb_out ? reinterpret_cast<float *>(base + L.comb_out) : nullptr;
  d.pre_out = host->pre_out ? reinterpret_cast<float *>(base + L.pre_out) : nullptr;
  d.mixes_out = host->mixes_out ? reinterpret_cast<float *>(base + L.mixes_out) : nullptr;
  d.reduced_out = host->reduced_out ? base + L.reduced_out : nullptr;
  d.mxfp8_values = host->mxfp8_values ? base + L.mx_values : nullptr;
  d.mxfp8_scales = host->mxfp8_scales ? base + L.mx_scales : nullptr;
  std::string msg;
  mhc_status_t s = validate(b, &d, false, msg);
  if (s != MHC_OK) {
    b->last_error = msg;
    return s;
  }
  DeviceGuard guard(b->device);
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  // Token chunks: chunk k's inputs go up on the h2d stream, its kernels run on
  // `stream` once they are there, and its outputs come back on the d2h
  // stream once the kernels are done, so the copies of one chunk overlap the
  // kernels and the opposite-direction copies of its neighbours.  Chunk k
  // uses its own part of every staging buffer ([tp][mc][H] partials at tp *
  // t0 * H, the other tensors at their token offset), so no chunk waits for
  // another's buffers.
  const int n_chunks = std::max(1, std::min(HOST_CHUNKS_MAX, m / HOST_CHUNK_MIN));
  const int per_chunk = (m + n_chunks - 1) / n_chunks;
  const int chunk = n_chunks == 1 ? m : (per_chunk + 127) / 128 * 128;
  // chunk k: tokens [t0s[k], t0s[k] + mcs[k]); a tail under 128 tokens joins
  // the chunk before it, so that every chunk takes the same kernels as the
  // whole call would
  int t0s[HOST_CHUNKS_MAX], mcs[HOST_CHUNKS_MAX], nk = 0;
  for (int t0 = 0; t0 < m && nk < HOST_CHUNKS_MAX; t0 += mcs[nk++]) {
    t0s[nk] = t0;
    mcs[nk] = std::min(chunk, m - t0);
    if (m - (t0 + mcs[nk]) < 128 || nk == HOST_CHUNKS_MAX - 1) mcs[nk] = m - t0;
  }
  const int tp = c.tp;
  auto ptr = [](const void *p, size_t off) -> const unsigned char * {
    return p ? static_cast<const unsigned char *>(p) + off : nullptr;
  };
  auto mptr = [](void *p, size_t off) -> unsigned char * {
    return p ? static_cast<unsigned char *>(p) + off : nullptr;
  };
  cudaError_t e = cudaEventRecord(b->host_start, stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(b->h2d, b->host_start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(b->d2h, b->host_start, 0);
  // the call's weights once, before the first chunk's inputs
  struct Copy { void *dst; const void *src; size_t bytes; };
  const Copy weights[] = {
      {base + L.hc_fn, host->hc_fn ? static_cast<const void *>(host->hc_fn) : host->hc_fn_bf16,
       size_t(HC) * H * MIX * (host->hc_fn ? 4 : 2)},
      {base + L.scale, host->scale, 3 * 4},
      {base + L.base, host->base, MIX * 4},
      {base + L.gamma, host->norm_weight, H * 2}};
  for (const Copy &x : weights)
    if (e == cudaSuccess && x.src) e = cudaMemcpyAsync(x.dst, x.src, x.bytes, cudaMemcpyHostToDevice, b->h2d);
  for (int k = 0; k < nk && e == cudaSuccess; ++k) {
    const size_t T0 = size_t(t0s[k]), MC = size_t(mcs[k]);
    // partials: tp row runs of mc x H, one 2-D copy (host rows m x H apart)
    if (host->partials)
      e = cudaMemcpy2DAsync(base + L.partials + size_t(tp) * T0 * H * 2, MC * H * 2,
                            ptr(host->partials, T0 * H * 2), M * H * 2, MC * H * 2, size_t(tp),
                            cudaMemcpyHostToDevice, b->h2d);
    const Copy in[] = {{base + L.residual + T0 * HC * H * 2, ptr(host->residual, T0 * HC * H * 2), MC * HC * H * 2},
                       {base + L.post + T0 * HC * 4, ptr(host->post, T0 * HC * 4), MC * HC * 4},
                       {base + L.comb + T0 * HC * HC * 4, ptr(host->comb, T0 * HC * HC * 4), MC * HC * HC * 4}};
    for (const Copy &x : in)
      if (e == cudaSuccess && x.src) e = cudaMemcpyAsync(x.dst, x.src, x.bytes, cudaMemcpyHostToDevice, b->h2d);
    if (e == cudaSuccess) e = cudaEventRecord(b->in_done[k], b->h2d);
  }
  if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "host to device copy: %s", cudaGetErrorString(e));
  for (int k = 0; k < nk; ++k) {
    const size_t T0 = size_t(t0s[k]);
    mhc_run_args_t dk = d;
    dk.m = mcs[k];
    dk.partials = mptr(const_cast<void *>(d.partials), size_t(tp) * T0 * H * 2);
    dk.residual = mptr(const_cast<void *>(d.residual), T0 * HC * H * 2);
    dk.post = reinterpret_cast<float *>(mptr(const_cast<float *>(d.post), T0 * HC * 4));
    dk.comb = reinterpret_cast<float *>(mptr(const_cast<float *>(d.comb), T0 * HC * HC * 4));
    dk.residual_out = mptr(d.residual_out, T0 * HC * H * 2);
    dk.layer_input = mptr(d.layer_input, T0 * H * 2);
    dk.post_out = reinterpret_cast<float *>(mptr(d.post_out, T0 * HC * 4));
    dk.comb_out = reinterpret_cast<float *>(mptr(d.comb_out, T0 * HC * HC * 4));
    dk.pre_out = reinterpret_cast<float *>(mptr(d.pre_out, T0 * HC * 4));
    dk.mixes_out = reinterpret_cast<float *>(mptr(d.mixes_out, T0 * MIX * 4));
    dk.reduced_out = mptr(d.reduced_out, T0 * H * 2);
    dk.mxfp8_values = reinterpret_cast<uint8_t *>(mptr(d.mxfp8_values, T0 * H));
    dk.mxfp8_scales = reinterpret_cast<uint8_t *>(mptr(d.mxfp8_scales, T0 * (H / 32)));
    e = cudaStreamWaitEvent(stream, b->in_done[k], 0);
    if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "copy wait: %s", cudaGetErrorString(e));
    s = launch_call(b, &dk, nullptr, stream);
    if (s != MHC_OK) return s;
    if (b->side_pending) e = cudaStreamWaitEvent(stream, b->side_done, 0);
    if (e == cudaSuccess) e = cudaEventRecord(b->run_done[k], stream);
    if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "chunk event: %s", cudaGetErrorString(e));
  }
  for (int k = 0; k < nk && e == cudaSuccess; ++k) {
    const size_t T0 = size_t(t0s[k]), MC = size_t(mcs[k]);
    e = cudaStreamWaitEvent(b->d2h, b->run_done[k], 0);
    const Copy out[] = {
        {mptr(host->residual_out, T0 * HC * H * 2), ptr(d.residual_out, T0 * HC * H * 2), MC * HC * H * 2},
        {mptr(host->layer_input, T0 * H * 2), ptr(d.layer_input, T0 * H * 2), MC * H * 2},
        {mptr(host->post_out, T0 * HC * 4), ptr(d.post_out, T0 * HC * 4), MC * HC * 4},
        {mptr(host->comb_out, T0 * HC * HC * 4), ptr(d.comb_out, T0 * HC * HC * 4), MC * HC * HC * 4},
        {mptr(host->pre_out, T0 * HC * 4), ptr(d.pre_out, T0 * HC * 4), MC * HC * 4},
        {mptr(host->mixes_out, T0 * MIX * 4), ptr(d.mixes_out, T0 * MIX * 4), MC * MIX * 4},
        {mptr(host->reduced_out, T0 * H * 2), ptr(d.reduced_out, T0 * H * 2), MC * H * 2},
        {mptr(host->mxfp8_values, T0 * H), ptr(d.mxfp8_values, T0 * H), MC * H},
        {mptr(host->mxfp8_scales, T0 * (H / 32)), ptr(d.mxfp8_scales, T0 * (H / 32)), scale_bytes(mcs[k], c.hidden)}};
    for (const Copy &x : out)
      if (e == cudaSuccess && x.dst) e = cudaMemcpyAsync(x.dst, x.src, x.bytes, cudaMemcpyDeviceToHost, b->d2h);
  }
  if (e == cudaSuccess) e = cudaEventRecord(b->host_end, b->d2h);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, b->host_end, 0);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "device to host copy: %s", cudaGetErrorString(e));
  return MHC_OK;
}

mhc_status_t mhc_boundary_check_errors(mhc_boundary_t *b) {
  if (!b) return MHC_ERR_INVALID_ARG;
  DeviceGuard guard(b->device);
  unsigned int flag = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&flag, b->err, sizeof flag, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && flag) e = cudaMemset(b->err, 0, sizeof flag);
  if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "check_errors: %s", cudaGetErrorString(e));
  if (flag & 2u)
    return fail(b->last_error, MHC_ERR_TIMEOUT,
                "a kernel gave up one of its bounded waits (copies or tensor-core work); its outputs are not valid");
  if (flag & 1u)
    return fail(b->last_error, MHC_ERR_INVALID_ARG,
                "a MoE route index was outside [-1, rows_per_rank); the route was skipped");
  return MHC_OK;
}

mhc_status_t mhc_boundary_destroy(mhc_boundary_t *b) {
  if (!b) return MHC_OK;
  {
    DeviceGuard guard(b->device);
    release(b);
  }
  delete b;
  return MHC_OK;
}

size_t mhc_mxfp8_scale_bytes(int32_t m, int32_t hidden) { return scale_bytes(m, hidden); }

int32_t mhc_boundary_launches_per_call(const mhc_boundary_t *b) {
  if (!b) return 0;
  // for a call of max_num_tokens tokens (either weight form): the one-kernel
  // path, or the stage and finish kernels; plus a separate post / Sinkhorn
  // kernel, plus the owner reduce
  const bool owner = (b->cfg.flags & MHC_FLAG_OWNER_REDUCE) != 0;
  const int tp = owner ? 1 : b->cfg.tp;
  const int core = small_clusters_for(b, b->cfg.max_num_tokens, tp) > 0 ? 1 : 2;
  return core + ((b->cfg.flags & (MHC_FLAG_SIDE_MIXES | MHC_FLAG_SYNC_MIXES)) ? 1 : 0) + (owner ? 1 : 0);
}

mhc_status_t mhc_boundary_profile_begin(mhc_boundary_t *b, int32_t max_calls) {
  if (!b) return MHC_ERR_INVALID_ARG;
  if (max_calls < 1 || max_calls > (1 << 16))
    return fail(b->last_error, MHC_ERR_INVALID_ARG, "max_calls must be in [1, 65536]");
  DeviceGuard guard(b->device);
  cudaDeviceSynchronize();
  destroy_profile_events(b);
  b->prof_events.assign(size_t(max_calls) * 6, nullptr);
  for (cudaEvent_t &ev : b->prof_events) {
    const cudaError_t e = cudaEventCreate(&ev);
    if (e != cudaSuccess) {
      destroy_profile_events(b);
      return fail(b->last_error, MHC_ERR_CUDA, "profile_begin: %s", cudaGetErrorString(e));
    }
  }
  b->prof_capacity = max_calls;
  b->prof_calls = 0;
  return MHC_OK;
}

mhc_status_t mhc_boundary_profile_end(mhc_boundary_t *b, mhc_profile_t *out) {
  if (!b || !out) return MHC_ERR_INVALID_ARG;
  DeviceGuard guard(b->device);
  mhc_profile_t sum = {};
  cudaError_t e = cudaDeviceSynchronize();
  for (int i = 0; e == cudaSuccess && i < b->prof_calls; ++i) {
    const cudaEvent_t *ev = &b->prof_events[size_t(i) * 6];
    float ms[3] = {0.f, 0.f, 0.f};
    for (int k = 0; k < 3 && e == cudaSuccess; ++k) e = cudaEventElapsedTime(&ms[k], ev[2 * k], ev[2 * k + 1]);
    sum.stage_ms += ms[0];
    sum.finish_ms += ms[1];
    sum.mixes_ms += ms[2];
  }
  sum.calls = b->prof_calls;
  destroy_profile_events(b);
  if (e != cudaSuccess) return fail(b->last_error, MHC_ERR_CUDA, "profile_end: %s", cudaGetErrorString(e));
  *out = sum;
  return MHC_OK;
}

const char *mhc_status_string(mhc_status_t status) {
  switch (status) {
    case MHC_OK: return "ok";
    case MHC_ERR_INVALID_ARG: return "invalid argument";
    case MHC_ERR_UNSUPPORTED: return "unsupported";
    case MHC_ERR_CAPACITY: return "token count outside capacity";
    case MHC_ERR_CUDA: return "CUDA error";
    case MHC_ERR_OOM: return "out of device memory";
    case MHC_ERR_TIMEOUT: return "timeout";
  }
  return "unknown status";
}

const char *mhc_last_error(const mhc_boundary_t *b) {
  return b ? b->last_error.c_str() : g_create_error.c_str();
}

}  // extern "C"

mhc_status_t mhc_test_stall_stage_copies(int32_t on) {
  cudaError_t e = stage_tc_stall_copies(on ? 1 : 0);
  if (e == cudaSuccess) e = small_stall_copies(on ? 1 : 0);
  return e == cudaSuccess ? MHC_OK : MHC_ERR_CUDA;
}
