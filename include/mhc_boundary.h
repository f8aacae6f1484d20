/*
 * mhc_boundary.h -- C ABI of the GB300 mHC sublayer boundary library.
 *
 * The mHC (multi-stream hyper-connection) sublayer boundary of a
 * DSV4.1 / GLM-style decoder, for one GPU where the tp partial sublayer
 * outputs already sit in local HBM.  One call, in order:
 *   1. sums the tp BF16 partials in FP32 in rank order, rounds to BF16
 *      (or folds an unfinalised MoE output: top-k weighted routed rows plus
 *      the shared expert, per rank, then the same rank-order sum);
 *   2. post-mixes the hc = 4 residual streams;
 *   3. takes the 24-way prenorm GEMV of the new streams against hc_fn and
 *      their sum of squares;
 *   4. derives pre (on the caller's stream) and, on a library side stream,
 *      post and the Sinkhorn residual mix for the next boundary;
 *   5. collapses the streams with pre and RMS-normalises the result, with an
 *      optional MXFP8 copy (E4M3 values, UE8M0 scales per 32 elements in the
 *      swizzled 128x4 layout).
 *
 * Sources (web pages, by title and the class / method on them):
 *   [GLM] vllm.models.glm5next.nvidia.specialized_decode.all_reduce_mhc --
 *         AllReduceMhcBoundary.__init__ / __call__ / join,
 *         _BoundaryDeviceKernel.kernel, _MixesDeviceKernel._sinkhorn.
 *   [DSV] vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc --
 *         AllReduceMHC.__call__ / finalize / _check / _consumer,
 *         _LamportMHCDeviceKernel.kernel, _QuadFinalizePublishDeviceKernel.
 *
 * Conventions for every entry point:
 *   - BF16 tensors are passed as their 16-bit patterns (void pointers).
 *   - Unless a function says "host", pointers are DEVICE pointers on the
 *     handle's device; the caller allocates and owns every buffer.  The
 *     library owns only its handle, a side stream, two events and scratch
 *     that it allocates in mhc_boundary_create (nothing is allocated later).
 *   - Tensors are dense row-major with the shapes given below.  BF16, FP8,
 *     hc_fn, post and comb pointers must be 16-byte aligned (the kernels move
 *     them with 16-byte vector loads and TMA tensor copies), the other FP32 /
 *     int32 pointers 4-byte aligned.
 *   - Errors: every argument is checked before the first launch; on error
 *     the call returns a non-zero status, launches nothing and leaves the
 *     handle's state unchanged ([DSV] AllReduceMHC._consumer: a bad argument
 *     raises with the state untouched).  A CUDA launch failure returns
 *     MHC_ERR_CUDA.  mhc_last_error() gives the message.  Nothing aborts,
 *     exits or traps.
 *   - A handle is not safe for concurrent use from several host threads.
 */
#ifndef MHC_BOUNDARY_H
#define MHC_BOUNDARY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream); NULL is the legacy default stream. */
typedef struct CUstream_st *mhc_stream_t;

typedef enum {
  MHC_OK = 0,
  MHC_ERR_INVALID_ARG = 1, /* a pointer, size, alignment or shape is wrong */
  MHC_ERR_UNSUPPORTED = 2, /* valid request the library does not implement */
  MHC_ERR_CAPACITY = 3,    /* m outside [1, max_num_tokens] */
  MHC_ERR_CUDA = 4,        /* a CUDA call failed */
  MHC_ERR_OOM = 5,         /* device allocation failed in create */
  MHC_ERR_TIMEOUT = 6      /* a kernel gave up a bounded wait (see check_errors) */
} mhc_status_t;

/* Config flags. */
enum {
  /* Accept mxfp8_values / mxfp8_scales (needs hidden % 128 == 0);
   * [DSV] AllReduceMHC(quantize_layer_input=True). */
  MHC_FLAG_MXFP8 = 1u << 0,
  /* Compute post / Sinkhorn in a separate one-warp-per-32-tokens kernel on
   * the caller's stream (takes precedence over MHC_FLAG_SIDE_MIXES).  Without
   * either flag the finish kernel computes them itself, on the caller's
   * stream, beside the collapse of the same token.  All three forms give the
   * same bits; with no side stream, join() is a no-op. */
  MHC_FLAG_SYNC_MIXES = 1u << 1,
  /* Allocate device staging buffers in create so that mhc_boundary_run_host
   * can take host pointers. */
  MHC_FLAG_HOST_STAGING = 1u << 2,
  /* [GLM] AllReduceMhcBoundary's layout: post / Sinkhorn in a separate kernel
   * on the library side stream, so that they overlap whatever the caller
   * enqueues next; post_out / comb_out are then valid only after
   * mhc_boundary_join (or the next call, which joins automatically). */
  MHC_FLAG_SIDE_MIXES = 1u << 3,
  /* The prenorm weight (hc_fn or hc_fn_bf16) is a layer weight: it is written
   * before the first call, by work the call's stream has already waited for,
   * and not while calls run.  The stage kernel is a programmatic dependent
   * launch: its CTAs set up while the kernel before it on the stream is
   * finishing, and with this flag they also stage the weight and split it
   * into tensor-core operands then, ahead of the wait for that kernel.  The
   * partials, streams, post and comb are read only after the wait in any
   * case.  Results are the same bits with or without the flag. */
  MHC_FLAG_STATIC_WEIGHT = 1u << 4,
  /* [DSV] two-shot (BT) reduction, emulated on one GPU: an owner-reduce
   * kernel first sums the tp partials of every token (token t's owner is
   * rank t % tp) in FP32 from rank 0 and rounds to BF16, into a library
   * buffer of max_num_tokens x H BF16 allocated in create; the boundary then
   * takes those sums as its one partial.  Same bits as the direct sum; one
   * more kernel and 4H more bytes a token.  Applies to mhc_boundary_run and
   * to mhc_boundary_consume with partials; a MoE call folds its routes
   * instead. */
  MHC_FLAG_OWNER_REDUCE = 1u << 5,
  /* mhc_boundary_run_static only (mhc_boundary_create rejects it): after
   * launching, the call synchronises its stream and reads the error word of
   * the allocation-free calls on this device, which a kernel sets when one of
   * its bounded waits gives up; a set word returns MHC_ERR_TIMEOUT (and is
   * cleared).  Without the flag the word keeps the report until a call with
   * the flag reads it. */
  MHC_FLAG_CHECK_ERRORS = 1u << 6
};

/* Construction arguments ([GLM] AllReduceMhcBoundary.__init__, [DSV]
 * AllReduceMHC.__init__).  hc_mult must be 4 (the 24 mixes are
 * 2*hc + hc*hc); hidden % 8 == 0; 1 <= tp <= 32; top_k = 0 disables
 * finalize_moe, else 1 <= top_k <= 64. */
typedef struct {
  int32_t hidden;          /* H */
  int32_t hc_mult;         /* hc, must be 4 */
  int32_t tp;              /* number of partial sums per token */
  int32_t max_num_tokens;  /* capacity: largest m of any call */
  int32_t sinkhorn_repeat; /* Sinkhorn rounds, >= 1 */
  int32_t top_k;           /* routes per token for finalize_moe (0: none) */
  float rms_eps;           /* epsilon of the prenorm RMS */
  float hc_eps;            /* pre-mix offset and Sinkhorn epsilon */
  float post_mult;         /* post-mix multiplier */
  float norm_eps;          /* RMSNorm epsilon */
  uint32_t flags;          /* MHC_FLAG_* */
} mhc_boundary_config_t;

typedef struct mhc_boundary mhc_boundary_t; /* opaque, library-owned */

/* Arguments of one boundary call over m tokens.
 * Inputs:
 *   partials    [tp][m][H] bf16: rank r's partial sublayer output (rank-major)
 *   residual    [m][4][H]  bf16: the hc residual streams
 *   post        [m][4]     f32 : post-mix of the previous boundary
 *   comb        [m][4][4]  f32 : residual mix, indexed [source][target]
 *   hc_fn       [4H][24]   f32 : prenorm GEMV weight, row j*H + h
 *                                  (or NULL when hc_fn_bf16 is given)
 *   scale       [3]        f32 : mix scales (pre, post, comb)
 *   base        [24]       f32 : mix biases (pre 0..3, post 4..7, comb 8..23)
 *   norm_weight [H]        bf16: RMSNorm weight
 * Outputs (required):
 *   residual_out [m][4][H] bf16: post-mixed streams
 *   layer_input  [m][H]    bf16: RMS-normalised collapse
 *   post_out     [m][4]    f32 : next boundary's post-mix   (side stream)
 *   comb_out     [m][4][4] f32 : next boundary's Sinkhorn mix (side stream)
 * Outputs (optional, NULL = not written):
 *   pre_out      [m][4]    f32 : pre-mix used for the collapse
 *   mixes_out    [m][24]   f32 : normalised GEMV outputs ("raw mixes")
 *   reduced_out  [m][H]    bf16: the stage-1 sum
 *   mxfp8_values [m][H]    u8  : E4M3 copy of layer_input   (MHC_FLAG_MXFP8)
 *   mxfp8_scales mhc_mxfp8_scale_bytes(m, H) u8: UE8M0 scales, 128x4
 *                swizzled, padding rows zeroed; both or neither. */
typedef struct {
  int32_t m;
  const void *partials;
  const void *residual;
  const float *post;
  const float *comb;
  const float *hc_fn;
  const float *scale;
  const float *base;
  const void *norm_weight;
  void *residual_out;
  void *layer_input;
  float *post_out;
  float *comb_out;
  float *pre_out;
  float *mixes_out;
  void *reduced_out;
  uint8_t *mxfp8_values;
  uint8_t *mxfp8_scales;
  /* The prenorm weight in the GLM page's form instead of hc_fn ([GLM]
   * AllReduceMhcBoundary.__call__, fn): [24][4H] bf16, output i, stream j,
   * column h at i*4H + j*H + h.  Exactly one of hc_fn and hc_fn_bf16 is
   * non-NULL; hc_fn_bf16 needs tp <= 8 (MHC_ERR_UNSUPPORTED otherwise). */
  const void *hc_fn_bf16;
} mhc_run_args_t;

/* Arguments of a boundary call whose stage 1 folds an unfinalised MoE output
 * ([DSV] AllReduceMHC.finalize and _QuadFinalizePublishDeviceKernel; [GLM]
 * AllReduceMhcBoundary.__call__ with a MoEOutput).  run.partials must be
 * NULL; every other field of run is as for mhc_boundary_run.
 *   routed  [tp][rows_per_rank][H] bf16: each rank's unweighted expert rows
 *   idx     [tp][m][top_k] int32: row of each route in routed[r], -1 for a
 *           route the rank does not hold; any other out-of-range value adds
 *           nothing and is reported by mhc_boundary_check_errors
 *   weights [m][top_k] f32: routing weights, already scaled
 *   shared  [tp][m][H] bf16: each rank's shared-expert partial output
 * Per rank: x_r = bf16(sum_k weights * routed_r[idx] + shared_r), the routes
 * in k order as fused multiply-adds; then the stage-1 sum over r. */
typedef struct {
  mhc_run_args_t run;
  int32_t rows_per_rank;
  const void *routed;
  const int32_t *idx;
  const float *weights;
  const void *shared;
} mhc_moe_args_t;

/* Creates a boundary on `device` (it becomes current only inside library
 * calls).  Allocates the side stream, its events and the scratch for
 * max_num_tokens tokens.  *out is set only on MHC_OK. */
mhc_status_t mhc_boundary_create(const mhc_boundary_config_t *config, int device,
                                 mhc_boundary_t **out);

/* One boundary call on `stream` ([GLM] AllReduceMhcBoundary.__call__): the
 * stage and finish kernels on `stream`; post / Sinkhorn inside the finish
 * kernel, or (flags) in a separate kernel.  With MHC_FLAG_SIDE_MIXES the call
 * first makes `stream` wait for the previous call's side-stream kernel (the
 * automatic join) and post_out / comb_out are valid for `stream` only after
 * mhc_boundary_join (or the next call); otherwise they are ordered like every
 * other output.
 * Stream capture: calls may be recorded into a CUDA graph.  Inside a capture
 * the automatic join covers only side kernels of the same capture, so join
 * and finish eager calls before the capture begins, and call
 * mhc_boundary_join on the capturing stream before ending the capture (the
 * side stream's branch must rejoin it).  Profiling events are not recorded
 * inside a capture. */
mhc_status_t mhc_boundary_run(mhc_boundary_t *b, const mhc_run_args_t *args,
                              mhc_stream_t stream);

/* mhc_boundary_run with the MoE fold as stage 1 (needs top_k > 0): a fold
 * kernel writes the stage-1 sum to library scratch ([cap][H] bf16, allocated
 * in create when top_k > 0), which the stage kernel reads as its only
 * partial. */
mhc_status_t mhc_boundary_finalize_moe(mhc_boundary_t *b, const mhc_moe_args_t *args,
                                       mhc_stream_t stream);

/* Arguments of a delayed-mHC consumer call ([DSV] AllReduceMHC.__call__ /
 * finalize): the boundary without the prenorm GEMV, for a model that carries
 * the pre-mix from elsewhere.
 *   partials     [tp][m][H] bf16, or NULL to fold an unfinalised MoE output
 *                (rows_per_rank, routed, idx, weights, shared as in
 *                mhc_moe_args_t; needs top_k > 0)
 *   residual, post, comb: as for mhc_boundary_run
 *   pre          [m][4] f32: carried pre-mix of the collapse; NULL together
 *                with norm_weight and layer_input for residual_only ([DSV]
 *                AllReduceMHC(residual_only=True)): only the post-mixed
 *                streams are written
 *   norm_weight  [H] bf16
 *   residual_out [m][4][H] bf16, layer_input [m][H] bf16 (NULL iff pre is NULL)
 *   reduced_out  optional [m][H] bf16: the stage-1 sum
 *   mxfp8_values / mxfp8_scales: optional, as for mhc_boundary_run, not with
 *                residual_only ([DSV]: "a residual-only consumer has no layer
 *                input to quantize")
 * No post_out / comb_out / mixes: the consumer leaves the next mixes to the
 * caller.  Up to twelve tokens (four with residual_only) it runs one kernel
 * of CTA clusters where the shape fits; otherwise the stage kernel without
 * its GEMV and, unless residual_only, the finish kernel with the carried
 * pre; all on `stream` (after the MoE fold for a MoE output). */
typedef struct {
  int32_t m;
  const void *partials;
  int32_t rows_per_rank;
  const void *routed;
  const int32_t *idx;
  const float *weights;
  const void *shared;
  const void *residual;
  const float *post;
  const float *comb;
  const float *pre;
  const void *norm_weight;
  void *residual_out;
  void *layer_input;
  void *reduced_out;
  uint8_t *mxfp8_values;
  uint8_t *mxfp8_scales;
} mhc_consume_args_t;

mhc_status_t mhc_boundary_consume(mhc_boundary_t *b, const mhc_consume_args_t *args,
                                  mhc_stream_t stream);

/* Makes `stream` wait for the last side-stream kernel ([GLM]
 * AllReduceMhcBoundary.join).  Cheap; may be called any number of times.
 * On a capturing stream it joins a side kernel of the same capture; a side
 * kernel that ran in a captured graph is ordered by the graph itself. */
mhc_status_t mhc_boundary_join(mhc_boundary_t *b, mhc_stream_t stream);

/* mhc_boundary_run with HOST pointers in `args` (every tensor in host
 * memory; pinned memory makes the copies asynchronous).  Needs
 * MHC_FLAG_HOST_STAGING.  The call is split into token chunks (one chunk
 * below 512 tokens, else up to 8 chunks of at least 256 tokens, each a
 * multiple of 128): each chunk's inputs are copied to the library staging
 * buffers on the handle's host-to-device stream, its kernels run on `stream`
 * once they have arrived, and its outputs are copied back on the handle's
 * device-to-host stream, so copies in both directions overlap the kernels.
 * Each chunk is one boundary call over its tokens (the same bits as one
 * call over all of them).  The copy streams start after the work already on
 * `stream`, and the call synchronises `stream`, which is ordered after the
 * last copy, before returning (so it cannot be captured). */
mhc_status_t mhc_boundary_run_host(mhc_boundary_t *b, const mhc_run_args_t *args,
                                   mhc_stream_t stream);

/* Synchronises the handle's streams and reports device-detected errors of
 * earlier calls: MHC_ERR_TIMEOUT if a kernel gave up one of its bounded
 * waits (for copies or tensor-core work; its outputs are then invalid),
 * MHC_ERR_INVALID_ARG
 * for an out-of-range MoE route index, else MHC_OK (the flags are cleared). */
mhc_status_t mhc_boundary_check_errors(mhc_boundary_t *b);

/* Waits for the side stream, frees everything the handle owns. NULL is OK. */
mhc_status_t mhc_boundary_destroy(mhc_boundary_t *b);

/* Bytes of the MXFP8 scale buffer: rows padded to a multiple of 128 times
 * the 32-element blocks per row padded to a multiple of 4 ([DSV]
 * mxfp8_scale_bytes). 0 if hidden % 32 != 0 or m < 1. */
size_t mhc_mxfp8_scale_bytes(int32_t m, int32_t hidden);

/* One boundary call that allocates nothing.  The pages have no counterpart
 * of this entry point: it exists for callers that cannot allocate device
 * memory when they need a boundary -- a framework whose caching allocator
 * already owns the device's memory budget, code that must not trigger the
 * implicit device synchronisation a cudaMalloc / cudaFree can cause, or a
 * thread that may not create a handle (mhc_boundary_create allocates scratch,
 * a stream and events).  It needs no handle: `config` is read as for
 * mhc_boundary_create (top_k is ignored) and `args` as for mhc_boundary_run,
 * device pointers the caller allocated and owns.  config->flags may hold:
 *   MHC_FLAG_MXFP8          accept mxfp8_values / mxfp8_scales;
 *   MHC_FLAG_STATIC_WEIGHT  the prenorm weight is a layer weight: the stage
 *                           kernel reads it before it waits for the kernel
 *                           ahead of it on `stream`, so no kernel enqueued
 *                           before the call may write hc_fn / hc_fn_bf16;
 *   MHC_FLAG_SYNC_MIXES     accepted and without effect here: post / Sinkhorn
 *                           always run in a separate kernel on `stream`;
 *   MHC_FLAG_CHECK_ERRORS   synchronise and report device-side failures (see
 *                           the flag).
 * The stage kernel, the finish kernel and the post / Sinkhorn kernel run on
 * `stream` in order, so post_out / comb_out need no join.
 * Scratch: an 8 MiB array of this library's device memory, which every GPU
 * that loads the library holds until the process exits; a call needs
 * m * (4 * ceil(25 * ceil(H / 64) / 4) + 24) * 4 + 256 bytes of it (H = 6144: up to 865 tokens),
 * and a larger m returns MHC_ERR_CAPACITY with nothing launched.  Every call
 * on a device shares that array and it keeps the last call's contents
 * (nothing needs clearing: each call writes every scratch word it reads
 * before reading it, unless one of its kernels gave up a bounded wait, which
 * the error word records), so calls whose kernels overlap on the GPU race:
 * order them on one stream or with events.  The first call on a device looks
 * up the addresses of the array and of the error word and sets kernel
 * attributes there; make that first call before any stream capture.  Runs on
 * the current device.  On failure the message is written to
 * error[0 .. error_len-1] (error may be NULL) and nothing is launched, except
 * for the report of MHC_FLAG_CHECK_ERRORS, which comes after the launches. */
mhc_status_t mhc_boundary_run_static(const mhc_boundary_config_t *config, const mhc_run_args_t *args,
                                     mhc_stream_t stream, char *error, size_t error_len);

/* Device time of each kernel, summed over the calls recorded between
 * mhc_boundary_profile_begin and mhc_boundary_profile_end (for measurement
 * tools; off by default). */
typedef struct {
  int32_t calls;    /* calls recorded */
  float stage_ms;   /* stage kernel (with the MoE fold or owner reduce before it):
                       stage 1, post-mix, partial GEMV */
  float finish_ms;  /* finish kernel: pre, collapse, RMSNorm, MXFP8 */
  float mixes_ms;   /* side kernel: post and Sinkhorn */
} mhc_profile_t;

/* Records CUDA events around every kernel of the next max_calls calls (events
 * are created here, not per call).  Calls beyond max_calls are not recorded. */
mhc_status_t mhc_boundary_profile_begin(mhc_boundary_t *b, int32_t max_calls);
/* Synchronises the recorded events, writes the sums to *out and stops
 * recording (the events are destroyed). */
mhc_status_t mhc_boundary_profile_end(mhc_boundary_t *b, mhc_profile_t *out);

/* Kernels one mhc_boundary_run call of max_num_tokens tokens launches: one
 * (the one-kernel path, up to twelve tokens where the shape fits) or two
 * (stage + finish), plus the post / Sinkhorn kernel with MHC_FLAG_SIDE_MIXES
 * or MHC_FLAG_SYNC_MIXES, plus the owner reduce with MHC_FLAG_OWNER_REDUCE.
 * mhc_boundary_finalize_moe launches the MoE fold in its place, or one more
 * kernel without that flag. */
int32_t mhc_boundary_launches_per_call(const mhc_boundary_t *b);

const char *mhc_status_string(mhc_status_t status);
/* Message of the handle's last failure ("" if none); NULL handle: the last
 * failure of mhc_boundary_create on this thread. */
const char *mhc_last_error(const mhc_boundary_t *b);

#ifdef __cplusplus
}
#endif
#endif /* MHC_BOUNDARY_H */
