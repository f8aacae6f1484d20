// launch.cuh -- parameter blocks and launchers of the boundary kernels
// (internal to the library; the public surface is include/mhc_boundary.h).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mhc {

constexpr int HC = 4;           // residual streams
constexpr int MIX = 24;         // 2*HC + HC*HC mixes
constexpr int VALUES = MIX + 1; // the mixes and the sum of squares
constexpr int VEC = 8;          // BF16 values per 16-byte fragment

// Hidden elements a CUDA-core stage CTA owns (8 fragments of 8 BF16 values).
constexpr int SLICE = 64;
// Hidden columns of one tensor-core stage unit (256-byte rows).
constexpr int TC_GROUP_COLS = 128;
// Ranks one TMA box of the tensor-core stage kernel covers; calls with more
// partials run the CUDA-core stage kernel.
constexpr int TP_TMA_MAX = 8;
// Floats per token row of the partial-sum scratch: slices x 25, padded to a
// multiple of 4 so that every row starts on a 16-byte boundary.
constexpr int part_row_floats(int slices) { return (slices * VALUES + 3) / 4 * 4; }
// Dynamic shared memory the stage kernel may use (of 227 KB per CTA).
constexpr size_t STAGE_SMEM_LIMIT = 200 * 1024;
// Largest hidden size the finish kernel's register tiling covers.
constexpr int MAX_HIDDEN = 16384;

// Stage kernel: stage-1 sum, post-mix, partial GEMV + sum of squares for one
// (token tile, hidden slice).  A MoE call's fold kernel runs first and the
// stage kernel takes its output as the one partial.
struct StageParams {
  int m, hidden, tp, slices;
  const uint16_t *partials;   // [tp][m][H]
  const uint16_t *residual;   // [m][4][H]
  const float *post;          // [m][4]
  const float *comb;          // [m][4][4]
  const float *hc_fn;         // [4H][24] f32, or null
  const uint16_t *hc_fn_bf16; // [24][4H] bf16 (tensor-core kernel only), or null
  int fn_terms;               // BF16 terms of B: 3 for the FP32 weight, 1 for the BF16 one,
                              // 0 for no GEMV (the delayed-mHC consumer: streams only)
  int early_weight;           // the weight is a layer weight: stage and split it before
                              // waiting for the preceding kernel (tensor-core kernel)
  int group_aligned;          // set by the launcher: every CTA's units lie in one column group
  uint16_t *residual_out;     // [m][4][H]
  uint16_t *reduced_out;      // [m][H] or null
  float *part;                // [m][part_stride]: [slices][25] partial GEMV outputs + sum of squares
  int part_stride;            // floats per token row of part (part_row_floats(slices))
  unsigned int *err;          // device error word (bit 1: a bounded wait gave up), or null
};

// Finish kernel: per token, the partial sums, mixes, pre, collapse, RMSNorm,
// the optional MXFP8 copy and, with post_out / comb_out set, the next
// boundary's post-mix and Sinkhorn mix.
struct FinishParams {
  int m, hidden, slices, part_stride;
  const float *part;
  const float *scale;
  const float *base;
  const uint16_t *gamma;
  const uint16_t *streams;    // the residual_out the stage kernel wrote
  float rms_eps, hc_eps, norm_eps;
  float *mixes;               // [m][24] raw mixes for the side kernel, or null
  float *mixes_out;           // optional copy
  const float *pre_in;        // [m][4] carried pre-mix (delayed-mHC consumer), or null
  float *post_out;            // [m][4]: post-mix computed here (fused), or null
  float *comb_out;            // [m][4][4]: Sinkhorn mix computed here (fused), or null
  float post_mult;
  int repeat;                 // Sinkhorn rounds
  float *pre_out;             // optional
  uint16_t *layer_input;      // [m][H]
  uint8_t *mx_values;         // [m][H] or null
  uint8_t *mx_scales;         // mxfp8_scale_bytes(m, H) or null
  unsigned int *err;          // device error word (bit 1: a wait gave up) or null
};

// The boundary of a few tokens in one kernel (k_small.cu): clusters of `cs`
// CTAs, each cluster up to SMALL_B_MAX tokens, each CTA a column range.
constexpr int SMALL_B_MAX = 8;
constexpr int SMALL_ITEMS_MAX = 512;   // (token, 16-byte fragment) items of a CTA
// Largest call the one-kernel path takes (larger calls run the stage and
// finish kernels).  Up to twelve tokens it takes six or fewer clusters and is
// the faster path (two tokens a cluster: at H = 6144 tp = 4, 9.1 / 9.3 us a
// call at 10 / 12 tokens against 10.1 for the stage and finish kernels);
// from 16 tokens on its clusters hold most of the SMs, so the next call's
// CTAs cannot start their prologue beside it, and the two kernels are faster
// (10.1 against 10.8 us at 16 tokens; the same at H = 5120 tp = 8).
constexpr int SMALL_M_MAX = 12;
struct SmallParams {
  int m, hidden, tp;
  int cs;                     // CTAs a cluster (8 or 16)
  int cols_max;               // small_cols_max(hidden, cs)
  const uint16_t *partials;   // [tp][m][H]
  const uint16_t *residual;   // [m][4][H]
  const float *post;          // [m][4]
  const float *comb;          // [m][4][4]
  const float *hc_fn;         // [4H][24] f32, or null
  const uint16_t *hc_fn_bf16; // [24][4H] bf16, or null (exactly one of the two; neither for the consumer)
  const float *scale;         // [3] (not read by the consumer)
  const float *base;          // [24] (not read by the consumer)
  const uint16_t *gamma;      // [H]
  int consume;                // the delayed-mHC consumer: no GEMV and no mixes; pre comes from pre_in
  const float *pre_in;        // [m][4] carried pre of the consumer, or null: the post-mixed streams only
  int early_weight;           // the weight is a layer weight: load it before the wait
  float rms_eps, hc_eps, norm_eps, post_mult;
  int repeat;
  uint16_t *residual_out;     // [m][4][H]
  uint16_t *reduced_out;      // [m][H] or null
  uint16_t *layer_input;      // [m][H]
  float *mixes;               // [m][24] for a separate post / Sinkhorn kernel, or null
  float *mixes_out, *pre_out; // optional
  float *post_out, *comb_out; // null when a separate kernel computes them
  uint8_t *mx_values;         // [m][H] or null
  uint8_t *mx_scales;         // mxfp8_scale_bytes(m, H) or null
  unsigned int *err;          // bit 1: a copy wait gave up
};

// Two-shot reduction (single-GPU emulation of the owner reduce): the tp
// partials [tp][m][H] summed per token into sums [m][H].
struct OwnerParams {
  int m, hidden, tp;
  const uint16_t *partials;   // [tp][m][H]
  uint16_t *sums;             // [m][H]
};

// MoE fold: stage 1 of a MoE-finalize call into a [m][H] BF16 buffer.
struct FoldParams {
  int m, hidden, tp, top_k, rows_per_rank;
  const uint16_t *routed;     // [tp][rows][H]
  const int32_t *idx;         // [tp][m][K]
  const float *weights;       // [m][K]
  const uint16_t *shared;     // [tp][m][H]
  uint16_t *y;                // [m][H]
  unsigned int *err;          // bit 0: route index outside [-1, rows)
};

// Side kernel: post-mix and Sinkhorn residual mix of the next boundary.
struct MixesParams {
  int m, repeat;
  const float *mixes;
  const float *scale;
  const float *base;
  float post_mult, eps;
  float *post_out;            // [m][4]
  float *comb_out;            // [m][4][4]
};

// Token tile of the stage kernel for a call of m tokens.
int stage_tile_tokens(int m);
size_t stage_smem_bytes(int tile_tokens);
cudaError_t stage_set_attributes();
cudaError_t launch_stage(const StageParams &p, cudaStream_t stream);
// Stage kernel with the GEMV on tcgen05 tensor cores (non-MoE calls):
// persistent, at most `ctas` CTAs of one per SM.
size_t stage_tc_smem_bytes();
cudaError_t stage_tc_set_attributes();
cudaError_t stage_tc_stall_copies(int on);   // test hook, see include/mhc_boundary_test.h
// `grid_out`, if given, receives the number of CTAs launched.
cudaError_t launch_stage_tc(const StageParams &p, int ctas, cudaStream_t stream, int *grid_out = nullptr);
// Finish kernel: persistent CTAs (at most `ctas`), programmatic dependent
// launch after the stage kernel when `pdl`.  `stage_grid`: the CTAs of the
// tensor-core stage kernel of this call (0 if another stage kernel ran); a
// call of the same shape launches that many again next, and the finish
// kernel's CTAs per SM are chosen with them in mind.
cudaError_t finish_set_attributes();
cudaError_t launch_finish(const FinishParams &p, int ctas, cudaStream_t stream, bool pdl, int stage_grid = 0);
cudaError_t launch_mixes(const MixesParams &p, cudaStream_t stream);
// The boundary of a few tokens in one kernel: columns a CTA, shared memory,
// tokens a cluster (0: the shape does not fit), attributes, clusters that
// run at once, launch on `clusters` clusters.
int small_cols_max(int hidden, int cs);
size_t small_smem_bytes(int hidden, int tp, int cs, int tokens);
int small_tokens_max(int hidden, int tp, int cs);
cudaError_t small_set_attributes();
cudaError_t small_stall_copies(int on);   // test hook, see include/mhc_boundary_test.h
int small_active_clusters(int cs, size_t smem);
cudaError_t launch_small(const SmallParams &p, int clusters, cudaStream_t stream);
// MoE fold: CTAs of 256 threads, at most three for each of the GPU's `sms`
// SMs; the attributes allow its rank buffer of up to 64 KB.
cudaError_t moe_fold_set_attributes();
cudaError_t launch_moe_fold(const FoldParams &p, int sms, cudaStream_t stream);
cudaError_t launch_owner_reduce(const OwnerParams &p, int ctas, cudaStream_t stream);

}  // namespace mhc
