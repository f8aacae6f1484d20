/*
 * mhc_oracle.h -- plain, slow CPU statement of the mHC sublayer boundary.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this code; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * Sources (web pages, cited by title and by the class / method on them):
 *   [GLM] "vllm.models.glm5next.nvidia.specialized_decode.all_reduce_mhc"
 *         (AllReduceMhcBoundary, _BoundaryDeviceKernel, _MixesDeviceKernel)
 *   [DSV] "vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc"
 *         (AllReduceMHC, _LamportMHCDeviceKernel,
 *          _QuadFinalizePublishDeviceKernel, _OwnerReduceMulticastDeviceKernel)
 *
 * Arithmetic: IEEE FP32 one operation at a time (the library is compiled with
 * floating-point contraction off); fmaf() only where the reading of the pages
 * is a fused multiply-add.  BF16 rounding is round-to-nearest-even.  Sums whose
 * order the pages leave free (the prenorm GEMV, both sums of squares) are
 * taken in FP64 and rounded once to FP32.
 *
 * Layouts (all row-major, element counts):
 *   partials  [tp][m][H]  bf16      residual  [m][4][H] bf16
 *   post      [m][4] f32            comb      [m][4][4] f32, [source][target]
 *   hc_fn     [4H][24] f32, row j*H+h holds the 24 weights of stream j, column h
 *   scale     [3] f32 (pre, post, comb)        base [24] f32
 *   gamma     [H] bf16
 *   routed    [tp][rows][H] bf16   idx [tp][m][K] i32   weights [m][K] f32
 *   shared    [tp][m][H] bf16
 * BF16 values travel as their 16-bit patterns (uint16_t).
 */
#ifndef MHC_ORACLE_H
#define MHC_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_HC = 4, ORACLE_MIX = 24 };

typedef struct {
  int32_t hidden;          /* H */
  int32_t tp;              /* number of partial sums */
  int32_t m;               /* tokens in the whole problem (row stride) */
  int32_t top_k;           /* K, MoE only */
  int32_t rows_per_rank;   /* rows of routed[r], MoE only */
  int32_t sinkhorn_repeat; /* Sinkhorn rounds */
  float rms_eps;           /* epsilon of the mix RMS */
  float hc_eps;            /* pre-mix offset and Sinkhorn epsilon */
  float post_mult;         /* post-mix multiplier */
  float norm_eps;          /* RMSNorm epsilon */
} oracle_config_t;

/* Scalar conversions (exposed so the tests can pin them). */
float oracle_bf16_to_f32(uint16_t bits);
uint16_t oracle_f32_to_bf16(float value);
uint8_t oracle_f32_to_e4m3(float value);       /* RNE, saturate to +-448 */
double oracle_e4m3_to_f64(uint8_t bits);
uint8_t oracle_ue8m0_of_amax(float amax);      /* scale exponent of a block */
size_t oracle_mxfp8_scale_bytes(int32_t m, int32_t hidden);
size_t oracle_swizzle_128x4(int32_t row, int32_t col, int32_t scale_cols);
/* Element-wise loops over the two conversions above, for exhaustive tests. */
void oracle_f32_to_bf16_array(size_t n, const float *in, uint16_t *out);
void oracle_f32_to_e4m3_array(size_t n, const float *in, uint8_t *out);

/* Steps, each over tokens [t0, t1).  Outputs are indexed like inputs. */
void oracle_stage1(const oracle_config_t *c, int32_t t0, int32_t t1,
                   const uint16_t *partials, uint16_t *y);
void oracle_moe_fold(const oracle_config_t *c, int32_t t0, int32_t t1,
                     const uint16_t *routed, const int32_t *idx,
                     const float *weights, const uint16_t *shared, uint16_t *y);
void oracle_post_mix(const oracle_config_t *c, int32_t t0, int32_t t1,
                     const uint16_t *y, const uint16_t *residual,
                     const float *post, const float *comb, uint16_t *streams);
void oracle_prenorm_gemv(const oracle_config_t *c, int32_t t0, int32_t t1,
                         const uint16_t *streams, const float *hc_fn,
                         float *raw, float *sum_squares);
/* The same with the weight in the GLM page's form: fn [24][4H] BF16, output i,
 * stream j, column h at i * 4H + j * H + h. */
void oracle_prenorm_gemv_bf16(const oracle_config_t *c, int32_t t0, int32_t t1,
                              const uint16_t *streams, const uint16_t *fn,
                              float *raw, float *sum_squares);
void oracle_mixes_and_pre(const oracle_config_t *c, int32_t t0, int32_t t1,
                          const float *raw, const float *sum_squares,
                          const float *scale, const float *base,
                          float *mixes, float *pre);
void oracle_post_from_mixes(const oracle_config_t *c, int32_t t0, int32_t t1,
                            const float *mixes, const float *scale,
                            const float *base, float *post_out);
void oracle_sinkhorn(const oracle_config_t *c, int32_t t0, int32_t t1,
                     const float *mixes, const float *scale, const float *base,
                     float *comb_out);
void oracle_collapse_norm(const oracle_config_t *c, int32_t t0, int32_t t1,
                          const uint16_t *streams, const float *pre,
                          const uint16_t *gamma, uint16_t *layer_input);
/* Quantizes rows [t0, t1) of a BF16 [m][H] matrix; scales must hold
 * oracle_mxfp8_scale_bytes(m, H) bytes.  With pad != 0 it also zeroes the
 * scales of the padding rows m .. ceil(m/128)*128 - 1. */
void oracle_mxfp8(const oracle_config_t *c, int32_t t0, int32_t t1,
                  const uint16_t *layer_input, uint8_t *values,
                  uint8_t *scales, int pad);

/* The whole boundary over tokens [t0, t1), in the pages' order.  moe != 0
 * takes the MoE fold for stage 1 (routed/idx/weights/shared), else partials.
 * Any of mixes, pre, reduced, mx_values/mx_scales may be NULL. */
typedef struct {
  const uint16_t *partials;
  const uint16_t *routed;
  const int32_t *idx;
  const float *weights;
  const uint16_t *shared;
  const uint16_t *residual;
  const float *post;
  const float *comb;
  const float *hc_fn;
  const uint16_t *hc_fn_bf16; /* [24][4H] bf16; used instead of hc_fn when set */
  const float *scale;
  const float *base;
  const uint16_t *gamma;
  uint16_t *residual_out;
  uint16_t *layer_input;
  float *post_out;
  float *comb_out;
  float *mixes;
  float *pre;
  uint16_t *reduced;
  uint8_t *mx_values;
  uint8_t *mx_scales;
  /* [DSV] delayed-mHC consumer: when set, the carried pre-mix [m][4] of the
   * collapse; there is no GEMV, no mixes, no post / Sinkhorn, and with
   * layer_input NULL only the post-mixed streams are written (residual only). */
  const float *pre_in;
} oracle_io_t;

int oracle_boundary(const oracle_config_t *c, int32_t t0, int32_t t1, int moe,
                    const oracle_io_t *io);

#ifdef __cplusplus
}
#endif
#endif /* MHC_ORACLE_H */
