/*
 * mhc_oracle.c -- plain, slow CPU statement of the mHC sublayer boundary.
 *
 * TEST INFRASTRUCTURE ONLY (tests, smoke check, the benchmark's CPU
 * baseline).  The CUDA library never includes, links or calls this file.
 * Compile with -ffp-contract=off so that every FP32 expression below rounds
 * after each operation exactly as written.
 *
 * Pages cited (title, then class / method / block on the page):
 *   [GLM] vllm.models.glm5next.nvidia.specialized_decode.all_reduce_mhc
 *   [DSV] vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc
 * Parity pins for every function live in tests/test_oracle_*.py.
 */
#include "mhc_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define HC ORACLE_HC
#define MIX ORACLE_MIX

/* ------------------------------------------------------------------------ */
/* Scalar conversions                                                        */
/* ------------------------------------------------------------------------ */

float oracle_bf16_to_f32(uint16_t bits) {
  /* A BF16 value is the upper half of the FP32 with the same bits. */
  uint32_t word = (uint32_t)bits << 16;
  float value;
  memcpy(&value, &word, sizeof value);
  return value;
}

uint16_t oracle_f32_to_bf16(float value) {
  /* Round to nearest, ties to even, on the 16 low bits that BF16 drops.  A
   * carry out of the mantissa bumps the exponent (and overflows to inf), as
   * rounding requires.  NaN stays a quiet NaN. */
  uint32_t word;
  memcpy(&word, &value, sizeof word);
  if ((word & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((word >> 16) | 0x0040u);
  uint32_t kept = word >> 16;
  uint32_t dropped = word & 0xffffu;
  if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;
  return (uint16_t)kept;
}

uint8_t oracle_f32_to_e4m3(float value) {
  /* OCP E4M3 (bias 7, no infinities, S.1111.111 is NaN, largest finite 448):
   * normal numbers (1 + f/8) * 2^(E-7) for E = 1..15, subnormals f * 2^-9.
   * The value nearest to x is taken with ties to even, and anything beyond
   * 448 saturates to 448 (the "satfinite" conversion of the MXFP8 reading). */
  uint8_t sign = signbit(value) ? 0x80u : 0x00u;
  if (isnan(value)) return (uint8_t)(sign | 0x7fu);
  if (isinf(value)) return (uint8_t)(sign | 0x7eu);
  double a = fabs((double)value);
  if (a == 0.0) return sign;
  int e;
  (void)frexp(a, &e);           /* a in [2^(e-1), 2^e) */
  int k = e - 1;                /* floor(log2 a) */
  double quantum = (k < -6) ? ldexp(1.0, -9) : ldexp(1.0, k - 3);
  double q = nearbyint(a / quantum) * quantum; /* default mode: ties to even */
  if (q > 448.0) q = 448.0;
  if (q == 0.0) return sign;
  if (q < ldexp(1.0, -6)) {     /* subnormal: f * 2^-9 */
    int f = (int)(q / ldexp(1.0, -9));
    return (uint8_t)(sign | f);
  }
  int eq;
  (void)frexp(q, &eq);
  int kq = eq - 1;
  int biased = kq + 7;
  int f = (int)(q / ldexp(1.0, kq) * 8.0) - 8;
  return (uint8_t)(sign | (biased << 3) | f);
}

double oracle_e4m3_to_f64(uint8_t bits) {
  int biased = (bits >> 3) & 0xf;
  int f = bits & 0x7;
  double magnitude;
  if (biased == 0xf && f == 0x7) return NAN;
  if (biased == 0)
    magnitude = f * ldexp(1.0, -9);
  else
    magnitude = (1.0 + f / 8.0) * ldexp(1.0, biased - 7);
  return (bits & 0x80) ? -magnitude : magnitude;
}

uint8_t oracle_ue8m0_of_amax(float amax) {
  /* [DSV] _LamportMHCDeviceKernel.kernel, MXFP8 epilogue: the block scale is
   * the UE8M0 code of amax * (FP32 reciprocal of the E4M3 maximum 448).
   * Reading: the smallest power of two 2^(e-127) at or above that product,
   * e clamped to [0, 254]; a zero block gets e = 0. */
  const float inv_e4m3_max = 1.0f / 448.0f;
  float s = amax * inv_e4m3_max;
  if (!(s > 0.0f)) return 0;
  int e;
  double f = frexp((double)s, &e); /* s = f * 2^e, f in [0.5, 1) */
  int exponent = (f == 0.5) ? e - 1 : e; /* ceil(log2 s) */
  int biased = exponent + 127;
  if (biased < 0) biased = 0;
  if (biased > 254) biased = 254;
  return (uint8_t)biased;
}

size_t oracle_mxfp8_scale_bytes(int32_t m, int32_t hidden) {
  /* [DSV] AllReduceMHC.__call__ (mxfp8_out): the scale buffer covers the
   * rows padded up to a multiple of 128 and the 32-element blocks padded up
   * to a multiple of 4 columns. */
  size_t rows = ((size_t)m + 127) / 128 * 128;
  size_t cols = ((size_t)hidden / 32 + 3) / 4 * 4;
  return rows * cols;
}

size_t oracle_swizzle_128x4(int32_t row, int32_t col, int32_t scale_cols) {
  /* The 128x4 block-scale layout that MXFP8 GEMMs read ([DSV] names it
   * "swizzled 128x4"): tiles of 128 rows x 4 columns are 512 bytes each,
   * tile-row major; inside a tile, row r sits at (r % 32) * 16 +
   * (r / 32) * 4 and column c at c % 4. */
  size_t cols_padded = ((size_t)scale_cols + 3) / 4 * 4;
  size_t tile = (size_t)(row / 128) * (cols_padded / 4) + (size_t)(col / 4);
  int32_t r = row % 128;
  return tile * 512 + (size_t)(r % 32) * 16 + (size_t)(r / 32) * 4 + (size_t)(col % 4);
}

void oracle_f32_to_bf16_array(size_t n, const float *in, uint16_t *out) {
  for (size_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(in[i]);
}

void oracle_f32_to_e4m3_array(size_t n, const float *in, uint8_t *out) {
  for (size_t i = 0; i < n; ++i) out[i] = oracle_f32_to_e4m3(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Steps                                                                      */
/* ------------------------------------------------------------------------ */

#define BF(x) oracle_bf16_to_f32(x)
#define TO_BF(x) oracle_f32_to_bf16(x)

void oracle_stage1(const oracle_config_t *c, int32_t t0, int32_t t1,
                   const uint16_t *partials, uint16_t *y) {
  /* [DSV] _LamportMHCDeviceKernel.kernel (lane_sum) and
   * _OwnerReduceMulticastDeviceKernel.kernel (reduced): FP32 sum of the tp
   * contributions from rank 0 upward, starting at +0, one add at a time,
   * rounded to BF16 once ("FP32 from rank 0, rounded to BF16", module text
   * of [DSV]; "BF16, as the collective returns it", [GLM] kernel). */
  const size_t H = (size_t)c->hidden, M = (size_t)c->m;
  for (int32_t t = t0; t < t1; ++t) {
    for (size_t h = 0; h < H; ++h) {
      float acc = 0.0f;
      for (int32_t r = 0; r < c->tp; ++r) acc = acc + BF(partials[((size_t)r * M + t) * H + h]);
      y[(size_t)t * H + h] = TO_BF(acc);
    }
  }
}

void oracle_moe_fold(const oracle_config_t *c, int32_t t0, int32_t t1,
                     const uint16_t *routed, const int32_t *idx,
                     const float *weights, const uint16_t *shared, uint16_t *y) {
  /* [DSV] _QuadFinalizePublishDeviceKernel.kernel: per rank r, an FP32
   * accumulator starts at 0 and takes, route by route in k order, the
   * routed row times its FP32 weight (read as a fused multiply-add); routes
   * whose index is -1 (an expert the rank does not hold) add nothing.  The
   * rank's shared-expert row is added and the result rounded to BF16: that is
   * the rank's contribution, which stage 1 then sums in rank order. */
  const size_t H = (size_t)c->hidden, M = (size_t)c->m, K = (size_t)c->top_k;
  const size_t rows = (size_t)c->rows_per_rank;
  for (int32_t t = t0; t < t1; ++t) {
    for (size_t h = 0; h < H; ++h) {
      float total = 0.0f;
      for (int32_t r = 0; r < c->tp; ++r) {
        float acc = 0.0f;
        for (size_t k = 0; k < K; ++k) {
          int32_t row = idx[((size_t)r * M + t) * K + k];
          if (row == -1) continue;
          acc = fmaf(BF(routed[((size_t)r * rows + (size_t)row) * H + h]),
                     weights[(size_t)t * K + k], acc);
        }
        float contribution = acc + BF(shared[((size_t)r * M + t) * H + h]);
        total = total + BF(TO_BF(contribution));
      }
      y[(size_t)t * H + h] = TO_BF(total);
    }
  }
}

void oracle_post_mix(const oracle_config_t *c, int32_t t0, int32_t t1,
                     const uint16_t *y, const uint16_t *residual,
                     const float *post, const float *comb, uint16_t *streams) {
  /* [GLM] _BoundaryDeviceKernel.kernel (mixed = x * post_mix; mixed +=
   * stream_k * comb[k][j]) and [DSV] _LamportMHCDeviceKernel.kernel: stream j
   * of the new residual is bf16(y * post_j + sum_k res_k * comb[k][j]), comb
   * indexed [source][target], the k terms added in source order, each as a
   * fused multiply-add. */
  const size_t H = (size_t)c->hidden;
  for (int32_t t = t0; t < t1; ++t) {
    for (int j = 0; j < HC; ++j) {
      for (size_t h = 0; h < H; ++h) {
        float mixed = BF(y[(size_t)t * H + h]) * post[(size_t)t * HC + j];
        for (int k = 0; k < HC; ++k)
          mixed = fmaf(BF(residual[((size_t)t * HC + k) * H + h]),
                       comb[((size_t)t * HC + k) * HC + j], mixed);
        streams[((size_t)t * HC + j) * H + h] = TO_BF(mixed);
      }
    }
  }
}

void oracle_prenorm_gemv(const oracle_config_t *c, int32_t t0, int32_t t1,
                         const uint16_t *streams, const float *hc_fn,
                         float *raw, float *sum_squares) {
  /* [GLM] _BoundaryDeviceKernel.kernel (partial[row], partial[MIX]): the 24
   * prenorm outputs are dot products of hc_fn's columns with the flattened
   * BF16-rounded new streams (element j*H + h), and the 25th value is their
   * sum of squares.  The order of these sums is not fixed by the pages; they
   * are taken here in FP64 and rounded once. */
  const size_t H = (size_t)c->hidden;
  for (int32_t t = t0; t < t1; ++t) {
    double acc[MIX];
    double squares = 0.0;
    for (int i = 0; i < MIX; ++i) acc[i] = 0.0;
    for (int j = 0; j < HC; ++j) {
      for (size_t h = 0; h < H; ++h) {
        double v = (double)BF(streams[((size_t)t * HC + j) * H + h]);
        const float *row = hc_fn + ((size_t)j * H + h) * MIX;
        for (int i = 0; i < MIX; ++i) acc[i] += (double)row[i] * v;
        squares += v * v;
      }
    }
    for (int i = 0; i < MIX; ++i) raw[(size_t)t * MIX + i] = (float)acc[i];
    sum_squares[t] = (float)squares;
  }
}

void oracle_prenorm_gemv_bf16(const oracle_config_t *c, int32_t t0, int32_t t1,
                              const uint16_t *streams, const uint16_t *fn,
                              float *raw, float *sum_squares) {
  /* The same 24 dot products with the weight as the GLM page passes it
   * ([GLM] AllReduceMhcBoundary.__call__, fn: [24, hc * hidden] BF16;
   * _BoundaryDeviceKernel.kernel reads element row * (hc * hidden) +
   * lane * hidden + column, i.e. output i, stream j, column h at
   * i * 4H + j * H + h).  Each BF16 x BF16 product is exact; the sums are
   * taken in FP64 and rounded once, as for the FP32 weight. */
  const size_t H = (size_t)c->hidden;
  for (int32_t t = t0; t < t1; ++t) {
    double acc[MIX];
    double squares = 0.0;
    for (int i = 0; i < MIX; ++i) acc[i] = 0.0;
    for (int j = 0; j < HC; ++j) {
      for (size_t h = 0; h < H; ++h) {
        double v = (double)BF(streams[((size_t)t * HC + j) * H + h]);
        for (int i = 0; i < MIX; ++i) acc[i] += (double)BF(fn[(size_t)i * HC * H + (size_t)j * H + h]) * v;
        squares += v * v;
      }
    }
    for (int i = 0; i < MIX; ++i) raw[(size_t)t * MIX + i] = (float)acc[i];
    sum_squares[t] = (float)squares;
  }
}

static float sigmoid_f32(float x) { return 1.0f / (1.0f + expf(-x)); }

void oracle_mixes_and_pre(const oracle_config_t *c, int32_t t0, int32_t t1,
                          const float *raw, const float *sum_squares,
                          const float *scale, const float *base,
                          float *mixes, float *pre) {
  /* [GLM] _BoundaryDeviceKernel.kernel: rstd = rsqrt(ss / (hc*H) + rms_eps);
   * mixes = raw * rstd (the raw mixes the side kernel finishes);
   * pre_j = sigmoid(mixes_j * scale[0] + base[j]) + hc_eps. */
  const float n = (float)(HC * c->hidden);
  for (int32_t t = t0; t < t1; ++t) {
    float rstd = 1.0f / sqrtf(sum_squares[t] / n + c->rms_eps);
    for (int i = 0; i < MIX; ++i) mixes[(size_t)t * MIX + i] = raw[(size_t)t * MIX + i] * rstd;
    for (int j = 0; j < HC; ++j) {
      float z = mixes[(size_t)t * MIX + j] * scale[0] + base[j];
      pre[(size_t)t * HC + j] = sigmoid_f32(z) + c->hc_eps;
    }
  }
}

void oracle_post_from_mixes(const oracle_config_t *c, int32_t t0, int32_t t1,
                            const float *mixes, const float *scale,
                            const float *base, float *post_out) {
  /* [GLM] _MixesDeviceKernel.kernel:
   * post_j = sigmoid(mixes_{4+j} * scale[1] + base[4+j]) * post_mult. */
  for (int32_t t = t0; t < t1; ++t)
    for (int j = 0; j < HC; ++j) {
      float z = mixes[(size_t)t * MIX + HC + j] * scale[1] + base[HC + j];
      post_out[(size_t)t * HC + j] = sigmoid_f32(z) * c->post_mult;
    }
}

void oracle_sinkhorn(const oracle_config_t *c, int32_t t0, int32_t t1,
                     const float *mixes, const float *scale, const float *base,
                     float *comb_out) {
  /* [GLM] _MixesDeviceKernel._sinkhorn, step for step:
   *  1. logits c[r][k] = mixes_{8+4r+k} * scale[2] + base[8+4r+k];
   *  2. per row: subtract the row maximum, exponentiate, multiply by the
   *     reciprocal of the row sum, add eps;
   *  3. `repeat` rounds; from the second round on a round first multiplies
   *     each row by 1/(row sum + eps); every round then multiplies each
   *     column by 1/(column sum + eps).
   * Four-term sums are paired ((a + b) + (c + d)) as on the page; the
   * reciprocal is 1/x. */
  const float eps = c->hc_eps;
  for (int32_t t = t0; t < t1; ++t) {
    float m[HC * HC];
    for (int i = 0; i < HC * HC; ++i)
      m[i] = mixes[(size_t)t * MIX + 2 * HC + i] * scale[2] + base[2 * HC + i];
    for (int r = 0; r < HC; ++r) {
      float *row = m + r * HC;
      float peak = fmaxf(fmaxf(row[0], row[1]), fmaxf(row[2], row[3]));
      for (int k = 0; k < HC; ++k) row[k] = expf(row[k] - peak);
      float inv = 1.0f / ((row[0] + row[1]) + (row[2] + row[3]));
      for (int k = 0; k < HC; ++k) row[k] = row[k] * inv + eps;
    }
    for (int it = 0; it < c->sinkhorn_repeat; ++it) {
      if (it > 0) {
        for (int r = 0; r < HC; ++r) {
          float *row = m + r * HC;
          float inv = 1.0f / ((row[0] + row[1]) + (row[2] + row[3]) + eps);
          for (int k = 0; k < HC; ++k) row[k] = row[k] * inv;
        }
      }
      for (int k = 0; k < HC; ++k) {
        float inv = 1.0f / ((m[k] + m[HC + k]) + (m[2 * HC + k] + m[3 * HC + k]) + eps);
        for (int r = 0; r < HC; ++r) m[r * HC + k] = m[r * HC + k] * inv;
      }
    }
    for (int i = 0; i < HC * HC; ++i) comb_out[(size_t)t * HC * HC + i] = m[i];
  }
}

void oracle_collapse_norm(const oracle_config_t *c, int32_t t0, int32_t t1,
                          const uint16_t *streams, const float *pre,
                          const uint16_t *gamma, uint16_t *layer_input) {
  /* [GLM] _BoundaryDeviceKernel.kernel (collapse, prenorm, inv_rms, result)
   * and [DSV] _LamportMHCDeviceKernel.kernel: c = bf16(sum_j new_j * pre_j)
   * with the four products paired as the page's lane butterfly pairs them;
   * inv_rms = rsqrt(sum c^2 / H + norm_eps) (sum order free: FP64);
   * out = bf16((c * inv_rms) * gamma). */
  const size_t H = (size_t)c->hidden;
  uint16_t *collapsed = (uint16_t *)malloc(H * sizeof(uint16_t));
  if (!collapsed) return;
  for (int32_t t = t0; t < t1; ++t) {
    const float *p = pre + (size_t)t * HC;
    double squares = 0.0;
    for (size_t h = 0; h < H; ++h) {
      float v[HC];
      for (int j = 0; j < HC; ++j) v[j] = BF(streams[((size_t)t * HC + j) * H + h]) * p[j];
      collapsed[h] = TO_BF((v[0] + v[1]) + (v[2] + v[3]));
      double cv = (double)BF(collapsed[h]);
      squares += cv * cv;
    }
    float inv_rms = 1.0f / sqrtf((float)squares / (float)H + c->norm_eps);
    for (size_t h = 0; h < H; ++h) {
      float normed = BF(collapsed[h]) * inv_rms;
      layer_input[(size_t)t * H + h] = TO_BF(normed * BF(gamma[h]));
    }
  }
  free(collapsed);
}

void oracle_mxfp8(const oracle_config_t *c, int32_t t0, int32_t t1,
                  const uint16_t *layer_input, uint8_t *values,
                  uint8_t *scales, int pad) {
  /* [DSV] _LamportMHCDeviceKernel.kernel, quantize branch: per 32-element
   * block of the BF16 layer input, amax = max |x|, scale code e from
   * oracle_ue8m0_of_amax, inverse scale 2^(127 - e), each element converted
   * as e4m3(x * inv) in FP32; the scale byte lands at the 128x4 swizzled
   * index; scales of the padding rows up to a multiple of 128 are zero. */
  const int32_t H = c->hidden;
  const int32_t cols = H / 32;
  for (int32_t t = t0; t < t1; ++t) {
    for (int32_t b = 0; b < cols; ++b) {
      const uint16_t *block = layer_input + (size_t)t * H + (size_t)b * 32;
      float amax = 0.0f;
      for (int i = 0; i < 32; ++i) {
        float a = fabsf(BF(block[i]));
        if (a > amax) amax = a;
      }
      uint8_t e = oracle_ue8m0_of_amax(amax);
      float inv = ldexpf(1.0f, 127 - (int)e);
      for (int i = 0; i < 32; ++i)
        values[(size_t)t * H + (size_t)b * 32 + i] = oracle_f32_to_e4m3(BF(block[i]) * inv);
      scales[oracle_swizzle_128x4(t, b, cols)] = e;
    }
  }
  if (pad) {
    int32_t padded = (c->m + 127) / 128 * 128;
    int32_t cols_padded = (cols + 3) / 4 * 4;
    for (int32_t r = c->m; r < padded; ++r)
      for (int32_t b = 0; b < cols_padded; ++b) scales[oracle_swizzle_128x4(r, b, cols)] = 0;
  }
}

int oracle_boundary(const oracle_config_t *c, int32_t t0, int32_t t1, int moe,
                    const oracle_io_t *io) {
  /* [GLM] AllReduceMhcBoundary.__call__ order: stage 1 (or the MoE fold),
   * post-mix, prenorm GEMV, mixes and pre, collapse + RMSNorm; then the side
   * kernel's post and Sinkhorn; [DSV] adds the MXFP8 copy.  With io->pre_in
   * set, [DSV] AllReduceMHC's delayed-mHC consumer instead: stage 1, post-mix,
   * and the collapse with the carried pre (or the streams alone). */
  if (!c || c->hidden <= 0 || c->m <= 0 || t0 < 0 || t1 > c->m || t0 > t1) return -1;
  if (c->tp <= 0) return -1;
  if (moe) {
    if (c->top_k <= 0 || c->rows_per_rank <= 0) return -1;
    const size_t n = (size_t)c->tp * (size_t)c->m * (size_t)c->top_k;
    for (size_t i = 0; i < n; ++i)
      if (io->idx[i] < -1 || io->idx[i] >= c->rows_per_rank) return -2;
  }
  if ((io->mx_values || io->mx_scales) && c->hidden % 128) return -1;
  const size_t H = (size_t)c->hidden, M = (size_t)c->m;
  uint16_t *y = io->reduced ? io->reduced : (uint16_t *)calloc(M * H, sizeof(uint16_t));
  float *raw = (float *)calloc(M * MIX, sizeof(float));
  float *ss = (float *)calloc(M, sizeof(float));
  float *mixes = io->mixes ? io->mixes : (float *)calloc(M * MIX, sizeof(float));
  float *pre = io->pre ? io->pre : (float *)calloc(M * HC, sizeof(float));
  int status = 0;
  if (!y || !raw || !ss || !mixes || !pre) {
    status = -3;
  } else {
    if (moe)
      oracle_moe_fold(c, t0, t1, io->routed, io->idx, io->weights, io->shared, y);
    else
      oracle_stage1(c, t0, t1, io->partials, y);
    oracle_post_mix(c, t0, t1, y, io->residual, io->post, io->comb, io->residual_out);
    if (io->pre_in) {
      /* [DSV] AllReduceMHC.__call__ / finalize: the collapse takes the carried
       * pre-mix; residual_only writes the post-mixed streams alone */
      if (io->layer_input) {
        oracle_collapse_norm(c, t0, t1, io->residual_out, io->pre_in, io->gamma, io->layer_input);
        if (io->mx_values && io->mx_scales)
          oracle_mxfp8(c, t0, t1, io->layer_input, io->mx_values, io->mx_scales, t1 == c->m);
      }
    } else {
    if (io->hc_fn_bf16)
      oracle_prenorm_gemv_bf16(c, t0, t1, io->residual_out, io->hc_fn_bf16, raw, ss);
    else
      oracle_prenorm_gemv(c, t0, t1, io->residual_out, io->hc_fn, raw, ss);
    oracle_mixes_and_pre(c, t0, t1, raw, ss, io->scale, io->base, mixes, pre);
    oracle_collapse_norm(c, t0, t1, io->residual_out, pre, io->gamma, io->layer_input);
    oracle_post_from_mixes(c, t0, t1, mixes, io->scale, io->base, io->post_out);
    oracle_sinkhorn(c, t0, t1, mixes, io->scale, io->base, io->comb_out);
    if (io->mx_values && io->mx_scales)
      oracle_mxfp8(c, t0, t1, io->layer_input, io->mx_values, io->mx_scales, t1 == c->m);
    }
  }
  if (!io->reduced) free(y);
  free(raw);
  free(ss);
  if (!io->mixes) free(mixes);
  if (!io->pre) free(pre);
  return status;
}
