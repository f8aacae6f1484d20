// device_common.cuh -- device helpers shared by the boundary kernels:
// BF16 packing (hardware round-to-nearest-even conversions), vector loads
// and stores with cache hints, warp reductions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "launch.cuh"

namespace mhc {

// ---------------------------------------------------------------- BF16
// A BF16 value is the upper half of the FP32 with the same bits.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two FP32 values to a BF16 pair, nearest-even (lo in bits 0..15).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void unpack8(const uint4 &v, float (&x)[8]) {
  x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x);
  x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
  x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z);
  x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
  return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                    pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
}

// Rounds eight FP32 values to BF16 in place (the value a BF16 store keeps).
__device__ __forceinline__ uint4 round8(float (&x)[8]) {
  uint4 p = pack8(x);
  unpack8(p, x);
  return p;
}

// ------------------------------------------------------------- memory
// Streaming read of data used once: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Read-only 16-byte read, cached in L1 (data no kernel of the call writes
// and the CTA re-reads, such as a weight).  Not ordered after the thread's
// own earlier stores, so independent reads issue back to back.
__device__ __forceinline__ uint4 ld_ro(const void *p) {
  uint4 v;
  asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Plain 16-byte read through L1 (data other threads of the CTA re-read).
__device__ __forceinline__ uint4 ld_vec(const void *p) {
  return *reinterpret_cast<const uint4 *>(p);
}

__device__ __forceinline__ void st_vec(void *p, const uint4 &v) {
  *reinterpret_cast<uint4 *>(p) = v;
}

// ----------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Programmatic dependent launch: wait until the preceding kernel on the
// stream has completed and its memory is visible (a no-op without PDL).
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next kernel on the stream start its launch early.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// --------------------------------------------------- mixes and MXFP8 steps
// sigmoid(z) = 1 / (1 + exp(-z)) with a correctly rounded reciprocal.
__device__ __forceinline__ float sigmoid(float z) {
  return __frcp_rn(__fadd_rn(1.0f, expf(-z)));
}

// The Sinkhorn normalisation reciprocal: the hardware's approximate
// reciprocal instruction (rcp.approx, within 1 ulp of 1/x; the sums it takes
// are at least eps = 1e-6 and at most a few units, far from subnormal, so
// the flush-to-zero form is exact in its range).  One instruction on the
// chain of 40 dependent normalisations a token.
__device__ __forceinline__ float rcp_fast(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// A BF16 pair as FP32 (exact).
__device__ __forceinline__ float2 bf16_pair(uint32_t w) { return make_float2(bf16_lo(w), bf16_hi(w)); }

// UE8M0 code of the smallest power of two >= s (s >= 0), clamped to [0, 254].
__device__ __forceinline__ uint32_t ue8m0_ceil(float s) {
  const uint32_t bits = __float_as_uint(s);
  const uint32_t ex = bits >> 23, man = bits & 0x7fffffu;
  uint32_t e;
  if (bits == 0u) e = 0u;
  else if (ex == 0u) e = man > (1u << 22) ? 1u : 0u;   // subnormal s
  else e = ex + (man != 0u ? 1u : 0u);
  return e > 254u ? 254u : e;
}

// 2^(127 - e) as an FP32 (normal for e < 254, 2^-127 otherwise).
__device__ __forceinline__ float inv_scale(uint32_t e) {
  return e < 254u ? __uint_as_float((254u - e) << 23) : __uint_as_float(0x00400000u);
}

// Lane-wise maximum of two BF16 pairs (finite, non-negative here).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Four FP32 values to E4M3, nearest-even, saturating (a in the lowest byte).
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  unsigned short lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return uint32_t(lo) | (uint32_t(hi) << 16);
}

// Byte offset of scale (row, col) in the 128x4 swizzled block-scale layout
// with `cols` scale columns (a multiple of 4).
__device__ __forceinline__ size_t swizzle_128x4(int row, int col, int cols) {
  const size_t tile = size_t(row / 128) * (cols / 4) + col / 4;
  const int r = row % 128;
  return tile * 512 + (r % 32) * 16 + (r / 32) * 4 + (col % 4);
}

// Next boundary's post-mix and Sinkhorn residual mix of one token, from its
// normalised mixes, in one thread ([GLM] _MixesDeviceKernel):
//   post_j = sigmoid(mixes_{4+j} * scale[1] + base[4+j]) * post_mult
//   logits c[r][k] = mixes_{8+4r+k} * scale[2] + base[8+4r+k]
//   rows: c = exp(c - max_k c) / sum_k + eps
//   `repeat` rounds: (from the second round) rows c /= (row sum + eps);
//                    columns c /= (column sum + eps)
// with the four-term sums paired ((a + b) + (c + d)) and reciprocals
// multiplied in (rcp_fast), the same operations as the side-stream kernel, so
// both give the same bits.
__device__ __forceinline__ float sum4_paired(float a, float b, float c, float d) {
  return __fadd_rn(__fadd_rn(a, b), __fadd_rn(c, d));
}

// Its arguments are values, not a kernel's parameter block by reference (an
// out-of-line function would read that through a generic pointer into
// parameter space, which is slow).
struct MixArgs {
  const float *scale, *base;
  float *post_out, *comb_out;
  float post_mult, eps;
  int repeat;
};

static __device__ __noinline__ void post_and_sinkhorn(const MixArgs p, int t, const float *mix) {
#pragma unroll
  for (int j = 0; j < HC; ++j) {
    const float z = __fadd_rn(__fmul_rn(mix[HC + j], p.scale[1]), p.base[HC + j]);
    p.post_out[(size_t)t * HC + j] = __fmul_rn(sigmoid(z), p.post_mult);
  }
  const float eps = p.eps, s2 = p.scale[2];
  float c[HC * HC];
#pragma unroll
  for (int i = 0; i < HC * HC; ++i) c[i] = __fadd_rn(__fmul_rn(mix[2 * HC + i], s2), p.base[2 * HC + i]);
#pragma unroll
  for (int r = 0; r < HC; ++r) {
    float *x = c + HC * r;
    const float peak = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
#pragma unroll
    for (int k = 0; k < HC; ++k) x[k] = expf(__fsub_rn(x[k], peak));
    const float inv = rcp_fast(sum4_paired(x[0], x[1], x[2], x[3]));
#pragma unroll
    for (int k = 0; k < HC; ++k) x[k] = __fadd_rn(__fmul_rn(x[k], inv), eps);
  }
  auto cols = [&]() {
#pragma unroll
    for (int k = 0; k < HC; ++k) {
      const float inv = rcp_fast(__fadd_rn(sum4_paired(c[k], c[HC + k], c[2 * HC + k], c[3 * HC + k]), eps));
#pragma unroll
      for (int r = 0; r < HC; ++r) c[HC * r + k] = __fmul_rn(c[HC * r + k], inv);
    }
  };
  // round 1: columns; rounds 2 .. repeat: rows, then columns
  cols();
#pragma unroll 4
  for (int it = 1; it < p.repeat; ++it) {
#pragma unroll
    for (int r = 0; r < HC; ++r) {
      float *x = c + HC * r;
      const float inv = rcp_fast(__fadd_rn(sum4_paired(x[0], x[1], x[2], x[3]), eps));
#pragma unroll
      for (int k = 0; k < HC; ++k) x[k] = __fmul_rn(x[k], inv);
    }
    cols();
  }
  float *dst = p.comb_out + (size_t)t * HC * HC;
#pragma unroll
  for (int i = 0; i < HC * HC; ++i) dst[i] = c[i];
}

// Paired four-term sum over the lanes that differ in bits a and 2a.
__device__ __forceinline__ float lane_sum4(float x, int a) {
  const float s = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, a));
  return __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 2 * a));
}

// The same post-mix and Sinkhorn mix with a token spread over 16 lanes, one
// matrix element each (lane 4r + k of the token's half-warp; the whole warp
// calls it, a half-warp per token): a row sum is two butterfly shuffles over
// lanes 4r .. 4r+3 (xor 1 then xor 2 gives (c0 + c1) + (c2 + c3) on every
// lane of the row), a column sum two over lanes k, k+4, k+8, k+12 (xor 4
// then xor 8); lanes 0-3 of the token also compute post.  The operations are
// those of post_and_sinkhorn, so the bits are the same.  `mix` points at the
// token's 24 normalised mixes; half-warps with live == false compute on zeros
// and store nothing.
__device__ __forceinline__ void post_and_sinkhorn16(const MixArgs p, int t, const float *mix, bool live) {
  const int e = threadIdx.x & (HC * HC - 1);
  if (live && e < HC) {
    const float z = __fadd_rn(__fmul_rn(mix[HC + e], p.scale[1]), p.base[HC + e]);
    p.post_out[(size_t)t * HC + e] = __fmul_rn(sigmoid(z), p.post_mult);
  }
  const float eps = p.eps;
  float x = live ? __fadd_rn(__fmul_rn(mix[2 * HC + e], p.scale[2]), p.base[2 * HC + e]) : 0.f;
  // row softmax
  float peak = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  peak = fmaxf(peak, __shfl_xor_sync(0xffffffffu, peak, 2));
  x = expf(__fsub_rn(x, peak));
  x = __fadd_rn(__fmul_rn(x, rcp_fast(lane_sum4(x, 1))), eps);
  // round 1: columns; rounds 2 .. repeat: rows, then columns
  x = __fmul_rn(x, rcp_fast(__fadd_rn(lane_sum4(x, HC), eps)));
#pragma unroll 4
  for (int it = 1; it < p.repeat; ++it) {
    x = __fmul_rn(x, rcp_fast(__fadd_rn(lane_sum4(x, 1), eps)));
    x = __fmul_rn(x, rcp_fast(__fadd_rn(lane_sum4(x, HC), eps)));
  }
  if (live) p.comb_out[(size_t)t * HC * HC + e] = x;
}

// The same post-mix and Sinkhorn mix with a token spread over 4 lanes, one
// matrix row each (lane r of the token's quad): a row sum is the paired sum
// in registers, a column sum two butterfly shuffles over the quad (xor 1
// then xor 2 gives (c0k + c1k) + (c2k + c3k) on every lane), the four
// columns' chains side by side; lane r also computes post_r.  The
// operations are those of post_and_sinkhorn, so the bits are the same.  The
// whole warp calls it, a quad per token; quads with live == false compute on
// zeros and store nothing.
__device__ __forceinline__ void post_and_sinkhorn4(const MixArgs p, int t, const float *mix, bool live) {
  const int r = threadIdx.x & (HC - 1);
  if (live) {
    const float z = __fadd_rn(__fmul_rn(mix[HC + r], p.scale[1]), p.base[HC + r]);
    p.post_out[(size_t)t * HC + r] = __fmul_rn(sigmoid(z), p.post_mult);
  }
  const float eps = p.eps, s2 = p.scale[2];
  float c[HC];
#pragma unroll
  for (int k = 0; k < HC; ++k)
    c[k] = live ? __fadd_rn(__fmul_rn(mix[2 * HC + HC * r + k], s2), p.base[2 * HC + HC * r + k]) : 0.f;
  {
    const float peak = fmaxf(fmaxf(c[0], c[1]), fmaxf(c[2], c[3]));
#pragma unroll
    for (int k = 0; k < HC; ++k) c[k] = expf(__fsub_rn(c[k], peak));
    const float inv = rcp_fast(sum4_paired(c[0], c[1], c[2], c[3]));
#pragma unroll
    for (int k = 0; k < HC; ++k) c[k] = __fadd_rn(__fmul_rn(c[k], inv), eps);
  }
  auto cols = [&]() {
    float s[HC];
#pragma unroll
    for (int k = 0; k < HC; ++k) s[k] = __fadd_rn(c[k], __shfl_xor_sync(0xffffffffu, c[k], 1));
#pragma unroll
    for (int k = 0; k < HC; ++k) s[k] = __fadd_rn(s[k], __shfl_xor_sync(0xffffffffu, s[k], 2));
#pragma unroll
    for (int k = 0; k < HC; ++k) c[k] = __fmul_rn(c[k], rcp_fast(__fadd_rn(s[k], eps)));
  };
  // round 1: columns; rounds 2 .. repeat: rows, then columns
  cols();
#pragma unroll 4
  for (int it = 1; it < p.repeat; ++it) {
    const float inv = rcp_fast(__fadd_rn(sum4_paired(c[0], c[1], c[2], c[3]), eps));
#pragma unroll
    for (int k = 0; k < HC; ++k) c[k] = __fmul_rn(c[k], inv);
    cols();
  }
  if (live) {
    float *dst = p.comb_out + (size_t)t * HC * HC + HC * r;
#pragma unroll
    for (int k = 0; k < HC; ++k) dst[k] = c[k];
  }
}

}  // namespace mhc
