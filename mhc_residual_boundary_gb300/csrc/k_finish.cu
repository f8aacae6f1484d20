// k_finish.cu -- finish kernel of the mHC boundary: one CTA per token.
//
//  1. sums the stage kernel's per-slice partials in slice order (24 GEMV
//     outputs and the sum of squares of the new streams);
//  2. rstd = 1/sqrt(ss / (4H) + rms_eps), mixes = raw * rstd (kept for the
//     side kernel), pre_j = sigmoid(mixes_j * scale[0] + base[j]) + hc_eps
//     ([GLM] _BoundaryDeviceKernel.kernel, "rstd", "pre_mix");
//  3. collapse c = bf16(sum_j new_j * pre_j), inv_rms = 1/sqrt(sum c^2 / H +
//     norm_eps), out = bf16((c * inv_rms) * gamma) ([GLM] "collapse",
//     "prenorm", "inv_rms"; [DSV] _LamportMHCDeviceKernel.kernel);
//  4. optionally the MXFP8 copy of out: per 32-element block the UE8M0 code of
//     amax * (1/448) rounded up to a power of two, E4M3 values of
//     out * 2^(127 - e) with hardware nearest-even satfinite conversions,
//     scales at the 128x4 swizzled offset, padding-row scales zeroed ([DSV]
//     _LamportMHCDeviceKernel.kernel, quantize branch).
//
// Pages: [GLM] vllm.models.glm5next.nvidia.specialized_decode.all_reduce_mhc,
//        [DSV] vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc.
#include "device_common.cuh"
#include "launch.cuh"

namespace mhc {
namespace {

constexpr int NT = 256;
constexpr int MAXF = MAX_HIDDEN / VEC / NT;   // fragments per thread at most
static_assert(MAXF == 8, "launch_finish dispatches NF = 1 .. 8");

__device__ __forceinline__ float sigmoid(float z) {
  return __frcp_rn(__fadd_rn(1.0f, expf(-z)));
}

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

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  unsigned short lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return uint32_t(lo) | (uint32_t(hi) << 16);
}

__device__ __forceinline__ size_t swizzle_128x4(int row, int col, int cols) {
  const size_t tile = size_t(row / 128) * (cols / 4) + col / 4;
  const int r = row % 128;
  return tile * 512 + (r % 32) * 16 + (r / 32) * 4 + (col % 4);
}

// NF: 16-byte fragments of a stream row per thread (ceil(H / 8 / 256)).
template <int NF>
__global__ void __launch_bounds__(NT) k_finish(const FinishParams p) {
  extern __shared__ float part_s[];   // [slices][25] of this token
  __shared__ float tot_s[VALUES];
  __shared__ float pre_s[HC];
  __shared__ float red_s[NT / 32];
  __shared__ float ir_s;
  const int t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.hidden;
  const int nfrag = H / VEC;

  // Nothing below may read the stage kernel's outputs before this point.
  pdl_wait();

  // the token's new streams go to registers first, so that their latency
  // overlaps the partial-sum reduction
  uint4 sv[NF][HC];
#pragma unroll
  for (int i = 0; i < NF; ++i) {
    const int fr = tid + i * NT;
#pragma unroll
    for (int j = 0; j < HC; ++j)
      sv[i][j] = fr < nfrag ? ld_stream(p.streams + ((size_t)t * HC + j) * H + (size_t)fr * VEC)
                            : make_uint4(0u, 0u, 0u, 0u);
  }
  const int np = p.slices * VALUES;
  const float *prow = p.part + (size_t)t * np;
  for (int e = tid; e < np; e += NT) part_s[e] = prow[e];
  __syncthreads();

  // 1. partial sums over the slices, in slice order within each lane
  for (int v = warp; v < VALUES; v += NT / 32) {
    float s = 0.f;
    for (int sl = lane; sl < p.slices; sl += 32) s += part_s[sl * VALUES + v];
    s = warp_sum(s);
    if (lane == 0) tot_s[v] = s;
  }
  __syncthreads();

  // 2. mixes and pre
  if (tid < MIX) {
    const float rstd = __frcp_rn(sqrtf(__fadd_rn(__fdiv_rn(tot_s[MIX], float(HC * H)), p.rms_eps)));
    const float mix = __fmul_rn(tot_s[tid], rstd);
    p.mixes[(size_t)t * MIX + tid] = mix;
    if (p.mixes_out) p.mixes_out[(size_t)t * MIX + tid] = mix;
    if (tid < HC) {
      const float z = __fadd_rn(__fmul_rn(mix, p.scale[0]), p.base[tid]);
      const float pre = __fadd_rn(sigmoid(z), p.hc_eps);
      pre_s[tid] = pre;
      if (p.pre_out) p.pre_out[(size_t)t * HC + tid] = pre;
    }
  }
  __syncthreads();
  pdl_launch_dependents();

  // 3. collapse, kept in registers as BF16 for the normalisation
  const float p0 = pre_s[0], p1 = pre_s[1], p2 = pre_s[2], p3 = pre_s[3];
  uint4 cfr[NF];
  float ssq = 0.f;
#pragma unroll
  for (int i = 0; i < NF; ++i) {
    float n0[8], n1[8], n2[8], n3[8], c[8];
    unpack8(sv[i][0], n0);
    unpack8(sv[i][1], n1);
    unpack8(sv[i][2], n2);
    unpack8(sv[i][3], n3);
#pragma unroll
    for (int e = 0; e < 8; ++e)
      c[e] = __fadd_rn(__fadd_rn(__fmul_rn(n0[e], p0), __fmul_rn(n1[e], p1)),
                       __fadd_rn(__fmul_rn(n2[e], p2), __fmul_rn(n3[e], p3)));
    cfr[i] = round8(c);   // fragments past H hold zeros and add nothing
#pragma unroll
    for (int e = 0; e < 8; ++e) ssq = fmaf(c[e], c[e], ssq);
  }
  ssq = warp_sum(ssq);
  if (lane == 0) red_s[warp] = ssq;
  __syncthreads();
  if (tid == 0) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) s += red_s[w];
    ir_s = __frcp_rn(sqrtf(__fadd_rn(__fdiv_rn(s, float(H)), p.norm_eps)));
  }
  __syncthreads();
  const float ir = ir_s;

  // 4. normalise, store, optional MXFP8 (4 consecutive lanes = one block)
  const int cols = H / 32;
#pragma unroll
  for (int i = 0; i < NF; ++i) {
    const int fr = tid + i * NT;
    const bool live = fr < nfrag;
    float o[8];
    uint4 ob = make_uint4(0u, 0u, 0u, 0u);
    if (live) {
      float c[8], g[8];
      unpack8(cfr[i], c);
      unpack8(ld_vec(p.gamma + (size_t)fr * VEC), g);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = __fmul_rn(__fmul_rn(c[e], ir), g[e]);
      ob = round8(o);
      st_vec(p.layer_input + (size_t)t * H + (size_t)fr * VEC, ob);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = 0.f;
    }
    if (p.mx_values) {
      float amax = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(o[e]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const uint32_t e8 = ue8m0_ceil(__fmul_rn(amax, 1.0f / 448.0f));
      const float inv = inv_scale(e8);
      if (live) {
        uint2 q;
        q.x = e4m3x4(__fmul_rn(o[0], inv), __fmul_rn(o[1], inv), __fmul_rn(o[2], inv), __fmul_rn(o[3], inv));
        q.y = e4m3x4(__fmul_rn(o[4], inv), __fmul_rn(o[5], inv), __fmul_rn(o[6], inv), __fmul_rn(o[7], inv));
        *reinterpret_cast<uint2 *>(p.mx_values + (size_t)t * H + (size_t)fr * VEC) = q;
        if ((fr & 3) == 0) p.mx_scales[swizzle_128x4(t, fr / 4, cols)] = uint8_t(e8);
      }
    }
  }

  // padding rows of the scale layout: zero their scales (4 columns a store)
  if (p.mx_scales) {
    const int padded = (p.m + 127) / 128 * 128;
    for (int row = p.m + t; row < padded; row += gridDim.x)
      for (int c4 = tid; c4 < cols / 4; c4 += NT)
        *reinterpret_cast<uint32_t *>(p.mx_scales + swizzle_128x4(row, c4 * 4, cols)) = 0u;
  }
}

}  // namespace

cudaError_t launch_finish(const FinishParams &p, cudaStream_t stream, bool pdl) {
  using Kernel = void (*)(FinishParams);
  static const Kernel kernels[MAXF] = {k_finish<1>, k_finish<2>, k_finish<3>, k_finish<4>,
                                       k_finish<5>, k_finish<6>, k_finish<7>, k_finish<8>};
  const int nf = (p.hidden / VEC + NT - 1) / NT;
  if (nf < 1 || nf > MAXF) return cudaErrorInvalidValue;
  const size_t smem = size_t(p.slices) * VALUES * sizeof(float);
  if (smem > 48 * 1024) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.m);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernels[nf - 1], p);
}

}  // namespace mhc
