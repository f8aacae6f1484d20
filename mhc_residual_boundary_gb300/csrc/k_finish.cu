// k_finish.cu -- finish kernel of the mHC boundary.  Per token:
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
// Layout on the GPU: persistent CTAs of 256 threads, two per SM where the
// shared memory allows, each taking tokens blockIdx.x, blockIdx.x + gridDim.x,
// ...  A token's four new streams are one contiguous 8H-byte run of
// residual_out and its partial sums one 16-byte-padded row, so each token
// arrives in shared memory by two bulk copies into a two-slot ring; thread 0
// refills a slot as soon as the token in it has been collapsed, so the next
// token's copies are in flight while this one is normalised and stored, and
// the two CTAs of an SM interleave their per-token barriers.  gamma is held in
// registers for the whole kernel.  Every wait is bounded; a
// wait that gives up sets bit 1 of the error word.
//
// Pages: [GLM] vllm.models.glm5next.nvidia.specialized_decode.all_reduce_mhc,
//        [DSV] vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc.
#include "device_common.cuh"
#include "launch.cuh"
#include "tcgen05.cuh"

namespace mhc {
namespace {

constexpr int NT = 256;
constexpr int NFMAX = MAX_HIDDEN / VEC / NT;   // fragments of a stream row per thread at most
static_assert(NFMAX == 8, "launch_finish dispatches NF = 1 .. 8");
constexpr int MAX_SLOTS = 2;
constexpr size_t SMEM_BUDGET = 110 * 1024;     // ring bytes of one CTA: two CTAs fit an SM
constexpr size_t SMEM_LIMIT = 200 * 1024;      // one slot at H = 16384 is 153 KB
constexpr uint32_t WAIT_LIMIT = 1u << 22;      // polls before a wait gives up

// Bytes of one ring slot: the token's four stream rows, then its partial-sum row.
__host__ __device__ inline size_t slot_bytes(int hidden, int part_stride) {
  return size_t(HC) * hidden * 2 + size_t(part_stride) * 4;
}
inline int ring_slots(int hidden, int part_stride) {
  const size_t n = SMEM_BUDGET / slot_bytes(hidden, part_stride);
  return n < 1 ? 1 : n > size_t(MAX_SLOTS) ? MAX_SLOTS : int(n);
}

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
__global__ void __launch_bounds__(NT, 2) k_finish(const FinishParams p, int slots) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[MAX_SLOTS];
  __shared__ float tot_s[VALUES];
  __shared__ float red_s[NT / 32];
  __shared__ int abort_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.hidden;
  const int nfrag = H / VEC;
  const size_t sbytes = slot_bytes(H, p.part_stride);
  const uint32_t stream_bytes = uint32_t(HC) * H * 2, part_bytes = uint32_t(p.part_stride) * 4;
  // tokens of this CTA: blockIdx.x + k * gridDim.x, k < n_tok
  const int n_tok = (p.m - int(blockIdx.x) + int(gridDim.x) - 1) / int(gridDim.x);

  if (tid == 0) {
    for (int i = 0; i < slots; ++i) tc::mbar_init(&full[i], 1);
    abort_s = 0;
    tc::mbar_init_fence();
  }
  __syncthreads();

  // Nothing below may read the stage kernel's outputs before this point.
  pdl_wait();

  auto fill = [&](int k) {   // thread 0: token k of this CTA into slot k % slots
    const int t = int(blockIdx.x) + k * int(gridDim.x);
    unsigned char *dst = smem + size_t(k % slots) * sbytes;
    uint64_t *bar = &full[k % slots];
    tc::mbar_arrive_expect_tx(bar, stream_bytes + part_bytes);
    tc::bulk_load(dst, p.streams + (size_t)t * HC * H, stream_bytes, bar);
    tc::bulk_load(dst + stream_bytes, p.part + (size_t)t * p.part_stride, part_bytes, bar);
  };
  int filled = 0;   // tokens whose copies were issued (thread 0)
  if (tid == 0)
    for (; filled < slots && filled < n_tok; ++filled) fill(filled);

  const int cols = H / 32;
  uint4 gam[NF];   // this thread's fragments of gamma, the same for every token
#pragma unroll
  for (int i = 0; i < NF; ++i) {
    const int fr = tid + i * NT;
    gam[i] = fr < nfrag ? ld_vec(p.gamma + (size_t)fr * VEC) : make_uint4(0u, 0u, 0u, 0u);
  }
  for (int k = 0; k < n_tok; ++k) {
    const int t = int(blockIdx.x) + k * int(gridDim.x);
    const unsigned char *slot = smem + size_t(k % slots) * sbytes;
    if (!tc::mbar_wait_bounded(&full[k % slots], uint32_t(k / slots) & 1u, WAIT_LIMIT)) abort_s = 1;
    const uint16_t *sv = reinterpret_cast<const uint16_t *>(slot);
    const float *part_s = reinterpret_cast<const float *>(slot + stream_bytes);

    // 1. partial sums over the slices, in slice order within each lane
    for (int v = warp; v < VALUES; v += NT / 32) {
      float s = 0.f;
      for (int sl = lane; sl < p.slices; sl += 32) s += part_s[sl * VALUES + v];
      s = warp_sum(s);
      if (lane == 0) tot_s[v] = s;
    }
    __syncthreads();
    if (abort_s) break;

    // 2. mixes (for the side kernel) and pre, the latter on every thread
    const float rstd = __frcp_rn(sqrtf(__fadd_rn(__fdiv_rn(tot_s[MIX], float(HC * H)), p.rms_eps)));
    if (tid < MIX) {
      const float mix = __fmul_rn(tot_s[tid], rstd);
      p.mixes[(size_t)t * MIX + tid] = mix;
      if (p.mixes_out) p.mixes_out[(size_t)t * MIX + tid] = mix;
    }
    float pre[HC];
#pragma unroll
    for (int j = 0; j < HC; ++j) {
      const float z = __fadd_rn(__fmul_rn(__fmul_rn(tot_s[j], rstd), p.scale[0]), p.base[j]);
      pre[j] = __fadd_rn(sigmoid(z), p.hc_eps);
    }
    if (p.pre_out && tid < HC)
      p.pre_out[(size_t)t * HC + tid] = tid == 0 ? pre[0] : tid == 1 ? pre[1] : tid == 2 ? pre[2] : pre[3];

    // 3. collapse, kept in registers as BF16 for the normalisation
    const float p0 = pre[0], p1 = pre[1], p2 = pre[2], p3 = pre[3];
    uint4 cfr[NF];
    float ssq = 0.f;
#pragma unroll
    for (int i = 0; i < NF; ++i) {
      const int fr = tid + i * NT;
      cfr[i] = make_uint4(0u, 0u, 0u, 0u);
      if (fr < nfrag) {
        float n0[8], n1[8], n2[8], n3[8], c[8];
        const uint16_t *s = sv + (size_t)fr * VEC;
        unpack8(*reinterpret_cast<const uint4 *>(s), n0);
        unpack8(*reinterpret_cast<const uint4 *>(s + H), n1);
        unpack8(*reinterpret_cast<const uint4 *>(s + 2 * H), n2);
        unpack8(*reinterpret_cast<const uint4 *>(s + 3 * H), n3);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          c[e] = __fadd_rn(__fadd_rn(__fmul_rn(n0[e], p0), __fmul_rn(n1[e], p1)),
                           __fadd_rn(__fmul_rn(n2[e], p2), __fmul_rn(n3[e], p3)));
        cfr[i] = round8(c);
#pragma unroll
        for (int e = 0; e < 8; ++e) ssq = fmaf(c[e], c[e], ssq);
      }
    }
    ssq = warp_sum(ssq);
    if (lane == 0) red_s[warp] = ssq;
    // the slot's next fill is an async-proxy write after these generic reads
    tc::fence_proxy_async_smem();
    __syncthreads();
    // the slot has been read: it takes the token `slots` places further on
    if (tid == 0 && filled < n_tok) fill(filled++);
    float sq = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) sq += red_s[w];
    const float ir = __frcp_rn(sqrtf(__fadd_rn(__fdiv_rn(sq, float(H)), p.norm_eps)));

    // 4. normalise, store, optional MXFP8 (4 consecutive lanes = one block)
#pragma unroll
    for (int i = 0; i < NF; ++i) {
      const int fr = tid + i * NT;
      const bool live = fr < nfrag;
      float o[8];
      if (live) {
        float c[8], g[8];
        unpack8(cfr[i], c);
        unpack8(gam[i], g);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = __fmul_rn(__fmul_rn(c[e], ir), g[e]);
        st_vec(p.layer_input + (size_t)t * H + (size_t)fr * VEC, round8(o));
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
  }
  pdl_launch_dependents();

  // padding rows of the scale layout: zero their scales (4 columns a store)
  if (p.mx_scales) {
    const int padded = (p.m + 127) / 128 * 128;
    for (int row = p.m + int(blockIdx.x); row < padded; row += int(gridDim.x))
      for (int c4 = tid; c4 < cols / 4; c4 += NT)
        *reinterpret_cast<uint32_t *>(p.mx_scales + swizzle_128x4(row, c4 * 4, cols)) = 0u;
  }
  if (tid == 0) {
    if (abort_s && p.err) atomicOr(p.err, 2u);
    // copies still in flight land before the CTA may exit
    for (int k = filled - slots; k < filled; ++k)
      if (k >= 0) tc::mbar_wait_bounded(&full[k % slots], uint32_t(k / slots) & 1u, WAIT_LIMIT);
  }
}

}  // namespace

using FinishKernel = void (*)(FinishParams, int);
constexpr FinishKernel kFinish[NFMAX] = {k_finish<1>, k_finish<2>, k_finish<3>, k_finish<4>,
                                         k_finish<5>, k_finish<6>, k_finish<7>, k_finish<8>};

cudaError_t finish_set_attributes() {
  for (FinishKernel k : kFinish) {
    const cudaError_t e =
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(SMEM_LIMIT));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_finish(const FinishParams &p, int ctas, cudaStream_t stream, bool pdl) {
  const int nf = (p.hidden / VEC + NT - 1) / NT;
  if (nf < 1 || nf > NFMAX || p.part_stride % 4 || p.part_stride < p.slices * VALUES) return cudaErrorInvalidValue;
  const int slots = ring_slots(p.hidden, p.part_stride);
  const size_t smem = size_t(slots) * slot_bytes(p.hidden, p.part_stride);
  if (smem > SMEM_LIMIT) return cudaErrorInvalidValue;
  // two CTAs an SM when their rings fit beside each other (227 KB an SM)
  const int per_sm = smem <= SMEM_BUDGET ? 2 : 1;
  const int grid = ctas * per_sm;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.m < grid ? p.m : grid);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kFinish[nf - 1], p, slots);
}

}  // namespace mhc
