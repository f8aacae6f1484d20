// k_mixes.cu -- side-stream kernel: the next boundary's post-mix and Sinkhorn
// residual mix from this boundary's raw mixes, one thread per token, one warp
// per CTA ([GLM] _MixesDeviceKernel.kernel and _MixesDeviceKernel._sinkhorn).
//
//   post_j = sigmoid(mixes_{4+j} * scale[1] + base[4+j]) * post_mult
//   logits c[r][k] = mixes_{8+4r+k} * scale[2] + base[8+4r+k]
//   rows: c = exp(c - max_k c) / sum_k + eps
//   `repeat` rounds: (from the second round) rows c /= (row sum + eps);
//                    columns c /= (column sum + eps)
// with the four-term sums paired ((a + b) + (c + d)) and 1/x reciprocals, as
// on the page.  The matrix lives in 16 registers.
//
// Page: [GLM] vllm.models.glm5next.nvidia.specialized_decode.all_reduce_mhc.
#include "device_common.cuh"
#include "launch.cuh"

namespace mhc {
namespace {

__device__ __forceinline__ float sigmoid(float z) {
  return __frcp_rn(__fadd_rn(1.0f, expf(-z)));
}

__global__ void __launch_bounds__(32) k_mixes(const MixesParams p) {
  const int t = blockIdx.x * 32 + threadIdx.x;
  if (t >= p.m) return;
  const float *row = p.mixes + (size_t)t * MIX;
  const float s1 = p.scale[1], s2 = p.scale[2], eps = p.eps;
#pragma unroll
  for (int j = 0; j < HC; ++j) {
    const float z = __fadd_rn(__fmul_rn(row[HC + j], s1), p.base[HC + j]);
    p.post_out[(size_t)t * HC + j] = __fmul_rn(sigmoid(z), p.post_mult);
  }
  float c[HC * HC];
#pragma unroll
  for (int i = 0; i < HC * HC; ++i) c[i] = __fadd_rn(__fmul_rn(row[2 * HC + i], s2), p.base[2 * HC + i]);
#pragma unroll
  for (int r = 0; r < HC; ++r) {
    float *x = c + r * HC;
    const float peak = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
#pragma unroll
    for (int k = 0; k < HC; ++k) x[k] = expf(__fsub_rn(x[k], peak));
    const float inv = __frcp_rn(__fadd_rn(__fadd_rn(x[0], x[1]), __fadd_rn(x[2], x[3])));
#pragma unroll
    for (int k = 0; k < HC; ++k) x[k] = __fadd_rn(__fmul_rn(x[k], inv), eps);
  }
  for (int it = 0; it < p.repeat; ++it) {
    if (it > 0) {
#pragma unroll
      for (int r = 0; r < HC; ++r) {
        float *x = c + r * HC;
        const float inv = __frcp_rn(__fadd_rn(__fadd_rn(__fadd_rn(x[0], x[1]), __fadd_rn(x[2], x[3])), eps));
#pragma unroll
        for (int k = 0; k < HC; ++k) x[k] = __fmul_rn(x[k], inv);
      }
    }
#pragma unroll
    for (int k = 0; k < HC; ++k) {
      const float inv = __frcp_rn(__fadd_rn(
          __fadd_rn(__fadd_rn(c[k], c[HC + k]), __fadd_rn(c[2 * HC + k], c[3 * HC + k])), eps));
#pragma unroll
      for (int r = 0; r < HC; ++r) c[r * HC + k] = __fmul_rn(c[r * HC + k], inv);
    }
  }
#pragma unroll
  for (int i = 0; i < HC * HC; ++i) p.comb_out[(size_t)t * HC * HC + i] = c[i];
}

}  // namespace

cudaError_t launch_mixes(const MixesParams &p, cudaStream_t stream) {
  k_mixes<<<(p.m + 31) / 32, 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mhc
