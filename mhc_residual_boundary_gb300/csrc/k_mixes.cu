// k_mixes.cu -- side-stream kernel: the next boundary's post-mix and Sinkhorn
// residual mix from this boundary's raw mixes ([GLM] _MixesDeviceKernel.kernel
// and _MixesDeviceKernel._sinkhorn).
//
//   post_j = sigmoid(mixes_{4+j} * scale[1] + base[4+j]) * post_mult
//   logits c[r][k] = mixes_{8+4r+k} * scale[2] + base[8+4r+k]
//   rows: c = exp(c - max_k c) / sum_k + eps
//   `repeat` rounds: (from the second round) rows c /= (row sum + eps);
//                    columns c /= (column sum + eps)
// with the four-term sums paired ((a + b) + (c + d)) and reciprocals
// multiplied in, as on the page.
//
// The rounds are a chain of dependent steps per token, so the kernel spreads
// a token over 16 lanes, one matrix element each (lane 4r + k of the token's
// half-warp): a row sum is two butterfly shuffles over lanes 4r .. 4r+3
// (xor 1 then xor 2 gives (c0 + c1) + (c2 + c3) on every lane of the row), a
// column sum two over lanes k, k+4, k+8, k+12 (xor 4 then xor 8).  Lanes 0-3
// of the token also compute post.  Two tokens per warp, eight per CTA.
//
// Page: [GLM] vllm.models.glm5next.nvidia.specialized_decode.all_reduce_mhc.
#include "device_common.cuh"
#include "launch.cuh"

namespace mhc {
namespace {

constexpr int NT = 128;
constexpr int LANES = HC * HC;             // lanes per token
constexpr int TOKENS = NT / LANES;         // tokens per CTA

__global__ void __launch_bounds__(NT) k_mixes(const MixesParams p) {
  const int t = blockIdx.x * TOKENS + threadIdx.x / LANES;
  // the whole warp runs the shuffles; lanes of a token past m compute on zeros
  const bool live = t < p.m;
  const MixArgs ma = {p.scale, p.base, p.post_out, p.comb_out, p.post_mult, p.eps, p.repeat};
  post_and_sinkhorn16(ma, t, p.mixes + (size_t)(live ? t : 0) * MIX, live);
}

}  // namespace

cudaError_t launch_mixes(const MixesParams &p, cudaStream_t stream) {
  k_mixes<<<(p.m + TOKENS - 1) / TOKENS, NT, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mhc
