// k_moe_fold.cu -- stage 1 of a MoE-finalize boundary ([DSV]
// _QuadFinalizePublishDeviceKernel.kernel, then the rank-order sum of
// _LamportMHCDeviceKernel.kernel): per rank r
//
//   x_r = bf16( fma-chain_k( routed_r[idx_r[t][k]], w[t][k] ) + shared_r[t] )
//
// (one fused multiply-add per held route in k order, from +0; a route index
// of -1 is a route the rank does not hold), then y = bf16(sum_r x_r) added in
// rank order from +0.  y goes to a [m][H] BF16 buffer that the tensor-core
// stage kernel takes as its single partial (a one-term rank sum from +0
// returns y unchanged), so the MoE call shares the post-mix and GEMV path.
// An index outside [-1, rows) sets bit 0 of the error word and is treated as
// a route not held.
//
// Layout: one CTA of 128 threads per (token, 1024-column chunk), grid-stride;
// the token's indices and weights are staged in shared memory, and each
// thread takes one 16-byte fragment, loading eight routes' fragments before
// the multiply-adds so that eight loads are in flight per thread.
//
// Page: [DSV] vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc.
#include "device_common.cuh"
#include "launch.cuh"

namespace mhc {
namespace {

constexpr int NT = 128;
constexpr int KB = 8;                        // routes loaded per batch
constexpr int MAX_ROUTES = 32 * 64;          // tp * top_k the shared staging holds

__global__ void __launch_bounds__(NT) k_moe_fold(const FoldParams p) {
  __shared__ int idx_s[MAX_ROUTES];
  __shared__ float w_s[64];
  const int H = p.hidden, K = p.top_k, routes = p.tp * p.top_k;
  const int nfrag = H / VEC, chunks = (nfrag + NT - 1) / NT;
  for (int job = blockIdx.x; job < p.m * chunks; job += gridDim.x) {
    const int t = job / chunks, fr = (job % chunks) * NT + threadIdx.x;
    __syncthreads();   // the previous token's routes are no longer read
    for (int e = threadIdx.x; e < routes; e += NT) {
      const int r = e / K, k = e % K;
      int row = p.idx[((size_t)r * p.m + t) * K + k];
      if (row < -1 || row >= p.rows_per_rank) {
        atomicOr(p.err, 1u);
        row = -1;
      }
      idx_s[e] = row;
    }
    for (int k = threadIdx.x; k < K; k += NT) w_s[k] = p.weights[(size_t)t * K + k];
    __syncthreads();
    if (fr < nfrag) {
      const size_t h = size_t(fr) * VEC;
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = 0.f;
#pragma unroll 1
      for (int r = 0; r < p.tp; ++r) {
        const uint16_t *rows_r = p.routed + (size_t)r * p.rows_per_rank * H + h;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll 1
        for (int k0 = 0; k0 < K; k0 += KB) {
          uint4 x[KB];
#pragma unroll
          for (int i = 0; i < KB; ++i) {
            const int k = k0 + i;
            const int row = k < K ? idx_s[r * K + k] : -1;
            x[i] = row >= 0 ? ld_stream(rows_r + (size_t)row * H) : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int i = 0; i < KB; ++i) {
            const int k = k0 + i;
            if (k < K && idx_s[r * K + k] >= 0) {
              float v[8];
              unpack8(x[i], v);
              const float w = w_s[k];
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[e] = __fmaf_rn(v[e], w, acc[e]);
            }
          }
        }
        float s[8];
        unpack8(ld_stream(p.shared + ((size_t)r * p.m + t) * H + h), s);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], s[e]);
        round8(acc);
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = __fadd_rn(y[e], acc[e]);
      }
      st_vec(p.y + (size_t)t * H + h, round8(y));
    }
  }
}

}  // namespace

cudaError_t launch_moe_fold(const FoldParams &p, int ctas, cudaStream_t stream) {
  if (p.tp < 1 || p.top_k < 1 || p.top_k > 64 || p.tp * p.top_k > MAX_ROUTES || p.hidden % VEC)
    return cudaErrorInvalidValue;
  const int jobs = p.m * ((p.hidden / VEC + NT - 1) / NT);
  const int grid = jobs < ctas ? jobs : ctas;
  k_moe_fold<<<grid, NT, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mhc
