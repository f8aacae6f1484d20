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
// Layout: CTAs of 8 warps, grid-stride over (token, 256-column chunk) jobs.
// Lane l of every warp takes the chunk's 16-byte fragment l, so that a warp
// reads 512 contiguous bytes of a route row; warp w folds ranks w, w + 8, ...,
// loading a rank's routes four at a time before their multiply-adds.
// The folded x_r go to shared memory, and warp 0 adds them in rank order.
//
// Page: [DSV] vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc.
#include "device_common.cuh"
#include "launch.cuh"

namespace mhc {
namespace {

constexpr int WARPS = 8;
constexpr int NT = WARPS * 32;
constexpr int KB = 4;                        // routes loaded per batch
constexpr int TP_MAX = 32;

// Four routes a batch and six CTAs an SM (40 registers a thread, 24 bytes
// spilled): more warps with gathers in flight than eight routes at four CTAs,
// measured 4 % faster a MoE call at 256 tokens; eight routes at six CTAs
// spill 268 bytes and ran 27 % slower.
__global__ void __launch_bounds__(NT, 6) k_moe_fold(const FoldParams p) {
  extern __shared__ float4 xs[];             // [tp][32][2]: x_r of the chunk's 32 fragments
  const int H = p.hidden, K = p.top_k, nfrag = H / VEC;
  const int warp = int(threadIdx.x) >> 5, lane = int(threadIdx.x) & 31;
  const int chunks = (nfrag + 31) / 32;
  for (int job = blockIdx.x; job < p.m * chunks; job += gridDim.x) {
    const int t = job / chunks, fr = (job % chunks) * 32 + lane;
    const bool live = fr < nfrag;
#pragma unroll 1
    for (int r = warp; r < p.tp; r += WARPS) {
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = 0.f;
      if (live) {
        // the shared expert's row does not depend on the route indices: its
        // load is in flight with theirs and the routes'
        const uint4 sv = ld_stream(p.shared + ((size_t)r * p.m + t) * H + (size_t)fr * VEC);
        const int32_t *ix = p.idx + ((size_t)r * p.m + t) * K;
        const float *wt = p.weights + (size_t)t * K;
        const uint16_t *rows = p.routed + (size_t)r * p.rows_per_rank * H + (size_t)fr * VEC;
#pragma unroll 1
        for (int k0 = 0; k0 < K; k0 += KB) {
          int row[KB];
          uint4 v[KB];
#pragma unroll
          for (int i = 0; i < KB; ++i) {
            row[i] = k0 + i < K ? ix[k0 + i] : -1;
            if (row[i] < -1 || row[i] >= p.rows_per_rank) {
              atomicOr(p.err, 1u);
              row[i] = -1;
            }
            v[i] = row[i] >= 0 ? ld_stream(rows + (size_t)row[i] * H) : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int i = 0; i < KB; ++i) {
            if (row[i] >= 0) {
              float a[8];
              unpack8(v[i], a);
              const float w = wt[k0 + i];
#pragma unroll
              for (int e = 0; e < 8; ++e) x[e] = __fmaf_rn(a[e], w, x[e]);
            }
          }
        }
        float s[8];
        unpack8(sv, s);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = __fadd_rn(x[e], s[e]);
        round8(x);
      }
      xs[(r * 32 + lane) * 2] = make_float4(x[0], x[1], x[2], x[3]);
      xs[(r * 32 + lane) * 2 + 1] = make_float4(x[4], x[5], x[6], x[7]);
    }
    __syncthreads();
    if (warp == 0 && live) {
      // y = bf16(((0 + x_0) + x_1) + ...)
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = 0.f;
#pragma unroll 1
      for (int r = 0; r < p.tp; ++r) {
        const float4 a = xs[(r * 32 + lane) * 2], b = xs[(r * 32 + lane) * 2 + 1];
        y[0] = __fadd_rn(y[0], a.x); y[1] = __fadd_rn(y[1], a.y);
        y[2] = __fadd_rn(y[2], a.z); y[3] = __fadd_rn(y[3], a.w);
        y[4] = __fadd_rn(y[4], b.x); y[5] = __fadd_rn(y[5], b.y);
        y[6] = __fadd_rn(y[6], b.z); y[7] = __fadd_rn(y[7], b.w);
      }
      st_vec(p.y + (size_t)t * H + (size_t)fr * VEC, round8(y));
    }
    __syncthreads();   // the next job's x_r overwrite these
  }
}

}  // namespace

cudaError_t launch_moe_fold(const FoldParams &p, int ctas, cudaStream_t stream) {
  if (p.tp < 1 || p.tp > TP_MAX || p.top_k < 1 || p.top_k > 64 || p.hidden % VEC) return cudaErrorInvalidValue;
  const int jobs = p.m * ((p.hidden / VEC + 31) / 32);
  const int grid = jobs < ctas ? jobs : ctas;
  k_moe_fold<<<grid, NT, size_t(p.tp) * 32 * 2 * sizeof(float4), stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mhc
