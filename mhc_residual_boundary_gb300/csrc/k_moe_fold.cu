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
// Layout: CTAs of 8 warps, three to an SM, grid-stride over (token,
// 1024-column chunk) jobs.  Lane l of every warp takes the chunk's 16-byte
// fragments l, l + 32, l + 64 and l + 96, so that a warp reads 2 KB of a
// route row in four 512-byte runs, with eight loads of two routes in flight
// a lane; warp w folds ranks w, w + 8, ...  The shared expert's row of the
// rank is copied by cp.async into the rank's slots of the rank buffer (2 KB a
// rank), where it waits without holding registers; the folded x_r, rounded
// to BF16, replace it there, and warps 0-3 add them in rank order, a
// fragment a lane.  Every CTA lets the stage kernel's launch begin at
// its start, so that stage CTAs take the SMs this grid leaves as they empty.
//
// Page: [DSV] vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc.
#include "device_common.cuh"
#include "launch.cuh"
#include "tcgen05.cuh"

namespace mhc {
namespace {

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

constexpr int WARPS = 8;
constexpr int NT = WARPS * 32;
constexpr int KB = 2;                        // routes loaded per batch
constexpr int FR = 4;                        // 16-byte fragments a lane, 512 bytes apart
constexpr int CHUNK = 32 * FR;               // fragments a job (2 KB of a route row)
constexpr int TP_MAX = 32;

__global__ void __launch_bounds__(NT, 3) k_moe_fold(const FoldParams p) {
  extern __shared__ uint4 xs[];              // [tp][CHUNK]: x_r of the chunk's fragments, BF16 (rounded already)
  const int H = p.hidden, K = p.top_k, nfrag = H / VEC;
  const int warp = int(threadIdx.x) >> 5, lane = int(threadIdx.x) & 31;
  const int chunks = (nfrag + CHUNK - 1) / CHUNK;
  const uint32_t xs_addr = tc::smem_addr(xs);
  // the stage kernel that follows may place its CTAs on SMs this grid leaves
  // and stage its layer weight there; it reads y only after this grid ends
  pdl_launch_dependents();
  for (int job = blockIdx.x; job < p.m * chunks; job += gridDim.x) {
    const int t = job / chunks, fr0 = (job % chunks) * CHUNK + lane;
#pragma unroll 1
    for (int r = warp; r < p.tp; r += WARPS) {
      float x[FR][8];
#pragma unroll
      for (int g = 0; g < FR; ++g)
#pragma unroll
        for (int e = 0; e < 8; ++e) x[g][e] = 0.f;
      // the shared expert's rows do not depend on the route indices: they
      // are copied into this rank's slots of the rank buffer, in flight with
      // the routes' loads and holding no registers
#pragma unroll
      for (int g = 0; g < FR; ++g)
        if (fr0 + 32 * g < nfrag)
          cp_async16(xs_addr + uint32_t(r * CHUNK + 32 * g + lane) * 16u,
                     p.shared + ((size_t)r * p.m + t) * H + (size_t)(fr0 + 32 * g) * VEC);
      cp_async_commit();
      const int32_t *ix = p.idx + ((size_t)r * p.m + t) * K;
      const float *wt = p.weights + (size_t)t * K;
      const uint16_t *rows = p.routed + (size_t)r * p.rows_per_rank * H + (size_t)fr0 * VEC;
#pragma unroll 1
      for (int k0 = 0; k0 < K; k0 += KB) {
        int row[KB];
        uint4 v[KB][FR];
#pragma unroll
        for (int i = 0; i < KB; ++i) {
          row[i] = k0 + i < K ? ix[k0 + i] : -1;
          if (row[i] < -1 || row[i] >= p.rows_per_rank) {
            atomicOr(p.err, 1u);
            row[i] = -1;
          }
#pragma unroll
          for (int g = 0; g < FR; ++g)
            v[i][g] = row[i] >= 0 && fr0 + 32 * g < nfrag ? ld_stream(rows + (size_t)row[i] * H + 32 * g * VEC)
                                                          : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < KB; ++i) {
          if (row[i] >= 0) {
            const float w = wt[k0 + i];
#pragma unroll
            for (int g = 0; g < FR; ++g) {
              float a[8];
              unpack8(v[i][g], a);
#pragma unroll
              for (int e = 0; e < 8; ++e) x[g][e] = __fmaf_rn(a[e], w, x[g][e]);
            }
          }
        }
      }
      cp_async_wait_all();                   // this lane's own shared-row fragments
#pragma unroll
      for (int g = 0; g < FR; ++g) {
        if (fr0 + 32 * g < nfrag) {
          float s[8];
          unpack8(xs[r * CHUNK + 32 * g + lane], s);
#pragma unroll
          for (int e = 0; e < 8; ++e) x[g][e] = __fadd_rn(x[g][e], s[e]);
          round8(x[g]);
        }
        xs[r * CHUNK + 32 * g + lane] = make_uint4(pack_bf16x2(x[g][0], x[g][1]), pack_bf16x2(x[g][2], x[g][3]),
                                                   pack_bf16x2(x[g][4], x[g][5]), pack_bf16x2(x[g][6], x[g][7]));
      }
    }
    __syncthreads();
    // y = bf16(((0 + x_0) + x_1) + ...): warps 0 .. FR - 1 take a fragment each
    if (warp < FR && fr0 + 32 * warp < nfrag) {
      const int fi = 32 * warp + lane;
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = 0.f;
#pragma unroll 1
      for (int r = 0; r < p.tp; ++r) {
        float a[8];
        unpack8(xs[r * CHUNK + fi], a);
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = __fadd_rn(y[e], a[e]);
      }
      st_vec(p.y + (size_t)t * H + (size_t)(fr0 + 32 * warp) * VEC, round8(y));
    }
    __syncthreads();   // the next job's x_r overwrite these
  }
}

}  // namespace

// The rank buffer: tp x CHUNK fragments x 16 bytes.
cudaError_t moe_fold_set_attributes() {
  return cudaFuncSetAttribute(k_moe_fold, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              TP_MAX * CHUNK * int(sizeof(uint4)));
}

cudaError_t launch_moe_fold(const FoldParams &p, int sms, cudaStream_t stream) {
  const int ctas = sms * 3;   // the CTAs resident at once (launch bounds)
  if (p.tp < 1 || p.tp > TP_MAX || p.top_k < 1 || p.top_k > 64 || p.hidden % VEC) return cudaErrorInvalidValue;
  const int jobs = p.m * ((p.hidden / VEC + CHUNK - 1) / CHUNK);
  const int grid = jobs < ctas ? jobs : ctas;
  k_moe_fold<<<grid, NT, size_t(p.tp) * CHUNK * sizeof(uint4), stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mhc
