// k_owner_reduce.cu -- single-GPU emulation of the two-shot (BT) reduction
// of the tp partials ([DSV] module text on the BT protocol,
// _OwnerReduceMulticastDeviceKernel.kernel): token t belongs to owner rank
// t % tp, and the owner sums the tp ranks' contributions of its tokens in
// FP32 from rank 0, in rank order, rounded to BF16:
//
//   sums[t] = bf16(((+0 + x_0[t]) + x_1[t]) + ... + x_{tp-1}[t])
//
// -- the same order and precision as the direct stage-1 sum, so the boundary
// that then takes sums as its one partial gives the same bits.  On one GPU
// the publish step (each rank storing its contribution into the owner's
// mailbox) would only copy the partials, so the owners read them where they
// are; the multicast of the sums becomes one [m][H] BF16 buffer.
//
// Layout: CTAs of 128 threads, grid-stride over (owner, owner token,
// 1024-column chunk) jobs, owners first, so that an owner's tokens are
// reduced together; a thread takes one 16-byte fragment and keeps eight
// ranks' fragments in flight.  Every CTA lets the stage kernel's launch
// begin at its start.
//
// Page: [DSV] vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc.
#include "device_common.cuh"
#include "launch.cuh"

namespace mhc {
namespace {

constexpr int NT = 128;
constexpr int RB = 8;                        // ranks loaded per batch

__global__ void __launch_bounds__(NT) k_owner_reduce(const OwnerParams p) {
  const int H = p.hidden, nfrag = H / VEC, chunks = (nfrag + NT - 1) / NT;
  const int per_owner = (p.m + p.tp - 1) / p.tp;     // tokens an owner may hold
  const long long jobs = (long long)p.tp * per_owner * chunks;
  // the stage kernel that follows may place its CTAs beside this grid's and
  // stage its layer weight; it reads the sums only after this grid ends
  pdl_launch_dependents();
  for (long long job = blockIdx.x; job < jobs; job += gridDim.x) {
    const int owner = int(job / ((long long)per_owner * chunks));
    const int rest = int(job % ((long long)per_owner * chunks));
    const int t = owner + p.tp * (rest / chunks);    // the owner's (rest / chunks)-th token
    const int fr = (rest % chunks) * NT + int(threadIdx.x);
    if (t >= p.m || fr >= nfrag) continue;
    const uint16_t *src = p.partials + (size_t)t * H + (size_t)fr * VEC;
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = 0.f;
#pragma unroll 1
    for (int r0 = 0; r0 < p.tp; r0 += RB) {
      uint4 v[RB];
#pragma unroll
      for (int i = 0; i < RB; ++i)
        v[i] = r0 + i < p.tp ? ld_stream(src + (size_t)(r0 + i) * p.m * H) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int i = 0; i < RB; ++i) {
        if (r0 + i < p.tp) {
          float x[8];
          unpack8(v[i], x);
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = __fadd_rn(y[e], x[e]);
        }
      }
    }
    st_vec(p.sums + (size_t)t * H + (size_t)fr * VEC, round8(y));
  }
}

}  // namespace

cudaError_t launch_owner_reduce(const OwnerParams &p, int ctas, cudaStream_t stream) {
  if (p.tp < 1 || p.tp > 32 || p.m < 1 || p.hidden % VEC) return cudaErrorInvalidValue;
  const long long jobs = (long long)p.tp * ((p.m + p.tp - 1) / p.tp) * ((p.hidden / VEC + NT - 1) / NT);
  const int grid = jobs < ctas ? int(jobs) : ctas;
  k_owner_reduce<<<grid, NT, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mhc
