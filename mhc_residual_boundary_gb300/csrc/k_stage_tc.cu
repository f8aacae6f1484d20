// k_stage_tc.cu -- stage kernel with the prenorm GEMV on tcgen05 tensor cores.
//
// Work unit: 128 tokens x one 64-column hidden slice.  Units are numbered
// slice-major and every CTA (one per SM, persistent) takes a contiguous range
// of them, so a CTA stages each hc_fn slice it meets once.
//
//   phase A (CUDA cores, thread = token x 16-byte fragment, loads prefetched
//     one item ahead in registers): stage-1 sum of the tp BF16 partials in
//     FP32 in rank order, rounded to BF16 ([DSV] _LamportMHCDeviceKernel
//     .kernel, lane_sum); post-mix of the four residual streams ([GLM]
//     _BoundaryDeviceKernel.kernel, "mixed"), stored to residual_out and, as
//     the MMA's A operand, to shared memory; the slice's sum of squares.
//   GEMV (tensor cores): D[token][output] = sum_k new[token][k] * fn[k][output]
//     over the slice's 256 inputs ([GLM] _BoundaryDeviceKernel.kernel,
//     "partial").  hc_fn is FP32; it is split exactly enough into three BF16
//     terms (hi + mid + lo, the remainder below 2^-24 relative) so that each
//     BF16 x BF16 product is exact and the sum accumulates in FP32 in tensor
//     memory: 3 x 16 MMAs of M=128, N=32 (24 outputs used), K=16 per unit.
//   epilogue: the 24 sums of each token (tcgen05.ld) and its sum of squares
//     go to the partial-sum scratch the finish kernel reduces.
// Two A buffers and two TMEM accumulators let the tensor core work on one
// unit while the threads load and mix the next.
//
// Pages: [GLM] vllm.models.glm5next.nvidia.specialized_decode.all_reduce_mhc,
//        [DSV] vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc.
#include "device_common.cuh"
#include "launch.cuh"
#include "tcgen05.cuh"

namespace mhc {
namespace {

constexpr int NT = 256;                       // threads
constexpr int UT = 128;                       // tokens per unit (MMA M)
constexpr int UN = 32;                        // MMA N: 24 outputs + 8 zero rows
constexpr int UK = HC * SLICE;                // 256 GEMV inputs per unit
constexpr int KCOLS = UK / 8;                 // core-matrix columns of 8 BF16
constexpr int A_KCOL = UT * 16 + 16;          // bytes between A core columns (+16: no bank conflicts)
constexpr int A_BYTES = KCOLS * A_KCOL;       // one A buffer
constexpr int B_KCOL = UN * 16;               // bytes between B core columns
constexpr int B_BYTES = 3 * KCOLS * B_KCOL;   // hi, mid, lo
constexpr int ITEMS = UT * (SLICE / VEC) / NT;  // (token, fragment) items per thread per unit
constexpr int TPF = 8;                        // ranks whose loads are prefetched
constexpr uint32_t TMEM_COLS = 64;            // two 32-column accumulators
constexpr uint32_t WAIT_LIMIT = 1u << 22;     // mbarrier polls before giving up

struct Layout {
  static constexpr size_t a0 = 0;
  static constexpr size_t a1 = A_BYTES;
  static constexpr size_t b = 2 * size_t(A_BYTES);
  static constexpr size_t ss = b + B_BYTES;                 // float [2][UT]
  static constexpr size_t bar = ss + 2 * UT * 4;            // uint64 [2]
  static constexpr size_t slot = bar + 16;                  // TMEM address
  static constexpr size_t total = slot + 16;
  static_assert(a1 % 16 == 0 && b % 16 == 0 && bar % 8 == 0, "alignment");
};

struct Item {
  uint4 x[TPF];
  uint4 res[HC];
  float post[HC];
  float comb[HC * HC];   // [source][target]
};

__device__ __forceinline__ void load_item(const StageParams &p, int t, int h, bool act, Item &it) {
  if (!act) return;
#pragma unroll
  for (int q = 0; q < TPF; ++q)
    if (q < p.tp) it.x[q] = ld_stream(p.partials + ((size_t)q * p.m + t) * p.hidden + h);
#pragma unroll
  for (int k = 0; k < HC; ++k) it.res[k] = ld_stream(p.residual + ((size_t)t * HC + k) * p.hidden + h);
  // post / comb are only 4-byte aligned by contract: scalar loads
#pragma unroll
  for (int j = 0; j < HC; ++j) it.post[j] = __ldg(p.post + (size_t)t * HC + j);
#pragma unroll
  for (int c = 0; c < HC * HC; ++c) it.comb[c] = __ldg(p.comb + (size_t)t * HC * HC + c);
}

// Stage 1 and post-mix of one item; returns the new streams as BF16 fragments
// and adds their squares to ss.
__device__ __forceinline__ void mix_item(const StageParams &p, int t, int h, const Item &it, uint4 (&nv)[HC],
                                         float &ss) {
  float y[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) y[e] = 0.f;
#pragma unroll
  for (int q = 0; q < TPF; ++q) {
    if (q < p.tp) {
      float x[8];
      unpack8(it.x[q], x);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = __fadd_rn(y[e], x[e]);
    }
  }
  for (int q = TPF; q < p.tp; ++q) {  // ranks beyond the prefetched ones
    float x[8];
    unpack8(ld_stream(p.partials + ((size_t)q * p.m + t) * p.hidden + h), x);
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = __fadd_rn(y[e], x[e]);
  }
  const uint4 yb = round8(y);
  if (p.reduced_out) st_vec(p.reduced_out + (size_t)t * p.hidden + h, yb);
  float res[HC][8];
#pragma unroll
  for (int k = 0; k < HC; ++k) unpack8(it.res[k], res[k]);
#pragma unroll
  for (int j = 0; j < HC; ++j) {
    float o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float v = __fmul_rn(y[e], it.post[j]);
#pragma unroll
      for (int k = 0; k < HC; ++k) v = __fmaf_rn(res[k][e], it.comb[k * HC + j], v);
      o[e] = v;
    }
    nv[j] = round8(o);
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(o[e], o[e], ss);
    st_vec(p.residual_out + ((size_t)t * HC + j) * p.hidden + h, nv[j]);
  }
}

// The slice's hc_fn as three BF16 B operands (hi, mid, lo), K-major core
// matrices: [term][core column][8-output group][8 outputs][8 inputs].
__device__ void build_b(const StageParams &p, int h0, unsigned char *b_s) {
  for (int e = threadIdx.x; e < (UK / 2) * MIX; e += NT) {
    const int kp = e / MIX, i = e % MIX;
    const int k = 2 * kp, j = k / SLICE, col = k % SLICE, h = h0 + col;
    const float *src = p.hc_fn + ((size_t)j * p.hidden + h) * MIX + i;
    const float x0 = h < p.hidden ? __ldg(src) : 0.f;
    const float x1 = h + 1 < p.hidden ? __ldg(src + MIX) : 0.f;
    const uint32_t hi = pack_bf16x2(x0, x1);
    const float r0 = __fsub_rn(x0, bf16_lo(hi)), r1 = __fsub_rn(x1, bf16_hi(hi));
    const uint32_t mid = pack_bf16x2(r0, r1);
    const uint32_t lo = pack_bf16x2(__fsub_rn(r0, bf16_lo(mid)), __fsub_rn(r1, bf16_hi(mid)));
    const size_t inner = size_t(i / 8) * 128 + (i % 8) * 16 + (k % 8) * 2;
    *reinterpret_cast<uint32_t *>(b_s + size_t(0 * KCOLS + k / 8) * B_KCOL + inner) = hi;
    *reinterpret_cast<uint32_t *>(b_s + size_t(1 * KCOLS + k / 8) * B_KCOL + inner) = mid;
    *reinterpret_cast<uint32_t *>(b_s + size_t(2 * KCOLS + k / 8) * B_KCOL + inner) = lo;
  }
}

__global__ void __launch_bounds__(NT, 1) k_stage_tc(const StageParams p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *b_s = smem + Layout::b;
  float *ss_s = reinterpret_cast<float *>(smem + Layout::ss);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + Layout::bar);
  uint32_t *slot = reinterpret_cast<uint32_t *>(smem + Layout::slot);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.slices;
  const int n_tiles = (p.m + UT - 1) / UT;
  const int units = n_tiles * S;
  const int u_begin = int((long long)blockIdx.x * units / gridDim.x);
  const int u_end = int((long long)(blockIdx.x + 1) * units / gridDim.x);

  if (tid == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    tc::mbar_init_fence();
  }
  if (warp == 0) tc::tmem_alloc(slot, TMEM_COLS);
  for (int i = tid; i < B_BYTES / 16; i += NT) reinterpret_cast<uint4 *>(b_s)[i] = make_uint4(0u, 0u, 0u, 0u);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *slot;
  const uint32_t idesc = tc::idesc_bf16_f32(UT, UN);

  bool ok = true;
  // Reads unit i's accumulator once its MMAs are done and writes the partial
  // sums of its tokens; warps 0-3 take outputs 0-15, warps 4-7 outputs 16-23
  // and the sum of squares.
  auto epilogue = [&](int i) {
    const int u = u_begin + i, s = u / n_tiles, tile = u % n_tiles, stage = i & 1;
    if (ok && !tc::mbar_wait_bounded(&bar[stage], (i >> 1) & 1, WAIT_LIMIT)) ok = false;
    tc::fence_after_sync();
    const int tl = 32 * (warp & 3) + lane, t = tile * UT + tl, c0 = (warp >> 2) * 16;
    float v[16];
    tc::tmem_ld16(tmem + (uint32_t(32 * (warp & 3)) << 16) + uint32_t(stage * UN + c0), v);
    if (ok && t < p.m) {
      float *dst = p.part + ((size_t)t * S + s) * VALUES;
#pragma unroll
      for (int c = 0; c < 16; ++c)
        if (c0 + c < MIX) dst[c0 + c] = v[c];
      if (warp >= 4) dst[MIX] = ss_s[stage * UT + tl];
    }
    tc::fence_before_sync();
  };

  int cur_slice = -1, pending = -1;
  for (int i = 0; u_begin + i < u_end; ++i) {
    const int u = u_begin + i, s = u / n_tiles, tile = u % n_tiles, stage = i & 1;
    if (s != cur_slice) {
      // B is about to change: the previous unit's MMAs must be done with it
      if (pending >= 0) epilogue(pending);
      pending = -1;
      __syncthreads();
      build_b(p, s * SLICE, b_s);
      tc::fence_proxy_async_smem();
      __syncthreads();
      cur_slice = s;
    }

    // phase A: items r = 0..ITEMS-1, token tl = tid/8 + 32r, fragment tid%8;
    // the loads of item r+1 are issued before item r is mixed
    const int f = tid & 7, h = s * SLICE + f * VEC;
    unsigned char *a = smem + (stage ? Layout::a1 : Layout::a0);
    Item cur, nxt;
    {
      const int t = tile * UT + (tid >> 3);
      load_item(p, t, h, t < p.m && h < p.hidden, cur);
    }
#pragma unroll
    for (int r = 0; r < ITEMS; ++r) {
      const int tl = (tid >> 3) + 32 * r, t = tile * UT + tl;
      const bool act = t < p.m && h < p.hidden;
      if (r + 1 < ITEMS) {
        const int tn = t + 32;
        load_item(p, tn, h, tn < p.m && h < p.hidden, nxt);
      }
      uint4 nv[HC] = {};
      float ssi = 0.f;
      if (act) mix_item(p, t, h, cur, nv, ssi);
#pragma unroll
      for (int j = 0; j < HC; ++j)
        *reinterpret_cast<uint4 *>(a + size_t(j * (SLICE / VEC) + f) * A_KCOL + (tl / 8) * 128 + (tl % 8) * 16) = nv[j];
      ssi += __shfl_xor_sync(0xffffffffu, ssi, 1);
      ssi += __shfl_xor_sync(0xffffffffu, ssi, 2);
      ssi += __shfl_xor_sync(0xffffffffu, ssi, 4);
      if (f == 0) ss_s[stage * UT + tl] = ssi;
      if (r + 1 < ITEMS) cur = nxt;
    }

    // hand the A buffer to the tensor core
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0 && ok) {
      tc::fence_after_sync();
      const uint32_t a_addr = tc::smem_addr(a), b_addr = tc::smem_addr(b_s);
#pragma unroll 1
      for (int term = 0; term < 3; ++term) {
#pragma unroll
        for (int ks = 0; ks < UK / 16; ++ks) {
          const uint64_t ad = tc::smem_desc(a_addr + uint32_t(2 * ks * A_KCOL), A_KCOL, 128);
          const uint64_t bd = tc::smem_desc(b_addr + uint32_t((term * KCOLS + 2 * ks) * B_KCOL), B_KCOL, 128);
          tc::mma_bf16(tmem + uint32_t(stage * UN), ad, bd, idesc, (term | ks) != 0);
        }
      }
      tc::mma_commit(&bar[stage]);
    }
    if (pending >= 0) epilogue(pending);
    pending = i;
    // a wait that gave up anywhere ends the loop everywhere
    if (__syncthreads_or(!ok)) {
      ok = false;
      break;
    }
  }
  if (pending >= 0) epilogue(pending);
  if (!ok) {
    // a barrier wait gave up: report it and give the MMAs still in flight
    // one more bounded wait before their tensor memory is released
    if (tid == 0) {
      if (p.err) atomicOr(p.err, 2u);
      if (pending >= 0) tc::mbar_wait_bounded(&bar[pending & 1], (pending >> 1) & 1, WAIT_LIMIT);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

size_t stage_tc_smem_bytes() { return Layout::total; }

cudaError_t stage_tc_set_attributes() {
  return cudaFuncSetAttribute(k_stage_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Layout::total));
}

cudaError_t launch_stage_tc(const StageParams &p, int ctas, cudaStream_t stream) {
  const int units = ((p.m + UT - 1) / UT) * p.slices;
  const int grid = units < ctas ? units : ctas;
  k_stage_tc<<<grid, NT, Layout::total, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mhc
