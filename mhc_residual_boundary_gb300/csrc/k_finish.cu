// k_finish.cu -- finish kernel of the mHC boundary.  Per token:
//
//  1. sums the stage kernel's per-group partials in group order (24 GEMV
//     outputs and the sum of squares of the new streams), one value per
//     lane of the mixes warp;
//  2. rstd = 1/sqrt(ss / (4H) + rms_eps), mixes = raw * rstd,
//     pre_j = sigmoid(mixes_j * scale[0] + base[j]) + hc_eps
//     ([GLM] _BoundaryDeviceKernel.kernel, "rstd", "pre_mix");
//  3. collapse c = bf16(sum_j new_j * pre_j), inv_rms = 1/sqrt(sum c^2 / H +
//     norm_eps), out = bf16((c * inv_rms) * gamma) ([GLM] "collapse",
//     "prenorm", "inv_rms"; [DSV] _LamportMHCDeviceKernel.kernel);
//  4. optionally the MXFP8 copy of out: per 32-element block the UE8M0 code of
//     amax * (1/448) rounded up to a power of two, E4M3 values of
//     out * 2^(127 - e) with hardware nearest-even satfinite conversions,
//     scales at the 128x4 swizzled offset, padding-row scales zeroed ([DSV]
//     _LamportMHCDeviceKernel.kernel, quantize branch);
//  With `pre_in` set (the [DSV] delayed-mHC consumer) steps 1-2 and 5 are
//  skipped: the collapse takes the carried pre-mix.
//  5. with `post_out` set, the next boundary's post-mix and Sinkhorn residual
//     mix as well ([GLM] _MixesDeviceKernel.kernel and _sinkhorn): the mixes
//     warp keeps the normalised mixes of up to 32 of the CTA's tokens and
//     runs their Sinkhorn chains one token per lane, while the other seven
//     warps collapse the batch's last token; otherwise the raw mixes go to
//     `mixes` for the side kernel.
//
// Layout on the GPU: persistent CTAs of 256 threads (7 collapse warps and
// the mixes warp), up to four per SM as the shared memory allows, each
// taking tokens blockIdx.x, blockIdx.x + gridDim.x, ...  A token's four new
// streams are one contiguous 8H-byte run of residual_out and its partial
// sums one 16-byte-padded row, so each token arrives in shared memory by two
// bulk copies into a ring of one or two slots, each on its own barrier: the
// mixes warp reduces token k + 1's partial-sum row (and issues the copy of
// the row that takes its place) while the collapse warps work on token k.
// The collapse keeps c in registers (BF16 pairs), so thread 0 refills the
// slot's stream rows as soon as the collapse has read them, and the next
// token's copy is in flight while this one is normalised and stored; the
// collapse and normalisation run on FP32 pairs with each operation rounded
// as written above.  Every wait is bounded; a wait that gives up sets bit 1
// of the error word, and the CTA's stop decision is the barrier's OR of its
// threads' failed waits.
//
// Pages: [GLM] vllm.models.glm5next.nvidia.specialized_decode.all_reduce_mhc,
//        [DSV] vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc.
#include <atomic>

#include "device_common.cuh"
#include "launch.cuh"
#include "tcgen05.cuh"

namespace mhc {
namespace {

constexpr int NT = 256;
constexpr int CWARPS = 7;                      // collapse warps
constexpr int CT = CWARPS * 32;                // collapse threads
constexpr int MIX_WARP = CWARPS;               // the mixes warp
constexpr int MAX_SLOTS = 2;
constexpr int BATCH = 32;                      // tokens per lane-parallel Sinkhorn batch
constexpr size_t SMEM_SM = 216 * 1024;         // ring bytes of all CTAs of an SM (of 228 KB)
constexpr size_t SMEM_LIMIT = 200 * 1024;      // one slot at H = 16384 is 133 KB
constexpr uint32_t WAIT_LIMIT = 1u << 22;      // polls before a wait gives up
static_assert(CT % 4 == 0, "a 32-element MXFP8 block is four consecutive collapse threads");

// Bytes of one ring slot: the token's four stream rows, then its partial-sum row.
__host__ __device__ inline size_t slot_bytes(int hidden, int part_stride) {
  return size_t(HC) * hidden * 2 + size_t(part_stride) * 4;
}
// CTAs per SM (up to 4) and ring slots per CTA.  Up to DEEP_TOKENS tokens an
// SM: as many CTAs as fit with one slot each (more warps, and a CTA's first
// token arrives sooner), then a second slot.  Above it, where each CTA runs a
// long chain of tokens, two slots a CTA first (each CTA has its next token's
// copies in flight during the current one's normalisation): at H = 6144 this
// trades 4 CTAs x 1 slot for 2 x 2, which measured 2 % faster a call at 4096
// tokens on 152 SMs and 1-2 % slower at 512-1024.
constexpr int DEEP_TOKENS = 12;
constexpr int SPREAD_TOKENS = 6;   // see launch_finish
struct Occupancy {
  int ctas, slots;
};
inline Occupancy occupancy(int hidden, int part_stride, bool deep) {
  const size_t slot = slot_bytes(hidden, part_stride);
  int ctas = int(SMEM_SM / (deep ? 2 * slot : slot));
  ctas = ctas < 1 ? 1 : ctas > 4 ? 4 : ctas;
  const int slots = ctas * 2 * slot <= SMEM_SM ? 2 : 1;
  return {ctas, slots};
}

// NF: 16-byte fragments of a row per collapse thread (ceil(H / 8 / 224)).
// The register bound follows the CTAs per SM that the shared memory allows
// at that width (a slot is 8H bytes and more): 4 up to NF = 5, then 3, 2, 1.
template <int NF>
__global__ void __launch_bounds__(NT, NF <= 5 ? 4 : NF <= 7 ? 3 : NF <= 9 ? 2 : 1)
    k_finish(const FinishParams p, int slots) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t sfull[MAX_SLOTS];   // a slot's four stream rows arrived
  __shared__ __align__(8) uint64_t pfull[MAX_SLOTS];   // a slot's partial-sum row arrived
  __shared__ float pre_s[2][HC];                       // pre of token k in pre_s[k & 1]
  __shared__ float red_s[CWARPS];
  __shared__ float mix_s[BATCH][MIX];
  __shared__ int abort_s;   // some wait gave up (reported after the loop)
  bool bad = false;         // one of this thread's waits gave up
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.hidden;
  const int nfrag = H / VEC;
  const size_t sbytes = slot_bytes(H, p.part_stride);
  const uint32_t stream_bytes = uint32_t(HC) * H * 2;
  const uint32_t part_bytes = p.pre_in ? 0u : uint32_t(p.part_stride) * 4;   // no GEMV sums with a carried pre
  // tokens of this CTA: blockIdx.x + k * gridDim.x, k < n_tok
  const int n_tok = (p.m - int(blockIdx.x) + int(gridDim.x) - 1) / int(gridDim.x);

  if (tid == 0) {
    for (int i = 0; i < slots; ++i) {
      tc::mbar_init(&sfull[i], 1);
      tc::mbar_init(&pfull[i], 1);
    }
    abort_s = 0;
    tc::mbar_init_fence();
  }
  __syncthreads();

  // Nothing below may read the stage kernel's outputs before this point.
  pdl_wait();
  // The next kernel on the stream may start its own setup on the SMs this
  // grid leaves free (it waits for this grid before it touches its inputs).
  pdl_launch_dependents();

  const uint64_t read_once = tc::policy_evict_first();   // the new streams are read once more, here
  // Token k of this CTA goes to slot k % slots, on two barriers: its four
  // stream rows (thread 0, once the collapse has read the slot) and its
  // partial-sum row (the mixes warp, once it has reduced the row that the
  // slot held before; a token earlier, so that the copy is hidden).
  auto fill_streams = [&](int k) {
    const int t = int(blockIdx.x) + k * int(gridDim.x);
    tc::mbar_arrive_expect_tx(&sfull[k % slots], stream_bytes);
    tc::bulk_load_hint(smem + size_t(k % slots) * sbytes, p.streams + (size_t)t * HC * H, stream_bytes,
                       &sfull[k % slots], read_once);
  };
  auto fill_part = [&](int k) {
    const int t = int(blockIdx.x) + k * int(gridDim.x);
    tc::mbar_arrive_expect_tx(&pfull[k % slots], part_bytes);
    tc::bulk_load(smem + size_t(k % slots) * sbytes + stream_bytes, p.part + (size_t)t * p.part_stride, part_bytes,
                  &pfull[k % slots]);
  };
  // partial-sum rows (mixes warp): copies issued for tokens < pissued, rows
  // reduced for tokens < preduced
  int pissued = part_bytes ? (slots < n_tok ? slots : n_tok) : 0, preduced = 0;
  // the pre-mix's scale and base, read once (not after every token's
  // reduction, where the load would add a round trip to the chain)
  const float pre_scale = warp == MIX_WARP && !p.pre_in ? p.scale[0] : 0.f;
  const float pre_base = warp == MIX_WARP && !p.pre_in && lane < HC ? p.base[lane] : 0.f;
  // mixes warp: steps 1-2 for token k of this CTA (its pre into pre_s[k & 1])
  auto token_pre = [&](int k) {
    const int t = int(blockIdx.x) + k * int(gridDim.x);
    if (p.pre_in) {
      // the delayed-mHC consumer: the collapse takes the carried pre-mix
      if (lane < HC) pre_s[k & 1][lane] = p.pre_in[(size_t)t * HC + lane];
      return;
    }
    if (!tc::mbar_wait_bounded(&pfull[k % slots], uint32_t(k / slots) & 1u, WAIT_LIMIT)) bad = true;
    const float *part_s = reinterpret_cast<const float *>(smem + size_t(k % slots) * sbytes + stream_bytes);
    // each of lanes 0-24 sums one value over the groups, in group order
    float v = 0.f;
    if (lane < VALUES) {
#pragma unroll 8
      for (int g = 0; g < p.slices; ++g) v = __fadd_rn(v, part_s[g * VALUES + lane]);
    }
    // the row's next fill is an async-proxy write after these generic reads
    tc::fence_proxy_async_smem();
    __syncwarp();
    preduced = k + 1;
    if (k + slots < n_tok) {
      if (lane == 0) fill_part(k + slots);
      pissued = k + slots + 1;
    }
    const float ss = __shfl_sync(0xffffffffu, v, MIX);
    const float rstd = __frcp_rn(sqrtf(__fadd_rn(__fdiv_rn(ss, float(HC * H)), p.rms_eps)));
    if (lane < MIX) {
      const float mix = __fmul_rn(v, rstd);
      mix_s[k % BATCH][lane] = mix;
      if (p.mixes) p.mixes[(size_t)t * MIX + lane] = mix;
      if (p.mixes_out) p.mixes_out[(size_t)t * MIX + lane] = mix;
      if (lane < HC) {
        const float pre = __fadd_rn(sigmoid(__fadd_rn(__fmul_rn(mix, pre_scale), pre_base)), p.hc_eps);
        pre_s[k & 1][lane] = pre;
        if (p.pre_out) p.pre_out[(size_t)t * HC + lane] = pre;
      }
    }
  };

  int filled = 0;   // tokens whose stream copies were issued (thread 0)
  if (tid == 0)
    for (; filled < slots && filled < n_tok; ++filled) {
      if (part_bytes) fill_part(filled);
      fill_streams(filled);
    }
  if (warp == MIX_WARP && n_tok > 0) token_pre(0);

  const int cols = H / 32;
  for (int k = 0; k < n_tok; ++k) {
    const int t = int(blockIdx.x) + k * int(gridDim.x);
    unsigned char *slot = smem + size_t(k % slots) * sbytes;
    // pre of token k is ready; token k - 1 is done with its slot and pre_s
    // entry.  Every thread takes the same decision: the barrier's own OR of
    // the threads' failed waits.
    if (__syncthreads_or(bad)) break;

    if (warp == MIX_WARP) {
      // (fused) post + Sinkhorn per batch of tokens, one token per lane; it
      // runs before token k + 1's mixes overwrite the batch's first entry
      const int b = k % BATCH;
      if (p.post_out && !p.pre_in && (b == BATCH - 1 || k == n_tok - 1)) {
        const MixArgs ma = {p.scale, p.base, p.post_out, p.comb_out, p.post_mult, p.hc_eps, p.repeat};
        if (b < 8) {
          // a batch of at most 8 tokens (a CTA's last, or all it has at
          // small M, where the chain sits on the CTA's critical path): four
          // lanes a token, a shorter chain with the same bits
          const int i = lane >> 2;
          post_and_sinkhorn4(ma, int(blockIdx.x) + (k - b + (i <= b ? i : 0)) * int(gridDim.x),
                             mix_s[i <= b ? i : 0], i <= b);
        } else if (lane <= b) {
          post_and_sinkhorn(ma, int(blockIdx.x) + (k - b + lane) * int(gridDim.x), mix_s[lane]);
        }
        __syncwarp();
      }
      // steps 1-2 of the next token, beside this token's collapse (its
      // partial-sum row was issued with its streams, at the last refill)
      if (k + 1 < n_tok) token_pre(k + 1);
    } else {
      // 3. collapse, kept in registers as BF16; sum of squares of c
      if (!tc::mbar_wait_bounded(&sfull[k % slots], uint32_t(k / slots) & 1u, WAIT_LIMIT)) bad = true;
      // on element pairs (FP32x2): c = (n0 * pre0 + n1 * pre1) + (n2 * pre2 +
      // n3 * pre3), each product and sum rounded on its own
      float2 pre2[HC];
#pragma unroll
      for (int j = 0; j < HC; ++j) pre2[j] = make_float2(pre_s[k & 1][j], pre_s[k & 1][j]);
      const uint16_t *sv = reinterpret_cast<const uint16_t *>(slot);
      uint4 cfr[NF];
      float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < NF; ++i) {
        const int fr = tid + i * CT;
        cfr[i] = make_uint4(0u, 0u, 0u, 0u);
        if (fr < nfrag) {
          const uint16_t *s = sv + (size_t)fr * VEC;
          const uint4 w0 = *reinterpret_cast<const uint4 *>(s), w1 = *reinterpret_cast<const uint4 *>(s + H);
          const uint4 w2 = *reinterpret_cast<const uint4 *>(s + 2 * H), w3 = *reinterpret_cast<const uint4 *>(s + 3 * H);
          const uint32_t n0[4] = {w0.x, w0.y, w0.z, w0.w}, n1[4] = {w1.x, w1.y, w1.z, w1.w};
          const uint32_t n2[4] = {w2.x, w2.y, w2.z, w2.w}, n3[4] = {w3.x, w3.y, w3.z, w3.w};
          uint32_t c[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 a = __fadd2_rn(__fmul2_rn(bf16_pair(n0[e]), pre2[0]), __fmul2_rn(bf16_pair(n1[e]), pre2[1]));
            const float2 b = __fadd2_rn(__fmul2_rn(bf16_pair(n2[e]), pre2[2]), __fmul2_rn(bf16_pair(n3[e]), pre2[3]));
            const float2 v = __fadd2_rn(a, b);
            c[e] = pack_bf16x2(v.x, v.y);
            const float2 r = bf16_pair(c[e]);   // the rounded value, as stored
            ss2 = __ffma2_rn(r, r, ss2);
          }
          cfr[i] = make_uint4(c[0], c[1], c[2], c[3]);
        }
      }
      float ssq = __fadd_rn(ss2.x, ss2.y);
      // the norm weight's fragments, all requested before any store of this
      // token, so that they cost one round trip, overlapping the reduction
      uint4 gw[NF];
#pragma unroll
      for (int i = 0; i < NF; ++i)
        gw[i] = tid + i * CT < nfrag ? ld_ro(p.gamma + (size_t)(tid + i * CT) * VEC) : make_uint4(0u, 0u, 0u, 0u);
      ssq = warp_sum(ssq);
      if (lane == 0) red_s[warp] = ssq;
      // the slot's next fill is an async-proxy write after these generic reads
      tc::fence_proxy_async_smem();
      asm volatile("bar.sync 1, %0;" ::"n"(CT) : "memory");
      // the slot's stream rows have been read: they take the token `slots`
      // places further on, whose copy then overlaps this token's normalisation
      if (tid == 0 && filled < n_tok) fill_streams(filled++);
      float sq = 0.f;
#pragma unroll
      for (int w = 0; w < CWARPS; ++w) sq += red_s[w];
      const float ir = __frcp_rn(sqrtf(__fadd_rn(__fdiv_rn(sq, float(H)), p.norm_eps)));

      // 4. normalise (pairs: (c * inv_rms) * gamma), store, optional MXFP8
      // (4 consecutive lanes = one 32-element block)
      const float2 ir2 = make_float2(ir, ir);
#pragma unroll
      for (int i = 0; i < NF; ++i) {
        const int fr = tid + i * CT;
        const bool live = fr < nfrag;
        const uint32_t cw[4] = {cfr[i].x, cfr[i].y, cfr[i].z, cfr[i].w};
        const uint32_t gv[4] = {gw[i].x, gw[i].y, gw[i].z, gw[i].w};
        uint32_t ow[4] = {0u, 0u, 0u, 0u};   // the output as stored (BF16 pairs); 0 for no fragment
        if (live) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 o = __fmul2_rn(__fmul2_rn(bf16_pair(cw[e]), ir2), bf16_pair(gv[e]));
            ow[e] = pack_bf16x2(o.x, o.y);
          }
          st_vec(p.layer_input + (size_t)t * H + (size_t)fr * VEC, make_uint4(ow[0], ow[1], ow[2], ow[3]));
        }
        if (p.mx_values) {
          // the block's largest magnitude, on the stored BF16 pairs
          const uint32_t m2 = bf16x2_max(bf16x2_max(ow[0] & 0x7fff7fffu, ow[1] & 0x7fff7fffu),
                                         bf16x2_max(ow[2] & 0x7fff7fffu, ow[3] & 0x7fff7fffu));
          float amax = fmaxf(bf16_lo(m2), bf16_hi(m2));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
          const uint32_t e8 = ue8m0_ceil(__fmul_rn(amax, 1.0f / 448.0f));
          const float2 inv2 = make_float2(inv_scale(e8), inv_scale(e8));
          if (live) {
            const float2 q0 = __fmul2_rn(bf16_pair(ow[0]), inv2), q1 = __fmul2_rn(bf16_pair(ow[1]), inv2);
            const float2 q2 = __fmul2_rn(bf16_pair(ow[2]), inv2), q3 = __fmul2_rn(bf16_pair(ow[3]), inv2);
            uint2 q;
            q.x = e4m3x4(q0.x, q0.y, q1.x, q1.y);
            q.y = e4m3x4(q2.x, q2.y, q3.x, q3.y);
            *reinterpret_cast<uint2 *>(p.mx_values + (size_t)t * H + (size_t)fr * VEC) = q;
            if ((fr & 3) == 0) p.mx_scales[swizzle_128x4(t, fr / 4, cols)] = uint8_t(e8);
          }
        }
      }
    }
  }
  if (bad) abort_s = 1;
  __syncthreads();

  // padding rows of the scale layout: zero their scales (4 columns a store)
  if (p.mx_scales) {
    const int padded = (p.m + 127) / 128 * 128;
    for (int row = p.m + int(blockIdx.x); row < padded; row += int(gridDim.x))
      for (int c4 = tid; c4 < cols / 4; c4 += NT)
        *reinterpret_cast<uint32_t *>(p.mx_scales + swizzle_128x4(row, c4 * 4, cols)) = 0u;
  }
  if (tid == 0) {
    if (abort_s && p.err) atomicOr(p.err, 2u);
    // stream copies still in flight land before the CTA may exit
    for (int k = filled - slots; k < filled; ++k) {
      if (k < 0) continue;
      tc::mbar_wait_bounded(&sfull[k % slots], uint32_t(k / slots) & 1u, WAIT_LIMIT);
    }
  }
  if (warp == MIX_WARP && lane == 0) {
    // partial-sum rows copied but not reduced (only after a failed wait)
    for (int k = preduced; k < pissued; ++k)
      tc::mbar_wait_bounded(&pfull[k % slots], uint32_t(k / slots) & 1u, WAIT_LIMIT);
  }
}

}  // namespace

constexpr int NFMAX = (MAX_HIDDEN / VEC + CT - 1) / CT;
static_assert(NFMAX == 10, "launch_finish dispatches NF = 1 .. 10");
using FinishKernel = void (*)(FinishParams, int);
constexpr FinishKernel kFinish[NFMAX] = {k_finish<1>, k_finish<2>, k_finish<3>, k_finish<4>, k_finish<5>,
                                         k_finish<6>, k_finish<7>, k_finish<8>, k_finish<9>, k_finish<10>};

cudaError_t finish_set_attributes() {
  for (FinishKernel k : kFinish) {
    const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(SMEM_LIMIT));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_finish(const FinishParams &p, int ctas, cudaStream_t stream, bool pdl, int stage_grid) {
  if (p.hidden % VEC || p.hidden > MAX_HIDDEN || p.part_stride % 4 || p.part_stride < p.slices * VALUES)
    return cudaErrorInvalidValue;
  const bool deep = p.m >= DEEP_TOKENS * ctas;
  Occupancy occ = occupancy(p.hidden, p.part_stride, deep);
  // Spread: at most two CTAs an SM (two slots each when they fit), when up to
  // SPREAD_TOKENS tokens an SM, packed CTAs would leave fewer SMs free than
  // the stage kernel of the next call needs.  A stage CTA takes a whole SM,
  // so its CTAs wait for this kernel's CTAs to leave; packed four an SM, the
  // ones that found no free SM start several us late and end late, while
  // two an SM delay every stage CTA about alike.  Two an SM also share an
  // SM's issue slots among fewer post / Sinkhorn chains.  Same box, CUDA
  // graph of back-to-back calls, us a call (packed -> spread): H = 6144 tp = 4
  // at M = 96 15.9 -> 14.3, M = 256 22.0 -> 19.9, M = 512 31.3 -> 30.4,
  // M = 768 40.8 -> 38.2; H = 5120 tp = 8 at M = 256 21.5 -> 20.1; and where
  // the stage grid fits beside the packed CTAs (H = 5120 tp = 8, M = 128:
  // 120 CTAs, 120 free SMs) packing stays ahead, 15.7 against 17.1.
  const size_t slot = slot_bytes(p.hidden, p.part_stride);
  size_t smem = size_t(occ.slots) * slot;
  if (!deep && stage_grid > 0 && occ.ctas > 2 && p.m <= SPREAD_TOKENS * ctas &&
      ctas - (p.m + occ.ctas - 1) / occ.ctas < stage_grid) {
    occ.ctas = 2;
    occ.slots = 2 * slot <= SMEM_SM / 2 ? 2 : 1;
    // a third CTA must not fit beside two
    smem = SMEM_SM / 2 > size_t(occ.slots) * slot ? SMEM_SM / 2 : size_t(occ.slots) * slot;
  }
  const int slots = occ.slots;
  if (smem > SMEM_LIMIT) return cudaErrorInvalidValue;
  const int nf = (p.hidden / VEC + CT - 1) / CT;
  // persistent: as many CTAs as are resident at once (the runtime's count, so
  // that the static shared memory and the per-CTA reservation are included)
  // (cached per kernel and ring size: the query costs host time on every call)
  static std::atomic<uint64_t> cache[NFMAX][MAX_SLOTS];
  std::atomic<uint64_t> &entry = cache[nf - 1][slots - 1];
  const uint64_t cached = entry.load(std::memory_order_relaxed);
  int resident = 0;
  if (cached && (cached >> 8) == smem) {
    resident = int(cached & 0xff);
  } else {
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, kFinish[nf - 1], NT, smem);
    if (e != cudaSuccess) return e;
    entry.store((uint64_t(smem) << 8) | uint64_t(resident & 0xff), std::memory_order_relaxed);
  }
  resident = resident < 1 ? 1 : resident > occ.ctas ? occ.ctas : resident;
  const int grid = ctas * resident;
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
