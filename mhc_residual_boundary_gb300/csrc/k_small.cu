// k_small.cu -- the whole boundary of a few tokens in one kernel.
//
// A cluster of CS CTAs (16, or 8 where 16 do not fit) owns up to B_MAX tokens
// and every CTA of it one contiguous range of the hidden columns (whole
// 32-column blocks when H is a multiple of 32), as the pages lay out their
// boundary kernels ([GLM] _BoundaryDeviceKernel.kernel: one token per CTA
// cluster, the 24-way GEMV summed over the cluster through distributed shared
// memory).  Per CTA, in one pass:
//   1. bulk copies bring the CTA's prenorm weight rows (FP32, [4][cols][24];
//      for a layer weight before the wait for the preceding kernel) and each
//      token's partials, streams, post and comb for its columns;
//   2. stage-1 sum of the tp partials in FP32 in rank order, rounded to BF16
//      ([DSV] _LamportMHCDeviceKernel.kernel, lane_sum), post-mix of the four
//      streams ([GLM] "mixed"), with the operations of the tensor-core stage
//      kernel (so the same bits); residual_out stored, the new streams kept in
//      shared memory;
//   3. the CTA's part of the GEMV and the sum of squares ([GLM] "partial"):
//      FP32 fused multiply-adds of the BF16 streams (exact as FP32) with the
//      FP32 weight, split over threads by (4 outputs, row phase) with every
//      token of the cluster in each thread (the weight is read once), summed
//      back in a fixed shuffle tree;
//   4. every CTA sends its partial sums of each token into every CTA's
//      inbox (remote stores that count their bytes on the receiver's
//      mbarrier), then sums its own inbox in rank order: rstd, mixes and pre
//      ([GLM] "rstd", "pre_mix") -- the same values in every CTA;
//   5. collapse c = bf16((n0 p0 + n1 p1) + (n2 p2 + n3 p3)) of its columns
//      and their sum of c^2, exchanged the same way; inv_rms from the CS sums
//      in rank order; out = bf16((c * inv_rms) * gamma) and the optional MXFP8
//      copy ([GLM] "collapse", "inv_rms"; [DSV] quantize branch);
//   6. token t's post and Sinkhorn mix ([GLM] _MixesDeviceKernel) in four
//      lanes of CTA rank t % CS's last warp (the same operations as the
//      finish kernel's, so the same bits), from right after step 4, while
//      the other warps collapse and normalise.
// The delayed-mHC consumer ([DSV] AllReduceMHC.__call__ with a carried pre)
// runs steps 1, 2, 5 and its exchange only: no weight, GEMV, first exchange
// or mixes, pre copied in with the token's inputs; without a carried pre
// (residual only) it stops after step 2.
// One cluster barrier, after every CTA has armed its inboxes, orders the
// first remote store after the arming; a CTA leaves only once its inboxes
// are complete, so no store reaches a CTA that has left.  Every wait is
// bounded; a CTA whose copies do not arrive skips its work (its outputs are
// invalid), still sends (zeros) to every inbox, and sets bit 1 of the error
// word.
//
// Pages: [GLM] vllm.models.glm5next.nvidia.specialized_decode.all_reduce_mhc,
//        [DSV] vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc.
#include "device_common.cuh"
#include "launch.cuh"
#include "tcgen05.cuh"

namespace mhc {
namespace {

// Test hook (mhc_test_stall_stage_copies): when set, no token data copies are
// issued, so the kernel's bounded wait runs out and it reports the timeout
// through the error word instead of hanging.
__device__ int g_stall_copies = 0;

constexpr int NT = 512;
constexpr int NWARP = NT / 32;
constexpr int SINK_WARP = NWARP - 1;           // post / Sinkhorn, no collapse items
static_assert(SMALL_B_MAX <= 8, "a CTA owns at most one token's post / Sinkhorn (clusters of 8 or 16)");
constexpr int ITEM_THREADS = NT - 32;          // threads of the collapse and normalisation items
constexpr int GEMV_ROWS_WARP = 5;              // weight rows a warp takes at once (30 lanes)
constexpr int GEMV_ROWS_PASS = GEMV_ROWS_WARP * NWARP;   // 80
constexpr uint32_t WAIT_LIMIT = 1u << 22;      // polls before a copy wait gives up
constexpr int SMEM_MAX = 227 * 1024;
constexpr int IN1_STRIDE = 28;                 // floats of a token's partials in an inbox (7 x 16 bytes)

// Shared memory: control block, then the weight rows, then one slot per token.
struct Ctl {
  static constexpr int wbar = 0;               // uint64: weight rows arrived
  static constexpr int dbar = 8;               // uint64: token data arrived
  static constexpr int ibar1 = 16;             // uint64: every CTA's GEMV partials arrived
  static constexpr int ibar2 = 24;             // uint64: every CTA's sums of c^2 arrived
  static constexpr int inbox1 = 32;            // f32 [16 ranks][SMALL_B_MAX][28]: partials + sum of squares (padded)
  static constexpr int inbox2 = inbox1 + 16 * SMALL_B_MAX * IN1_STRIDE * 4;   // f32 [16 ranks][8]: sums of c^2
  static constexpr int red = inbox2 + 16 * 8 * 4;   // f32 [SMALL_B_MAX][25]: GEMV partials + sum of squares
  static constexpr int red2 = red + SMALL_B_MAX * VALUES * 4;   // f32 [SMALL_B_MAX]: sum of c^2
  static constexpr int pre = red2 + SMALL_B_MAX * 4;             // f32 [SMALL_B_MAX][4]
  static constexpr int ir = pre + SMALL_B_MAX * 16;              // f32 [SMALL_B_MAX]
  static constexpr int mix = ir + SMALL_B_MAX * 4;               // f32 [SMALL_B_MAX][24]
  static constexpr int item_ss = mix + SMALL_B_MAX * MIX * 4;    // f32 [SMALL_ITEMS_MAX]
  static constexpr int gred = item_ss + SMALL_ITEMS_MAX * 4;     // f32 [16 warps][SMALL_B_MAX][24]: the warps' GEMV sums
  static constexpr int sb = gred + NWARP * SMALL_B_MAX * MIX * 4;  // f32 [28]: scale[3], base[24]
  static constexpr int smix = sb + 28 * 4;                         // f32 [24]: the post / Sinkhorn token's mixes
  static constexpr int bad = smix + MIX * 4;                       // int: a copy wait gave up
  static constexpr int end = (bad + 4 + 127) / 128 * 128;
};

__host__ __device__ constexpr int weight_bytes(int cols) { return HC * cols * MIX * 4; }
// A token's slot: partials [tp][cols] bf16, streams [4][cols] bf16, post [4]
// and comb [16] f32.
__host__ __device__ constexpr int slot_res(int tp, int cols) { return tp * cols * 2; }
__host__ __device__ constexpr int slot_post(int tp, int cols) { return slot_res(tp, cols) + HC * cols * 2; }
__host__ __device__ constexpr int slot_bytes(int tp, int cols) { return (slot_post(tp, cols) + 80 + 127) / 128 * 128; }

// Column range of cluster rank r (whole units of `unit` columns).
__device__ __forceinline__ void col_range(int hidden, int cs, int r, int &c0, int &c1) {
  const int unit = hidden % 32 == 0 ? 32 : VEC, n = hidden / unit;
  c0 = (r * n / cs) * unit;   // r < 16 and n <= 2048: no overflow
  c1 = ((r + 1) * n / cs) * unit;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster: arrive (release), then wait (acquire).
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_sync() {
  cluster_arrive();
  cluster_wait();
}

// The 15 warps other than the post / Sinkhorn warp.
__device__ __forceinline__ void item_sync() { asm volatile("bar.sync 1, %0;" ::"n"(ITEM_THREADS) : "memory"); }

// Sum over the 32 lanes of a warp in a fixed tree (every lane gets it).
__device__ __forceinline__ float tree_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// This CTA's shared address `p` in cluster CTA `rank`.
__device__ __forceinline__ uint32_t remote_addr(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(tc::smem_addr(p)), "r"(rank));
  return r;
}
// 16 bytes into cluster shared memory, counted in bytes on the receiver's
// mbarrier when they land.
__device__ __forceinline__ void st_async16(uint32_t remote, float4 v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
               ::"r"(remote), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
               : "memory");
}

__device__ __forceinline__ float2 dup(float x) { return make_float2(x, x); }

// Loads from this CTA's shared memory by 32-bit shared-window address: the
// GEMV below is a separate function, so a generic pointer would reach it
// without its address space.
__device__ __forceinline__ float4 lds_f4(uint32_t a) {
  float4 v;
  asm("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds_u2(uint32_t a) {
  uint2 v;
  asm("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  unsigned short h;
  asm("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(a));
  return h;
}

struct GemvArgs {
  const void *w;               // the weight rows [4 * cols][24], FP32 or BF16
  const unsigned char *x;      // token 0's new streams [4][cols] bf16; token t at + t * sbytes
  int sbytes, K;               // K = 4 * cols rows
  float *gred;                 // [16 warps][SMALL_B_MAX][24]: each warp's sums
};

// This CTA's part of the GEMV for B tokens: lane l < 30 of warp w takes
// outputs 4 * (l % 6) .. +3 of rows k = 5 * w + l / 6, + 80, + 160, ... (a warp
// reads 5 whole weight rows of 96 (FP32) or 48 (BF16) bytes, without bank
// conflicts); each warp's five row lanes of an output quad are summed in
// order into gred.  A BF16 weight widens exactly to FP32.
template <int B, bool BF16W>
__device__ __noinline__ void gemv_part(const GemvArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int iq = lane % 6, rr = lane / 6;
  float4 acc[B];
#pragma unroll
  for (int t = 0; t < B; ++t) acc[t] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (lane < 30) {
    const uint32_t w0 = tc::smem_addr(a.w) + uint32_t(iq * 4 * (BF16W ? 2 : 4)), x0 = tc::smem_addr(a.x);
    // two rows' loads ahead of their multiply-adds (each sum keeps its order)
#pragma unroll 2
    for (int k = GEMV_ROWS_WARP * warp + rr; k < a.K; k += GEMV_ROWS_PASS) {
      float4 wv;
      if (BF16W) {
        const uint2 q = lds_u2(w0 + uint32_t(k * MIX * 2));
        wv = make_float4(bf16_lo(q.x), bf16_hi(q.x), bf16_lo(q.y), bf16_hi(q.y));
      } else {
        wv = lds_f4(w0 + uint32_t(k * MIX * 4));
      }
#pragma unroll
      for (int t = 0; t < B; ++t) {
        const float x = __uint_as_float(lds_u16(x0 + uint32_t(t * a.sbytes + k * 2)) << 16);
        acc[t].x = fmaf(wv.x, x, acc[t].x);
        acc[t].y = fmaf(wv.y, x, acc[t].y);
        acc[t].z = fmaf(wv.z, x, acc[t].z);
        acc[t].w = fmaf(wv.w, x, acc[t].w);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < B; ++t) {
    float4 v = acc[t];
#pragma unroll
    for (int r = 1; r < GEMV_ROWS_WARP; ++r) {
      const int src = (lane + 6 * r) & 31;
      v.x = __fadd_rn(v.x, __shfl_sync(0xffffffffu, acc[t].x, src));
      v.y = __fadd_rn(v.y, __shfl_sync(0xffffffffu, acc[t].y, src));
      v.z = __fadd_rn(v.z, __shfl_sync(0xffffffffu, acc[t].z, src));
      v.w = __fadd_rn(v.w, __shfl_sync(0xffffffffu, acc[t].w, src));
    }
    if (lane < 6) *reinterpret_cast<float4 *>(a.gred + ((warp * SMALL_B_MAX) + t) * MIX + lane * 4) = v;
  }
}

// One instantiation a weight form, so that the FP32 kernel carries none of
// the BF16 form's code.
template <bool BF16W>
__global__ void __launch_bounds__(NT, 1) k_small(const SmallParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *wbar = reinterpret_cast<uint64_t *>(smem + Ctl::wbar);
  uint64_t *dbar = reinterpret_cast<uint64_t *>(smem + Ctl::dbar);
  float *red = reinterpret_cast<float *>(smem + Ctl::red);
  float *red2 = reinterpret_cast<float *>(smem + Ctl::red2);
  float *pre_s = reinterpret_cast<float *>(smem + Ctl::pre);
  float *ir_s = reinterpret_cast<float *>(smem + Ctl::ir);
  float *mix_s = reinterpret_cast<float *>(smem + Ctl::mix);
  float *item_ss = reinterpret_cast<float *>(smem + Ctl::item_ss);
  volatile int *bad = reinterpret_cast<volatile int *>(smem + Ctl::bad);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.hidden, tp = p.tp, cs = p.cs;
  const uint32_t rank = cluster_rank();
  const int cluster = int(blockIdx.x) / cs;
  // tokens of this cluster: [t0, t1)
  const int n_clusters = int(gridDim.x) / cs;
  const int t0 = int((long long)cluster * p.m / n_clusters), t1 = int((long long)(cluster + 1) * p.m / n_clusters);
  const int b = t1 - t0;
  int c0, c1;
  col_range(H, cs, int(rank), c0, c1);
  const int cols = c1 - c0, F = cols / VEC;           // 16-byte fragments of a row piece
  unsigned char *w_s = smem + Ctl::end;
  unsigned char *slots = w_s + weight_bytes(p.cols_max);
  const int sbytes = slot_bytes(tp, p.cols_max);

  uint64_t *ibar1 = reinterpret_cast<uint64_t *>(smem + Ctl::ibar1);
  uint64_t *ibar2 = reinterpret_cast<uint64_t *>(smem + Ctl::ibar2);
  float *inbox1 = reinterpret_cast<float *>(smem + Ctl::inbox1);
  float *inbox2 = reinterpret_cast<float *>(smem + Ctl::inbox2);
  const int in2_vecs = (b + 3) / 4;   // 16-byte pieces of a CTA's sums of c^2
  // the delayed-mHC consumer takes no weight, runs no GEMV and computes no
  // mixes (no first exchange); without a carried pre it writes the
  // post-mixed streams only (no collapse, no second exchange)
  const bool gemv = !p.consume, collapse = gemv || p.pre_in != nullptr;
  if (tid == 0) {
    tc::mbar_init(wbar, 1);
    tc::mbar_init(dbar, 1);
    tc::mbar_init(ibar1, 1);
    tc::mbar_init(ibar2, 1);
    *bad = 0;
    tc::mbar_init_fence();
    // the inboxes expect every CTA's pieces
    if (b > 0 && gemv) tc::mbar_arrive_expect_tx(ibar1, uint32_t(cs * b * IN1_STRIDE * 4));
    if (b > 0 && collapse) tc::mbar_arrive_expect_tx(ibar2, uint32_t(cs * in2_vecs * 16));
  }
  // every CTA's inboxes are armed before any CTA sends
  cluster_sync();
  pdl_launch_dependents();

  // the weight rows of this CTA's columns (a layer weight: before the wait).
  // FP32 ([4H][24]): stream j's rows are one run, [4 * cols][24] as copied.
  // BF16 ([GLM] [24][4H]): the 96 row pieces (output i, stream j) are staged
  // [i][j][cols] in the second half of the weight area, then transposed to
  // [4 * cols][24] BF16 in the first half.
  constexpr bool bf16w = BF16W;
  unsigned char *stg = w_s + weight_bytes(p.cols_max) / 2;
  auto load_weight = [&]() {
    if (warp == 0 && cols > 0) {
      if (lane == 0) tc::mbar_arrive_expect_tx(wbar, uint32_t(bf16w ? weight_bytes(cols) / 2 : weight_bytes(cols)));
      __syncwarp();
      if (bf16w) {
        for (int e = lane; e < MIX * HC; e += 32)
          tc::bulk_load(stg + e * cols * 2, p.hc_fn_bf16 + (size_t)(e / HC) * HC * H + (size_t)(e % HC) * H + c0,
                        uint32_t(cols * 2), wbar);
      } else if (lane < HC) {
        tc::bulk_load(w_s + lane * cols * MIX * 4, p.hc_fn + ((size_t)lane * H + c0) * MIX, uint32_t(cols * MIX * 4), wbar);
      }
    }
  };
  auto transpose_weight = [&]() {
    const uint16_t *src = reinterpret_cast<const uint16_t *>(stg);
    for (int k = tid; k < HC * cols; k += NT) {
      const int j = k / cols, c = k % cols;
      uint32_t w[MIX / 2];
#pragma unroll
      for (int i2 = 0; i2 < MIX / 2; ++i2)
        w[i2] = uint32_t(src[((2 * i2) * HC + j) * cols + c]) | (uint32_t(src[((2 * i2 + 1) * HC + j) * cols + c]) << 16);
      uint4 *d = reinterpret_cast<uint4 *>(w_s + k * MIX * 2);
      d[0] = make_uint4(w[0], w[1], w[2], w[3]);
      d[1] = make_uint4(w[4], w[5], w[6], w[7]);
      d[2] = make_uint4(w[8], w[9], w[10], w[11]);
    }
  };
  if (p.early_weight && gemv) {
    load_weight();
    if (bf16w) {
      // staged and transposed while the kernel ahead finishes
      if (cols > 0 && !tc::mbar_wait_bounded(wbar, 0u, WAIT_LIMIT)) *bad = 1;
      __syncthreads();
      if (*bad == 0) transpose_weight();
      __syncthreads();
    }
  }
  pdl_wait();
  if (!p.early_weight && gemv) load_weight();
  // scale and base into shared memory now, beside the token's copies: pre and
  // the post / Sinkhorn warp would otherwise wait on an L2 round trip for them
  float *sb_s = reinterpret_cast<float *>(smem + Ctl::sb);
  float *smix_s = reinterpret_cast<float *>(smem + Ctl::smix);
  if (gemv && warp == 1 && lane < 3 + MIX) sb_s[lane] = lane < 3 ? p.scale[lane] : p.base[lane - 3];
  // the consumer's carried pre of this cluster's tokens (b * 4 <= 32 values)
  if (!gemv && p.pre_in && warp == 1 && lane < b * HC) pre_s[lane] = p.pre_in[(size_t)t0 * HC + lane];
  // each token's partials, streams, post and comb (lanes of warp 0 issue)
  const bool stall = *static_cast<volatile int *>(&g_stall_copies) != 0;
  if (warp == 0 && b > 0 && !stall) {
    const uint32_t per_token = uint32_t((tp + HC) * cols * 2 + 80);
    if (lane == 0) tc::mbar_arrive_expect_tx(dbar, cols > 0 ? per_token * uint32_t(b) : uint32_t(b) * 80u);
    __syncwarp();
    const int per = tp + HC + 2;
    for (int e = lane; e < b * per; e += 32) {
      const int tl = e / per, k = e % per, t = t0 + tl;
      unsigned char *st = slots + tl * sbytes;
      if (k < tp) {
        if (cols > 0) tc::bulk_load(st + k * cols * 2, p.partials + ((size_t)k * p.m + t) * H + c0, uint32_t(cols * 2), dbar);
      } else if (k < tp + HC) {
        const int j = k - tp;
        if (cols > 0)
          tc::bulk_load(st + slot_res(tp, cols) + j * cols * 2, p.residual + ((size_t)t * HC + j) * H + c0,
                        uint32_t(cols * 2), dbar);
      } else if (k == tp + HC) {
        tc::bulk_load(st + slot_post(tp, cols), p.post + (size_t)t * HC, 16u, dbar);
      } else {
        tc::bulk_load(st + slot_post(tp, cols) + 16, p.comb + (size_t)t * HC * HC, 64u, dbar);
      }
    }
  }
  if (b > 0 && !tc::mbar_wait_bounded(dbar, 0u, WAIT_LIMIT)) *bad = 1;
  if (b > 0 && cols > 0 && gemv && !tc::mbar_wait_bounded(wbar, 0u, WAIT_LIMIT)) *bad = 1;
  __syncthreads();
  if (bf16w && !p.early_weight) {
    if (*bad == 0) transpose_weight();
    __syncthreads();
  }
  const bool ok = *bad == 0;

  // ---- 2. stage-1 sum and post-mix: item (token, fragment), four threads an
  // item (a quad of lanes), thread j of the quad computing new stream j; the
  // stage-1 sum is computed by all four (the same bits), thread 0 stores it
  const int n_items = b * F;
  for (int base = warp * 32; base < n_items * HC; base += NT) {
    const int q = base + lane, item = q >> 2, j = q & 3;
    const bool act = ok && item < n_items;
    const int tl = act ? item / F : 0, f = act ? item % F : 0, t = t0 + tl;
    unsigned char *st = slots + tl * sbytes;
    unsigned char *rs = st + slot_res(tp, cols) + f * 16;
    float2 y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = make_float2(0.f, 0.f);
    uint4 res[HC];
    float pj = 0.f;
    float ck[HC];
    if (act) {
      for (int r = 0; r < tp; ++r) {
        const uint4 w = *reinterpret_cast<const uint4 *>(st + r * cols * 2 + f * 16);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          y[e].x = __fadd_rn(y[e].x, bf16_lo(ww[e]));
          y[e].y = __fadd_rn(y[e].y, bf16_hi(ww[e]));
        }
      }
#pragma unroll
      for (int k = 0; k < HC; ++k) res[k] = *reinterpret_cast<const uint4 *>(rs + k * cols * 2);
      const float *pc = reinterpret_cast<const float *>(st + slot_post(tp, cols));
      pj = pc[j];
#pragma unroll
      for (int k = 0; k < HC; ++k) ck[k] = pc[4 + k * HC + j];   // comb[k][j]
    }
    const uint4 yb = make_uint4(pack_bf16x2(y[0].x, y[0].y), pack_bf16x2(y[1].x, y[1].y),
                                pack_bf16x2(y[2].x, y[2].y), pack_bf16x2(y[3].x, y[3].y));
    const uint32_t ybw[4] = {yb.x, yb.y, yb.z, yb.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = bf16_pair(ybw[e]);
    if (act && j == 0 && p.reduced_out) st_vec(p.reduced_out + (size_t)t * H + c0 + f * VEC, yb);
    // new_j = y * post_j + sum_k res_k * comb[k][j], one fused multiply-add a
    // source in source order, on FP32 element pairs
    float2 o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = __fmul2_rn(y[e], dup(pj));
#pragma unroll
    for (int k = 0; k < HC; ++k) {
      const uint32_t ww[4] = {res[k].x, res[k].y, res[k].z, res[k].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = __ffma2_rn(bf16_pair(ww[e]), dup(ck[k]), o[e]);
    }
    const uint4 nv = make_uint4(pack_bf16x2(o[0].x, o[0].y), pack_bf16x2(o[1].x, o[1].y),
                                pack_bf16x2(o[2].x, o[2].y), pack_bf16x2(o[3].x, o[3].y));
    const uint32_t nw[4] = {nv.x, nv.y, nv.z, nv.w};
    float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 r2 = bf16_pair(nw[e]);
      ss2 = __ffma2_rn(r2, r2, ss2);
    }
    // the item's sum of squares over its four streams: ((s0 + s1) + (s2 + s3))
    float s4 = act ? __fadd_rn(ss2.x, ss2.y) : 0.f;
    s4 = __fadd_rn(s4, __shfl_xor_sync(0xffffffffu, s4, 1));
    s4 = __fadd_rn(s4, __shfl_xor_sync(0xffffffffu, s4, 2));
    // every thread of the quad has read the source streams before any of
    // them is replaced: the new stream j takes source stream j's place in the
    // slot (each item owns its 16 bytes of every stream)
    __syncwarp();
    if (act) {
      *reinterpret_cast<uint4 *>(rs + j * cols * 2) = nv;
      st_vec(p.residual_out + ((size_t)t * HC + j) * H + c0 + f * VEC, nv);
      if (j == 0) item_ss[item] = s4;
    }
  }
  __syncthreads();

  // steps 3 and 4 (and the mixes) are the boundary's; the consumer's pre
  // was copied in with its inputs
  if (gemv) {
    // ---- 3. this CTA's part of the GEMV (gemv_part: the loop over the
    // cluster's tokens unrolled for their number)
    float *gred = reinterpret_cast<float *>(smem + Ctl::gred);
    {
      const GemvArgs ga = {w_s, slots + slot_res(tp, cols), sbytes, HC * cols, gred};
      switch (ok ? b : 0) {
        case 1: gemv_part<1, BF16W>(ga); break;
        case 2: gemv_part<2, BF16W>(ga); break;
        case 3: gemv_part<3, BF16W>(ga); break;
        case 4: gemv_part<4, BF16W>(ga); break;
        case 5: gemv_part<5, BF16W>(ga); break;
        case 6: gemv_part<6, BF16W>(ga); break;
        case 7: gemv_part<7, BF16W>(ga); break;
        case 8: gemv_part<8, BF16W>(ga); break;
        default: break;
      }
    }
    // the sum of squares of token `warp`'s new streams, over its fragments in
    // a fixed tree
    if (warp < b) {
      float s = 0.f;
      for (int f = lane; f < F; f += 32) s = __fadd_rn(s, ok ? item_ss[warp * F + f] : 0.f);
      s = tree_sum(s);
      if (lane == 0) red[warp * VALUES + MIX] = s;
    }
    __syncthreads();
    // the 16 warps' sums of output i of token t, in warp order
    if (tid < b * MIX) {
      const int t = tid / MIX, i = tid % MIX;
      float v = 0.f;
  #pragma unroll
      for (int w = 0; w < NWARP; ++w) v = __fadd_rn(v, gred[((w * SMALL_B_MAX) + t) * MIX + i]);
      red[t * VALUES + i] = v;
    }
    __syncthreads();
    // ---- 4. this CTA's partials of every token into every CTA's inbox (slot
    // `rank`): thread (peer, token, 16-byte piece)
    {
      constexpr int PIECES = IN1_STRIDE / 4;
      for (int e = tid; e < cs * b * PIECES; e += NT) {
        const int peer = e / (b * PIECES), rest = e % (b * PIECES), t = rest / PIECES, k = rest % PIECES;
        const float *src = red + t * VALUES + k * 4;
        float4 v;
        v.x = k * 4 + 0 < VALUES ? src[0] : 0.f;
        v.y = k * 4 + 1 < VALUES ? src[1] : 0.f;
        v.z = k * 4 + 2 < VALUES ? src[2] : 0.f;
        v.w = k * 4 + 3 < VALUES ? src[3] : 0.f;
        const float *dst = inbox1 + ((int(rank) * SMALL_B_MAX) + t) * IN1_STRIDE + k * 4;
        st_async16(remote_addr(dst, uint32_t(peer)), v, remote_addr(ibar1, uint32_t(peer)));
      }
    }
    // every CTA's partials, summed in rank order; rstd, mixes, pre
    if (b > 0 && !tc::mbar_wait_bounded(ibar1, 0u, WAIT_LIMIT)) *bad = 1;
    if (warp < b) {
      float v = 0.f;
      // (a compile-time bound, so that the 16 loads issue before the adds)
      if (lane < VALUES) {
  #pragma unroll
        for (int r = 0; r < 16; ++r)
          if (r < cs) v = __fadd_rn(v, inbox1[((r * SMALL_B_MAX) + warp) * IN1_STRIDE + lane]);
      }
      const int t = t0 + warp;
      const float ss = __shfl_sync(0xffffffffu, v, MIX);
      const float rstd = __frcp_rn(sqrtf(__fadd_rn(__fdiv_rn(ss, float(HC * H)), p.rms_eps)));
      const float mix = lane < MIX ? __fmul_rn(v, rstd) : 0.f;
      const bool mine = int(rank) == t % cs;   // this CTA writes the token's mixes, pre, post, comb
      if (lane < MIX) {
        mix_s[warp * MIX + lane] = mix;
        if (mine && p.mixes) p.mixes[(size_t)t * MIX + lane] = mix;
        if (mine && p.mixes_out) p.mixes_out[(size_t)t * MIX + lane] = mix;
      }
      if (lane < HC) {
        const float pr = __fadd_rn(sigmoid(__fadd_rn(__fmul_rn(mix, sb_s[0]), sb_s[3 + lane])), p.hc_eps);
        pre_s[warp * HC + lane] = pr;
        if (mine && p.pre_out) p.pre_out[(size_t)t * HC + lane] = pr;
      }
    } else if (warp == SINK_WARP && p.post_out) {
      // The post / Sinkhorn warp computes the mixes of its token itself (the
      // same operations as above, so the same bits) and starts at once, not
      // after the barrier below: its chain is the longest of the call.  A CTA
      // has at most one such token (b <= 8 <= cs).
      const int first = (int(rank) - t0 % cs + cs) % cs;
      if (first < b) {
        float v = 0.f;
        if (lane < VALUES) {
  #pragma unroll
          for (int r = 0; r < 16; ++r)
            if (r < cs) v = __fadd_rn(v, inbox1[((r * SMALL_B_MAX) + first) * IN1_STRIDE + lane]);
        }
        const float ss = __shfl_sync(0xffffffffu, v, MIX);
        const float rstd = __frcp_rn(sqrtf(__fadd_rn(__fdiv_rn(ss, float(HC * H)), p.rms_eps)));
        if (lane < MIX) smix_s[lane] = __fmul_rn(v, rstd);
      }
      __syncwarp();
    }
  }
  // the collapse needs every token's pre; the post / Sinkhorn warp goes on
  if (warp != SINK_WARP) item_sync();

  // ---- 5. collapse of this CTA's columns (kept in registers for step 7);
  // meanwhile the last warp runs post and the Sinkhorn mix of this CTA's
  // tokens (it has no items and sends nothing more)
  constexpr int IPT = (SMALL_ITEMS_MAX + ITEM_THREADS - 1) / ITEM_THREADS;   // items a thread
  uint32_t cw[IPT][4];
  if (warp == SINK_WARP) {
    cluster_arrive_relaxed();
    if (p.post_out) {
      // the token t of this cluster with t % cs == rank (first < b), on the
      // first quad of lanes; the other quads compute on the same mixes and
      // store nothing
      const int first = (int(rank) - t0 % cs + cs) % cs;   // local index with (t0 + i) % cs == rank
      const MixArgs ma = {sb_s, sb_s + 3, p.post_out, p.comb_out, p.post_mult, p.hc_eps, p.repeat};
      if (first < b) {
        const bool live = ok && lane < 4;
        post_and_sinkhorn4(ma, t0 + first, smix_s, live);
      }
    }
  } else if (!collapse) {
    // the consumer without a carried pre: nothing more to compute or send
    cluster_arrive_relaxed();
  } else {
#pragma unroll
    for (int n = 0; n < IPT; ++n) {
      const int item = tid + n * ITEM_THREADS;
      float s = 0.f;
      if (ok && item < n_items) {
        const int tl = item / F, f = item % F;
        const unsigned char *rs = slots + tl * sbytes + slot_res(tp, cols) + f * 16;
        const float4 pr = *reinterpret_cast<const float4 *>(pre_s + tl * HC);
        const uint4 w0 = *reinterpret_cast<const uint4 *>(rs), w1 = *reinterpret_cast<const uint4 *>(rs + cols * 2);
        const uint4 w2 = *reinterpret_cast<const uint4 *>(rs + 2 * cols * 2);
        const uint4 w3 = *reinterpret_cast<const uint4 *>(rs + 3 * cols * 2);
        const uint32_t n0[4] = {w0.x, w0.y, w0.z, w0.w}, n1[4] = {w1.x, w1.y, w1.z, w1.w};
        const uint32_t n2[4] = {w2.x, w2.y, w2.z, w2.w}, n3[4] = {w3.x, w3.y, w3.z, w3.w};
        float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 a = __fadd2_rn(__fmul2_rn(bf16_pair(n0[e]), dup(pr.x)), __fmul2_rn(bf16_pair(n1[e]), dup(pr.y)));
          const float2 c = __fadd2_rn(__fmul2_rn(bf16_pair(n2[e]), dup(pr.z)), __fmul2_rn(bf16_pair(n3[e]), dup(pr.w)));
          const float2 v = __fadd2_rn(a, c);
          cw[n][e] = pack_bf16x2(v.x, v.y);
          const float2 r2 = bf16_pair(cw[n][e]);
          ss2 = __ffma2_rn(r2, r2, ss2);
        }
        s = __fadd_rn(ss2.x, ss2.y);
      }
      if (item < n_items) item_ss[item] = s;
    }
    item_sync();
    // sum of c^2 of token `warp`, over its fragments in a fixed tree
    if (warp < b) {
      float s = 0.f;
      for (int f = lane; f < F; f += 32) s = __fadd_rn(s, item_ss[warp * F + f]);
      s = tree_sum(s);
      if (lane == 0) red2[warp] = s;
    }
    item_sync();
    // ---- 6. this CTA's sums of c^2 into every CTA's inbox (slot `rank`)
    if (tid < cs * in2_vecs) {
      const int peer = tid / in2_vecs, k = tid % in2_vecs;
      float4 v;
      v.x = k * 4 + 0 < b ? red2[k * 4 + 0] : 0.f;
      v.y = k * 4 + 1 < b ? red2[k * 4 + 1] : 0.f;
      v.z = k * 4 + 2 < b ? red2[k * 4 + 2] : 0.f;
      v.w = k * 4 + 3 < b ? red2[k * 4 + 3] : 0.f;
      st_async16(remote_addr(inbox2 + int(rank) * 8 + k * 4, uint32_t(peer)), v, remote_addr(ibar2, uint32_t(peer)));
    }
    // this CTA sends nothing more
    cluster_arrive_relaxed();
    // the norm-weight fragments, requested before the wait
    uint4 gw[IPT];
#pragma unroll
    for (int n = 0; n < IPT; ++n) {
      const int item = tid + n * ITEM_THREADS;
      gw[n] = ok && item < n_items ? ld_ro(p.gamma + c0 + (item % F) * VEC) : make_uint4(0u, 0u, 0u, 0u);
    }
    // ---- 7. inv_rms of each token (the CS sums in rank order), normalisation
    if (b > 0 && !tc::mbar_wait_bounded(ibar2, 0u, WAIT_LIMIT)) *bad = 1;
    if (warp < b && lane == 0) {
      float s = 0.f;
#pragma unroll
      for (int r = 0; r < 16; ++r)
        if (r < cs) s = __fadd_rn(s, inbox2[r * 8 + warp]);
      ir_s[warp] = __frcp_rn(sqrtf(__fadd_rn(__fdiv_rn(s, float(H)), p.norm_eps)));
    }
    item_sync();
    const int scols = H / 32;
#pragma unroll
    for (int n = 0; n < IPT; ++n) {
      const int item = tid + n * ITEM_THREADS;
      // items of a token are consecutive threads, so that a 32-element
      // block is four consecutive lanes (cols and c0 are multiples of 32
      // with MXFP8)
      const bool live = ok && item < n_items;
      const int tl = live ? item / F : 0, f = live ? item % F : 0, t = t0 + tl, h = c0 + f * VEC;
      const float ir = ir_s[tl];
      const uint32_t gv[4] = {gw[n].x, gw[n].y, gw[n].z, gw[n].w};
      uint32_t ow[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 o = __fmul2_rn(__fmul2_rn(bf16_pair(cw[n][e]), dup(ir)), bf16_pair(gv[e]));
        ow[e] = live ? pack_bf16x2(o.x, o.y) : 0u;
      }
      if (live) st_vec(p.layer_input + (size_t)t * H + h, make_uint4(ow[0], ow[1], ow[2], ow[3]));
      if (p.mx_values) {
        const uint32_t m2 = bf16x2_max(bf16x2_max(ow[0] & 0x7fff7fffu, ow[1] & 0x7fff7fffu),
                                       bf16x2_max(ow[2] & 0x7fff7fffu, ow[3] & 0x7fff7fffu));
        float amax = fmaxf(bf16_lo(m2), bf16_hi(m2));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const uint32_t e8 = ue8m0_ceil(__fmul_rn(amax, 1.0f / 448.0f));
        const float2 inv2 = dup(inv_scale(e8));
        if (live) {
          const float2 q0 = __fmul2_rn(bf16_pair(ow[0]), inv2), q1 = __fmul2_rn(bf16_pair(ow[1]), inv2);
          const float2 q2 = __fmul2_rn(bf16_pair(ow[2]), inv2), q3 = __fmul2_rn(bf16_pair(ow[3]), inv2);
          uint2 q;
          q.x = e4m3x4(q0.x, q0.y, q1.x, q1.y);
          q.y = e4m3x4(q2.x, q2.y, q3.x, q3.y);
          *reinterpret_cast<uint2 *>(p.mx_values + (size_t)t * H + h) = q;
          if ((f & 3) == 0) p.mx_scales[swizzle_128x4(t, h / 32, scols)] = uint8_t(e8);
        }
      }
    }
  }
  // MXFP8 padding rows of the scale layout (cluster 0): scales zeroed
  if (p.mx_scales && cluster == 0) {
    const int padded = (p.m + 127) / 128 * 128, scols = H / 32;
    for (int row = p.m + int(rank); row < padded; row += cs)
      for (int c4 = tid; c4 < scols / 4; c4 += NT)
        *reinterpret_cast<uint32_t *>(p.mx_scales + swizzle_128x4(row, c4 * 4, scols)) = 0u;
  }
  // no CTA leaves before every CTA has issued its remote stores (its own
  // inboxes are complete, so nothing more arrives here)
  cluster_wait();
  if (tid == 0 && *bad != 0 && p.err) atomicOr(p.err, 2u);
}

}  // namespace

cudaError_t small_stall_copies(int on) { return cudaMemcpyToSymbol(g_stall_copies, &on, sizeof on); }

int small_cols_max(int hidden, int cs) {
  const int unit = hidden % 32 == 0 ? 32 : VEC, n = hidden / unit;
  return (n + cs - 1) / cs * unit;
}

size_t small_smem_bytes(int hidden, int tp, int cs, int tokens) {
  const int cols = small_cols_max(hidden, cs);
  return size_t(Ctl::end) + size_t(weight_bytes(cols)) + size_t(tokens) * slot_bytes(tp, cols);
}

// Tokens one cluster can take at this shape (0: the path does not apply).
int small_tokens_max(int hidden, int tp, int cs) {
  const int cols = small_cols_max(hidden, cs), f = cols / VEC;
  int b = SMALL_B_MAX;
  while (b > 0 && (small_smem_bytes(hidden, tp, cs, b) > size_t(SMEM_MAX) || b * f > SMALL_ITEMS_MAX)) --b;
  return b;
}

cudaError_t small_set_attributes() {
  cudaError_t e = cudaSuccess;
  for (auto k : {k_small<false>, k_small<true>}) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  }
  return e;
}

// Clusters of `cs` CTAs that can run at once with `smem` bytes a CTA.
int small_active_clusters(int cs, size_t smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_small<false>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_small(const SmallParams &p, int clusters, cudaStream_t stream) {
  if (p.cs != 8 && p.cs != 16) return cudaErrorInvalidValue;
  const int b_max = small_tokens_max(p.hidden, p.tp, p.cs);
  if (b_max < 1 || clusters < 1 || (p.m + clusters - 1) / clusters > b_max) return cudaErrorInvalidValue;
  // one weight form for the boundary, none for the consumer
  if (p.consume ? (p.hc_fn || p.hc_fn_bf16) : !p.hc_fn == !p.hc_fn_bf16) return cudaErrorInvalidValue;
  if (p.cols_max != small_cols_max(p.hidden, p.cs)) return cudaErrorInvalidValue;
  const int b = (p.m + clusters - 1) / clusters;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(clusters * p.cs);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = small_smem_bytes(p.hidden, p.tp, p.cs, b);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return p.hc_fn_bf16 ? cudaLaunchKernelEx(&cfg, k_small<true>, p) : cudaLaunchKernelEx(&cfg, k_small<false>, p);
}

}  // namespace mhc
