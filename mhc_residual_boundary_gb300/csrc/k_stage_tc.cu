// k_stage_tc.cu -- stage kernel: TMA-fed load pipeline, post-mix on CUDA
// cores, prenorm GEMV on tcgen05 tensor cores.
//
// Work unit: 32 tokens x one group of 128 hidden columns, so that every row
// piece a unit reads is a 256-byte run (HBM serves these about 10% faster
// than 128-byte pieces of rows 12 KB apart).  Units are numbered group-major
// and every CTA (one per SM, persistent) takes a contiguous range of them, so
// a CTA stages each group's hc_fn once.  Per CTA (8 warps):
//
//   loads: stage q (tokens 8q .. 8q+7) of every unit goes to ring slot q by
//     four TMA tensor copies -- the partials [tp][m][H] (one 3-D box: 128
//     columns x 8 tokens x tp ranks), the residual streams [m][4][H], post
//     [m][4] and comb [m][4][4] -- tracked by the slot's mbarrier transaction
//     count.  Out-of-range tokens and columns arrive as zeros.  Lane 0 of
//     warp q issues them: the next unit's copies as soon as warps q and q + 4
//     have moved the current stage to registers.
//   mixing: warps q and q + 4 own slot q.  A thread handles two (token,
//     16-byte fragment) items of its stage: stage-1 sum of the tp partials in
//     FP32 in rank order, rounded to BF16 ([DSV]
//     _LamportMHCDeviceKernel.kernel, lane_sum); post-mix of the four streams
//     ([GLM] _BoundaryDeviceKernel.kernel, "mixed"), stored to residual_out
//     and, as the MMA's A operand, to shared memory; the sum of squares of
//     the new streams, reduced over the token's 16 lanes and written to the
//     partial-sum scratch.
//   GEMV (tensor cores): the MMA's 128 rows are (token t, stream j) with
//     row = 4t + j, its K the unit's 128 columns and its 96 columns (stream
//     j', output i): D[(t,j)][(j',i)] = sum_h new_j[t][h] * fn[j'*H + h][i];
//     the j' = j block of each row is that stream's part of the prenorm GEMV
//     ([GLM] _BoundaryDeviceKernel.kernel, "partial").  hc_fn is FP32; it is
//     split into three BF16 terms (hi + mid + lo, remainder below 2^-24
//     relative) so that each BF16 x BF16 product is exact and the sum
//     accumulates in FP32 in tensor memory: 3 x 8 MMAs of M=128, N=96, K=16,
//     issued by one thread into one of two accumulators (by unit parity).
//   epilogue (one unit later, so that it overlaps the next unit's loads):
//     TMEM lane quarter q holds the rows of stage q's tokens, four lanes per
//     token; warp q reads outputs 0-11 and warp q + 4 outputs 12-23 of all
//     four blocks, the four streams of a token are added in the order
//     ((j0 + j1) + (j2 + j3)) with warp shuffles, and the sums go to the
//     scratch rows [m][groups][25] (24 sums + the sum of squares; rows padded
//     to 16 bytes) that the finish kernel reduces.
// Every wait is bounded; a wait that gives up sets bit 1 of the error word.
//
// Pages: [GLM] vllm.models.glm5next.nvidia.specialized_decode.all_reduce_mhc,
//        [DSV] vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "device_common.cuh"
#include "launch.cuh"
#include "tcgen05.cuh"

namespace mhc {
namespace {

constexpr int NT = 256;                       // 8 warps (256 threads leave 255 registers a thread)
constexpr int UT = 32;                        // tokens per unit
constexpr int ROWS = HC * UT;                 // MMA M: (token, stream) rows
constexpr int UK = TC_GROUP_COLS;             // MMA K per term: the unit's 128 columns
constexpr int KCOLS = UK / 8;                 // core-matrix columns of 8 BF16
constexpr int UN = HC * MIX;                  // MMA N: (stream', output) columns
constexpr int QT = 8;                         // tokens per pipeline stage
constexpr int NSTAGE = UT / QT;               // ring slots = stages per unit
constexpr int SLOT_THREADS = 64;              // threads per slot (two warps)
constexpr int FRAGS = UK / VEC;               // 16-byte fragments per row piece
constexpr int A_KCOL = ROWS * 16 + 16;        // bytes between A core columns (+16: no bank conflicts)
constexpr int A_BYTES = KCOLS * A_KCOL;
constexpr int B_KCOL = UN * 16;               // bytes between B core columns
constexpr int B_BYTES = 3 * KCOLS * B_KCOL;   // hi, mid, lo
constexpr int ROW = UK * 2;                   // bytes of one 128-column BF16 row piece
constexpr int STAGE_PART = 0;                 // [tp][8 tokens][128] bf16
constexpr int STAGE_RES = TP_TMA_MAX * QT * ROW;          // [8 tokens][4][128] bf16
constexpr int STAGE_POST = STAGE_RES + QT * HC * ROW;     // [8][4] f32
constexpr int STAGE_COMB = STAGE_POST + 128;              // [8][16] f32
constexpr int STAGE_BYTES = STAGE_COMB + QT * HC * HC * 4;
constexpr int OUT_HALF = MIX / 2;             // outputs one epilogue warp reads per block
constexpr uint32_t D_STRIDE = 128;            // TMEM columns between the two accumulators
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t WAIT_LIMIT = 1u << 22;     // polls before a wait gives up
static_assert(QT * HC * 4 <= 128, "post block");
static_assert(UK % 16 == 0 && UN % 16 == 0 && UN <= 256, "MMA shape");
static_assert(QT * FRAGS == 2 * SLOT_THREADS, "two items per thread");
static_assert(ROWS == 4 * 32 && QT * HC == 32, "one TMEM lane quarter per stage");
static_assert(OUT_HALF % 4 == 0 && OUT_HALF == 3 * HC, "epilogue split");

struct Layout {
  static constexpr size_t a = 0;
  static constexpr size_t b = A_BYTES;
  static constexpr size_t stages = ((b + B_BYTES + 127) / 128) * 128;
  static constexpr size_t full = stages + size_t(NSTAGE) * STAGE_BYTES;  // uint64 [NSTAGE]
  static constexpr size_t empty = full + 8 * NSTAGE;                     // uint64 [NSTAGE]
  static constexpr size_t mma = empty + 8 * NSTAGE;                      // uint64 [2]
  static constexpr size_t slot = mma + 16;                               // TMEM address
  static constexpr size_t cabort = slot + 4;                             // int
  static constexpr size_t total = cabort + 12;
  static_assert(b % 16 == 0 && STAGE_BYTES % 128 == 0, "TMA / MMA alignment");
  static_assert(STAGE_RES % 128 == 0 && STAGE_POST % 128 == 0 && STAGE_COMB % 128 == 0, "TMA alignment");
  static_assert(full % 8 == 0, "mbarrier alignment");
  static_assert(total <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ void cta_sync() { asm volatile("bar.sync 0;" ::: "memory"); }

// The group's hc_fn as three BF16 B operands (hi, mid, lo), K-major core
// matrices [term][core column][8-column block][8 columns][8 inputs];
// column n = stream * 24 + output, input k = column in the group.  Every
// thread issues all its loads before the first split, so the build costs
// one memory latency rather than one per element pair.
constexpr int B_PAIRS = (UK / 2) * UN / NT;   // element pairs per thread
static_assert((UK / 2) * UN % NT == 0, "B build split");
__device__ __noinline__ void build_b(const StageParams &p, int h0, unsigned char *b_s) {
  float x0[B_PAIRS], x1[B_PAIRS];
#pragma unroll
  for (int it = 0; it < B_PAIRS; ++it) {
    const int e = threadIdx.x + it * NT;
    const int kp = e / UN, n = e % UN, j = n / MIX, i = n % MIX;
    const int h = h0 + 2 * kp;
    const float *src = p.hc_fn + ((size_t)j * p.hidden + h) * MIX + i;
    x0[it] = h < p.hidden ? __ldg(src) : 0.f;
    x1[it] = h + 1 < p.hidden ? __ldg(src + MIX) : 0.f;
  }
#pragma unroll
  for (int it = 0; it < B_PAIRS; ++it) {
    const int e = threadIdx.x + it * NT;
    const int kp = e / UN, n = e % UN, k = 2 * kp;
    const uint32_t hi = pack_bf16x2(x0[it], x1[it]);
    const float r0 = __fsub_rn(x0[it], bf16_lo(hi)), r1 = __fsub_rn(x1[it], bf16_hi(hi));
    const uint32_t mid = pack_bf16x2(r0, r1);
    const uint32_t lo = pack_bf16x2(__fsub_rn(r0, bf16_lo(mid)), __fsub_rn(r1, bf16_hi(mid)));
    const size_t inner = size_t(n / 8) * 128 + (n % 8) * 16 + (k % 8) * 2;
    *reinterpret_cast<uint32_t *>(b_s + size_t(0 * KCOLS + k / 8) * B_KCOL + inner) = hi;
    *reinterpret_cast<uint32_t *>(b_s + size_t(1 * KCOLS + k / 8) * B_KCOL + inner) = mid;
    *reinterpret_cast<uint32_t *>(b_s + size_t(2 * KCOLS + k / 8) * B_KCOL + inner) = lo;
  }
}

// Two BF16 values of a packed word as an FP32 pair.
__device__ __forceinline__ float2 unpack2(uint32_t w) { return make_float2(bf16_lo(w), bf16_hi(w)); }
__device__ __forceinline__ void unpack4x2(const uint4 &v, float2 (&x)[4]) {
  x[0] = unpack2(v.x);
  x[1] = unpack2(v.y);
  x[2] = unpack2(v.z);
  x[3] = unpack2(v.w);
}
// Rounds four FP32 pairs to BF16 in place; returns the packed words.
__device__ __forceinline__ uint4 round4x2(float2 (&x)[4]) {
  const uint4 w = make_uint4(pack_bf16x2(x[0].x, x[0].y), pack_bf16x2(x[1].x, x[1].y),
                             pack_bf16x2(x[2].x, x[2].y), pack_bf16x2(x[3].x, x[3].y));
  unpack4x2(w, x);
  return w;
}
__device__ __forceinline__ float lane4(const float4 &v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}
__device__ __forceinline__ float2 dup(float x) { return make_float2(x, x); }

// One (token, fragment) of a filled stage, copied to registers so that the
// ring slot can be released before the arithmetic.
struct Item {
  uint4 part[TP_TMA_MAX];
  uint4 res[HC];
  float4 post;
  float4 comb[HC];
};

__device__ __forceinline__ void load_item(int tp, const unsigned char *st, int tl, int f, Item &it) {
#pragma unroll
  for (int q = 0; q < TP_TMA_MAX; ++q)
    if (q < tp) it.part[q] = *reinterpret_cast<const uint4 *>(st + STAGE_PART + (q * QT + tl) * ROW + f * 16);
#pragma unroll
  for (int k = 0; k < HC; ++k)
    it.res[k] = *reinterpret_cast<const uint4 *>(st + STAGE_RES + (tl * HC + k) * ROW + f * 16);
  it.post = *reinterpret_cast<const float4 *>(st + STAGE_POST + tl * HC * 4);
#pragma unroll
  for (int k = 0; k < HC; ++k)
    it.comb[k] = *reinterpret_cast<const float4 *>(st + STAGE_COMB + (tl * HC + k) * HC * 4);
}

// Stage 1 and post-mix of two items in one instruction stream; returns the
// stage-1 sums and the new streams as BF16 fragments and each item's sum of
// squares.  The post-mix runs on FP32 element pairs (packed mul / fma, each
// lane rounded to nearest as the scalar operation would be).
__device__ __forceinline__ void mix_pair(int tp, const Item (&it)[2], uint4 (&yb)[2], uint4 (&nv)[2][HC],
                                         float (&ss)[2]) {
  float2 y[2][4];
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int e = 0; e < 4; ++e) y[k][e] = make_float2(0.f, 0.f);
#pragma unroll
  for (int q = 0; q < TP_TMA_MAX; ++q) {
    if (q < tp) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        // FP32 += BF16 with the widening folded into the add (exact, so
        // each lane rounds once, as the FP32 add of the widened value would)
        const uint32_t ww[4] = {it[k].part[q].x, it[k].part[q].y, it[k].part[q].z, it[k].part[q].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          asm("{.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tadd.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;}"
              : "+f"(y[k][e].x), "+f"(y[k][e].y) : "r"(ww[e]));
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    yb[k] = round4x2(y[k]);
    float2 res[HC][4];
#pragma unroll
    for (int c = 0; c < HC; ++c) unpack4x2(it[k].res[c], res[c]);
    float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < HC; ++j) {
      float2 o[4];
      const float2 pj = dup(lane4(it[k].post, j));
      // comb[i][j] weighs source stream i in output stream j
      const float2 c0 = dup(lane4(it[k].comb[0], j)), c1 = dup(lane4(it[k].comb[1], j));
      const float2 c2 = dup(lane4(it[k].comb[2], j)), c3 = dup(lane4(it[k].comb[3], j));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float2 v = __fmul2_rn(y[k][e], pj);
        v = __ffma2_rn(res[0][e], c0, v);
        v = __ffma2_rn(res[1][e], c1, v);
        v = __ffma2_rn(res[2][e], c2, v);
        v = __ffma2_rn(res[3][e], c3, v);
        o[e] = v;
      }
      nv[k][j] = round4x2(o);
#pragma unroll
      for (int e = 0; e < 4; ++e) ss2 = __ffma2_rn(o[e], o[e], ss2);
    }
    ss[k] = ss2.x + ss2.y;
  }
}

// Unit i's GEMV sums, once its MMAs are done (the tensor memory holds two
// accumulators, by unit parity).  Lane l of a warp in lane quarter q holds
// row 32q + l = (token 8q + l/4, stream l%4); the warp reads outputs
// 12*half .. 12*half+11 of all four stream blocks, each lane takes its own
// stream's block from the four lanes of its token and adds them in the order
// ((j0 + j1) + (j2 + j3)); lane j of the token writes three of the sums.
__device__ __forceinline__ void epilogue(const StageParams &p, uint32_t tmem, uint64_t *mma_bar, int i,
                                         int u_begin, int n_tiles, int q, int half, bool &ok) {
  const int lane = threadIdx.x & 31;
  const int u = u_begin + i, grpc = u / n_tiles, tile = u % n_tiles, d = i & 1;
  if (ok && !tc::mbar_wait_bounded(&mma_bar[d], (i >> 1) & 1, WAIT_LIMIT)) ok = false;
  tc::fence_after_sync();
  uint32_t raw[HC][OUT_HALF];
  const uint32_t base = tmem + (uint32_t(32 * q) << 16) + uint32_t(d) * D_STRIDE + uint32_t(OUT_HALF * half);
#pragma unroll
  for (int jb = 0; jb < HC; ++jb)
#pragma unroll
    for (int c = 0; c < OUT_HALF; c += 4) tc::tmem_ld4_async(base + uint32_t(jb * MIX + c), &raw[jb][c]);
  tc::tmem_wait_ld();
#pragma unroll
  for (int jb = 0; jb < HC; ++jb)
#pragma unroll
    for (int c = 0; c < OUT_HALF; c += 4) tc::tmem_hold4(&raw[jb][c]);
  const int src = lane & ~3, j = lane & 3;
  float out[3] = {0.f, 0.f, 0.f};
#pragma unroll
  for (int c = 0; c < OUT_HALF; ++c) {
    const float s0 = __shfl_sync(0xffffffffu, __uint_as_float(raw[0][c]), src + 0);
    const float s1 = __shfl_sync(0xffffffffu, __uint_as_float(raw[1][c]), src + 1);
    const float s2 = __shfl_sync(0xffffffffu, __uint_as_float(raw[2][c]), src + 2);
    const float s3 = __shfl_sync(0xffffffffu, __uint_as_float(raw[3][c]), src + 3);
    const float sum = (s0 + s1) + (s2 + s3);
    if (c / 3 == j) out[c % 3] = sum;
  }
  const int t = tile * UT + q * QT + (lane >> 2);
  if (ok && t < p.m) {
    float *dst = p.part + (size_t)t * p.part_stride + grpc * VALUES + OUT_HALF * half + 3 * j;
    dst[0] = out[0];
    dst[1] = out[1];
    dst[2] = out[2];
  }
}

__global__ void __launch_bounds__(NT, 1)
    k_stage_tc(const StageParams p, const __grid_constant__ CUtensorMap tm_part,
               const __grid_constant__ CUtensorMap tm_res, const __grid_constant__ CUtensorMap tm_post,
               const __grid_constant__ CUtensorMap tm_comb) {
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *a_s = smem + Layout::a;
  unsigned char *b_s = smem + Layout::b;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + Layout::full);
  uint64_t *empty = reinterpret_cast<uint64_t *>(smem + Layout::empty);
  uint64_t *mma_bar = reinterpret_cast<uint64_t *>(smem + Layout::mma);
  uint32_t *slot = reinterpret_cast<uint32_t *>(smem + Layout::slot);
  // Set before a CTA barrier and read after it: every thread takes the same
  // decision to stop.
  volatile int *cabort_s = reinterpret_cast<volatile int *>(smem + Layout::cabort);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.slices;                               // 128-column groups
  const int n_tiles = (p.m + UT - 1) / UT;
  const int units = n_tiles * G;
  const int u_begin = int((long long)blockIdx.x * units / gridDim.x);
  const int u_end = int((long long)(blockIdx.x + 1) * units / gridDim.x);
  const int n_units = u_end - u_begin;

  if (tid == 0) {
    for (int i = 0; i < NSTAGE; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], SLOT_THREADS);
    }
    tc::mbar_init(&mma_bar[0], 1);
    tc::mbar_init(&mma_bar[1], 1);
    *cabort_s = 0;
    tc::mbar_init_fence();
  }
  if (warp == 0) tc::tmem_alloc(slot, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *slot;

  const uint32_t idesc = tc::idesc_bf16_f32(ROWS, UN);
  const int q = warp & 3, half = warp >> 2, f = lane & (FRAGS - 1);
  // this thread's two tokens of stage q
  int tl[2];
  tl[0] = 4 * half + (lane >> 4);
  tl[1] = tl[0] + 2;
  unsigned char *stage = smem + Layout::stages + size_t(q) * STAGE_BYTES;
  bool ok = true;
  const bool filler = half == 0 && lane == 0;   // issues slot q's copies
  const uint32_t tx = uint32_t(p.tp) * QT * ROW + QT * HC * ROW + QT * HC * 4 + QT * HC * HC * 4;
  int fills = 0;                                 // copies issued into slot q (by the filler)
  auto fill = [&](int n) {
    const int u = u_begin + n, h0 = (u / n_tiles) * UK, t0 = (u % n_tiles) * UT + q * QT;
    tc::mbar_arrive_expect_tx(&full[q], tx);
    tc::tma_load_3d(stage + STAGE_PART, &tm_part, h0, t0, 0, &full[q]);
    tc::tma_load_3d(stage + STAGE_RES, &tm_res, h0, 0, t0, &full[q]);
    tc::tma_load_2d(stage + STAGE_POST, &tm_post, 0, t0, &full[q]);
    tc::tma_load_2d(stage + STAGE_COMB, &tm_comb, 0, t0, &full[q]);
    fills = n + 1;
  };
  if (filler && n_units > 0) {
    tc::tma_prefetch_desc(&tm_part);
    tc::tma_prefetch_desc(&tm_res);
    tc::tma_prefetch_desc(&tm_post);
    tc::tma_prefetch_desc(&tm_comb);
    fill(0);
  }

  int cur_group = -1, pending = -1, issued = -1;
  for (int i = 0; i < n_units; ++i) {
    const int u = u_begin + i, gc = u / n_tiles, tile = u % n_tiles;
    if (gc != cur_group) {
      // B is about to change: the previous unit's MMAs must be done with it
      if (pending >= 0) epilogue(p, tmem, mma_bar, pending, u_begin, n_tiles, q, half, ok);
      pending = -1;
      cta_sync();
      build_b(p, gc * UK, b_s);
      tc::fence_proxy_async_smem();
      cta_sync();
      cur_group = gc;
    }
    const int h = gc * UK + f * VEC;
    if (ok && !tc::mbar_wait_bounded(&full[q], i & 1, WAIT_LIMIT)) ok = false;
    Item it[2];
    if (ok) {
      load_item(p.tp, stage, tl[0], f, it[0]);
      load_item(p.tp, stage, tl[1], f, it[1]);
    }
    // The slot's next fill is an async-proxy write: the generic-proxy reads
    // above are ordered before it by a proxy fence ahead of the release.
    tc::fence_proxy_async_smem();
    tc::mbar_arrive(&empty[q]);
    // once both warps of the slot hold unit i's stage, the slot takes unit i + 1's
    if (filler && ok && i + 1 < n_units) {
      if (tc::mbar_wait_bounded(&empty[q], i & 1, WAIT_LIMIT))
        fill(i + 1);
      else
        ok = false;
    }
    uint4 yb[2], nv[2][HC];
    float ss[2];
    mix_pair(p.tp, it, yb, nv, ss);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int t = tile * UT + q * QT + tl[k];
      if (ok && t < p.m && h < p.hidden) {
        if (p.reduced_out) st_vec(p.reduced_out + (size_t)t * p.hidden + h, yb[k]);
#pragma unroll
        for (int j = 0; j < HC; ++j) st_vec(p.residual_out + ((size_t)t * HC + j) * p.hidden + h, nv[k][j]);
      } else {
        // columns past H and tokens past m contribute nothing to the GEMV
#pragma unroll
        for (int j = 0; j < HC; ++j) nv[k][j] = make_uint4(0, 0, 0, 0);
        ss[k] = 0.f;
      }
    }
    // the A buffer is free once the previous unit's MMAs are done
    if (pending >= 0) epilogue(p, tmem, mma_bar, pending, u_begin, n_tiles, q, half, ok);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
#pragma unroll
      for (int j = 0; j < HC; ++j) {
        const int row = 32 * q + 4 * tl[k] + j;
        *reinterpret_cast<uint4 *>(a_s + size_t(f) * A_KCOL + (row / 8) * 128 + (row % 8) * 16) = nv[k][j];
      }
      // the 16 fragments of a token are 16 consecutive lanes
      float s = ss[k];
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      s += __shfl_xor_sync(0xffffffffu, s, 4);
      s += __shfl_xor_sync(0xffffffffu, s, 8);
      const int t = tile * UT + q * QT + tl[k];
      if (f == 0 && ok && t < p.m) p.part[(size_t)t * p.part_stride + gc * VALUES + MIX] = s;
    }
    pending = -1;
    // hand the A buffer to the tensor core
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    if (!ok) *cabort_s = 1;
    cta_sync();
    if (*cabort_s) {
      ok = false;
      break;
    }
    if (tid == 0) {
      tc::fence_after_sync();
      const uint32_t a_addr = tc::smem_addr(a_s), b_addr = tc::smem_addr(b_s);
      const uint32_t d = uint32_t(i & 1) * D_STRIDE;
#pragma unroll 1
      for (int term = 0; term < 3; ++term) {
#pragma unroll
        for (int ks = 0; ks < UK / 16; ++ks) {
          const uint64_t ad = tc::smem_desc(a_addr + uint32_t(2 * ks * A_KCOL), A_KCOL, 128);
          const uint64_t bd = tc::smem_desc(b_addr + uint32_t((term * KCOLS + 2 * ks) * B_KCOL), B_KCOL, 128);
          tc::mma_bf16(tmem + d, ad, bd, idesc, (term | ks) != 0);
        }
      }
      tc::mma_commit(&mma_bar[i & 1]);
    }
    pending = issued = i;
  }
  if (pending >= 0) epilogue(p, tmem, mma_bar, pending, u_begin, n_tiles, q, half, ok);
  // copies still in flight land before the CTA may exit
  if (filler && fills > 0) tc::mbar_wait_bounded(&full[q], (fills - 1) & 1, WAIT_LIMIT);
  if (!ok && tid == 0) {
    if (p.err) atomicOr(p.err, 2u);
    // MMAs still in flight finish before their tensor memory is released
    if (issued >= 0) tc::mbar_wait_bounded(&mma_bar[issued & 1], (issued >> 1) & 1, WAIT_LIMIT);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

bool encode(CUtensorMap *map, CUtensorMapDataType type, int rank, const void *base, const cuuint64_t *dims,
            const cuuint64_t *strides, const cuuint32_t *box) {
  const cuuint32_t ones[3] = {1, 1, 1};
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  return fn(map, type, cuuint32_t(rank), const_cast<void *>(base), dims, strides, box, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t stage_tc_smem_bytes() { return Layout::total; }

cudaError_t stage_tc_set_attributes() {
  if (!encode_fn()) return cudaErrorNotSupported;
  return cudaFuncSetAttribute(k_stage_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Layout::total));
}

cudaError_t launch_stage_tc(const StageParams &p, int ctas, cudaStream_t stream) {
  if (p.tp < 1 || p.tp > TP_TMA_MAX) return cudaErrorInvalidValue;
  if (p.slices != (p.hidden + TC_GROUP_COLS - 1) / TC_GROUP_COLS) return cudaErrorInvalidValue;
  const cuuint64_t H = cuuint64_t(p.hidden), M = cuuint64_t(p.m), TP = cuuint64_t(p.tp);
  CUtensorMap tm_part, tm_res, tm_post, tm_comb;
  const cuuint64_t part_dims[3] = {H, M, TP}, part_strides[2] = {H * 2, M * H * 2};
  const cuuint32_t part_box[3] = {UK, QT, cuuint32_t(p.tp)};
  const cuuint64_t res_dims[3] = {H, HC, M}, res_strides[2] = {H * 2, HC * H * 2};
  const cuuint32_t res_box[3] = {UK, HC, QT};
  const cuuint64_t post_dims[2] = {HC, M}, post_strides[1] = {HC * 4};
  const cuuint32_t post_box[2] = {HC, QT};
  const cuuint64_t comb_dims[2] = {HC * HC, M}, comb_strides[1] = {HC * HC * 4};
  const cuuint32_t comb_box[2] = {HC * HC, QT};
  if (!encode(&tm_part, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.partials, part_dims, part_strides, part_box) ||
      !encode(&tm_res, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.residual, res_dims, res_strides, res_box) ||
      !encode(&tm_post, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.post, post_dims, post_strides, post_box) ||
      !encode(&tm_comb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.comb, comb_dims, comb_strides, comb_box))
    return cudaErrorInvalidValue;
  const int units = ((p.m + UT - 1) / UT) * p.slices;
  const int grid = units < ctas ? units : ctas;
  k_stage_tc<<<grid, NT, Layout::total, stream>>>(p, tm_part, tm_res, tm_post, tm_comb);
  return cudaGetLastError();
}

}  // namespace mhc
