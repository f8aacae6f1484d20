// k_stage_tc.cu -- stage kernel: TMA-fed load pipeline, post-mix on CUDA
// cores, prenorm GEMV on tcgen05 tensor cores.
//
// Work unit: 32 tokens x one group of 128 hidden columns.  Every row a unit
// reads is a 256-byte run (HBM delivers 128-byte pieces of rows 12 KB apart
// far more slowly).  Units are numbered group-major and every CTA (one per
// SM, persistent) takes a contiguous range of them, so a CTA stages each
// group's hc_fn once.  Per CTA:
//
//   producer warp (one thread): for every 8-token stage of a unit, four TMA
//     tensor copies into a four-slot shared-memory ring -- the partials
//     [tp][m][H] (one 3-D box: 128 columns x 8 tokens x tp ranks), the
//     residual streams [m][4][H], post [m][4] and comb [m][4][4] -- tracked by
//     the slot's mbarrier transaction count.  Out-of-range tokens and columns
//     arrive as zeros.
//   8 consumer warps in two groups taking alternate stages, thread = token x
//   16-byte fragment: stage-1 sum of the tp partials in FP32 in rank order,
//     rounded to BF16 ([DSV] _LamportMHCDeviceKernel.kernel, lane_sum);
//     post-mix of the four streams ([GLM] _BoundaryDeviceKernel.kernel,
//     "mixed"), stored to residual_out and, as the MMA's A operand, to shared
//     memory; the sum of squares of the new streams.
//   GEMV (tensor cores): the MMA's 128 rows are (stream j, token t), its K the
//     unit's 128 columns and its 96 columns (stream j', output i):
//     D[(j,t)][(j',i)] = sum_h new_j[t][h] * fn[j'*H + h][i]; the j' = j block
//     of each row is that stream's part of the prenorm GEMV ([GLM]
//     _BoundaryDeviceKernel.kernel, "partial").  hc_fn is FP32; it is split
//     into three BF16 terms (hi + mid + lo, remainder below 2^-24 relative) so
//     that each BF16 x BF16 product is exact and the sum accumulates in FP32
//     in tensor memory: 3 x 8 MMAs of M=128, N=96, K=16 per unit.
//   epilogue: each warp reads its stream's 24 sums per token (tcgen05.ld),
//     the four streams are added through shared memory, and each token's 24
//     sums and its sum of squares go to the partial-sum scratch [m][groups][25]
//     that the finish kernel reduces.
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

constexpr int CONSUMERS = 256;                // 8 consumer warps
constexpr int NT = CONSUMERS + 32;            // + the producer warp
constexpr int UT = 32;                        // tokens per unit
constexpr int ROWS = HC * UT;                 // MMA M: (stream, token) rows
constexpr int UK = TC_GROUP_COLS;             // MMA K per term: the unit's 128 columns
constexpr int KCOLS = UK / 8;                 // core-matrix columns of 8 BF16
constexpr int UN = HC * MIX;                  // MMA N: (stream', output) columns
constexpr int QT = 8;                         // tokens per pipeline stage
constexpr int STAGES_PER_UNIT = UT / QT;      // even ones to warps 0-3, odd ones to warps 4-7
constexpr int A_KCOL = ROWS * 16 + 16;        // bytes between A core columns (+16: no bank conflicts)
constexpr int A_BYTES = KCOLS * A_KCOL;
constexpr int B_KCOL = UN * 16;               // bytes between B core columns
constexpr int B_BYTES = 3 * KCOLS * B_KCOL;   // hi, mid, lo
constexpr int ROW = UK * 2;                   // bytes of one 128-column BF16 row
constexpr int STAGE_PART = 0;                 // [tp][8 tokens][128] bf16
constexpr int STAGE_RES = TP_TMA_MAX * QT * ROW;          // [8 tokens][4][128] bf16
constexpr int STAGE_POST = STAGE_RES + QT * HC * ROW;     // [8][4] f32
constexpr int STAGE_COMB = STAGE_POST + 128;              // [8][16] f32
constexpr int STAGE_BYTES = STAGE_COMB + QT * HC * HC * 4;
constexpr int NSTAGE = 4;                     // ring slots
constexpr int GROUP = CONSUMERS / 2;          // consumer threads per stage
constexpr uint32_t D_STRIDE = 128;            // TMEM columns between the two accumulators
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t WAIT_LIMIT = 1u << 22;     // polls before a wait gives up
static_assert(QT * HC * 4 <= 128, "post block");
static_assert(UK % 16 == 0 && UN % 16 == 0 && UN <= 256, "MMA shape");

struct Layout {
  static constexpr size_t a = 0;
  static constexpr size_t b = A_BYTES;
  static constexpr size_t stages = ((b + B_BYTES + 127) / 128) * 128;
  static constexpr size_t red = stages + size_t(NSTAGE) * STAGE_BYTES;  // float [4][UT][24]
  static constexpr size_t ss = red + size_t(HC) * UT * MIX * 4;         // float [2][UT]
  static constexpr size_t full = ss + 2 * UT * 4;                       // uint64 [NSTAGE]
  static constexpr size_t empty = full + 8 * NSTAGE;                    // uint64 [NSTAGE]
  static constexpr size_t mma = empty + 8 * NSTAGE;                     // uint64 [2]
  static constexpr size_t slot = mma + 16;                              // TMEM address
  static constexpr size_t abort = slot + 4;                             // int
  static constexpr size_t fill = abort + 4;                             // int [NSTAGE]
  static constexpr size_t cabort = fill + 4 * NSTAGE;                   // int
  static constexpr size_t total = cabort + 8;
  static_assert(b % 16 == 0 && STAGE_BYTES % 128 == 0, "TMA / MMA alignment");
  static_assert(STAGE_RES % 128 == 0 && STAGE_POST % 128 == 0 && STAGE_COMB % 128 == 0, "TMA alignment");
  static_assert(full % 8 == 0, "mbarrier alignment");
  static_assert(total <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// The group's hc_fn as three BF16 B operands (hi, mid, lo), K-major core
// matrices [term][core column][8-column block][8 columns][8 inputs];
// column n = stream * 24 + output, input k = column in the group.
__device__ void build_b(const StageParams &p, int h0, unsigned char *b_s) {
  for (int e = threadIdx.x; e < (UK / 2) * UN; e += CONSUMERS) {
    const int kp = e / UN, n = e % UN, j = n / MIX, i = n % MIX;
    const int k = 2 * kp, h = h0 + k;
    const float *src = p.hc_fn + ((size_t)j * p.hidden + h) * MIX + i;
    const float x0 = h < p.hidden ? __ldg(src) : 0.f;
    const float x1 = h + 1 < p.hidden ? __ldg(src + MIX) : 0.f;
    const uint32_t hi = pack_bf16x2(x0, x1);
    const float r0 = __fsub_rn(x0, bf16_lo(hi)), r1 = __fsub_rn(x1, bf16_hi(hi));
    const uint32_t mid = pack_bf16x2(r0, r1);
    const uint32_t lo = pack_bf16x2(__fsub_rn(r0, bf16_lo(mid)), __fsub_rn(r1, bf16_hi(mid)));
    const size_t inner = size_t(n / 8) * 128 + (n % 8) * 16 + (k % 8) * 2;
    *reinterpret_cast<uint32_t *>(b_s + size_t(0 * KCOLS + k / 8) * B_KCOL + inner) = hi;
    *reinterpret_cast<uint32_t *>(b_s + size_t(1 * KCOLS + k / 8) * B_KCOL + inner) = mid;
    *reinterpret_cast<uint32_t *>(b_s + size_t(2 * KCOLS + k / 8) * B_KCOL + inner) = lo;
  }
}

// Stage 1 and post-mix of one (token, fragment) from a filled stage; returns
// the new streams as BF16 fragments and their sum of squares.
__device__ __forceinline__ void mix_item(const StageParams &p, const unsigned char *st, int tl, int f, int t,
                                         int h, uint4 (&nv)[HC], float &ss) {
  float y[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) y[e] = 0.f;
#pragma unroll
  for (int q = 0; q < TP_TMA_MAX; ++q) {
    if (q < p.tp) {
      float x[8];
      unpack8(*reinterpret_cast<const uint4 *>(st + STAGE_PART + (q * QT + tl) * ROW + f * 16), x);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = __fadd_rn(y[e], x[e]);
    }
  }
  const uint4 yb = round8(y);
  if (p.reduced_out) st_vec(p.reduced_out + (size_t)t * p.hidden + h, yb);
  float res[HC][8];
#pragma unroll
  for (int k = 0; k < HC; ++k)
    unpack8(*reinterpret_cast<const uint4 *>(st + STAGE_RES + (tl * HC + k) * ROW + f * 16), res[k]);
  const float *post = reinterpret_cast<const float *>(st + STAGE_POST) + tl * HC;
  const float *comb = reinterpret_cast<const float *>(st + STAGE_COMB) + tl * HC * HC;
#pragma unroll
  for (int j = 0; j < HC; ++j) {
    float o[8];
    const float pj = post[j];
    const float c0 = comb[0 * HC + j], c1 = comb[1 * HC + j], c2 = comb[2 * HC + j], c3 = comb[3 * HC + j];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float v = __fmul_rn(y[e], pj);
      v = __fmaf_rn(res[0][e], c0, v);
      v = __fmaf_rn(res[1][e], c1, v);
      v = __fmaf_rn(res[2][e], c2, v);
      v = __fmaf_rn(res[3][e], c3, v);
      o[e] = v;
    }
    nv[j] = round8(o);
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(o[e], o[e], ss);
    st_vec(p.residual_out + ((size_t)t * HC + j) * p.hidden + h, nv[j]);
  }
}

__global__ void __launch_bounds__(NT, 1)
    k_stage_tc(const StageParams p, const __grid_constant__ CUtensorMap tm_part,
               const __grid_constant__ CUtensorMap tm_res, const __grid_constant__ CUtensorMap tm_post,
               const __grid_constant__ CUtensorMap tm_comb) {
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *a_s = smem + Layout::a;
  unsigned char *b_s = smem + Layout::b;
  float *red_s = reinterpret_cast<float *>(smem + Layout::red);
  float *ss_s = reinterpret_cast<float *>(smem + Layout::ss);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + Layout::full);
  uint64_t *empty = reinterpret_cast<uint64_t *>(smem + Layout::empty);
  uint64_t *mma_bar = reinterpret_cast<uint64_t *>(smem + Layout::mma);
  uint32_t *slot = reinterpret_cast<uint32_t *>(smem + Layout::slot);
  volatile int *abort_s = reinterpret_cast<volatile int *>(smem + Layout::abort);
  // Index of the fill a ring slot last received: a consumer waits until its
  // slot holds its own fill before the parity wait, so that the parity wait
  // can never be satisfied by an older phase of the same slot.
  volatile int *fill_s = reinterpret_cast<volatile int *>(smem + Layout::fill);
  // Set only by consumers, before a consumer barrier, and read after it: all
  // consumers take the same decision to stop (the producer's flag may change
  // at any time).
  volatile int *cabort_s = reinterpret_cast<volatile int *>(smem + Layout::cabort);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.slices;                               // 128-column groups
  const int n_tiles = (p.m + UT - 1) / UT;
  const int units = n_tiles * G;
  const int u_begin = int((long long)blockIdx.x * units / gridDim.x);
  const int u_end = int((long long)(blockIdx.x + 1) * units / gridDim.x);

  if (tid == 0) {
    for (int i = 0; i < NSTAGE; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], GROUP);
      fill_s[i] = -1;
    }
    tc::mbar_init(&mma_bar[0], 1);
    tc::mbar_init(&mma_bar[1], 1);
    *abort_s = 0;
    *cabort_s = 0;
    tc::mbar_init_fence();
  }
  if (warp == 0) tc::tmem_alloc(slot, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *slot;

  if (warp == CONSUMERS / 32) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tc::tma_prefetch_desc(&tm_part);
      tc::tma_prefetch_desc(&tm_res);
      tc::tma_prefetch_desc(&tm_post);
      tc::tma_prefetch_desc(&tm_comb);
      const uint32_t tx = uint32_t(p.tp) * QT * ROW + QT * HC * ROW + QT * HC * 4 + QT * HC * HC * 4;
      int g = 0;
      for (int u = u_begin; u < u_end && !*abort_s; ++u) {
        const int h0 = (u / n_tiles) * UK, tile = u % n_tiles;
        for (int q = 0; q < STAGES_PER_UNIT; ++q, ++g) {
          const int st = g % NSTAGE, n = g / NSTAGE;
          if (n >= 1 && !tc::mbar_wait_bounded(&empty[st], (n - 1) & 1, WAIT_LIMIT)) {
            *abort_s = 1;
            break;
          }
          unsigned char *dst = smem + Layout::stages + size_t(st) * STAGE_BYTES;
          const int t0 = tile * UT + q * QT;
          tc::mbar_arrive_expect_tx(&full[st], tx);
          tc::tma_load_3d(dst + STAGE_PART, &tm_part, h0, t0, 0, &full[st]);
          tc::tma_load_3d(dst + STAGE_RES, &tm_res, h0, 0, t0, &full[st]);
          tc::tma_load_2d(dst + STAGE_POST, &tm_post, 0, t0, &full[st]);
          tc::tma_load_2d(dst + STAGE_COMB, &tm_comb, 0, t0, &full[st]);
          __threadfence_block();
          fill_s[st] = g;
        }
      }
      // copies still in flight complete before the CTA may exit
      for (int k = g - NSTAGE; k < g; ++k)
        if (k >= 0) tc::mbar_wait_bounded(&full[k % NSTAGE], (k / NSTAGE) & 1, WAIT_LIMIT);
    }
  } else {
    // ----------------------------------------------------------- consumers
    const uint32_t idesc = tc::idesc_bf16_f32(ROWS, UN);
    // thread = (token of the stage, 16-byte fragment of the 128 columns)
    const int grp = warp >> 2, gt = tid & (GROUP - 1), tl = gt >> 4, f = gt & 15;
    bool ok = true;
    // Reads unit i's accumulator once its MMAs are done: warp w holds rows
    // (stream w%4, token lane); it reads its stream's 24 sums (warps 0-3
    // outputs 0-15, warps 4-7 outputs 16-23) into red_s, the streams are added
    // in order ((j0 + j1) + (j2 + j3)), and the 24 sums plus the sum of
    // squares of every token go to the scratch.
    auto epilogue = [&](int i) {
      const int u = u_begin + i, grpc = u / n_tiles, tile = u % n_tiles, d = i & 1;
      if (ok && !tc::mbar_wait_bounded(&mma_bar[d], (i >> 1) & 1, WAIT_LIMIT)) ok = false;
      tc::fence_after_sync();
      const int j = warp & 3, c0 = (warp >> 2) * 16;
      const uint32_t col = tmem + (uint32_t(32 * j) << 16) + uint32_t(d) * D_STRIDE + uint32_t(j * MIX + c0);
      float v[16];
      tc::tmem_ld8(col, v);
      tc::tmem_ld8(col + 8, v + 8);
#pragma unroll
      for (int c = 0; c < 16; ++c)
        if (c0 + c < MIX) red_s[(j * UT + lane) * MIX + c0 + c] = v[c];
      tc::fence_before_sync();
      consumer_sync();
      for (int e = tid; e < UT * VALUES; e += CONSUMERS) {
        const int et = e / VALUES, k = e % VALUES, t = tile * UT + et;
        if (!ok || t >= p.m) continue;
        float val;
        if (k < MIX)
          val = (red_s[(0 * UT + et) * MIX + k] + red_s[(1 * UT + et) * MIX + k]) +
                (red_s[(2 * UT + et) * MIX + k] + red_s[(3 * UT + et) * MIX + k]);
        else
          val = ss_s[d * UT + et];
        p.part[((size_t)t * G + grpc) * VALUES + k] = val;
      }
    };

    int cur_group = -1, pending = -1, issued = -1;
    for (int i = 0; u_begin + i < u_end; ++i) {
      const int u = u_begin + i, gc = u / n_tiles, tile = u % n_tiles;
      if (gc != cur_group) {
        // B is about to change: the previous unit's MMAs must be done with it
        if (pending >= 0) epilogue(pending);
        pending = -1;
        consumer_sync();
        build_b(p, gc * UK, b_s);
        tc::fence_proxy_async_smem();
        consumer_sync();
        cur_group = gc;
      }
      const int h = gc * UK + f * VEC;
      for (int jj = 0; jj < STAGES_PER_UNIT / 2; ++jj) {
        const int q = 2 * jj + grp, gq = i * STAGES_PER_UNIT + q, st = gq % NSTAGE;
        if (ok) {
          uint32_t n = 0;
          while (fill_s[st] != gq && n < WAIT_LIMIT) {
            if (*abort_s) break;
            if (++n > 64) __nanosleep(64);
          }
          if (fill_s[st] != gq || !tc::mbar_wait_bounded(&full[st], (gq / NSTAGE) & 1, WAIT_LIMIT)) ok = false;
        }
        const unsigned char *stage = smem + Layout::stages + size_t(st) * STAGE_BYTES;
        const int ut = q * QT + tl, t = tile * UT + ut;
        uint4 nv[HC] = {};
        float ssi = 0.f;
        if (ok && t < p.m && h < p.hidden) mix_item(p, stage, tl, f, t, h, nv, ssi);
        tc::mbar_arrive(&empty[st]);   // the slot may be refilled
        if (jj == 0 && pending >= 0) {
          // the A buffer is free once the previous unit's MMAs are done
          epilogue(pending);
        }
#pragma unroll
        for (int c = 0; c < HC; ++c) {
          const int row = c * UT + ut;
          *reinterpret_cast<uint4 *>(a_s + size_t(f) * A_KCOL + (row / 8) * 128 + (row % 8) * 16) = nv[c];
        }
        // the 16 fragments of a token are 16 consecutive lanes
        ssi += __shfl_xor_sync(0xffffffffu, ssi, 1);
        ssi += __shfl_xor_sync(0xffffffffu, ssi, 2);
        ssi += __shfl_xor_sync(0xffffffffu, ssi, 4);
        ssi += __shfl_xor_sync(0xffffffffu, ssi, 8);
        if (f == 0) ss_s[(i & 1) * UT + ut] = ssi;
      }
      pending = -1;
      // hand the A buffer to the tensor core
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      if (!ok) {
        *abort_s = 1;
        *cabort_s = 1;
      }
      consumer_sync();
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
    if (pending >= 0) epilogue(pending);
    if (!ok) {
      *abort_s = 1;
      if (tid == 0) {
        if (p.err) atomicOr(p.err, 2u);
        // MMAs still in flight finish before their tensor memory is released
        if (issued >= 0) tc::mbar_wait_bounded(&mma_bar[issued & 1], (issued >> 1) & 1, WAIT_LIMIT);
      }
    }
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
