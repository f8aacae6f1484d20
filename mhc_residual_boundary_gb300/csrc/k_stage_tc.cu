// k_stage_tc.cu -- stage kernel: TMA-fed load pipeline, post-mix on CUDA
// cores, prenorm GEMV on tcgen05 tensor cores.
//
// Work unit: 32 tokens x one group of 128 hidden columns (every row piece a
// unit reads is a 256-byte run).  Units are numbered group-major.  Each CTA
// (persistent, one per SM) takes a contiguous range of them, or, when that
// costs no more than 10 % in its largest share, the CTAs are shared out over
// the groups and each takes a contiguous range of its group's token tiles
// (the launcher decides).  Roles in a CTA of 18 warps:
//
//   producer warp (one lane issues): refills ring slots as soon as the mixer
//     warps release them -- stage q (tokens 8q .. 8q+7) of every unit by four
//     TMA tensor copies: the partials [tp][m][H] (one 3-D box of 128 columns
//     x 8 tokens x tp ranks), the residual streams [m][4][H], post [m][4] and
//     comb [m][4][4], counted on the slot's mbarrier; out-of-range tokens and
//     columns arrive as zeros.
//   MMA warp (one lane issues): a unit's MMAs as soon as its A operand is
//     complete, then the unit's new streams from A to residual_out by two
//     swizzled TMA tensor stores; it releases A (the MMA barrier) once the
//     MMAs are done and the stores have read A.  It also owns the tensor
//     memory.
//   16 mixer warps: four per stage, one (token, 16-byte fragment) item per
//     thread.  Stage-1 sum of the tp partials in FP32 in rank order, rounded
//     to BF16 ([DSV] _LamportMHCDeviceKernel.kernel, lane_sum); post-mix of
//     the four streams ([GLM] _BoundaryDeviceKernel.kernel, "mixed"), written
//     as the MMA's A operand to shared memory; the sum of squares of the new
//     streams over the token's 16 lanes.  They also build the B operand when
//     the group changes and read the accumulators.
//   GEMV (tensor cores): the MMA's 128 rows are (token t, stream j) with
//     row = 4t + j, its K the unit's 128 columns and its 96 columns (stream
//     j', output i): D[(t,j)][(j',i)] = sum_h new_j[t][h] * fn[j'*H + h][i];
//     the j' = j block of each row is that stream's part of the prenorm GEMV
//     ([GLM] _BoundaryDeviceKernel.kernel, "partial").  hc_fn is FP32; it is
//     split into three BF16 terms (hi + mid + lo, remainder below 2^-24
//     relative) so that each BF16 x BF16 product is exact and the sum
//     accumulates in FP32 in tensor memory: 3 x 8 MMAs of M=128, N=96, K=16
//     into one of two accumulators (by unit parity).  A BF16 weight ([GLM]
//     `fn`, [24][4H]) is one term: 8 MMAs.
//   order of a mixer iteration: post-mix of unit i, wait for unit i - 1's
//     MMAs (and stores), A rows of unit i to shared memory and to the MMA
//     warp, then -- while those MMAs run -- the token sums of squares and the
//     epilogue of unit i - 1.
//   epilogue (one unit later):
//     warp w reads TMEM lane quarter w % 4 (the rows of stage w % 4's
//     tokens, four lanes per token) and six of the 24 outputs of all four
//     stream blocks; each lane keeps its own stream's block and the four
//     lanes of a token add them in the order ((j0 + j1) + (j2 + j3)).  The
//     sums go to the scratch rows [m][groups][25] (24 sums + the sum of
//     squares; rows padded to 16 bytes) that the finish kernel reduces.
//
// A group's weight rows arrive by bulk (FP32) or tiled (BF16) copies into
// the A buffer, which is idle at that point, and the mixers split or place
// them into B from shared memory.  The kernel is a programmatic dependent
// launch: set-up, and for a layer weight the first group's staging and
// split, happen before it waits for the preceding kernel; the producer
// prefetches the later groups' rows into L2.  Without the GEMV (the
// delayed-mHC consumer) there is no A, B or MMA, and the mixers store the
// new streams themselves.  Every wait is bounded; a wait that gives up sets
// bit 1 of the error word and stops the CTA.
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

// Test hook (mhc_test_stall_stage_copies): when set, the producer issues no
// input copies, so the kernel's bounded waits run out and it reports the
// timeout through the error word instead of hanging.
__device__ int g_stall_copies = 0;

constexpr int MIX_WARPS = 16;                 // mixer warps
constexpr int PROD_WARP = MIX_WARPS;          // the TMA producer warp
constexpr int MMA_WARP = MIX_WARPS + 1;       // the MMA warp
constexpr int NT = (MIX_WARPS + 2) * 32;      // 576 threads
constexpr int MIX_THREADS = MIX_WARPS * 32;
constexpr int UT = 32;                        // tokens per unit
constexpr int ROWS = HC * UT;                 // MMA M: (token, stream) rows
constexpr int UK = TC_GROUP_COLS;             // MMA K per term: the unit's 128 columns
constexpr int KCOLS = UK / 8;                 // core-matrix columns of 8 BF16
constexpr int UN = HC * MIX;                  // MMA N: (stream', output) columns
constexpr int QT = 8;                         // tokens per pipeline stage
constexpr int NSTAGE = UT / QT;               // stages per unit
constexpr int STAGE_WARPS = MIX_WARPS / NSTAGE;   // mixer warps per stage
constexpr int FRAGS = UK / VEC;               // 16-byte fragments per row piece
// A: two halves of 64 columns, each 128 rows of 128 bytes in the 128-byte
// swizzled K-major layout (16-byte chunk c of row r at chunk c ^ (r % 8)),
// which the tensor core reads and a swizzled TMA store writes out as is.
constexpr int A_ROW = 128;                    // bytes of one row of a half
constexpr int A_HALF = ROWS * A_ROW;          // 16 KB
constexpr int A_BYTES = 2 * A_HALF;
constexpr int B_KCOL = UN * 16;               // bytes between B core columns
constexpr int TERM_BYTES = KCOLS * B_KCOL;    // one BF16 term of B
constexpr int ROW = UK * 2;                   // bytes of one 128-column BF16 row piece
constexpr int MAX_SLOTS = 8;
constexpr uint32_t D_STRIDE = 128;            // TMEM columns between the two accumulators
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t WAIT_LIMIT = 1u << 22;     // polls before a wait gives up
constexpr int SMEM_MAX = 227 * 1024;          // dynamic shared memory of one CTA
constexpr int B_PAIRS = (UK / 2) * UN / MIX_THREADS;   // hc_fn element pairs per mixer thread
constexpr int OUTS = MIX / STAGE_WARPS;       // outputs one epilogue warp reads per block (6)
constexpr int HC_ROWS_BYTES = UK * MIX * 4;   // one stream's hc_fn rows of a group (FP32)
constexpr int STAGING = HC * HC_ROWS_BYTES;   // a group's hc_fn rows, staged over the A buffer
constexpr int FN_SEG = UK * 2;                // BF16 weight: one (output, stream) row piece of a group
constexpr int STAGING_BF16 = MIX * HC * FN_SEG;   // a group's 96 row pieces
static_assert(QT * FRAGS == STAGE_WARPS * 32, "one item per mixer thread");
static_assert(ROWS == 4 * 32 && QT * HC == 32, "one TMEM lane quarter per stage");
static_assert((UK / 2) * UN % MIX_THREADS == 0 && B_PAIRS == 12, "B build split");
static_assert(OUTS == 6, "epilogue split: four outputs plus two");
static_assert(UK % 16 == 0 && UN % 16 == 0 && UN <= 256, "MMA shape");

// Shared memory: control block, B (three BF16 terms for an FP32 weight, one
// for a BF16 weight), A (whose space also takes a group's staged weight
// rows), then the ring of stage slots.
struct Layout {
  static constexpr int full = 0;                        // uint64 [MAX_SLOTS][2] (see full_bar)
  static constexpr int empty = full + 16 * MAX_SLOTS;   // uint64 [MAX_SLOTS]
  static constexpr int afull = empty + 8 * MAX_SLOTS;   // uint64: A operand complete
  static constexpr int mma = afull + 8;                 // uint64 [2]: MMAs of a unit done
  static constexpr int bfull = mma + 16;                // uint64: a group's hc_fn rows staged
  static constexpr int bbuilt = bfull + 8;              // uint64: every mixer warp has split a group into B
  static constexpr int slot = bbuilt + 8;               // TMEM address
  static constexpr int abort = slot + 4;                // int
  static constexpr int b = 1024;
  static_assert(abort + 4 <= b, "control block");
  // A (after B) starts on a 1024-byte boundary: the swizzle pattern repeats
  // every 8 rows of 128 bytes
  static_assert(b % 1024 == 0 && TERM_BYTES % 1024 == 0 && A_BYTES % 128 == 0, "TMA / MMA alignment");
};
__host__ __device__ constexpr int layout_a(int terms) { return Layout::b + terms * TERM_BYTES; }
__host__ __device__ constexpr int layout_ring(int terms) {
  return terms == 0 ? Layout::b   // no GEMV (the delayed-mHC consumer): neither B nor A
                    : layout_a(terms) + (terms == 3 ? (A_BYTES > STAGING ? A_BYTES : STAGING)
                                                    : (A_BYTES > STAGING_BF16 ? A_BYTES : STAGING_BF16));
}
static_assert(layout_ring(3) % 128 == 0 && layout_ring(1) % 128 == 0, "TMA alignment");

// A stage slot: partials [tp][8][128] bf16, streams [8][4][128] bf16,
// post [8][4] f32, comb [8][16] f32 (each part 128-byte aligned).
__host__ __device__ constexpr int slot_res(int tp) { return tp * QT * ROW; }
__host__ __device__ constexpr int slot_post(int tp) { return slot_res(tp) + QT * HC * ROW; }
__host__ __device__ constexpr int slot_comb(int tp) { return slot_post(tp) + QT * HC * 4; }
__host__ __device__ constexpr int slot_bytes(int tp) { return slot_comb(tp) + QT * HC * HC * 4; }
// Ring slots: 8, 6 or 4 (as many as the shared memory holds).  Slot n % nslot
// takes stage n % 4.  With 4 or 8 slots every use of a slot is consumed by
// the same four warps in order.  With 6 a slot alternates between two
// stages' warps; an mbarrier tells phases apart only by parity, so each slot
// then has two "full" barriers, one for its even and one for its odd uses,
// each consumed by one stage's warps in order (full_bar).
__host__ __device__ constexpr int ring_slots(int tp, int terms) {
  return (SMEM_MAX - layout_ring(terms)) / slot_bytes(tp) >= 8   ? 8
         : (SMEM_MAX - layout_ring(terms)) / slot_bytes(tp) >= 6 ? 6
                                                                 : 4;
}
static_assert(slot_bytes(1) % 128 == 0 && slot_post(1) % 128 == 0 && slot_comb(1) % 128 == 0, "slot alignment");
static_assert(ring_slots(TP_TMA_MAX, 3) >= NSTAGE, "a unit's four stages fit the ring");
static_assert(MAX_SLOTS == 8 && (SMEM_MAX - layout_ring(3)) / slot_bytes(TP_TMA_MAX) >= 4, "ring of 4, 6 or 8 slots");

// The "full" barrier of fill n (slot n % nslot, use n / nslot) and the parity
// of that use's phase on it.
struct FullBar {
  int index;
  uint32_t parity;
};
__device__ __forceinline__ FullBar full_bar(int n, int nslot) {
  const int s = n % nslot, use = n / nslot;
  if (nslot % NSTAGE == 0) return {2 * s, uint32_t(use & 1)};
  return {2 * s + (use & 1), uint32_t((use >> 1) & 1)};
}

__device__ __forceinline__ float2 unpack2(uint32_t w) { return make_float2(bf16_lo(w), bf16_hi(w)); }
__device__ __forceinline__ float lane4(const float4 &v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}
__device__ __forceinline__ float2 dup(float x) { return make_float2(x, x); }

// Rounds four FP32 pairs to BF16 in place; returns the packed words.
__device__ __forceinline__ uint4 round4x2(float2 (&x)[4]) {
  const uint4 w = make_uint4(pack_bf16x2(x[0].x, x[0].y), pack_bf16x2(x[1].x, x[1].y),
                             pack_bf16x2(x[2].x, x[2].y), pack_bf16x2(x[3].x, x[3].y));
  x[0] = unpack2(w.x);
  x[1] = unpack2(w.y);
  x[2] = unpack2(w.z);
  x[3] = unpack2(w.w);
  return w;
}

// FP32 pair += the BF16 pair of a packed word; the widening is folded into
// the add (exact, so each lane rounds once, as the FP32 add of the widened
// value would).
__device__ __forceinline__ void add_bf16x2(float2 &acc, uint32_t w) {
  asm("{.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tadd.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;}"
      : "+f"(acc.x), "+f"(acc.y)
      : "r"(w));
}

// ------------------------------------------------------------- B operand
// The group's hc_fn as three BF16 B operands (hi, mid, lo), K-major core
// matrices [term][core column][8-column block][8 columns][8 inputs];
// column n = stream * 24 + output, input k = column in the group.  Mixer
// thread `tid` owns element pairs e = tid + 512 * it (inputs 2kp, 2kp + 1 of
// column n), with (kp, n) chosen so that a warp's 32 stores fill 32 banks:
// with rest = e / 32, kp = 4 (rest / 12) + e % 4 and n = 8 (rest % 12) +
// (e / 4) % 8.

// Splits the group's staged hc_fn rows (stream j's rows at stg + j * 128 * 24
// floats; rows past `rows` are treated as zero) into B.  A plain loop: the
// code is short, and every load is a shared-memory read.  The operands are
// addressed through their 32-bit shared-window addresses: this is a separate
// function, which generic pointers would reach without their address space.
__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts_u32(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __noinline__ void convert_b(const float *stg, int rows, unsigned char *b_s) {
  const uint32_t s0 = tc::smem_addr(stg), b0 = tc::smem_addr(b_s);
  // Element pair e = tid + 512 * it (above): rest = e / 32 grows by 16 = 12 + 4
  // an iteration, so its quotient q and remainder r by 12 are carried along;
  // then kp = 4q + e % 4, n = 8r + c with c = (e / 4) % 8 (fixed), and n's
  // stream j = r / 3, output i = 8 (r % 3) + c.
  const int c = (int(threadIdx.x) >> 2) & 7, kq = int(threadIdx.x) & 3;
  int q = 0, r = int(threadIdx.x) >> 5;   // rest < 16 at it = 0
  if (r >= 12) {
    q = 1;
    r -= 12;
  }
#pragma unroll 2
  for (int it = 0; it < B_PAIRS; ++it) {
    const int kp = 4 * q + kq, k = 2 * kp;
    const int j = (r * 11) >> 5, i = (r - 3 * j) * 8 + c;   // r / 3 for r < 12
    const uint32_t src = s0 + uint32_t(((j * UK + k) * MIX + i) * 4);
    const float x0 = k < rows ? lds_f32(src) : 0.f;
    const float x1 = k + 1 < rows ? lds_f32(src + MIX * 4) : 0.f;
    const uint32_t hi = pack_bf16x2(x0, x1);
    const float r0 = __fsub_rn(x0, bf16_lo(hi)), r1 = __fsub_rn(x1, bf16_hi(hi));
    const uint32_t mid = pack_bf16x2(r0, r1);
    const uint32_t lo = pack_bf16x2(__fsub_rn(r0, bf16_lo(mid)), __fsub_rn(r1, bf16_hi(mid)));
    const uint32_t dst = b0 + uint32_t(q * B_KCOL + r * 128 + c * 16 + kq * 4);
    sts_u32(dst, hi);
    sts_u32(dst + KCOLS * B_KCOL, mid);
    sts_u32(dst + 2 * KCOLS * B_KCOL, lo);
    q += 1;
    r += 4;
    if (r >= 12) {
      q += 1;
      r -= 12;
    }
  }
}

// The BF16 weight's group: its 96 staged row pieces (output i, stream j at
// stg + (j * 24 + i) * 256 bytes, 128 columns each; columns past `rows` are
// zero) are already BF16, so B is their 16-byte pieces moved to the core-
// matrix layout: piece (n, kc) of row n = j * 24 + i to core column kc.
__device__ __noinline__ void place_b_bf16(const unsigned char *stg, int rows, unsigned char *b_s) {
  constexpr int PIECES = UN * KCOLS;
  static_assert(PIECES % MIX_THREADS == 0, "B placement split");
#pragma unroll
  for (int it = 0; it < PIECES / MIX_THREADS; ++it) {
    const int e = threadIdx.x + it * MIX_THREADS;
    const int kc = e % KCOLS, n = e / KCOLS;
    const uint4 v = kc * 8 < rows ? *reinterpret_cast<const uint4 *>(stg + n * FN_SEG + kc * 16)
                                  : make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4 *>(b_s + kc * B_KCOL + (n >> 3) * 128 + (n & 7) * 16) = v;
  }
}

// Rows of group g (at most 128; fewer in the last group).
__device__ __forceinline__ int group_rows(int hidden, int g) {
  return hidden - g * UK < UK ? hidden - g * UK : UK;
}

// Group g's weight rows into `stg`, counted on `bar`; called by a whole warp.
// FP32 weight: four bulk copies (one per stream, 128 rows of 24 floats).
// BF16 weight: four tiled copies (one per stream: 24 rows of 128 columns).
__device__ __forceinline__ void stage_hc_fn(const StageParams &p, const CUtensorMap *tm_fn, int g,
                                            unsigned char *stg, uint64_t *bar) {
  const int rows = group_rows(p.hidden, g);
  if (tc::elect_one()) {
    if (p.fn_terms == 3) {
      tc::mbar_arrive_expect_tx(bar, uint32_t(HC * rows * MIX * 4));
      for (int j = 0; j < HC; ++j)
        tc::bulk_load(stg + j * HC_ROWS_BYTES, p.hc_fn + ((size_t)j * p.hidden + (size_t)g * UK) * MIX,
                      uint32_t(rows * MIX * 4), bar);
    } else {
      // the full boxes arrive (columns past the weight are zero-filled)
      tc::mbar_arrive_expect_tx(bar, uint32_t(HC * MIX * FN_SEG));
      for (int j = 0; j < HC; ++j)
        tc::tma_load_2d(stg + j * MIX * FN_SEG, tm_fn, j * p.hidden + g * UK, 0, bar);
    }
  }
  __syncwarp();
}

// Splits (FP32) or places (BF16) the staged weight rows of group g into B.
__device__ __forceinline__ void build_b(const StageParams &p, int g, const unsigned char *stg, unsigned char *b_s) {
  if (p.fn_terms == 3)
    convert_b(reinterpret_cast<const float *>(stg), group_rows(p.hidden, g), b_s);
  else
    place_b_bf16(stg, group_rows(p.hidden, g), b_s);
}

// The mixer warps' barrier after splitting weight group number `loads`
// (1, 2, ...): each warp arrives once, then waits, with a bound, for the
// phase of that group; a barrier with a bounded wait, so that a warp that has
// left the loop after a failed wait cannot hold the others forever.
__device__ __forceinline__ bool b_built(uint64_t *bbuilt, int loads, int lane) {
  __syncwarp();
  if (lane == 0) tc::mbar_arrive(bbuilt);
  return tc::mbar_wait_bounded(bbuilt, uint32_t((loads - 1) & 1), WAIT_LIMIT);
}

// ------------------------------------------------------------- epilogue
// Unit `i`'s GEMV sums once its MMAs are done.  Warp w reads lane quarter
// w % 4 -- row 32q + l = (token 8q + l/4, stream l%4) -- and outputs
// 4s .. 4s+3 and 16+2s, 17+2s (s = w / 4) of all four stream blocks; each
// lane takes its own stream's block, the four lanes of a token add them in
// the order ((j0 + j1) + (j2 + j3)) and lane o % 4 writes output o.
// Everything it reads is passed by value: an out-of-line function that took
// the kernel's parameter block by reference would read every field through a
// generic pointer into parameter space, which is slow.
struct Epi {
  float *part;             // the partial-sum scratch
  int part_stride, m;
  uint32_t tmem;
  uint64_t *mma_bar;
  volatile int *abort_s;
  int i, tile, group;
};

__device__ __noinline__ void epilogue(const Epi e) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3, s = warp >> 2, j = lane & 3, d = e.i & 1;
  const bool ok = tc::mbar_wait_bounded(&e.mma_bar[d], (e.i >> 1) & 1, WAIT_LIMIT);
  if (!ok) *e.abort_s = 1;
  tc::fence_after_sync();
  const uint32_t base = e.tmem + (uint32_t(32 * q) << 16) + uint32_t(d) * D_STRIDE;
  uint32_t r4[HC][4], r2[HC][2];
#pragma unroll
  for (int jb = 0; jb < HC; ++jb) {
    tc::tmem_ld4_async(base + uint32_t(jb * MIX + 4 * s), r4[jb]);
    tc::tmem_ld2_async(base + uint32_t(jb * MIX + 16 + 2 * s), r2[jb]);
  }
  tc::tmem_wait_ld();
#pragma unroll
  for (int jb = 0; jb < HC; ++jb) {
    tc::tmem_hold4(r4[jb]);
    tc::tmem_hold2(r2[jb]);
  }
  const int t = e.tile * UT + q * QT + (lane >> 2);
  float *dst = e.part + (size_t)t * e.part_stride + e.group * VALUES;
#pragma unroll
  for (int o = 0; o < OUTS; ++o) {
    const int c = o < 4 ? o : o - 4;
    const uint32_t v0 = o < 4 ? r4[0][c] : r2[0][c], v1 = o < 4 ? r4[1][c] : r2[1][c];
    const uint32_t v2 = o < 4 ? r4[2][c] : r2[2][c], v3 = o < 4 ? r4[3][c] : r2[3][c];
    const float v = __uint_as_float(j == 0 ? v0 : j == 1 ? v1 : j == 2 ? v2 : v3);
    float sum = v + __shfl_xor_sync(0xffffffffu, v, 1);
    sum = sum + __shfl_xor_sync(0xffffffffu, sum, 2);
    const int out = o < 4 ? 4 * s + o : 16 + 2 * s + (o - 4);
    if (ok && j == (o & 3) && t < e.m) dst[out] = sum;
  }
}

// ----------------------------------------------------------------- mixing
// One item (token tl of the stage, fragment f) of a filled slot, moved to
// registers so that the slot can be released before the post-mix: the
// stage-1 sum of the tp partials in rank order (still FP32), the four source
// streams, post and comb.
struct Item {
  float2 y[4];
  uint4 res[HC];
  float4 post;
  float4 comb[HC];
};

__device__ __forceinline__ void load_item(int tp, const unsigned char *st, int tl, int f, Item &it) {
#pragma unroll
  for (int e = 0; e < 4; ++e) it.y[e] = make_float2(0.f, 0.f);
#pragma unroll
  for (int r = 0; r < TP_TMA_MAX; ++r) {
    if (r < tp) {
      const uint4 w = *reinterpret_cast<const uint4 *>(st + (r * QT + tl) * ROW + f * 16);
      add_bf16x2(it.y[0], w.x);
      add_bf16x2(it.y[1], w.y);
      add_bf16x2(it.y[2], w.z);
      add_bf16x2(it.y[3], w.w);
    }
  }
  const unsigned char *rs = st + slot_res(tp) + tl * HC * ROW + f * 16;
#pragma unroll
  for (int k = 0; k < HC; ++k) it.res[k] = *reinterpret_cast<const uint4 *>(rs + k * ROW);
  it.post = *reinterpret_cast<const float4 *>(st + slot_post(tp) + tl * HC * 4);
#pragma unroll
  for (int k = 0; k < HC; ++k)
    it.comb[k] = *reinterpret_cast<const float4 *>(st + slot_comb(tp) + (tl * HC + k) * HC * 4);
}

// The stage-1 sum rounded to BF16 (yb) and the post-mixed streams
// new_j = y * post_j + sum_k res_k * comb[k][j] (one fused multiply-add per
// source in source order, on FP32 element pairs), rounded to BF16 (nv).
// Returns the sum of squares of the rounded streams.
__device__ __forceinline__ float mix_item(Item &it, uint4 &yb, uint4 (&nv)[HC]) {
  yb = round4x2(it.y);
  float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < HC; ++j) {
    const float2 pj = dup(lane4(it.post, j));
    // comb[k][j] weighs source stream k in output stream j
    float2 o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = __fmul2_rn(it.y[e], pj);
#pragma unroll
    for (int k = 0; k < HC; ++k) {
      const float2 ck = dup(lane4(it.comb[k], j));
      const uint32_t ww[4] = {it.res[k].x, it.res[k].y, it.res[k].z, it.res[k].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = __ffma2_rn(unpack2(ww[e]), ck, o[e]);
    }
    nv[j] = round4x2(o);
#pragma unroll
    for (int e = 0; e < 4; ++e) ss2 = __ffma2_rn(o[e], o[e], ss2);
  }
  return ss2.x + ss2.y;
}

// ------------------------------------------------------------------ kernel
// 18 warps put five on one SM sub-partition (16384 registers each), so a
// thread may use at most 96 registers.
__global__ void __launch_bounds__(NT, 1)
    k_stage_tc(const StageParams p, const __grid_constant__ CUtensorMap tm_part,
               const __grid_constant__ CUtensorMap tm_res, const __grid_constant__ CUtensorMap tm_post,
               const __grid_constant__ CUtensorMap tm_comb, const __grid_constant__ CUtensorMap tm_fn,
               const __grid_constant__ CUtensorMap tm_out) {
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + Layout::full);
  uint64_t *empty = reinterpret_cast<uint64_t *>(smem + Layout::empty);
  uint64_t *afull = reinterpret_cast<uint64_t *>(smem + Layout::afull);
  uint64_t *mma_bar = reinterpret_cast<uint64_t *>(smem + Layout::mma);
  uint64_t *bfull = reinterpret_cast<uint64_t *>(smem + Layout::bfull);
  uint64_t *bbuilt = reinterpret_cast<uint64_t *>(smem + Layout::bbuilt);
  uint32_t *slot = reinterpret_cast<uint32_t *>(smem + Layout::slot);
  volatile int *abort_s = reinterpret_cast<volatile int *>(smem + Layout::abort);
  unsigned char *a_s = smem + layout_a(p.fn_terms);
  unsigned char *b_s = smem + Layout::b;
  unsigned char *ring = smem + layout_ring(p.fn_terms);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = (p.m + UT - 1) / UT;
  const int units = n_tiles * p.slices;
  // Units are numbered group-major.  Either each CTA takes a contiguous
  // share of them, or (group_aligned) the C CTAs are shared out over the G
  // groups -- group g gets CTAs floor(g * C / G) .. floor((g + 1) * C / G) - 1
  // -- and each takes a contiguous share of its group's tiles, so that no CTA
  // splits a second weight group.
  // (32-bit unsigned divisions where the products fit, as they do at every
  // size but a million tokens and more: a 64-bit division by a run-time
  // value is a long software routine, and this is on every CTA's start)
  int u_begin, u_end;
  const unsigned C = gridDim.x, b = blockIdx.x;
  if (p.group_aligned) {
    const unsigned G = unsigned(p.slices), T = unsigned(n_tiles);
    const unsigned g = ((b + 1) * G - 1) / C;   // G, C <= 1024
    const unsigned c0 = g * C / G, c1 = (g + 1) * C / G;
    const unsigned k = b - c0, n = c1 - c0;
    const bool narrow = T <= 0xffffffffu / C;
    u_begin = int(g * T + (narrow ? k * T / n : unsigned((unsigned long long)k * T / n)));
    u_end = int(g * T + (narrow ? (k + 1) * T / n : unsigned((unsigned long long)(k + 1) * T / n)));
  } else {
    const unsigned U = unsigned(units);
    const bool narrow = U <= 0xffffffffu / C;
    u_begin = int(narrow ? b * U / C : unsigned((unsigned long long)b * U / C));
    u_end = int(narrow ? (b + 1) * U / C : unsigned((unsigned long long)(b + 1) * U / C));
  }
  const int n_units = u_end - u_begin;             // >= 1: the grid is at most `units`
  const int nslot = ring_slots(p.tp, p.fn_terms), sbytes = slot_bytes(p.tp);
  const int total_fills = n_units * NSTAGE;
  const int first_group = u_begin / n_tiles;
  const bool gemv = p.fn_terms > 0;                // false: streams only (delayed-mHC consumer)

  // The finish kernel may be scheduled on SMs as they free up; it waits for
  // this whole grid (and its memory) before it reads anything this grid writes.
  pdl_launch_dependents();

  // Stage `n` (unit n / 4, stage n % 4) into ring slot n % nslot; called by
  // the whole producer warp, one lane issues.
  auto fill = [&](int n) {
    const int u = u_begin + n / NSTAGE, q = n % NSTAGE;
    const int h0 = (u / n_tiles) * UK, t0 = (u % n_tiles) * UT + q * QT, s = n % nslot;
    unsigned char *st = ring + s * sbytes;
    if (tc::elect_one()) {
      uint64_t *bar = &full[full_bar(n, nslot).index];
      tc::mbar_arrive_expect_tx(bar, uint32_t(sbytes));
      tc::tma_load_3d(st, &tm_part, h0, t0, 0, bar);
      tc::tma_load_3d(st + slot_res(p.tp), &tm_res, h0, 0, t0, bar);
      tc::tma_load_2d(st + slot_post(p.tp), &tm_post, 0, t0, bar);
      tc::tma_load_2d(st + slot_comb(p.tp), &tm_comb, 0, t0, bar);
    }
    __syncwarp();
  };

  if (warp == PROD_WARP) {
    if (tc::elect_one()) {
      for (int s = 0; s < nslot; ++s) {
        tc::mbar_init(&full[2 * s], 1);
        tc::mbar_init(&full[2 * s + 1], 1);
        tc::mbar_init(&empty[s], STAGE_WARPS);
      }
      tc::mbar_init(afull, MIX_WARPS);
      tc::mbar_init(&mma_bar[0], 1);
      tc::mbar_init(&mma_bar[1], 1);
      tc::mbar_init(bfull, 1);
      tc::mbar_init(bbuilt, MIX_WARPS);
      *abort_s = 0;
      tc::mbar_init_fence();
      tc::tma_prefetch_desc(&tm_part);
      tc::tma_prefetch_desc(&tm_res);
      tc::tma_prefetch_desc(&tm_post);
      tc::tma_prefetch_desc(&tm_comb);
      if (p.fn_terms == 1) tc::tma_prefetch_desc(&tm_fn);
      if (gemv) tc::tma_prefetch_desc(&tm_out);
    }
    __syncwarp();
    // a layer weight: the first group's rows while the preceding kernel
    // finishes (nothing before the wait below may read the call's inputs)
    if (gemv && p.early_weight) stage_hc_fn(p, &tm_fn, first_group, a_s, bfull);
  } else if (warp == MMA_WARP) {
    tc::tmem_alloc(slot, TMEM_COLS);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *slot;

  if (warp == PROD_WARP) {
    // The inputs, and the outputs that the preceding kernel may still read,
    // are touched only after it has completed.
    pdl_wait();
    const bool stall = *static_cast<volatile int *>(&g_stall_copies) != 0;
    if (gemv && !p.early_weight) stage_hc_fn(p, &tm_fn, first_group, a_s, bfull);
    for (int n = 0; !stall && n < nslot && n < total_fills; ++n) fill(n);
    // the later groups' weight rows, so that their staging copies read L2
    const int last_group = gemv ? (u_end - 1) / n_tiles : first_group;
    for (int g = first_group + 1; g <= last_group && g <= first_group + 16; ++g) {
      const int rows = group_rows(p.hidden, g);
      if (p.fn_terms == 3) {
        for (int j = lane; j < HC; j += 32)
          tc::prefetch_l2(p.hc_fn + ((size_t)j * p.hidden + (size_t)g * UK) * MIX, uint32_t(rows * MIX * 4));
      } else {
        for (int j = lane; j < HC; j += 32) tc::tma_prefetch_2d(&tm_fn, j * p.hidden + g * UK, 0);
      }
      __syncwarp();
    }
    // refill each slot as soon as its previous stage has been read
    int nf = stall ? 0 : nslot < total_fills ? nslot : total_fills;
    for (; !stall && nf < total_fills; ++nf) {
      const int s = nf % nslot;
      if (!tc::mbar_wait_bounded(&empty[s], uint32_t((nf / nslot - 1) & 1), WAIT_LIMIT) || *abort_s) {
        if (lane == 0) *abort_s = 1;
        break;
      }
      fill(nf);
    }
    // copies still in flight land before exit
    for (int n = nf - nslot < 0 ? 0 : nf - nslot; n < nf; ++n)
      tc::mbar_wait_bounded(&full[full_bar(n, nslot).index], full_bar(n, nslot).parity, WAIT_LIMIT);
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // a unit's 3 x 8 MMAs once its A operand is complete
    const uint32_t idesc = tc::idesc_bf16_f32(ROWS, UN);
    // A: 128-byte swizzle (layout type 2), 8-row groups 1024 bytes apart
    const uint64_t a0 = tc::smem_desc(tc::smem_addr(a_s), 16, 8 * A_ROW) | (uint64_t(2) << 61);
    const uint64_t b0 = tc::smem_desc(tc::smem_addr(b_s), B_KCOL, 128);
    int nm = 0;
    for (; gemv && nm < n_units; ++nm) {
      if (!tc::mbar_wait_bounded(afull, uint32_t(nm & 1), WAIT_LIMIT) || *abort_s) {
        if (lane == 0) *abort_s = 1;
        break;
      }
      tc::fence_after_sync();
      const uint32_t d = tmem + uint32_t(nm & 1) * D_STRIDE;
      if (tc::elect_one()) {
#pragma unroll 1
        for (int term = 0; term < p.fn_terms; ++term) {
#pragma unroll
          for (int ks = 0; ks < UK / 16; ++ks) {
            // K step ks: half ks / 4, byte 32 * (ks % 4) of the swizzled row
            const uint64_t ad = a0 + uint64_t(((ks >> 2) * A_HALF + (ks & 3) * 32) >> 4);
            const uint64_t bd = b0 + uint64_t(((term * KCOLS + 2 * ks) * B_KCOL) >> 4);
            tc::mma_bf16(d, ad, bd, idesc, (term | ks) != 0);
          }
        }
        // the unit's new streams, A as it stands, to residual_out: one
        // swizzled tensor store per half (rows past m, columns past H are
        // not written); A is released (the MMA barrier) only after both
        // stores have read it
        const int u = u_begin + nm, h0 = (u / n_tiles) * UK, t0 = (u % n_tiles) * UT;
        tc::tma_store_3d(&tm_out, a_s, h0, 0, t0);
        if (h0 + UK / 2 < p.hidden) tc::tma_store_3d(&tm_out, a_s + A_HALF, h0 + UK / 2, 0, t0);
        tc::bulk_commit_group();
        tc::bulk_wait_read_all();
        tc::mma_commit(&mma_bar[nm & 1]);
      }
      __syncwarp();
    }
    // issued MMAs complete before the tensor memory is released, and the
    // stores before the CTA exits
    if (nm > 0) tc::mbar_wait_bounded(&mma_bar[(nm - 1) & 1], uint32_t(((nm - 1) >> 1) & 1), WAIT_LIMIT);
    if (tc::elect_one()) tc::bulk_wait_all();
    __syncwarp();
  } else {
    const int q = warp / STAGE_WARPS, item = (warp % STAGE_WARPS) * 32 + lane;
    const int tl = item / FRAGS, f = item % FRAGS;
    Epi ep = {p.part, p.part_stride, p.m, tmem, mma_bar, abort_s, -1, 0, 0};
    int cur_group = -1, loads = 0;   // hc_fn groups staged so far
    if (gemv && p.early_weight) {
      // the first group's B, split while the preceding kernel finishes
      if (!tc::mbar_wait_bounded(bfull, 0u, WAIT_LIMIT)) *abort_s = 1;
      ++loads;
      build_b(p, first_group, a_s, b_s);
      // every mixer has read the staged rows before any A row is written
      if (!b_built(bbuilt, loads, lane)) *abort_s = 1;
      cur_group = first_group;
    }
    pdl_wait();
    for (int i = 0; i < n_units; ++i) {
      if (*abort_s) break;
      const int u = u_begin + i, g = u / n_tiles, tile = u % n_tiles;
      const int n = i * NSTAGE + q, s = n % nslot;
      const FullBar fb = full_bar(n, nslot);
      if (!tc::mbar_wait_bounded(&full[fb.index], fb.parity, WAIT_LIMIT)) {
        *abort_s = 1;
        break;
      }
      Item it;
      load_item(p.tp, ring + s * sbytes, tl, f, it);
      // The slot's next fill is an async-proxy write: the generic-proxy reads
      // above are ordered before it by a proxy fence ahead of the release.
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[s]);
      uint4 yb, nv[HC];
      float ss = mix_item(it, yb, nv);
      const int t = tile * UT + q * QT + tl, h = g * UK + f * VEC;
      const bool live = t < p.m && h < p.hidden;
      if (!gemv) {
        if (live) {
          if (p.reduced_out) st_vec(p.reduced_out + (size_t)t * p.hidden + h, yb);
#pragma unroll
          for (int j = 0; j < HC; ++j) st_vec(p.residual_out + ((size_t)t * HC + j) * p.hidden + h, nv[j]);
        }
        continue;
      }
      // The A buffer (and B) are free once the previous unit's MMAs are done.
      if (i > 0 && !tc::mbar_wait_bounded(&mma_bar[(i - 1) & 1], uint32_t(((i - 1) >> 1) & 1), WAIT_LIMIT)) {
        *abort_s = 1;
        break;
      }
      if (g != cur_group) {
        // B and the A space change; the first group's rows were staged at
        // kernel start, so their split overlaps the first unit's loads
        if (cur_group >= 0 && warp == 0) stage_hc_fn(p, &tm_fn, g, a_s, bfull);
        if (!tc::mbar_wait_bounded(bfull, uint32_t(loads & 1), WAIT_LIMIT)) {
          *abort_s = 1;
          break;
        }
        ++loads;
        build_b(p, g, a_s, b_s);
        // every mixer has read the staged rows before any A row is written
        if (!b_built(bbuilt, loads, lane)) {
          *abort_s = 1;
          break;
        }
        cur_group = g;
      }
#pragma unroll
      for (int j = 0; j < HC; ++j) {
        const int row = 32 * q + 4 * tl + j;
        *reinterpret_cast<uint4 *>(a_s + (f >> 3) * A_HALF + row * A_ROW + (((f & 7) ^ (row & 7)) << 4)) = nv[j];
      }
      // hand the A rows (and a new B) to the tensor core
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(afull);
      // while the tensor core runs (and the MMA warp stores the new streams
      // from A): the stage-1 sum if asked for, the token's sum of squares (its
      // 16 fragments are 16 consecutive lanes) and the previous unit's sums
      // (its MMAs are done: waited for above)
      if (live && p.reduced_out) st_vec(p.reduced_out + (size_t)t * p.hidden + h, yb);
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      ss += __shfl_xor_sync(0xffffffffu, ss, 2);
      ss += __shfl_xor_sync(0xffffffffu, ss, 4);
      ss += __shfl_xor_sync(0xffffffffu, ss, 8);
      if (f == 0 && t < p.m) p.part[(size_t)t * p.part_stride + g * VALUES + MIX] = ss;
      if (ep.i >= 0) epilogue(ep);
      ep.i = i;
      ep.tile = tile;
      ep.group = g;
    }
    if (ep.i >= 0 && !*abort_s) epilogue(ep);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == MMA_WARP) tc::tmem_dealloc(tmem, TMEM_COLS);
  if (tid == 0 && *abort_s && p.err) atomicOr(p.err, 2u);
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
            const cuuint64_t *strides, const cuuint32_t *box,
            CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
  const cuuint32_t ones[3] = {1, 1, 1};
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  return fn(map, type, cuuint32_t(rank), const_cast<void *>(base), dims, strides, box, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t stage_tc_smem_bytes() { return size_t(SMEM_MAX); }

cudaError_t stage_tc_stall_copies(int on) {
  return cudaMemcpyToSymbol(g_stall_copies, &on, sizeof on);
}

cudaError_t stage_tc_set_attributes() {
  if (!encode_fn()) return cudaErrorNotSupported;
  return cudaFuncSetAttribute(k_stage_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX);
}

cudaError_t launch_stage_tc(const StageParams &p, int ctas, cudaStream_t stream, int *grid_out) {
  if (p.tp < 1 || p.tp > TP_TMA_MAX) return cudaErrorInvalidValue;
  if (p.slices != (p.hidden + TC_GROUP_COLS - 1) / TC_GROUP_COLS) return cudaErrorInvalidValue;
  if (!(p.fn_terms == 3 && p.hc_fn) && !(p.fn_terms == 1 && p.hc_fn_bf16) && p.fn_terms != 0)
    return cudaErrorInvalidValue;
  const cuuint64_t H = cuuint64_t(p.hidden), M = cuuint64_t(p.m), TP = cuuint64_t(p.tp);
  CUtensorMap tm_part, tm_res, tm_post, tm_comb, tm_fn = {}, tm_out = {};
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
  if (p.fn_terms > 0) {
    // residual_out [m][4][H], written from A: box of 64 columns x 4 streams x
    // 32 tokens, 128-byte swizzle (one half of A)
    const cuuint32_t out_box[3] = {UK / 2, HC, UT};
    if (!encode(&tm_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.residual_out, res_dims, res_strides, out_box,
                CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  if (p.fn_terms == 1) {
    // the BF16 weight [24][4H]: box of 128 columns x 24 rows (one stream of a group)
    const cuuint64_t fn_dims[2] = {HC * H, MIX}, fn_strides[1] = {HC * H * 2};
    const cuuint32_t fn_box[2] = {UK, MIX};
    if (!encode(&tm_fn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.hc_fn_bf16, fn_dims, fn_strides, fn_box))
      return cudaErrorInvalidValue;
  }
  // One unit per CTA when there are no more units than CTAs.  Else the
  // group-aligned split on floor(ctas / groups) CTAs per group, when its
  // largest share is within 10 % of the contiguous split's: no CTA then
  // stages and splits a second weight group on its critical path, and the
  // CTAs of all groups sweep the same token tiles together, so that the
  // tokens' rows are read from HBM close together in time.
  const int tiles = (p.m + UT - 1) / UT, units = tiles * p.slices;
  int grid = units < ctas ? units : ctas;
  StageParams q = p;
  q.group_aligned = 0;
  if (units > ctas && ctas >= p.slices && p.fn_terms > 0) {
    const int per = ctas / p.slices;
    if (10 * ((tiles + per - 1) / per) <= 11 * ((units + ctas - 1) / ctas)) {
      q.group_aligned = 1;
      grid = per * p.slices;
    }
  }
  if (grid_out) *grid_out = grid;
  const size_t smem = size_t(layout_ring(p.fn_terms)) + size_t(ring_slots(p.tp, p.fn_terms)) * slot_bytes(p.tp);
  // programmatic dependent launch: the CTAs' setup (and, for a layer weight,
  // its staging and split) overlaps the end of the preceding kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_stage_tc, q, tm_part, tm_res, tm_post, tm_comb, tm_fn, tm_out);
}

}  // namespace mhc
