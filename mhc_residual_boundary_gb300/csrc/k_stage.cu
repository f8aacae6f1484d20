// k_stage.cu -- stage kernel of the mHC boundary.
//
// One CTA owns a hidden slice of SLICE = 64 columns for a tile of T tokens:
//   phase A  (thread = token x 16-byte fragment): stage-1 sum of the tp BF16
//            partials in FP32 in rank order, rounded to BF16 ([DSV]
//            _LamportMHCDeviceKernel.kernel, lane_sum); then the post-mix of
//            the four residual streams ([GLM] _BoundaryDeviceKernel.kernel,
//            "mixed"), written to residual_out and to shared memory, and the
//            slice's sum of squares of the new streams;
//   phase B  the slice's part of the 24-way prenorm GEMV ([GLM]
//            _BoundaryDeviceKernel.kernel, "partial"): a [T x 256] x [256 x 24]
//            product from shared memory, hc_fn's slice staged once per CTA and
//            reused by all T tokens.
// The 25 per-token partial sums go to a scratch array that the finish kernel
// reduces in a fixed order.
//
// Pages: [GLM] vllm.models.glm5next.nvidia.specialized_decode.all_reduce_mhc,
//        [DSV] vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_reduce_mhc.
#include "device_common.cuh"
#include "launch.cuh"

namespace mhc {
namespace {

constexpr int KW = HC * SLICE;   // GEMV inputs of a slice: 4 streams x 64 columns
constexpr int FN_LD = KW + 4;    // fn_s row stride in floats (bank offset 4 per row)
constexpr int NEW_LD = KW + 8;   // new_s row stride in BF16 (bank offset 4 per row)
constexpr int MIX_LD = 20;       // post[4] + comb[16] per token

template <int T>
struct StageLayout {
  static constexpr size_t fn = 0;
  static constexpr size_t fn_bytes = size_t(MIX) * FN_LD * 4;
  static constexpr size_t news = fn + fn_bytes;
  static constexpr size_t news_bytes = size_t(T) * NEW_LD * 2;
  static constexpr size_t mixs = news + news_bytes;
  static constexpr size_t mixs_bytes = size_t(T) * MIX_LD * 4;
  static constexpr size_t ss = mixs + mixs_bytes;
  static constexpr size_t end = ss + size_t(T) * 4;
  // the GEMV partials of every warp reuse the fn_s / new_s region
  static constexpr size_t red_bytes = size_t(T / 4) * T * MIX * 4;
  static_assert(red_bytes <= fn_bytes + news_bytes, "reduction scratch must fit");
  static_assert(news % 16 == 0 && mixs % 16 == 0, "alignment");
};

template <int T>
__global__ void __launch_bounds__(T * 8) k_stage(const StageParams p) {
  constexpr int NT = T * 8;         // one thread per (token, fragment)
  constexpr int WARPS = NT / 32;
  constexpr int TT = T / 8;         // tokens per lane in phase B
  constexpr int KP = KW / WARPS;    // GEMV inputs per warp in phase B
  using L = StageLayout<T>;
  extern __shared__ __align__(16) unsigned char smem[];
  float *fn_s = reinterpret_cast<float *>(smem + L::fn);
  uint16_t *new_s = reinterpret_cast<uint16_t *>(smem + L::news);
  float *mix_s = reinterpret_cast<float *>(smem + L::mixs);
  float *ss_s = reinterpret_cast<float *>(smem + L::ss);

  const int tid = threadIdx.x;
  const int slice = blockIdx.x;
  const int h0 = slice * SLICE;
  const int t0 = blockIdx.y * T;
  const int H = p.hidden;

  // ---- stage hc_fn's slice as fn_s[output][k], k = stream * 64 + column
  for (int e = tid; e < KW * (MIX / 4); e += NT) {
    const int k = e / (MIX / 4), q = e % (MIX / 4);
    const int j = k / SLICE, col = k % SLICE;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (h0 + col < H)
      v = *reinterpret_cast<const float4 *>(p.hc_fn + ((size_t)j * H + h0 + col) * MIX + q * 4);
    fn_s[(q * 4 + 0) * FN_LD + k] = v.x;
    fn_s[(q * 4 + 1) * FN_LD + k] = v.y;
    fn_s[(q * 4 + 2) * FN_LD + k] = v.z;
    fn_s[(q * 4 + 3) * FN_LD + k] = v.w;
  }
  // ---- per-token post [4] and comb [source][target] [16]
  for (int e = tid; e < T * MIX_LD; e += NT) {
    const int tl = e / MIX_LD, c = e % MIX_LD, t = t0 + tl;
    float v = 0.f;
    if (t < p.m) v = c < HC ? p.post[(size_t)t * HC + c] : p.comb[(size_t)t * HC * HC + (c - HC)];
    mix_s[e] = v;
  }
  __syncthreads();

  // ---- phase A: one thread per (token, fragment of 8 columns)
  const int tl = tid >> 3, f = tid & 7;
  const int t = t0 + tl;
  const int h = h0 + f * VEC;
  const bool act = (t < p.m) && (h < H);
  uint4 nv[HC] = {};
  float ss = 0.f;
  if (act) {
    float y[8];
    // stage 1: acc = +0, then + rank 0, + rank 1, ... (one FP32 add each)
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = 0.f;
    for (int r = 0; r < p.tp; ++r) {
      float x[8];
      unpack8(ld_stream(p.partials + ((size_t)r * p.m + t) * H + h), x);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = __fadd_rn(y[e], x[e]);
    }
    const uint4 yb = round8(y);
    if (p.reduced_out) st_vec(p.reduced_out + (size_t)t * H + h, yb);

    // post-mix: new_j = bf16(y * post_j + sum_k res_k * comb[k][j]), the k
    // terms in source order as fused multiply-adds
    float res[HC][8];
#pragma unroll
    for (int k = 0; k < HC; ++k) unpack8(ld_stream(p.residual + ((size_t)t * HC + k) * H + h), res[k]);
    const float *mx = mix_s + tl * MIX_LD;
#pragma unroll
    for (int j = 0; j < HC; ++j) {
      const float pj = mx[j];
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float v = __fmul_rn(y[e], pj);
#pragma unroll
        for (int k = 0; k < HC; ++k) v = __fmaf_rn(res[k][e], mx[HC + k * HC + j], v);
        o[e] = v;
      }
      nv[j] = round8(o);
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(o[e], o[e], ss);
      st_vec(p.residual_out + ((size_t)t * HC + j) * H + h, nv[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < HC; ++j)
    *reinterpret_cast<uint4 *>(new_s + tl * NEW_LD + j * SLICE + f * VEC) = nv[j];
  // the 8 fragments of a token are 8 consecutive lanes
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);
  ss += __shfl_xor_sync(0xffffffffu, ss, 4);
  if (f == 0) ss_s[tl] = ss;
  __syncthreads();

  // ---- phase B: lane (g, q) accumulates outputs 6g..6g+5 for tokens
  // q, q+8, ... over this warp's range of the 256 GEMV inputs
  const int warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 3, q = lane & 7;
  float acc[TT][6];
#pragma unroll
  for (int a = 0; a < TT; ++a)
#pragma unroll
    for (int i = 0; i < 6; ++i) acc[a][i] = 0.f;
  const int kbeg = warp * KP;
#pragma unroll 2
  for (int k = kbeg; k < kbeg + KP; k += 8) {
    float x[TT][8];
#pragma unroll
    for (int a = 0; a < TT; ++a)
      unpack8(*reinterpret_cast<const uint4 *>(new_s + (q + 8 * a) * NEW_LD + k), x[a]);
#pragma unroll
    for (int i = 0; i < 6; ++i) {
      const float4 w0 = *reinterpret_cast<const float4 *>(fn_s + (6 * g + i) * FN_LD + k);
      const float4 w1 = *reinterpret_cast<const float4 *>(fn_s + (6 * g + i) * FN_LD + k + 4);
#pragma unroll
      for (int a = 0; a < TT; ++a) {
        float s = acc[a][i];
        s = fmaf(x[a][0], w0.x, s);
        s = fmaf(x[a][1], w0.y, s);
        s = fmaf(x[a][2], w0.z, s);
        s = fmaf(x[a][3], w0.w, s);
        s = fmaf(x[a][4], w1.x, s);
        s = fmaf(x[a][5], w1.y, s);
        s = fmaf(x[a][6], w1.z, s);
        s = fmaf(x[a][7], w1.w, s);
        acc[a][i] = s;
      }
    }
  }
  __syncthreads();  // fn_s / new_s are free from here on
  float *red_s = fn_s;  // [WARPS][T][MIX]
#pragma unroll
  for (int a = 0; a < TT; ++a)
#pragma unroll
    for (int i = 0; i < 6; ++i) red_s[(warp * T + q + 8 * a) * MIX + 6 * g + i] = acc[a][i];
  __syncthreads();
  for (int e = tid; e < T * VALUES; e += NT) {
    const int tl2 = e / VALUES, v = e % VALUES, tok = t0 + tl2;
    if (tok >= p.m) continue;
    float s;
    if (v < MIX) {
      s = 0.f;
#pragma unroll
      for (int w = 0; w < WARPS; ++w) s += red_s[(w * T + tl2) * MIX + v];
    } else {
      s = ss_s[tl2];
    }
    p.part[(size_t)tok * p.part_stride + slice * VALUES + v] = s;
  }
}

template <int T>
cudaError_t launch_t(const StageParams &p, cudaStream_t stream) {
  const dim3 grid(p.slices, (p.m + T - 1) / T);
  k_stage<T><<<grid, T * 8, stage_smem_bytes(T), stream>>>(p);
  return cudaGetLastError();
}

template <int T>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(k_stage<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(STAGE_SMEM_LIMIT));
}

}  // namespace

int stage_tile_tokens(int m) {
  // Small calls spread their tokens over more CTAs; large calls take 32
  // tokens per CTA so that each staged hc_fn slice serves more tokens.
  if (m <= 64) return 8;
  if (m <= 256) return 16;
  return 32;
}

size_t stage_smem_bytes(int tile_tokens) {
  switch (tile_tokens) {
    case 8: return StageLayout<8>::end;
    case 16: return StageLayout<16>::end;
    default: return StageLayout<32>::end;
  }
}

cudaError_t stage_set_attributes() {
  cudaError_t e;
  if ((e = set_attr<8>()) != cudaSuccess) return e;
  if ((e = set_attr<16>()) != cudaSuccess) return e;
  return set_attr<32>();
}

cudaError_t launch_stage(const StageParams &p, cudaStream_t stream) {
  switch (stage_tile_tokens(p.m)) {
    case 8: return launch_t<8>(p, stream);
    case 16: return launch_t<16>(p, stream);
    default: return launch_t<32>(p, stream);
  }
}

}  // namespace mhc
