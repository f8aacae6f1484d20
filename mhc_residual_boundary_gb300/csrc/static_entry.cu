// static_entry.cu -- mhc_boundary_run_static: one boundary call that
// allocates nothing.
//
// Some callers cannot allocate device memory when they need a boundary: a
// framework whose caching allocator already owns the device memory budget,
// code that must not trigger the implicit device synchronisation a
// cudaMalloc / cudaFree can cause, or a host thread that may not create a
// handle (mhc_boundary_create allocates its scratch, a side stream and
// events).  This entry point runs the stage kernel, the finish kernel and the
// separate post / Sinkhorn kernel, all on the caller's stream, with their
// scratch (the per-group GEMV partial sums and the raw mixes) in a
// fixed-size array of this library's device memory instead of memory a
// handle allocated.
//
// The array and the error word are file-scope __device__ variables: every
// GPU that loads this library holds STATIC_SCRATCH_BYTES of them until the
// process exits.  In host code their names are only host-side stand-ins,
// never device addresses, so the host asks the runtime for the device
// addresses (cudaGetSymbolAddress) once per device, with that device
// current, and passes those pointers to the kernels.
#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "launch.cuh"
#include "mhc_boundary.h"

using namespace mhc;

namespace {

// Scratch of every call: [m] rows of partial sums ([slices][25] padded to a
// multiple of 4 floats), then [m][24] mixes.
constexpr size_t STATIC_SCRATCH_BYTES = size_t(8) << 20;   // 8 MiB per device
static __device__ __align__(256) float g_scratch[STATIC_SCRATCH_BYTES / sizeof(float)];
// Error word of the allocation-free calls: bit 1 is set by a stage or finish
// kernel whose bounded wait gave up (its outputs are then invalid).  It stays
// set until a call with MHC_FLAG_CHECK_ERRORS reads and clears it.
static __device__ unsigned int g_static_err;

constexpr int MAX_DEVICES = 64;
std::mutex g_setup_mutex;
std::atomic<float *> g_scratch_ptr[MAX_DEVICES];
unsigned int *g_err_ptr[MAX_DEVICES];
int g_sm_count[MAX_DEVICES];

mhc_status_t report(char *error, size_t error_len, mhc_status_t status, const char *fmt, ...) {
  if (error && error_len) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(error, error_len, fmt, ap);
    va_end(ap);
  }
  return status;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device addresses of g_scratch and g_static_err on the current device,
// looked up once per device; the first call on a device also raises the
// stage kernels' shared memory limits there and reads its SM count.
mhc_status_t scratch_on_device(int device, float **out, unsigned int **err, char *error, size_t error_len) {
  if (device < 0 || device >= MAX_DEVICES)
    return report(error, error_len, MHC_ERR_UNSUPPORTED, "device %d is beyond the %d devices supported",
                  device, MAX_DEVICES);
  float *ptr = g_scratch_ptr[device].load(std::memory_order_acquire);
  if (!ptr) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    ptr = g_scratch_ptr[device].load(std::memory_order_relaxed);
    if (!ptr) {
      void *addr = nullptr, *err_addr = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&addr, g_scratch);
      if (e == cudaSuccess) e = cudaGetSymbolAddress(&err_addr, g_static_err);
      if (e == cudaSuccess) e = stage_set_attributes();
      if (e == cudaSuccess) e = stage_tc_set_attributes();
      if (e == cudaSuccess) e = finish_set_attributes();
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_sm_count[device], cudaDevAttrMultiProcessorCount, device);
      if (e != cudaSuccess)
        return report(error, error_len, MHC_ERR_CUDA, "set-up on device %d: %s", device, cudaGetErrorString(e));
      ptr = static_cast<float *>(addr);
      g_err_ptr[device] = static_cast<unsigned int *>(err_addr);
      g_scratch_ptr[device].store(ptr, std::memory_order_release);
    }
  }
  *out = ptr;
  *err = g_err_ptr[device];
  return MHC_OK;
}

}  // namespace

extern "C" mhc_status_t mhc_boundary_run_static(const mhc_boundary_config_t *config, const mhc_run_args_t *a,
                                                mhc_stream_t stream_, char *error, size_t error_len) {
  if (error && error_len) error[0] = '\0';
  if (!config || !a) return report(error, error_len, MHC_ERR_INVALID_ARG, "config and args are required");
  const mhc_boundary_config_t &c = *config;
  if (c.hc_mult != HC) return report(error, error_len, MHC_ERR_UNSUPPORTED, "hc_mult must be 4");
  if (c.hidden <= 0 || c.hidden % VEC)
    return report(error, error_len, MHC_ERR_INVALID_ARG, "hidden must be a positive multiple of 8");
  if (c.hidden > MAX_HIDDEN) return report(error, error_len, MHC_ERR_UNSUPPORTED, "hidden > %d", MAX_HIDDEN);
  if (c.tp < 1 || c.tp > 32) return report(error, error_len, MHC_ERR_INVALID_ARG, "tp must be in [1, 32]");
  if (c.sinkhorn_repeat < 1 || c.sinkhorn_repeat > 10000)
    return report(error, error_len, MHC_ERR_INVALID_ARG, "sinkhorn_repeat must be in [1, 10000]");
  if (c.flags & ~uint32_t(MHC_FLAG_MXFP8 | MHC_FLAG_SYNC_MIXES | MHC_FLAG_STATIC_WEIGHT | MHC_FLAG_CHECK_ERRORS))
    return report(error, error_len, MHC_ERR_UNSUPPORTED,
                  "only MHC_FLAG_MXFP8, MHC_FLAG_SYNC_MIXES, MHC_FLAG_STATIC_WEIGHT and MHC_FLAG_CHECK_ERRORS apply");
  if ((c.flags & MHC_FLAG_MXFP8) && c.hidden % 128)
    return report(error, error_len, MHC_ERR_INVALID_ARG, "MXFP8 output needs hidden %% 128 == 0");

  const int slices = (c.hidden + SLICE - 1) / SLICE;
  const size_t per_token = size_t(part_row_floats(slices)) + MIX;    // floats
  // the mixes start at a 64-float boundary after the partial sums
  const size_t max_m = (STATIC_SCRATCH_BYTES / sizeof(float) - 64) / per_token;
  if (a->m < 1 || size_t(a->m) > max_m)
    return report(error, error_len, MHC_ERR_CAPACITY,
                  "M=%d is outside [1, %zu]: the static scratch (%zu bytes) holds %zu floats per token at hidden=%d",
                  a->m, max_m, STATIC_SCRATCH_BYTES, per_token, c.hidden);
  struct Need { const void *p; const char *name; size_t align; };
  const Need required[] = {
      {a->partials, "partials", 16}, {a->residual, "residual", 16}, {a->post, "post", 16},
      {a->comb, "comb", 16}, {a->scale, "scale", 4}, {a->base, "base", 4},
      {a->norm_weight, "norm_weight", 16}, {a->residual_out, "residual_out", 16},
      {a->layer_input, "layer_input", 16}, {a->post_out, "post_out", 4}, {a->comb_out, "comb_out", 4}};
  for (const Need &n : required) {
    if (!n.p) return report(error, error_len, MHC_ERR_INVALID_ARG, "%s is NULL", n.name);
    if (!aligned(n.p, n.align))
      return report(error, error_len, MHC_ERR_INVALID_ARG, "%s is not %zu-byte aligned", n.name, n.align);
  }
  const Need optional[] = {{a->pre_out, "pre_out", 4}, {a->mixes_out, "mixes_out", 4},
                           {a->reduced_out, "reduced_out", 16}, {a->mxfp8_values, "mxfp8_values", 16},
                           {a->mxfp8_scales, "mxfp8_scales", 16}};
  for (const Need &n : optional)
    if (n.p && !aligned(n.p, n.align))
      return report(error, error_len, MHC_ERR_INVALID_ARG, "%s is not %zu-byte aligned", n.name, n.align);
  if ((a->mxfp8_values == nullptr) != (a->mxfp8_scales == nullptr))
    return report(error, error_len, MHC_ERR_INVALID_ARG, "mxfp8_values and mxfp8_scales go together");
  if ((a->hc_fn == nullptr) == (a->hc_fn_bf16 == nullptr))
    return report(error, error_len, MHC_ERR_INVALID_ARG, "exactly one of hc_fn and hc_fn_bf16 is required");
  if (!aligned(a->hc_fn ? static_cast<const void *>(a->hc_fn) : a->hc_fn_bf16, 16))
    return report(error, error_len, MHC_ERR_INVALID_ARG, "the prenorm weight is not 16-byte aligned");
  if (a->hc_fn_bf16 && c.tp > TP_TMA_MAX)
    return report(error, error_len, MHC_ERR_UNSUPPORTED, "hc_fn_bf16 needs tp <= %d", TP_TMA_MAX);
  if (a->mxfp8_values && !(c.flags & MHC_FLAG_MXFP8))
    return report(error, error_len, MHC_ERR_UNSUPPORTED, "MXFP8 outputs need MHC_FLAG_MXFP8");

  int device = -1;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return report(error, error_len, MHC_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  float *scratch = nullptr;
  unsigned int *err = nullptr;
  const mhc_status_t s = scratch_on_device(device, &scratch, &err, error, error_len);
  if (s != MHC_OK) return s;
  // every scratch word a kernel reads was written earlier in the same call,
  // so nothing needs clearing between calls (the error word is cleared only
  // when it is read, below)
  float *part = scratch;
  // the tensor-core stage kernel writes one partial group per 128 columns,
  // the CUDA-core one per 64; the capacity rule above counts the latter
  const bool tc_path = c.tp <= TP_TMA_MAX;
  const int groups = tc_path ? (c.hidden + TC_GROUP_COLS - 1) / TC_GROUP_COLS : slices;
  float *mixes = scratch + (size_t(a->m) * part_row_floats(groups) + 63) / 64 * 64;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  StageParams sp = {};
  sp.m = a->m;
  sp.hidden = c.hidden;
  sp.tp = c.tp;
  sp.slices = groups;
  sp.partials = static_cast<const uint16_t *>(a->partials);
  sp.residual = static_cast<const uint16_t *>(a->residual);
  sp.post = a->post;
  sp.comb = a->comb;
  sp.hc_fn = a->hc_fn;
  sp.hc_fn_bf16 = static_cast<const uint16_t *>(a->hc_fn_bf16);
  sp.fn_terms = a->hc_fn_bf16 ? 1 : 3;
  sp.early_weight = (c.flags & MHC_FLAG_STATIC_WEIGHT) != 0;
  sp.residual_out = static_cast<uint16_t *>(a->residual_out);
  sp.reduced_out = static_cast<uint16_t *>(a->reduced_out);
  sp.part = part;
  sp.part_stride = part_row_floats(groups);
  sp.err = err;   // a stage-kernel wait that gives up sets bit 1
  int stage_grid = 0;
  e = tc_path ? launch_stage_tc(sp, g_sm_count[device], stream, &stage_grid) : launch_stage(sp, stream);
  if (e != cudaSuccess) return report(error, error_len, MHC_ERR_CUDA, "stage kernel: %s", cudaGetErrorString(e));

  FinishParams fp = {};
  fp.m = a->m;
  fp.hidden = c.hidden;
  fp.slices = groups;
  fp.part = part;
  fp.part_stride = sp.part_stride;
  fp.scale = a->scale;
  fp.base = a->base;
  fp.gamma = static_cast<const uint16_t *>(a->norm_weight);
  fp.streams = static_cast<const uint16_t *>(a->residual_out);
  fp.rms_eps = c.rms_eps;
  fp.hc_eps = c.hc_eps;
  fp.norm_eps = c.norm_eps;
  fp.err = err;
  fp.mixes = mixes;
  fp.mixes_out = a->mixes_out;
  fp.pre_out = a->pre_out;
  fp.layer_input = static_cast<uint16_t *>(a->layer_input);
  fp.mx_values = a->mxfp8_values;
  fp.mx_scales = a->mxfp8_scales;
  e = launch_finish(fp, g_sm_count[device], stream, true, stage_grid);
  if (e != cudaSuccess) return report(error, error_len, MHC_ERR_CUDA, "finish kernel: %s", cudaGetErrorString(e));

  MixesParams mp = {};
  mp.m = a->m;
  mp.repeat = c.sinkhorn_repeat;
  mp.mixes = mixes;
  mp.scale = a->scale;
  mp.base = a->base;
  mp.post_mult = c.post_mult;
  mp.eps = c.hc_eps;
  mp.post_out = a->post_out;
  mp.comb_out = a->comb_out;
  e = launch_mixes(mp, stream);
  if (e != cudaSuccess) return report(error, error_len, MHC_ERR_CUDA, "mixes kernel: %s", cudaGetErrorString(e));
  if (!(c.flags & MHC_FLAG_CHECK_ERRORS)) return MHC_OK;

  // the caller asked for the kernels' own failure reports: wait for this call
  // and read (then clear) the error word of this and earlier calls
  unsigned int word = 0;
  e = cudaMemcpyAsync(&word, err, sizeof word, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess && word) e = cudaMemsetAsync(err, 0, sizeof word, stream);
  if (e == cudaSuccess && word) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return report(error, error_len, MHC_ERR_CUDA, "error check: %s", cudaGetErrorString(e));
  if (word & 2u)
    return report(error, error_len, MHC_ERR_TIMEOUT,
                  "a kernel gave up one of its bounded waits; the outputs of the call that set it are not valid");
  return MHC_OK;
}
