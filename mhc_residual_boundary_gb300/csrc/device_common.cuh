// device_common.cuh -- device helpers shared by the boundary kernels:
// BF16 packing (hardware round-to-nearest-even conversions), vector loads
// and stores with cache hints, warp reductions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "launch.cuh"

namespace mhc {

// ---------------------------------------------------------------- BF16
// A BF16 value is the upper half of the FP32 with the same bits.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two FP32 values to a BF16 pair, nearest-even (lo in bits 0..15).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void unpack8(const uint4 &v, float (&x)[8]) {
  x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x);
  x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
  x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z);
  x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
  return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                    pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
}

// Rounds eight FP32 values to BF16 in place (the value a BF16 store keeps).
__device__ __forceinline__ uint4 round8(float (&x)[8]) {
  uint4 p = pack8(x);
  unpack8(p, x);
  return p;
}

// ------------------------------------------------------------- memory
// Streaming read of data used once: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Read-only 16-byte read, cached in L1 (data no kernel of the call writes
// and the CTA re-reads, such as a weight).  Not ordered after the thread's
// own earlier stores, so independent reads issue back to back.
__device__ __forceinline__ uint4 ld_ro(const void *p) {
  uint4 v;
  asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Plain 16-byte read through L1 (data other threads of the CTA re-read).
__device__ __forceinline__ uint4 ld_vec(const void *p) {
  return *reinterpret_cast<const uint4 *>(p);
}

__device__ __forceinline__ void st_vec(void *p, const uint4 &v) {
  *reinterpret_cast<uint4 *>(p) = v;
}

// ----------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Programmatic dependent launch: wait until the preceding kernel on the
// stream has completed and its memory is visible (a no-op without PDL).
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next kernel on the stream start its launch early.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace mhc
