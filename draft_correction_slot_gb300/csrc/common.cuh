// common.cuh -- device helpers shared by the library's kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define DC_FULL_MASK 0xffffffffu

namespace dc {

// Device error bits, OR-ed into the handle's device status word.
enum : int {
  kErrBadCandidateId = 1,   // a gathered token id was outside [0, V)
  kErrTimeout = 2,          // a bounded wait inside a kernel expired
};

// ---- bf16 bit helpers ------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}
// fp32 -> bf16 bits, round to nearest even.
__device__ __forceinline__ uint32_t bf16_rn_bits(float f) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Order-preserving 16-bit key of a bf16 value: larger key <=> larger value.
// -0 is folded onto +0 first so the two compare equal.
__device__ __forceinline__ uint32_t bf16_order_key(uint32_t bits16) {
  bits16 &= 0xFFFFu;
  if (bits16 == 0x8000u) bits16 = 0u;
  return (bits16 & 0x8000u) ? (~bits16 & 0xFFFFu) : (bits16 | 0x8000u);
}

// Inverse of bf16_order_key (for keys of real values).
__device__ __forceinline__ float order_key_to_float(uint32_t key) {
  uint32_t bits = (key & 0x8000u) ? (key & 0x7FFFu) : (~key & 0xFFFFu);
  return bf16_bits_to_float(bits);
}

// Streaming 16-byte load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Packed bf16x2 maximum (one instruction on sm_90+).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(DC_FULL_MASK, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(DC_FULL_MASK, v, o));
  return v;
}

// Programmatic dependent launch.  pdl_trigger lets the next kernel in the
// stream be scheduled; pdl_wait blocks until the previous kernel has finished
// and its memory operations are visible (a no-op without a programmatic
// dependency).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace dc
