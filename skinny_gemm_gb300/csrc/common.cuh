// common.cuh -- device helpers shared by the W4A16 kernels (not by the oracle).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace w4a16 {

constexpr int kGroup = 64;  // codes per (row, group) scale/bias pair

// bf16 bit patterns <-> fp32.  Widening is exact: the bf16 bits are the high
// half of the fp32 pattern.
__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// fp32 -> bf16, IEEE round to nearest even (CUDA intrinsic).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Streaming 16-byte load of packed weights: read-only path, no L1
// allocation (each byte is used once), 256-byte L2 prefetch granularity.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Read-only 16-byte load that may stay in L1 (activations, reused by rows).
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint16_t ld_nc_u16(const uint16_t* p) {
  unsigned short v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// Code j (0..7) of a packed word as an exact fp32, without a variable shift.
// The masked nibble sits inside the mantissa of 2^23; one FMA removes the
// 2^23 offset and the nibble's place value 16^(j%4) at once, exactly, because
// (2^23 + q*16^i) * 16^-i - 2^(23-4i) = q has an exact intermediate.  This
// is the "read packed int4 values through a 16-bit mask, avoiding a shift
// for every weight" idea of tiny-llm "Week 2 Day 2: Keep W4 Packed",
// section "Stage 2: SIMD Matvec", applied to the weights instead of
// pre-scaling the activations.
template <int I>
__device__ __forceinline__ float nibble_in_half(uint32_t half16) {
  constexpr uint32_t mask = 0xFu << (4 * I);
  constexpr float inv = 1.0f / (float)(1u << (4 * I));
  constexpr float off = -8388608.0f / (float)(1u << (4 * I));
  return __fmaf_rn(__uint_as_float((half16 & mask) | 0x4B000000u), inv, off);
}

__device__ __forceinline__ void unpack8_f32(uint32_t w, float q[8]) {
  const uint32_t hi = w >> 16;
  q[0] = nibble_in_half<0>(w);
  q[1] = nibble_in_half<1>(w);
  q[2] = nibble_in_half<2>(w);
  q[3] = nibble_in_half<3>(w);
  q[4] = nibble_in_half<0>(hi);
  q[5] = nibble_in_half<1>(hi);
  q[6] = nibble_in_half<2>(hi);
  q[7] = nibble_in_half<3>(hi);
}

// Eight bf16 activations (one 16-byte chunk) widened to fp32.
__device__ __forceinline__ void widen8(const uint4& v, float f[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

}  // namespace w4a16
