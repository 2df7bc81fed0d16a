// quant.cuh -- device-side primitives of the zero-aware asymmetric group
// quantizer ("Echo: Error-Compensated 4-Bit Tensor-Parallel Communication",
// Table 8 "zero-aware asymmetric, g=128"; transport of b-bit integers with one
// fp16 step and one fp16 zero point per group, article "Your All-Reduce Is 4x
// Overpriced", section "The cancellation rule").
//
// Reading of the unprinted formula: lo = min(0, min v), hi = max(0, max v);
// s = (hi - lo) / (2^b - 1) rounded up to fp16 (1 for an all-zero group);
// z = clamp(rint(-lo / s), 0, 2^b - 1); q = clamp(rint(v / s) + z, 0, 2^b - 1);
// decoded value s * (q - z).  Each step is one IEEE fp32 operation with
// explicit round-to-nearest intrinsics, so no multiply-add is ever fused.
//
// One warp handles one group of 128 values, 4 consecutive values per lane.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace echo {

constexpr unsigned kFull = 0xFFFFFFFFu;

struct GroupGrid {
  float s;        // step (an fp16 value)
  float zf;       // zero point as a float (an integer value)
  int z;          // zero point
  uint32_t meta;  // fp16 step bits | fp16 zero-point bits << 16
  bool finite;    // false when the step overflowed fp16 (or the range was NaN)
};

// Warp-wide zero-aware range: every lane passes its 4 values, all lanes get
// (lo, hi) with lo <= 0 <= hi.
__device__ __forceinline__ void warp_range(const float v[4], float& lo, float& hi) {
  lo = fminf(fminf(fminf(0.0f, v[0]), fminf(v[1], v[2])), v[3]);
  hi = fmaxf(fmaxf(fmaxf(0.0f, v[0]), fmaxf(v[1], v[2])), v[3]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(kFull, lo, off));
    hi = fmaxf(hi, __shfl_xor_sync(kFull, hi, off));
  }
}

// Step and zero point of a group from its range.
__device__ __forceinline__ GroupGrid make_grid(float lo, float hi, float L) {
  const float s32 = __fdiv_rn(__fsub_rn(hi, lo), L);
  __half sh = __float2half_ru(s32);
  float s = __half2float(sh);
  if (s == 0.0f) {
    sh = __ushort_as_half((unsigned short)0x3C00);  // 1.0
    s = 1.0f;
  }
  float zf = rintf(__fdiv_rn(-lo, s));
  zf = fminf(fmaxf(zf, 0.0f), L);
  GroupGrid gg;
  gg.z = (int)zf;
  gg.zf = (float)gg.z;
  gg.s = s;
  gg.meta = (uint32_t)__half_as_ushort(sh) |
            ((uint32_t)__half_as_ushort(__int2half_rn(gg.z)) << 16);
  gg.finite = isfinite(s);
  return gg;
}

__device__ __forceinline__ int encode(float v, const GroupGrid& gg, float L) {
  float c = __fadd_rn(rintf(__fdiv_rn(v, gg.s)), gg.zf);
  c = fminf(fmaxf(c, 0.0f), L);
  return (int)c;
}

// s * (q - z): an integer difference, an exact conversion, one multiply.
__device__ __forceinline__ float decode(int q, int z, float s) {
  return __fmul_rn((float)(q - z), s);
}

// Meta word -> (step, zero point).
__device__ __forceinline__ void unpack_meta(uint32_t meta, float& s, int& z) {
  s = __half2float(__ushort_as_half((unsigned short)(meta & 0xFFFFu)));
  z = (int)__half2float(__ushort_as_half((unsigned short)(meta >> 16)));
}

// 4 codes of one lane <-> its slice of the packed group.  4-bit: element 2i in
// the low nibble of byte i, so 4 consecutive codes form one little-endian
// 16-bit word; 8-bit: one byte each, one 32-bit word.
template <int BITS>
__device__ __forceinline__ uint32_t pack4(const int q[4]) {
  if (BITS == 4) {
    return (uint32_t)q[0] | ((uint32_t)q[1] << 4) | ((uint32_t)q[2] << 8) | ((uint32_t)q[3] << 12);
  } else {
    return (uint32_t)q[0] | ((uint32_t)q[1] << 8) | ((uint32_t)q[2] << 16) | ((uint32_t)q[3] << 24);
  }
}

template <int BITS>
__device__ __forceinline__ void unpack4(uint32_t w, int q[4]) {
  constexpr int SH = BITS;
  constexpr uint32_t MASK = (1u << BITS) - 1;
#pragma unroll
  for (int k = 0; k < 4; ++k) q[k] = (int)((w >> (SH * k)) & MASK);
}

// 4 bf16 values in 8 bytes <-> floats.
__device__ __forceinline__ void bf16x4_to_f32(uint2 r, float f[4]) {
  f[0] = __uint_as_float(r.x << 16);
  f[1] = __uint_as_float(r.x & 0xFFFF0000u);
  f[2] = __uint_as_float(r.y << 16);
  f[3] = __uint_as_float(r.y & 0xFFFF0000u);
}

__device__ __forceinline__ uint2 f32x4_to_bf16(const float f[4], float back[4]) {
  const __nv_bfloat16 b0 = __float2bfloat16_rn(f[0]);
  const __nv_bfloat16 b1 = __float2bfloat16_rn(f[1]);
  const __nv_bfloat16 b2 = __float2bfloat16_rn(f[2]);
  const __nv_bfloat16 b3 = __float2bfloat16_rn(f[3]);
  back[0] = __bfloat162float(b0);
  back[1] = __bfloat162float(b1);
  back[2] = __bfloat162float(b2);
  back[3] = __bfloat162float(b3);
  uint2 r;
  r.x = (uint32_t)__bfloat16_as_ushort(b0) | ((uint32_t)__bfloat16_as_ushort(b1) << 16);
  r.y = (uint32_t)__bfloat16_as_ushort(b2) | ((uint32_t)__bfloat16_as_ushort(b3) << 16);
  return r;
}

__device__ __forceinline__ bool all_finite4(const float v[4]) {
  return isfinite(v[0]) && isfinite(v[1]) && isfinite(v[2]) && isfinite(v[3]);
}

}  // namespace echo
