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
// Thread mapping: NL = g/16 lanes per group of g values (4 lanes for g = 64,
// a quarter warp for 128, half a warp for 256); lane q of the group holds 16
// values in two halves of 8 consecutive elements, half h being elements
// [8 NL h + 8q, 8 NL h + 8q + 8), so that every warp-wide access to a half
// covers 32/NL contiguous runs, one per group, with 16- or 32-byte accesses
// per lane.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace echo {

constexpr unsigned kFull = 0xFFFFFFFFu;

// NaN-propagating min / max (PTX min.NaN / max.NaN).  For finite and infinite
// values they equal fminf / fmaxf; a NaN anywhere in a group makes its range,
// hence its step, NaN, which flags the group (see make_grid).
__device__ __forceinline__ float min_nan(float a, float b) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Three-input forms (one instruction on the sm_100 family).
__device__ __forceinline__ float min3_nan(float a, float b, float c) {
  float r;
  asm("min.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// The largest of three, NaN operands ignored (NaN only if all three are).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Butterfly over the NL lanes of a group (aligned lane blocks of NL).
template <int NL>
__device__ __forceinline__ float group_min(float x) {
#pragma unroll
  for (int off = NL / 2; off > 0; off >>= 1) x = min_nan(x, __shfl_xor_sync(kFull, x, off));
  return x;
}
template <int NL>
__device__ __forceinline__ float group_max(float x) {
#pragma unroll
  for (int off = NL / 2; off > 0; off >>= 1) x = max_nan(x, __shfl_xor_sync(kFull, x, off));
  return x;
}

// Zero-aware range of a group over its NL lanes (all 32 lanes must call it;
// each block of NL lanes reduces its own group).
#ifndef ECHO_RANGE3
#define ECHO_RANGE3 1
#endif
template <int NL>
__device__ __forceinline__ void group_range(const float v[16], float& lo, float& hi) {
#if !ECHO_RANGE3
  float a2[4], b2[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    a2[k] = min_nan(min_nan(v[4 * k], v[4 * k + 1]), min_nan(v[4 * k + 2], v[4 * k + 3]));
    b2[k] = max_nan(max_nan(v[4 * k], v[4 * k + 1]), max_nan(v[4 * k + 2], v[4 * k + 3]));
  }
  lo = group_min<NL>(min_nan(min_nan(min_nan(a2[0], a2[1]), min_nan(a2[2], a2[3])), 0.0f));
  hi = group_max<NL>(max_nan(max_nan(max_nan(b2[0], b2[1]), max_nan(b2[2], b2[3])), 0.0f));
  return;
#endif
  // 16 values and 0 in 8 three-input steps each (two independent chains).
  float a = min3_nan(v[0], v[1], 0.0f), c = min3_nan(v[2], v[3], v[4]);
  float b = max3_nan(v[0], v[1], 0.0f), d = max3_nan(v[2], v[3], v[4]);
  a = min3_nan(a, v[5], v[6]);   c = min3_nan(c, v[7], v[8]);
  b = max3_nan(b, v[5], v[6]);   d = max3_nan(d, v[7], v[8]);
  a = min3_nan(a, v[9], v[10]);  c = min3_nan(c, v[11], v[12]);
  b = max3_nan(b, v[9], v[10]);  d = max3_nan(d, v[11], v[12]);
  lo = group_min<NL>(min3_nan(a, c, min_nan(v[13], min_nan(v[14], v[15]))));
  hi = group_max<NL>(max3_nan(b, d, max_nan(v[13], max_nan(v[14], v[15]))));
}

struct GroupGrid {
  float s;        // step (an fp16 value)
  float inv;      // 1/s rounded to nearest (fast path of v/s, see encode)
  float zf;       // zero point as a float (an integer value)
  uint32_t meta;  // fp16 step bits | fp16 zero-point bits << 16
  bool finite;    // false: non-finite input or step overflow; results unspecified
};

// ------------------------------------------------------------- pairs ----
// Elementwise fp32 add / sub / mul / fma on pairs of values.  Each half is
// rounded to nearest exactly as by __fadd_rn / __fsub_rn / __fmul_rn /
// __fmaf_rn (IEEE, subnormals kept); the sm_100 family issues one packed
// f32x2 instruction per pair, half the instructions of the scalar form.
#ifndef ECHO_F32X2
#define ECHO_F32X2 1
#endif

#if ECHO_F32X2
#define ECHO_PAIR_OP(NAME, OP)                                                              \
  __device__ __forceinline__ void NAME(float& r0, float& r1, float a0, float a1, float b0,  \
                                       float b1) {                                          \
    asm("{\n\t.reg .b64 pa, pb, pr;\n\t"                                                   \
        "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t" OP                             \
        " pr, pa, pb;\n\tmov.b64 {%0, %1}, pr;\n\t}"                                        \
        : "=f"(r0), "=f"(r1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));                        \
  }
ECHO_PAIR_OP(add2, "add.rn.f32x2")
ECHO_PAIR_OP(sub2, "sub.rn.f32x2")
ECHO_PAIR_OP(mul2, "mul.rn.f32x2")
#undef ECHO_PAIR_OP
__device__ __forceinline__ void fma2(float& r0, float& r1, float a0, float a1, float b0, float b1,
                                     float c0, float c1) {
  asm("{\n\t.reg .b64 pa, pb, pc, pr;\n\t"
      "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\tmov.b64 pc, {%6, %7};\n\t"
      "fma.rn.f32x2 pr, pa, pb, pc;\n\tmov.b64 {%0, %1}, pr;\n\t}"
      : "=f"(r0), "=f"(r1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
#else
__device__ __forceinline__ void add2(float& r0, float& r1, float a0, float a1, float b0, float b1) {
  r0 = __fadd_rn(a0, b0); r1 = __fadd_rn(a1, b1);
}
__device__ __forceinline__ void sub2(float& r0, float& r1, float a0, float a1, float b0, float b1) {
  r0 = __fsub_rn(a0, b0); r1 = __fsub_rn(a1, b1);
}
__device__ __forceinline__ void mul2(float& r0, float& r1, float a0, float a1, float b0, float b1) {
  r0 = __fmul_rn(a0, b0); r1 = __fmul_rn(a1, b1);
}
__device__ __forceinline__ void fma2(float& r0, float& r1, float a0, float a1, float b0, float b1,
                                     float c0, float c1) {
  r0 = __fmaf_rn(a0, b0, c0); r1 = __fmaf_rn(a1, b1, c1);
}
#endif

// Arrays of N (even) values: r = a + b, r = a - b, r = a * b, r = a * s.
template <int N>
__device__ __forceinline__ void add_n(float* r, const float* a, const float* b) {
#pragma unroll
  for (int k = 0; k < N; k += 2) add2(r[k], r[k + 1], a[k], a[k + 1], b[k], b[k + 1]);
}
template <int N>
__device__ __forceinline__ void sub_n(float* r, const float* a, const float* b) {
#pragma unroll
  for (int k = 0; k < N; k += 2) sub2(r[k], r[k + 1], a[k], a[k + 1], b[k], b[k + 1]);
}
template <int N>
__device__ __forceinline__ void mul_ns(float* r, const float* a, float s) {
#pragma unroll
  for (int k = 0; k < N; k += 2) mul2(r[k], r[k + 1], a[k], a[k + 1], s, s);
}

// rint(t) for |t| < 2^22 with two fp32 adds: at 1.5 * 2^23 the fp32 spacing
// is 1, so the first add rounds t to an integer (to nearest, ties to even)
// and the second removes the offset exactly.  Runs on the FMA pipe.
__device__ __forceinline__ float rint_small(float t) {
  return __fsub_rn(__fadd_rn(t, 12582912.0f), 12582912.0f);
}

// Largest distance from an integer at which rint(x * (1/s)) is taken as
// rint(x / s).  For a finite group |x / s| < 256, so the correctly rounded
// reciprocal and product are within 256 * 3 * 2^-24 < 2^-13 of the correctly
// rounded quotient; when the product lies farther than that from every
// half-integer, both round to the same integer.  Otherwise the quotient itself
// is computed (IEEE division).
constexpr float kFastRintLimit = 0.5f - 1.0f / 8192.0f;

// Step and zero point of a group from its range.
__device__ __forceinline__ GroupGrid make_grid(float lo, float hi, float L) {
  const float s32 = __fdiv_rn(__fsub_rn(hi, lo), L);
  __half sh = __float2half_ru(s32);
  float s = __half2float(sh);
  if (s == 0.0f) {
    sh = __ushort_as_half((unsigned short)0x3C00);  // 1.0
    s = 1.0f;
  }
  const float inv = __frcp_rn(s);
  // z = rint(-lo / s); -lo / s lies in [0, L(1 + 2^-22)] for a finite group.
  const float t = __fmul_rn(-lo, inv);
  float zf = rint_small(t);
  if (!(fabsf(__fsub_rn(t, zf)) < kFastRintLimit)) zf = rintf(__fdiv_rn(-lo, s));
  zf = fminf(fmaxf(zf, 0.0f), L);
  GroupGrid gg;
  gg.s = s;
  gg.inv = inv;
  gg.zf = zf;
  gg.meta = (uint32_t)__half_as_ushort(sh) |
            ((uint32_t)__half_as_ushort(__float2half_rn(zf)) << 16);
  gg.finite = isfinite(s);
  return gg;
}

// Codes (as integer-valued floats in [0, L]) and decoded values of 8 values:
// c = clamp(rint(v / s) + z, 0, L), d = (c - z) * s.
//
// rint(v / s) comes from the product with the reciprocal unless some value of
// the 8 lies near a rounding boundary, in which case all 8 are recomputed with
// IEEE division.  Only the upper clamp is applied: for a finite group v >= lo,
// so rint(fl(v / s)) >= rint(fl(lo / s)) = -z (division and rint are monotonic
// and odd-symmetric), and c >= 0 already.  (For a non-finite group the codes
// are unspecified; pack8 still confines each packed word to its own bytes.)
//
// Since r and z are small integers, clamp(r + z, L) - z = min(r, L - z)
// exactly: the clamped offset cm = q - z gives both c = cm + z and d = cm * s.
__device__ __forceinline__ void quantize8(const float v[8], const GroupGrid& gg, float L,
                                          float c[8], float d[8]) {
  constexpr float M = 12582912.0f;                 // 1.5 * 2^23, see rint_small
  float t[8], r[8], e[8];
  mul_ns<8>(t, v, gg.inv);
#pragma unroll
  for (int k = 0; k < 8; k += 2) {
    add2(r[k], r[k + 1], t[k], t[k + 1], M, M);
    sub2(r[k], r[k + 1], r[k], r[k + 1], M, M);
  }
  sub_n<8>(e, t, r);
  // max |e| (NaN operands ignored, as by fmaxf), three at a time
  float dev = max3(fabsf(e[0]), fabsf(e[1]), fabsf(e[2]));
  dev = max3(dev, fabsf(e[3]), fabsf(e[4]));
  dev = max3(dev, fabsf(e[5]), fabsf(e[6]));
  dev = fmaxf(dev, fabsf(e[7]));
  if (dev >= kFastRintLimit) {
    // (+ 0 turns a -0 from rintf into +0, as the fast path gives, so that
    // cm * s below is +0 where (q - z) * s is.)
#pragma unroll
    for (int k = 0; k < 8; ++k) r[k] = __fadd_rn(rintf(__fdiv_rn(v[k], gg.s)), 0.0f);
  }
  const float lz = __fsub_rn(L, gg.zf);            // exact
  float cm[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) cm[k] = fminf(r[k], lz);
#pragma unroll
  for (int k = 0; k < 8; k += 2) add2(c[k], c[k + 1], cm[k], cm[k + 1], gg.zf, gg.zf);
  mul_ns<8>(d, cm, gg.s);
}

// Quantizer variants: the method's zero-aware asymmetric quantizer and the two
// ablations of Table 8.  Readings of the unprinted formulas:
//   kNaiveZeroPoint  range [min v, max v] without 0; offset m = fp16 rounding
//                    of min v toward -inf, carried in the meta word's zero-point
//                    half; s = (max v - m) / (2^b - 1) rounded up to fp16;
//                    q = clamp(rint((v - m) / s), 0, 2^b - 1); decoded m + s*q.
//   kSymmetric       s = max|v| / (2^(b-1) - 1) rounded up to fp16; zero point
//                    2^(b-1); q = clamp(rint(v / s), +-(2^(b-1) - 1)) + 2^(b-1).
enum QuantMode : int { kZeroAware = 0, kNaiveZeroPoint = 1, kSymmetric = 2 };

// The grid of one group held by NL lanes (16 values per lane); every lane of
// the warp must call it.  For kNaiveZeroPoint, zf holds the offset m.
template <int MODE, int NL>
__device__ __forceinline__ GroupGrid group_grid(const float v[16], float L) {
  if constexpr (MODE == kZeroAware) {
    float lo, hi;
    group_range<NL>(v, lo, hi);
    return make_grid(lo, hi, L);
  } else if constexpr (MODE == kSymmetric) {
    float a = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k) a = max_nan(a, fabsf(v[k]));
    a = group_max<NL>(a);
    const float zf = __fadd_rn(__fmul_rn(L, 0.5f), 0.5f);   // 2^(b-1), exact
    __half sh = __float2half_ru(__fdiv_rn(a, __fsub_rn(zf, 1.0f)));
    float s = __half2float(sh);
    if (s == 0.0f) {
      sh = __ushort_as_half((unsigned short)0x3C00);
      s = 1.0f;
    }
    GroupGrid gg;
    gg.s = s;
    gg.inv = __frcp_rn(s);
    gg.zf = zf;
    gg.meta = (uint32_t)__half_as_ushort(sh) | ((uint32_t)__half_as_ushort(__float2half_rn(zf)) << 16);
    gg.finite = isfinite(s);
    return gg;
  } else {
    float lo = v[0], hi = v[0];
#pragma unroll
    for (int k = 1; k < 16; ++k) {
      lo = min_nan(lo, v[k]);
      hi = max_nan(hi, v[k]);
    }
    lo = group_min<NL>(lo);
    hi = group_max<NL>(hi);
    const __half mh = __float2half_rd(lo);
    const float m = __half2float(mh);
    __half sh = __float2half_ru(__fdiv_rn(__fsub_rn(hi, m), L));
    float s = __half2float(sh);
    if (s == 0.0f) {
      sh = __ushort_as_half((unsigned short)0x3C00);
      s = 1.0f;
    }
    GroupGrid gg;
    gg.s = s;
    gg.inv = __frcp_rn(s);
    gg.zf = m;
    gg.meta = (uint32_t)__half_as_ushort(sh) | ((uint32_t)__half_as_ushort(mh) << 16);
    gg.finite = isfinite(s) && isfinite(m);
    return gg;
  }
}

// Codes (integer-valued floats) and decoded values of 8 values in any mode.
// The quotient is rint(x / s) with x = v (or v - m for the naive offset),
// taken through the reciprocal as in quantize8; |x / s| < 256 in every mode.
template <int MODE>
__device__ __forceinline__ void quantize8_mode(const float v[8], const GroupGrid& gg, float L,
                                               float c[8], float d[8]) {
  if constexpr (MODE == kZeroAware) {
    quantize8(v, gg, L, c, d);
  } else {
    float x[8], r[8];
    float dev = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      x[k] = MODE == kNaiveZeroPoint ? __fsub_rn(v[k], gg.zf) : v[k];
      const float t = __fmul_rn(x[k], gg.inv);
      r[k] = rint_small(t);
      dev = fmaxf(dev, fabsf(__fsub_rn(t, r[k])));
    }
    if (dev >= kFastRintLimit) {
#pragma unroll
      for (int k = 0; k < 8; ++k) r[k] = rintf(__fdiv_rn(x[k], gg.s));
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if constexpr (MODE == kSymmetric) {
        const float lh = __fsub_rn(gg.zf, 1.0f);
        c[k] = __fadd_rn(fminf(fmaxf(r[k], -lh), lh), gg.zf);
        d[k] = __fmul_rn(__fsub_rn(c[k], gg.zf), gg.s);
      } else {
        c[k] = fminf(fmaxf(r[k], 0.0f), L);
        d[k] = __fadd_rn(__fmul_rn(c[k], gg.s), gg.zf);   // m + s*q
      }
    }
  }
}

// Meta word -> (step, zero point as float).
__device__ __forceinline__ void unpack_meta(uint32_t meta, float& s, float& zf) {
  s = __half2float(__ushort_as_half((unsigned short)(meta & 0xFFFFu)));
  zf = __half2float(__ushort_as_half((unsigned short)(meta >> 16)));
}

// Packing of 4 consecutive codes.  4-bit: element 2i in the low nibble of
// byte i, so 4 codes form one little-endian 16-bit word; 8-bit: one byte
// each, one 32-bit word.  The codes are integer-valued floats, so the word is
// built with exact fp arithmetic (every intermediate is an integer below
// 2^16) and read out of the mantissa of 2^23 + word.  Two runs of 4 (c[0..3]
// into w0, c[4..7] into w1) at once, on pairs.
template <int BITS>
__device__ __forceinline__ void pack8(const float c[8], uint32_t& w0, uint32_t& w1) {
  constexpr float B = 8388608.0f;                  // 2^23
  float a0, a1;
  if (BITS == 4) {
    fma2(a0, a1, c[1], c[5], 16.0f, 16.0f, c[0], c[4]);
    fma2(a0, a1, c[2], c[6], 256.0f, 256.0f, a0, a1);
    fma2(a0, a1, c[3], c[7], 4096.0f, 4096.0f, a0, a1);
    add2(a0, a1, a0, a1, B, B);
    w0 = __float_as_uint(a0) & 0xFFFFu;
    w1 = __float_as_uint(a1) & 0xFFFFu;
  } else {
    float b0, b1;
    fma2(a0, a1, c[1], c[5], 256.0f, 256.0f, c[0], c[4]);   // bytes 0, 1
    fma2(b0, b1, c[3], c[7], 256.0f, 256.0f, c[2], c[6]);   // bytes 2, 3
    add2(a0, a1, a0, a1, B, B);
    add2(b0, b1, b0, b1, B, B);
    w0 = __byte_perm(__float_as_uint(a0), __float_as_uint(b0), 0x5410);
    w1 = __byte_perm(__float_as_uint(a1), __float_as_uint(b1), 0x5410);
  }
}

// Decoding of a packed chunk word: (q - z) * s for its 4 codes.  The code is
// turned into a float exactly by placing it in the mantissa of 2^23.
template <int BITS>
__device__ __forceinline__ void decode4(uint32_t w, float s, float zf, float d[4]) {
  constexpr uint32_t MASK = (1u << BITS) - 1;
  const float bias = __fadd_rn(8388608.0f, zf);   // 2^23 + z, exact
  float q23[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) q23[k] = __uint_as_float(0x4B000000u | ((w >> (BITS * k)) & MASK));
#pragma unroll
  for (int k = 0; k < 4; k += 2) {
    sub2(d[k], d[k + 1], q23[k], q23[k + 1], bias, bias);   // q - z exact
    mul2(d[k], d[k + 1], d[k], d[k + 1], s, s);
  }
}

// Decoding in any mode: s * (q - z), or m + s * q for the naive offset
// (zf then holds m).
template <int BITS, int MODE>
__device__ __forceinline__ void decode4_mode(uint32_t w, float s, float zf, float d[4]) {
  if constexpr (MODE != kNaiveZeroPoint) {
    decode4<BITS>(w, s, zf, d);
  } else {
    constexpr uint32_t MASK = (1u << BITS) - 1;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float q = __fsub_rn(__uint_as_float(0x4B000000u | ((w >> (BITS * k)) & MASK)), 8388608.0f);
      d[k] = __fadd_rn(__fmul_rn(q, s), zf);
    }
  }
}

// bf16 <-> f32 for 8 values held in 16 bytes.
__device__ __forceinline__ void bf16x8_to_f32(uint4 r, float f[8]) {
  f[0] = __uint_as_float(r.x << 16); f[1] = __uint_as_float(r.x & 0xFFFF0000u);
  f[2] = __uint_as_float(r.y << 16); f[3] = __uint_as_float(r.y & 0xFFFF0000u);
  f[4] = __uint_as_float(r.z << 16); f[5] = __uint_as_float(r.z & 0xFFFF0000u);
  f[6] = __uint_as_float(r.w << 16); f[7] = __uint_as_float(r.w & 0xFFFF0000u);
}

// The entry pass of 8 values: v[k] = float(x_k) + e[k] for 8 bf16 values in
// 16 bytes and their fp32 held errors, one IEEE fp32 add each (the bf16 value
// widens exactly).  With ECHO_MIXED_ADD (the default) the sm_100 family's
// mixed-precision add (add.rn.f32.bf16) takes the bf16 half of a register as
// it is, with no separate widening instruction: 2 instructions per pair
// instead of 3 (measured +0.9% on a call with 2-byte state, +0.1% with fp32
// state); 0 widens the values and adds them in pairs.
#ifndef ECHO_MIXED_ADD
#define ECHO_MIXED_ADD 1
#endif
__device__ __forceinline__ float add_bf16_f32(uint32_t w, int half, float e) {
  float r;
  if (half == 0)
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.bf16 %0, lo, %2;\n\t}"
        : "=f"(r) : "r"(w), "f"(e));
  else
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.bf16 %0, hi, %2;\n\t}"
        : "=f"(r) : "r"(w), "f"(e));
  return r;
}

__device__ __forceinline__ void entry8(uint4 x, const float e[8], float v[8]) {
#if ECHO_MIXED_ADD
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[2 * k] = add_bf16_f32(w[k], 0, e[2 * k]);
    v[2 * k + 1] = add_bf16_f32(w[k], 1, e[2 * k + 1]);
  }
#else
  bf16x8_to_f32(x, v);
  add_n<8>(v, v, e);
#endif
}

// 8 values rounded to bf16 (nearest even) two at a time, packed into 16 bytes
// (element 2k in the low half of word k), with the rounded values widened
// back to fp32 exactly in `back`.
__device__ __forceinline__ uint4 f32x8_to_bf16(const float f[8], float back[8]) {
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);
    w[k] = *reinterpret_cast<const uint32_t*>(&h);
    back[2 * k] = __uint_as_float(w[k] << 16);
    back[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Storage of the compensator state: none (uncompensated), fp32, or bf16 or
// fp16 (each rounded to nearest even).  Element i of rank p lives at p*n + i
// in every format.
enum StateFmt : int { kNoState = 0, kStateF32 = 1, kStateBF16 = 2, kStateF16 = 3 };

// The state format of a call: its comp pointer and the plan's format code
// (0 fp32, 1 bf16, 2 fp16).
__host__ __device__ inline int state_fmt_of(const void* comp, int code) {
  return comp == nullptr ? kNoState : code == 1 ? kStateBF16 : code == 2 ? kStateF16 : kStateF32;
}

template <int SF>
constexpr int state_bytes() { return SF == kStateF32 ? 4 : (SF == kNoState ? 0 : 2); }

// The 8 state values of a half at element index i (a multiple of 8) of a
// stage in shared memory, as fp32 (exact for both formats).
template <int SF>
__device__ __forceinline__ void state_load8(const uint8_t* base, int i, float e[8]) {
  if constexpr (SF == kStateF32) {
    const float4 a = *reinterpret_cast<const float4*>(base + 4 * i);
    const float4 b = *reinterpret_cast<const float4*>(base + 4 * i + 16);
    e[0] = a.x; e[1] = a.y; e[2] = a.z; e[3] = a.w;
    e[4] = b.x; e[5] = b.y; e[6] = b.z; e[7] = b.w;
  } else if constexpr (SF == kStateBF16) {
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(base + 2 * i), e);
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(base + 2 * i);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[k]));
      e[2 * k] = f.x;
      e[2 * k + 1] = f.y;
    }
  }
}

// Keeps the revealed errors r of a half in global memory at element index i
// (a multiple of 8; the state buffer is 32-byte aligned): decay * r, stored
// as fp32 (one 32-byte store) or rounded to bf16 or fp16 (one 16-byte
// store).  With DECAY false the multiply is skipped, for decay 1: r * 1 is r
// itself for every value (a NaN from the subtraction is already the
// canonical one a multiply would give).
template <int SF, bool DECAY = true>
__device__ __forceinline__ void state_store8(uint8_t* base, int64_t i, const float r[8],
                                             float decay) {
  float t[8];
  if constexpr (DECAY) {
    mul_ns<8>(t, r, decay);
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) t[k] = r[k];
  }
  if constexpr (SF == kStateF32) {
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :: "l"(base + 4 * i), "f"(t[0]), "f"(t[1]), "f"(t[2]), "f"(t[3]), "f"(t[4]),
                    "f"(t[5]), "f"(t[6]), "f"(t[7]) : "memory");
  } else if constexpr (SF == kStateBF16) {
    float back[8];
    *reinterpret_cast<uint4*>(base + 2 * i) = f32x8_to_bf16(t, back);
  } else {
    uint32_t u[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 h = __floats2half2_rn(t[2 * k], t[2 * k + 1]);
      u[k] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(base + 2 * i) = make_uint4(u[0], u[1], u[2], u[3]);
  }
}

// Element offset, within a group, of half h (0, 1) of lane q (0..NL-1) of the
// group's NL lanes.
template <int NL>
__device__ __forceinline__ int half_at(int h, int q) { return 8 * NL * h + 8 * q; }

// Byte offset, within a group's packed codes, of half h of lane q: 8 codes of
// BITS bits each, stored contiguously (4 or 8 bytes).
template <int BITS, int NL>
__device__ __forceinline__ int half_code_byte(int h, int q) { return half_at<NL>(h, q) * BITS / 8; }

}  // namespace echo
