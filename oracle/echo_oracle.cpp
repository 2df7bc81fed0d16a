// echo_oracle.cpp -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, single-threaded CPU restatement of the per-call arithmetic of
// Echo, the error-compensated 4-bit tensor-parallel all-reduce described in
// "Echo: Error-Compensated 4-Bit Tensor-Parallel Communication for LLM Training
// and Inference" (arXiv 2610.14277) and in the article "Your All-Reduce Is 4x
// Overpriced: Echo's 4-Bit Error-Feedback Trick for Tensor-Parallel Training".
//
// It exists so that the GPU library can be checked against something obviously
// correct.  Only the test suite, the smoke check and the bench's CPU-baseline
// leg load it.  It shares no source, header, table or helper with the GPU
// library, and it never reads anything the GPU library produced.
//
// Numerics: every floating-point step is a single IEEE-754 binary32 operation
// rounded to nearest-even.  The file is compiled with -O2 -ffp-contract=off so
// that no multiply and add are fused.  Conversions to binary16 and bfloat16 are
// written below from the definitions of those formats, not taken from a library.
//
// Where the pages leave a step open, the reading taken here is stated at the
// step (the quantizer formula itself, "Eqn. (8)" in the paper's appendix, is not
// printed on the pages):
//   * quantizer: zero-aware asymmetric min/max quantizer with an integer zero
//     point; the range [lo, hi] is widened to contain 0 so that 0 is encoded
//     exactly (Table 8 row "zero-aware asymmetric, g=128", against the ablation
//     rows "naive zero-point" and "symmetric grid");
//   * per-group parameters in half precision: an fp16 scale and an fp16 zero
//     point, 4 bytes per group (article, section "The cancellation rule": 4-bit
//     integers with half-precision quantization parameters per group);
//   * the scale is rounded toward +infinity to fp16, so that no code is clamped
//     by more than half a step; an all-zero group gets scale 1;
//   * codes are rint (half-to-even) of v/s plus the zero point, clamped to
//     [0, 2^b - 1];
//   * the two quantizers of the ablation in Table 8 (their formulas are not
//     printed either) are read as: "naive zero-point" -- range [min v, max v]
//     without 0, a float offset m (fp16, rounded down from min v) stored where
//     the zero point goes, codes rint((v - m)/s), decoded m + s*q, so 0 is in
//     general not exactly representable; "symmetric grid" -- s from max|v| over
//     2^(b-1) - 1 levels, a fixed zero point 2^(b-1), codes rint(v/s) + 2^(b-1);
//   * options of the compensator (the pages print none of its constants): the
//     held error may be stored in bf16 (rounded to nearest even) instead of
//     fp32, and it may be decayed, e' = decay * (revealed error), before it is
//     stored; decay 1 with fp32 storage is the plain error feedback above;
//   * owner segments are contiguous: rank o owns elements [o*m, (o+1)*m) with
//     m = n/P; groups are consecutive runs of g elements inside a segment, the
//     last one shorter when g does not divide m (Fig. 2(a), Fig. 4);
//   * the owner's high-precision sum is an fp32 sum in ascending rank order,
//     starting from rank 0's term (Fig. 2(a): "sums them ... in high precision");
//   * compensator: full error feedback, each error held where it is revealed.
//     A sender keeps, for each element it quantized for the push, the stage-1
//     error v - deq(q); the owner keeps, for each element of its segment, the
//     stage-2 error sum - bf16 output.  The next call adds the held error to the
//     input before quantizing (the "entry pass"); the update itself does not
//     change the values computed by the call (article, "The cancellation rule";
//     paper abstract: "the summation reveals each injected error, and Echo feeds
//     it back into later calls").
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

uint32_t f32_bits(float x) {
  uint32_t u;
  std::memcpy(&u, &x, 4);
  return u;
}

float bits_f32(uint32_t u) {
  float x;
  std::memcpy(&x, &u, 4);
  return x;
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// Number formats.
// ---------------------------------------------------------------------------

// IEEE 754 binary16 -> binary32 (exact).
float oracle_f16_to_f32(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int ex = (h >> 10) & 0x1F;
  const int man = h & 0x3FF;
  float mag;
  if (ex == 0) {
    mag = std::ldexp((float)man, -24);                 // subnormal: man * 2^-24
  } else if (ex == 31) {
    mag = man ? NAN : INFINITY;
  } else {
    mag = std::ldexp((float)(1024 + man), ex - 25);    // (1.man) * 2^(ex-15)
  }
  return sign ? -mag : mag;
}

// binary32 -> binary16, rounding toward +infinity.
// The magnitude is first truncated to the binary16 grid, remembering whether
// any bits were dropped; a positive inexact value then moves one binary16 step
// up, a negative one keeps the truncated magnitude (which is the larger value).
uint16_t oracle_f32_to_f16_ru(float x) {
  const uint32_t u = f32_bits(x);
  const uint16_t sign = (uint16_t)((u >> 16) & 0x8000);
  const uint32_t a = u & 0x7FFFFFFF;
  const int ex32 = (int)(a >> 23);
  const uint32_t man32 = a & 0x7FFFFF;
  if (ex32 == 0xFF) {                          // inf or NaN
    return (uint16_t)(sign | (man32 ? 0x7E00 : 0x7C00));
  }
  uint16_t trunc;   // binary16 magnitude bits, rounded toward zero
  bool inexact;
  if (ex32 == 0) {                             // binary32 zero or subnormal: below 2^-126
    trunc = 0;
    inexact = man32 != 0;
  } else {
    const int e = ex32 - 127;                  // unbiased exponent
    const uint32_t M = (1u << 23) | man32;     // 24-bit significand, value M * 2^(e-23)
    if (e > 15) {                              // at least 2^16: beyond the largest finite
      trunc = 0x7BFF;                          // 65504
      inexact = true;
    } else if (e >= -14) {                     // binary16 normal range
      trunc = (uint16_t)(((e + 15) << 10) | (man32 >> 13));
      inexact = (man32 & 0x1FFF) != 0;
    } else {                                   // binary16 subnormal: units of 2^-24
      const int shift = -(e + 1);              // value / 2^-24 = M * 2^(e+1)
      if (shift >= 32) {
        trunc = 0;
        inexact = true;
      } else {
        trunc = (uint16_t)(M >> shift);
        inexact = (M & ((1u << shift) - 1)) != 0;
      }
    }
  }
  if (sign) {
    return (uint16_t)(sign | trunc);           // toward +inf = toward zero for negatives
  }
  return (uint16_t)(trunc + (inexact ? 1 : 0));  // 0x7BFF + 1 carries into +inf
}

float oracle_bf16_to_f32(uint16_t b) { return bits_f32((uint32_t)b << 16); }

// binary32 -> bfloat16, round to nearest, ties to even.
uint16_t oracle_f32_to_bf16_rn(float x) {
  const uint32_t u = f32_bits(x);
  if ((u & 0x7FFFFFFF) > 0x7F800000) {         // NaN: keep sign, force quiet
    return (uint16_t)((u >> 16) | 0x0040);
  }
  const uint32_t kept_lsb = (u >> 16) & 1;
  return (uint16_t)((u + 0x7FFF + kept_lsb) >> 16);
}

// Element-wise array forms of the conversions above.
void oracle_f32_to_f16_ru_n(const float* x, int64_t count, uint16_t* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = oracle_f32_to_f16_ru(x[i]);
}

void oracle_f16_to_f32_n(const uint16_t* h, int64_t count, float* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = oracle_f16_to_f32(h[i]);
}

void oracle_f32_to_bf16_rn_n(const float* x, int64_t count, uint16_t* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = oracle_f32_to_bf16_rn(x[i]);
}

// binary32 -> binary16, rounding toward -infinity: the negation of rounding
// the negated value toward +infinity.
uint16_t oracle_f32_to_f16_rd(float x) {
  return (uint16_t)(oracle_f32_to_f16_ru(-x) ^ 0x8000);
}

void oracle_f32_to_f16_rd_n(const float* x, int64_t count, uint16_t* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = oracle_f32_to_f16_rd(x[i]);
}

// binary32 -> binary16, round to nearest, ties to even: whichever of the two
// directed roundings lies nearer to x (distances compared exactly in double,
// where every binary16 and binary32 value and their differences here are
// exact); on a tie, the one whose last significand bit is 0.  Beyond the
// largest finite value the next step up is taken to be 2^16 (as IEEE rounding
// does), so x >= 65520 rounds to infinity.  NaN stays NaN.
uint16_t oracle_f32_to_f16_rn(float x) {
  const uint16_t up = oracle_f32_to_f16_ru(x);
  if (x != x) return up;
  const uint16_t dn = oracle_f32_to_f16_rd(x);
  if (up == dn) return up;
  const double xd = (double)x;
  const double vu = up == 0x7C00 ? 65536.0 : (double)oracle_f16_to_f32(up);
  const double vd = dn == 0xFC00 ? -65536.0 : (double)oracle_f16_to_f32(dn);
  const double du = vu - xd, dd = xd - vd;
  if (du < dd) return up;
  if (dd < du) return dn;
  return (up & 1) == 0 ? up : dn;
}

void oracle_f32_to_f16_rn_n(const float* x, int64_t count, uint16_t* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = oracle_f32_to_f16_rn(x[i]);
}

// Quantizer variants (a mode argument where the functions take one).
enum { kZeroAware = 0, kNaiveZeroPoint = 1, kSymmetric = 2 };

// ---------------------------------------------------------------------------
// The quantizer Q_b on one group of `len` fp32 values.
//
// Returns 1 when the group holds a non-finite value or its scale does not fit
// fp16 (the results are then unspecified), else 0.  Writes the codes q[i] in
// [0, 2^b-1], the fp16 scale bits and the fp16 zero-point bits.  When `ties`
// is not NULL, adds the number of exact rounding ties met: each rint whose
// fp32 argument lies exactly on a half-integer (both neighbours equally near,
// settled half-to-even), whether that argument is negative or positive and
// whether or not the code is clamped afterwards.
// ---------------------------------------------------------------------------
static int quantize_naive(const float* v, int len, int bits, uint8_t* q, uint16_t* s_bits,
                          uint16_t* z_bits, int64_t* ties);
static int quantize_symmetric(const float* v, int len, int bits, uint8_t* q, uint16_t* s_bits,
                              uint16_t* z_bits, int64_t* ties);

int oracle_quantize_group(const float* v, int len, int bits, uint8_t* q,
                          uint16_t* s_bits, uint16_t* z_bits,
                          int64_t* ties) {
  const int L = (1 << bits) - 1;
  const float Lf = (float)L;
  int bad = 0;

  // Step 1: the zero-aware range always contains 0.
  float lo = 0.0f, hi = 0.0f;
  for (int i = 0; i < len; ++i) {
    if (!std::isfinite(v[i])) bad = 1;
    lo = std::fmin(lo, v[i]);
    hi = std::fmax(hi, v[i]);
  }

  // Steps 2-3: step size, rounded up to fp16; an all-zero group gets 1.
  const float s32 = (hi - lo) / Lf;
  uint16_t sb = oracle_f32_to_f16_ru(s32);
  float s = oracle_f16_to_f32(sb);
  if (s == 0.0f) {
    sb = 0x3C00;
    s = 1.0f;
  }
  if (!std::isfinite(s)) bad = 1;

  // Step 4: integer zero point, the code that decodes to exactly 0.  Its
  // rint is a rounding decision like a code's, so an exact tie here counts too.
  const float rz = -lo / s;
  if (ties && std::isfinite(rz) && (rz - std::floor(rz)) == 0.5f) ++*ties;
  float zf = std::rint(rz);
  zf = std::fmin(std::fmax(zf, 0.0f), Lf);
  const int z = (int)zf;

  // Step 5: codes.
  for (int i = 0; i < len; ++i) {
    const float r = v[i] / s;
    if (ties && std::isfinite(r) && (r - std::floor(r)) == 0.5f) ++*ties;
    float c = std::rint(r) + (float)z;
    c = std::fmin(std::fmax(c, 0.0f), Lf);
    q[i] = (uint8_t)(int)c;
  }
  *s_bits = sb;
  *z_bits = oracle_f32_to_f16_ru((float)z);    // exact: a small integer
  return bad;
}

// Step 6: deq(q) = s * (q - z): integer difference, exact conversion, one multiply.
void oracle_dequantize_group(const uint8_t* q, int len, uint16_t s_bits,
                             uint16_t z_bits, float* out) {
  const float s = oracle_f16_to_f32(s_bits);
  const int z = (int)oracle_f16_to_f32(z_bits);
  for (int i = 0; i < len; ++i) out[i] = (float)((int)q[i] - z) * s;
}

// Ablation "naive zero-point" (Table 8): the group's own range, no 0 in it; a
// float offset m = fp16 rounding of min v toward -inf, so that v - m >= 0; step
// (max v - m) / L rounded up to fp16; codes rint((v - m) / s) in [0, L].  The
// meta word carries m where the zero point otherwise goes.
static int quantize_naive(const float* v, int len, int bits, uint8_t* q, uint16_t* s_bits,
                          uint16_t* z_bits, int64_t* ties) {
  const float Lf = (float)((1 << bits) - 1);
  int bad = 0;
  float lo = INFINITY, hi = -INFINITY;
  for (int i = 0; i < len; ++i) {
    if (!std::isfinite(v[i])) bad = 1;
    lo = std::fmin(lo, v[i]);
    hi = std::fmax(hi, v[i]);
  }
  const uint16_t mb = oracle_f32_to_f16_rd(lo);
  const float m = oracle_f16_to_f32(mb);
  uint16_t sb = oracle_f32_to_f16_ru((hi - m) / Lf);
  float s = oracle_f16_to_f32(sb);
  if (s == 0.0f) {
    sb = 0x3C00;
    s = 1.0f;
  }
  if (!std::isfinite(s) || !std::isfinite(m)) bad = 1;
  for (int i = 0; i < len; ++i) {
    const float r = (v[i] - m) / s;
    if (ties && std::isfinite(r) && (r - std::floor(r)) == 0.5f) ++*ties;
    const float c = std::fmin(std::fmax(std::rint(r), 0.0f), Lf);
    q[i] = (uint8_t)(int)c;
  }
  *s_bits = sb;
  *z_bits = mb;
  return bad;
}

// Ablation "symmetric grid" (Table 8): step max|v| / (2^(b-1) - 1) rounded up
// to fp16, fixed zero point 2^(b-1), codes rint(v/s) clamped to
// [-(2^(b-1) - 1), 2^(b-1) - 1] plus the zero point; decoded as s * (q - z).
static int quantize_symmetric(const float* v, int len, int bits, uint8_t* q, uint16_t* s_bits,
                              uint16_t* z_bits, int64_t* ties) {
  const int half = 1 << (bits - 1);
  const float Lh = (float)(half - 1);
  int bad = 0;
  float a = 0.0f;
  for (int i = 0; i < len; ++i) {
    if (!std::isfinite(v[i])) bad = 1;
    a = std::fmax(a, std::fabs(v[i]));
  }
  uint16_t sb = oracle_f32_to_f16_ru(a / Lh);
  float s = oracle_f16_to_f32(sb);
  if (s == 0.0f) {
    sb = 0x3C00;
    s = 1.0f;
  }
  if (!std::isfinite(s)) bad = 1;
  for (int i = 0; i < len; ++i) {
    const float r = v[i] / s;
    if (ties && std::isfinite(r) && (r - std::floor(r)) == 0.5f) ++*ties;
    const float c = std::fmin(std::fmax(std::rint(r), -Lh), Lh) + (float)half;
    q[i] = (uint8_t)(int)c;
  }
  *s_bits = sb;
  *z_bits = oracle_f32_to_f16_ru((float)half);   // exact: a small integer
  return bad;
}

int oracle_quantize_group_mode(const float* v, int len, int bits, int mode, uint8_t* q,
                               uint16_t* s_bits, uint16_t* z_bits, int64_t* ties) {
  if (mode == kNaiveZeroPoint) return quantize_naive(v, len, bits, q, s_bits, z_bits, ties);
  if (mode == kSymmetric) return quantize_symmetric(v, len, bits, q, s_bits, z_bits, ties);
  return oracle_quantize_group(v, len, bits, q, s_bits, z_bits, ties);
}

// Decoding for any mode: s * (q - z), or m + s * q for the naive zero point
// (one multiply, then one add).
void oracle_dequantize_group_mode(const uint8_t* q, int len, int mode, uint16_t s_bits,
                                  uint16_t z_bits, float* out) {
  if (mode != kNaiveZeroPoint) {
    oracle_dequantize_group(q, len, s_bits, z_bits, out);
    return;
  }
  const float s = oracle_f16_to_f32(s_bits);
  const float m = oracle_f16_to_f32(z_bits);
  for (int i = 0; i < len; ++i) out[i] = (float)q[i] * s + m;
}

// Wire packing of codes.  b=4: element 2i in the low nibble of byte i, element
// 2i+1 in its high nibble (an odd count leaves the last high nibble 0).  b=8:
// one byte per element.
void oracle_pack_codes(const uint8_t* q, int64_t count, int bits, uint8_t* out) {
  if (bits == 8) {
    for (int64_t i = 0; i < count; ++i) out[i] = q[i];
    return;
  }
  for (int64_t i = 0; i < (count + 1) / 2; ++i) {
    const uint8_t lo = q[2 * i] & 0xF;
    const uint8_t hi = (2 * i + 1 < count) ? (q[2 * i + 1] & 0xF) : 0;
    out[i] = (uint8_t)(lo | (hi << 4));
  }
}

// ---------------------------------------------------------------------------
// One group position: the same `len` elements of all P ranks, in the segment
// owned by rank `o`.  Group positions are independent of one another, so a
// whole call is this function applied to every position (oracle_allreduce),
// and a sample of positions can be checked on its own.
//
//   x      [P][len]  bf16 bits of each rank's input
//   e      [P][len]  compensator state (updated in place), or NULL for an
//                    uncompensated call (no state is read or written)
//   y      [len]     bf16 bits of the value every rank receives
//   q1     [P][len]  stage-1 codes of each sender (row o untouched), or NULL
//   m1     [P]       stage-1 meta (fp16 s | fp16 z << 16) per sender, or NULL
//   q2     [len]     stage-2 codes, or NULL;  m2 [1] stage-2 meta, or NULL
//   acc    [len]     the owner's fp32 sum, or NULL
//   nq     [P][len]  number of quantizations each rank's contribution went
//                    through before reaching y, or NULL
//   ties   counter of exact rounding ties, or NULL: every rint of the two
//          quantizations whose fp32 argument is exactly k + 1/2 (a code's v/s,
//          or (v - m)/s for the naive zero point, and the zero-aware zero
//          point's -lo/s), counted before any clamp
// Returns the number of quantizations flagged non-finite (0 when all is fine).
// ---------------------------------------------------------------------------
// The value the state keeps for a revealed error r: decay * r (one fp32
// multiply), rounded to nearest-even bf16 or fp16 when the state is stored in
// that type (state_fmt 1 or 2; 0 is fp32).  The state array itself stays fp32
// (holding bf16 or fp16 values in those cases).
static float keep_error(float r, int state_fmt, float decay) {
  const float t = decay * r;
  if (state_fmt == 1) return oracle_bf16_to_f32(oracle_f32_to_bf16_rn(t));
  if (state_fmt == 2) return oracle_f16_to_f32(oracle_f32_to_f16_rn(t));
  return t;
}

int oracle_group_position_ex(int P, int o, int len, int bits, int mode, int state_fmt,
                             float decay, const uint16_t* x, float* e, uint16_t* y,
                             uint8_t* q1, uint32_t* m1, uint8_t* q2, uint32_t* m2,
                             float* acc_out, uint8_t* nq, int64_t* ties) {
  int bad = 0;
  std::vector<float> v(len), d((size_t)P * len), acc(len);
  std::vector<uint8_t> q(len);
  uint16_t sb, zb;
  if (nq) std::memset(nq, 0, (size_t)P * len);

  // Fig. 2(a), push: every rank other than the owner quantizes its copy of the
  // segment.  The entry pass first adds the error that rank holds.
  for (int p = 0; p < P; ++p) {
    if (p == o) continue;
    const uint16_t* xp = x + (size_t)p * len;
    float* ep = e ? e + (size_t)p * len : nullptr;
    for (int i = 0; i < len; ++i) {
      v[i] = ep ? oracle_bf16_to_f32(xp[i]) + ep[i] : oracle_bf16_to_f32(xp[i]);
    }
    bad += oracle_quantize_group_mode(v.data(), len, bits, mode, q.data(), &sb, &zb, ties);
    float* dp = d.data() + (size_t)p * len;
    oracle_dequantize_group_mode(q.data(), len, mode, sb, zb, dp);
    if (q1) std::memcpy(q1 + (size_t)p * len, q.data(), len);
    if (m1) m1[p] = (uint32_t)sb | ((uint32_t)zb << 16);
    if (nq) for (int i = 0; i < len; ++i) nq[(size_t)p * len + i] += 1;
    // The push reveals this rank's stage-1 error; the rank keeps it.
    if (ep) for (int i = 0; i < len; ++i) ep[i] = keep_error(v[i] - dp[i], state_fmt, decay);
  }

  // The owner's own copy is not quantized; its entry pass adds its held error.
  {
    const uint16_t* xo = x + (size_t)o * len;
    const float* eo = e ? e + (size_t)o * len : nullptr;
    float* dst = d.data() + (size_t)o * len;
    for (int i = 0; i < len; ++i) {
      dst[i] = eo ? oracle_bf16_to_f32(xo[i]) + eo[i] : oracle_bf16_to_f32(xo[i]);
    }
  }

  // Reduce: fp32 sum in ascending rank order, starting from rank 0's term.
  for (int i = 0; i < len; ++i) {
    float a = d[i];
    for (int p = 1; p < P; ++p) a = a + d[(size_t)p * len + i];
    acc[i] = a;
  }

  // Gather: the sum is quantized once; every rank decodes the same code.
  bad += oracle_quantize_group_mode(acc.data(), len, bits, mode, q.data(), &sb, &zb, ties);
  oracle_dequantize_group_mode(q.data(), len, mode, sb, zb, v.data());
  for (int i = 0; i < len; ++i) y[i] = oracle_f32_to_bf16_rn(v[i]);
  if (q2) std::memcpy(q2, q.data(), len);
  if (m2) m2[0] = (uint32_t)sb | ((uint32_t)zb << 16);
  if (nq) for (size_t k = 0; k < (size_t)P * len; ++k) nq[k] += 1;
  if (acc_out) std::memcpy(acc_out, acc.data(), sizeof(float) * len);

  // The owner keeps the stage-2 error, measured against what ranks receive.
  if (e) {
    float* eo = e + (size_t)o * len;
    for (int i = 0; i < len; ++i) eo[i] = keep_error(acc[i] - oracle_bf16_to_f32(y[i]), state_fmt, decay);
  }
  return bad;
}

int oracle_group_position_mode(int P, int o, int len, int bits, int mode, const uint16_t* x,
                               float* e, uint16_t* y, uint8_t* q1, uint32_t* m1,
                               uint8_t* q2, uint32_t* m2, float* acc_out,
                               uint8_t* nq, int64_t* ties) {
  return oracle_group_position_ex(P, o, len, bits, mode, 0, 1.0f, x, e, y, q1, m1, q2, m2,
                                  acc_out, nq, ties);
}

int oracle_group_position(int P, int o, int len, int bits, const uint16_t* x,
                          float* e, uint16_t* y, uint8_t* q1, uint32_t* m1,
                          uint8_t* q2, uint32_t* m2, float* acc_out,
                          uint8_t* nq, int64_t* ties) {
  return oracle_group_position_mode(P, o, len, bits, kZeroAware, x, e, y, q1, m1, q2, m2,
                                    acc_out, nq, ties);
}

// A list of independent group positions, each of `len` elements, processed one
// after the other by oracle_group_position.  Arrays are position-major:
//   owners [npos]; x [npos][P][len]; e [npos][P][len] or NULL; y [npos][len];
//   q1 [npos][P][len], m1 [npos][P], q2 [npos][len], m2 [npos] (each or NULL).
// Returns the number of flagged quantizations, or -1 for invalid arguments.
int64_t oracle_group_positions_ex(int P, int64_t npos, const int* owners, int len,
                                  int bits, int mode, int state_fmt, float decay,
                                  const uint16_t* x, float* e, uint16_t* y,
                                  uint8_t* q1, uint32_t* m1, uint8_t* q2,
                                  uint32_t* m2, int64_t* ties) {
  if (P < 1 || npos < 0 || len < 1 || (bits != 4 && bits != 8) || mode < 0 || mode > 2) return -1;
  const size_t blk = (size_t)P * len;
  int64_t bad = 0;
  for (int64_t k = 0; k < npos; ++k) {
    if (owners[k] < 0 || owners[k] >= P) return -1;
    bad += oracle_group_position_ex(P, owners[k], len, bits, mode, state_fmt, decay, x + k * blk,
                                      e ? e + k * blk : nullptr, y + k * len,
                                      q1 ? q1 + k * blk : nullptr, m1 ? m1 + k * P : nullptr,
                                      q2 ? q2 + k * len : nullptr, m2 ? m2 + k : nullptr,
                                      nullptr, nullptr, ties);
  }
  return bad;
}

int64_t oracle_group_positions_mode(int P, int64_t npos, const int* owners, int len,
                                    int bits, int mode, const uint16_t* x, float* e, uint16_t* y,
                                    uint8_t* q1, uint32_t* m1, uint8_t* q2,
                                    uint32_t* m2, int64_t* ties) {
  return oracle_group_positions_ex(P, npos, owners, len, bits, mode, 0, 1.0f, x, e, y, q1, m1,
                                   q2, m2, ties);
}

int64_t oracle_group_positions(int P, int64_t npos, const int* owners, int len,
                               int bits, const uint16_t* x, float* e, uint16_t* y,
                               uint8_t* q1, uint32_t* m1, uint8_t* q2,
                               uint32_t* m2, int64_t* ties) {
  return oracle_group_positions_mode(P, npos, owners, len, bits, kZeroAware, x, e, y, q1, m1,
                                     q2, m2, ties);
}

// ---------------------------------------------------------------------------
// One whole call over P ranks of n elements each (n a multiple of P; g need
// not divide m = n/P, the last group of a segment is then shorter).
//
//   x    [P][n] bf16 bits;  out [P][n] bf16 bits (every row equal)
//   e    [P][n] fp32 state, updated in place, or NULL (uncompensated)
//   q1   [P][n]        stage-1 code of element i sent by rank p (own segment
//                      entries 0), or NULL
//   m1   [P][P][Gs]    stage-1 meta of rank p for group j of segment o
//                      (entries with p == o are 0), or NULL; Gs = ceil(m/g)
//   q2   [n]           stage-2 codes, or NULL;  m2 [P][Gs] stage-2 meta, or NULL
//   acc  [n]           the owners' fp32 sums, or NULL
//   nq   [P][n]        quantization counts, or NULL
//   ties               exact-tie counter, or NULL
// Returns the number of flagged quantizations, or -1 for invalid arguments.
// ---------------------------------------------------------------------------
int64_t oracle_allreduce_ex(int P, int64_t n, int g, int bits, int mode, int state_fmt,
                            float decay, const uint16_t* x,
                            uint16_t* out, float* e, uint8_t* q1, uint32_t* m1,
                            uint8_t* q2, uint32_t* m2, float* acc, uint8_t* nq,
                            int64_t* ties) {
  if (P < 1 || n < 0 || g < 1 || (bits != 4 && bits != 8) || n % P != 0) return -1;
  if (mode < 0 || mode > 2) return -1;
  const int64_t m = n / P;
  const int64_t Gs = (m + g - 1) / g;
  if (q1) std::memset(q1, 0, (size_t)(P * n));
  if (m1) std::memset(m1, 0, sizeof(uint32_t) * (size_t)(P * P * Gs));

  std::vector<uint16_t> xg((size_t)P * g), yg(g);
  std::vector<float> eg((size_t)P * g), accg(g);
  std::vector<uint8_t> q1g((size_t)P * g), q2g(g), nqg((size_t)P * g);
  std::vector<uint32_t> m1g(P);
  int64_t bad = 0;

  for (int o = 0; o < P; ++o) {
    for (int64_t j = 0; j < Gs; ++j) {
      const int64_t start = o * m + j * g;
      const int len = (int)std::min<int64_t>(g, m - j * g);
      for (int p = 0; p < P; ++p) {
        for (int i = 0; i < len; ++i) {
          xg[(size_t)p * len + i] = x[p * n + start + i];
          if (e) eg[(size_t)p * len + i] = e[p * n + start + i];
        }
      }
      uint32_t m2g = 0;
      bad += oracle_group_position_ex(P, o, len, bits, mode, state_fmt, decay, xg.data(),
                                      e ? eg.data() : nullptr, yg.data(), q1g.data(), m1g.data(),
                                      q2g.data(), &m2g, accg.data(), nqg.data(), ties);
      for (int p = 0; p < P; ++p) {
        for (int i = 0; i < len; ++i) {
          out[p * n + start + i] = yg[i];
          if (e) e[p * n + start + i] = eg[(size_t)p * len + i];
          if (nq) nq[p * n + start + i] = nqg[(size_t)p * len + i];
          if (q1 && p != o) q1[p * n + start + i] = q1g[(size_t)p * len + i];
        }
        if (m1 && p != o) m1[((int64_t)p * P + o) * Gs + j] = m1g[p];
      }
      for (int i = 0; i < len; ++i) {
        if (q2) q2[start + i] = q2g[i];
        if (acc) acc[start + i] = accg[i];
      }
      if (m2) m2[o * Gs + j] = m2g;
    }
  }
  return bad;
}

int64_t oracle_allreduce_mode(int P, int64_t n, int g, int bits, int mode, const uint16_t* x,
                              uint16_t* out, float* e, uint8_t* q1, uint32_t* m1,
                              uint8_t* q2, uint32_t* m2, float* acc, uint8_t* nq,
                              int64_t* ties) {
  return oracle_allreduce_ex(P, n, g, bits, mode, 0, 1.0f, x, out, e, q1, m1, q2, m2, acc, nq,
                             ties);
}

int64_t oracle_allreduce(int P, int64_t n, int g, int bits, const uint16_t* x,
                         uint16_t* out, float* e, uint8_t* q1, uint32_t* m1,
                         uint8_t* q2, uint32_t* m2, float* acc, uint8_t* nq,
                         int64_t* ties) {
  return oracle_allreduce_mode(P, n, g, bits, kZeroAware, x, out, e, q1, m1, q2, m2, acc, nq,
                               ties);
}

}  // extern "C"
