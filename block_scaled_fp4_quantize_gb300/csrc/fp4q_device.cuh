// fp4q_device.cuh -- device-side numerics of the block-scaled FP4 quantizer.
//
// Every floating-point step that decides a bit of the output is written with
// explicit PTX (div.rn / mul.rn / add.rn / sub.rn without .ftz), so results
// keep subnormals and do not change under -use_fast_math or -ftz=true.
// Absolute maxima are integer maxima of |x| bit patterns (monotone for
// non-negative finite binary32), and scale encoders work on exponent and
// mantissa bits; nothing here depends on log2/exp2 approximations.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fp4q {

// ---------------------------------------------------------------------------
// IEEE binary32, round to nearest even, subnormals preserved
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ieee_div(float a, float b) {
  float r;
  asm("div.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float ieee_mul(float a, float b) {
  float r;
  asm("mul.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float ieee_add(float a, float b) {
  float r;
  asm("add.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float ieee_sub(float a, float b) {
  float r;
  asm("sub.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ uint32_t fbits(float f) { return __float_as_uint(f); }
__device__ __forceinline__ float bitsf(uint32_t b) { return __uint_as_float(b); }
__device__ __forceinline__ uint32_t abs_bits(float f) { return __float_as_uint(f) & 0x7FFFFFFFu; }
// +-0 carrying the sign of v
__device__ __forceinline__ float signed_zero(float v) { return bitsf(fbits(v) & 0x80000000u); }

// bf16 <-> binary32
__device__ __forceinline__ float bf16lo(uint32_t w) { return bitsf(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return bitsf(w & 0xFFFF0000u); }
// two binary32 -> packed bf16x2 (lo in bits 0-15), round to nearest even
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------------------
// Inner-scale formats: E4M3 (bias 7, max 448, codes 0..0x7E) and UE5M3
// (bias 15, max 114688, codes 0..0xFE).  Byte c = exponent e (bits 7..3)
// and mantissa m (bits 2..0): e == 0 -> m * 2^(-2-bias); else
// (8 + m) * 2^(e - 3 - bias).
// ---------------------------------------------------------------------------
struct ScaleFmt {
  int bias;
  uint32_t maxcode;
  uint32_t maxbits;  // binary32 bits of the largest finite value
  float denom;       // largest finite value * 6 (the outer-scale denominator)
};

__host__ __device__ inline ScaleFmt scale_fmt(int ue5m3) {
  ScaleFmt f;
  if (ue5m3) { f.bias = 15; f.maxcode = 0xFE; f.maxbits = 0x47E00000u; f.denom = 688128.0f; }
  else       { f.bias = 7;  f.maxcode = 0x7E; f.maxbits = 0x43E00000u; f.denom = 2688.0f; }
  return f;
}

// Nearest code to v >= 0 (finite), ties to even, saturating at the maximum.
__device__ __forceinline__ uint32_t enc_scale(float v, const ScaleFmt& f) {
  uint32_t b = fbits(v);
  if (b >= f.maxbits) return f.maxcode;
  int ev = (int)(b >> 23) - 127;
  uint32_t sig = b & 0x7FFFFFu;
  if (b >> 23) sig |= 0x800000u; else ev = -126;
  const bool normal = ev >= 1 - f.bias;
  const int sh = normal ? 20 : 21 - f.bias - ev;  // bits below the kept mantissa
  uint32_t m = 0;
  if (sh < 32) {
    m = sig >> sh;
    const uint32_t rem = sig & ((1u << sh) - 1u);
    const uint32_t half = 1u << (sh - 1);
    m += (rem > half || (rem == half && (m & 1u))) ? 1u : 0u;
  }
  const uint32_t code = normal ? ((uint32_t)(ev + f.bias) << 3) + m - 8u : m;
  return code < f.maxcode ? code : f.maxcode;
}

// UE5M3 code of v >= 0 (finite): enc_scale with the UE5M3 format in fewer
// steps.  Normal range (v >= 2^-14): round the binary32 significand to 3
// bits, ties to even, on the bit pattern (a carry moves into the exponent)
// and rebias the exponent from 127 to 15.  Subnormal range: m = RN(v 2^17)
// from one FMA onto 2^23 (v 2^17 < 8 is exact, the sum rounds to an
// integer with ties to even); m = 8 is the smallest normal code.  Saturates
// at 0xFE.  Equal to enc_scale for every finite v >= 0
// (tests/gpu_scale_check.cu).
__device__ __forceinline__ uint32_t enc_ue5m3(float v) {
  const uint32_t b = fbits(v);
  const uint32_t r = (b + 0x7FFFFu + ((b >> 20) & 1u)) >> 20;
  const uint32_t n = r - ((127u - 15u) << 3);
  float s;
  asm("fma.rn.f32 %0, %1, 0f48000000, 0f4B000000;" : "=f"(s) : "f"(v));
  const uint32_t code = b < 0x38800000u ? (fbits(s) & 0xFu) : n;
  return code < 0xFEu ? code : 0xFEu;
}

__device__ __forceinline__ float dec_scale(uint32_t c, const ScaleFmt& f) {
  const uint32_t e = c >> 3, m = c & 7u;
  if (e == 0) return ieee_mul((float)m, bitsf((uint32_t)(127 - 2 - f.bias) << 23));
  return bitsf(((e - f.bias + 127u) << 23) | (m << 20));
}

// ---------------------------------------------------------------------------
// E2M1: code = sign << 3 | k, magnitude index k into {0,.5,1,1.5,2,3,4,6}
// ---------------------------------------------------------------------------

// Round-to-nearest-even with saturation, two values at a time (hardware
// conversion).  Returns a byte: `lo` in bits 0-3, `hi` in bits 4-7.
__device__ __forceinline__ uint32_t e2m1x2_rne(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Decode a byte of two codes to binary32 (exact).
__device__ __forceinline__ void e2m1x2_decode(uint32_t byte, float& lo, float& hi) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(byte));
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi) : "r"(h2));
}

// Stochastic rounding of t onto the E2M1 grid with the 32-bit random word w:
// between neighbours lo < |t| < hi the result is hi iff (w >> 8) < f * 2^24,
// f = (|t| - lo) / (hi - lo); the value is returned, sign kept (a grid value,
// so the hardware E2M1 conversion encodes it exactly).
// On the bit pattern b of |t| >= 1/2 the grid keeps one mantissa bit above 1
// and none in [1/2, 1) (its points there are 1/2 and 1), so the d = 22 (or
// 23) bits below the kept ones hold f * 2^d exactly.  Adding (2^d - 1) - (w >>
// (32 - d)) to b carries into the kept bits iff (w >> (32 - d)) < f * 2^d,
// which for integers is the condition above, and clearing the d bits leaves
// the chosen neighbour (a carry out of the mantissa lands on the next binade's
// first point).  Above 6 the result saturates at 6.  Below 1/2 the neighbours
// are 0 and 1/2, f * 2^24 = |t| * 2^25, compared in binary32 (both sides exact).
__device__ __forceinline__ float e2m1_sr_value(float t, uint32_t w) {
  const uint32_t b = abs_bits(t);
  const bool ge1 = b >= 0x3F800000u;
  const uint32_t mask = ge1 ? 0x3FFFFFu : 0x7FFFFFu;
  const uint32_t rnd = ge1 ? (w >> 10) : (w >> 9);
  uint32_t r = (b + (rnd ^ mask)) & ~mask;
  r = r < 0x40C00000u ? r : 0x40C00000u;
  float t25, u24;
  asm("mul.rn.f32 %0, %1, 0f4C000000;" : "=f"(t25) : "f"(bitsf(b)));
  asm("cvt.rn.f32.u32 %0, %1;" : "=f"(u24) : "r"(w >> 8));
  uint32_t half;
  asm("{\n\t.reg .pred p;\n\tsetp.lt.f32 p, %1, %2;\n\tselp.u32 %0, 0x3F000000, 0, p;\n\t}"
      : "=r"(half) : "f"(u24), "f"(t25));
  r = b < 0x3F000000u ? half : r;
  return bitsf(r | (fbits(t) & 0x80000000u));
}

// The E2M1 code of e2m1_sr_value.
__device__ __forceinline__ uint32_t e2m1_sr(float t, uint32_t w) { return e2m1x2_rne(e2m1_sr_value(t, w), 0.0f) & 0xFu; }

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11)
// ---------------------------------------------------------------------------

// The ten round keys of a 64-bit key: round r uses (k0 + r W0, k1 + r W1),
// W0 = 0x9E3779B9, W1 = 0xBB67AE85.  The kernels take them precomputed from
// their parameter block, so the rounds read them as constant operands.
struct PhiloxKeys {
  uint32_t k0[10], k1[10];
};

__host__ __device__ inline PhiloxKeys philox_keys(uint64_t key) {
  PhiloxKeys K;
  uint32_t k0 = (uint32_t)key, k1 = (uint32_t)(key >> 32);
  for (int r = 0; r < 10; ++r) {
    K.k0[r] = k0;
    K.k1[r] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return K;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxKeys& K) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c.x, p1 = (uint64_t)0xCD9E8D57u * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ K.k0[r], (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ K.k1[r],
                   (uint32_t)p0);
  }
  return c;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
  return philox4x32_10(c, philox_keys(((uint64_t)k1 << 32) | k0));
}

// Random words of elements 4*blk .. 4*blk+3 of an orientation's flat index
// space: counter (blk lo, blk hi, step, orient), key = seed (as round keys).
__device__ __forceinline__ uint4 sr_words(const PhiloxKeys& K, uint32_t step, uint32_t orient, uint64_t blk) {
  return philox4x32_10(make_uint4((uint32_t)blk, (uint32_t)(blk >> 32), step, orient), K);
}

// ---------------------------------------------------------------------------
// Exact binary32 division without div.rn
// ---------------------------------------------------------------------------

// RN(1 / s), the IEEE reciprocal.
__device__ __forceinline__ float ieee_rcp(float s) {
  float r;
  asm("rcp.rn.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

// RN(1 / s) for 2^-125 <= s <= 2^125 without the special-case handling of
// rcp.rn: the hardware approximation y, the residual e = RN(1 - s y) (exact:
// it fits in 24 bits when y is within an ulp of 1 / s) and one correction
// RN(y + e y) (Markstein's reciprocal refinement, same paper as
// div_markstein).  Its agreement with rcp.rn.f32 is checked for every
// binary32 of the range by tests/gpu_rcp_check.cu.
__device__ __forceinline__ float rcp_markstein(float s) {
  float r;
  asm("{\n\t.reg .f32 y, e;\n\trcp.approx.ftz.f32 y, %1;\n\tneg.f32 e, %1;\n\t"
      "fma.rn.f32 e, e, y, 0f3F800000;\n\tfma.rn.f32 %0, e, y, y;\n\t}"
      : "=f"(r) : "f"(s));
  return r;
}

// RN(u / S) from r = RN(1 / S) by Markstein's correction step (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990): q = RN(u r), e = RN(q S - u)
// (exact), result RN(q - e r).  Written with the remainder negated so that a
// zero quotient keeps the sign of u.  Exact whenever S is normal, |u / S| <
// 2^126 and |u| >= 2^-100 (the remainder is then representable); callers
// take div.rn outside that range.
__device__ __forceinline__ float div_markstein(float u, float S, float r) {
  float x;
  asm("{\n\t.reg .f32 q, e, nu, nr;\n\tmul.rn.f32 q, %1, %3;\n\tneg.f32 nu, %1;\n\t"
      "fma.rn.f32 e, q, %2, nu;\n\tneg.f32 nr, %3;\n\tfma.rn.f32 %0, e, nr, q;\n\t}"
      : "=f"(x) : "f"(u), "f"(S), "f"(r));
  return x;
}

// RN(y / d) for a divisor d known in advance through zh = RD(1 / d) and
// zl = RN(1 / d - zh) (N. Brisebarre, J.-M. Muller, S. K. Raina,
// "Accelerating correctly rounded floating-point division when the divisor is
// known in advance", IEEE Trans. Computers 53(8), 2004): RN(y zh + RN(y zl)).
// Exact for every y whose product y zl does not underflow, for the divisor
// significands this library uses (integers 1..15 and 21, checked over every
// dividend significand); zh, zl >= 0 keep the sign of a zero y.
__device__ __forceinline__ float div_bmr(float y, float zh, float zl) {
  float r;
  asm("{\n\t.reg .f32 p;\n\tmul.rn.f32 p, %1, %3;\n\tfma.rn.f32 %0, %1, %2, p;\n\t}"
      : "=f"(r) : "f"(y), "f"(zh), "f"(zl));
  return r;
}

// max(m, |a|, |b|) with NaN propagating and subnormals kept.
__device__ __forceinline__ float amax3(float m, float a, float b) {
  float r;
  asm("{\n\t.reg .f32 x, y;\n\tabs.f32 x, %2;\n\tabs.f32 y, %3;\n\tmax.NaN.f32 %0, %1, x, y;\n\t}"
      : "=f"(r) : "f"(m), "f"(a), "f"(b));
  return r;
}

// S > 0 for a binary32 bit pattern (NaN and negative values are not), without
// a float compare that -ftz could flush.
__device__ __forceinline__ bool positive(float S) {
  const int b = (int)fbits(S);
  return b > 0 && b <= 0x7F800000;
}
// S is a normal, finite, positive binary32.
__device__ __forceinline__ bool positive_normal(float S) {
  const uint32_t b = fbits(S);
  return b >= 0x00800000u && b < 0x7F800000u;
}

// E4M3 code of v >= 0 (RNE, saturating at 448) by the hardware conversion.
__device__ __forceinline__ uint32_t enc_e4m3_hw(float v) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, 0f00000000, %1;\n\tcvt.u32.u16 %0, t;\n\t}"
      : "=r"(r) : "f"(v));
  return r & 0xFFu;
}

// One 256-bit store (p 32-byte aligned): a lane fills a whole 32-byte sector.
__device__ __forceinline__ void st256(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// ---------------------------------------------------------------------------
// Packed binary32 pairs (f32x2, one 64-bit register): two lanes of the same
// IEEE operation per instruction, round to nearest even, subnormals kept.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// Markstein's quotient (see div_markstein) for a pair, from the NEGATED
// dividends nu = -u: q = RN(nu * -r) = RN(u r), e = RN(q S + nu), x =
// RN(e * -r + q).  S2 = (S, S), NR2 = (-r, -r).  The zero quotient keeps the
// sign of u.
__device__ __forceinline__ uint64_t markstein2(uint64_t nu, uint64_t S2, uint64_t NR2) {
  const uint64_t q = mul2(nu, NR2);
  const uint64_t e = fma2(q, S2, nu);
  return fma2(e, NR2, q);
}

// Brisebarre-Muller-Raina quotient (see div_bmr) for a pair: RN(y zh + RN(y zl)).
__device__ __forceinline__ uint64_t bmr2(uint64_t y, uint64_t ZH2, uint64_t ZL2) {
  return fma2(y, ZH2, mul2(y, ZL2));
}

// Negated bf16 -> binary32 (low / high half of a bf16x2 word): -(w << 16) and
// -(w & 0xFFFF0000), one integer instruction each.
__device__ __forceinline__ float nbf16lo(uint32_t w) { return bitsf(w * 65536u + 0x80000000u); }
__device__ __forceinline__ float nbf16hi(uint32_t w) { return bitsf((w & 0xFFFF0000u) ^ 0x80000000u); }

// max(|a|, |b|) of bf16x2 lanes with NaN propagating (lane signs garbage).
__device__ __forceinline__ uint32_t bf16x2_amax(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// max(|a|, |b|) of binary32 (sign garbage), subnormals kept.
__device__ __forceinline__ float f32_amax(float a, float b) {
  float r;
  asm("max.NaN.xorsign.abs.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Four pairs -> one word of eight E2M1 codes, RNE with saturation; pair i
// goes to byte i, its first value in the low nibble.
__device__ __forceinline__ uint32_t e2m1x8_rne(const float* t) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(t[0]), "f"(t[1]), "f"(t[2]), "f"(t[3]), "f"(t[4]), "f"(t[5]), "f"(t[6]), "f"(t[7]));
  return r;
}

// NaN -> +0, +-inf -> +- the largest finite value of the input dtype.
__device__ __forceinline__ float sanitize(float u, uint32_t maxfinite_bits) {
  const uint32_t b = fbits(u);
  if ((b & 0x7F800000u) != 0x7F800000u) return u;
  if (b & 0x7FFFFFu) return 0.0f;
  return bitsf((b & 0x80000000u) | maxfinite_bits);
}

}  // namespace fp4q
