// fp4q_block.cuh -- per-block steps shared by the fast quantize kernels
// (rowwise flat kernel and cast-transpose tile kernel): outer and inner
// scales, the normalization u -> x' = u / S and the E2M1 encode, each with
// the exact FMA division sequences of fp4q_device.cuh.
#pragma once

#include "fp4q_device.cuh"

namespace fp4q {
namespace {

// RD(1/M) and RN(1/M - RD(1/M)) for M = 0..15 (M = 0 unused); see div_bmr.
__constant__ uint32_t kRcpHi[16] = {0x00000000u, 0x3F800000u, 0x3F000000u, 0x3EAAAAAAu, 0x3E800000u, 0x3E4CCCCCu,
                                    0x3E2AAAAAu, 0x3E124924u, 0x3E000000u, 0x3DE38E38u, 0x3DCCCCCCu, 0x3DBA2E8Bu,
                                    0x3DAAAAAAu, 0x3D9D89D8u, 0x3D924924u, 0x3D888888u};
__constant__ uint32_t kRcpLo[16] = {0x00000000u, 0x00000000u, 0x00000000u, 0x32AAAAABu, 0x00000000u, 0x324CCCCDu,
                                    0x322AAAABu, 0x32124925u, 0x00000000u, 0x31E38E39u, 0x31CCCCCDu, 0x31A2E8BAu,
                                    0x31AAAAABu, 0x319D89D9u, 0x31924925u, 0x31888889u};
// 1/6 split the same way (a / 6 for the inner scale)
constexpr uint32_t kSixHi = 0x3E2AAAAAu, kSixLo = 0x322AAAABu;
// 1/2688 (E4M3: 448 * 6 = 21 * 2^7) and 1/688128 (UE5M3: 114688 * 6 = 21 * 2^15)
constexpr uint32_t kDenHiE4 = 0x39C30C30u, kDenLoE4 = 0x2DC30C31u;
constexpr uint32_t kDenHiU5 = 0x35C30C30u, kDenLoU5 = 0x29C30C31u;

// amax bits below which the FMA division paths are not used (2^-90)
constexpr uint32_t kTiny = 0x12800000u;

__device__ __forceinline__ uint32_t umax(uint32_t a, uint32_t b) { return a > b ? a : b; }

// outer scale amax / (scale_max * 6)
template <bool UE5M3>
__device__ __forceinline__ float outer_scale(float A) {
  if (fbits(A) >= kTiny)
    return div_bmr(A, bitsf(UE5M3 ? kDenHiU5 : kDenHiE4), bitsf(UE5M3 ? kDenLoU5 : kDenLoE4));
  return ieee_div(A, UE5M3 ? 688128.0f : 2688.0f);
}

template <bool UE5M3>
__device__ __forceinline__ uint32_t encode_scale(float v) {
  if (UE5M3) return enc_ue5m3(v);
  return enc_e4m3_hw(v);
}

// Per-block state of the normalization u -> x' = u / S.
struct Norm {
  float S, r;
  bool none, pos, fast;
};

// Inner scale of a block with |u| maximum `am` (binary32, finite): returns
// the code and fills (s, zh, zl) from the table; `n.fast` is narrowed to the
// range where the Markstein path is exact.
template <bool UE5M3, class SM>
__device__ __forceinline__ uint32_t block_scale(const SM& sm, float am, Norm& n, float4& T) {
  float a;
  if (n.none) {
    a = am;
  } else if (!n.pos) {
    a = 0.0f;
  } else {
    n.fast = n.fast && fbits(am) >= kTiny;
    a = n.fast ? div_markstein(am, n.S, n.r) : ieee_div(am, n.S);
    n.fast = n.fast && fbits(a) < 0x7E800000u;
  }
  const float v = div_bmr(a, bitsf(kSixHi), bitsf(kSixLo));
  const uint32_t sc = encode_scale<UE5M3>(v);
  T = sm.tab[sc];
  return sc;
}


// Rare path of normalize16 (tiny, subnormal or non-positive scales).
__device__ __noinline__ float div_slow(float u, float S, bool pos) { return pos ? ieee_div(u, S) : signed_zero(u); }

// |u| bits below which Markstein's remainder can underflow (2^-100)
constexpr uint32_t kTinyElem = 0x0D800000u;

// Elements 0 < |u| < 2^-100 of a block whose maximum is at least 2^-90 get
// x' from div.rn.  With round-to-nearest they cannot matter: |x'| / a <=
// 2^-10, so |t| = |x'| / s < 0.01 and the code is +-0 whichever x' is
// taken (the dequantized value and the residual follow).  Stochastic
// rounding compares t itself with a random threshold, so its callers pass
// TINY = true.
template <bool TINY>
__device__ __forceinline__ void fix_tiny(const float (&u)[16], float (&x)[16], const Norm& n, uint32_t sgn) {
  if (!TINY) return;
  bool any = false;
#pragma unroll
  for (int i = 0; i < 16; ++i) any |= abs_bits(u[i]) - 1u < kTinyElem - 1u;
  if (any) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (abs_bits(u[i]) - 1u < kTinyElem - 1u) x[i] = ieee_div(bitsf(fbits(u[i]) ^ sgn), n.S);
  }
}

// x' = u / S for a whole block: one block-uniform branch, the fast path two
// values per instruction.
template <bool TINY>
__device__ __forceinline__ void normalize16(const float (&u)[16], float (&x)[16], const Norm& n) {
  if (n.none) {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = u[i];
  } else if (n.fast) {
    const float nr = bitsf(fbits(n.r) ^ 0x80000000u);
    const uint64_t S2 = pk2(n.S, n.S), NR2 = pk2(nr, nr);
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const uint64_t nu = pk2(bitsf(fbits(u[i]) ^ 0x80000000u), bitsf(fbits(u[i + 1]) ^ 0x80000000u));
      upk2(markstein2(nu, S2, NR2), x[i], x[i + 1]);
    }
    fix_tiny<TINY>(u, x, n, 0u);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = div_slow(u[i], n.S, n.pos);
  }
}

// normalize16 from the NEGATED values nu = -u (bf16 inputs widen to -u in
// one instruction, so the negation the sign-safe Markstein form needs costs
// nothing); same results.  Not for mode none.
template <bool TINY>
__device__ __forceinline__ void normalize16_neg(const float (&nu)[16], float (&x)[16], const Norm& n) {
  if (n.fast) {
    const float nr = bitsf(fbits(n.r) ^ 0x80000000u);
    const uint64_t S2 = pk2(n.S, n.S), NR2 = pk2(nr, nr);
#pragma unroll
    for (int i = 0; i < 16; i += 2) upk2(markstein2(pk2(nu[i], nu[i + 1]), S2, NR2), x[i], x[i + 1]);
    fix_tiny<TINY>(nu, x, n, 0x80000000u);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = div_slow(bitsf(fbits(nu[i]) ^ 0x80000000u), n.S, n.pos);
  }
}

// 16 values -> 16 codes (two 32-bit words, element 2i in the low nibble of
// byte i); optional dequantized values (e2m1 * s) * S.
template <bool SR, bool DEQ>
__device__ __forceinline__ void encode16(const float (&x)[16], const float4& T, const Norm& n, const PhiloxKeys& K,
                                         uint32_t step, uint32_t orient, uint64_t n0, uint32_t& w0, uint32_t& w1,
                                         float (&deq)[16]) {
  float t[16];
  {
    const uint64_t ZH2 = pk2(T.y, T.y), ZL2 = pk2(T.z, T.z);
#pragma unroll
    for (int i = 0; i < 16; i += 2) upk2(bmr2(pk2(x[i], x[i + 1]), ZH2, ZL2), t[i], t[i + 1]);
  }
  uint32_t byte[8];
  if (!SR && !DEQ) {
    w0 = e2m1x8_rne(t);
    w1 = e2m1x8_rne(t + 8);
    return;
  }
  if (SR) {  // the chosen grid values, encoded by the hardware conversion (exact)
    float g[16];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint4 rw = sr_words(K, step, orient, (n0 >> 2) + (uint64_t)w);
      g[4 * w] = e2m1_sr_value(t[4 * w], rw.x);
      g[4 * w + 1] = e2m1_sr_value(t[4 * w + 1], rw.y);
      g[4 * w + 2] = e2m1_sr_value(t[4 * w + 2], rw.z);
      g[4 * w + 3] = e2m1_sr_value(t[4 * w + 3], rw.w);
    }
    w0 = e2m1x8_rne(g);
    w1 = e2m1x8_rne(g + 8);
    if (DEQ) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float d = ieee_mul(g[i], T.x);
        if (!n.none) d = ieee_mul(d, n.S);
        deq[i] = d;
      }
    }
    return;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) byte[i] = e2m1x2_rne(t[2 * i], t[2 * i + 1]);
  }
  w0 = __byte_perm(__byte_perm(byte[0], byte[1], 0x0040), __byte_perm(byte[2], byte[3], 0x0040), 0x5410);
  w1 = __byte_perm(__byte_perm(byte[4], byte[5], 0x0040), __byte_perm(byte[6], byte[7], 0x0040), 0x5410);
  if (DEQ) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float g0, g1;
      e2m1x2_decode(byte[i], g0, g1);
      float d0 = ieee_mul(g0, T.x), d1 = ieee_mul(g1, T.x);
      if (!n.none) { d0 = ieee_mul(d0, n.S); d1 = ieee_mul(d1, n.S); }
      deq[2 * i] = d0;
      deq[2 * i + 1] = d1;
    }
  }
}


// Per-block steps for a block the FMA division sequences cover
// (fast_block below): `a` = RN(am / S) is already known and no step needs a
// fallback.  OUTER: an outer scale applies; NEG: the values arrive negated.
template <bool SR, bool UE5M3, bool OUTER, bool NEG, class TabT>
__device__ __forceinline__ uint32_t block_fast(const TabT& tab, const float (&v)[16], float a, float S, float r,
                                               const PhiloxKeys& K, uint32_t step, uint32_t orient, uint64_t n0,
                                               uint32_t& w0, uint32_t& w1) {
  const uint32_t sc = encode_scale<UE5M3>(div_bmr(a, bitsf(kSixHi), bitsf(kSixLo)));
  const float4 T = tab[sc];
  Norm n;
  n.none = !OUTER;
  n.S = S;
  n.r = r;
  n.pos = true;
  n.fast = true;
  float x[16], dq[16];
  if (NEG) normalize16_neg<SR>(v, x, n);
  else normalize16<SR>(v, x, n);
  encode16<SR, false>(x, T, n, K, step, orient, n0, w0, w1, dq);
  return sc;
}

// A block is covered by block_fast when its outer scale S and 1 / S are
// normal, its |u| maximum am is 0 or at least 2^-90 and a = RN(am / S) is
// below 2^126: the conditions under which block_scale and normalize16 take
// no fallback (am = 0 gives a = +0 and signed-zero quotients either way).
// Returns a.
__device__ __forceinline__ bool fast_block(float am, float S, float R, float& a) {
  a = div_markstein(am, S, R);
  return (fbits(S) - 0x00800000u) < 0x7F000000u && (fbits(R) - 0x00800000u) < 0x7F000000u &&
         fbits(am) - 1u >= kTiny - 1u && fbits(a) < 0x7E800000u;
}

// Outer scale S = RN(A / (scale_max * 6)) and R = RN(1 / S), called by a
// whole warp: when every lane's A is at least 2^-90, S lies in
// [2^-110, 2^117] and both come from the FMA sequences; otherwise the warp
// takes the general path.  Returns true on the first branch (warp-uniform):
// then S and R are normal and RN(am / S) < 2^126 for every am <= A.
template <bool UE5M3>
__device__ __forceinline__ bool outer_sr(float A, float& S, float& R) {
  if (__all_sync(0xFFFFFFFFu, fbits(A) >= kTiny)) {
    S = div_bmr(A, bitsf(UE5M3 ? kDenHiU5 : kDenHiE4), bitsf(UE5M3 ? kDenLoU5 : kDenLoE4));
    R = rcp_markstein(S);
    return true;
  }
  S = outer_scale<UE5M3>(A);
  R = ieee_rcp(S);
  return false;
}

// outer_sr for two outer blocks at once (one branch for both).
template <bool UE5M3>
__device__ __forceinline__ bool outer_sr2(float A0, float A1, float (&S)[2], float (&R)[2]) {
  if (__all_sync(0xFFFFFFFFu, fbits(A0) >= kTiny && fbits(A1) >= kTiny)) {
    S[0] = div_bmr(A0, bitsf(UE5M3 ? kDenHiU5 : kDenHiE4), bitsf(UE5M3 ? kDenLoU5 : kDenLoE4));
    S[1] = div_bmr(A1, bitsf(UE5M3 ? kDenHiU5 : kDenHiE4), bitsf(UE5M3 ? kDenLoU5 : kDenLoE4));
    R[0] = rcp_markstein(S[0]);
    R[1] = rcp_markstein(S[1]);
    return true;
  } else {
    S[0] = outer_scale<UE5M3>(A0);
    S[1] = outer_scale<UE5M3>(A1);
    R[0] = ieee_rcp(S[0]);
    R[1] = ieee_rcp(S[1]);
  }
  return false;
}

// max |u| over 16 values (NaN propagates), as a tree of magnitude maxima.
__device__ __forceinline__ float amax_pair(float a, float b) {
  float r;
  asm("{\n\t.reg .f32 x, y;\n\tabs.f32 x, %1;\n\tabs.f32 y, %2;\n\tmax.NaN.f32 %0, x, y;\n\t}" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float amax16(const float (&u)[16]) {
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = amax_pair(u[2 * i], u[2 * i + 1]);
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = max_nan(m[2 * i], m[2 * i + 1]);
  return max_nan(max_nan(m[0], m[1]), max_nan(m[2], m[3]));
}

// Sanitized copy of a bf16 pair (NaN -> +0, +-inf -> +-largest finite).
__device__ __forceinline__ uint32_t sanitize_bf16x2(uint32_t w) {
  uint32_t r = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t v = (w >> (16 * h)) & 0xFFFFu;
    const uint32_t a = v & 0x7FFFu;
    if (a > 0x7F80u) v = 0u;
    else if (a == 0x7F80u) v = (v & 0x8000u) | 0x7F7Fu;
    r |= v << (16 * h);
  }
  return r;
}

// max |.| of the two halves of a packed bf16 maximum, as binary32.
__device__ __forceinline__ float bf16x2_hmax(uint32_t m) {
  m &= 0x7FFF7FFFu;
  const uint32_t hi = m >> 16, lo = m & 0xFFFFu;
  return bitsf((hi > lo ? hi : lo) << 16);
}

// Inner-scale table entry of code c: (DEC(c), zh, zl, 0) with zh + zl the
// split reciprocal of DEC(c) used by div_bmr.
template <bool UE5M3>
__device__ __forceinline__ float4 scale_entry(uint32_t c) {
  const int bias = UE5M3 ? 15 : 7;
  const uint32_t e = c >> 3, m = c & 7u;
  const uint32_t M = e ? 8u + m : m;
  const int ex = e ? (int)e - 3 - bias : -2 - bias;
  const uint32_t hi = kRcpHi[M], lo = kRcpLo[M];
  return make_float4(dec_scale(c, scale_fmt(UE5M3 ? 1 : 0)), M ? bitsf((uint32_t)((int)hi - ex * 8388608)) : 0.0f,
                     lo ? bitsf((uint32_t)((int)lo - ex * 8388608)) : 0.0f, 0.0f);
}

// Inner-scale table in shared memory (entries of scale_entry).
template <bool UE5M3>
__device__ __forceinline__ void build_scale_table(float4* tab, int t, int nthreads) {
  for (int c = t; c < 256; c += nthreads) tab[c] = scale_entry<UE5M3>((uint32_t)c);
}

}  // namespace
}  // namespace fp4q
