// k_ct.cu -- fast fused quantize / cast-transpose / QDQ kernel.
//
// One CTA of 256 threads owns a 128 (M) x 64 (K) tile at a time (grid-stride
// over tiles, grid sized to the resident CTAs).  Rowwise pass: thread t owns
// the 1 x 16 blocks (row t/4, block t%4) and (row t/4 + 64, block t%4), loaded
// straight from HBM with 128-bit loads; a 1 x 64 outer block is the 4 lanes
// of one row, reduced with two xor-shuffles.  The columnwise pass reads the
// tile back from a swizzled binary32 staging buffer in shared memory (thread
// owns 2 columns x 16 rows), so x is read from HBM once for both
// orientations ("Block-Scaled FP8 and FP4 Weight Quantization", section 3).
// With a 2-D outer scale, tensorwise or no outer scale, the normalized value
// x' = u / S is computed once and staged; with 1-D outer scales u is staged
// and each orientation normalizes by its own scale.
//
// Division: every quotient the method defines is one IEEE binary32 division.
// Here they are computed exactly with FMA sequences: u / S with Markstein's
// correction from RN(1/S), x' / s and a / 6 and amax / (scale_max * 6) with
// the Brisebarre-Muller-Raina method for divisors known in advance (the inner
// scale s has a 4-bit significand).  Blocks outside the proven range (tiny or
// subnormal scales) take div.rn.
//
// Covers: inner 1 x 16 blocks, 16-byte-aligned inputs; modes none, tensorwise,
// outer-block 1-D / 2-D with ob in {16, 32, 64} computed in the tile or any ob
// read from the outer buffers; RNE / SR; error feedback; QDQ along K or M.
#include "fp4q_device.cuh"
#include "fp4q_internal.h"

namespace fp4q {
namespace {

constexpr int TM = 128, TK = 64, NT = 256;

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

template <bool COL>
struct Smem {
  float stage[COL ? TM * TK : 4];  // columnwise staging (swizzled), binary32
  float4 tab[256];         // per inner-scale code: (s, zh, zl, -)
  uint32_t red2d[32];      // 2-D sub-block amax (bits)
  float2 sr2d[32];         // 2-D sub-block (S, 1/S)
  uint32_t redcol[8][TK];  // 1-D columnwise outer amax per (row block, column)
};

// swizzled index of (row, col) in the staging tile: 16-byte units of a row are
// permuted so that the rowwise stores and the columnwise loads are free of
// bank conflicts
__device__ __forceinline__ int sidx(int row, int col) {
  const int unit = col >> 2;
  const int phys = unit ^ (((unit >> 3) & 1) << 1) ^ (row & 1);
  return row * TK + phys * 4 + (col & 3);
}

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
  if (UE5M3) return enc_scale(v, scale_fmt(1));
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

__device__ __forceinline__ float normalize(float u, const Norm& n) {
  if (n.none) return u;
  if (n.fast) return div_markstein(u, n.S, n.r);
  return n.pos ? ieee_div(u, n.S) : signed_zero(u);
}

// 16 values -> 16 codes (two 32-bit words, element 2i in the low nibble of
// byte i); optional dequantized values (e2m1 * s) * S.
template <bool SR, bool DEQ>
__device__ __forceinline__ void encode16(const float (&x)[16], const float4& T, const Norm& n, uint64_t seed,
                                         uint32_t step, uint32_t orient, uint64_t n0, uint32_t& w0, uint32_t& w1,
                                         float (&deq)[16]) {
  float t[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) t[i] = div_bmr(x[i], T.y, T.z);
  uint32_t byte[8];
  if (SR) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint4 rw = sr_words(seed, step, orient, (n0 >> 2) + (uint64_t)w);
      byte[2 * w] = e2m1_sr(t[4 * w], rw.x) | (e2m1_sr(t[4 * w + 1], rw.y) << 4);
      byte[2 * w + 1] = e2m1_sr(t[4 * w + 2], rw.z) | (e2m1_sr(t[4 * w + 3], rw.w) << 4);
    }
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

template <bool IN_BF16>
__device__ __forceinline__ void load16(const QuantJob& j, int64_t g, int64_t m, int64_t k, float (&u)[16]) {
  if (IN_BF16) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(j.x) + (g * j.M + m) * j.ld + k);
    const uint4 a = __ldg(p), b = __ldg(p + 1);
    u[0] = bf16lo(a.x); u[1] = bf16hi(a.x); u[2] = bf16lo(a.y); u[3] = bf16hi(a.y);
    u[4] = bf16lo(a.z); u[5] = bf16hi(a.z); u[6] = bf16lo(a.w); u[7] = bf16hi(a.w);
    u[8] = bf16lo(b.x); u[9] = bf16hi(b.x); u[10] = bf16lo(b.y); u[11] = bf16hi(b.y);
    u[12] = bf16lo(b.z); u[13] = bf16hi(b.z); u[14] = bf16lo(b.w); u[15] = bf16hi(b.w);
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(j.x) + (g * j.M + m) * j.ld + k);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v = __ldg(p + q);
      u[4 * q] = v.x; u[4 * q + 1] = v.y; u[4 * q + 2] = v.z; u[4 * q + 3] = v.w;
    }
  }
  if (j.residual) {
    const float4* rp = reinterpret_cast<const float4*>(j.residual + (g * j.M + m) * j.K + k);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v = rp[q];
      u[4 * q] = ieee_add(u[4 * q], v.x); u[4 * q + 1] = ieee_add(u[4 * q + 1], v.y);
      u[4 * q + 2] = ieee_add(u[4 * q + 2], v.z); u[4 * q + 3] = ieee_add(u[4 * q + 3], v.w);
    }
  }
}

__device__ __forceinline__ float amax16(const float (&u)[16]) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; i += 2) a = amax3(a, u[i], u[i + 1]);
  return a;
}

__device__ __forceinline__ void store16(void* y, int out_bf16, int64_t idx, const float (&v)[16]) {
  if (out_bf16) {
    uint4* p = reinterpret_cast<uint4*>(static_cast<uint16_t*>(y) + idx);
    p[0] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
    p[1] = make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]), pack_bf16x2(v[12], v[13]),
                      pack_bf16x2(v[14], v[15]));
  } else {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(y) + idx);
#pragma unroll
    for (int q = 0; q < 4; ++q) p[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  }
}

template <bool IN_BF16, bool SR, bool COL, bool UE5M3>
__global__ void __launch_bounds__(NT) ct_kernel(const QuantJob j) {
  __shared__ __align__(16) Smem<COL> sm;
  const int t = threadIdx.x;
  const uint32_t maxfin = IN_BF16 ? 0x7F7F0000u : 0x7F7FFFFFu;

  // inner-scale table: value, and the divisor split of its reciprocal
  {
    const uint32_t c = (uint32_t)t;
    const int bias = UE5M3 ? 15 : 7;
    const uint32_t e = c >> 3, m = c & 7u;
    const uint32_t M = e ? 8u + m : m;
    const int ex = e ? (int)e - 3 - bias : -2 - bias;
    const float s = dec_scale(c, scale_fmt(UE5M3 ? 1 : 0));
    const uint32_t hi = kRcpHi[M], lo = kRcpLo[M];
    const float zh = M ? bitsf((uint32_t)((int)hi - ex * 8388608)) : 0.0f;
    const float zl = lo ? bitsf((uint32_t)((int)lo - ex * 8388608)) : 0.0f;
    sm.tab[c] = make_float4(s, zh, zl, 0.0f);
    if (t < 32) sm.red2d[t] = 0u;
    for (int i = t; i < 8 * TK; i += NT) (&sm.redcol[0][0])[i] = 0u;
  }

  const int64_t tiles_m = (j.M + TM - 1) / TM, tiles_k = (j.K + TK - 1) / TK;
  const int64_t ntiles = j.G * tiles_m * tiles_k;
  const int ob = j.ob;
  const bool none = j.s_src == S_ONE;
  const bool shared_S = none || j.mode == 1 || j.outer_2d;  // one normalization for both orientations
  float S_tw = 1.0f, r_tw = 1.0f;
  if (j.s_src == S_TENSORWISE_WS) {
    S_tw = ieee_div(bitsf(*j.tw_amax), UE5M3 ? 688128.0f : 2688.0f);
    r_tw = ieee_rcp(S_tw);
    if (blockIdx.x == 0 && t == 0 && j.tile_outer) j.tile_outer[0] = S_tw;
  }
  const bool deq_row = j.qdq_orient == 1 || j.residual != nullptr;
  const int b = t & 3, rr = t >> 2;
  __syncthreads();

  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t tk = tile % tiles_k;
    const int64_t tm = (tile / tiles_k) % tiles_m;
    const int64_t g = tile / (tiles_k * tiles_m);
    const int64_t m0 = tm * TM, k0 = tk * TK;
    const int64_t kb = k0 + 16 * b;

    // ---------------------------------------------------------------- load
    float u[2][16];
    float am[2];
    bool valid[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t m = m0 + rr + 64 * h;
      valid[h] = m < j.M && kb < j.K;
      if (valid[h]) {
        load16<IN_BF16>(j, g, m, kb, u[h]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) u[h][i] = 0.0f;
      }
      am[h] = amax16(u[h]);
      if (fbits(am[h]) >= 0x7F800000u) {  // inf or NaN present: sanitize this block
#pragma unroll
        for (int i = 0; i < 16; ++i) u[h][i] = sanitize(u[h][i], maxfin);
        am[h] = amax16(u[h]);
      }
    }

    // ---------------------------------------------------- outer scale (rows)
    Norm nr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      nr[h].none = none;
      nr[h].S = 1.0f;
      nr[h].r = 1.0f;
    }
    if (j.s_src == S_TENSORWISE_WS) {
#pragma unroll
      for (int h = 0; h < 2; ++h) { nr[h].S = S_tw; nr[h].r = r_tw; }
    } else if (j.s_src == S_IN_TILE && j.outer_2d) {
      // reduce over the ob x ob sub-blocks of the tile in shared memory
      const int nbk = TK / ob;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v = fbits(am[h]);
        v = umax(v, __shfl_xor_sync(0xFFFFFFFFu, v, 4));
        v = umax(v, __shfl_xor_sync(0xFFFFFFFFu, v, 8));
        v = umax(v, __shfl_xor_sync(0xFFFFFFFFu, v, 16));
        if (ob >= 32) v = umax(v, __shfl_xor_sync(0xFFFFFFFFu, v, 1));
        if (ob >= 64) v = umax(v, __shfl_xor_sync(0xFFFFFFFFu, v, 2));
        const int row = rr + 64 * h;
        if ((t & 31) < 4 && (b % (ob / 16)) == 0) atomicMax(&sm.red2d[(row / ob) * nbk + (16 * b) / ob], v);
      }
      __syncthreads();
      const int nsub = (TM / ob) * nbk;
      if (t < nsub) {
        const float A = bitsf(sm.red2d[t]);
        sm.red2d[t] = 0u;
        const float S = outer_scale<UE5M3>(A);
        sm.sr2d[t] = make_float2(S, ieee_rcp(S));
        const int64_t mi = m0 + (int64_t)(t / nbk) * ob, kj = k0 + (int64_t)(t % nbk) * ob;
        if (j.tile_outer && mi < j.M && kj < j.K) j.tile_outer[(g * (j.M / ob) + mi / ob) * (j.K / ob) + kj / ob] = S;
      }
      __syncthreads();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float2 sr = sm.sr2d[((rr + 64 * h) / ob) * nbk + (16 * b) / ob];
        nr[h].S = sr.x;
        nr[h].r = sr.y;
      }
    } else if (j.s_src == S_IN_TILE && j.do_row) {
      // 1-D along K: the 4 lanes of a row hold the 4 blocks of 1 x 64
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v = fbits(am[h]);
        if (ob >= 32) v = umax(v, __shfl_xor_sync(0xFFFFFFFFu, v, 1));
        if (ob >= 64) v = umax(v, __shfl_xor_sync(0xFFFFFFFFu, v, 2));
        const float S = outer_scale<UE5M3>(bitsf(v));
        nr[h].S = S;
        nr[h].r = ieee_rcp(S);
        const int64_t m = m0 + rr + 64 * h;
        if (valid[h] && (b % (ob / 16)) == 0 && j.row_outer) j.row_outer[(g * j.M + m) * (j.K / ob) + kb / ob] = S;
      }
    } else if (j.s_src == S_FROM_BUFFER && (j.do_row || shared_S)) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (!valid[h]) continue;
        const int64_t m = m0 + rr + 64 * h;
        float S;
        if (j.mode == 1) S = j.tile_outer[0];
        else if (j.outer_2d) S = j.tile_outer[(g * (j.M / ob) + m / ob) * (j.K / ob) + kb / ob];
        else S = j.row_outer[(g * j.M + m) * (j.K / ob) + kb / ob];
        nr[h].S = S;
        nr[h].r = ieee_rcp(S);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      nr[h].pos = none || positive(nr[h].S);
      nr[h].fast = !none && positive_normal(nr[h].S);
    }

    // ---------------------------------------------------------- rowwise pass
    if (j.do_row || (COL && shared_S)) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float4 T;
        const uint32_t sc = block_scale<UE5M3>(sm, am[h], nr[h], T);
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = normalize(u[h][i], nr[h]);
        const int row = rr + 64 * h;
        if (COL && shared_S) {
          float4* d = reinterpret_cast<float4*>(sm.stage);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            d[sidx(row, 16 * b + 4 * q) >> 2] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
        }
        if (j.do_row) {
          const int64_t m = m0 + row;
          const uint64_t n0 = (uint64_t)((g * j.M + m) * j.K + kb);
          uint32_t w0, w1;
          float deq[16];
          if (deq_row) encode16<SR, true>(x, T, nr[h], j.seed, j.step, 0u, n0, w0, w1, deq);
          else encode16<SR, false>(x, T, nr[h], j.seed, j.step, 0u, n0, w0, w1, deq);
          if (valid[h]) {
            if (j.row_codes) *reinterpret_cast<uint2*>(j.row_codes + n0 / 2) = make_uint2(w0, w1);
            if (j.row_scales) j.row_scales[n0 / 16] = (uint8_t)sc;
            if (j.residual) {
              float4* rp = reinterpret_cast<float4*>(j.residual + n0);
#pragma unroll
              for (int q = 0; q < 4; ++q)
                rp[q] = make_float4(ieee_sub(u[h][4 * q], deq[4 * q]), ieee_sub(u[h][4 * q + 1], deq[4 * q + 1]),
                                    ieee_sub(u[h][4 * q + 2], deq[4 * q + 2]), ieee_sub(u[h][4 * q + 3], deq[4 * q + 3]));
            }
            if (j.qdq_orient == 1) store16(j.y, j.out_bf16, (int64_t)n0, deq);
          }
        }
      }
    }
    if (!COL) continue;

    if (!shared_S) {
      // 1-D outer scales: stage u, each orientation normalizes by its own S
      float4* d = reinterpret_cast<float4*>(sm.stage);
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int q = 0; q < 4; ++q)
          d[sidx(rr + 64 * h, 16 * b + 4 * q) >> 2] =
              make_float4(u[h][4 * q], u[h][4 * q + 1], u[h][4 * q + 2], u[h][4 * q + 3]);
    }
    __syncthreads();

    // -------------------------------------------------------- columnwise pass
    {
      const int cp = t & 31, seg = t >> 5;
      const int64_t kc = k0 + 2 * cp, mb = m0 + 16 * seg;
      const bool cvalid = kc < j.K && mb < j.M;
      float v[2][16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 p = *reinterpret_cast<const float2*>(&sm.stage[sidx(16 * seg + i, 2 * cp)]);
        v[0][i] = p.x;
        v[1][i] = p.y;
      }
      Norm nc[2];
      float cam[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        cam[c] = amax16(v[c]);
        nc[c].none = true;
        nc[c].S = 1.0f;
        nc[c].r = 1.0f;
        nc[c].pos = true;
        nc[c].fast = false;
      }
      if (shared_S) {
        // staged values are already normalized; keep S for the dequantized output
        if (!none) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            if (j.s_src == S_TENSORWISE_WS) nc[c].S = S_tw;
            else if (j.s_src == S_IN_TILE) nc[c].S = sm.sr2d[((16 * seg) / ob) * (TK / ob) + (2 * cp) / ob].x;
            else if (cvalid) {
              const int64_t k = kc + c;
              nc[c].S = j.mode == 1 ? j.tile_outer[0]
                                    : j.tile_outer[(g * (j.M / ob) + mb / ob) * (j.K / ob) + k / ob];
            }
          }
        }
      } else {
        // 1-D along M
        if (j.s_src == S_IN_TILE) {
          const int segs = ob / 16;
#pragma unroll
          for (int c = 0; c < 2; ++c) atomicMax(&sm.redcol[seg / segs][2 * cp + c], fbits(cam[c]));
          __syncthreads();
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const float S = outer_scale<UE5M3>(bitsf(sm.redcol[seg / segs][2 * cp + c]));
            nc[c].S = S;
            const int64_t k = kc + c;
            if (cvalid && (seg % segs) == 0 && j.col_outer) j.col_outer[(g * j.K + k) * (j.M / ob) + mb / ob] = S;
          }
          __syncthreads();
          if (seg % segs == 0) {
            sm.redcol[seg / segs][2 * cp] = 0u;
            sm.redcol[seg / segs][2 * cp + 1] = 0u;
          }
        } else if (cvalid) {
#pragma unroll
          for (int c = 0; c < 2; ++c) nc[c].S = j.col_outer[(g * j.K + kc + c) * (j.M / ob) + mb / ob];
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          nc[c].none = false;
          nc[c].r = ieee_rcp(nc[c].S);
          nc[c].pos = positive(nc[c].S);
          nc[c].fast = positive_normal(nc[c].S);
        }
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float4 T;
        uint32_t sc;
        float x[16];
        if (shared_S) {
          Norm pass = nc[c];
          pass.none = true;  // values already normalized: inner amax is max |x'|
          sc = block_scale<UE5M3>(sm, cam[c], pass, T);
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] = v[c][i];
        } else {
          sc = block_scale<UE5M3>(sm, cam[c], nc[c], T);
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] = normalize(v[c][i], nc[c]);
        }
        const int64_t k = kc + c;
        const uint64_t n0 = (uint64_t)((g * j.K + k) * j.M + mb);
        uint32_t w0, w1;
        float deq[16];
        Norm dq = nc[c];
        dq.none = none;
        if (j.qdq_orient == 2) encode16<SR, true>(x, T, dq, j.seed, j.step, 1u, n0, w0, w1, deq);
        else encode16<SR, false>(x, T, dq, j.seed, j.step, 1u, n0, w0, w1, deq);
        if (cvalid) {
          if (j.col_codes) *reinterpret_cast<uint2*>(j.col_codes + n0 / 2) = make_uint2(w0, w1);
          if (j.col_scales) j.col_scales[n0 / 16] = (uint8_t)sc;
          if (j.qdq_orient == 2) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int64_t yi = (g * j.M + mb + i) * j.K + k;
              if (j.out_bf16) static_cast<uint16_t*>(j.y)[yi] = (uint16_t)(pack_bf16x2(deq[i], 0.0f) & 0xFFFFu);
              else static_cast<float*>(j.y)[yi] = deq[i];
            }
          }
        }
      }
    }
    __syncthreads();
  }
}

template <bool IN_BF16, bool SR, bool COL, bool UE5M3>
cudaError_t launch_t(const QuantJob& j, cudaStream_t st) {
  auto kern = ct_kernel<IN_BF16, SR, COL, UE5M3>;
  static int per_sm_cache[128] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int per_sm = (dev >= 0 && dev < 128) ? per_sm_cache[dev] : 0;
  if (per_sm == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    if (dev >= 0 && dev < 128) per_sm_cache[dev] = per_sm;
  }
  const int64_t tiles = j.G * ((j.M + TM - 1) / TM) * ((j.K + TK - 1) / TK);
  const int64_t cap = (int64_t)num_sms() * per_sm;
  kern<<<(int)(tiles < cap ? tiles : cap), NT, 0, st>>>(j);
  return cudaGetLastError();
}

template <bool IN_BF16, bool SR>
cudaError_t launch_c(const QuantJob& j, cudaStream_t st) {
  const bool col = j.do_col != 0;
  if (j.ue5m3) return col ? launch_t<IN_BF16, SR, true, true>(j, st) : launch_t<IN_BF16, SR, false, true>(j, st);
  return col ? launch_t<IN_BF16, SR, true, false>(j, st) : launch_t<IN_BF16, SR, false, false>(j, st);
}

}  // namespace

bool ct_supports(const QuantJob& j) {
  if (j.inner_2d) return false;
  if (j.s_src == S_IN_TILE && !(j.ob == 16 || j.ob == 32 || j.ob == 64)) return false;
  return true;
}

cudaError_t launch_ct(const QuantJob& j, cudaStream_t st) {
  if (j.in_bf16) return j.sr ? launch_c<true, true>(j, st) : launch_c<true, false>(j, st);
  return j.sr ? launch_c<false, true>(j, st) : launch_c<false, false>(j, st);
}

}  // namespace fp4q
