// k_ctl.cu -- the bf16 cast-transpose quantize in its whole-tile form: both
// orientations of NVFP4 / AMD-FP4 codes from one TMA-staged 128 x 64 tile
// ("Block-Scaled FP8 and FP4 Weight Quantization", section 3: the fused
// cast-transpose; section 6: a 2-D outer scale computed once and shared by
// both orientations; "NVFP4 / AMD-FP4 outer-block (two-level) scaling for FP4
// training", "Technical design": outer and inner scales), for the calls whose
// facts let every bound check fold away: M a multiple of 128, K of 64, bf16
// input, round-to-nearest, both orientations, linear scale layout, and an
// outer scale that is none, one per tensor, 1 x 64 / 64 x 1 or 64 x 64.
// Every other call takes the general cast-transpose kernel (k_ctb.cuh), which
// gives the same bits.
//
// Per tile, one CTA barrier.  Before it, every thread takes the block maxima
// it needs from the raw tile (rowwise: its half row, two 1 x 16 blocks;
// columnwise: its two 16 x 1 column blocks) and publishes what other warps
// need (the columns' 64-row maxima for 64 x 1 outer blocks, the warp's
// maximum for 64 x 64 blocks).  After it, the columnwise pass (its 16 words
// still in registers) and the rowwise pass (four 16-byte reloads) compute
// scales and codes.  The barrier also orders the previous tile's staged
// columnwise codes and scales before their stores (tensor store of the
// codes, 8-byte stores of the scales), so staging alternates between two
// buffers by tile parity, and the tile after next is copied into the slot
// whose last reader is past this barrier.
//
// The arithmetic is that of fp4q_block.cuh: x' = u / S by Markstein's
// correction from RN(1 / S), a = RN(amax / S) and v = RN(a / 6) two blocks
// per instruction (packed binary32 pairs), t = x' / s by the known-divisor
// method, E2M1 and E4M3 by the hardware conversions.  A warp whose outer
// scales or block maxima leave the range those sequences cover (maxima
// below 2^-90, non-finite inputs) takes the general per-block steps with
// div.rn for its tile.
#include "fp4q_block.cuh"
#include "fp4q_device.cuh"
#include "fp4q_internal.h"
#include "fp4q_tma.cuh"

namespace fp4q {
namespace {

constexpr int LT = 256;           // threads per CTA
constexpr int LM = 128, LK = 64;  // tile
constexpr int LRAW = LM * LK * 2; // bytes of one raw bf16 tile

// Shared memory (offsets from the 1024-byte aligned base)
struct LL {
  __host__ __device__ static constexpr int raw(int s) { return s * LRAW; }             // 2 slots
  __host__ __device__ static constexpr int ccs(int s) { return 2 * LRAW + s * 4096; }  // col codes, [64][64] swizzled
  __host__ __device__ static constexpr int sst(int s) { return 2 * LRAW + 2 * 4096 + s * 512; }  // col scales [64][8]
  static constexpr int tab = 2 * LRAW + 2 * 4096 + 2 * 512;                            // 256 x (s, zh, zl, -)
  __host__ __device__ static constexpr int red(int s) { return tab + 4096 + s * 1024; }  // [8 warps][32 lanes] u32
  static constexpr int ztab = tab + 4096 + 2 * 1024;                                   // 128 x (zh, zl)
  static constexpr int bars = ztab + 1024;                                             // 2 mbarriers
  static constexpr int total = bars + 16 + 1024;                                       // + alignment slack
};

// Outer-scale form of a launch
enum LO : int { LO_NONE = 0, LO_UNIFORM = 1, LO_1D = 2, LO_2D = 3 };

// Set by a tile wait that ran out; read and cleared by fp4q_device_status.
__device__ unsigned int g_ctl_timeout = 0;

__device__ __forceinline__ void issue_tile(const CUtensorMap* map, const TilePos& p, unsigned char* raw, uint64_t* bar) {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_tx(bar, (uint32_t)LRAW);
  tma_load3(raw, map, (int)p.k0, (int)p.m0, (int)p.g, bar);
}

// |max| of the 16 bf16 words of two column blocks (column 2 lane in the low
// halves, 2 lane + 1 in the high halves), NaN propagating, signs cleared.
__device__ __forceinline__ uint32_t colmax16(const uint32_t (&w)[16]) {
  uint32_t m = bf16x2_amax(w[0], w[1]);
#pragma unroll
  for (int i = 2; i < 16; i += 2) m = bf16x2_amax(m, bf16x2_amax(w[i], w[i + 1]));
  return m & 0x7FFF7FFFu;
}

// |max| of two row blocks (words a[0..1] and a[2..3]) as one word: block 0 in
// the low half, block 1 in the high half, NaN propagating, signs cleared.
__device__ __forceinline__ uint32_t rowmax2(const uint4 (&a)[4]) {
  uint32_t m[2];
#pragma unroll
  for (int b = 0; b < 2; ++b)
    m[b] = bf16x2_amax(bf16x2_amax(bf16x2_amax(a[2 * b].x, a[2 * b].y), bf16x2_amax(a[2 * b].z, a[2 * b].w)),
                       bf16x2_amax(bf16x2_amax(a[2 * b + 1].x, a[2 * b + 1].y),
                                   bf16x2_amax(a[2 * b + 1].z, a[2 * b + 1].w)));
  return bf16x2_amax(__byte_perm(m[0], m[1], 0x5410), __byte_perm(m[0], m[1], 0x7632)) & 0x7FFF7FFFu;
}

// A packed pair of |max| bf16 halves holds a non-finite value.
__device__ __forceinline__ bool nonfinite2(uint32_t m) {
  return (m & 0xFFFFu) >= 0x7F80u || (m >> 16) >= 0x7F80u;
}

// x' for a pair of values (lo, hi) packed from a bf16x2 word w.
template <int NM>
__device__ __forceinline__ uint64_t norm2(uint32_t w, uint64_t P, uint64_t Q) {
  if (NM == NM_MARK) return markstein2(pk2(nbf16lo(w), nbf16hi(w)), P, Q);
  if (NM == NM_BMR) return bmr2(pk2(bf16lo(w), bf16hi(w)), P, Q);
  return pk2(bf16lo(w), bf16hi(w));
}

// Inner scales of two blocks at once: a = RN(am / S) (or am), v = RN(a /
// 6), codes (low byte block 0), and their table entries.  am2: the blocks'
// maxima as bf16 halves.
template <bool UE5M3, int NM>
__device__ __forceinline__ uint32_t scales2(const float4* tab, uint32_t am2, uint64_t P, uint64_t Q, float4& T0,
                                            float4& T1) {
  const float m0 = bitsf(am2 << 16), m1 = bitsf(am2 & 0xFFFF0000u);
  uint64_t a2;
  if (NM == NM_MARK) a2 = markstein2(pk2(bitsf(fbits(m0) | 0x80000000u), bitsf(fbits(m1) | 0x80000000u)), P, Q);
  else if (NM == NM_BMR) a2 = bmr2(pk2(m0, m1), P, Q);
  else a2 = pk2(m0, m1);
  const uint64_t v2 = bmr2(a2, pk2(bitsf(kSixHi), bitsf(kSixHi)), pk2(bitsf(kSixLo), bitsf(kSixLo)));
  float v0, v1;
  upk2(v2, v0, v1);
  uint32_t sc;
  if (UE5M3) {
    sc = enc_ue5m3(v0) | (enc_ue5m3(v1) << 8);
  } else {
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\tcvt.u32.u16 %0, t;\n\t}" : "=r"(sc) : "f"(v1), "f"(v0));
  }
  T0 = tab[sc & 0xFFu];
  T1 = tab[sc >> 8];
  return sc;
}

// Codes of one rowwise block from its 8 words (4 per uint4): x' (NM) and
// t = x' / s, two values per instruction; element 2i in the low nibble of
// byte i.
template <int NM>
__device__ __forceinline__ void row_codes16(const uint4& p, const uint4& q, uint64_t P, uint64_t Q, const float4& T,
                                            uint32_t& w0, uint32_t& w1) {
  const uint64_t ZH2 = pk2(T.y, T.y), ZL2 = pk2(T.z, T.z);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4& v = h ? q : p;
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
    float t[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) upk2(bmr2(norm2<NM>(wd[i], P, Q), ZH2, ZL2), t[2 * i], t[2 * i + 1]);
    (h ? w1 : w0) = e2m1x8_rne(t);
  }
}

// Codes of the two column blocks of a lane from its 16 words (word i: row i,
// column 2 lane in the low half, 2 lane + 1 in the high half): the pairs run
// across the two columns, each with its own outer and inner scale; c[0],
// c[1]: column 2 lane, rows 0-7 and 8-15; c[2], c[3]: column 2 lane + 1.
template <int NM>
__device__ __forceinline__ void col_codes16(const uint32_t (&w)[16], uint64_t P, uint64_t Q, const float4& T0,
                                            const float4& T1, uint32_t (&c)[4]) {
  const uint64_t ZH2 = pk2(T0.y, T1.y), ZL2 = pk2(T0.z, T1.z);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float t0[8], t1[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) upk2(bmr2(norm2<NM>(w[8 * h + i], P, Q), ZH2, ZL2), t0[i], t1[i]);
    c[h] = e2m1x8_rne(t0);
    c[2 + h] = e2m1x8_rne(t1);
  }
}

// The general per-block steps (div.rn where the FMA sequences do not reach):
// 16 values u (as -u when NEG), block maximum am, outer scale S, R = 1 / S.
template <bool UE5M3, bool NEG>
__device__ __forceinline__ uint32_t slow_block(const float4* tab, const float (&v)[16], float am, float S, float R,
                                               bool none, const PhiloxKeys& K, uint32_t& w0, uint32_t& w1) {
  Norm n;
  n.none = none;
  n.S = S;
  n.r = R;
  n.pos = none || positive(S);
  n.fast = !none && positive_normal(S) && positive_normal(R);
  struct {
    const float4* tab;
  } tv{tab};
  float4 T;
  const uint32_t sc = block_scale<UE5M3>(tv, am, n, T);
  float x[16], dq[16];
  if (NEG) normalize16_neg<false>(v, x, n);
  else normalize16<false>(v, x, n);
  encode16<false, false>(x, T, n, K, 0u, 0u, 0ull, w0, w1, dq);
  return sc;
}

// Fast-path mode of a pass, warp-uniform: the general per-block steps, or
// NM_NONE / NM_MARK / NM_BMR.
constexpr int PM_SLOW = -1;

template <bool UE5M3, int LOF>
__global__ void __launch_bounds__(LT, LOF == LO_2D ? 3 : 4) ctl_kernel(const QuantJob j, const __grid_constant__ CUtensorMap tmap,
                                                                        const __grid_constant__ CUtensorMap cmap) {
  constexpr bool OUTER = LOF != LO_NONE;
  pdl_wait_then_release();
  extern __shared__ __align__(16) unsigned char smem_dyn[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  float4* tab = reinterpret_cast<float4*>(smem + LL::tab);
  float2* ztab = reinterpret_cast<float2*>(smem + LL::ztab);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LL::bars);

  TileIter cur;
  cur.init<LM>(j);
  if (t == 0) {
    mbar_init(&bars[0]);
    mbar_init(&bars[1]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (t == 0) {  // the first two tiles; later tiles take a slot once its reads are past a barrier
    if (cur.valid()) issue_tile(&tmap, cur.pos<LM>(), smem + LL::raw(0), &bars[0]);
    if (cur.idx + (int)gridDim.x < cur.ntiles)
      issue_tile(&tmap, cur.pos_of<LM>(cur.idx + (int)gridDim.x), smem + LL::raw(1), &bars[1]);
  }
  build_scale_table<UE5M3>(tab, t, LT);
  if (OUTER) build_ztab(ztab, t);
  const float denh = bitsf(UE5M3 ? kDenHiU5 : kDenHiE4), denl = bitsf(UE5M3 ? kDenLoU5 : kDenLoE4);

  // rowwise: thread t owns row t / 2, columns 32 (t mod 2) .. + 31 (two
  // blocks); its four 16-byte chunks sit at these swizzled offsets
  const int rr = t >> 1, rh = t & 1;
  uint32_t roff[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) roff[q] = (uint32_t)(rr * 128 + (((4 * rh + q) ^ (rr & 7)) << 4));
  // columnwise: warp w owns rows 16 w .. + 15, lane l columns 2 l, 2 l + 1
  const uint32_t coff = (uint32_t)(warp * 2048 + (lane & 3) * 4);
  const int cunit = lane >> 2;
  __syncthreads();

  // one scale for the whole tensor: from the amax in the workspace, or given
  float S_u = 1.0f, R_u = 1.0f, zh_u = 0.0f, zl_u = 0.0f;
  int um = NM_MARK;  // the uniform scale's fast mode (CTA-uniform)
  bool u_ok = true;  // S_u and 1 / S_u normal
  if (LOF == LO_UNIFORM) {
    uint32_t Ab = 0;
    if (j.s_src == S_TENSORWISE_WS) {
      Ab = *j.tw_amax;
      S_u = ieee_div(bitsf(Ab), UE5M3 ? 688128.0f : 2688.0f);
      if (blockIdx.x == 0 && t == 0 && j.tile_outer) j.tile_outer[0] = S_u;
    } else {
      S_u = j.tile_outer[0];
    }
    R_u = ieee_rcp(S_u);
    u_ok = positive_normal(S_u) && positive_normal(R_u);
    // an amax that is a bf16 value (every bf16 tensor's is) in range
    if (j.s_src == S_TENSORWISE_WS && (Ab & 0xFFFFu) == 0u && Ab >= kTiny && fbits(S_u) < 0x6C800000u) {
      um = NM_BMR;
      zsplit(Ab, S_u, ztab, zh_u, zl_u);
    }
  }

  int slot = 0;
  uint32_t phase = 0;
  int pg = 0, pm0 = 0, pk0 = 0;  // the previous tile
  int prev_par = 0;
  bool have_prev = false;
  for (int it = 0; cur.valid(); ++it) {
    const int par = it & 1;
    const int tg = cur.g, tm0 = cur.tm * LM, tk0 = cur.tk * LK;  // this tile
    const int after = cur.idx + 2 * (int)gridDim.x;              // the tile that takes this slot next
    cur.next();
    const unsigned char* raw = smem + LL::raw(slot);
    // a wait that runs out raises the error flag; the walk goes on (every
    // later wait is bounded and every barrier is still reached)
    if (!mbar_wait(&bars[slot], phase, 1u << 22)) atomicExch(&g_ctl_timeout, 1u);
    uint32_t* red = reinterpret_cast<uint32_t*>(smem + LL::red(par));
    const int64_t row = (int64_t)tg * j.M + tm0 + rr;  // this thread's row of the [G M, K] view

    // rowwise: scales, codes and stores of the thread's two blocks; mode:
    // the fast form (P, Q its constants), or PM_SLOW
    auto row_pass = [&](const uint4 (&a)[4], uint32_t ram, int mode, float S, float R, uint64_t P, uint64_t Q) {
      uint32_t c[4], sc;
      if (mode == NM_BMR || mode == NM_NONE) {
        float4 T0, T1;
        if (LOF == LO_NONE) {
          sc = scales2<UE5M3, NM_NONE>(tab, ram, P, Q, T0, T1);
          row_codes16<NM_NONE>(a[0], a[1], P, Q, T0, c[0], c[1]);
          row_codes16<NM_NONE>(a[2], a[3], P, Q, T1, c[2], c[3]);
        } else {
          sc = scales2<UE5M3, NM_BMR>(tab, ram, P, Q, T0, T1);
          row_codes16<NM_BMR>(a[0], a[1], P, Q, T0, c[0], c[1]);
          row_codes16<NM_BMR>(a[2], a[3], P, Q, T1, c[2], c[3]);
        }
      } else if (OUTER && mode == NM_MARK) {
        float4 T0, T1;
        sc = scales2<UE5M3, NM_MARK>(tab, ram, P, Q, T0, T1);
        row_codes16<NM_MARK>(a[0], a[1], P, Q, T0, c[0], c[1]);
        row_codes16<NM_MARK>(a[2], a[3], P, Q, T1, c[2], c[3]);
      } else {
        const float am0 = bitsf(ram << 16), am1 = bitsf(ram & 0xFFFF0000u);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const uint32_t wd[8] = {a[2 * b].x, a[2 * b].y, a[2 * b].z, a[2 * b].w,
                                  a[2 * b + 1].x, a[2 * b + 1].y, a[2 * b + 1].z, a[2 * b + 1].w};
          float u[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            u[2 * i] = bf16lo(wd[i]);
            u[2 * i + 1] = bf16hi(wd[i]);
          }
          const uint32_t s1 = slow_block<UE5M3, false>(tab, u, b ? am1 : am0, S, R, !OUTER, j.srk, c[2 * b], c[2 * b + 1]);
          sc = b ? (sc | (s1 << 8)) : s1;
        }
      }
      const int64_t e = row * j.K + tk0 + 32 * rh;  // flat index of the thread's first element
      *reinterpret_cast<uint4*>(j.row_codes + (e >> 1)) = make_uint4(c[0], c[1], c[2], c[3]);
      *reinterpret_cast<uint16_t*>(j.row_scales + (e >> 4)) = (uint16_t)sc;
    };
    // Markstein's form with a scale not taken from a bf16 amax: every
    // block maximum must be 0 or at least 2^-90 and a = RN(am / S) < 2^126
    auto mark_ok = [&](uint32_t am2, float S, float R) {
      float d0, d1;
      return __all_sync(0xFFFFFFFFu, u_ok && fast_block(bitsf(am2 << 16), S, R, d0) &&
                                         fast_block(bitsf(am2 & 0xFFFF0000u), S, R, d1));
    };

    // ------------------------------------------ before the barrier: every read of the raw tile
    uint4 a[4];  // row rr, columns 32 rh .. + 31
#pragma unroll
    for (int q = 0; q < 4; ++q) a[q] = *reinterpret_cast<const uint4*>(raw + roff[q]);
    uint32_t ram = rowmax2(a);  // |max| of the two row blocks: block 0 low half, block 1 high half
    if (nonfinite2(ram)) {      // sanitize (NaN -> +0, +-inf -> +-largest finite)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        a[q].x = sanitize_bf16x2(a[q].x); a[q].y = sanitize_bf16x2(a[q].y);
        a[q].z = sanitize_bf16x2(a[q].z); a[q].w = sanitize_bf16x2(a[q].w);
      }
      ram = rowmax2(a);
    }
    if (LOF == LO_2D) {  // the warp's 16 x 64 maximum, for the 64 x 64 block's scale
      uint32_t m = umax(ram & 0xFFFFu, ram >> 16);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = umax(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      if (lane == 0) red[warp * 32] = m;
    } else if (LOF == LO_NONE) {  // the rowwise pass needs nothing from other warps: done here
      row_pass(a, ram, NM_NONE, 1.0f, 1.0f, 0ull, 0ull);
    } else if (LOF == LO_UNIFORM) {
      if (um == NM_BMR) row_pass(a, ram, NM_BMR, S_u, R_u, pk2(zh_u, zh_u), pk2(zl_u, zl_u));
      else row_pass(a, ram, mark_ok(ram, S_u, R_u) ? NM_MARK : PM_SLOW, S_u, R_u, pk2(S_u, S_u), pk2(-R_u, -R_u));
    } else {  // 1 x 64: the row's 64 columns are this thread's two blocks and its partner's
      uint32_t g = umax(ram & 0xFFFFu, ram >> 16);
      g = umax(g, __shfl_xor_sync(0xFFFFFFFFu, g, 1)) << 16;
      const float S = div_bmr(bitsf(g), denh, denl);  // exact for g >= 2^-90
      float* so = j.row_outer + row * (j.K >> 6) + (tk0 >> 6);
      if (__all_sync(0xFFFFFFFFu, g >= kTiny && fbits(S) < 0x6C800000u)) {
        if (rh == 0) *so = S;
        float zh, zl;
        zsplit(g, S, ztab, zh, zl);
        row_pass(a, ram, NM_BMR, S, 1.0f, pk2(zh, zh), pk2(zl, zl));
      } else {
        const float S1 = outer_scale<UE5M3>(bitsf(g));
        if (rh == 0) *so = S1;
        row_pass(a, ram, PM_SLOW, S1, ieee_rcp(S1), 0ull, 0ull);
      }
    }
    uint32_t wv[16];  // rows 16 warp .. + 15, columns 2 lane (low halves) and 2 lane + 1 (high)
    {
      const unsigned char* rb = raw + coff;
#pragma unroll
      for (int i = 0; i < 16; ++i) wv[i] = *reinterpret_cast<const uint32_t*>(rb + i * 128 + ((cunit ^ (i & 7)) << 4));
    }
    uint32_t cam = colmax16(wv);
    if (nonfinite2(cam)) {
#pragma unroll
      for (int i = 0; i < 16; ++i) wv[i] = sanitize_bf16x2(wv[i]);
      cam = colmax16(wv);
    }
    if (LOF == LO_1D) red[warp * 32 + lane] = cam;
    // the store that read this staging parity two tiles ago is done with it
    if (t == 0) bulk_wait_read_0();
    __syncthreads();

    if (t == 0) {  // refill the slot, store the previous tile's staged column codes
      if (after < cur.ntiles) issue_tile(&tmap, cur.pos_of<LM>(after), smem + LL::raw(slot), &bars[slot]);
      if (have_prev) {
        tma_store3(&cmap, smem + LL::ccs(par ^ 1), pm0 >> 1, pk0, pg);
        bulk_commit();
      }
    }
    if (have_prev && t < 64) {  // the previous tile's column scales: 8 bytes per column
      const uint2 v = *reinterpret_cast<const uint2*>(smem + LL::sst(par ^ 1) + t * 8);
      *reinterpret_cast<uint2*>(j.col_scales + ((int64_t)pg * j.K + pk0 + t) * (j.M >> 4) + (pm0 >> 4)) = v;
    }
    if (++slot == 2) {
      slot = 0;
      phase ^= 1u;
    }

    // ---------------------------------------- after the barrier: registers and staging only
    float S2f = 1.0f, zh2 = 0.0f, zl2 = 0.0f;  // the 64 x 64 block's scale (2-D): both orientations
    bool f2 = true;
    if (LOF == LO_2D) {
      const uint32_t* rq = red + (warp >> 2) * 128;
      const uint32_t A = umax(umax(rq[0], rq[32]), umax(rq[64], rq[96])) << 16;
      S2f = div_bmr(bitsf(A), denh, denl);
      f2 = A >= kTiny && fbits(S2f) < 0x6C800000u;  // uniform over the CTA half
      if (f2) zsplit(A, S2f, ztab, zh2, zl2);
      else S2f = outer_scale<UE5M3>(bitsf(A));
      if ((warp & 3) == 0 && lane == 0)
        j.tile_outer[((int64_t)tg * (j.M >> 6) + (tm0 >> 6) + (warp >> 2)) * (j.K >> 6) + (tk0 >> 6)] = S2f;
      if (f2) row_pass(a, ram, NM_BMR, S2f, 1.0f, pk2(zh2, zh2), pk2(zl2, zl2));
      else row_pass(a, ram, PM_SLOW, S2f, ieee_rcp(S2f), 0ull, 0ull);
    }
    // ----------------------------------------------------------- columnwise
    {
      float S[2] = {1.0f, 1.0f}, R[2] = {1.0f, 1.0f};
      int mode = NM_NONE;
      uint64_t P = 0ull, Q = 0ull;
      if (LOF == LO_UNIFORM) {
        S[0] = S[1] = S_u;
        R[0] = R[1] = R_u;
        if (um == NM_BMR) {
          mode = NM_BMR;
          P = pk2(zh_u, zh_u);
          Q = pk2(zl_u, zl_u);
        } else {
          mode = mark_ok(cam, S_u, R_u) ? NM_MARK : PM_SLOW;
          P = pk2(S_u, S_u);
          Q = pk2(-R_u, -R_u);
        }
      } else if (LOF == LO_2D) {
        S[0] = S[1] = S2f;
        if (!f2) R[0] = R[1] = ieee_rcp(S2f);  // the general steps take 1 / S
        mode = f2 ? NM_BMR : PM_SLOW;
        P = pk2(zh2, zh2);
        Q = pk2(zl2, zl2);
      } else if (LOF == LO_1D) {  // the columns' 64-row maxima over the 4 warps of this half
        const uint32_t* rq = red + (warp >> 2) * 128 + lane;
        const uint32_t g = bf16x2_amax(bf16x2_amax(rq[0], rq[32]), bf16x2_amax(rq[64], rq[96])) & 0x7FFF7FFFu;
        const uint32_t g0 = g << 16, g1 = g & 0xFFFF0000u;
        float Sv0, Sv1;
        upk2(bmr2(pk2(bitsf(g0), bitsf(g1)), pk2(denh, denh), pk2(denl, denl)), Sv0, Sv1);
        S[0] = Sv0;  // exact for g >= 2^-90
        S[1] = Sv1;
        if (__all_sync(0xFFFFFFFFu, umin(g0, g1) >= kTiny && umax(fbits(S[0]), fbits(S[1])) < 0x6C800000u)) {
          float zh0, zl0, zh1, zl1;
          zsplit(g0, S[0], ztab, zh0, zl0);
          zsplit(g1, S[1], ztab, zh1, zl1);
          mode = NM_BMR;
          P = pk2(zh0, zh1);
          Q = pk2(zl0, zl1);
        } else {
          mode = PM_SLOW;
          S[0] = outer_scale<UE5M3>(bitsf(g0));
          S[1] = outer_scale<UE5M3>(bitsf(g1));
          R[0] = ieee_rcp(S[0]);
          R[1] = ieee_rcp(S[1]);
        }
        if ((warp & 3) == 0) {
          const int64_t M64 = j.M >> 6;
          float* d = j.col_outer + ((int64_t)tg * j.K + tk0 + 2 * lane) * M64 + (tm0 >> 6) + (warp >> 2);
          d[0] = S[0];
          d[M64] = S[1];
        }
      }
      uint32_t c[4], sc;
      if (mode == NM_BMR || mode == NM_NONE) {
        float4 T0, T1;
        if (LOF == LO_NONE) {
          sc = scales2<UE5M3, NM_NONE>(tab, cam, P, Q, T0, T1);
          col_codes16<NM_NONE>(wv, P, Q, T0, T1, c);
        } else {
          sc = scales2<UE5M3, NM_BMR>(tab, cam, P, Q, T0, T1);
          col_codes16<NM_BMR>(wv, P, Q, T0, T1, c);
        }
      } else if (LOF == LO_UNIFORM && mode == NM_MARK) {
        float4 T0, T1;
        sc = scales2<UE5M3, NM_MARK>(tab, cam, P, Q, T0, T1);
        col_codes16<NM_MARK>(wv, P, Q, T0, T1, c);
      } else {
        const float am0 = bitsf(cam << 16), am1 = bitsf(cam & 0xFFFF0000u);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          float u[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) u[i] = k ? bf16hi(wv[i]) : bf16lo(wv[i]);
          const uint32_t s1 = slow_block<UE5M3, false>(tab, u, k ? am1 : am0, S[k], R[k], !OUTER, j.srk, c[2 * k], c[2 * k + 1]);
          sc = k ? (sc | (s1 << 8)) : s1;
        }
      }
      // stage: codes of column 2 lane + k, rows 16 warp .. + 15 go to row
      // 2 lane + k of the tensor-store box at byte 8 warp, whose 16-byte
      // chunk the 64-byte swizzle XORs with (row / 2) mod 4 = lane mod 4
      unsigned char* cb = smem + LL::ccs(par);
      unsigned char* sb = smem + LL::sst(par);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        *reinterpret_cast<uint2*>(cb + ((((2 * lane + k) << 6) + 8 * warp) ^ ((lane & 3) << 4))) =
            make_uint2(c[2 * k], c[2 * k + 1]);
        sb[(2 * lane + k) * 8 + warp] = (uint8_t)(sc >> (8 * k));
      }
      fence_proxy_async();
    }
    pg = tg;
    pm0 = tm0;
    pk0 = tk0;
    prev_par = par;
    have_prev = true;
  }
  // the last tile's columnwise codes and scales
  __syncthreads();
  if (have_prev) {
    if (t == 0) {
      tma_store3(&cmap, smem + LL::ccs(prev_par), pm0 >> 1, pk0, pg);
      bulk_commit();
    }
    if (t < 64) {
      const uint2 v = *reinterpret_cast<const uint2*>(smem + LL::sst(prev_par) + t * 8);
      *reinterpret_cast<uint2*>(j.col_scales + ((int64_t)pg * j.K + pk0 + t) * (j.M >> 4) + (pm0 >> 4)) = v;
    }
  }
  if (t == 0) bulk_wait_all();
}

template <bool UE5M3, int LOF>
cudaError_t launch_ctl_t(const QuantJob& j, const CUtensorMap& map, const CUtensorMap& cmap, cudaStream_t st) {
  auto kern = ctl_kernel<UE5M3, LOF>;
  static int per_sm_cache[128] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 128) dev = 0;
  int& per_sm = per_sm_cache[dev];
  if (per_sm == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LL::total);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, LT, LL::total);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
  }
  const int64_t tiles = j.G * (j.M / LM) * (j.K / LK);
  const int64_t cap = (int64_t)num_sms() * per_sm;
  return launch_pdl(kern, dim3((unsigned)(tiles < cap ? tiles : cap)), dim3(LT), (size_t)LL::total, st, j, map, cmap);
}

template <bool UE5M3>
cudaError_t launch_ctl_f(const QuantJob& j, int lof, const CUtensorMap& map, const CUtensorMap& cmap, cudaStream_t st) {
  switch (lof) {
    case LO_NONE: return launch_ctl_t<UE5M3, LO_NONE>(j, map, cmap, st);
    case LO_UNIFORM: return launch_ctl_t<UE5M3, LO_UNIFORM>(j, map, cmap, st);
    case LO_1D: return launch_ctl_t<UE5M3, LO_1D>(j, map, cmap, st);
    default: return launch_ctl_t<UE5M3, LO_2D>(j, map, cmap, st);
  }
}

bool aligned_to(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0u; }

}  // namespace

// The whole-tile form, when the call's facts allow it (false: the caller
// takes the general cast-transpose kernel).  FP4Q_NO_CTL_KERNEL=1 turns it
// off (the parity tests run every kernel that can take a case).
bool launch_ctl(const QuantJob& j, cudaStream_t st, cudaError_t* err) {
  if (!j.in_bf16 || !j.do_row || !j.do_col || j.sr || j.inner_2d || j.residual || j.qdq_orient || j.ngroups ||
      j.col_rht || j.rsl.mma || j.csl.mma || j.M % LM || j.K % LK)
    return false;
  if (!aligned_to(j.x, 16) || (j.ld * 2) % 16 || !aligned_to(j.row_codes, 16) || !aligned_to(j.row_scales, 2) ||
      !aligned_to(j.col_codes, 16) || !aligned_to(j.col_scales, 8))
    return false;
  int lof;
  if (j.s_src == S_ONE) lof = LO_NONE;
  else if (j.mode == 1) lof = LO_UNIFORM;  // tensorwise: from the workspace amax or a given scale
  else if (j.s_src == S_IN_TILE && j.ob == 64) lof = j.outer_2d ? LO_2D : LO_1D;
  else return false;
  if (getenv_flag("FP4Q_NO_CTL_KERNEL")) return false;
  CUtensorMap map, cmap;
  if (!make_bf16_tile_map(j, &map, LM) || !make_col_map(j, &cmap)) return false;
  *err = j.ue5m3 ? launch_ctl_f<true>(j, lof, map, cmap, st) : launch_ctl_f<false>(j, lof, map, cmap, st);
  return true;
}

cudaError_t ctl_timeout_flag(uint32_t* v, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(v, g_ctl_timeout, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_ctl_timeout, &z, sizeof z);
  }
  return e;
}

}  // namespace fp4q
