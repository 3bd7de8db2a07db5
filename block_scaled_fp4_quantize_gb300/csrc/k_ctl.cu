// k_ctl.cu -- the bf16 cast-transpose quantize in its whole-tile form: both
// orientations of NVFP4 / AMD-FP4 codes from one TMA-staged 128 x 64 tile
// ("Block-Scaled FP8 and FP4 Weight Quantization", section 3: the fused
// cast-transpose; section 6: a 2-D outer scale computed once and shared by
// both orientations; "NVFP4 / AMD-FP4 outer-block (two-level) scaling for FP4
// training", "Technical design": outer and inner scales), for the calls whose
// facts let every bound check fold away: M a multiple of 128 (64 for ragged
// groups), K of 64, bf16 input, round-to-nearest, both orientations, linear
// scale layout, and an outer scale that is none, one per tensor (from the
// tensorwise amax), 1 x 64 / 64 x 1 or 64 x 64.  Every other call takes the
// general cast-transpose kernel (k_ctb.cuh), which gives the same bits.
//
// Per tile, one CTA barrier.  Before it, every thread reads what it needs
// from the raw tile (rowwise: its half row, two 1 x 16 blocks; columnwise:
// its two 16 x 1 column blocks, kept in registers) and publishes what other
// warps need (the columns' 64-row maxima for 64 x 1 outer blocks, the warp's
// maximum for 64 x 64 blocks).  After it, the rowwise and columnwise passes
// compute scales and codes and stage the codes in shared memory.  The barrier
// also orders the previous tile's staged codes and scales before their
// stores (tensor stores of the rowwise and columnwise codes, 8-byte stores of
// the column scales), so staging alternates between two buffers by tile
// parity, and the tile after next is copied into the slot whose last reader
// is past this barrier.  Staging the rowwise codes for tensor stores costs
// the shared memory of a fourth CTA per SM and still measured faster than
// 16-byte stores from registers at four CTAs.
//
// The arithmetic.  The outer amax A of bf16 data is a bf16 value, so S =
// RN(A / (scale_max * 6)) has one of 128 significands (set by the 7 mantissa
// bits m of A) and an inner scale s one of 8 (its 3 mantissa bits j).  For
// every pair (j, m) the table of fp4q_pairtab.cuh holds multipliers c1, c2
// with which RN(RN(u c1) c2) has the E2M1 code of the two rounded divisions
// RN(RN(u / S) / s) for every bf16 u (checked by enumeration): two packed
// multiplies per pair of values.  The inner scale itself, a = RN(am / S) and
// v = RN(a / 6), comes from the known-divisor method (exact for bf16
// dividends), its E4M3 code from the hardware conversion.  The table rows sit
// in shared memory with the exponent of S folded in (one bulk copy of a
// precomputed image per CTA), so a block's multipliers are two table loads
// and two integer adds.  A warp whose outer amax lies outside [2^-90, 2^101)
// (2^109 for UE5M3 scales), where the scaled entries stay normal, takes the
// general per-block steps with div.rn.
#include "fp4q_block.cuh"
#include "fp4q_device.cuh"
#include "fp4q_internal.h"
#include "fp4q_pair.cuh"
#include "fp4q_tma.cuh"

#include <type_traits>

namespace fp4q {
namespace {

constexpr int LT = 256;           // threads per CTA
constexpr int LM = 128, LK = 64;  // tile
constexpr int LRAW = LM * LK * 2; // bytes of one raw bf16 tile
static_assert(LT == 256, "one thread per scale code builds the code tables");

// Shared memory (offsets from the 1024-byte aligned base).  Buffers that
// tensor copies read or write start on 1024-byte boundaries (the copies need
// 128, the swizzled loads 1024).
struct LL {
  __host__ __device__ static constexpr int raw(int s) { return s * LRAW; }                   // 2 input slots
  __host__ __device__ static constexpr int ccs(int s) { return 2 * LRAW + s * 4096; }        // col codes, [64][64] swizzled
  __host__ __device__ static constexpr int rcs(int s) { return 2 * LRAW + 8192 + s * 4096; } // row codes [128][32]
  __host__ __device__ static constexpr int sst(int s) { return 2 * LRAW + 16384 + s * 512; }  // col scales [64][8]
  __host__ __device__ static constexpr int red(int s) { return 2 * LRAW + 17408 + s * 1024; }  // [8 warps][32 lanes] u32
  static constexpr int pt = 2 * LRAW + 19456;  // 10 rows x 128 x (u32, u32), rows 1024 bytes apart
                                               // (no outer scale: 256 x (c1, c2) by scale code)
  static constexpr int ctab = pt + 10240;      // 256 x u32: scale code -> row and exponent of 1 / s
  static constexpr int bars = ctab + 1024;     // 3 mbarriers: two input slots, the tables
  static constexpr int total = bars + 32 + 1024;  // + alignment slack
};
static_assert(LL::rcs(0) % 1024 == 0 && LL::rcs(1) % 1024 == 0 && LL::ccs(1) % 1024 == 0,
              "tensor-copy staging alignment");
static_assert(LL::pt % 16 == 0 && LL::bars % 8 == 0, "bulk-copy and mbarrier alignment");
static_assert(LL::sst(0) == LL::rcs(2) && LL::red(0) == LL::sst(2) && LL::pt == LL::red(2), "regions back to back");
// resident CTAs per SM (shared memory: 3 x LL::total fit)
constexpr int kCtlPerSm = 3;

// Outer-scale form of a launch
enum LO : int { LO_NONE = 0, LO_UNIFORM = 1, LO_1D = 2, LO_2D = 3 };

// Set by a tile wait that ran out; read and cleared by fp4q_device_status.
__device__ unsigned int g_ctl_timeout = 0;

// Column loads of rows c and c + 8 (shared-memory offset OFF of the slot;
// ca: the lane's address in slot 0, row 0; the 128-byte swizzle XORs the
// 16-byte chunk index, address bits 4..6, with the row mod 8).
template <int OFF, int c>
__device__ __forceinline__ void lds_col(uint32_t ca, uint32_t (&wv)[16]) {
  const uint32_t a = ca ^ ((uint32_t)c << 4);
  asm volatile("ld.shared.b32 %0, [%1+%2];" : "=r"(wv[c]) : "r"(a), "n"(OFF + c * 128) : "memory");
  asm volatile("ld.shared.b32 %0, [%1+%2];" : "=r"(wv[c + 8]) : "r"(a), "n"(OFF + c * 128 + 1024) : "memory");
}

// One bulk copy of `bytes` (a multiple of 16, both addresses 16-byte
// aligned) into shared memory, completion on an mbarrier.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

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

// A packed pair of |max| bf16 halves (each at most 0x7FFF) holds a
// non-finite value: a half at or above 0x7F80 carries into its bit 15.
__device__ __forceinline__ bool nonfinite2(uint32_t m) { return ((m + 0x00800080u) & 0x80008000u) != 0u; }

// Inner-scale codes of two blocks (block 0 in the low byte) from their
// maxima am2 (bf16 halves): a = am, or RN(am / S) from the split reciprocal
// pairs (ZH, ZL); v = RN(a / 6); the E4M3 / UE5M3 code of v.
template <bool UE5M3, bool OUTER>
__device__ __forceinline__ uint32_t codes2(uint32_t am2, uint64_t ZH, uint64_t ZL) {
  uint64_t a2 = pk2(bitsf(am2 << 16), bitsf(am2 & 0xFFFF0000u));
  if (OUTER) a2 = bmr2(a2, ZH, ZL);
  float v0, v1;
  upk2(bmr2(a2, pk2(bitsf(kSixHi), bitsf(kSixHi)), pk2(bitsf(kSixLo), bitsf(kSixLo))), v0, v1);
  if (UE5M3) return enc_ue5m3(v0) | (enc_ue5m3(v1) << 8);
  uint32_t sc;
  asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\tcvt.u32.u16 %0, t;\n\t}" : "=r"(sc) : "f"(v1), "f"(v0));
  return sc;
}

// t = RN(RN(u c1) c2) for the pair of values of bf16x2 word w
__device__ __forceinline__ uint64_t t2(uint32_t w, uint64_t C1, uint64_t C2) {
  return mul2(mul2(pk2(bf16lo(w), bf16hi(w)), C1), C2);
}

// Codes of one rowwise block from its 8 words (4 per uint4); element 2i in
// the low nibble of byte i.
__device__ __forceinline__ void row_codes16(const uint4& p, const uint4& q, uint64_t C1, uint64_t C2, uint32_t& w0,
                                            uint32_t& w1) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4& v = h ? q : p;
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
    float t[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) upk2(t2(wd[i], C1, C2), t[2 * i], t[2 * i + 1]);
    (h ? w1 : w0) = e2m1x8_rne(t);
  }
}

// Codes of the two column blocks of a lane from its 16 words (word i: row i,
// column 2 lane in the low half, 2 lane + 1 in the high half): the pairs run
// across the two columns, each with its own multipliers; c[0], c[1]: column
// 2 lane, rows 0-7 and 8-15; c[2], c[3]: column 2 lane + 1.
__device__ __forceinline__ void col_codes16(const uint32_t (&w)[16], uint64_t C1, uint64_t C2, uint32_t (&c)[4]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float t0[8], t1[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) upk2(t2(w[8 * h + i], C1, C2), t0[i], t1[i]);
    c[h] = e2m1x8_rne(t0);
    c[2 + h] = e2m1x8_rne(t1);
  }
}


// The general per-block steps (div.rn where the FMA sequences do not reach):
// 16 values u, block maximum am, outer scale S, R = 1 / S.
template <bool UE5M3>
__device__ __forceinline__ uint32_t slow_block(const float (&v)[16], float am, float S, float R, bool none,
                                               const PhiloxKeys& K, uint32_t& w0, uint32_t& w1) {
  Norm n;
  n.none = none;
  n.S = S;
  n.r = R;
  n.pos = none || positive(S);
  n.fast = !none && positive_normal(S) && positive_normal(R);
  struct {
    EntryCalc<UE5M3> tab;
  } tv;
  float4 T;
  const uint32_t sc = block_scale<UE5M3>(tv, am, n, T);
  float x[16], dq[16];
  normalize16<false>(v, x, n);
  encode16<false, false>(x, T, n, K, 0u, 0u, 0ull, w0, w1, dq);
  return sc;
}

// GR: ragged groups (rows [goff[e], goff[e + 1]) form group e, quantized as a
// matrix of its own, every group a whole number of 64-row outer blocks): the
// walk covers each group's 128-row tiles, the last one of a group possibly a
// half tile of 64 rows; the columnwise outputs go to the group's own
// transpose by vector stores (its row length differs from group to group).
template <bool UE5M3, int LOF, bool GR>
__global__ void __launch_bounds__(LT, kCtlPerSm) ctl_kernel(const QuantJob j, const __grid_constant__ CUtensorMap tmap,
                                                                       const __grid_constant__ CUtensorMap cmap,
                                                                       const __grid_constant__ CUtensorMap rmap,
                                                                       const __grid_constant__ CUtensorMap rmap64) {
  constexpr bool OUTER = LOF != LO_NONE;
  static_assert(!GR || LOF == LO_1D || LOF == LO_2D, "groups: outer-block forms only");
  extern __shared__ __align__(16) unsigned char smem_dyn[];
  unsigned char* smem = smem_align1024(smem_dyn);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const unsigned char* ptb = smem + LL::pt;
  const uint32_t* ctab = reinterpret_cast<const uint32_t*>(smem + LL::ctab);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LL::bars);

  if (t == 0) {
    mbar_init(&bars[0]);
    mbar_init(&bars[1]);
    mbar_init(&bars[2]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // the tables are constant data: their copy may start before the
    // previous grid on the stream has finished
    const uint32_t* img = kCtlTab[UE5M3 ? 1 : 0] + (OUTER ? 0 : kImgOuter / 4);
    mbar_expect_tx(&bars[2], OUTER ? kImgOuter : kImgUnit);
    bulk_load(smem + LL::pt, img, OUTER ? kImgOuter : kImgUnit, &bars[2]);
  }
  pdl_wait_then_release();
  __syncthreads();
  const uint32_t* gtp = GR ? group_tprefix(j.gws) : nullptr;
  if (GR && j.gws->bad) {  // invalid offsets: write nothing (once the table copy has landed)
    if (!mbar_wait(&bars[2], 0u, 1u << 22)) atomicExch(&g_ctl_timeout, 1u);
    return;
  }
  TileIter cur;
  if (GR) cur.init_n((int)(j.K / LK), (int)j.gws->mtiles, 1);
  else cur.init<LM>(j);
  GroupCursor gc, pc;  // the group of the processed tile (all threads), of the prefetched one (thread 0)
  auto tile_at = [&](int i) -> TilePos {
    if (!GR) return cur.pos_of<LM>(i);
    const uint32_t q = (uint32_t)(i / cur.tiles_k);
    pc.seek(gtp, q);
    return TilePos{0, j.goff[pc.e] + LM * (int64_t)(q - pc.lo), (int64_t)(i - (int)q * cur.tiles_k) * LK};
  };
  if (t == 0) {  // the first two tiles; later tiles take a slot once its reads are past a barrier
    if (cur.valid()) issue_tile(&tmap, tile_at(cur.idx), smem + LL::raw(0), &bars[0]);
    if (cur.idx + (int)gridDim.x < cur.ntiles) issue_tile(&tmap, tile_at(cur.idx + (int)gridDim.x), smem + LL::raw(1), &bars[1]);
  }
  const float denh = bitsf(UE5M3 ? kDenHiU5 : kDenHiE4), denl = bitsf(UE5M3 ? kDenLoU5 : kDenLoE4);

  // rowwise: thread t owns row t / 2, columns 32 (t mod 2) .. + 31 (two
  // blocks); its four 16-byte chunks sit at these swizzled offsets
  const int rr = t >> 1, rh = t & 1;
  uint32_t roff[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) roff[q] = (uint32_t)(rr * 128 + (((4 * rh + q) ^ (rr & 7)) << 4));
  // columnwise: warp w owns rows 16 w .. + 15, lane l columns 2 l, 2 l + 1
  const uint32_t ca = smem_u32(smem) + (uint32_t)(warp * 2048 + (lane & 3) * 4 + ((lane >> 2) << 4));
  if (!mbar_wait(&bars[2], 0u, 1u << 22)) atomicExch(&g_ctl_timeout, 1u);

  // one scale for the whole tensor, from the tensorwise amax in the
  // workspace (a bf16 value: the table path when in range)
  uint32_t A_u = unit_amax<UE5M3>();
  float S_u = 1.0f, R_u = 1.0f;
  uint64_t ZH_u = 0ull, ZL_u = 0ull;
  bool u_fast = true;
  if (LOF == LO_UNIFORM) {
    A_u = *j.tw_amax;
    S_u = ieee_div(bitsf(A_u), UE5M3 ? 688128.0f : 2688.0f);
    if (blockIdx.x == 0 && t == 0 && j.tile_outer) j.tile_outer[0] = S_u;
    R_u = ieee_rcp(S_u);
    u_fast = (A_u & 0xFFFFu) == 0u && table_ok<UE5M3>(A_u);
    if (u_fast) {
      float zh, zl;
      outer_rcp(ptb, A_u, zh, zl);
      ZH_u = pk2(zh, zh);
      ZL_u = pk2(zl, zl);
    }
  }

  // c1, c2 of a block with scale code sc and outer amax bits A
  auto mults = [&](uint32_t sc, uint32_t A, float& c1, float& c2) {
    if (OUTER) {
      pair_mults(ptb, ctab, sc, A, c1, c2);
    } else {
      const uint2 e = reinterpret_cast<const uint2*>(ptb)[sc];
      c1 = bitsf(e.x);
      c2 = bitsf(e.y);
    }
  };

  uint32_t phase = 0;
  int pg = 0, pm0 = 0, pk0 = 0;  // the previous tile
  int64_t pgb = 0, pgm = 0, pmr = 0;  // its matrix (a group, or matrix pg): first row, rows; its row in it
  bool phalf = false;            // it was a half tile
  int prev_par = 0;
  bool have_prev = false;
  // The previous tile's staged outputs (parity pp): the tensor stores (t ==
  // 0, one bulk group), and the vector stores of the grouped columnwise
  // codes and of the column scales (8 bytes per column: 64 x 1 block rows
  // of the tile; 4 for a half tile).
  auto store_prev = [&](int pp) {
    if (t == 0) {
      if (!GR) tma_store3(&cmap, smem + LL::ccs(pp), pm0 >> 1, pk0, pg);
      tma_store2(phalf ? &rmap64 : &rmap, smem + LL::rcs(pp), pk0 >> 1, (int)(pg * j.M + pm0));
      bulk_commit();
    }
    const int64_t cb = j.K * pgb + pmr;  // columnwise index of (k, first row): cb + k pgm (the matrix's transpose)
    if (GR) {  // 16-byte chunk q of column c: bytes 16 q .. of its 64 (32 for a half tile)
      const int c = t >> 2, q = t & 3;
      if (!phalf || q < 2) {
        const uint4 v = *reinterpret_cast<const uint4*>(smem + LL::ccs(pp) + c * 64 + ((q ^ ((c >> 1) & 3)) << 4));
        *reinterpret_cast<uint4*>(j.col_codes + ((cb + (pk0 + c) * pgm) >> 1) + q * 16) = v;
      }
    }
    if (t < 64) {
      const uint2 v = *reinterpret_cast<const uint2*>(smem + LL::sst(pp) + t * 8);
      uint8_t* d = j.col_scales + ((cb + (pk0 + t) * pgm) >> 4);
      if (!GR) {
        *reinterpret_cast<uint2*>(d) = v;
      } else {  // 4-byte aligned only (a group's rows / 16 is a multiple of 4)
        reinterpret_cast<uint32_t*>(d)[0] = v.x;
        if (!phalf) reinterpret_cast<uint32_t*>(d)[1] = v.y;
      }
    }
  };
  // One tile; the walk alternates the two input slots and the two staging
  // buffers, so the loop runs two tiles per iteration with the parity a
  // compile-time constant (shared-memory offsets fold into the loads).
  auto tile = [&](auto PC) {
    constexpr int par = decltype(PC)::value;  // input slot and staging buffer
    const int tk0 = cur.tk * LK;
    int tg, tm0;        // this tile: matrix, first row (of the matrix; of the [M, K] view with groups)
    int64_t gb, gm, mr; // its matrix: first row of the [G M] view, rows; the tile's first row in it
    bool half = false;  // the tile's last 64 rows belong to the next group
    if (GR) {
      gc.seek(gtp, (uint32_t)cur.tm);
      gb = j.goff[gc.e];
      gm = j.goff[gc.e + 1] - gb;
      tg = 0;
      mr = LM * (int64_t)((uint32_t)cur.tm - gc.lo);
      tm0 = (int)(gb + mr);
      half = gm - mr == 64;
    } else {
      tg = cur.g;
      tm0 = cur.tm * LM;
      gb = (int64_t)tg * j.M;
      gm = j.M;
      mr = tm0;
    }
    const bool rvalid = !half || rr < 64;  // this thread's row belongs to the tile's matrix
    const int after = cur.idx + 2 * (int)gridDim.x;  // the tile that takes this slot next
    cur.next();
    const unsigned char* raw = smem + LL::raw(par);
    // a wait that runs out raises the error flag; the walk goes on (every
    // later wait is bounded and every barrier is still reached)
    if (!mbar_wait(&bars[par], phase, 1u << 22)) atomicExch(&g_ctl_timeout, 1u);
    uint32_t* red = reinterpret_cast<uint32_t*>(smem + LL::red(par));
    const int64_t row = (int64_t)tg * j.M + tm0 + rr;  // this thread's row of the [G M, K] view

    auto row_store = [&](const uint32_t (&c)[4], uint32_t sc) {
      const int64_t e = row * j.K + tk0 + 32 * rh;  // flat index of the thread's first element
      *reinterpret_cast<uint4*>(smem + LL::rcs(par) + rr * 32 + rh * 16) = make_uint4(c[0], c[1], c[2], c[3]);
      if (rvalid) *reinterpret_cast<uint16_t*>(j.row_scales + (e >> 4)) = (uint16_t)sc;
    };
    // rowwise scales, codes and stores of the thread's two blocks, table path
    // (A: the outer amax bits, ZH / ZL: the split reciprocal of S)
    auto row_fast = [&](const uint4 (&a)[4], uint32_t ram, uint32_t A, uint64_t ZH, uint64_t ZL) {
      const uint32_t sc = codes2<UE5M3, OUTER>(ram, ZH, ZL);
      float c10, c20, c11, c21;
      mults(sc & 0xFFu, A, c10, c20);
      mults(sc >> 8, A, c11, c21);
      uint32_t c[4];
      row_codes16(a[0], a[1], pk2(c10, c10), pk2(c20, c20), c[0], c[1]);
      row_codes16(a[2], a[3], pk2(c11, c11), pk2(c21, c21), c[2], c[3]);
      row_store(c, sc);
    };
    // the same by the general per-block steps
    auto row_slow = [&](const uint4 (&a)[4], uint32_t ram, float S, float R) {
      uint32_t c[4], sc = 0;
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
        const float am = bitsf(b ? (ram & 0xFFFF0000u) : (ram << 16));
        sc |= slow_block<UE5M3>(u, am, S, R, !OUTER, j.srk, c[2 * b], c[2 * b + 1]) << (8 * b);
      }
      row_store(c, sc);
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
    }
    // 1 x 64 (after the barrier): the row's 64 columns are this thread's two
    // blocks and its partner's
    auto row_1d = [&]() {
      uint32_t g = umax(ram & 0xFFFFu, ram >> 16);
      g = umax(g, __shfl_xor_sync(0xFFFFFFFFu, g, 1)) << 16;
      float* so = j.row_outer + row * (j.K >> 6) + (tk0 >> 6);
      if (__all_sync(0xFFFFFFFFu, table_ok<UE5M3>(g))) {
        if (rh == 0 && rvalid) *so = div_bmr(bitsf(g), denh, denl);  // exact for g >= 2^-90
        float zh, zl;
        outer_rcp(ptb, g, zh, zl);
        row_fast(a, ram, g, pk2(zh, zh), pk2(zl, zl));
      } else {
        const float S1 = outer_scale<UE5M3>(bitsf(g));
        if (rh == 0 && rvalid) *so = S1;
        row_slow(a, ram, S1, ieee_rcp(S1));
      }
    };
    // rows 16 warp .. + 15, columns 2 lane (low halves) and 2 lane + 1
    // (high): row i's word sits in 16-byte chunk cunit ^ (i mod 8), which is
    // the per-lane base address with bits 4..6 XORed by i mod 8
    uint32_t wv[16];
    lds_col<LL::raw(par), 0>(ca, wv);
    lds_col<LL::raw(par), 1>(ca, wv);
    lds_col<LL::raw(par), 2>(ca, wv);
    lds_col<LL::raw(par), 3>(ca, wv);
    lds_col<LL::raw(par), 4>(ca, wv);
    lds_col<LL::raw(par), 5>(ca, wv);
    lds_col<LL::raw(par), 6>(ca, wv);
    lds_col<LL::raw(par), 7>(ca, wv);
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

    // refill the slot, store the previous tile's staged outputs
    if (t == 0 && after < cur.ntiles) issue_tile(&tmap, tile_at(after), smem + LL::raw(par), &bars[par]);
    if (have_prev) store_prev(par ^ 1);

    // ---------------------------------------- after the barrier: registers and staging only
    if (LOF == LO_1D) {
      row_1d();
    } else if (LOF == LO_NONE) {
      row_fast(a, ram, unit_amax<UE5M3>(), 0ull, 0ull);
    } else if (LOF == LO_UNIFORM) {
      if (u_fast) row_fast(a, ram, A_u, ZH_u, ZL_u);
      else row_slow(a, ram, S_u, R_u);
    }
    uint32_t A2 = 0;  // the 64 x 64 block's amax (2-D): both orientations
    float S2f = 1.0f;
    uint64_t ZH2 = 0ull, ZL2 = 0ull;
    bool f2 = true;
    if (LOF == LO_2D) {
      const uint32_t* rq = red + (warp >> 2) * 128;
      A2 = umax(umax(rq[0], rq[32]), umax(rq[64], rq[96])) << 16;
      f2 = table_ok<UE5M3>(A2);  // uniform over the CTA half
      if (f2) {
        S2f = div_bmr(bitsf(A2), denh, denl);
        float zh, zl;
        outer_rcp(ptb, A2, zh, zl);
        ZH2 = pk2(zh, zh);
        ZL2 = pk2(zl, zl);
      } else {
        S2f = outer_scale<UE5M3>(bitsf(A2));
      }
      if ((warp & 3) == 0 && lane == 0 && (!half || warp < 4))
        j.tile_outer[((int64_t)tg * (j.M >> 6) + (tm0 >> 6) + (warp >> 2)) * (j.K >> 6) + (tk0 >> 6)] = S2f;
      if (f2) row_fast(a, ram, A2, ZH2, ZL2);
      else row_slow(a, ram, S2f, ieee_rcp(S2f));
    }
    // ----------------------------------------------------------- columnwise
    {
      uint32_t A0 = unit_amax<UE5M3>(), A1 = A0;  // the two columns' outer amax bits
      uint64_t ZH = 0ull, ZL = 0ull;
      float S[2] = {1.0f, 1.0f};
      bool fast = true;
      if (LOF == LO_UNIFORM) {
        A0 = A1 = A_u;
        ZH = ZH_u;
        ZL = ZL_u;
        S[0] = S[1] = S_u;
        fast = u_fast;
      } else if (LOF == LO_2D) {
        A0 = A1 = A2;
        ZH = ZH2;
        ZL = ZL2;
        S[0] = S[1] = S2f;
        fast = f2;
      } else if (LOF == LO_1D) {  // the columns' 64-row maxima over the 4 warps of this half
        const uint32_t* rq = red + (warp >> 2) * 128 + lane;
        const uint32_t g = bf16x2_amax(bf16x2_amax(rq[0], rq[32]), bf16x2_amax(rq[64], rq[96])) & 0x7FFF7FFFu;
        A0 = g << 16;
        A1 = g & 0xFFFF0000u;
        fast = __all_sync(0xFFFFFFFFu, table_ok<UE5M3>(A0) && table_ok<UE5M3>(A1));
        if (fast) {
          upk2(bmr2(pk2(bitsf(A0), bitsf(A1)), pk2(denh, denh), pk2(denl, denl)), S[0], S[1]);  // exact
          float zh0, zl0, zh1, zl1;
          outer_rcp(ptb, A0, zh0, zl0);
          outer_rcp(ptb, A1, zh1, zl1);
          ZH = pk2(zh0, zh1);
          ZL = pk2(zl0, zl1);
        } else {
          S[0] = outer_scale<UE5M3>(bitsf(A0));
          S[1] = outer_scale<UE5M3>(bitsf(A1));
        }
        if ((warp & 3) == 0 && (!half || warp < 4)) {  // the matrix's [K, rows / 64] outer scales
          const int64_t M64 = gm >> 6;
          float* d = j.col_outer + ((j.K * gb + mr) >> 6) + (tk0 + 2 * lane) * M64 + (warp >> 2);
          d[0] = S[0];
          d[M64] = S[1];
        }
      }
      uint32_t c[4], sc;
      if (fast) {
        sc = codes2<UE5M3, OUTER>(cam, ZH, ZL);
        float c10, c20, c11, c21;
        mults(sc & 0xFFu, A0, c10, c20);
        mults(sc >> 8, A1, c11, c21);
        col_codes16(wv, pk2(c10, c11), pk2(c20, c21), c);
      } else {
        sc = 0;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          float u[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) u[i] = k ? bf16hi(wv[i]) : bf16lo(wv[i]);
          const float am = bitsf(k ? (cam & 0xFFFF0000u) : (cam << 16));
          sc |= slow_block<UE5M3>(u, am, S[k], ieee_rcp(S[k]), !OUTER, j.srk, c[2 * k], c[2 * k + 1]) << (8 * k);
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
    pgb = gb;
    pgm = gm;
    pmr = mr;
    phalf = half;
    prev_par = par;
    have_prev = true;
  };
  while (cur.valid()) {
    tile(std::integral_constant<int, 0>{});
    if (!cur.valid()) break;
    tile(std::integral_constant<int, 1>{});
    phase ^= 1u;
  }
  // the last tile's staged outputs
  __syncthreads();
  if (have_prev) store_prev(prev_par);
  if (t == 0) bulk_wait_all();
}

template <bool UE5M3, int LOF, bool GR>
cudaError_t launch_ctl_t(const QuantJob& j, const CUtensorMap& map, const CUtensorMap& cmap, const CUtensorMap& rmap,
                         const CUtensorMap& rmap64, cudaStream_t st) {
  auto kern = ctl_kernel<UE5M3, LOF, GR>;
  constexpr int smem = LL::total;
  static int per_sm_cache[128] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 128) dev = 0;
  int& per_sm = per_sm_cache[dev];
  if (per_sm == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, LT, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
  }
  // grouped: the tile count lives on the device; at most ceil(M / 128) +
  // groups 128-row tiles per 64-column strip
  const int64_t tiles = GR ? (j.M / LM + j.ngroups) * (j.K / LK) : j.G * (j.M / LM) * (j.K / LK);
  const int64_t cap = (int64_t)num_sms() * per_sm;
  return launch_pdl(kern, dim3((unsigned)(tiles < cap ? tiles : cap)), dim3(LT), (size_t)smem, st, j, map, cmap, rmap,
                    rmap64);
}

template <bool UE5M3>
cudaError_t launch_ctl_f(const QuantJob& j, int lof, const CUtensorMap& map, const CUtensorMap& cmap,
                         const CUtensorMap& rmap, const CUtensorMap& rmap64, cudaStream_t st) {
  if (j.ngroups > 0) {
    return lof == LO_1D ? launch_ctl_t<UE5M3, LO_1D, true>(j, map, cmap, rmap, rmap64, st)
                        : launch_ctl_t<UE5M3, LO_2D, true>(j, map, cmap, rmap, rmap64, st);
  }
  switch (lof) {
    case LO_NONE: return launch_ctl_t<UE5M3, LO_NONE, false>(j, map, cmap, rmap, rmap64, st);
    case LO_UNIFORM: return launch_ctl_t<UE5M3, LO_UNIFORM, false>(j, map, cmap, rmap, rmap64, st);
    case LO_1D: return launch_ctl_t<UE5M3, LO_1D, false>(j, map, cmap, rmap, rmap64, st);
    default: return launch_ctl_t<UE5M3, LO_2D, false>(j, map, cmap, rmap, rmap64, st);
  }
}

bool aligned_to(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0u; }

// Tensor map of the rowwise codes as a [G M][K / 2] byte matrix for the tile
// store (box: 32 bytes x box_m rows, no swizzle: the staging holds row r at
// byte 32 r).  Needs rows of a multiple of 16 bytes (K a multiple of 32), a
// 16-byte aligned base and G M below 2^31 (a 32-bit coordinate).
bool make_row_map(const QuantJob& j, CUtensorMap* map, int box_m) {
  if (j.K % 32 || !aligned_to(j.row_codes, 16) || j.G * j.M >= ((int64_t)1 << 31)) return false;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)(j.K / 2), (cuuint64_t)(j.G * j.M)};
  const cuuint64_t strides[1] = {(cuuint64_t)(j.K / 2)};
  const cuuint32_t box[2] = {32u, (cuuint32_t)box_m};
  const cuuint32_t es[2] = {1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, j.row_codes, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// The whole-tile form, when the call's facts allow it (false: the caller
// takes the general cast-transpose kernel).  FP4Q_NO_CTL_KERNEL=1 turns it
// off (the parity tests run every kernel that can take a case).  Ragged
// groups take it with 1-D or 2-D outer blocks of 64 (every group then a
// multiple of 64 rows).
bool launch_ctl(const QuantJob& j, cudaStream_t st, cudaError_t* err) {
  const bool gr = j.ngroups > 0;
  if (!j.in_bf16 || !j.do_row || !j.do_col || j.sr || j.inner_2d || j.residual || j.qdq_orient || j.col_rht ||
      j.rsl.mma || j.csl.mma || j.K % LK || (gr ? (j.G != 1 || j.M % 64) : j.M % LM))
    return false;
  if (!aligned_to(j.x, 16) || (j.ld * 2) % 16 || !aligned_to(j.row_codes, 16) || !aligned_to(j.row_scales, 2) ||
      !aligned_to(j.col_codes, 16) || !aligned_to(j.col_scales, gr ? 4 : 8))
    return false;
  int lof;
  if (j.s_src == S_ONE) lof = LO_NONE;
  else if (j.mode == 1 && j.s_src == S_TENSORWISE_WS) lof = LO_UNIFORM;  // tensorwise, from the workspace amax
  else if (j.s_src == S_IN_TILE && j.ob == 64) lof = j.outer_2d ? LO_2D : LO_1D;
  else return false;
  if (gr && lof != LO_1D && lof != LO_2D) return false;
  if (getenv_flag("FP4Q_NO_CTL_KERNEL")) return false;
  CUtensorMap map, cmap = {}, rmap = {}, rmap64 = {};
  if (!make_bf16_tile_map(j, &map, LM) || (!gr && !make_col_map(j, &cmap))) return false;
  if (!make_row_map(j, &rmap, LM) || (gr && !make_row_map(j, &rmap64, 64))) return false;
  *err = j.ue5m3 ? launch_ctl_f<true>(j, lof, map, cmap, rmap, rmap64, st)
                 : launch_ctl_f<false>(j, lof, map, cmap, rmap, rmap64, st);
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
