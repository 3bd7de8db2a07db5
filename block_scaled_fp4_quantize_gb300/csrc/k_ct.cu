// k_ct.cu -- generic cast-transpose quantize / QDQ kernel (binary32 or bf16
// input; the columnwise bf16 quantize has its own kernel in k_ctb.cu).
//
// A CTA of 256 threads walks TM x 64 tiles of x (bf16: 128 rows, binary32:
// 64 rows; 16 KB either way), fed by 3-D tensor copies with the 128-byte
// swizzle, several tiles in flight on mbarriers with bounded waits.  Rowwise
// pass: a thread owns consecutive 1 x 16 blocks of one row.  Columnwise pass:
// a thread owns one column and a quarter of the tile's rows.  With a 2-D
// outer scale, tensorwise or no outer scale, x' = u / S is computed once in
// the rowwise pass and staged in shared memory (binary32) for the columnwise
// pass; with 1-D outer scales each orientation normalizes by its own scale
// ("Block-Scaled FP8 and FP4 Weight Quantization", sections 3 and 6).
//
// Covers: inner 1 x 16 blocks, 16-byte-aligned inputs; modes none,
// tensorwise, outer-block 1-D / 2-D with ob in {16, 32, 64} computed in the
// tile or any ob read from the outer buffers; RNE / SR; error feedback; QDQ
// along K or M.  The per-block arithmetic (exact division sequences, scale
// encode, E2M1 encode) is in fp4q_block.cuh.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "fp4q_block.cuh"
#include "fp4q_tma.cuh"
#include "fp4q_device.cuh"
#include "fp4q_internal.h"

namespace fp4q {
namespace {

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



// ---------------------------------------------------------------------------
// Pipelined tile kernel: 128 threads, TM x 64 tiles (bf16: 128 rows,
// binary32: 64 rows; 16 KB raw either way), double-buffered with cp.async.
// Rowwise pass: a thread owns RPT consecutive 1 x 16 blocks of one row (bf16:
// the whole 1 x 64 row segment).  Columnwise pass: a thread owns one column
// and TM / 2 rows.  Both passes write whole 32-byte (bf16) code runs.
// ---------------------------------------------------------------------------
constexpr int NT = 256;

template <bool IN_BF16>
struct Geo {
  static constexpr int TM = IN_BF16 ? 128 : 64;
  static constexpr int E = IN_BF16 ? 2 : 4;      // bytes per element
  static constexpr int UPR = 64 * E / 16;        // 16-byte units per raw row
  static constexpr int RAW = TM * 64 * E;        // bytes of one raw tile
  static constexpr int RPT = TM / 64;            // row pass: 1 x 16 blocks per thread
  static constexpr int TPR = 4 / RPT;            // threads per row
  static constexpr int CB = TM / 64;             // column pass: 16 x 1 blocks per thread (4 parts)
};

// Swizzled 16-byte unit within a row (bank-conflict-free copies, block
// reads, staging writes and column reads).  bf16 raw rows have 8 units;
// binary32 rows (raw and staged) have 16.
// Byte offset of 16-byte unit `unit` of tile row `row` in a raw tile as the
// tensor copy writes it: 128-byte rows (bf16: one per tile row; binary32: the
// tile is two 32-column halves), 16-byte units permuted by the 128-byte
// swizzle (unit ^ (row mod 8)), which also keeps the block and column reads
// free of bank conflicts.
template <bool IN_BF16>
__device__ __forceinline__ int raw_off(int row, int unit) {
  if (IN_BF16) return (row * 8 + (unit ^ (row & 7))) * 16;
  return (unit >> 3) * (Geo<false>::TM * 128) + (row * 8 + ((unit & 7) ^ (row & 7))) * 16;
}
template <bool IN_BF16>
__device__ __forceinline__ int stage_swz(int row, int unit) {
  return (unit & 8) | ((unit & 7) ^ ((2 * row + (unit >> 3)) & 7));
}

// Shared memory: [raw tiles 0 .. NS - 1][x' staging][table (s, zh, zl)]
// [2-D and 1-D reductions][tile-arrival barriers]
template <bool IN_BF16, int NS>
struct Layout {
  __host__ __device__ static constexpr int raw(int s) { return s * Geo<IN_BF16>::RAW; }
  static constexpr int stage = NS * Geo<IN_BF16>::RAW;
  static constexpr int stage_bytes = Geo<IN_BF16>::TM * 64 * 4;
  __host__ __device__ static int tab(bool staged) { return stage + (staged ? stage_bytes : 0); }
  __host__ __device__ static int red(bool staged) { return tab(staged) + 256 * 16; }
  __host__ __device__ static int total(bool staged) { return red(staged) + (32 + 128 + 2 * 32) * 4 + 8 * NS + 1024; }
};

// Tile copies in flight per CTA: enough bytes per SM to cover HBM latency
// at the CTA counts each variant runs (2 with the columnwise pass, 3 without).
template <bool COL>
struct Stages {
  static constexpr int NS = COL ? 3 : 4;
};

// Set when a tile copy did not arrive within the wait limit (the kernel then
// stops early).
__device__ unsigned int g_tile_timeout = 0;

// Issue the copy of one raw tile (one thread): bf16 one 64 x TM box,
// binary32 two 32 x TM boxes (the 128-byte swizzle spans at most 128 bytes).
template <bool IN_BF16>
__device__ __forceinline__ void issue_tile(const CUtensorMap* map, const TilePos& p, unsigned char* raw, uint64_t* bar) {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_tx(bar, (uint32_t)Geo<IN_BF16>::RAW);
  if (IN_BF16) {
    tma_load3(raw, map, (int)p.k0, (int)p.m0, (int)p.g, bar);
  } else {
    tma_load3(raw, map, (int)p.k0, (int)p.m0, (int)p.g, bar);
    tma_load3(raw + Geo<false>::TM * 128, map, (int)p.k0 + 32, (int)p.m0, (int)p.g, bar);
  }
}

// The 16 values of block b (columns 16 b .. 16 b + 15) of tile row `row`.
template <bool IN_BF16>
__device__ __forceinline__ void read_block(const unsigned char* raw, int row, int b, float (&u)[16]) {
  using G = Geo<IN_BF16>;
  constexpr int upb = G::UPR / 4;
#pragma unroll
  for (int q = 0; q < upb; ++q) {
    const uint4 w = *reinterpret_cast<const uint4*>(raw + raw_off<IN_BF16>(row, b * upb + q));
    if (IN_BF16) {
      u[8 * q + 0] = bf16lo(w.x); u[8 * q + 1] = bf16hi(w.x); u[8 * q + 2] = bf16lo(w.y); u[8 * q + 3] = bf16hi(w.y);
      u[8 * q + 4] = bf16lo(w.z); u[8 * q + 5] = bf16hi(w.z); u[8 * q + 6] = bf16lo(w.w); u[8 * q + 7] = bf16hi(w.w);
    } else {
      u[4 * q + 0] = bitsf(w.x); u[4 * q + 1] = bitsf(w.y); u[4 * q + 2] = bitsf(w.z); u[4 * q + 3] = bitsf(w.w);
    }
  }
}

// Element (row, col) of the raw tile.
template <bool IN_BF16>
__device__ __forceinline__ float raw_elem(const unsigned char* raw, int row, int col) {
  using G = Geo<IN_BF16>;
  constexpr int epu = 16 / G::E;
  const unsigned char* p = raw + raw_off<IN_BF16>(row, col / epu) + (col % epu) * G::E;
  if (IN_BF16) return bitsf((uint32_t)(*reinterpret_cast<const uint16_t*>(p)) << 16);
  return *reinterpret_cast<const float*>(p);
}

// x' staging: binary32 [TM][64], 16 units per row.
template <bool IN_BF16>
__device__ __forceinline__ void stage_block(float* xs, int row, int b, const float (&x)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    reinterpret_cast<float4*>(xs)[row * 16 + stage_swz<IN_BF16>(row, 4 * b + q)] =
        make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
}
template <bool IN_BF16>
__device__ __forceinline__ float staged_elem(const float* xs, int row, int col) {
  return xs[(row * 16 + stage_swz<IN_BF16>(row, col >> 2)) * 4 + (col & 3)];
}

// Residual-corrected, sanitized values of one block and their |max|.
template <bool IN_BF16>
__device__ __forceinline__ float load_block(const QuantJob& j, const unsigned char* raw, int row, int b, int64_t n0,
                                            bool valid, float (&u)[16]) {
  read_block<IN_BF16>(raw, row, b, u);
  if (j.residual && valid) {
    const float4* rp = reinterpret_cast<const float4*>(j.residual + n0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v = rp[q];
      u[4 * q] = ieee_add(u[4 * q], v.x); u[4 * q + 1] = ieee_add(u[4 * q + 1], v.y);
      u[4 * q + 2] = ieee_add(u[4 * q + 2], v.z); u[4 * q + 3] = ieee_add(u[4 * q + 3], v.w);
    }
  }
  float am = amax16(u);
  if (fbits(am) >= 0x7F800000u) {
#pragma unroll
    for (int i = 0; i < 16; ++i) u[i] = sanitize(u[i], IN_BF16 ? 0x7F7F0000u : 0x7F7FFFFFu);
    am = amax16(u);
  }
  return am;
}

// |max| of block (row, b) for the outer-scale reductions: packed bf16 pairs
// when nothing is added, else the full residual-corrected, sanitized block.
template <bool IN_BF16>
__device__ __forceinline__ float pre_amax(const QuantJob& j, const unsigned char* raw, int row, int b, int64_t n0,
                                          bool valid) {
  if (IN_BF16 && !j.residual) {
    const uint4 a = *reinterpret_cast<const uint4*>(raw + raw_off<true>(row, 2 * b));
    const uint4 c = *reinterpret_cast<const uint4*>(raw + raw_off<true>(row, 2 * b + 1));
    uint32_t m = bf16x2_amax(bf16x2_amax(bf16x2_amax(a.x, a.y), bf16x2_amax(a.z, a.w)),
                             bf16x2_amax(bf16x2_amax(c.x, c.y), bf16x2_amax(c.z, c.w)));
    m &= 0x7FFF7FFFu;
    const uint32_t hi = m >> 16, lo = m & 0xFFFFu;
    const float am = bitsf((hi > lo ? hi : lo) << 16);
    if (fbits(am) < 0x7F800000u) return am;
  }
  float u[16];
  return load_block<IN_BF16>(j, raw, row, b, n0, valid, u);
}

// Outer scale of a rowwise block from S sources other than the in-tile 1-D
// reduction (which needs the neighbours' maxima).
struct OuterCtx {
  float S_tw, r_tw;
  const float2* sr2d;
  int ob, lob;
};

template <bool IN_BF16, bool SR, bool COL, bool UE5M3>
__global__ void __launch_bounds__(NT, COL ? 2 : 3) cp_kernel(const QuantJob j, const __grid_constant__ CUtensorMap tmap) {
  using G = Geo<IN_BF16>;
  constexpr int NS = Stages<COL>::NS;
  using L = Layout<IN_BF16, NS>;
  extern __shared__ __align__(16) unsigned char smem_dyn[];
  // the 128-byte swizzle of the tensor copies needs 1024-byte aligned tiles
  unsigned char* smem = smem_align1024(smem_dyn);
  const int t = threadIdx.x;
  const bool none = j.s_src == S_ONE;
  const bool shared_S = none || j.mode == 1 || j.outer_2d;
  const bool staged = COL && shared_S;
  float* xs = reinterpret_cast<float*>(smem + L::stage);
  const float4* tab = reinterpret_cast<const float4*>(smem + L::tab(staged));
  uint32_t* red2d = reinterpret_cast<uint32_t*>(smem + L::red(staged));  // [32]
  uint32_t* redcol = red2d + 32;                                          // [2][64]
  float2* sr2d = reinterpret_cast<float2*>(redcol + 128);                 // [32]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sr2d + 32);                // [NS] tile-arrival barriers
  struct {
    const float4* tab;
  } tv{tab};

  TileIter cur;
  cur.init<Geo<IN_BF16>::TM>(j);
  if (t == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(&bars[s]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // prologue: the first NS - 1 tiles of this CTA's walk
  if (t == 0) {
#pragma unroll
    for (int s = 0; s < NS - 1; ++s) {
      const int i = cur.idx + s * (int)gridDim.x;
      if (i < cur.ntiles) issue_tile<IN_BF16>(&tmap, cur.pos_of<Geo<IN_BF16>::TM>(i), smem + L::raw(s), &bars[s]);
    }
  }

  // inner-scale table: value and the divisor split of its reciprocal
  build_scale_table<UE5M3>(reinterpret_cast<float4*>(smem + L::tab(staged)), t, NT);
  if (t < 32) red2d[t] = 0u;
  if (t < 128) redcol[t] = 0u;
  const int ob = j.ob;
  const bool ob_pow2 = ob > 0 && (ob & (ob - 1)) == 0;
  const int lob = ob > 0 ? 31 - __clz(ob) : 0;  // log2(ob) for power-of-two blocks
  const int mob = ob > 0 ? (int)(j.M / ob) : 0, kob = ob > 0 ? (int)(j.K / ob) : 0;
  auto dob = [&](int v) { return ob_pow2 ? (v >> lob) : v / ob; };
  float S_tw = 1.0f, r_tw = 1.0f;
  if (j.s_src == S_TENSORWISE_WS) {
    S_tw = ieee_div(bitsf(*j.tw_amax), UE5M3 ? 688128.0f : 2688.0f);
    r_tw = ieee_rcp(S_tw);
    if (blockIdx.x == 0 && t == 0 && j.tile_outer) j.tile_outer[0] = S_tw;
  }
  const bool deq_row = j.qdq_orient == 1 || j.residual != nullptr;
  const int row = t / G::TPR, bq0 = (t % G::TPR) * G::RPT;  // rowwise: blocks bq0 .. bq0 + RPT - 1 of `row`
  const int col = t & 63, part = t >> 6;                     // columnwise: column, rows part * TM/4 ..
  const bool wide_codes = (j.K % 32) == 0 && (j.M % 32) == 0 &&
                          ((reinterpret_cast<uintptr_t>(j.row_codes) | reinterpret_cast<uintptr_t>(j.col_codes)) & 15u) == 0;
  const bool wide_scales = (j.K % 64) == 0 && (j.M % 64) == 0 &&
                           ((reinterpret_cast<uintptr_t>(j.row_scales) | reinterpret_cast<uintptr_t>(j.col_scales)) & 3u) == 0;
  __syncthreads();

  int slot = 0;
  uint32_t phase = 0;
  for (int it = 0; cur.valid(); ++it) {
    unsigned char* raw = smem + L::raw(slot);
    const TilePos p = cur.pos<Geo<IN_BF16>::TM>();
    // refill the slot the previous tile used (every thread has left it)
    if (t == 0) {
      const int i = cur.idx + (NS - 1) * (int)gridDim.x;
      const int s = slot == 0 ? NS - 1 : slot - 1;
      if (i < cur.ntiles) issue_tile<IN_BF16>(&tmap, cur.pos_of<Geo<IN_BF16>::TM>(i), smem + L::raw(s), &bars[s]);
    }
    cur.next();
    // bounded wait for this tile's copy; on a timeout every thread leaves
    const bool arrived = mbar_wait(&bars[slot], phase, 1u << 22);
    if (!__syncthreads_and(arrived)) {
      if (t == 0) {
        atomicExch(&g_tile_timeout, 1u);
        // let the later copies still in flight land before the CTA exits
        for (int d = 1; d < NS; ++d) {
          const int i = it + d;
          if (cur.idx + (d - 1) * (int)gridDim.x < cur.ntiles)
            mbar_wait(&bars[i % NS], (uint32_t)(i / NS) & 1u, 1u << 22);
        }
      }
      return;
    }
    if (++slot == NS) {
      slot = 0;
      phase ^= 1u;
    }

    const int K32 = (int)j.K, M32 = (int)j.M;
    const int64_t rbase = (p.g * j.M + p.m0) * j.K + p.k0;  // rowwise element index of the tile origin
    const int64_t cbase = (p.g * j.K + p.k0) * j.M + p.m0;  // the same in the transposed tensor
    const int64_t m = p.m0 + row;
    const bool rvalid = m < j.M;
    const int64_t nrow = rbase + (int64_t)row * K32;         // element index of (row, column 0)

    // block maxima of this thread's row segment
    float am[G::RPT];
#pragma unroll
    for (int q = 0; q < G::RPT; ++q) {
      const int b = bq0 + q;
      am[q] = pre_amax<IN_BF16>(j, raw, row, b, nrow + 16 * b, rvalid && p.k0 + 16 * b < j.K);
    }

    // 2-D outer scales of the tile's ob x ob sub-blocks (ob in {16, 32, 64})
    if (j.s_src == S_IN_TILE && j.outer_2d) {
      const int nbk = 64 >> lob;
#pragma unroll
      for (int q = 0; q < G::RPT; ++q) {
        // lanes hold consecutive rows (bf16) or row halves (binary32); reduce
        // over the rows of the sub-block that fall in this warp
        uint32_t v = fbits(am[q]);
        for (int o = G::TPR; o < 32 && o < ob * G::TPR; o <<= 1) v = umax(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
        const int b = bq0 + q;
        if (((t & 31) % (ob * G::TPR < 32 ? ob * G::TPR : 32)) < G::TPR)
          atomicMax(&red2d[(row >> lob) * nbk + ((16 * b) >> lob)], v);
      }
      __syncthreads();
      const int nsub = (G::TM >> lob) * nbk;
      if (t < nsub) {
        const float A = bitsf(red2d[t]);
        red2d[t] = 0u;
        const float S = outer_scale<UE5M3>(A);
        sr2d[t] = make_float2(S, ieee_rcp(S));
        const int64_t mi = p.m0 + (int64_t)(t / nbk) * ob, kj = p.k0 + (int64_t)(t % nbk) * ob;
        if (j.tile_outer && mi < j.M && kj < j.K)
          j.tile_outer[(p.g * (j.M / ob) + mi / ob) * (j.K / ob) + kj / ob] = S;
      }
      __syncthreads();
    }

    // ------------------------------------------------------------- rowwise
    if (j.do_row || staged) {
      // outer scale of each block
      float Sq[G::RPT], rq[G::RPT];
#pragma unroll
      for (int q = 0; q < G::RPT; ++q) { Sq[q] = 1.0f; rq[q] = 1.0f; }
      if (j.s_src == S_TENSORWISE_WS) {
#pragma unroll
        for (int q = 0; q < G::RPT; ++q) { Sq[q] = S_tw; rq[q] = r_tw; }
      } else if (j.s_src == S_IN_TILE && j.outer_2d) {
#pragma unroll
        for (int q = 0; q < G::RPT; ++q) {
          const float2 sr = sr2d[(row >> lob) * (64 >> lob) + ((16 * (bq0 + q)) >> lob)];
          Sq[q] = sr.x;
          rq[q] = sr.y;
        }
      } else if (j.s_src == S_IN_TILE) {
        // 1-D along K: the ob / 16 blocks of an outer block are this thread's
        // (or, for 1 x 64 binary32, this thread's and its neighbour's)
        const int per = ob / 16, lper = lob - 4;
        uint32_t gmax[G::RPT];
#pragma unroll
        for (int q = 0; q < G::RPT; ++q) {
          uint32_t v = 0;
#pragma unroll
          for (int q2 = 0; q2 < G::RPT; ++q2)
            if (((bq0 + q2) >> lper) == ((bq0 + q) >> lper)) v = umax(v, fbits(am[q2]));
          gmax[q] = v;
        }
        for (int o = 1; o < per / G::RPT; o <<= 1) {  // neighbours holding the rest of the outer block
#pragma unroll
          for (int q = 0; q < G::RPT; ++q) gmax[q] = umax(gmax[q], __shfl_xor_sync(0xFFFFFFFFu, gmax[q], o));
        }
#pragma unroll
        for (int q = 0; q < G::RPT; ++q) {
          if (((bq0 + q) & (per - 1)) == 0 || q == 0) {
            Sq[q] = outer_scale<UE5M3>(bitsf(gmax[q]));
            rq[q] = ieee_rcp(Sq[q]);
          } else {
            Sq[q] = Sq[q - 1];
            rq[q] = rq[q - 1];
          }
          const int64_t kb = p.k0 + 16 * (bq0 + q);
          if (j.row_outer && rvalid && kb < j.K && ((bq0 + q) & (per - 1)) == 0 && j.do_row)
            j.row_outer[(nrow + 16 * (bq0 + q)) >> (31 - __clz(ob))] = Sq[q];
        }
      } else if (j.s_src == S_FROM_BUFFER && rvalid) {
#pragma unroll
        for (int q = 0; q < G::RPT; ++q) {
          const int64_t kb = p.k0 + 16 * (bq0 + q);
          if (kb >= j.K) continue;
          if (j.mode == 1) Sq[q] = j.tile_outer[0];
          else if (j.outer_2d) Sq[q] = j.tile_outer[((int64_t)p.g * mob + dob((int)m)) * kob + dob((int)kb)];
          else Sq[q] = j.row_outer[((int64_t)p.g * j.M + m) * kob + dob((int)kb)];
          rq[q] = ieee_rcp(Sq[q]);
        }
      }
      uint32_t cw[2 * G::RPT];
      uint32_t scw = 0;
#pragma unroll
      for (int q = 0; q < G::RPT; ++q) {
        const int b = bq0 + q;
        const int64_t kb = p.k0 + 16 * b;
        const bool valid = rvalid && kb < j.K;
        const int64_t n0 = nrow + 16 * b;
        float u[16];
        const float amq = load_block<IN_BF16>(j, raw, row, b, n0, valid, u);
        Norm n;
        n.none = none;
        n.S = Sq[q];
        n.r = rq[q];
        n.pos = none || positive(n.S);
        n.fast = !none && positive_normal(n.S) && positive_normal(n.r);
        float4 T;
        const uint32_t sc = block_scale<UE5M3>(tv, amq, n, T);
        float x[16];
        normalize16<SR>(u, x, n);
        if (staged) stage_block<IN_BF16>(xs, row, b, x);
        if (j.do_row) {
          float deq[16];
          if (deq_row) encode16<SR, true>(x, T, n, j.srk, j.step, 0u, sr_row_n(j, n0), cw[2 * q], cw[2 * q + 1], deq);
          else encode16<SR, false>(x, T, n, j.srk, j.step, 0u, sr_row_n(j, n0), cw[2 * q], cw[2 * q + 1], deq);
          scw |= sc << (8 * q);
          if (valid) {
            if (j.residual) {
              float4* rp = reinterpret_cast<float4*>(j.residual + n0);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                rp[i] = make_float4(ieee_sub(u[4 * i], deq[4 * i]), ieee_sub(u[4 * i + 1], deq[4 * i + 1]),
                                    ieee_sub(u[4 * i + 2], deq[4 * i + 2]), ieee_sub(u[4 * i + 3], deq[4 * i + 3]));
            }
            if (j.qdq_orient == 1) store16(j.y, j.out_bf16, n0, deq);
          }
        }
      }
      if (j.do_row && rvalid && j.row_codes) {
        const int64_t c0 = nrow + 16 * bq0;  // first element of this thread's run
        const int nb = (int)min((int64_t)G::RPT, (j.K - p.k0 - 16 * bq0 + 15) / 16);
        if (nb == G::RPT && wide_codes && G::RPT >= 2) {
          uint4* d = reinterpret_cast<uint4*>(j.row_codes + c0 / 2);
#pragma unroll
          for (int q = 0; q < G::RPT / 2; ++q) d[q] = make_uint4(cw[4 * q], cw[4 * q + 1], cw[4 * q + 2], cw[4 * q + 3]);
        } else {
#pragma unroll
          for (int q = 0; q < G::RPT; ++q)
            if (q < nb) *reinterpret_cast<uint2*>(j.row_codes + (c0 + 16 * q) / 2) = make_uint2(cw[2 * q], cw[2 * q + 1]);
        }
        if (nb == G::RPT && wide_scales && G::RPT == 2 && !j.rsl.mma) {
          *reinterpret_cast<uint16_t*>(j.row_scales + c0 / 16) = (uint16_t)scw;
        } else {
#pragma unroll
          for (int q = 0; q < G::RPT; ++q)
            if (q < nb) j.row_scales[sf_from_linear(j.rsl, c0 / 16 + q)] = (uint8_t)(scw >> (8 * q));
        }
      }
    }
    if (!COL) {
      __syncthreads();
      continue;
    }

    // ---------------------------------------------------------- columnwise
    if (staged) __syncthreads();
    const int64_t k = p.k0 + col;
    const bool kvalid = k < j.K;
    const int rbeg = part * 16 * G::CB;  // first tile row of this thread
    float cam[G::CB];
    // column block maxima (from the staged x' or the raw tile)
#pragma unroll
    for (int q = 0; q < G::CB; ++q) {
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = rbeg + 16 * q + i;
        v[i] = staged ? staged_elem<IN_BF16>(xs, r, col) : raw_elem<IN_BF16>(raw, r, col);
      }
      cam[q] = amax16(v);
      if (!staged && fbits(cam[q]) >= 0x7F800000u) {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = sanitize(v[i], IN_BF16 ? 0x7F7F0000u : 0x7F7FFFFFu);
        cam[q] = amax16(v);
      }
    }
    float Sc[G::CB];
#pragma unroll
    for (int q = 0; q < G::CB; ++q) Sc[q] = 1.0f;
    if (shared_S) {
#pragma unroll
      for (int q = 0; q < G::CB; ++q) {
        const int64_t mb = p.m0 + rbeg + 16 * q;
        if (j.s_src == S_TENSORWISE_WS) Sc[q] = S_tw;
        else if (j.s_src == S_IN_TILE && !none) Sc[q] = sr2d[((rbeg + 16 * q) >> lob) * (64 >> lob) + (col >> lob)].x;
        else if (j.s_src == S_FROM_BUFFER && mb < j.M && kvalid)
          Sc[q] = j.mode == 1 ? j.tile_outer[0] : j.tile_outer[((int64_t)p.g * mob + dob((int)mb)) * kob + dob((int)k)];
      }
    } else if (j.s_src == S_IN_TILE) {
      // 1-D along M: an outer block is ob / 16 of this thread's blocks, or
      // (binary32, ob = 64) spans both threads of the column
      const int per = ob / 16, lper = lob - 4;
      uint32_t gmax[G::CB];
#pragma unroll
      for (int q = 0; q < G::CB; ++q) {
        uint32_t v = 0;
#pragma unroll
        for (int q2 = 0; q2 < G::CB; ++q2)
          if ((q2 >> lper) == (q >> lper)) v = umax(v, fbits(cam[q2]));
        gmax[q] = v;
      }
      if (per > G::CB) {  // the outer block spans several parts: reduce in shared memory
        uint32_t* slot = &redcol[(rbeg >> lob) * 64 + col];
#pragma unroll
        for (int q = 0; q < G::CB; ++q) atomicMax(slot, gmax[q]);
        __syncthreads();
#pragma unroll
        for (int q = 0; q < G::CB; ++q) gmax[q] = *slot;
        __syncthreads();
        if ((rbeg & (ob - 1)) == 0) *slot = 0u;
      }
#pragma unroll
      for (int q = 0; q < G::CB; ++q) {
        Sc[q] = outer_scale<UE5M3>(bitsf(gmax[q]));
        const int64_t mb = p.m0 + rbeg + 16 * q;
        if (j.col_outer && kvalid && mb < j.M && ((rbeg / 16 + q) & (per - 1)) == 0)
          j.col_outer[((int64_t)p.g * j.K + k) * mob + dob((int)mb)] = Sc[q];
      }
    } else if (kvalid) {
#pragma unroll
      for (int q = 0; q < G::CB; ++q) {
        const int64_t mb = p.m0 + rbeg + 16 * q;
        if (mb < j.M) Sc[q] = j.col_outer[((int64_t)p.g * j.K + k) * mob + dob((int)mb)];
      }
    }
    uint32_t ccw[2 * G::CB];
    uint32_t cscw = 0;
#pragma unroll
    for (int q = 0; q < G::CB; ++q) {
      const int64_t mb = p.m0 + rbeg + 16 * q;
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = rbeg + 16 * q + i;
        v[i] = staged ? staged_elem<IN_BF16>(xs, r, col) : raw_elem<IN_BF16>(raw, r, col);
      }
      if (!staged && fbits(amax16(v)) >= 0x7F800000u) {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = sanitize(v[i], IN_BF16 ? 0x7F7F0000u : 0x7F7FFFFFu);
      }
      Norm n;
      n.none = none;
      n.S = Sc[q];
      float4 T;
      uint32_t sc;
      float x[16];
      if (shared_S) {
        n.r = 1.0f;
        n.pos = true;
        n.fast = false;
        Norm pass = n;
        pass.none = true;  // staged values are normalized: the inner amax is max |x'|
        sc = block_scale<UE5M3>(tv, cam[q], pass, T);
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = v[i];
      } else {
        n.r = ieee_rcp(n.S);
        n.pos = positive(n.S);
        n.fast = positive_normal(n.S) && positive_normal(n.r);
        sc = block_scale<UE5M3>(tv, cam[q], n, T);
        normalize16<SR>(v, x, n);
      }
      // SR index of the column block: row g K + k0 + col of x transposed
      const uint64_t n0 = sr_col_n(j, p.g * j.K + p.k0 + col, p.m0 + rbeg + 16 * q);
      float deq[16];
      if (j.qdq_orient == 2) encode16<SR, true>(x, T, n, j.srk, j.step, 1u, n0, ccw[2 * q], ccw[2 * q + 1], deq);
      else encode16<SR, false>(x, T, n, j.srk, j.step, 1u, n0, ccw[2 * q], ccw[2 * q + 1], deq);
      cscw |= sc << (8 * q);
      if (j.qdq_orient == 2 && kvalid && mb < j.M) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int64_t yi = rbase + (int64_t)(rbeg + 16 * q + i) * K32 + col;
          if (j.out_bf16) static_cast<uint16_t*>(j.y)[yi] = (uint16_t)(pack_bf16x2(deq[i], 0.0f) & 0xFFFFu);
          else static_cast<float*>(j.y)[yi] = deq[i];
        }
      }
    }
    if (j.col_codes && kvalid) {
      const int64_t c0 = cbase + (int64_t)col * M32 + rbeg;
      const int nb = (int)min((int64_t)G::CB, (j.M - p.m0 - rbeg + 15) / 16);
      if (nb == G::CB && wide_codes && G::CB >= 2) {
        uint4* d = reinterpret_cast<uint4*>(j.col_codes + c0 / 2);
#pragma unroll
        for (int q = 0; q < G::CB / 2; ++q) d[q] = make_uint4(ccw[4 * q], ccw[4 * q + 1], ccw[4 * q + 2], ccw[4 * q + 3]);
      } else {
#pragma unroll
        for (int q = 0; q < G::CB; ++q)
          if (q < nb) *reinterpret_cast<uint2*>(j.col_codes + (c0 + 16 * q) / 2) = make_uint2(ccw[2 * q], ccw[2 * q + 1]);
      }
      if (nb == G::CB && wide_scales && G::CB == 2 && !j.csl.mma) {
        *reinterpret_cast<uint16_t*>(j.col_scales + c0 / 16) = (uint16_t)cscw;
      } else {
#pragma unroll
        for (int q = 0; q < G::CB; ++q)
          if (q < nb) j.col_scales[sf_from_linear(j.csl, c0 / 16 + q)] = (uint8_t)(cscw >> (8 * q));
      }
    }
    __syncthreads();
  }
}

// Tensor map of x as a (K, M, G) tensor with TM x 64 (bf16) or TM x 32
// (binary32) boxes and the 128-byte swizzle; false if it cannot be built.
template <bool IN_BF16>
bool make_tensor_map(const QuantJob& j, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t E = IN_BF16 ? 2 : 4;
  const cuuint64_t dims[3] = {(cuuint64_t)j.K, (cuuint64_t)j.M, (cuuint64_t)j.G};
  const cuuint64_t strides[2] = {(cuuint64_t)j.ld * E, (cuuint64_t)j.M * (cuuint64_t)j.ld * E};
  const cuuint32_t box[3] = {IN_BF16 ? 64u : 32u, (cuuint32_t)Geo<IN_BF16>::TM, 1u};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  const CUresult r = enc(map, IN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                         const_cast<void*>(j.x), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool IN_BF16, bool SR, bool COL, bool UE5M3>
cudaError_t launch_cp(const QuantJob& j, cudaStream_t st) {
  using L = Layout<IN_BF16, Stages<COL>::NS>;
  CUtensorMap map;
  if (!make_tensor_map<IN_BF16>(j, &map)) return launch_quant_tile(j, true, st);
  auto kern = cp_kernel<IN_BF16, SR, COL, UE5M3>;
  const bool staged = COL && (j.s_src == S_ONE || j.mode == 1 || j.outer_2d);
  const int smem = L::total(staged);
  static int per_sm_cache[2][128] = {{0}};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 128) dev = 0;
  int& per_sm = per_sm_cache[staged ? 1 : 0][dev];
  if (per_sm == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::total(true));
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
  }
  const int64_t tiles = j.G * ((j.M + Geo<IN_BF16>::TM - 1) / Geo<IN_BF16>::TM) * ((j.K + 63) / 64);
  const int64_t cap = (int64_t)num_sms() * per_sm;
  kern<<<(int)(tiles < cap ? tiles : cap), NT, smem, st>>>(j, map);
  return cudaGetLastError();
}

template <bool IN_BF16, bool SR>
cudaError_t launch_c(const QuantJob& j, cudaStream_t st) {
  const bool col = j.do_col != 0;
  if (j.ue5m3) return col ? launch_cp<IN_BF16, SR, true, true>(j, st) : launch_cp<IN_BF16, SR, false, true>(j, st);
  return col ? launch_cp<IN_BF16, SR, true, false>(j, st) : launch_cp<IN_BF16, SR, false, false>(j, st);
}

}  // namespace

bool ct_supports(const QuantJob& j) {
  if (j.inner_2d) return false;
  // 32-bit offsets inside a tile and a 32-bit tile counter
  const int64_t e = j.in_bf16 ? 2 : 4;
  if (j.ld * e >= (int64_t(1) << 24) || j.M >= (int64_t(1) << 24) || j.K >= (int64_t(1) << 24)) return false;
  if (j.G * ((j.M + 63) / 64) * ((j.K + 63) / 64) >= (int64_t(1) << 31)) return false;
  if (j.s_src == S_IN_TILE && !(j.ob == 16 || j.ob == 32 || j.ob == 64)) return false;
  return true;
}

cudaError_t launch_ct(const QuantJob& j, cudaStream_t st) {
  if (j.in_bf16) return j.sr ? launch_c<true, true>(j, st) : launch_c<true, false>(j, st);
  return j.sr ? launch_c<false, true>(j, st) : launch_c<false, false>(j, st);
}

cudaError_t ct_timeout_flag(uint32_t* v, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(v, g_tile_timeout, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_tile_timeout, &z, sizeof z);
  }
  return e;
}

}  // namespace fp4q
