// k_ctb.cuh -- the bf16 cast-transpose kernel body, instantiated without
// groups in k_ctb.cu and with ragged groups in k_ctb_grouped.cu (two
// translation units, compiled in parallel).  Design notes: k_ctb.cu.
#pragma once

#include "fp4q_block.cuh"
#include "fp4q_device.cuh"
#include "fp4q_internal.h"
#include "fp4q_tma.cuh"

namespace fp4q {
namespace {

constexpr int BT = 256;             // threads per CTA
constexpr int BM = 128, BK = 64;    // tile
constexpr int BNS = 2;              // tiles in flight (2 stages x 4 resident CTAs per SM)
constexpr int BRAW = BM * BK * 2;   // bytes of one raw tile
constexpr int CST = 72;             // bytes per staged column of codes (64 + 8 against bank conflicts)

// Shared memory (offsets from the 1024-byte aligned base)
struct BL {
  __host__ __device__ static constexpr int raw(int s) { return s * BRAW; }
  // Staging of the columnwise codes, scales and 1-D outer maxima comes in
  // two buffers picked by tile parity, so that one CTA barrier per tile
  // separates a tile's writes from its readers and the next tile's writes.
  // Codes: for the tensor store, [64 columns][64 bytes] with the 64-byte
  // swizzle (ccs, 1024-byte aligned); for the thread copy-out, 64 columns x
  // CST bytes (cst, the same region).
  __host__ __device__ static constexpr int ccs(int s) { return BNS * BRAW + s * 4096; }
  __host__ __device__ static constexpr int cst(int s) { return BNS * BRAW + s * 64 * CST; }
  static constexpr int tab = BNS * BRAW + 2 * 64 * CST;                     // 256 x (s, zh, zl, -)
  __host__ __device__ static constexpr int scales(int s) { return tab + 256 * 16 + s * 512; }  // 64 x 8
  // 2-D sub-tile maxima: 2 x 32 u32, picked by tile parity
  static constexpr int red2d = tab + 256 * 16 + 2 * 512;
  __host__ __device__ static constexpr int redc(int s) { return red2d + 256 + s * 1024; }  // 64 x 4 u32
  static constexpr int bars = red2d + 256 + 2 * 1024;                       // BNS mbarriers
  static constexpr int total = bars + 8 * BNS + 1024;                       // + alignment slack
};

// Outer-scale source of a launch
enum BOuter : int { BO_NONE = 0, BO_UNIFORM, BO_T1D, BO_T2D, BO_B1D, BO_B2D };

// Set by a tile wait that ran out (one flag per translation unit that
// includes this body); read and cleared from the host by fp4q_device_status.
__device__ unsigned int g_ctb_timeout = 0;

// Host side: this translation unit's flag on the current device.
inline cudaError_t ctb_flag_rw(uint32_t* v, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(v, g_ctb_timeout, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_ctb_timeout, &z, sizeof z);
  }
  return e;
}

__device__ __forceinline__ void issue_bf16_tile(const CUtensorMap* map, const TilePos& p, unsigned char* raw,
                                                uint64_t* bar) {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_tx(bar, (uint32_t)BRAW);
  tma_load3(raw, map, (int)p.k0, (int)p.m0, (int)p.g, bar);
}

__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Random Hadamard transform of a lane's two column blocks (16 rows each, the
// pair (column 2 l, column 2 l + 1) packed per row): signs, the fast
// Walsh-Hadamard butterfly h = 1, 2, 4, 8 in binary32, times 1/4 -- the
// same operations in the same order as the definition.
__device__ __forceinline__ void rht16x2(const uint32_t (&wv)[16], uint32_t signs, float (&z0)[16], float (&z1)[16]) {
  uint64_t p[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint64_t neg = ((signs >> i) & 1u) ? 0x8000000080000000ull : 0ull;
    p[i] = pk2(bf16lo(wv[i]), bf16hi(wv[i])) ^ neg;
  }
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & h) continue;
      const uint64_t a = p[i], b = p[i + h];
      p[i] = add2(a, b);
      p[i + h] = sub2(a, b);
    }
  }
  const uint64_t q = pk2(0.25f, 0.25f);
#pragma unroll
  for (int i = 0; i < 16; ++i) upk2(mul2(p[i], q), z0[i], z1[i]);
}

// Per-block steps shared by both passes: inner scale, x' = u / S, codes.
// With an outer scale (NEG) the block arrives negated, v = -u.
template <bool SR, bool UE5M3, bool NEG>
__device__ __forceinline__ uint32_t quant_block(const float4* tab, const float (&v)[16], float am, float S, float r,
                                                bool none, const QuantJob& j, uint32_t orient, uint64_t n0,
                                                uint32_t& w0, uint32_t& w1) {
  Norm n;
  n.none = none;
  n.S = S;
  n.r = r;
  n.pos = none || positive(S);
  n.fast = !none && positive_normal(S) && positive_normal(r);
  struct {
    const float4* tab;
  } tv{tab};
  float4 T;
  const uint32_t sc = block_scale<UE5M3>(tv, am, n, T);
  float x[16], dq[16];
  if (NEG) normalize16_neg<SR>(v, x, n);
  else normalize16<SR>(v, x, n);
  encode16<SR, false>(x, T, n, j.srk, j.step, orient, n0, w0, w1, dq);
  return sc;
}

// FT, bit 0: every tile is whole along K (K a multiple of 64), so the
// column edge checks fold away.  Bit 1: whole along M too (M a multiple of
// 128, no groups), both orientations are written, the columnwise codes
// leave by the tensor store, the row codes are 16-byte aligned and the
// inner scales use the linear layout, so the row edge checks and these
// branches fold away as well.
template <bool SR, bool UE5M3, int BO, bool GR, bool RHT, int OBC, int FT>
__global__ void __launch_bounds__(BT, (RHT || SR) ? 3 : 4) ctb_kernel(const QuantJob j, const __grid_constant__ CUtensorMap tmap,
                                                          const __grid_constant__ CUtensorMap cmap, int col_tma_) {
  constexpr bool FTK = (FT & 1) != 0, FTM = (FT & 2) != 0;
  const int col_tma = FTM ? 1 : col_tma_;
  pdl_wait_then_release();
  extern __shared__ __align__(16) unsigned char smem_dyn[];
  unsigned char* smem = smem_align1024(smem_dyn);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  float4* tab = reinterpret_cast<float4*>(smem + BL::tab);
  uint32_t* red2d = reinterpret_cast<uint32_t*>(smem + BL::red2d);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BL::bars);

  // grouped inputs: rows [goff[e], goff[e + 1]) form group e, quantized as
  // a matrix of its own; the walk covers each group's 128-row tiles
  constexpr bool gr = GR;
  const uint32_t* gtp = gr ? group_tprefix(j.gws) : nullptr;
  if (gr && j.gws->bad) return;  // invalid offsets: write nothing
  TileIter cur;
  if (gr) cur.init_n((int)((j.K + 63) / 64), (int)j.gws->mtiles, 1);
  else cur.init<BM>(j);
  GroupCursor gc, pc;  // processing cursor (all threads), prefetch cursor (thread 0)
  auto tile_at = [&](int i) -> TilePos {
    if (!gr) return cur.pos_of<BM>(i);
    const uint32_t q = (uint32_t)(i / cur.tiles_k);
    pc.seek(gtp, q);
    return TilePos{0, j.goff[pc.e] + 128 * (int64_t)(q - pc.lo), (int64_t)(i - (int)q * cur.tiles_k) * 64};
  };
  if (t == 0) {
#pragma unroll
    for (int s = 0; s < BNS; ++s) mbar_init(&bars[s]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (t == 0) {
#pragma unroll
    for (int s = 0; s < BNS - 1; ++s) {
      const int i = cur.idx + s * (int)gridDim.x;
      if (i < cur.ntiles) issue_bf16_tile(&tmap, tile_at(i), smem + BL::raw(s), &bars[s]);
    }
  }
  build_scale_table<UE5M3>(tab, t, BT);
  if (t < 64) red2d[t] = 0u;
  reinterpret_cast<uint32_t*>(smem + BL::redc(0))[t] = 0u;
  reinterpret_cast<uint32_t*>(smem + BL::redc(1))[t] = 0u;

  const bool none = BO == BO_NONE;
  // OBC: the outer block size fixed at compile time (0: taken from the job)
  const int ob = OBC ? OBC : j.ob;
  const int lob = OBC ? (OBC == 64 ? 6 : OBC == 32 ? 5 : 4) : (ob > 0 ? 31 - __clz(ob) : 0);
  const bool ob_pow2 = OBC ? true : (ob > 0 && (ob & (ob - 1)) == 0);
  const int64_t mob = ob > 0 ? j.M / ob : 0, kob = ob > 0 ? j.K / ob : 0;
  float S_u = 1.0f, r_u = 1.0f;
  int64_t s_group = -1;  // group whose tensorwise scale S_u holds (grouped path)
  if (BO == BO_UNIFORM && gr) {
  } else if (BO == BO_UNIFORM) {
    if (j.s_src == S_TENSORWISE_WS) {
      S_u = ieee_div(bitsf(*j.tw_amax), UE5M3 ? 688128.0f : 2688.0f);
      if (blockIdx.x == 0 && t == 0 && j.tile_outer) j.tile_outer[0] = S_u;
    } else {
      S_u = j.tile_outer[0];
    }
    r_u = ieee_rcp(S_u);
  }
  const int64_t M = j.M, K = j.K;
  const bool row_wide = FTM || ((K % 32) == 0 && ((reinterpret_cast<uintptr_t>(j.row_codes) & 15u) == 0) &&
                               ((reinterpret_cast<uintptr_t>(j.row_scales) & 1u) == 0));

  // rowwise ownership
  const int rr = t >> 1, rh = t & 1;
  // columnwise ownership: rows 16 warp .., columns 2 lane, 2 lane + 1; the
  // swizzled byte offset of this lane's pair in row 16 warp + i is
  // rowbase + (cunit ^ (i mod 8)) * 16 + cbyte
  const int cunit = lane >> 2, cbyte = (lane & 3) * 4;
  __syncthreads();

  int slot = 0;
  uint32_t phase = 0;
  for (int it = 0; cur.valid(); ++it) {
    const unsigned char* raw = smem + BL::raw(slot);
    unsigned char* cst = smem + BL::cst(it & 1);
    unsigned char* sst = smem + BL::scales(it & 1);
    uint32_t* redc = reinterpret_cast<uint32_t*>(smem + BL::redc(it & 1));
    TilePos p = cur.pos<BM>();
    // the tile's group: rows [goff, gend), columnwise index of (k, m) =
    // cbase + k * cstride + m (the group's own [K, rows] transpose)
    int64_t gend = M, goff = 0, cbase = p.g * K * M, cstride = M;
    if (gr) {
      gc.seek(gtp, (uint32_t)cur.tm);
      goff = j.goff[gc.e];
      gend = j.goff[gc.e + 1];
      p = TilePos{0, goff + 128 * (int64_t)((uint32_t)cur.tm - gc.lo), p.k0};
      cbase = K * goff - goff;
      cstride = gend - goff;
      if (BO == BO_UNIFORM && gc.e != s_group) {  // the group's tensorwise scale
        s_group = gc.e;
        S_u = ieee_div(bitsf(group_amax(j.gws, j.ngroups)[gc.e]), UE5M3 ? 688128.0f : 2688.0f);
        r_u = ieee_rcp(S_u);
      }
      if (BO == BO_UNIFORM && t == 0 && p.m0 == goff && p.k0 == 0 && j.tile_outer) j.tile_outer[gc.e] = S_u;
    }
    if (t == 0) {
      const int i = cur.idx + (BNS - 1) * (int)gridDim.x;
      const int s = slot == 0 ? BNS - 1 : slot - 1;
      if (i < cur.ntiles) issue_bf16_tile(&tmap, tile_at(i), smem + BL::raw(s), &bars[s]);
    }
    cur.next();
    // Each thread waits for the tile itself (no CTA barrier).  A wait that
    // runs out raises the error flag and the walk goes on with whatever the
    // slot holds: every later wait is bounded and every barrier is still
    // reached by all threads.
    if (!mbar_wait(&bars[slot], phase, 1u << 22)) atomicExch(&g_ctb_timeout, 1u);
    if (++slot == BNS) {
      slot = 0;
      phase ^= 1u;
    }

    // ------------------------------------------------------------ rowwise
    const int64_t m = p.m0 + rr;
    const bool rvalid = FTM || m < gend;
    const int64_t rel = (p.g * M + m) * K + p.k0 + 32 * rh;  // flat index of this thread's first element
    uint4 a[4] = {};
    float am[2] = {0.0f, 0.0f};
    if (FTM || j.do_row || BO == BO_T2D) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      a[q] = *reinterpret_cast<const uint4*>(raw + (rr * 8 + ((4 * rh + q) ^ (rr & 7))) * 16);
#pragma unroll
    for (int b = 0; b < 2; ++b)
      am[b] = bf16x2_hmax(bf16x2_amax(bf16x2_amax(bf16x2_amax(a[2 * b].x, a[2 * b].y), bf16x2_amax(a[2 * b].z, a[2 * b].w)),
                                      bf16x2_amax(bf16x2_amax(a[2 * b + 1].x, a[2 * b + 1].y),
                                                  bf16x2_amax(a[2 * b + 1].z, a[2 * b + 1].w))));
    if (fbits(am[0]) >= 0x7F800000u || fbits(am[1]) >= 0x7F800000u) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        a[q].x = sanitize_bf16x2(a[q].x); a[q].y = sanitize_bf16x2(a[q].y);
        a[q].z = sanitize_bf16x2(a[q].z); a[q].w = sanitize_bf16x2(a[q].w);
      }
#pragma unroll
      for (int b = 0; b < 2; ++b)
        am[b] = bf16x2_hmax(bf16x2_amax(bf16x2_amax(bf16x2_amax(a[2 * b].x, a[2 * b].y), bf16x2_amax(a[2 * b].z, a[2 * b].w)),
                                        bf16x2_amax(bf16x2_amax(a[2 * b + 1].x, a[2 * b + 1].y),
                                                    bf16x2_amax(a[2 * b + 1].z, a[2 * b + 1].w))));
    }
    }

    // 2-D outer scales of the tile's ob x ob sub-blocks: the maxima meet in
    // the tile's half of red2d; after one barrier every thread derives the S
    // and 1 / S it needs from them
    uint32_t* r2 = red2d + 32 * (it & 1);
    if (BO == BO_T2D) {
      uint32_t v = umax(fbits(am[0]), fbits(am[1]));
      uint32_t v0 = fbits(am[0]), v1 = fbits(am[1]);
      if (ob >= 32) v0 = v1 = v;
      if (ob == 64) { v0 = umax(v0, __shfl_xor_sync(0xFFFFFFFFu, v0, 1)); v1 = v0; }
      // rows of this warp: lanes 2 apart
#pragma unroll
      for (int o = 2; o < 32; o <<= 1) {
        v0 = umax(v0, __shfl_xor_sync(0xFFFFFFFFu, v0, o));
        v1 = umax(v1, __shfl_xor_sync(0xFFFFFFFFu, v1, o));
      }
      const int nbk = 64 >> lob;
      if (lane < 2) {
        // sub-block column of this thread's blocks: (32 rh + 16 b) >> lob
        const int sb0 = (32 * rh) >> lob, sb1 = (32 * rh + 16) >> lob;
        const int srow = (16 * warp) >> lob;
        if (ob == 16) {
          r2[srow * nbk + sb0] = v0;
          r2[srow * nbk + sb1] = v1;
        } else {
          atomicMax(&r2[srow * nbk + sb0], v0);
          if (sb1 != sb0) atomicMax(&r2[srow * nbk + sb1], v1);
        }
      }
      __syncthreads();
      // the next tile's half: its last readers (the previous tile) are past
      // the previous tile's final barrier, its next writers past this one's
      if (t < 32) red2d[32 * ((it + 1) & 1) + t] = 0u;
      const int nsub = (BM >> lob) * nbk;
      if (t < nsub && j.tile_outer) {
        const int64_t mi = p.m0 + (int64_t)(t / nbk) * ob, kj = p.k0 + (int64_t)(t % nbk) * ob;
        if ((FTM || mi < gend) && (FTK || kj < K)) j.tile_outer[(p.g * mob + mi / ob) * kob + kj / ob] = outer_scale<UE5M3>(bitsf(r2[t]));
      }
    }

    if (FTM || j.do_row) {
      float S[2] = {1.0f, 1.0f}, R[2] = {1.0f, 1.0f};
      if (BO == BO_UNIFORM) {
        S[0] = S[1] = S_u;
        R[0] = R[1] = r_u;
      } else if (BO == BO_T1D) {
        uint32_t g0 = fbits(am[0]), g1 = fbits(am[1]);
        if (ob >= 32) g0 = g1 = umax(g0, g1);
        if (ob == 64) { g0 = umax(g0, __shfl_xor_sync(0xFFFFFFFFu, g0, 1)); g1 = g0; }
        outer_sr<UE5M3>(bitsf(g0), S[0], R[0]);
        if (ob == 16) {
          outer_sr<UE5M3>(bitsf(g1), S[1], R[1]);
        } else {
          S[1] = S[0];
          R[1] = R[0];
        }
        if (j.row_outer && rvalid) {
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            const int64_t e = rel + 16 * b;
            if ((FTK || p.k0 + 32 * rh + 16 * b < K) && (e & (ob - 1)) == 0) j.row_outer[e >> lob] = S[b];
          }
        }
      } else if (BO == BO_T2D) {
        const int i0 = ((16 * warp + (lane >> 1)) >> lob) * (64 >> lob);
        outer_sr<UE5M3>(bitsf(r2[i0 + ((32 * rh) >> lob)]), S[0], R[0]);
        if (ob == 16) {
          outer_sr<UE5M3>(bitsf(r2[i0 + ((32 * rh + 16) >> lob)]), S[1], R[1]);
        } else {
          S[1] = S[0];
          R[1] = R[0];
        }
      } else if (BO == BO_B1D || BO == BO_B2D) {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const int64_t kb = p.k0 + 32 * rh + 16 * b;
          if (rvalid && (FTK || kb < K)) {
            if (BO == BO_B1D) S[b] = j.row_outer[ob_pow2 ? ((rel + 16 * b) >> lob) : (rel + 16 * b) / ob];
            else S[b] = j.tile_outer[(p.g * mob + m / ob) * kob + kb / ob];
          }
          R[b] = ieee_rcp(S[b]);
        }
      }
      uint32_t cw[4], scw = 0;
      // the fast form with RNE only (stochastic rounding is Philox-bound and
      // keeps the general form's register budget)
      float ab[2] = {am[0], am[1]};
      bool fast = !SR;
      if (!SR && BO != BO_NONE) {
#pragma unroll
        for (int b = 0; b < 2; ++b) fast = fast_block(am[b], S[b], R[b], ab[b]) && fast;
        fast = __all_sync(0xFFFFFFFFu, fast);
      }
      // block b of this thread as u (or -u with an outer scale)
      auto row_u = [&](int b, float (&u)[16]) {
        const uint32_t wd[8] = {a[2 * b].x, a[2 * b].y, a[2 * b].z, a[2 * b].w,
                                a[2 * b + 1].x, a[2 * b + 1].y, a[2 * b + 1].z, a[2 * b + 1].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          u[2 * i] = BO == BO_NONE ? bf16lo(wd[i]) : nbf16lo(wd[i]);
          u[2 * i + 1] = BO == BO_NONE ? bf16hi(wd[i]) : nbf16hi(wd[i]);
        }
      };
      if (fast) {  // one branch for both blocks: straight-line code the scheduler can interleave
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          float u[16];
          row_u(b, u);
          scw |= block_fast<SR, UE5M3, BO != BO_NONE, BO != BO_NONE>(tab, u, ab[b], S[b], R[b], j.srk, j.step, 0u,
                                                                      sr_row_n(j, rel + 16 * b), cw[2 * b],
                                                                      cw[2 * b + 1])
                 << (8 * b);
        }
      } else {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          float u[16];
          row_u(b, u);
          scw |= quant_block<SR, UE5M3, BO != BO_NONE>(tab, u, am[b], S[b], R[b], none, j, 0u,
                                                       sr_row_n(j, rel + 16 * b), cw[2 * b], cw[2 * b + 1])
                 << (8 * b);
        }
      }
      if (rvalid) {
        const int nb = FTK ? 2 : (int)min((int64_t)2, (K - p.k0 - 32 * rh) / 16);
        // scale byte offset: linear rel / 16; tensor-core tiles: the tile of
        // (m0 / 128, k0 / 64), row rr of it, columns 2 rh and 2 rh + 1
        const int64_t so = (!FTM && j.rsl.mma) ? ((p.g * j.rsl.nrb + (p.m0 >> 7)) * j.rsl.ncb + (p.k0 >> 6)) * 512 +
                                           ((rr & 31) << 4) + ((rr >> 5) << 2) + 2 * rh
                                     : rel / 16;
        if (nb == 2 && row_wide) {
          *reinterpret_cast<uint4*>(j.row_codes + rel / 2) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
          *reinterpret_cast<uint16_t*>(j.row_scales + so) = (uint16_t)scw;
        } else {
          if (nb >= 1) {
            *reinterpret_cast<uint2*>(j.row_codes + rel / 2) = make_uint2(cw[0], cw[1]);
            j.row_scales[so] = (uint8_t)scw;
          }
          if (nb >= 2) {
            *reinterpret_cast<uint2*>(j.row_codes + rel / 2 + 8) = make_uint2(cw[2], cw[3]);
            j.row_scales[so + 1] = (uint8_t)(scw >> 8);
          }
        }
      }
    }

    // --------------------------------------------------------- columnwise
    if (!FTM && !j.do_col) {  // rowwise-only call (tensor-core scale layout)
      __syncthreads();
      continue;
    }
    uint32_t wv[16];
    {
      const unsigned char* rb = raw + warp * 16 * 128 + cbyte;
#pragma unroll
      for (int i = 0; i < 16; ++i) wv[i] = *reinterpret_cast<const uint32_t*>(rb + i * 128 + ((cunit ^ (i & 7)) << 4));
    }
    uint32_t mx = bf16x2_amax(wv[0], wv[1]);
#pragma unroll
    for (int i = 2; i < 16; i += 2) mx = bf16x2_amax(mx, bf16x2_amax(wv[i], wv[i + 1]));
    mx &= 0x7FFF7FFFu;
    if ((mx & 0xFFFFu) >= 0x7F80u || (mx >> 16) >= 0x7F80u) {
#pragma unroll
      for (int i = 0; i < 16; ++i) wv[i] = sanitize_bf16x2(wv[i]);
      mx = bf16x2_amax(wv[0], wv[1]);
#pragma unroll
      for (int i = 2; i < 16; i += 2) mx = bf16x2_amax(mx, bf16x2_amax(wv[i], wv[i + 1]));
      mx &= 0x7FFF7FFFu;
    }
    float cam[2] = {bitsf(mx << 16), bitsf(mx & 0xFFFF0000u)};
    // columnwise Hadamard transform along M (the rowwise side is untouched)
    float z0[16], z1[16];
    if (RHT) {
      rht16x2(wv, j.rht_signs, z0, z1);
      cam[0] = amax16(z0);
      cam[1] = amax16(z1);
      if (fbits(cam[0]) >= 0x7F800000u || fbits(cam[1]) >= 0x7F800000u) {  // the sums left the range
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          z0[i] = sanitize(z0[i], 0x7F7F0000u);
          z1[i] = sanitize(z1[i], 0x7F7F0000u);
        }
        cam[0] = amax16(z0);
        cam[1] = amax16(z1);
      }
    }
    const int64_t mb = p.m0 + 16 * warp;  // first row of this lane's blocks
    const bool mvalid = FTM || mb < gend;
    float S[2] = {1.0f, 1.0f}, R[2] = {1.0f, 1.0f};
    if (BO == BO_UNIFORM) {
      S[0] = S[1] = S_u;
      R[0] = R[1] = r_u;
    } else if (BO == BO_T1D) {
      uint32_t g[2] = {fbits(cam[0]), fbits(cam[1])};
      if (ob > 16) {  // the outer block spans ob / 16 warps
        const int grp = (16 * warp) >> lob;
#pragma unroll
        for (int c = 0; c < 2; ++c) atomicMax(&redc[(2 * lane + c) * 4 + grp], g[c]);
        __syncthreads();
#pragma unroll
        for (int c = 0; c < 2; ++c) g[c] = redc[(2 * lane + c) * 4 + grp];
      }
      outer_sr2<UE5M3>(bitsf(g[0]), bitsf(g[1]), S, R);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int64_t k = p.k0 + 2 * lane + c;
        if (j.col_outer && (FTK || k < K) && mvalid && ((16 * warp) & (ob - 1)) == 0)
          j.col_outer[(cbase + k * cstride + mb) >> lob] = S[c];
      }
    } else if (BO == BO_T2D) {
      // columns 2 lane and 2 lane + 1 lie in one sub-block (ob >= 16)
      outer_sr<UE5M3>(bitsf(r2[((16 * warp) >> lob) * (64 >> lob) + ((2 * lane) >> lob)]), S[0], R[0]);
      S[1] = S[0];
      R[1] = R[0];
    } else if (BO == BO_B1D || BO == BO_B2D) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int64_t k = p.k0 + 2 * lane + c;
        if ((FTK || k < K) && mvalid) {
          if (BO == BO_B1D) S[c] = j.col_outer[ob_pow2 ? ((cbase + k * cstride + mb) >> lob) : (cbase + k * cstride + mb) / ob];
          else S[c] = j.tile_outer[(p.g * mob + (ob_pow2 ? (mb >> lob) : mb / ob)) * kob + (ob_pow2 ? (k >> lob) : k / ob)];
        }
        R[c] = ieee_rcp(S[c]);
      }
    }
    float ac[2] = {cam[0], cam[1]};
    bool cfast = !SR;
    if (!SR && BO != BO_NONE) {
#pragma unroll
      for (int c = 0; c < 2; ++c) cfast = fast_block(cam[c], S[c], R[c], ac[c]) && cfast;
      cfast = __all_sync(0xFFFFFFFFu, cfast);
    }
    // column c of this lane as u (or -u with an outer scale; the transformed
    // z with the Hadamard transform)
    auto col_u = [&](int c, float (&u)[16]) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        u[i] = RHT ? (c ? z1[i] : z0[i])
                   : (BO == BO_NONE ? (c ? bf16hi(wv[i]) : bf16lo(wv[i])) : (c ? nbf16hi(wv[i]) : nbf16lo(wv[i])));
    };
    // SR index of column 2 lane + c's block: the group's own flat index in
    // the concatenated group transposes, else the global index of x
    // transposed (row g K + k)
    auto col_sr = [&](int c) -> uint64_t {
      const int64_t k = p.k0 + 2 * lane + c;
      return GR ? (uint64_t)(cbase + k * cstride + mb) : sr_col_n(j, p.g * K + k, mb);
    };
    // codes of column 2 lane + c, rows 16 warp .. + 15: row 2 lane + c of
    // the tensor-store box at byte 8 warp, whose 16-byte chunk index the
    // 64-byte swizzle XORs with (row / 2) mod 4 = lane mod 4; or the padded
    // staging rows of the thread copy-out
    unsigned char* cbuf = smem + BL::ccs(it & 1);
    auto col_stage = [&](int c, uint32_t w0, uint32_t w1, uint32_t sc) {
      if (!GR && col_tma)
        *reinterpret_cast<uint2*>(cbuf + ((((2 * lane + c) << 6) + 8 * warp) ^ ((lane & 3) << 4))) = make_uint2(w0, w1);
      else
        *reinterpret_cast<uint2*>(cst + (2 * lane + c) * CST + 8 * warp) = make_uint2(w0, w1);
      sst[(2 * lane + c) * 8 + warp] = (uint8_t)sc;
    };
    if (cfast) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float u[16];
        col_u(c, u);
        uint32_t w0, w1;
        const uint32_t sc = block_fast<SR, UE5M3, BO != BO_NONE, BO != BO_NONE && !RHT>(
            tab, u, ac[c], S[c], R[c], j.srk, j.step, 1u, col_sr(c), w0, w1);
        col_stage(c, w0, w1, sc);
      }
    } else {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float u[16];
        col_u(c, u);
        uint32_t w0, w1;
        const uint32_t sc = quant_block<SR, UE5M3, BO != BO_NONE && !RHT>(
            tab, u, cam[c], S[c], R[c], none, j, 1u, col_sr(c), w0, w1);
        col_stage(c, w0, w1, sc);
      }
    }
    if (!GR && col_tma) fence_proxy_async();
    // the previous tile's store has read its buffer, which the next tile's
    // writers (past the barrier below) take over
    if (!GR && col_tma && t == 0) bulk_wait_read_0();
    __syncthreads();
    if (!GR && col_tma && t == 0) {  // the tile's columnwise codes: [64 columns][128 rows / 2] bytes
      tma_store3(&cmap, cbuf, (int)(p.m0 >> 1), (int)p.k0, (int)p.g);
      bulk_commit();
    }
    if (BO == BO_T1D && ob > 16 && ((16 * warp) & (ob - 1)) == 0) {
#pragma unroll
      for (int c = 0; c < 2; ++c) redc[(2 * lane + c) * 4 + ((16 * warp) >> lob)] = 0u;
    }
    // copy-out: thread t stores rows 32 (t mod 4) .. + 31 of column t / 4
    {
      const int col = t >> 2, ch = t & 3;
      const int64_t k = p.k0 + col;
      const int64_t m1 = p.m0 + 32 * ch;
      if ((GR || !col_tma) && (FTK || k < K) && (FTM || m1 < gend)) {
        const int nb = FTM ? 2 : (int)min((int64_t)2, (gend - m1) / 16);
        const uint2 c0 = *reinterpret_cast<const uint2*>(cst + col * CST + 16 * ch);
        const uint2 c1 = *reinterpret_cast<const uint2*>(cst + col * CST + 16 * ch + 8);
        uint8_t* d = j.col_codes + (cbase + k * cstride + m1) / 2;
        if (nb == 2 && (reinterpret_cast<uintptr_t>(d) & 15u) == 0) {
          *reinterpret_cast<uint4*>(d) = make_uint4(c0.x, c0.y, c1.x, c1.y);
        } else {
          *reinterpret_cast<uint2*>(d) = c0;
          if (nb == 2) *reinterpret_cast<uint2*>(d + 8) = c1;
        }
      }
      if (t < 64) {
        const int64_t kk = p.k0 + t;
        if (FTK || kk < K) {
          const int nbm = FTM ? 8 : (int)min((int64_t)8, (gend - p.m0) / 16);
          const uint2 v = *reinterpret_cast<const uint2*>(sst + t * 8);
          if (!FTM && j.csl.mma) {
            // scale columns m0 / 16 + 4 h .. + 3 of row kk: 4 bytes of tile
            // (kk / 128, m0 / 64 + h)
            uint8_t* d = j.col_scales + ((p.g * j.csl.nrb + (kk >> 7)) * j.csl.ncb + (p.m0 >> 6)) * 512 +
                         ((kk & 31) << 4) + (((kk >> 5) & 3) << 2);
            if (nbm == 8) {
              *reinterpret_cast<uint32_t*>(d) = v.x;
              *reinterpret_cast<uint32_t*>(d + 512) = v.y;
            } else {
              for (int q = 0; q < nbm; ++q) d[(q >> 2) * 512 + (q & 3)] = (uint8_t)((q < 4 ? v.x : v.y) >> (8 * (q & 3)));
            }
          } else {
            uint8_t* d = j.col_scales + (cbase + kk * cstride + p.m0) / 16;
            if (nbm == 8 && (reinterpret_cast<uintptr_t>(d) & 7u) == 0) {
              *reinterpret_cast<uint2*>(d) = v;
            } else {
              for (int q = 0; q < nbm; ++q) d[q] = (uint8_t)((q < 4 ? v.x : v.y) >> (8 * (q & 3)));
            }
          }
        }
      }
    }
  }
  if (!GR && col_tma && t == 0) bulk_wait_all();
}

bool make_bf16_map(const QuantJob& j, CUtensorMap* map) { return make_bf16_tile_map(j, map, BM); }

template <bool SR, bool UE5M3, int BO, bool GR, bool RHT, int OBC = 0, int FT = 0>
cudaError_t launch_ctb_t(const QuantJob& j, const CUtensorMap& map, const CUtensorMap& cmap, int col_tma,
                         cudaStream_t st) {
  auto kern = ctb_kernel<SR, UE5M3, BO, GR, RHT, OBC, FT>;
  static int per_sm_cache[128] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 128) dev = 0;
  int& per_sm = per_sm_cache[dev];
  if (per_sm == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BL::total);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, BT, BL::total);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
  }
  // grouped: the tile count lives on the device; an upper bound is
  // ceil(M / 128) + groups 128-row tiles per 64-column strip
  const int64_t tiles = j.ngroups > 0 ? ((j.M + BM - 1) / BM + j.ngroups) * ((j.K + BK - 1) / BK)
                                      : j.G * ((j.M + BM - 1) / BM) * ((j.K + BK - 1) / BK);
  const int64_t cap = (int64_t)num_sms() * per_sm;
  return launch_pdl(kern, dim3((unsigned)(tiles < cap ? tiles : cap)), dim3(BT), (size_t)BL::total, st, j, map, cmap,
                    col_tma);
}

template <bool SR, bool UE5M3, bool GR, bool RHT>
cudaError_t launch_ctb_o(const QuantJob& j, const CUtensorMap& map, const CUtensorMap& cmap, int col_tma,
                         cudaStream_t st) {
  // whole tiles: the edge checks folded away
  const bool whole = j.M % BM == 0 && j.K % BK == 0 && col_tma && j.do_row && j.do_col && !j.rsl.mma && !j.csl.mma &&
                     (reinterpret_cast<uintptr_t>(j.row_codes) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(j.row_scales) & 1u) == 0;
  if constexpr (RHT) {  // the transform is defined with no outer scale or 1-D outer blocks
    if constexpr (!SR && !GR) {
      if (whole && j.s_src == S_ONE) return launch_ctb_t<SR, UE5M3, BO_NONE, GR, true, 0, 3>(j, map, cmap, col_tma, st);
      if (whole && j.s_src == S_IN_TILE && j.ob == 64)
        return launch_ctb_t<SR, UE5M3, BO_T1D, GR, true, 64, 3>(j, map, cmap, col_tma, st);
    }
    if (j.s_src == S_ONE) return launch_ctb_t<SR, UE5M3, BO_NONE, GR, true>(j, map, cmap, col_tma, st);
    return launch_ctb_t<SR, UE5M3, BO_T1D, GR, true>(j, map, cmap, col_tma, st);
  } else {
    if constexpr (!SR && !GR) {
      if (whole) {
        if (j.s_src == S_ONE) return launch_ctb_t<SR, UE5M3, BO_NONE, GR, false, 0, 3>(j, map, cmap, col_tma, st);
        if (j.s_src == S_TENSORWISE_WS || j.mode == 1)
          return launch_ctb_t<SR, UE5M3, BO_UNIFORM, GR, false, 0, 3>(j, map, cmap, col_tma, st);
        if (j.s_src == S_IN_TILE && j.ob == 64)
          return j.outer_2d ? launch_ctb_t<SR, UE5M3, BO_T2D, GR, false, 64, 3>(j, map, cmap, col_tma, st)
                            : launch_ctb_t<SR, UE5M3, BO_T1D, GR, false, 64, 3>(j, map, cmap, col_tma, st);
      }
    }
    if (j.s_src == S_ONE) return launch_ctb_t<SR, UE5M3, BO_NONE, GR, false>(j, map, cmap, col_tma, st);
    if (j.s_src == S_TENSORWISE_WS || j.mode == 1)
      return launch_ctb_t<SR, UE5M3, BO_UNIFORM, GR, false>(j, map, cmap, col_tma, st);
    if constexpr (!SR) {  // the common 64-element outer block, its size folded into the code
      if (j.s_src == S_IN_TILE && j.ob == 64) {
        if constexpr (GR) {  // ragged groups: whole along K only
          if (j.K % BK == 0)
            return j.outer_2d ? launch_ctb_t<SR, UE5M3, BO_T2D, GR, false, 64, 1>(j, map, cmap, col_tma, st)
                              : launch_ctb_t<SR, UE5M3, BO_T1D, GR, false, 64, 1>(j, map, cmap, col_tma, st);
        }
        return j.outer_2d ? launch_ctb_t<SR, UE5M3, BO_T2D, GR, false, 64>(j, map, cmap, col_tma, st)
                          : launch_ctb_t<SR, UE5M3, BO_T1D, GR, false, 64>(j, map, cmap, col_tma, st);
      }
    }
    if (j.s_src == S_IN_TILE)
      return j.outer_2d ? launch_ctb_t<SR, UE5M3, BO_T2D, GR, false>(j, map, cmap, col_tma, st)
                        : launch_ctb_t<SR, UE5M3, BO_T1D, GR, false>(j, map, cmap, col_tma, st);
    return j.outer_2d ? launch_ctb_t<SR, UE5M3, BO_B2D, GR, false>(j, map, cmap, col_tma, st)
                      : launch_ctb_t<SR, UE5M3, BO_B1D, GR, false>(j, map, cmap, col_tma, st);
  }
}

// All variants of one grouping / transform mode: false if the tensor map
// cannot be built.
template <bool GR, bool RHT>
bool launch_ctb_all(const QuantJob& j, cudaStream_t st, cudaError_t* err) {
  CUtensorMap map, cmap;
  if (!make_bf16_map(j, &map)) return false;
  const int col_tma = make_col_map(j, &cmap) ? 1 : 0;
  if (!col_tma) cmap = map;  // unused by the kernel
  if (j.sr)
    *err = j.ue5m3 ? launch_ctb_o<true, true, GR, RHT>(j, map, cmap, col_tma, st)
                   : launch_ctb_o<true, false, GR, RHT>(j, map, cmap, col_tma, st);
  else
    *err = j.ue5m3 ? launch_ctb_o<false, true, GR, RHT>(j, map, cmap, col_tma, st)
                   : launch_ctb_o<false, false, GR, RHT>(j, map, cmap, col_tma, st);
  return true;
}

}  // namespace
}  // namespace fp4q
