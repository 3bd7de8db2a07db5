// k_tile.cu -- fused quantize / cast-transpose / QDQ tile kernel.
//
// One CTA of 256 threads owns a 64 x 64 tile of x at a time (grid-stride over
// tiles).  The tile is read from HBM once, widened to binary32 (plus the
// error-feedback residual, then sanitized) into shared memory, and from there
//   - the rowwise pass (one thread per 1 x 16 segment) writes rowwise codes,
//     inner scales, 1-D outer scales, the residual update and rowwise QDQ;
//   - the columnwise pass (one thread per 16 x 1 segment) writes the
//     transposed codes / scales / outer scales and columnwise QDQ.
// A 2-D outer scale (ob x ob, ob dividing 64) is reduced once per tile and
// shared by both passes ("Block-Scaled FP8 and FP4 Weight Quantization",
// section 6; "NVFP4 / AMD-FP4 outer-block scaling", "Implementation").
// Outer blocks that do not divide the tile come from a pre-pass kernel and
// are read back (S_FROM_BUFFER).
#include "fp4q_device.cuh"
#include "fp4q_internal.h"

namespace fp4q {
namespace {

constexpr int TILE = 64;
constexpr int LDS = TILE + 4;  // padded row stride of the shared tile (floats)
constexpr int NTHR = 256;

struct TileSmem {
  float u[TILE * LDS];
  uint32_t am_row[4][TILE];  // per (segment, row) 1x16 amax bits, rowwise pass
  uint32_t am_col[4][TILE];  // per (segment, column) 16x1 amax bits, columnwise pass
  uint32_t part[4][4];       // partial maxima for the 2-D outer reduction
  float S2[4][4];            // 2-D outer scales of the tile's ob x ob sub-tiles
};

__device__ __forceinline__ uint32_t umax(uint32_t a, uint32_t b) { return a > b ? a : b; }

// 1-D outer block amax over the segments [s0, s0 + n) of one row/column.
__device__ __forceinline__ uint32_t seg_group_max(const uint32_t (*am)[TILE], int s0, int n, int idx) {
  uint32_t v = 0;
  for (int s = s0; s < s0 + n; ++s) v = umax(v, am[s][idx]);
  return v;
}

// Shared per-segment arithmetic: from the 16 values u[] and the outer scale S
// (no_outer: S == 1), produce 16 codes (packed into 8 bytes), the inner-scale
// code and, if wanted, the dequantized values.
struct SegOut {
  uint32_t codes_lo, codes_hi;  // bytes 0-3 and 4-7
  uint32_t sc;
};

template <bool WANT_DEQ>
__device__ __forceinline__ SegOut quantize_segment(const float (&u)[16], float S, bool no_outer, uint32_t a_bits,
                                                   const ScaleFmt& f, bool sr, const PhiloxKeys& K, uint32_t step,
                                                   uint32_t orient, uint64_t n0, float (&deq)[16]) {
  // inner scale from the block amax in normalized space (a_bits, already
  // reduced over a 16x16 block when required)
  const float a = bitsf(a_bits);
  const float v = ieee_div(a, 6.0f);
  const uint32_t sc = enc_scale(v, f);
  const float s = dec_scale(sc, f);
  const bool s_pos = fbits(s) != 0u;
  const bool S_pos = fbits(S) != 0u;
  float t[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float xp = no_outer ? u[i] : (S_pos ? ieee_div(u[i], S) : signed_zero(u[i]));
    t[i] = s_pos ? ieee_div(xp, s) : signed_zero(xp);
  }
  uint32_t q[16];
  if (sr) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint4 r = sr_words(K, step, orient, (n0 >> 2) + (uint64_t)w);
      q[4 * w + 0] = e2m1_sr(t[4 * w + 0], r.x);
      q[4 * w + 1] = e2m1_sr(t[4 * w + 1], r.y);
      q[4 * w + 2] = e2m1_sr(t[4 * w + 2], r.z);
      q[4 * w + 3] = e2m1_sr(t[4 * w + 3], r.w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const uint32_t b = e2m1x2_rne(t[i], t[i + 1]);
      q[i] = b & 0xFu;
      q[i + 1] = b >> 4;
    }
  }
  SegOut o;
  o.codes_lo = 0;
  o.codes_hi = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) o.codes_lo |= q[i] << (4 * i);
#pragma unroll
  for (int i = 0; i < 8; ++i) o.codes_hi |= q[8 + i] << (4 * i);
  o.sc = sc;
  if (WANT_DEQ) {
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      float g0, g1;
      e2m1x2_decode(q[i] | (q[i + 1] << 4), g0, g1);
      float d0 = ieee_mul(g0, s), d1 = ieee_mul(g1, s);
      if (!no_outer) { d0 = ieee_mul(d0, S); d1 = ieee_mul(d1, S); }
      deq[i] = d0;
      deq[i + 1] = d1;
    }
  }
  return o;
}

template <bool IN_BF16, bool VEC>
__device__ __forceinline__ void load_tile(TileSmem& sm, const QuantJob& j, int64_t g, int64_t m0, int64_t k0) {
  const int t = threadIdx.x;
  const uint32_t maxfin = IN_BF16 ? 0x7F7F0000u : 0x7F7FFFFFu;
  if (VEC && IN_BF16) {
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const int v = t + NTHR * p;
      const int row = v >> 3, ch = v & 7;
      const int64_t m = m0 + row, k = k0 + ch * 8;
      float f[8];
      if (m < j.M && k < j.K) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(j.x) + (g * j.M + m) * j.ld + k));
        f[0] = bf16lo(w.x); f[1] = bf16hi(w.x); f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
        f[4] = bf16lo(w.z); f[5] = bf16hi(w.z); f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
        if (j.residual) {
          const float4* rp = reinterpret_cast<const float4*>(j.residual + (g * j.M + m) * j.K + k);
          const float4 r0 = rp[0], r1 = rp[1];
          f[0] = ieee_add(f[0], r0.x); f[1] = ieee_add(f[1], r0.y); f[2] = ieee_add(f[2], r0.z); f[3] = ieee_add(f[3], r0.w);
          f[4] = ieee_add(f[4], r1.x); f[5] = ieee_add(f[5], r1.y); f[6] = ieee_add(f[6], r1.z); f[7] = ieee_add(f[7], r1.w);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = sanitize(f[i], maxfin);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = 0.0f;
      }
      float4* dst = reinterpret_cast<float4*>(&sm.u[row * LDS + ch * 8]);
      dst[0] = make_float4(f[0], f[1], f[2], f[3]);
      dst[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
  } else if (VEC) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int v = t + NTHR * p;
      const int row = v >> 4, ch = v & 15;
      const int64_t m = m0 + row, k = k0 + ch * 4;
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (m < j.M && k < j.K) {
        f = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(j.x) + (g * j.M + m) * j.ld + k));
        if (j.residual) {
          const float4 r = *reinterpret_cast<const float4*>(j.residual + (g * j.M + m) * j.K + k);
          f.x = ieee_add(f.x, r.x); f.y = ieee_add(f.y, r.y); f.z = ieee_add(f.z, r.z); f.w = ieee_add(f.w, r.w);
        }
        f.x = sanitize(f.x, maxfin); f.y = sanitize(f.y, maxfin); f.z = sanitize(f.z, maxfin); f.w = sanitize(f.w, maxfin);
      }
      *reinterpret_cast<float4*>(&sm.u[row * LDS + ch * 4]) = f;
    }
  } else {
#pragma unroll 4
    for (int p = 0; p < 16; ++p) {
      const int e = t + NTHR * p;
      const int row = e >> 6, col = e & 63;
      const int64_t m = m0 + row, k = k0 + col;
      float f = 0.0f;
      if (m < j.M && k < j.K) {
        const int64_t xi = (g * j.M + m) * j.ld + k;
        f = IN_BF16 ? bitsf((uint32_t)static_cast<const uint16_t*>(j.x)[xi] << 16) : static_cast<const float*>(j.x)[xi];
        if (j.residual) f = ieee_add(f, j.residual[(g * j.M + m) * j.K + k]);
        f = sanitize(f, maxfin);
      }
      sm.u[row * LDS + col] = f;
    }
  }
}

__device__ __forceinline__ void store_vals(void* y, int out_bf16, int64_t idx, const float (&v)[16], bool vec) {
  if (out_bf16) {
    uint16_t* p = static_cast<uint16_t*>(y) + idx;
    if (vec) {
      uint4 a, b;
      a.x = pack_bf16x2(v[0], v[1]); a.y = pack_bf16x2(v[2], v[3]); a.z = pack_bf16x2(v[4], v[5]); a.w = pack_bf16x2(v[6], v[7]);
      b.x = pack_bf16x2(v[8], v[9]); b.y = pack_bf16x2(v[10], v[11]); b.z = pack_bf16x2(v[12], v[13]); b.w = pack_bf16x2(v[14], v[15]);
      reinterpret_cast<uint4*>(p)[0] = a;
      reinterpret_cast<uint4*>(p)[1] = b;
    } else {
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const uint32_t w = pack_bf16x2(v[i], v[i + 1]);
        p[i] = (uint16_t)(w & 0xFFFFu);
        p[i + 1] = (uint16_t)(w >> 16);
      }
    }
  } else {
    float* p = static_cast<float*>(y) + idx;
    if (vec) {
#pragma unroll
      for (int i = 0; i < 16; i += 4) reinterpret_cast<float4*>(p)[i / 4] = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) p[i] = v[i];
    }
  }
}

// 2-D outer scales of the tile's ob x ob sub-tiles (ob in {16, 32, 64}).
// Thread mapping: idx = t % 64 along the lane dimension, seg = t / 64 along
// the 16-wide dimension.  lanes_are_rows selects which tile axis the lanes
// run along (rows in the rowwise pass mapping).
__device__ __forceinline__ void reduce_outer_2d(TileSmem& sm, uint32_t amax16, int ob, const ScaleFmt& f,
                                                const QuantJob& j, int64_t g, int64_t m0, int64_t k0,
                                                bool lanes_are_rows) {
  const int t = threadIdx.x;
  const int idx = t & 63, seg = t >> 6;
  const int span = ob < 32 ? ob : 32;  // lanes reduced by shuffles
  uint32_t v = amax16;
  for (int o = 1; o < span; o <<= 1) v = umax(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  if ((idx % span) == 0) sm.part[seg][idx / span] = v;
  __syncthreads();
  const int nb = TILE / ob;  // sub-tiles per tile side
  if (t < nb * nb) {
    const int lb = t / nb, sb = t % nb;  // lane-axis block, segment-axis block
    const int segs = ob / 16, parts = ob / span;
    uint32_t A = 0;
    for (int s = sb * segs; s < (sb + 1) * segs; ++s)
      for (int p = lb * parts; p < (lb + 1) * parts; ++p) A = umax(A, sm.part[s][p]);
    const float S = ieee_div(bitsf(A), f.denom);
    const int rb = lanes_are_rows ? lb : sb, cb = lanes_are_rows ? sb : lb;
    sm.S2[rb][cb] = S;
    const int64_t mi = m0 + (int64_t)rb * ob, kj = k0 + (int64_t)cb * ob;
    if (j.tile_outer && mi < j.M && kj < j.K)
      j.tile_outer[(g * (j.M / ob) + mi / ob) * (j.K / ob) + kj / ob] = S;
  }
  __syncthreads();
}

template <bool IN_BF16, bool VEC, bool SR>
__global__ void __launch_bounds__(NTHR) quant_tile_kernel(const QuantJob j) {
  __shared__ __align__(16) TileSmem sm;
  const ScaleFmt f = scale_fmt(j.ue5m3);
  const int t = threadIdx.x;
  const int idx = t & 63, seg = t >> 6;
  const int64_t tiles_m = (j.M + TILE - 1) / TILE, tiles_k = (j.K + TILE - 1) / TILE;
  const int64_t ntiles = j.G * tiles_m * tiles_k;
  const int ob = j.ob;
  const bool no_outer = j.s_src == S_ONE;
  float S_tw = 1.0f;
  if (j.s_src == S_TENSORWISE_WS) {
    S_tw = ieee_div(bitsf(*j.tw_amax), f.denom);
    if (blockIdx.x == 0 && t == 0 && j.tile_outer) j.tile_outer[0] = S_tw;
  }
  const bool two_d_in_tile = j.s_src == S_IN_TILE && j.outer_2d;
  const bool qdq_row = j.qdq_orient == 1, qdq_col = j.qdq_orient == 2;
  const bool deq_row = qdq_row || j.residual != nullptr;

  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t tk = tile % tiles_k;
    const int64_t tm = (tile / tiles_k) % tiles_m;
    const int64_t g = tile / (tiles_k * tiles_m);
    const int64_t m0 = tm * TILE, k0 = tk * TILE;
    __syncthreads();
    load_tile<IN_BF16, VEC>(sm, j, g, m0, k0);
    __syncthreads();

    if (two_d_in_tile) {
      // amax of this thread's 1x16 row segment (rows along lanes)
      const float4* src = reinterpret_cast<const float4*>(&sm.u[idx * LDS + seg * 16]);
      uint32_t am = 0;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const float4 v = src[q4];
        am = umax(am, umax(umax(abs_bits(v.x), abs_bits(v.y)), umax(abs_bits(v.z), abs_bits(v.w))));
      }
      reduce_outer_2d(sm, am, ob, f, j, g, m0, k0, true);
    }

    // ------------------------------------------------------------------ rows
    if (j.do_row) {
      const int r = idx;
      const int64_t m = m0 + r, kb = k0 + seg * 16;
      const bool valid = m < j.M && kb < j.K;
      float u[16];
      {
        const float4* src = reinterpret_cast<const float4*>(&sm.u[r * LDS + seg * 16]);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 v = src[q4];
          u[4 * q4] = v.x; u[4 * q4 + 1] = v.y; u[4 * q4 + 2] = v.z; u[4 * q4 + 3] = v.w;
        }
      }
      uint32_t am = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) am = umax(am, abs_bits(u[i]));
      float S = 1.0f;
      if (j.s_src == S_TENSORWISE_WS) {
        S = S_tw;
      } else if (j.s_src == S_FROM_BUFFER) {
        if (valid) {
          if (j.mode == 1) S = j.tile_outer[0];
          else if (j.outer_2d) S = j.tile_outer[(g * (j.M / ob) + m / ob) * (j.K / ob) + kb / ob];
          else S = j.row_outer[(g * j.M + m) * (j.K / ob) + kb / ob];
        }
      } else if (j.s_src == S_IN_TILE) {
        if (j.outer_2d) {
          S = sm.S2[r / ob][(seg * 16) / ob];
        } else {
          sm.am_row[seg][r] = am;
          __syncthreads();
          const int segs = ob / 16;
          const int s0 = (seg / segs) * segs;
          const uint32_t A = seg_group_max(sm.am_row, s0, segs, r);
          S = ieee_div(bitsf(A), f.denom);
          if (valid && seg == s0 && j.row_outer) j.row_outer[(g * j.M + m) * (j.K / ob) + kb / ob] = S;
        }
      }
      // inner amax in normalized space: max |u / S| = max|u| / S (monotone)
      uint32_t a_bits = no_outer ? am : (fbits(S) != 0u ? fbits(ieee_div(bitsf(am), S)) : 0u);
      if (j.inner_2d) {
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) a_bits = umax(a_bits, __shfl_xor_sync(0xFFFFFFFFu, a_bits, o));
      }
      float deq[16];
      const uint64_t n0 = (uint64_t)((g * j.M + m) * j.K + kb);
      SegOut o;
      if (deq_row) o = quantize_segment<true>(u, S, no_outer, a_bits, f, SR, j.srk, j.step, 0u, sr_row_n(j, (int64_t)n0), deq);
      else o = quantize_segment<false>(u, S, no_outer, a_bits, f, SR, j.srk, j.step, 0u, sr_row_n(j, (int64_t)n0), deq);
      if (valid) {
        if (j.row_codes) *reinterpret_cast<uint2*>(j.row_codes + n0 / 2) = make_uint2(o.codes_lo, o.codes_hi);
        if (j.row_scales) j.row_scales[sf_offset(j.rsl, g, m, kb / 16)] = (uint8_t)o.sc;
        if (j.residual) {
          float rr[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) rr[i] = ieee_sub(u[i], deq[i]);
          float4* rp = reinterpret_cast<float4*>(j.residual + n0);
#pragma unroll
          for (int i = 0; i < 16; i += 4) rp[i / 4] = make_float4(rr[i], rr[i + 1], rr[i + 2], rr[i + 3]);
        }
        if (qdq_row) store_vals(j.y, j.out_bf16, (int64_t)n0, deq, VEC);
      }
    }

    // --------------------------------------------------------------- columns
    if (j.do_col) {
      const int c = idx;
      const int64_t k = k0 + c, mb = m0 + seg * 16;
      const bool valid = k < j.K && mb < j.M;
      float u[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) u[i] = sm.u[(seg * 16 + i) * LDS + c];
      uint32_t am = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) am = umax(am, abs_bits(u[i]));
      float S = 1.0f;
      if (j.s_src == S_TENSORWISE_WS) {
        S = S_tw;
      } else if (j.s_src == S_FROM_BUFFER) {
        if (valid) {
          if (j.mode == 1) S = j.tile_outer[0];
          else if (j.outer_2d) S = j.tile_outer[(g * (j.M / ob) + mb / ob) * (j.K / ob) + k / ob];
          else S = j.col_outer[(g * j.K + k) * (j.M / ob) + mb / ob];
        }
      } else if (j.s_src == S_IN_TILE) {
        if (j.outer_2d) {
          S = sm.S2[(seg * 16) / ob][c / ob];
        } else {
          sm.am_col[seg][c] = am;
          __syncthreads();
          const int segs = ob / 16;
          const int s0 = (seg / segs) * segs;
          const uint32_t A = seg_group_max(sm.am_col, s0, segs, c);
          S = ieee_div(bitsf(A), f.denom);
          if (valid && seg == s0 && j.col_outer) j.col_outer[(g * j.K + k) * (j.M / ob) + mb / ob] = S;
        }
      }
      uint32_t a_bits = no_outer ? am : (fbits(S) != 0u ? fbits(ieee_div(bitsf(am), S)) : 0u);
      if (j.inner_2d) {
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) a_bits = umax(a_bits, __shfl_xor_sync(0xFFFFFFFFu, a_bits, o));
      }
      float deq[16];
      const uint64_t n0 = (uint64_t)((g * j.K + k) * j.M + mb);
      SegOut o;
      const uint64_t nsr = sr_col_n(j, g * j.K + k, mb);
      if (qdq_col) o = quantize_segment<true>(u, S, no_outer, a_bits, f, SR, j.srk, j.step, 1u, nsr, deq);
      else o = quantize_segment<false>(u, S, no_outer, a_bits, f, SR, j.srk, j.step, 1u, nsr, deq);
      if (valid) {
        if (j.col_codes) *reinterpret_cast<uint2*>(j.col_codes + n0 / 2) = make_uint2(o.codes_lo, o.codes_hi);
        if (j.col_scales) j.col_scales[sf_offset(j.csl, g, k, mb / 16)] = (uint8_t)o.sc;
      }
      if (qdq_col) {
        // transpose the dequantized segment back to x's layout through smem
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 16; ++i) sm.u[(seg * 16 + i) * LDS + c] = deq[i];
        __syncthreads();
#pragma unroll
        for (int p = 0; p < 16; ++p) {
          const int e = t + NTHR * p;
          const int row = e >> 6, col = e & 63;
          const int64_t mm = m0 + row, kk = k0 + col;
          if (mm < j.M && kk < j.K) {
            const float v = sm.u[row * LDS + col];
            const int64_t yi = (g * j.M + mm) * j.K + kk;
            if (j.out_bf16) {
              const uint32_t w = pack_bf16x2(v, 0.0f);
              static_cast<uint16_t*>(j.y)[yi] = (uint16_t)(w & 0xFFFFu);
            } else {
              static_cast<float*>(j.y)[yi] = v;
            }
          }
        }
      }
    }
  }
}

template <bool IN_BF16, bool VEC, bool SR>
cudaError_t launch_t(const QuantJob& j, cudaStream_t st) {
  const int64_t tiles = j.G * ((j.M + TILE - 1) / TILE) * ((j.K + TILE - 1) / TILE);
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quant_tile_kernel<IN_BF16, VEC, SR>, NTHR, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t cap = (int64_t)num_sms() * per_sm;
  const int grid = (int)(tiles < cap ? tiles : cap);
  quant_tile_kernel<IN_BF16, VEC, SR><<<grid, NTHR, 0, st>>>(j);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_tile(const QuantJob& j, bool vec, cudaStream_t st) {
  const bool bf = j.in_bf16 != 0, sr = j.sr != 0;
  if (bf) {
    if (vec) return sr ? launch_t<true, true, true>(j, st) : launch_t<true, true, false>(j, st);
    return sr ? launch_t<true, false, true>(j, st) : launch_t<true, false, false>(j, st);
  }
  if (vec) return sr ? launch_t<false, true, true>(j, st) : launch_t<false, true, false>(j, st);
  return sr ? launch_t<false, false, true>(j, st) : launch_t<false, false, false>(j, st);
}

}  // namespace fp4q
