// k_aux.cu -- tensorwise amax, outer-scale pre-pass and dequantize kernels.
#include "fp4q_device.cuh"
#include "fp4q_internal.h"
#include "fp4q_tma.cuh"

namespace fp4q {
namespace {

__device__ __forceinline__ uint32_t umax(uint32_t a, uint32_t b) { return a > b ? a : b; }

// |u| bits of element (g, m, k): u = sanitize(x + residual).
__device__ __forceinline__ uint32_t abs_u(const QuantJob& j, int64_t g, int64_t m, int64_t k) {
  const int64_t xi = (g * j.M + m) * j.ld + k;
  float f = j.in_bf16 ? bitsf((uint32_t)static_cast<const uint16_t*>(j.x)[xi] << 16)
                      : static_cast<const float*>(j.x)[xi];
  if (j.residual) f = ieee_add(f, j.residual[(g * j.M + m) * j.K + k]);
  f = sanitize(f, j.in_bf16 ? 0x7F7F0000u : 0x7F7FFFFFu);
  return abs_bits(f);
}

__device__ __forceinline__ uint32_t block_max(uint32_t v, uint32_t* sh) {
  for (int o = 16; o > 0; o >>= 1) v = umax(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) sh[w] = v;
  __syncthreads();
  if (w == 0) {
    v = l < (int)(blockDim.x >> 5) ? sh[l] : 0u;
    for (int o = 16; o > 0; o >>= 1) v = umax(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  }
  return v;  // valid in thread 0
}

// Tensorwise amax: grid-stride over all elements, one atomicMax per CTA.
__global__ void __launch_bounds__(256) tensor_amax_kernel(const QuantJob j, uint32_t* amax) {
  __shared__ uint32_t sh[8];
  const int64_t n = j.G * j.M * j.K;
  uint32_t v = 0;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t k = e % j.K, gm = e / j.K;
    v = umax(v, abs_u(j, gm / j.M, gm % j.M, k));
  }
  v = block_max(v, sh);
  if (threadIdx.x == 0) atomicMax(amax, v);
}

// |max| without NaN propagation (a NaN operand yields the other one); the
// sign of the result is not meaningful.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ float absmax_f32(float a, float b) {
  float r;
  asm("max.xorsign.abs.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Sanitized |u| bits from an accumulated NaN-ignoring magnitude maximum of
// raw inputs: infinity stands for the largest finite value, a NaN (every
// input NaN) for zero.  Exact because no finite input exceeds that value.
__device__ __forceinline__ uint32_t fix_abs(uint32_t a, uint32_t inf_bits, uint32_t max_bits) {
  return a > inf_bits ? 0u : (a == inf_bits ? max_bits : a);
}

// Vector body of the contiguous tensorwise amax: one 16-byte unit of x (8
// bf16 or 4 binary32 values), plus its residual, folded into the running
// maxima.  Without a residual, `acc` is a packed NaN-ignoring maximum
// (bf16x2 bits, or binary32 bits); with one, sanitized |u| bits.
template <bool IN_BF16, bool RES>
__device__ __forceinline__ void amax_unit(const uint4 w, const float* res, uint32_t& acc) {
  if (!RES) {
    if (IN_BF16) {
      acc = absmax_bf16x2(acc, absmax_bf16x2(absmax_bf16x2(w.x, w.y), absmax_bf16x2(w.z, w.w)));
    } else {
      acc = fbits(absmax_f32(bitsf(acc), absmax_f32(absmax_f32(bitsf(w.x), bitsf(w.y)),
                                                     absmax_f32(bitsf(w.z), bitsf(w.w)))));
    }
    return;
  }
  constexpr int EPV = IN_BF16 ? 8 : 4;
  const uint32_t mx = IN_BF16 ? 0x7F7F0000u : 0x7F7FFFFFu;
  float u[EPV];
  if (IN_BF16) {
    u[0] = bf16lo(w.x); u[1] = bf16hi(w.x); u[2] = bf16lo(w.y); u[3] = bf16hi(w.y);
    u[4] = bf16lo(w.z); u[5] = bf16hi(w.z); u[6] = bf16lo(w.w); u[7] = bf16hi(w.w);
  } else {
    u[0] = bitsf(w.x); u[1] = bitsf(w.y); u[2] = bitsf(w.z); u[3] = bitsf(w.w);
  }
#pragma unroll
  for (int q = 0; q < EPV / 4; ++q) {
    const float4 r = reinterpret_cast<const float4*>(res)[q];
    u[4 * q] = ieee_add(u[4 * q], r.x); u[4 * q + 1] = ieee_add(u[4 * q + 1], r.y);
    u[4 * q + 2] = ieee_add(u[4 * q + 2], r.z); u[4 * q + 3] = ieee_add(u[4 * q + 3], r.w);
  }
#pragma unroll
  for (int i = 0; i < EPV; ++i) acc = umax(acc, abs_bits(sanitize(u[i], mx)));
}

// Tensorwise amax of a contiguous tensor (leading dimension K, 16-byte
// aligned x and residual): each warp streams 2 KB contiguous chunks (four
// 512-byte loads in flight), a scalar tail, one atomicMax per CTA.  (Four
// strided streams per thread, or more loads in flight, read slower.)
template <bool IN_BF16, bool RES>
__global__ void __launch_bounds__(256) tensor_amax_flat_kernel(const QuantJob j, uint32_t* amax) {
  pdl_wait_then_release();
  __shared__ uint32_t sh[8];
  constexpr int EPV = IN_BF16 ? 8 : 4;
  const int64_t n = j.G * j.M * j.K;
  const int64_t nv = n / EPV;
  const uint4* xv = static_cast<const uint4*>(j.x);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  // each warp reads 2 KB contiguous per iteration (four 512-byte loads)
  const int64_t wstride = stride * 4;
  int64_t i = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 128 + (threadIdx.x & 31);
  uint32_t acc = 0;
  for (; i + 96 < nv; i += wstride) {
    uint4 w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = __ldcs(xv + i + q * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q) amax_unit<IN_BF16, RES>(w[q], RES ? j.residual + (i + q * 32) * EPV : nullptr, acc);
  }
  for (; i < nv; i += 32) amax_unit<IN_BF16, RES>(__ldcs(xv + i), RES ? j.residual + i * EPV : nullptr, acc);
  uint32_t v;
  if (RES) {
    v = acc;
  } else if (IN_BF16) {
    v = umax(fix_abs(acc & 0x7FFFu, 0x7F80u, 0x7F7Fu), fix_abs((acc >> 16) & 0x7FFFu, 0x7F80u, 0x7F7Fu)) << 16;
  } else {
    v = fix_abs(acc & 0x7FFFFFFFu, 0x7F800000u, 0x7F7FFFFFu);
  }
  const int64_t e = nv * EPV + (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // scalar tail
  if (e < n) v = umax(v, abs_u(j, 0, 0, e));
  v = block_max(v, sh);
  if (threadIdx.x == 0) atomicMax(amax, v);
}

// Grouped path, one CTA: checks the offsets (0 = goff[0] <= ... <=
// goff[n] = M, every group a multiple of `align` rows), writes the prefix of
// 128-row tiles per group and the total, and clears the per-group amax.
__global__ void __launch_bounds__(1024) group_prep_kernel(const QuantJob j, int align) {
  __shared__ uint32_t part[1024];
  GroupWs* w = j.gws;
  const int64_t n = j.ngroups;
  uint32_t* tp = group_tprefix(w);
  uint32_t* am = group_amax(w, n);
  const int t = threadIdx.x;
  if (t == 0) w->bad = 0u;
  __syncthreads();
  const int64_t chunk = (n + 1023) / 1024;
  const int64_t e0 = t * chunk, e1 = e0 + chunk < n ? e0 + chunk : n;
  uint32_t bad = 0, sum = 0;
  if (t == 0 && (j.goff[0] != 0 || j.goff[n] != j.M)) bad = 1;
  for (int64_t e = e0; e < e1; ++e) {
    const int64_t a = j.goff[e], b = j.goff[e + 1];
    if (b < a || (b - a) % align) bad = 1;
    else sum += (uint32_t)((b - a + 127) / 128);
    am[e] = 0u;
    if (j.mode == 1 && j.tile_outer && b == a) j.tile_outer[e] = 0.0f;  // an empty group's tensorwise scale
  }
  if (bad) atomicOr(&w->bad, 1u);
  part[t] = sum;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {  // inclusive scan of the chunk sums
    const uint32_t v = t >= o ? part[t - o] : 0u;
    __syncthreads();
    part[t] += v;
    __syncthreads();
  }
  uint32_t run = t ? part[t - 1] : 0u;
  for (int64_t e = e0; e < e1; ++e) {
    tp[e] = run;
    const int64_t a = j.goff[e], b = j.goff[e + 1];
    if (b >= a) run += (uint32_t)((b - a + 127) / 128);
  }
  if (t == 1023) {
    tp[n] = part[1023];
    w->mtiles = part[1023];
  }
}

// Per-group tensorwise amax of a bf16 [M, K] input (row stride ld, 16-byte
// aligned rows): blockIdx.y = group, CTAs along x stride over its rows.
__global__ void __launch_bounds__(256) group_amax_kernel(const QuantJob j) {
  __shared__ uint32_t sh[8];
  GroupWs* w = j.gws;
  if (w->bad) return;
  const int64_t e = blockIdx.y;
  const int64_t r0 = j.goff[e], r1 = j.goff[e + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t units = j.K / 8;
  uint32_t acc = 0;
  for (int64_t r = r0 + (int64_t)blockIdx.x * 8 + warp; r < r1; r += (int64_t)gridDim.x * 8) {
    const uint4* row = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(j.x) + r * j.ld);
    for (int64_t u = lane; u < units; u += 32) amax_unit<true, false>(__ldcs(row + u), nullptr, acc);
  }
  uint32_t v = umax(fix_abs(acc & 0x7FFFu, 0x7F80u, 0x7F7Fu), fix_abs((acc >> 16) & 0x7FFFu, 0x7F80u, 0x7F7Fu)) << 16;
  v = block_max(v, sh);
  if (threadIdx.x == 0 && v) atomicMax(&group_amax(w, j.ngroups)[e], v);
}

// 1-D rowwise outer scales (ob along K): one warp per outer block.
__global__ void __launch_bounds__(256) outer_row_kernel(const QuantJob j) {
  const ScaleFmt f = scale_fmt(j.ue5m3);
  const int64_t nb_k = j.K / j.ob;
  const int64_t nblk = j.G * j.M * nb_k;
  const int lane = threadIdx.x & 31;
  for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < nblk;
       b += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int64_t jb = b % nb_k, gm = b / nb_k;
    uint32_t v = 0;
    for (int64_t k = jb * j.ob + lane; k < (jb + 1) * j.ob; k += 32) v = umax(v, abs_u(j, gm / j.M, gm % j.M, k));
    for (int o = 16; o > 0; o >>= 1) v = umax(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    if (lane == 0) j.row_outer[b] = ieee_div(bitsf(v), f.denom);
  }
}

// 1-D columnwise outer scales (ob along M): one thread per (g, block, k).
__global__ void __launch_bounds__(256) outer_col_kernel(const QuantJob j) {
  const ScaleFmt f = scale_fmt(j.ue5m3);
  const int64_t nb_m = j.M / j.ob;
  const int64_t n = j.G * nb_m * j.K;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t k = e % j.K, ib = (e / j.K) % nb_m, g = e / (j.K * nb_m);
    uint32_t v = 0;
    for (int64_t m = ib * j.ob; m < (ib + 1) * j.ob; ++m) v = umax(v, abs_u(j, g, m, k));
    j.col_outer[(g * j.K + k) * nb_m + ib] = ieee_div(bitsf(v), f.denom);
  }
}

// 2-D outer scales (ob x ob): one CTA per block.
__global__ void __launch_bounds__(256) outer_2d_kernel(const QuantJob j) {
  __shared__ uint32_t sh[8];
  const ScaleFmt f = scale_fmt(j.ue5m3);
  const int64_t nb_m = j.M / j.ob, nb_k = j.K / j.ob;
  const int64_t nblk = j.G * nb_m * nb_k;
  const int64_t ob2 = (int64_t)j.ob * j.ob;
  for (int64_t b = blockIdx.x; b < nblk; b += gridDim.x) {
    const int64_t jb = b % nb_k, ib = (b / nb_k) % nb_m, g = b / (nb_k * nb_m);
    uint32_t v = 0;
    for (int64_t e = threadIdx.x; e < ob2; e += blockDim.x)
      v = umax(v, abs_u(j, g, ib * j.ob + e / j.ob, jb * j.ob + e % j.ob));
    v = block_max(v, sh);
    if (threadIdx.x == 0) j.tile_outer[b] = ieee_div(bitsf(v), f.denom);
    __syncthreads();
  }
}

// Dequantize, linear scales without 2-D outer blocks: every index is a
// function of the flat block index b (codes at 8 b, scale at b, a 1 x ob
// outer scale at 16 b / ob), so there is no division.  One thread per
// microblock, DQ_IN_FLIGHT in flight per thread; OUTER: 0 none, 1 one scale, 2 1-D.
// W32: y is 32-byte aligned and each microblock's output leaves in 256-bit
// stores, so a warp's store instruction fills whole 32-byte sectors (two
// 16-byte stores a lane 32 bytes apart each fill half of every sector, and
// the sectors went to L2 twice).
constexpr int DQ_IN_FLIGHT = 4;  // microblocks per thread in flight (8 measured slower)
template <bool OUT_BF16, int OUTER, bool W32>
__global__ void __launch_bounds__(256) dequant_flat_kernel(const DequantJob j) {
  pdl_wait_then_release();
  const ScaleFmt f = scale_fmt(j.ue5m3);
  const int64_t nmb = j.G * j.R * (j.C / 16);
  const int lob = j.ob > 0 ? 31 - __clz(j.ob) : 0;
  const bool pow2 = j.ob > 0 && (j.ob & (j.ob - 1)) == 0;
  const float S1 = OUTER == 1 ? j.outer[0] : 1.0f;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t b0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b0 < nmb; b0 += DQ_IN_FLIGHT * stride) {
    uint2 cw[DQ_IN_FLIGHT];
    uint32_t sb[DQ_IN_FLIGHT];
    float S[DQ_IN_FLIGHT];
#pragma unroll
    for (int q = 0; q < DQ_IN_FLIGHT; ++q) S[q] = S1;
#pragma unroll
    for (int q = 0; q < DQ_IN_FLIGHT; ++q) {
      const int64_t b = b0 + q * stride;
      if (b < nmb) {
        cw[q] = __ldcs(reinterpret_cast<const uint2*>(j.codes) + b);
        sb[q] = j.scales[b];
        if (OUTER == 2) S[q] = j.outer[pow2 ? (b * 16) >> lob : (b * 16) / j.ob];
      }
    }
#pragma unroll
    for (int q = 0; q < DQ_IN_FLIGHT; ++q) {
      const int64_t b = b0 + q * stride;
      if (b >= nmb) continue;
      const float s = dec_scale(sb[q], f);
      uint32_t w[8];
      float v[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t byte = ((i < 4 ? cw[q].x : cw[q].y) >> (8 * (i & 3))) & 0xFFu;
        float g0, g1;
        e2m1x2_decode(byte, g0, g1);
        float d0 = ieee_mul(g0, s), d1 = ieee_mul(g1, s);
        if (OUTER) { d0 = ieee_mul(d0, S[q]); d1 = ieee_mul(d1, S[q]); }
        v[2 * i] = d0;
        v[2 * i + 1] = d1;
        w[i] = pack_bf16x2(d0, d1);
      }
      if (OUT_BF16 && W32) {
        st256(static_cast<uint16_t*>(j.y) + b * 16, w);
      } else if (OUT_BF16) {
        uint4* p = reinterpret_cast<uint4*>(static_cast<uint16_t*>(j.y) + b * 16);
        __stcs(p, make_uint4(w[0], w[1], w[2], w[3]));
        __stcs(p + 1, make_uint4(w[4], w[5], w[6], w[7]));
      } else if (W32) {
        float* p = static_cast<float*>(j.y) + b * 16;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t u[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) u[i] = fbits(v[8 * h + i]);
          st256(p + 8 * h, u);
        }
      } else {
        float4* p = reinterpret_cast<float4*>(static_cast<float*>(j.y) + b * 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) __stcs(p + i, make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
      }
    }
  }
}

// Dequantize: one thread per 1 x 16 microblock.
template <bool OUT_BF16>
__global__ void __launch_bounds__(256) dequant_kernel(const DequantJob j, int vec_out) {
  const ScaleFmt f = scale_fmt(j.ue5m3);
  const int64_t nmb = j.G * j.R * (j.C / 16);
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nmb; b += (int64_t)gridDim.x * blockDim.x) {
    const int64_t cb = b % (j.C / 16), gr = b / (j.C / 16);
    const int64_t r = gr % j.R, g = gr / j.R;
    const int64_t c0 = cb * 16;
    float S = 1.0f;
    const bool outer = j.mode != 0;
    if (j.mode == 1) {
      S = j.outer[0];
    } else if (j.mode == 2) {
      if (!j.outer_2d) {
        S = j.outer[(g * j.R + r) * (j.C / j.ob) + c0 / j.ob];
      } else {
        const int64_t mi = j.col ? c0 : r, kj = j.col ? r : c0;  // element's (m, k) in x
        S = j.outer[(g * (j.M / j.ob) + mi / j.ob) * (j.K / j.ob) + kj / j.ob];
      }
    }
    const float s = dec_scale(j.scales[sf_from_linear(j.sl, b)], f);
    const uint2 cw = *reinterpret_cast<const uint2*>(j.codes + b * 8);
    float v[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t byte = ((i < 4 ? cw.x : cw.y) >> (8 * (i & 3))) & 0xFFu;
      float g0, g1;
      e2m1x2_decode(byte, g0, g1);
      float d0 = ieee_mul(g0, s), d1 = ieee_mul(g1, s);
      if (outer) { d0 = ieee_mul(d0, S); d1 = ieee_mul(d1, S); }
      v[2 * i] = d0;
      v[2 * i + 1] = d1;
    }
    const int64_t yi = b * 16;
    if (OUT_BF16) {
      uint16_t* p = static_cast<uint16_t*>(j.y) + yi;
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
      if (vec_out) {
        reinterpret_cast<uint4*>(p)[0] = make_uint4(w[0], w[1], w[2], w[3]);
        reinterpret_cast<uint4*>(p)[1] = make_uint4(w[4], w[5], w[6], w[7]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) { p[2 * i] = (uint16_t)(w[i] & 0xFFFFu); p[2 * i + 1] = (uint16_t)(w[i] >> 16); }
      }
    } else {
      float* p = static_cast<float*>(j.y) + yi;
      if (vec_out) {
#pragma unroll
        for (int i = 0; i < 16; i += 4) reinterpret_cast<float4*>(p)[i / 4] = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) p[i] = v[i];
      }
    }
  }
}

int grid_for(int64_t work_items, int threads, int per_sm) {
  const int64_t need = (work_items + threads - 1) / threads;
  const int64_t cap = (int64_t)num_sms() * per_sm;
  int64_t g = need < cap ? need : cap;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_tensor_amax(const QuantJob& j, uint32_t* amax_ws, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(amax_ws, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  const int64_t n = j.G * j.M * j.K;
  const bool flat = (j.ld == j.K || j.M * j.G == 1) && vec_aligned(j.x, 0) &&
                    (!j.residual || vec_aligned(j.residual, 0));
  if (flat) {
    const int grid = grid_for(n / (j.in_bf16 ? 8 : 4) / 4 + 1, 256, 4);
    auto kern = j.in_bf16 ? (j.residual ? tensor_amax_flat_kernel<true, true> : tensor_amax_flat_kernel<true, false>)
                          : (j.residual ? tensor_amax_flat_kernel<false, true> : tensor_amax_flat_kernel<false, false>);
    return launch_pdl(kern, dim3((unsigned)grid), dim3(256), 0, st, j, amax_ws);
  }
  tensor_amax_kernel<<<grid_for(n, 256, 8), 256, 0, st>>>(j, amax_ws);
  return cudaGetLastError();
}

cudaError_t launch_group_prep(const QuantJob& j, int align, bool amax, cudaStream_t st) {
  group_prep_kernel<<<1, 1024, 0, st>>>(j, align);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (amax) {
    const int64_t per = (int64_t)num_sms() * 8 / (j.ngroups > 0 ? j.ngroups : 1);
    const dim3 grid((unsigned)(per < 1 ? 1 : (per > 64 ? 64 : per)), (unsigned)j.ngroups);
    group_amax_kernel<<<grid, 256, 0, st>>>(j);
    e = cudaGetLastError();
  }
  return e;
}

cudaError_t launch_outer_prepass(const QuantJob& j, cudaStream_t st) {
  if (j.outer_2d) {
    const int64_t nblk = j.G * (j.M / j.ob) * (j.K / j.ob);
    const int64_t cap = (int64_t)num_sms() * 8;
    outer_2d_kernel<<<(int)(nblk < cap ? nblk : cap), 256, 0, st>>>(j);
    return cudaGetLastError();
  }
  if (j.do_row) {
    outer_row_kernel<<<grid_for(j.G * j.M * (j.K / j.ob) * 32, 256, 8), 256, 0, st>>>(j);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (j.do_col) {
    outer_col_kernel<<<grid_for(j.G * (j.M / j.ob) * j.K, 256, 8), 256, 0, st>>>(j);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_dequant(const DequantJob& j, cudaStream_t st) {
  const int64_t nmb = j.G * j.R * (j.C / 16);
  const int vec = vec_aligned(j.y, 16);
  if (vec && !j.sl.mma && !(j.mode == 2 && j.outer_2d) && (reinterpret_cast<uintptr_t>(j.codes) & 7u) == 0) {
    const int grid = grid_for((nmb + DQ_IN_FLIGHT - 1) / DQ_IN_FLIGHT, 256, 8);
    const bool w32 = (reinterpret_cast<uintptr_t>(j.y) & 31u) == 0;
    void (*kern)(const DequantJob) =
        w32 ? (j.out_bf16 ? (j.mode == 0   ? dequant_flat_kernel<true, 0, true>
                             : j.mode == 1 ? dequant_flat_kernel<true, 1, true>
                                           : dequant_flat_kernel<true, 2, true>)
                          : (j.mode == 0   ? dequant_flat_kernel<false, 0, true>
                             : j.mode == 1 ? dequant_flat_kernel<false, 1, true>
                                           : dequant_flat_kernel<false, 2, true>))
            : (j.out_bf16 ? (j.mode == 0   ? dequant_flat_kernel<true, 0, false>
                             : j.mode == 1 ? dequant_flat_kernel<true, 1, false>
                                           : dequant_flat_kernel<true, 2, false>)
                          : (j.mode == 0   ? dequant_flat_kernel<false, 0, false>
                             : j.mode == 1 ? dequant_flat_kernel<false, 1, false>
                                           : dequant_flat_kernel<false, 2, false>));
    return launch_pdl(kern, dim3((unsigned)grid), dim3(256), 0, st, j);
  }
  const int grid = grid_for(nmb, 256, 8);
  if (j.out_bf16) dequant_kernel<true><<<grid, 256, 0, st>>>(j, vec);
  else dequant_kernel<false><<<grid, 256, 0, st>>>(j, vec);
  return cudaGetLastError();
}

}  // namespace fp4q
