// k_mxfp8.cu -- fused MXFP4 projection + MXFP8 re-encode ("MXFP4 weight QAT
// recipes on MXFP8 and FP8 block-scaling hosts", "Design": the projected
// weight goes to the host's MXFP8 quantizer, rowwise losslessly and
// columnwise (32 x 1) with bounded re-quantization; "Known limitations": a
// fused projection + quantize kernel is named as future work).
//
// MXFP8 follows the OCP Microscaling v1.0 rule: per block of 32 values a
// scale 2^X, X = floor(log2 amax) - 8 clamped to [-127, 127] (byte X + 127),
// elements E4M3(v / 2^X) with RNE and saturation; a block of zeros takes
// X = -127, a block holding a NaN (a poisoned MXFP4 block) is scale 0xFF
// with elements 0x7F.
//
// One CTA of 256 threads per 128 x 64 tile of x, read once:
//   rowwise: thread t owns the 1 x 32 block (row t / 2, columns 32 (t mod 2)
//     ..): MXFP4 projection (exponent from the integer bits of the block
//     maximum), the optional projected output, and the rowwise MXFP8 block.
//     Its scale needs no search: the projected maximum is
//     e2m1(q_max) 2^E, so X = E + floor(log2 e2m1(q_max)) - 8, and every
//     element y / 2^X = e2m1(q) 2^(E - X) is exact in E4M3.
//   the projected values are staged in shared memory as bf16 (exact: two
//     significant bits, exponents within bf16's range);
//   columnwise: a lane owns half (16 rows) of two 32 x 1 MXFP8 blocks of
//     adjacent columns, read from the staged tile as bf16 pairs; the block
//     maxima meet with one shuffle.
#include "fp4q_device.cuh"
#include "fp4q_internal.h"
#include "fp4q_tma.cuh"

namespace fp4q {
namespace {

constexpr int XT = 256;
constexpr int XM = 128, XK = 64;
// staged row stride in bytes; 16-byte unit u of row r sits at unit
// u ^ swz(r), swz(r) = (r mod 8) ^ 4 ((r / 16) mod 2): the rowwise stores of
// four consecutive rows and the columnwise loads of rows r and r + 16 both
// spread over all banks
constexpr int YS = XK * 2;
__device__ __forceinline__ int ys_swz(int r) { return (r & 7) ^ (((r >> 4) & 1) << 2); }

// MXFP4 block exponent (see k_mxfp4.cu): least E with 6 * 2^E >= max(A, 6 * 2^-126), capped at 125.
__device__ __forceinline__ int mx_exp(uint32_t amax_bits) {
  const uint32_t ac = amax_bits > 0x01C00000u ? amax_bits : 0x01C00000u;
  const int k = (int)(ac >> 23) - 127;
  const int e = (ac & 0x7FFFFFu) <= 0x400000u ? k - 2 : k - 1;
  return e < 125 ? e : 125;
}

// Two E4M3 bytes (RNE, satfinite): `lo` in bits 0-7, `hi` in bits 8-15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\tcvt.u32.u16 %0, t;\n\t}" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float pow2f(int e) { return bitsf((uint32_t)(e + 127) << 23); }  // -126 <= e <= 127

// Codes of a byte of two E2M1 values as binary16 pairs (exact), low nibble
// in the low half.
__device__ __forceinline__ uint32_t e2m1x2_f16x2(uint32_t byte) {
  uint32_t h;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h) : "r"(byte));
  return h;
}

// E4M3 bytes of a binary16 pair times 2^d (1 <= d <= 9: the products are
// exact in binary16 and in E4M3), low half in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_f16x2_scaled(uint32_t h, uint32_t p2) {
  uint32_t r;
  asm("{\n\t.reg .b32 m;\n\t.reg .b16 t;\n\tmul.rn.f16x2 m, %1, %2;\n\t"
      "cvt.rn.satfinite.e4m3x2.f16x2 t, m;\n\tcvt.u32.u16 %0, t;\n\t}"
      : "=r"(r) : "r"(h), "r"(p2));
  return r;
}

template <bool IN_BF16>
__device__ __forceinline__ void load_block32(const void* x, int64_t idx, float (&v)[32], uint32_t& amax) {
  // 32 elements from element index idx (16-byte aligned)
  if (IN_BF16) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + idx);
    uint32_t m = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = __ldcs(p + q);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[8 * q + 2 * i] = bf16lo(ww[i]);
        v[8 * q + 2 * i + 1] = bf16hi(ww[i]);
        m = q == 0 && i == 0 ? ww[i] : bf16x2_amax(m, ww[i]);
      }
    }
    m &= 0x7FFF7FFFu;
    const uint32_t hi = m >> 16, lo = m & 0xFFFFu;
    amax = (hi > lo ? hi : lo) << 16;
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(x) + idx);
    float m = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 w = __ldcs(p + q);
      v[4 * q] = w.x; v[4 * q + 1] = w.y; v[4 * q + 2] = w.z; v[4 * q + 3] = w.w;
      m = f32_amax(f32_amax(m, w.x), f32_amax(f32_amax(w.y, w.z), w.w));
    }
    amax = fbits(m) & 0x7FFFFFFFu;
  }
}

// Rowwise part of one 1 x 32 block (row m, columns k ..): projection, the
// optional projected output, the rowwise MXFP8 block and the bf16 staging of
// the projection for the columnwise part.  v: the block's values, amax:
// max |v| bits (inf / NaN: a poisoned block).
template <bool OUT_BF16>
__device__ __forceinline__ void row_work(const QuantJob& j, const float (&v)[32], uint32_t amax, int64_t g, int64_t m,
                                         int64_t k, int rr, int rh, unsigned char* ys) {
  const int64_t M = j.M, K = j.K;
  const bool poison = amax >= 0x7F800000u;
  const int E = mx_exp(amax);
  const float inv = pow2f(-E), sc = E >= -126 ? pow2f(E) : 0.0f;
  uint32_t qb[16];  // E2M1 code bytes
  const uint64_t INV2 = pk2(inv, inv);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float a, b;
    upk2(mul2(pk2(v[2 * i], v[2 * i + 1]), INV2), a, b);  // v 2^-E, two per instruction
    qb[i] = e2m1x2_rne(a, b);
  }
  // the largest code magnitude is the code of the block maximum (the
  // rounding is monotone); for a poisoned block it is not used
  const uint32_t qmax = e2m1x2_rne(ieee_mul(bitsf(amax), inv), 0.0f) & 7u;
  // projected values y = e2m1(q) 2^E (exact), recomputed from the codes
  // for each output so that no 32-value array stays live
  const int64_t n = (g * M + m) * K + k;  // element index of the block in the [G, M, K] outputs
  // a lane's 64 bytes of projection and 32 of rowwise codes leave in 256-bit
  // stores (whole 32-byte sectors) when both outputs are 32-byte aligned
  const bool w32 = ((reinterpret_cast<uintptr_t>(j.y) | reinterpret_cast<uintptr_t>(j.row_codes)) & 31u) == 0;
  if (j.y || j.col_codes) {
    const uint64_t SC2 = pk2(sc, sc);
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
      uint32_t w[8];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int q = 2 * qq + h;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float g0, g1;
          e2m1x2_decode(qb[4 * q + i], g0, g1);
          upk2(mul2(pk2(g0, g1), SC2), g0, g1);
          w[4 * h + i] = poison ? 0x7FC07FC0u : pack_bf16x2(g0, g1);
        }
        if (j.col_codes)  // staged as bf16 (exact; NaN for a poisoned block)
          *reinterpret_cast<uint4*>(ys + rr * YS + (((4 * rh + q) ^ ys_swz(rr)) << 4)) =
              make_uint4(w[4 * h], w[4 * h + 1], w[4 * h + 2], w[4 * h + 3]);
      }
      if (j.y && OUT_BF16) {
        uint16_t* d = static_cast<uint16_t*>(j.y) + n + 16 * qq;
        if (w32) {
          st256(d, w);
        } else {
          reinterpret_cast<uint4*>(d)[0] = make_uint4(w[0], w[1], w[2], w[3]);
          reinterpret_cast<uint4*>(d)[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    }
    if (j.y && !OUT_BF16) {
      float4* d = reinterpret_cast<float4*>(static_cast<float*>(j.y) + n);
      const float qn = bitsf(0x7FC00000u);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float g[4];
        e2m1x2_decode(qb[2 * q], g[0], g[1]);
        e2m1x2_decode(qb[2 * q + 1], g[2], g[3]);
        d[q] = poison ? make_float4(qn, qn, qn, qn)
                      : make_float4(ieee_mul(g[0], sc), ieee_mul(g[1], sc), ieee_mul(g[2], sc), ieee_mul(g[3], sc));
      }
    }
  }
  if (j.row_codes) {
    // X = E + floor(log2 e2m1(qmax)) - 8 (qmax: 0 -> zeros; 1 -> 0.5; 2,3 -> 1, 1.5; 4,5 -> 2, 3; 6,7 -> 4, 6)
    const int fl = qmax <= 1u ? -1 : (int)(qmax >> 1) - 1;
    int X = qmax == 0u ? -127 : E + fl - 8;
    X = X < -127 ? -127 : X;
    // 2^(E - X) in [2^1, 2^9] as a binary16 pair; e2m1(q) 2^(E - X) is exact
    // in binary16 and in E4M3
    const uint32_t p2 = (uint32_t)(E - X + 15) << 10, P2 = p2 | (p2 << 16);
    uint32_t cw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      cw[i] = e4m3x2_f16x2_scaled(e2m1x2_f16x2(qb[2 * i]), P2) |
              (e4m3x2_f16x2_scaled(e2m1x2_f16x2(qb[2 * i + 1]), P2) << 16);
      if (poison) cw[i] = 0x7F7F7F7Fu;
    }
    if (w32) {
      st256(j.row_codes + n, cw);
    } else {
      uint4* d = reinterpret_cast<uint4*>(j.row_codes + n);
      d[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      d[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
    }
    j.row_scales[n / 32] = poison ? (uint8_t)0xFF : (uint8_t)(X + 127);
  }
}

// Columnwise part of a 128 x 64 tile from the staged projection.
__device__ __forceinline__ void col_work(const QuantJob& j, const unsigned char* ys, int64_t g, int64_t m0, int64_t k0,
                                         int t) {
  const int64_t M = j.M, K = j.K;
  // ---- columnwise (M % 32 == 0): warp w takes the 32-row block w / 2 and
  // column half w mod 2; lane l the column pair 16 (w mod 2) + (l mod 16)
  // and rows 16 (l / 16) .. + 15 of the block, read as bf16 pairs (the two
  // row halves of a 64-byte run sit 64 bytes apart through the swizzle, so
  // a warp's loads do not conflict); the partner lane l ^ 16 holds the other
  // half of both blocks.
  const int lane = t & 31, warp = t >> 5;
  const int rb = warp >> 1, half = lane >> 4;
  const int col0 = 2 * (16 * (warp & 1) + (lane & 15));
  const int64_t k = k0 + col0, mb = m0 + 32 * rb;
  const bool valid = k < K && mb < M;  // K % 32 == 0: both columns or neither
  uint32_t wv[16];
  {
    // row 32 rb + 16 half + i: swz = (i mod 8) ^ 4 half
    const unsigned char* base = ys + (32 * rb + 16 * half) * YS + (col0 & 7) * 2;
    const int cu = (col0 >> 3) ^ (half << 2);
#pragma unroll
    for (int i = 0; i < 16; ++i) wv[i] = *reinterpret_cast<const uint32_t*>(base + i * YS + ((cu ^ (i & 7)) << 4));
  }
  uint32_t mx = bf16x2_amax(wv[0], wv[1]);
#pragma unroll
  for (int i = 2; i < 16; i += 2) mx = bf16x2_amax(mx, bf16x2_amax(wv[i], wv[i + 1]));
  mx = bf16x2_amax(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
  if (!valid) return;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint32_t a = (mx >> (16 * c)) & 0x7FFFu;  // |max| of the column's 32 values (NaN propagates)
    const bool nan = a > 0x7F80u;
    // X = floor(log2 amax) - 8 from the exponent bits (subnormal / zero amax: -127)
    const int ex = (int)(a >> 7);
    int X = ex == 0 ? -127 : ex - 127 - 8;
    X = X < -127 ? -127 : X;
    const float inv = pow2f(-X);
    const uint64_t INV2 = pk2(inv, inv);
    uint32_t cw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = c ? bf16hi(wv[4 * i + e]) : bf16lo(wv[4 * i + e]);
      upk2(mul2(pk2(v[0], v[1]), INV2), v[0], v[1]);  // v 2^-X, two per instruction
      upk2(mul2(pk2(v[2], v[3]), INV2), v[2], v[3]);
      cw[i] = e4m3x2(v[0], v[1]) | (e4m3x2(v[2], v[3]) << 16);
      if (nan) cw[i] = 0x7F7F7F7Fu;
    }
    const int64_t n = (g * K + k + c) * M + mb;  // block start in the [G, K, M] columnwise outputs
    *reinterpret_cast<uint4*>(j.col_codes + n + 16 * half) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    if (half == 0) j.col_scales[n / 32] = nan ? (uint8_t)0xFF : (uint8_t)(X + 127);
  }
}

template <bool IN_BF16, bool OUT_BF16>
__global__ void __launch_bounds__(XT, 4) mxfp8_kernel(const QuantJob j, int64_t tiles_m, int64_t tiles_k) {
  pdl_wait_then_release();
  __shared__ __align__(16) unsigned char ys[XM * YS];  // projected tile, bf16
  const int t = threadIdx.x;
  const int64_t tile = blockIdx.x;
  const int64_t tk = tile % tiles_k, tm = (tile / tiles_k) % tiles_m, g = tile / (tiles_k * tiles_m);
  const int64_t m0 = tm * XM, k0 = tk * XK;
  {
    const int rr = t >> 1, rh = t & 1;
    const int64_t m = m0 + rr, k = k0 + 32 * rh;
    if (m < j.M && k < j.K) {
      float v[32];
      uint32_t amax;
      load_block32<IN_BF16>(j.x, (g * j.M + m) * j.ld + k, v, amax);
      row_work<OUT_BF16>(j, v, amax, g, m, k, rr, rh, ys);
    }
  }
  if (!j.col_codes) return;
  __syncthreads();
  col_work(j, ys, g, m0, k0, t);
}

// ---- persistent form for bf16 input: 128 x 64 tiles copied by the tensor
// memory accelerator into two slots (128-byte swizzle), a CTA walking the
// tiles grid-stride, so the next tile is in flight while this one is
// processed.  Per tile: the rowwise pass reads its 1 x 32 block from the
// slot and stages the projection; a barrier frees the slot (refilled with
// the tile after next) and publishes the staging; the columnwise pass; a
// second barrier frees the staging.
constexpr int XLRAW = XM * XK * 2;
struct XL {
  __host__ __device__ static constexpr int raw(int s) { return s * XLRAW; }  // 2 slots
  static constexpr int ys = 2 * XLRAW;                                      // projected tile, bf16
  static constexpr int bars = ys + XM * YS;                                 // 2 mbarriers
  static constexpr int total = bars + 16 + 1024;                            // + alignment slack
};

// Set by a tile wait that ran out; read and cleared by fp4q_device_status.
__device__ unsigned int g_mx8_timeout = 0;

__device__ __forceinline__ void mx8_issue(const CUtensorMap* map, const TilePos& p, unsigned char* raw, uint64_t* bar) {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_tx(bar, (uint32_t)XLRAW);
  tma_load3(raw, map, (int)p.k0, (int)p.m0, (int)p.g, bar);
}

template <bool OUT_BF16>
__global__ void __launch_bounds__(XT, 4) mxfp8_tma_kernel(const QuantJob j, const __grid_constant__ CUtensorMap tmap) {
  pdl_wait_then_release();
  extern __shared__ __align__(16) unsigned char smem_dyn[];
  unsigned char* smem = smem_align1024(smem_dyn);
  const int t = threadIdx.x;
  unsigned char* ys = smem + XL::ys;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + XL::bars);
  TileIter cur;
  cur.init<XM>(j);
  if (t == 0) {
    mbar_init(&bars[0]);
    mbar_init(&bars[1]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (t == 0) {  // the first two tiles; later tiles take a slot once its reads are past a barrier
    if (cur.valid()) mx8_issue(&tmap, cur.pos<XM>(), smem + XL::raw(0), &bars[0]);
    if (cur.idx + (int)gridDim.x < cur.ntiles)
      mx8_issue(&tmap, cur.pos_of<XM>(cur.idx + (int)gridDim.x), smem + XL::raw(1), &bars[1]);
  }
  // rowwise: thread t owns row t / 2, columns 32 (t mod 2) .. + 31 (one
  // 1 x 32 block); its four 16-byte chunks sit at these swizzled offsets
  const int rr = t >> 1, rh = t & 1;
  uint32_t roff[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) roff[q] = (uint32_t)(rr * 128 + (((4 * rh + q) ^ (rr & 7)) << 4));
  int slot = 0;
  uint32_t phase = 0;
  while (cur.valid()) {
    const int64_t g = cur.g, m0 = (int64_t)cur.tm * XM, k0 = (int64_t)cur.tk * XK;
    const int after = cur.idx + 2 * (int)gridDim.x;  // the tile that takes this slot next
    cur.next();
    // a wait that runs out raises the error flag; the walk goes on (every
    // later wait is bounded and every barrier is still reached)
    if (!mbar_wait(&bars[slot], phase, 1u << 22)) atomicExch(&g_mx8_timeout, 1u);
    const unsigned char* raw = smem + XL::raw(slot);
    const int64_t m = m0 + rr, k = k0 + 32 * rh;
    if (m < j.M && k < j.K) {  // rows and columns past the edge arrive as zeros and are not used
      float v[32];
      uint32_t mx = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 w = *reinterpret_cast<const uint4*>(raw + roff[q]);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[8 * q + 2 * i] = bf16lo(ww[i]);
          v[8 * q + 2 * i + 1] = bf16hi(ww[i]);
          mx = q == 0 && i == 0 ? ww[i] : bf16x2_amax(mx, ww[i]);
        }
      }
      mx &= 0x7FFF7FFFu;
      const uint32_t hi = mx >> 16, lo = mx & 0xFFFFu;
      row_work<OUT_BF16>(j, v, (hi > lo ? hi : lo) << 16, g, m, k, rr, rh, ys);
    }
    __syncthreads();  // the staging is complete, the slot's reads are done
    if (t == 0 && after < cur.ntiles) mx8_issue(&tmap, cur.pos_of<XM>(after), smem + XL::raw(slot), &bars[slot]);
    if (j.col_codes) col_work(j, ys, g, m0, k0, t);
    __syncthreads();  // the staging is free for the next tile
    if (++slot == 2) {
      slot = 0;
      phase ^= 1u;
    }
  }
}

template <bool OUT_BF16>
cudaError_t launch_tma_t(const QuantJob& j, const CUtensorMap& map, cudaStream_t st) {
  auto kern = mxfp8_tma_kernel<OUT_BF16>;
  static int per_sm_cache[128] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 128) dev = 0;
  int& per_sm = per_sm_cache[dev];
  if (per_sm == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, XL::total);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, XT, XL::total);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
  }
  const int64_t tiles = j.G * ((j.M + XM - 1) / XM) * ((j.K + XK - 1) / XK);
  const int64_t cap = (int64_t)num_sms() * per_sm;
  return launch_pdl(kern, dim3((unsigned)(tiles < cap ? tiles : cap)), dim3(XT), (size_t)XL::total, st, j, map);
}

template <bool IN_BF16, bool OUT_BF16>
cudaError_t launch_t(const QuantJob& j, cudaStream_t st) {
  const int64_t tiles_m = (j.M + XM - 1) / XM, tiles_k = (j.K + XK - 1) / XK;
  return launch_pdl(mxfp8_kernel<IN_BF16, OUT_BF16>, dim3((unsigned)(j.G * tiles_m * tiles_k)), dim3(XT), 0, st, j,
                    tiles_m, tiles_k);
}

}  // namespace

// bf16 input whose rows the tensor copies can address (16-byte aligned base
// and row stride, tile counts in 32 bits) takes the persistent form;
// FP4Q_NO_MX8_TMA=1 turns it off (the tests run both forms).
cudaError_t launch_mxfp8(const QuantJob& j, cudaStream_t st) {
  if (j.in_bf16 && (reinterpret_cast<uintptr_t>(j.x) & 15u) == 0 && (j.ld * 2) % 16 == 0 &&
      j.G * ((j.M + XM - 1) / XM) * ((j.K + XK - 1) / XK) < ((int64_t)1 << 31) && !getenv_flag("FP4Q_NO_MX8_TMA")) {
    CUtensorMap map;
    if (make_bf16_tile_map(j, &map, XM)) return j.out_bf16 ? launch_tma_t<true>(j, map, st) : launch_tma_t<false>(j, map, st);
  }
  if (j.in_bf16) return j.out_bf16 ? launch_t<true, true>(j, st) : launch_t<true, false>(j, st);
  return j.out_bf16 ? launch_t<false, true>(j, st) : launch_t<false, false>(j, st);
}

cudaError_t mxfp8_timeout_flag(uint32_t* v, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(v, g_mx8_timeout, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_mx8_timeout, &z, sizeof z);
  }
  return e;
}

}  // namespace fp4q
