// k_mxfp4.cu -- MXFP4 fake-quantize ("MXFP4 weight QAT recipes on MXFP8 and
// FP8 block-scaling hosts", "Overview" and "Design").
//
// Pure streaming kernel: every 1 x 32 block is read once with 128-bit loads
// spread over 4 (bf16) or 8 (fp32) neighbouring lanes, its |x| maximum and
// inf/NaN flag are reduced with two or three xor-shuffles, the power-of-two
// exponent is derived from the maximum's exponent and mantissa bits, and the
// projected values are written back with 128-bit stores.
#include "fp4q_device.cuh"
#include "fp4q_internal.h"

namespace fp4q {
namespace {

constexpr int NT = 256;
constexpr int UNR = 4;   // independent 16-byte loads in flight per thread (16-byte path)
constexpr int WUNR = 2;  // independent 32-byte loads in flight per thread (32-byte path)

// Block exponent E for the block maximum |x| bits (finite): least E with
// 6 * 2^E >= max(A, 6 * 2^-126), capped at 125.  Writing the clamped maximum
// as (1 + f) 2^k: E = k - 2 if (1 + f) <= 1.5 else k - 1.
__device__ __forceinline__ int mx_exponent(uint32_t amax_bits) {
  const uint32_t ac = amax_bits > 0x01C00000u ? amax_bits : 0x01C00000u;  // 6 * 2^-126
  const int k = (int)(ac >> 23) - 127;
  const int e = (ac & 0x7FFFFFu) <= 0x400000u ? k - 2 : k - 1;
  return e < 125 ? e : 125;
}

// A 32-byte unit (two 16-byte halves) for the 256-bit access path.
struct U32B {
  uint4 a, b;
};

__device__ __forceinline__ U32B ld256_stream(const void* p) {
  U32B r;
  asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r.a.x), "=r"(r.a.y), "=r"(r.a.z), "=r"(r.a.w), "=r"(r.b.x), "=r"(r.b.y), "=r"(r.b.z),
                 "=r"(r.b.w)
               : "l"(p));
  return r;
}

template <typename TI>
struct InTraits;
template <>
struct InTraits<uint16_t> {
  static constexpr int EPU = 8;  // elements per 16-byte unit
  __device__ static void unpack(const uint4& w, float* x) {
    x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
    x[4] = bf16lo(w.z); x[5] = bf16hi(w.z); x[6] = bf16lo(w.w); x[7] = bf16hi(w.w);
  }
  __device__ static float load1(const void* p, int64_t i) {
    return bitsf((uint32_t) static_cast<const uint16_t*>(p)[i] << 16);
  }
};
template <>
struct InTraits<float> {
  static constexpr int EPU = 4;
  __device__ static void unpack(const uint4& w, float* x) {
    x[0] = bitsf(w.x); x[1] = bitsf(w.y); x[2] = bitsf(w.z); x[3] = bitsf(w.w);
  }
  __device__ static float load1(const void* p, int64_t i) { return static_cast<const float*>(p)[i]; }
};

// Project EPU values (the unit's share of one block) given the block's
// exponent; poisoned blocks become the canonical quiet NaN.
template <int EPU, bool OUT_BF16>
__device__ __forceinline__ void project_store(const float* x, int E, bool poison, void* y, int64_t yi) {
  const float inv = bitsf((uint32_t)(127 - E) << 23);
  const float sc = bitsf((uint32_t)(127 + E) << 23);
  float o[EPU];
#pragma unroll
  for (int i = 0; i < EPU; i += 2) {
    const uint32_t b = e2m1x2_rne(ieee_mul(x[i], inv), ieee_mul(x[i + 1], inv));
    float g0, g1;
    e2m1x2_decode(b, g0, g1);
    o[i] = ieee_mul(g0, sc);
    o[i + 1] = ieee_mul(g1, sc);
  }
  if (OUT_BF16) {
    uint32_t w[EPU / 2];
#pragma unroll
    for (int i = 0; i < EPU / 2; ++i) w[i] = poison ? 0x7FC07FC0u : pack_bf16x2(o[2 * i], o[2 * i + 1]);
    uint16_t* p = static_cast<uint16_t*>(y) + yi;
    if (EPU == 8) *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    else *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
  } else {
    float* p = static_cast<float*>(y) + yi;
    const float qn = bitsf(0x7FC00000u);
#pragma unroll
    for (int i = 0; i < EPU; i += 4)
      reinterpret_cast<float4*>(p)[i / 4] =
          poison ? make_float4(qn, qn, qn, qn) : make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
  }
}

template <typename TI, bool OUT_BF16, bool CONTIG>
__global__ void __launch_bounds__(NT) mxfp4_vec_kernel(const MxJob j) {
  constexpr int EPU = InTraits<TI>::EPU;
  constexpr int L = 32 / EPU;  // lanes per 1 x 32 block
  const int64_t units_per_row = j.K / EPU;
  const int64_t U = j.G * j.M * units_per_row;
  const TI* x = static_cast<const TI*>(j.x);
  for (int64_t base = (int64_t)blockIdx.x * NT * UNR; base < U; base += (int64_t)gridDim.x * NT * UNR) {
    uint4 w[UNR];
#pragma unroll
    for (int p = 0; p < UNR; ++p) {
      const int64_t u = base + p * NT + threadIdx.x;
      w[p] = make_uint4(0u, 0u, 0u, 0u);
      if (u < U) {
        const int64_t off = CONTIG ? u * EPU : (u / units_per_row) * j.ld + (u % units_per_row) * EPU;
        w[p] = __ldcs(reinterpret_cast<const uint4*>(x + off));
      }
    }
#pragma unroll
    for (int p = 0; p < UNR; ++p) {
      const int64_t u = base + p * NT + threadIdx.x;
      float v[EPU];
      InTraits<TI>::unpack(w[p], v);
      uint32_t am = 0;
#pragma unroll
      for (int i = 0; i < EPU; ++i) { const uint32_t a = abs_bits(v[i]); am = a > am ? a : am; }
#pragma unroll
      for (int o = 1; o < L; o <<= 1) { const uint32_t b = __shfl_xor_sync(0xFFFFFFFFu, am, o); am = b > am ? b : am; }
      if (u < U) project_store<EPU, OUT_BF16>(v, mx_exponent(am), am >= 0x7F800000u, j.y, u * EPU);
    }
  }
}

// bf16 in, bf16 out, contiguous and 32-byte aligned: every lane owns a
// 32-byte unit (half a 1 x 32 block), 256-bit loads and stores, one
// xor-shuffle per block.
//
// Launched with programmatic dependent launch: the kernel first waits for the
// previous grid on the stream to complete (griddepcontrol.wait: its writes are
// then visible), then lets the next grid be scheduled, so back-to-back calls
// overlap launch latency with the previous call's tail instead of idling.
// Without the launch attribute both instructions are no-ops.
__global__ void __launch_bounds__(NT) mxfp4_wide_kernel(const MxJob j) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int64_t U = j.G * j.M * j.K / 16;
  const uint16_t* x = static_cast<const uint16_t*>(j.x);
  uint16_t* y = static_cast<uint16_t*>(j.y);
  for (int64_t base = (int64_t)blockIdx.x * NT * WUNR; base < U; base += (int64_t)gridDim.x * NT * WUNR) {
    U32B w[WUNR];
#pragma unroll
    for (int p = 0; p < WUNR; ++p) {
      const int64_t u = base + p * NT + threadIdx.x;
      if (u < U) w[p] = ld256_stream(x + u * 16);
      else w[p] = U32B{make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
    }
#pragma unroll
    for (int p = 0; p < WUNR; ++p) {
      const int64_t u = base + p * NT + threadIdx.x;
      float v[16];
      InTraits<uint16_t>::unpack(w[p].a, v);
      InTraits<uint16_t>::unpack(w[p].b, v + 8);
      uint32_t am = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) { const uint32_t a = abs_bits(v[i]); am = a > am ? a : am; }
      { const uint32_t b = __shfl_xor_sync(0xFFFFFFFFu, am, 1); am = b > am ? b : am; }
      if (u < U) {
        const int E = mx_exponent(am);
        const bool poison = am >= 0x7F800000u;
        const float inv = bitsf((uint32_t)(127 - E) << 23);
        const float sc = bitsf((uint32_t)(127 + E) << 23);
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const uint32_t b = e2m1x2_rne(ieee_mul(v[i], inv), ieee_mul(v[i + 1], inv));
          float g0, g1;
          e2m1x2_decode(b, g0, g1);
          o[i / 2] = poison ? 0x7FC07FC0u : pack_bf16x2(ieee_mul(g0, sc), ieee_mul(g1, sc));
        }
        st256(y + u * 16, o);
      }
    }
  }
}

// Any alignment: one thread per 1 x 32 block, scalar accesses.
template <typename TI, bool OUT_BF16>
__global__ void __launch_bounds__(NT) mxfp4_scalar_kernel(const MxJob j) {
  const int64_t nb_row = j.K / 32;
  const int64_t nblk = j.G * j.M * nb_row;
  for (int64_t b = (int64_t)blockIdx.x * NT + threadIdx.x; b < nblk; b += (int64_t)gridDim.x * NT) {
    const int64_t row = b / nb_row, k0 = (b % nb_row) * 32;
    float v[32];
    uint32_t am = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      v[i] = InTraits<TI>::load1(j.x, row * j.ld + k0 + i);
      const uint32_t a = abs_bits(v[i]);
      am = a > am ? a : am;
    }
    const int E = mx_exponent(am);
    const bool poison = am >= 0x7F800000u;
    const float inv = bitsf((uint32_t)(127 - E) << 23);
    const float sc = bitsf((uint32_t)(127 + E) << 23);
    const int64_t yi = row * j.K + k0;
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const uint32_t q = e2m1x2_rne(ieee_mul(v[i], inv), ieee_mul(v[i + 1], inv));
      float g0, g1;
      e2m1x2_decode(q, g0, g1);
      const float o0 = ieee_mul(g0, sc), o1 = ieee_mul(g1, sc);
      if (OUT_BF16) {
        const uint32_t w = poison ? 0x7FC07FC0u : pack_bf16x2(o0, o1);
        static_cast<uint16_t*>(j.y)[yi + i] = (uint16_t)(w & 0xFFFFu);
        static_cast<uint16_t*>(j.y)[yi + i + 1] = (uint16_t)(w >> 16);
      } else {
        const float qn = bitsf(0x7FC00000u);
        static_cast<float*>(j.y)[yi + i] = poison ? qn : o0;
        static_cast<float*>(j.y)[yi + i + 1] = poison ? qn : o1;
      }
    }
  }
}

template <typename TI, bool OUT_BF16>
cudaError_t launch_typed(const MxJob& j, cudaStream_t st) {
  constexpr int EPU = InTraits<TI>::EPU;
  const int esz = (int)sizeof(TI);
  const bool vec = vec_aligned(j.x, j.ld * esz) && vec_aligned(j.y, 16) &&
                   (OUT_BF16 ? (EPU * 2) % 8 == 0 : true);
  const bool wide = sizeof(TI) == 2 && OUT_BF16 && (j.ld == j.K || j.G * j.M == 1) &&
                    ((reinterpret_cast<uintptr_t>(j.x) | reinterpret_cast<uintptr_t>(j.y)) & 31u) == 0 &&
                    !getenv_flag("FP4Q_MXFP4_NARROW");
  // grids of 8 CTAs per SM: more than are resident at once, which measured
  // faster than exactly the resident count (the hardware balances the tail)
  const int64_t cap = (int64_t)num_sms() * 8;
  if (wide) {
    const int64_t U = j.G * j.M * j.K / 16;
    const int64_t need = (U + NT * WUNR - 1) / (NT * WUNR);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(need < cap ? need : cap));
    cfg.blockDim = dim3(NT);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, mxfp4_wide_kernel, j);
    if (e != cudaSuccess) return e;
  } else if (vec) {
    const int64_t U = j.G * j.M * (j.K / EPU);
    const int64_t need = (U + NT * UNR - 1) / (NT * UNR);
    const int grid = (int)(need < cap ? need : cap);
    if (j.ld == j.K) mxfp4_vec_kernel<TI, OUT_BF16, true><<<grid, NT, 0, st>>>(j);
    else mxfp4_vec_kernel<TI, OUT_BF16, false><<<grid, NT, 0, st>>>(j);
  } else {
    const int64_t nblk = j.G * j.M * (j.K / 32);
    const int64_t need = (nblk + NT - 1) / NT;
    mxfp4_scalar_kernel<TI, OUT_BF16><<<(int)(need < cap ? need : cap), NT, 0, st>>>(j);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mxfp4(const MxJob& j, cudaStream_t st) {
  if (j.in_bf16) return j.out_bf16 ? launch_typed<uint16_t, true>(j, st) : launch_typed<uint16_t, false>(j, st);
  return j.out_bf16 ? launch_typed<float, true>(j, st) : launch_typed<float, false>(j, st);
}

}  // namespace fp4q
