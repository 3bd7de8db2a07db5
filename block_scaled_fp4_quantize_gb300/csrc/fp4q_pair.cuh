// fp4q_pair.cuh -- the pair-table path shared by the bf16 kernels: with a
// bf16 outer amax A (bits), S = RN(A / (scale_max * 6)) has one of 128
// significands and an inner scale s one of 8, and RN(RN(u c1) c2) with the
// pair's multipliers gives the E2M1 code of RN(RN(u / S) / s) for every
// bf16 u ("NVFP4 / AMD-FP4 outer-block (two-level) scaling for FP4
// training", "Technical design": x' = u / S and the code of x' / s; the
// table, its image in shared memory and the enumeration that checks it:
// gen_pairtab.py, fp4q_pairtab.cuh).
#pragma once

#include "fp4q_block.cuh"
#include "fp4q_device.cuh"
#include "fp4q_pairtab.cuh"

namespace fp4q {
namespace {

// row of the shared table holding the split reciprocal (zh, zl) of S (rows
// 0-7: the pairs by inner significand; row 8: a zero inner scale)
constexpr uint32_t PT_RCP = 9;
// bytes of the kCtlTab image the two forms copy: the rows and the code table
// (outer scales), or the table of the form without outer scale
constexpr uint32_t kImgOuter = (10 * 128 * 2 + 256) * 4, kImgUnit = 256 * 2 * 4;
static_assert(kImgOuter + kImgUnit == kCtlTabWords * 4, "image layout");

// bits of the amax A = scale_max * 6 (S = 1): the table position of "no outer scale"
template <bool UE5M3>
__device__ __forceinline__ constexpr uint32_t unit_amax() { return UE5M3 ? 0x49280000u : 0x45280000u; }

// The amax bits A (a bf16 value) admit the table path: A in [2^-90, 2^101)
// (E4M3) or [2^-90, 2^109) (UE5M3), so that 2^-90 < S < 2^90.
template <bool UE5M3>
__device__ __forceinline__ bool table_ok(uint32_t A) {
  return A - kTiny < (UE5M3 ? 0x76000000u : 0x72000000u) - kTiny;
}

// byte offset of the amax's mantissa in a table row
__device__ __forceinline__ uint32_t moff_of(uint32_t A) { return (A >> 13) & 0x3F8u; }

// c1 and c2 of a block with scale code sc whose outer amax has bits A
__device__ __forceinline__ void pair_mults(const unsigned char* ptb, const uint32_t* ctab, uint32_t sc, uint32_t A,
                                           float& c1, float& c2) {
  const uint32_t w = ctab[sc];
  const uint2 e = *reinterpret_cast<const uint2*>(ptb + (w & 0xFFFFu) + moff_of(A));
  c1 = bitsf(e.x - A);
  c2 = bitsf(e.y + (w & 0xFF800000u));
}

// split reciprocal (zh, zl) of S for the amax bits A
__device__ __forceinline__ void outer_rcp(const unsigned char* ptb, uint32_t A, float& zh, float& zl) {
  const uint2 e = *reinterpret_cast<const uint2*>(ptb + PT_RCP * 1024u + moff_of(A));
  zh = bitsf(e.x - A);
  zl = bitsf(e.y - A);
}

// c1, c2 of the form without outer scale (S = 1): the unit table entry of
// scale code sc
__device__ __forceinline__ void unit_mults(const unsigned char* ntb, uint32_t sc, float& c1, float& c2) {
  const uint2 e = reinterpret_cast<const uint2*>(ntb)[sc];
  c1 = bitsf(e.x);
  c2 = bitsf(e.y);
}

// Inner-scale table entries computed on demand (for the general steps).
template <bool UE5M3>
struct EntryCalc {
  __device__ __forceinline__ float4 operator[](uint32_t c) const { return scale_entry<UE5M3>(c); }
};

}  // namespace
}  // namespace fp4q
