// k_ctb.cu -- bf16 cast-transpose quantize: rowwise and columnwise NVFP4 /
// AMD-FP4 codes from one TMA-staged 128 x 64 tile
// ("Block-Scaled FP8 and FP4 Weight Quantization", section 3, the fused
// cast-transpose; "NVFP4 / AMD-FP4 outer-block (two-level) scaling for FP4
// training", "Technical design", outer and inner scales).
//
// A CTA of 256 threads walks 128 (M) x 64 (K) tiles of x; each tile arrives
// by a 3-D tensor copy with the 128-byte swizzle, two tiles in flight per
// CTA and four CTAs resident per SM.
//
//   Rowwise pass: thread t owns row t / 2 and the two 1 x 16 blocks of its
//   half (t mod 2) of the 64 columns; four 16-byte shared loads, block maxima
//   from packed bf16 maxima, then the per-block steps of fp4q_block.cuh.
//
//   Columnwise pass: warp w owns rows 16 w .. 16 w + 15, lane l columns 2 l
//   and 2 l + 1, so a lane holds two whole 16 x 1 blocks.  Each of its 16
//   shared loads is one 32-bit bf16 pair of one row (a warp reads one whole
//   128-byte row: no bank conflicts), and the two blocks' maxima come from
//   one packed maximum tree.  A 1-D outer block along M spanning several
//   warps is reduced in shared memory.  Codes and scales go to a staging
//   area and leave as 16-byte rows of the transposed outputs.
//
// Outer-scale sources are template cases: none, one scale for the tensor,
// 1-D or 2-D outer blocks computed in the tile (ob in {16, 32, 64}), and 1-D
// or 2-D outer scales read from the outer buffers.
#include "k_ctb.cuh"

namespace fp4q {

bool ctb_supports(const QuantJob& j) {
  // columnwise bf16 quantize, and rowwise-only bf16 quantize into the
  // tensor-core scale layout (tile-aligned scale addressing)
  return j.in_bf16 && (j.do_col || j.rsl.mma || j.ngroups > 0) && j.qdq_orient == 0 && !j.residual && !j.inner_2d &&
         (reinterpret_cast<uintptr_t>(j.x) & 15u) == 0 && (j.ld * 2) % 16 == 0;
}

// false: the tensor map could not be built (the caller takes another kernel)
bool launch_ctb(const QuantJob& j, cudaStream_t st, cudaError_t* err) {
  if (launch_ctl(j, st, err)) return true;  // the whole-tile form (k_ctl.cu)
  if (j.ngroups > 0) return launch_ctb_grouped(j, st, err);
  if (j.col_rht) return launch_ctb_rht(j, st, err);
  return launch_ctb_all<false, false>(j, st, err);
}

cudaError_t ctb_timeout_flag(uint32_t* v, bool clear) { return ctb_flag_rw(v, clear); }

cudaError_t set_ctb_timeout_flag() {
  const uint32_t one = 1;
  return cudaMemcpyToSymbol(g_ctb_timeout, &one, sizeof one);
}

}  // namespace fp4q
