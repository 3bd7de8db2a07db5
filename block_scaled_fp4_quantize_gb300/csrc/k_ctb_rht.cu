// k_ctb_rht.cu -- the bf16 cast-transpose kernel with a random Hadamard
// transform along M on the columnwise side ("NVFP4 / AMD-FP4 outer-block
// (two-level) scaling for FP4 training", "Op-level test coverage":
// outer-block scaling combined with an M-axis Hadamard transform): each
// 16-row column block is sign-flipped by a 16-bit mask, multiplied by the
// 16 x 16 Sylvester Hadamard matrix (fast Walsh-Hadamard butterfly in
// binary32) and scaled by 1/4 before its outer and inner scales are taken.
// Kernel body: k_ctb.cuh.
#include "k_ctb.cuh"

namespace fp4q {

bool launch_ctb_rht(const QuantJob& j, cudaStream_t st, cudaError_t* err) {
  return launch_ctb_all<false, true>(j, st, err);
}

cudaError_t ctb_rht_timeout_flag(uint32_t* v, bool clear) { return ctb_flag_rw(v, clear); }

}  // namespace fp4q
