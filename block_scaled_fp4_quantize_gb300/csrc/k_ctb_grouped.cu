// k_ctb_grouped.cu -- the bf16 cast-transpose kernel over ragged groups of
// rows (fp4_quantize_grouped): each group's 128-row tiles, its own
// columnwise transpose and tensorwise scale.  Kernel body: k_ctb.cuh.
#include "k_ctb.cuh"

namespace fp4q {

bool launch_ctb_grouped(const QuantJob& j, cudaStream_t st, cudaError_t* err) {
  return launch_ctb_all<true, false>(j, st, err);
}

cudaError_t ctb_grouped_timeout_flag(uint32_t* v, bool clear) { return ctb_flag_rw(v, clear); }

}  // namespace fp4q
