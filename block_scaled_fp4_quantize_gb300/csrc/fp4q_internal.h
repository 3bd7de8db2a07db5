// fp4q_internal.h -- launch interfaces shared by the C ABI and the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "fp4q_device.cuh"

namespace fp4q {

// Where a kernel takes the outer scale S from.
enum SSource : int {
  S_ONE = 0,            // mode none: S = 1, no normalization
  S_TENSORWISE_WS = 1,  // S = amax / denom from the tensorwise amax in the workspace
  S_IN_TILE = 2,        // computed inside the tile kernel (ob divides 64)
  S_FROM_BUFFER = 3,    // read from the outer-scale buffers (precomputed or pre-pass)
};

// Inner-scale buffer layout of one orientation: per matrix an R x C16 byte
// matrix, linear, or in 128 x 4 tiles of 512 bytes (tile-row-major; inside a
// tile byte (r, c) at (r mod 32) * 16 + (r / 32) * 4 + c), R padded to 128
// and C16 to 4 per matrix.
struct ScaleLayout {
  int mma;
  int64_t R, C16, nrb, ncb;  // rows, scales per row, tile rows, tile columns
};

inline ScaleLayout make_scale_layout(int mma, int64_t R, int64_t C16) {
  return ScaleLayout{mma, R, C16, (R + 127) / 128, (C16 + 3) / 4};
}

// Byte offset of scale (g, r, c).
__host__ __device__ __forceinline__ int64_t sf_offset(const ScaleLayout& L, int64_t g, int64_t r, int64_t c) {
  if (!L.mma) return (g * L.R + r) * L.C16 + c;
  return ((g * L.nrb + (r >> 7)) * L.ncb + (c >> 2)) * 512 + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (c & 3);
}

// Byte offset of the scale whose linear index is `lin` ((g R + r) C16 + c).
__host__ __device__ __forceinline__ int64_t sf_from_linear(const ScaleLayout& L, int64_t lin) {
  if (!L.mma) return lin;
  const int64_t row = lin / L.C16, c = lin - row * L.C16;
  const int64_t g = row / L.R, r = row - g * L.R;
  return sf_offset(L, g, r, c);
}

// Bytes of an orientation's scale buffer for G matrices.
inline int64_t sf_bytes(const ScaleLayout& L, int64_t G) {
  return L.mma ? G * L.nrb * L.ncb * 512 : G * L.R * L.C16;
}

// Device workspace of a grouped quantize: a validity flag and the tile count
// (set by the preparation kernel), the per-group prefix of 128-row tiles
// (tprefix[e] = tiles of the groups before e) and the per-group amax.
struct GroupWs {
  uint32_t bad;     // nonzero: offsets invalid, nothing is written
  uint32_t mtiles;  // total 128-row tiles over all groups
  uint32_t pad[2];
  // followed by uint32_t tprefix[ngroups + 1], then uint32_t amax[ngroups]
};

inline size_t group_ws_bytes(int64_t ngroups) {
  return (size_t)(16 + 4 * (ngroups + 1) + 4 * ngroups + 255) / 256 * 256;
}
__host__ __device__ __forceinline__ uint32_t* group_tprefix(GroupWs* w) {
  return reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(w) + 16);
}
__host__ __device__ __forceinline__ uint32_t* group_amax(GroupWs* w, int64_t ngroups) {
  return group_tprefix(w) + ngroups + 1;
}

// One quantize / qdq job.  Rowwise quantities are indexed [G, M, K], the
// columnwise ones [G, K, M].
struct QuantJob {
  const void* x;
  int64_t ld;
  int in_bf16;
  int64_t G, M, K;
  float* residual;  // [G, M, K] contiguous, rowwise only
  int mode, ob, outer_2d, inner_2d, ue5m3, sr;
  uint64_t seed;
  PhiloxKeys srk;   // the round keys of `seed` (stochastic rounding)
  uint32_t step;
  int do_row, do_col;
  int s_src;
  const uint32_t* tw_amax;  // tensorwise amax (binary32 bits), S_TENSORWISE_WS only
  uint8_t* row_codes;
  uint8_t* row_scales;
  float* row_outer;
  uint8_t* col_codes;
  uint8_t* col_scales;
  float* col_outer;
  float* tile_outer;
  void* y;          // qdq output [G, M, K] contiguous, or nullptr
  int out_bf16;
  int qdq_orient;   // 0: quantize; 1: qdq along K; 2: qdq along M
  ScaleLayout rsl, csl;  // rowwise / columnwise inner-scale layouts
  // ragged groups (0 = none): rows [goff[e], goff[e + 1]) of the [M, K]
  // input form group e, quantized as a matrix of its own
  int64_t ngroups;
  const int64_t* goff;  // device [ngroups + 1]
  GroupWs* gws;         // device workspace of the grouped path
  int col_rht;          // 1: Hadamard transform along M before the columnwise side
  uint32_t rht_signs;   // its sign mask (bit i: element i of each 16-block negated)
  // global index of the stochastic-rounding counter: rowwise element with
  // local flat index n draws word n + sr_row_off; columnwise element of row
  // gk = g K + k (of x transposed), column m draws sr_col_off + gk sr_col_ld + m
  int64_t sr_row_off, sr_col_off, sr_col_ld;
};

__host__ __device__ __forceinline__ uint64_t sr_row_n(const QuantJob& j, int64_t n) {
  return (uint64_t)(n + j.sr_row_off);
}
__host__ __device__ __forceinline__ uint64_t sr_col_n(const QuantJob& j, int64_t gk, int64_t m) {
  return (uint64_t)(j.sr_col_off + gk * j.sr_col_ld + m);
}

struct DequantJob {
  const uint8_t* codes;
  const uint8_t* scales;
  const float* outer;
  void* y;
  int64_t G, R, C;   // orientation's logical shape
  int64_t M, K;      // the quantized tensor's shape (2-D scale indexing)
  int col;           // 1: columnwise buffers (2-D scales read transposed)
  int mode, ob, outer_2d, ue5m3, out_bf16;
  ScaleLayout sl;    // the scale buffer's layout (R x C/16 per matrix)
};

struct MxJob {
  const void* x;
  int64_t ld;
  int in_bf16, out_bf16;
  int64_t G, M, K;
  void* y;
};

int num_sms();
int vec_aligned(const void* p, int64_t bytes_stride);
// true when the environment variable is set to a value other than "" or "0"
// (kernel-selection switches used by the parity tests)
bool getenv_flag(const char* name);

cudaError_t launch_quant_tile(const QuantJob& j, bool vec, cudaStream_t st);
bool ct_supports(const QuantJob& j);
bool row_supports(const QuantJob& j);
bool ctb_supports(const QuantJob& j);
bool launch_ctb(const QuantJob& j, cudaStream_t st, cudaError_t* err);
bool launch_ctl(const QuantJob& j, cudaStream_t st, cudaError_t* err);
bool launch_ctb_grouped(const QuantJob& j, cudaStream_t st, cudaError_t* err);
bool launch_ctb_rht(const QuantJob& j, cudaStream_t st, cudaError_t* err);
cudaError_t launch_row(const QuantJob& j, cudaStream_t st);
cudaError_t launch_ct(const QuantJob& j, cudaStream_t st);
cudaError_t launch_tensor_amax(const QuantJob& j, uint32_t* amax_ws, cudaStream_t st);
cudaError_t launch_outer_prepass(const QuantJob& j, cudaStream_t st);
cudaError_t launch_dequant(const DequantJob& j, cudaStream_t st);
cudaError_t launch_mxfp4(const MxJob& j, cudaStream_t st);
// fused MXFP4 projection + MXFP8 re-encode: x, ld, G, M, K, in_bf16, out_bf16,
// y (optional), row_codes / row_scales, col_codes / col_scales
cudaError_t launch_mxfp8(const QuantJob& j, cudaStream_t st);
// grouped path: offsets check + tile prefix (+ per-group amax for tensorwise)
cudaError_t launch_group_prep(const QuantJob& j, int align, bool amax, cudaStream_t st);

// Bounded-wait timeout flags of the TMA-fed kernels, one per translation
// unit that has such waits: read (and optionally clear) the flag of the
// current device (synchronous copies), or set it as a timed-out wait would.
cudaError_t ctb_timeout_flag(uint32_t* v, bool clear);
cudaError_t ctb_grouped_timeout_flag(uint32_t* v, bool clear);
cudaError_t ctb_rht_timeout_flag(uint32_t* v, bool clear);
cudaError_t row_timeout_flag(uint32_t* v, bool clear);
cudaError_t ct_timeout_flag(uint32_t* v, bool clear);
cudaError_t mxfp8_timeout_flag(uint32_t* v, bool clear);
cudaError_t ctl_timeout_flag(uint32_t* v, bool clear);
cudaError_t set_ctb_timeout_flag();

}  // namespace fp4q
