// fp4q_api.cu -- the C ABI: argument validation, path selection, launches.
//
// Nothing here allocates or frees, and only fp4q_device_status synchronizes;
// all work is enqueued on the caller's stream.  Validation happens before any launch, so an error other
// than FP4Q_ERR_CUDA leaves the stream untouched.
#include <cstdint>
#include <cstdlib>

#include "fp4q.h"
#include "fp4q_internal.h"

namespace fp4q {

int num_sms() {
  static int cache[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

int vec_aligned(const void* p, int64_t bytes_stride) {
  return (reinterpret_cast<uintptr_t>(p) % 16u == 0u) && (bytes_stride % 16 == 0);
}

bool getenv_flag(const char* name) {
  const char* v = std::getenv(name);
  return v && v[0] && v[0] != '0';
}

}  // namespace fp4q

using namespace fp4q;

namespace {

bool aligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0u; }

// Workspace of a tensorwise quantize: the amax word (the rest is padding).
constexpr size_t kTensorwiseWsBytes = 256;
static_assert(kTensorwiseWsBytes <= FP4Q_NOALLOC_SCRATCH_BYTES,
              "fp4_quantize_noalloc's static scratch must hold the tensorwise workspace");

int esize(int32_t dt) { return dt == FP4Q_BF16 ? 2 : 4; }

// The NVFP4 knobs that MXFP4 fake-quantize and the MXFP8 re-encode do not take.
bool mx_knobs_default(const fp4q_params_t* p) {
  return p->mode == FP4Q_MODE_NONE && p->outer_block_size == 0 && p->outer_2d == 0 && p->inner_2d == 0 &&
         p->scale_format == FP4Q_SCALE_E4M3 && p->use_precomputed_outer == 0 && p->scale_layout == 0 &&
         p->col_hadamard == 0 && p->precomputed_amax == 0;
}

int check_dtype(int32_t dt) {
  if (dt == FP4Q_BF16 || dt == FP4Q_FP32) return FP4Q_OK;
  return FP4Q_ERR_DTYPE;
}

// Rules shared by quantize and qdq; `mask` is the set of orientations produced.
int check_nvfp4(const fp4q_params_t* p, uint32_t mask) {
  if (!p) return FP4Q_ERR_NULL;
  if (p->struct_size != sizeof(fp4q_params_t)) return FP4Q_ERR_ABI;
  int rc = check_dtype(p->in_dtype);
  if (rc) return rc;
  if (mask == 0u || (mask & ~3u)) return FP4Q_ERR_MODE;
  if (p->mode < FP4Q_MODE_NONE || p->mode > FP4Q_MODE_OUTER_BLOCK) return FP4Q_ERR_MODE;
  if (p->scale_format != FP4Q_SCALE_E4M3 && p->scale_format != FP4Q_SCALE_UE5M3) return FP4Q_ERR_MODE;
  if (p->rounding != FP4Q_RNE && p->rounding != FP4Q_STOCHASTIC) return FP4Q_ERR_MODE;
  if ((p->outer_2d & ~1) || (p->inner_2d & ~1) || (p->use_precomputed_outer & ~1)) return FP4Q_ERR_MODE;
  if (p->scale_layout != FP4Q_SCALE_LAYOUT_LINEAR && p->scale_layout != FP4Q_SCALE_LAYOUT_MMA) return FP4Q_ERR_MODE;
  if (p->col_hadamard & ~1) return FP4Q_ERR_MODE;
  if (p->precomputed_amax & ~1) return FP4Q_ERR_MODE;
  if (p->precomputed_amax && (p->mode != FP4Q_MODE_TENSORWISE || p->use_precomputed_outer)) return FP4Q_ERR_MODE;
  if (p->G < 0 || p->M < 0 || p->K < 0 || p->ld < p->K) return FP4Q_ERR_SHAPE;
  // the stochastic-rounding counter's global index (a block of a larger tensor)
  if (p->sr_global_rows < 0 || p->sr_row_offset < 0 || p->sr_matrix_offset < 0) return FP4Q_ERR_SHAPE;
  if (p->sr_global_rows && p->sr_row_offset + p->M > p->sr_global_rows) return FP4Q_ERR_SHAPE;
  if (!p->sr_global_rows && p->sr_row_offset) return FP4Q_ERR_SHAPE;
  if (p->G > 1 && p->sr_global_rows && p->sr_global_rows != p->M) return FP4Q_ERR_UNSUPPORTED;
  if (p->K % 16) return FP4Q_ERR_SHAPE;
  const bool col = (mask & FP4Q_OUT_COL) != 0u;
  if ((col || p->inner_2d) && p->M % 16) return FP4Q_ERR_SHAPE;
  if (p->mode == FP4Q_MODE_OUTER_BLOCK) {
    const int64_t ob = p->outer_block_size;
    if (ob <= 0 || ob % 16) return FP4Q_ERR_SHAPE;
    if (p->K % ob) return FP4Q_ERR_SHAPE;
    if ((col || p->outer_2d) && p->M % ob) return FP4Q_ERR_SHAPE;
  } else {
    if (p->outer_block_size != 0 || p->outer_2d != 0) return FP4Q_ERR_MODE;
    if (p->mode == FP4Q_MODE_NONE && p->use_precomputed_outer) return FP4Q_ERR_MODE;
  }
  return FP4Q_OK;
}

void sizes_for(const fp4q_params_t* p, uint32_t mask, fp4q_sizes_t* s) {
  const int64_t G = p->G, M = p->M, K = p->K, ob = p->outer_block_size;
  const bool row = (mask & FP4Q_OUT_ROW) != 0u, col = (mask & FP4Q_OUT_COL) != 0u;
  const bool outer = p->mode == FP4Q_MODE_OUTER_BLOCK;
  s->row_codes = row ? (size_t)(G * M * K / 2) : 0;
  const int mma = p->scale_layout == FP4Q_SCALE_LAYOUT_MMA;
  s->row_scales = row ? (size_t)sf_bytes(make_scale_layout(mma, M, K / 16), G) : 0;
  s->col_codes = col ? (size_t)(G * K * M / 2) : 0;
  s->col_scales = col ? (size_t)sf_bytes(make_scale_layout(mma, K, M / 16), G) : 0;
  s->row_outer = (outer && !p->outer_2d && row) ? (size_t)(G * M * (K / ob)) * sizeof(float) : 0;
  s->col_outer = (outer && !p->outer_2d && col) ? (size_t)(G * K * (M / ob)) * sizeof(float) : 0;
  s->tile_outer = (outer && p->outer_2d) ? (size_t)(G * (M / ob) * (K / ob)) * sizeof(float)
                  : (p->mode == FP4Q_MODE_TENSORWISE ? sizeof(float) : 0);
  s->workspace = (p->mode == FP4Q_MODE_TENSORWISE && !p->use_precomputed_outer) ? kTensorwiseWsBytes : 0;
}

QuantJob base_job(const fp4q_params_t* p, const void* x, float* residual) {
  QuantJob j{};
  j.x = x;
  j.ld = p->ld;
  j.in_bf16 = p->in_dtype == FP4Q_BF16;
  j.G = p->G;
  j.M = p->M;
  j.K = p->K;
  j.residual = residual;
  j.mode = p->mode;
  j.ob = p->outer_block_size;
  j.outer_2d = p->outer_2d;
  j.inner_2d = p->inner_2d;
  j.ue5m3 = p->scale_format == FP4Q_SCALE_UE5M3;
  j.sr = p->rounding == FP4Q_STOCHASTIC;
  j.seed = p->seed;
  j.srk = philox_keys(p->seed);
  j.step = p->step;
  j.out_bf16 = p->out_dtype == FP4Q_BF16;
  const int mma = p->scale_layout == FP4Q_SCALE_LAYOUT_MMA;
  j.rsl = make_scale_layout(mma, p->M, p->K / 16);
  j.csl = make_scale_layout(mma, p->K, p->M / 16);
  // global index of the SR counter: this call is block [g0 : + G, r0 : + M]
  // of a [*, Mg, K] tensor (with G > 1, Mg == M and r0 == 0)
  const int64_t Mg = p->sr_global_rows ? p->sr_global_rows : p->M;
  j.sr_row_off = (p->sr_matrix_offset * Mg + p->sr_row_offset) * p->K;
  j.sr_col_off = p->sr_matrix_offset * p->K * Mg + p->sr_row_offset;
  j.sr_col_ld = Mg;
  return j;
}

// Pick the outer-scale source, running the amax / pre-pass kernels it needs.
int prepare_outer(const fp4q_params_t* p, QuantJob& j, void* ws, cudaStream_t st) {
  if (p->mode == FP4Q_MODE_NONE) {
    j.s_src = S_ONE;
    return FP4Q_OK;
  }
  if (p->use_precomputed_outer) {
    j.s_src = S_FROM_BUFFER;
    return FP4Q_OK;
  }
  if (p->mode == FP4Q_MODE_TENSORWISE) {
    j.s_src = S_TENSORWISE_WS;
    j.tw_amax = static_cast<uint32_t*>(ws);
    if (p->precomputed_amax) return FP4Q_OK;  // the caller's amax is in the workspace
    return launch_tensor_amax(j, static_cast<uint32_t*>(ws), st) == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
  }
  const int ob = p->outer_block_size;
  if (ob == 16 || ob == 32 || ob == 64) {
    j.s_src = S_IN_TILE;
    return FP4Q_OK;
  }
  j.s_src = S_FROM_BUFFER;
  return launch_outer_prepass(j, st) == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
}

// Kernel choice: rowwise-only work on a packed, 32-byte-aligned tensor
// streams through the flat rowwise kernel; other 16-byte-aligned work with
// 1 x 16 inner blocks runs in the cast-transpose tile kernel; everything
// else (16 x 16 inner blocks, unaligned views) in the general tile kernel.
// Columnwise bf16 quantize takes the bf16 cast-transpose kernel.
// FP4Q_GENERAL_KERNEL=1 forces the general kernel; FP4Q_NO_ROW_KERNEL=1 and
// FP4Q_NO_CTB_KERNEL=1 skip the flat and the bf16 cast-transpose kernels
// (for parity testing of each path).
int launch_quantizer(const QuantJob& j, bool vec, cudaStream_t st) {
  cudaError_t e;
  if (j.col_rht) {  // only the bf16 cast-transpose kernel has the transform
    if (!launch_ctb(j, st, &e)) return FP4Q_ERR_CUDA;
    return e == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
  }
  const bool fast = vec && ct_supports(j) && !getenv_flag("FP4Q_GENERAL_KERNEL");
  if (fast && row_supports(j) && !getenv_flag("FP4Q_NO_ROW_KERNEL")) e = launch_row(j, st);
  else if (fast && ctb_supports(j) && !getenv_flag("FP4Q_NO_CTB_KERNEL") && launch_ctb(j, st, &e)) {}
  else if (fast) e = launch_ct(j, st);
  else e = launch_quant_tile(j, vec, st);
  return e == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
}

bool vec_ok(const fp4q_params_t* p, const void* x, const float* residual, const void* y) {
  return vec_aligned(x, p->ld * esize(p->in_dtype)) && (!residual || aligned(residual, 16)) && (!y || aligned(y, 16));
}

}  // namespace

extern "C" {

void fp4q_params_init(fp4q_params_t* p) {
  if (!p) return;
  *p = fp4q_params_t{};
  p->struct_size = sizeof(fp4q_params_t);
  p->out_mask = FP4Q_OUT_ROW;
  p->G = 1;
  p->in_dtype = FP4Q_BF16;
  p->out_dtype = FP4Q_BF16;
  p->mode = FP4Q_MODE_NONE;
  p->scale_format = FP4Q_SCALE_E4M3;
  p->rounding = FP4Q_RNE;
}

int fp4q_query_sizes(const fp4q_params_t* p, fp4q_sizes_t* sizes) {
  if (!p || !sizes) return FP4Q_ERR_NULL;
  const int rc = check_nvfp4(p, p->out_mask);
  if (rc) return rc;
  sizes_for(p, p->out_mask, sizes);
  return FP4Q_OK;
}

int fp4_quantize(const fp4q_params_t* p, const void* x, const fp4q_outputs_t* out, float* residual, void* workspace,
                 size_t workspace_bytes, void* stream) {
  if (!p || !out) return FP4Q_ERR_NULL;
  int rc = check_nvfp4(p, p->out_mask);
  if (rc) return rc;
  const uint32_t mask = p->out_mask;
  const bool row = mask & FP4Q_OUT_ROW, col = mask & FP4Q_OUT_COL;
  if (residual && col) return FP4Q_ERR_UNSUPPORTED;
  fp4q_sizes_t s;
  sizes_for(p, mask, &s);
  const bool empty = p->G == 0 || p->M == 0 || p->K == 0;
  if (!empty) {
    if (!x) return FP4Q_ERR_NULL;
    if (row && (!out->row_codes || !out->row_scales)) return FP4Q_ERR_NULL;
    if (col && (!out->col_codes || !out->col_scales)) return FP4Q_ERR_NULL;
    if (s.row_outer && !out->row_outer) return FP4Q_ERR_NULL;
    if (s.col_outer && !out->col_outer) return FP4Q_ERR_NULL;
  }
  if (s.tile_outer && !out->tile_outer) return FP4Q_ERR_NULL;
  if (s.workspace && (!workspace || workspace_bytes < s.workspace)) return FP4Q_ERR_WORKSPACE;
  if (s.workspace && !aligned(workspace, 16)) return FP4Q_ERR_ALIGN;
  if (!aligned(x, (uintptr_t)esize(p->in_dtype))) return FP4Q_ERR_ALIGN;
  if ((row && !aligned(out->row_codes, 8)) || (col && !aligned(out->col_codes, 8))) return FP4Q_ERR_ALIGN;
  if (!aligned(out->row_outer, 4) || !aligned(out->col_outer, 4) || !aligned(out->tile_outer, 4)) return FP4Q_ERR_ALIGN;
  if (residual && !aligned(residual, 16)) return FP4Q_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (empty) {
    if (p->mode == FP4Q_MODE_TENSORWISE && !p->use_precomputed_outer && !p->precomputed_amax)
      return cudaMemsetAsync(out->tile_outer, 0, sizeof(float), st) == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
    return FP4Q_OK;
  }
  if (p->col_hadamard) {
    const int ob = p->outer_block_size;
    if (!col) return FP4Q_ERR_MODE;
    if (p->in_dtype != FP4Q_BF16 || p->inner_2d || p->mode == FP4Q_MODE_TENSORWISE || p->use_precomputed_outer ||
        (p->mode == FP4Q_MODE_OUTER_BLOCK && (p->outer_2d || !(ob == 16 || ob == 32 || ob == 64))) ||
        !vec_ok(p, x, residual, nullptr))
      return FP4Q_ERR_UNSUPPORTED;
  }
  QuantJob j = base_job(p, x, residual);
  j.col_rht = p->col_hadamard;
  j.rht_signs = p->hadamard_signs & 0xFFFFu;
  j.do_row = row;
  j.do_col = col;
  j.row_codes = row ? out->row_codes : nullptr;
  j.row_scales = row ? out->row_scales : nullptr;
  j.col_codes = col ? out->col_codes : nullptr;
  j.col_scales = col ? out->col_scales : nullptr;
  j.row_outer = s.row_outer ? out->row_outer : nullptr;
  j.col_outer = s.col_outer ? out->col_outer : nullptr;
  j.tile_outer = s.tile_outer ? out->tile_outer : nullptr;
  // tensor-core scale layout: the kernels write every real scale; the padding
  // of partial 128 x 4 tiles is zero
  if (j.rsl.mma && row && (p->M % 128 || (p->K / 16) % 4) &&
      cudaMemsetAsync(j.row_scales, 0, s.row_scales, st) != cudaSuccess)
    return FP4Q_ERR_CUDA;
  if (j.csl.mma && col && (p->K % 128 || (p->M / 16) % 4) &&
      cudaMemsetAsync(j.col_scales, 0, s.col_scales, st) != cudaSuccess)
    return FP4Q_ERR_CUDA;
  rc = prepare_outer(p, j, workspace, st);
  if (rc) return rc;
  return launch_quantizer(j, vec_ok(p, x, residual, nullptr), st);
}

int fp4q_query_sizes_grouped(const fp4q_params_t* p, int64_t ngroups, fp4q_sizes_t* sizes) {
  if (!p || !sizes) return FP4Q_ERR_NULL;
  const int rc = check_nvfp4(p, p->out_mask);
  if (rc) return rc;
  if (p->G != 1 || ngroups < 1 || ngroups > 65535) return FP4Q_ERR_SHAPE;
  sizes_for(p, p->out_mask, sizes);
  if (p->mode == FP4Q_MODE_TENSORWISE) sizes->tile_outer = (size_t)ngroups * sizeof(float);
  sizes->workspace = group_ws_bytes(ngroups);
  return FP4Q_OK;
}

int fp4_quantize_grouped(const fp4q_params_t* p, const void* x, const int64_t* offsets, int64_t ngroups,
                         const fp4q_outputs_t* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (!p || !out) return FP4Q_ERR_NULL;
  fp4q_sizes_t s;
  int rc = fp4q_query_sizes_grouped(p, ngroups, &s);
  if (rc) return rc;
  const uint32_t mask = p->out_mask;
  const bool row = mask & FP4Q_OUT_ROW, col = mask & FP4Q_OUT_COL;
  const bool small_ob = p->outer_block_size == 16 || p->outer_block_size == 32 || p->outer_block_size == 64;
  if (p->in_dtype != FP4Q_BF16 || p->inner_2d || p->scale_layout != FP4Q_SCALE_LAYOUT_LINEAR || p->col_hadamard ||
      p->precomputed_amax || p->sr_global_rows || p->sr_row_offset || p->sr_matrix_offset ||
      (p->use_precomputed_outer && p->mode != FP4Q_MODE_OUTER_BLOCK) ||
      (p->mode == FP4Q_MODE_OUTER_BLOCK && col && !p->outer_2d && !small_ob && !p->use_precomputed_outer))
    return FP4Q_ERR_UNSUPPORTED;
  if (!offsets || !workspace) return FP4Q_ERR_NULL;
  if (workspace_bytes < s.workspace) return FP4Q_ERR_WORKSPACE;
  if (!aligned(workspace, 16) || !aligned(offsets, 8)) return FP4Q_ERR_ALIGN;
  if (p->M == 0 || p->K == 0) return FP4Q_OK;
  if (!x) return FP4Q_ERR_NULL;
  if (row && (!out->row_codes || !out->row_scales)) return FP4Q_ERR_NULL;
  if (col && (!out->col_codes || !out->col_scales)) return FP4Q_ERR_NULL;
  if ((s.row_outer && !out->row_outer) || (s.col_outer && !out->col_outer) || (s.tile_outer && !out->tile_outer))
    return FP4Q_ERR_NULL;
  if (!vec_aligned(x, p->ld * 2)) return FP4Q_ERR_ALIGN;
  if ((row && !aligned(out->row_codes, 8)) || (col && !aligned(out->col_codes, 8))) return FP4Q_ERR_ALIGN;
  if (!aligned(out->row_outer, 4) || !aligned(out->col_outer, 4) || !aligned(out->tile_outer, 4)) return FP4Q_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  QuantJob j = base_job(p, x, nullptr);
  j.do_row = row;
  j.do_col = col;
  j.row_codes = row ? out->row_codes : nullptr;
  j.row_scales = row ? out->row_scales : nullptr;
  j.col_codes = col ? out->col_codes : nullptr;
  j.col_scales = col ? out->col_scales : nullptr;
  j.row_outer = s.row_outer ? out->row_outer : nullptr;
  j.col_outer = s.col_outer ? out->col_outer : nullptr;
  j.tile_outer = s.tile_outer ? out->tile_outer : nullptr;
  j.ngroups = ngroups;
  j.goff = offsets;
  j.gws = static_cast<GroupWs*>(workspace);
  // every group a whole number of the blocks that span rows
  int align = 1;
  if (col) align = 16;
  if (p->mode == FP4Q_MODE_OUTER_BLOCK && (p->outer_2d || col)) align = p->outer_block_size;
  const bool tw = p->mode == FP4Q_MODE_TENSORWISE;
  if (launch_group_prep(j, align, tw, st) != cudaSuccess) return FP4Q_ERR_CUDA;
  if (p->mode == FP4Q_MODE_NONE) {
    j.s_src = S_ONE;
  } else if (tw) {
    j.s_src = S_TENSORWISE_WS;  // per-group amax from the workspace
  } else if (p->use_precomputed_outer) {
    j.s_src = S_FROM_BUFFER;
  } else if (p->outer_block_size == 16 || p->outer_block_size == 32 || p->outer_block_size == 64) {
    j.s_src = S_IN_TILE;
  } else {
    j.s_src = S_FROM_BUFFER;  // group boundaries are whole outer blocks: the pre-pass of the whole tensor holds
    if (launch_outer_prepass(j, st) != cudaSuccess) return FP4Q_ERR_CUDA;
  }
  cudaError_t e = cudaSuccess;
  if (!launch_ctb(j, st, &e)) return FP4Q_ERR_CUDA;
  return e == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
}

int fp4_qdq(const fp4q_params_t* p, int orient, const void* x, void* y, float* residual, float* outer, void* workspace,
            size_t workspace_bytes, void* stream) {
  if (!p) return FP4Q_ERR_NULL;
  if (orient != (int)FP4Q_OUT_ROW && orient != (int)FP4Q_OUT_COL) return FP4Q_ERR_MODE;
  int rc = check_nvfp4(p, (uint32_t)orient);
  if (rc) return rc;
  rc = check_dtype(p->out_dtype);
  if (rc) return rc;
  if (residual && orient == (int)FP4Q_OUT_COL) return FP4Q_ERR_UNSUPPORTED;
  if (p->col_hadamard) return FP4Q_ERR_UNSUPPORTED;
  fp4q_sizes_t s;
  sizes_for(p, (uint32_t)orient, &s);
  const bool needs_outer = p->mode != FP4Q_MODE_NONE;
  if (needs_outer && !outer) return FP4Q_ERR_NULL;
  if (s.workspace && (!workspace || workspace_bytes < s.workspace)) return FP4Q_ERR_WORKSPACE;
  if (s.workspace && !aligned(workspace, 16)) return FP4Q_ERR_ALIGN;
  const bool empty = p->G == 0 || p->M == 0 || p->K == 0;
  if (!empty && (!x || !y)) return FP4Q_ERR_NULL;
  if (!aligned(x, (uintptr_t)esize(p->in_dtype)) || !aligned(y, (uintptr_t)esize(p->out_dtype))) return FP4Q_ERR_ALIGN;
  if (!aligned(outer, 4) || (residual && !aligned(residual, 16))) return FP4Q_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (empty) {
    if (p->mode == FP4Q_MODE_TENSORWISE && !p->use_precomputed_outer && !p->precomputed_amax)
      return cudaMemsetAsync(outer, 0, sizeof(float), st) == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
    return FP4Q_OK;
  }
  QuantJob j = base_job(p, x, residual);
  j.do_row = orient == (int)FP4Q_OUT_ROW;
  j.do_col = !j.do_row;
  j.qdq_orient = j.do_row ? 1 : 2;
  j.y = y;
  if (p->mode == FP4Q_MODE_TENSORWISE || (p->mode == FP4Q_MODE_OUTER_BLOCK && p->outer_2d)) j.tile_outer = outer;
  else if (p->mode == FP4Q_MODE_OUTER_BLOCK) (j.do_row ? j.row_outer : j.col_outer) = outer;
  rc = prepare_outer(p, j, workspace, st);
  if (rc) return rc;
  return launch_quantizer(j, vec_ok(p, x, residual, y), st);
}

int fp4_dequantize(const fp4q_params_t* p, int orient, const uint8_t* codes, const uint8_t* scales, const float* outer,
                   void* y, void* stream) {
  if (!p) return FP4Q_ERR_NULL;
  if (orient != (int)FP4Q_OUT_ROW && orient != (int)FP4Q_OUT_COL) return FP4Q_ERR_MODE;
  int rc = check_nvfp4(p, (uint32_t)orient);
  if (rc) return rc;
  rc = check_dtype(p->out_dtype);
  if (rc) return rc;
  if (p->use_precomputed_outer) return FP4Q_ERR_MODE;
  const bool empty = p->G == 0 || p->M == 0 || p->K == 0;
  if (empty) return FP4Q_OK;
  if (!codes || !scales || !y) return FP4Q_ERR_NULL;
  if (p->mode != FP4Q_MODE_NONE && !outer) return FP4Q_ERR_NULL;
  if (!aligned(codes, 8) || !aligned(outer, 4) || !aligned(y, (uintptr_t)esize(p->out_dtype))) return FP4Q_ERR_ALIGN;
  DequantJob j{};
  j.codes = codes;
  j.scales = scales;
  j.outer = outer;
  j.y = y;
  j.G = p->G;
  j.M = p->M;
  j.K = p->K;
  j.col = orient == (int)FP4Q_OUT_COL;
  j.R = j.col ? p->K : p->M;
  j.C = j.col ? p->M : p->K;
  j.mode = p->mode;
  j.ob = p->outer_block_size;
  j.outer_2d = p->outer_2d;
  j.ue5m3 = p->scale_format == FP4Q_SCALE_UE5M3;
  j.out_bf16 = p->out_dtype == FP4Q_BF16;
  j.sl = make_scale_layout(p->scale_layout == FP4Q_SCALE_LAYOUT_MMA, j.R, j.C / 16);
  return launch_dequant(j, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
}

int mxfp4_fake_quantize(const fp4q_params_t* p, const void* x, void* y, void* stream) {
  if (!p) return FP4Q_ERR_NULL;
  if (p->struct_size != sizeof(fp4q_params_t)) return FP4Q_ERR_ABI;
  int rc = check_dtype(p->in_dtype);
  if (rc) return rc;
  rc = check_dtype(p->out_dtype);
  if (rc) return rc;
  if (!mx_knobs_default(p)) return FP4Q_ERR_MODE;
  if (p->rounding != FP4Q_RNE) return FP4Q_ERR_UNSUPPORTED;
  if (p->G < 0 || p->M < 0 || p->K < 0 || p->ld < p->K || p->K % 32) return FP4Q_ERR_SHAPE;
  if (p->G == 0 || p->M == 0 || p->K == 0) return FP4Q_OK;
  if (!x || !y) return FP4Q_ERR_NULL;
  if (!aligned(x, (uintptr_t)esize(p->in_dtype)) || !aligned(y, (uintptr_t)esize(p->out_dtype))) return FP4Q_ERR_ALIGN;
  MxJob j{};
  j.x = x;
  j.ld = p->ld;
  j.in_bf16 = p->in_dtype == FP4Q_BF16;
  j.out_bf16 = p->out_dtype == FP4Q_BF16;
  j.G = p->G;
  j.M = p->M;
  j.K = p->K;
  j.y = y;
  return launch_mxfp4(j, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
}

int fp4_tensor_amax(const fp4q_params_t* p, const void* x, const float* residual, float* amax, void* stream) {
  if (!p || !amax) return FP4Q_ERR_NULL;
  if (p->struct_size != sizeof(fp4q_params_t)) return FP4Q_ERR_ABI;
  const int rc = check_dtype(p->in_dtype);
  if (rc) return rc;
  if (p->G < 0 || p->M < 0 || p->K < 0 || p->ld < p->K) return FP4Q_ERR_SHAPE;
  if (!aligned(amax, 4)) return FP4Q_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p->G == 0 || p->M == 0 || p->K == 0)
    return cudaMemsetAsync(amax, 0, sizeof(float), st) == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
  if (!x) return FP4Q_ERR_NULL;
  if (!aligned(x, (uintptr_t)esize(p->in_dtype)) || (residual && !aligned(residual, 4))) return FP4Q_ERR_ALIGN;
  QuantJob j = base_job(p, x, const_cast<float*>(residual));
  // the maximum of non-negative binary32 values is the maximum of their bits
  return launch_tensor_amax(j, reinterpret_cast<uint32_t*>(amax), st) == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
}

int mxfp4_project_mxfp8(const fp4q_params_t* p, const void* x, void* y, uint8_t* row_codes, uint8_t* row_scales,
                        uint8_t* col_codes, uint8_t* col_scales, void* stream) {
  if (!p) return FP4Q_ERR_NULL;
  if (p->struct_size != sizeof(fp4q_params_t)) return FP4Q_ERR_ABI;
  int rc = check_dtype(p->in_dtype);
  if (rc) return rc;
  rc = check_dtype(p->out_dtype);
  if (rc) return rc;
  if (!mx_knobs_default(p)) return FP4Q_ERR_MODE;
  if (p->rounding != FP4Q_RNE) return FP4Q_ERR_UNSUPPORTED;
  const uint32_t mask = p->out_mask;
  if (mask & ~3u) return FP4Q_ERR_MODE;
  const bool row = mask & FP4Q_OUT_ROW, col = mask & FP4Q_OUT_COL;
  if (p->G < 0 || p->M < 0 || p->K < 0 || p->ld < p->K || p->K % 32) return FP4Q_ERR_SHAPE;
  if (col && p->M % 32) return FP4Q_ERR_SHAPE;
  if (p->G == 0 || p->M == 0 || p->K == 0) return FP4Q_OK;
  if (!x) return FP4Q_ERR_NULL;
  if ((row && (!row_codes || !row_scales)) || (col && (!col_codes || !col_scales))) return FP4Q_ERR_NULL;
  if (!vec_aligned(x, p->ld * esize(p->in_dtype)) || (y && !aligned(y, 16)) || (row && !aligned(row_codes, 16)) ||
      (col && !aligned(col_codes, 16)))
    return FP4Q_ERR_ALIGN;
  QuantJob j{};
  j.x = x;
  j.ld = p->ld;
  j.in_bf16 = p->in_dtype == FP4Q_BF16;
  j.out_bf16 = p->out_dtype == FP4Q_BF16;
  j.G = p->G;
  j.M = p->M;
  j.K = p->K;
  j.y = y;
  j.row_codes = row ? row_codes : nullptr;
  j.row_scales = row ? row_scales : nullptr;
  j.col_codes = col ? col_codes : nullptr;
  j.col_scales = col ? col_scales : nullptr;
  return launch_mxfp8(j, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
}

const char* fp4q_status_string(int status) {
  switch (status) {
    case FP4Q_OK: return "FP4Q_OK";
    case FP4Q_ERR_NULL: return "FP4Q_ERR_NULL: a required pointer is NULL";
    case FP4Q_ERR_DTYPE: return "FP4Q_ERR_DTYPE: unsupported dtype (bf16 or fp32 only)";
    case FP4Q_ERR_SHAPE: return "FP4Q_ERR_SHAPE: a size or divisibility rule is violated";
    case FP4Q_ERR_MODE: return "FP4Q_ERR_MODE: inconsistent mode or knob combination";
    case FP4Q_ERR_UNSUPPORTED: return "FP4Q_ERR_UNSUPPORTED: combination not defined by the method";
    case FP4Q_ERR_WORKSPACE: return "FP4Q_ERR_WORKSPACE: workspace missing or too small";
    case FP4Q_ERR_CUDA: return "FP4Q_ERR_CUDA: a CUDA launch failed";
    case FP4Q_ERR_ABI: return "FP4Q_ERR_ABI: parameter struct size mismatch";
    case FP4Q_ERR_ALIGN: return "FP4Q_ERR_ALIGN: a buffer is not naturally aligned";
    case FP4Q_ERR_TIMEOUT: return "FP4Q_ERR_TIMEOUT: a kernel's bounded wait for its tile copy ran out";
    default: return "unknown fp4q status";
  }
}

int fp4q_abi_version(void) { return FP4Q_ABI_VERSION; }

int fp4q_device_status(int clear, void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FP4Q_ERR_CUDA;
  cudaError_t (*const readers[])(uint32_t*, bool) = {ctb_timeout_flag, ctb_grouped_timeout_flag, ctb_rht_timeout_flag,
                                                      ctl_timeout_flag, row_timeout_flag, ct_timeout_flag,
                                                      mxfp8_timeout_flag};
  uint32_t any = 0;
  for (auto rd : readers) {
    uint32_t v = 0;
    if (rd(&v, clear != 0) != cudaSuccess) return FP4Q_ERR_CUDA;
    any |= v;
  }
  return any ? FP4Q_ERR_TIMEOUT : FP4Q_OK;
}

int fp4q_set_device_timeout_flag(void) {
  return set_ctb_timeout_flag() == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
}

}  // extern "C"
