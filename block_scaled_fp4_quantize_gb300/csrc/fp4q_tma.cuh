// fp4q_tma.cuh -- tile walk and tensor-memory-access (TMA) copies shared by
// the tile kernels: a grid-stride walk over TM x 64 tiles of a [G, M, K]
// tensor, mbarrier-completed 3-D tensor copies with bounded waits, and the
// driver entry point that encodes tensor maps.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "fp4q_internal.h"

namespace fp4q {
namespace {

struct TilePos {
  int64_t g, m0, k0;
};

// Grid-stride walk over tiles without per-tile divisions (tile counts fit
// 32 bits: 2^31 tiles would be 2^44 elements).
struct TileIter {
  int tiles_k, tiles_m, ntiles, idx, tk, tm, g, dk, dm, dg;
  template <int TM>
  __device__ __forceinline__ void init(const QuantJob& j) {
    init_n((int)((j.K + 63) / 64), (int)((j.M + TM - 1) / TM), (int)j.G);
  }
  // a walk over G x tiles_m x tiles_k tiles (tk fastest)
  __device__ __forceinline__ void init_n(int tiles_k_, int tiles_m_, int g_count) {
    tiles_k = tiles_k_ > 0 ? tiles_k_ : 1;
    tiles_m = tiles_m_ > 0 ? tiles_m_ : 1;
    ntiles = (tiles_k_ > 0 && tiles_m_ > 0) ? g_count * tiles_m * tiles_k : 0;
    idx = (int)blockIdx.x;
    tk = idx % tiles_k;
    tm = (idx / tiles_k) % tiles_m;
    g = idx / (tiles_k * tiles_m);
    const int step = (int)gridDim.x;
    dk = step % tiles_k;
    dm = (step / tiles_k) % tiles_m;
    dg = step / (tiles_k * tiles_m);
  }
  __device__ __forceinline__ bool valid() const { return idx < ntiles; }
  __device__ __forceinline__ void next() {
    idx += (int)gridDim.x;
    tk += dk;
    int c = 0;
    if (tk >= tiles_k) { tk -= tiles_k; c = 1; }
    tm += dm + c;
    c = 0;
    if (tm >= tiles_m) { tm -= tiles_m; c = 1; }
    g += dg + c;
  }
  template <int TM>
  __device__ __forceinline__ TilePos pos() const {
    return TilePos{(int64_t)g, (int64_t)tm * TM, (int64_t)tk * 64};
  }
  // position of tile `i` (the copy issuer looks ahead of the walk)
  template <int TM>
  __device__ __forceinline__ TilePos pos_of(int i) const {
    const int q = i / tiles_k;
    return TilePos{(int64_t)(q / tiles_m), (int64_t)(q % tiles_m) * TM, (int64_t)(i - q * tiles_k) * 64};
  }
};

// Position in the grouped walk: group e owns the 128-row tiles
// tprefix[e] .. tprefix[e + 1] - 1 of the walk; a cursor only moves forward
// (a CTA's tile indices grow), so finding the group of a tile is amortized.
struct GroupCursor {
  int64_t e = -1;
  uint32_t lo = 0, hi = 0;
  __device__ __forceinline__ void seek(const uint32_t* tp, uint32_t q) {
    while (hi <= q) {
      ++e;
      lo = hi;
      hi = tp[e + 1];
    }
  }
};

// ---- programmatic dependent launch ----
// A kernel launched with programmatic stream serialization may start while
// the previous grid on the stream is still finishing: it waits for that
// grid's completion (its writes then visible) before touching global
// memory, then lets the next grid be scheduled.  Without the launch
// attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_wait_then_release() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
}

// Launch with programmatic stream serialization.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ---- tensor-memory-access (TMA) tile loads, completion on an mbarrier ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
// The dynamic shared-memory base rounded up to a 1024-byte boundary.  The
// result is an offset from `base`, not an integer cast back to a pointer, so
// the compiler still knows it points to shared memory: accesses through it
// compile to 32-bit shared loads and stores rather than 64-bit generic ones.
__device__ __forceinline__ unsigned char* smem_align1024(unsigned char* base) {
  return base + ((0u - smem_u32(base)) & 1023u);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar) {
  asm volatile("mbarrier.init.shared.b64 [%0], 1;" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// Wait for phase `parity` of the barrier, giving up after `limit` polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// One 3-D tensor copy (K, M, G) of a box into shared memory.
__device__ __forceinline__ void tma_load3(void* dst, const CUtensorMap* map, int k, int m, int g, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_u32(dst)), "l"(map), "r"(k), "r"(m), "r"(g), "r"(smem_u32(bar))
      : "memory");
}

// ---- tensor-memory-access (TMA) tile stores from shared memory ----
// Make this thread's shared-memory writes visible to the tensor copies
// (issued after a CTA barrier by one thread).
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// One 3-D tensor copy of a box from shared memory to global memory; the
// unit clips rows and columns outside the tensor.
__device__ __forceinline__ void tma_store3(const CUtensorMap* map, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
               ::"l"(map), "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
// One 2-D tensor copy of a box from shared memory to global memory.
__device__ __forceinline__ void tma_store2(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
               ::"l"(map), "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Every store group issued by this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Every store group issued by this thread is complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Tensor map of the bf16 input [G][M][K] (row stride ld) for tiles of
// `box_m` rows x 64 columns with the 128-byte swizzle.
bool make_bf16_tile_map(const QuantJob& j, CUtensorMap* map, int box_m) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)j.K, (cuuint64_t)j.M, (cuuint64_t)j.G};
  const cuuint64_t strides[2] = {(cuuint64_t)j.ld * 2, (cuuint64_t)j.M * (cuuint64_t)j.ld * 2};
  const cuuint32_t box[3] = {64u, (cuuint32_t)box_m, 1u};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(j.x), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of the columnwise codes [G][K][M / 2] bytes for the tile
// store (box: 64 columns x 64 bytes, 64-byte swizzle: the inner extent of
// the box equals the swizzle span).  Needs 16-byte aligned rows (M a
// multiple of 32) and a 16-byte aligned base; false when the codes leave by
// the thread copy-out instead.
bool make_col_map(const QuantJob& j, CUtensorMap* map) {
  if (j.ngroups > 0 || !j.do_col || j.M % 32 || (reinterpret_cast<uintptr_t>(j.col_codes) & 15u)) return false;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)(j.M / 2), (cuuint64_t)j.K, (cuuint64_t)j.G};
  const cuuint64_t strides[2] = {(cuuint64_t)(j.M / 2), (cuuint64_t)j.K * (cuuint64_t)(j.M / 2)};
  const cuuint32_t box[3] = {64u, 64u, 1u};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, j.col_codes, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace fp4q
