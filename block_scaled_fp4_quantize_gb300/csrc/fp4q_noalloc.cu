// fp4q_noalloc.cu -- fp4_quantize for callers that cannot allocate device memory.
//
// Tensorwise quantization needs a few bytes of device scratch for the
// cross-CTA amax; fp4_quantize takes it from the caller.  This entry point
// takes it instead from a file-scope static device array of
// FP4Q_NOALLOC_SCRATCH_BYTES bytes, so the caller passes only its inputs and
// outputs.  Each device that loads the library keeps the array until the
// process exits.
//
// Sharing: every call on a device uses the same array and leaves its last
// contents there.  The quantizer clears the part that must start at zero
// (the amax accumulator) at the start of every call, but calls whose work
// overlaps on the GPU (different streams, or different host threads without
// ordering) race on the array and may produce wrong scales.
#include <mutex>

#include <cuda_runtime.h>

#include "fp4q.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[FP4Q_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_noalloc_scratch on the current device.  Looked up once
// per device with that device current (the symbol's host-side name is only a
// stand-in and must never be handed to a kernel).  The address belongs to
// the device's primary context, the one the CUDA runtime (and torch) uses;
// after cudaDeviceReset, or from another context on the same device, it is
// not valid.
int scratch_address(void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP4Q_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return FP4Q_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return FP4Q_OK;
}

}  // namespace

extern "C" int fp4_quantize_noalloc(const fp4q_params_t* p, const void* x, const fp4q_outputs_t* out,
                                    float* residual, void* stream) {
  if (!p || !out) return FP4Q_ERR_NULL;
  fp4q_sizes_t s;
  int rc = fp4q_query_sizes(p, &s);
  if (rc != FP4Q_OK) return rc;
  // a precomputed tensorwise amax travels in the caller's workspace, which
  // this entry point does not take
  if (p->precomputed_amax) return FP4Q_ERR_UNSUPPORTED;
  if (s.workspace > (size_t)FP4Q_NOALLOC_SCRATCH_BYTES) return FP4Q_ERR_WORKSPACE;
  void* ws = nullptr;
  if (s.workspace > 0) {
    rc = scratch_address(&ws);
    if (rc != FP4Q_OK) return rc;
  }
  return fp4_quantize(p, x, out, residual, ws, s.workspace > 0 ? (size_t)FP4Q_NOALLOC_SCRATCH_BYTES : 0, stream);
}
