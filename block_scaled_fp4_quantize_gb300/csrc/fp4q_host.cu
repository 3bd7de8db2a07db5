// fp4q_host.cu -- host-buffer entry point: MXFP4 fake-quantize of a tensor in
// host memory, streamed through a caller-provided device staging area.
//
// The rows are cut into chunks.  Chunk c uses staging slot c mod 2 (an input
// and an output buffer per slot) and three engines run side by side:
//   copy stream A   host -> slot input            (waits: slot's kernel c-2)
//   the call stream kernel: slot input -> output  (waits: copy A of c, copy B of c-2)
//   copy stream B   slot output -> host           (waits: kernel c)
// so the host-to-device copy of chunk c+1, the kernel of chunk c and the
// device-to-host copy of chunk c-1 overlap.  The two copy streams are created
// once per device and reused; the call's completion is joined into the
// caller's stream.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fp4q.h"
#include "fp4q_internal.h"

namespace fp4q {
namespace {

struct HostPipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, in_ready[2] = {}, kern_done[2] = {}, out_done[2] = {};
};

std::mutex g_pipe_mu;
HostPipe g_pipes[128];

cudaError_t pipe_for_device(HostPipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  HostPipe& p = g_pipes[dev];
  if (!p.ready) {
    if ((e = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming)) != cudaSuccess) return e;
    for (int s = 0; s < 2; ++s) {
      if ((e = cudaEventCreateWithFlags(&p.in_ready[s], cudaEventDisableTiming)) != cudaSuccess) return e;
      if ((e = cudaEventCreateWithFlags(&p.kern_done[s], cudaEventDisableTiming)) != cudaSuccess) return e;
      if ((e = cudaEventCreateWithFlags(&p.out_done[s], cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    p.ready = true;
  }
  *out = &p;
  return cudaSuccess;
}

}  // namespace
}  // namespace fp4q

using namespace fp4q;

extern "C" int mxfp4_fake_quantize_host(const fp4q_params_t* p, const void* x, void* y, void* ws, size_t ws_bytes,
                                        void* stream) {
  if (!p) return FP4Q_ERR_NULL;
  if (p->struct_size != sizeof(fp4q_params_t)) return FP4Q_ERR_ABI;
  if ((p->in_dtype != FP4Q_BF16 && p->in_dtype != FP4Q_FP32) || (p->out_dtype != FP4Q_BF16 && p->out_dtype != FP4Q_FP32))
    return FP4Q_ERR_DTYPE;
  if (p->mode != FP4Q_MODE_NONE || p->outer_block_size != 0 || p->outer_2d != 0 || p->inner_2d != 0 ||
      p->scale_format != FP4Q_SCALE_E4M3 || p->use_precomputed_outer != 0 || p->scale_layout != 0 ||
      p->col_hadamard != 0 || p->precomputed_amax != 0)
    return FP4Q_ERR_MODE;
  if (p->rounding != FP4Q_RNE) return FP4Q_ERR_UNSUPPORTED;
  if (p->G < 0 || p->M < 0 || p->K < 0 || p->ld < p->K || p->K % 32) return FP4Q_ERR_SHAPE;
  const int64_t rows = p->G * p->M;
  if (rows == 0 || p->K == 0) return FP4Q_OK;
  if (!x || !y || !ws) return FP4Q_ERR_NULL;
  const int64_t ein = p->in_dtype == FP4Q_BF16 ? 2 : 4, eout = p->out_dtype == FP4Q_BF16 ? 2 : 4;
  if (reinterpret_cast<uintptr_t>(x) % (uintptr_t)ein || reinterpret_cast<uintptr_t>(y) % (uintptr_t)eout ||
      reinterpret_cast<uintptr_t>(ws) % 256u)
    return FP4Q_ERR_ALIGN;
  // staging: 2 slots x (input rows + output rows), each buffer 256-byte aligned
  const int64_t in_row = p->K * ein, out_row = p->K * eout;
  auto round256 = [](int64_t v) { return (v + 255) & ~int64_t(255); };
  // the largest chunk (whole rows) whose two input and two output buffers fit
  int64_t chunk = (int64_t)ws_bytes / (2 * (in_row + out_row));
  while (chunk > 1 && 2 * (round256(chunk * in_row) + round256(chunk * out_row)) > (int64_t)ws_bytes) --chunk;
  const int64_t cap = (int64_t)(FP4Q_HOST_CHUNK_BYTES / in_row);
  if (chunk > cap) chunk = cap;
  if (chunk < 1) chunk = 1;
  if (2 * (round256(chunk * in_row) + round256(chunk * out_row)) > (int64_t)ws_bytes) return FP4Q_ERR_WORKSPACE;
  unsigned char* base = static_cast<unsigned char*>(ws);
  unsigned char* in_buf[2] = {base, base + round256(chunk * in_row)};
  unsigned char* out_buf[2] = {base + 2 * round256(chunk * in_row),
                               base + 2 * round256(chunk * in_row) + round256(chunk * out_row)};

  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe* hp = nullptr;
  if (pipe_for_device(&hp) != cudaSuccess) return FP4Q_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  bool ok = cudaEventRecord(hp->start, st) == cudaSuccess && cudaStreamWaitEvent(hp->h2d, hp->start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(hp->d2h, hp->start, 0) == cudaSuccess;
  const int64_t nchunks = (rows + chunk - 1) / chunk;
  for (int64_t c = 0; ok && c < nchunks; ++c) {
    const int s = (int)(c & 1);
    const int64_t r0 = c * chunk, nr = (rows - r0 < chunk) ? rows - r0 : chunk;
    // host rows r0 .. r0 + nr of the [G * M, K] view (matrices back to back, row stride ld)
    const unsigned char* xs = static_cast<const unsigned char*>(x) + r0 * p->ld * ein;
    unsigned char* ys = static_cast<unsigned char*>(y) + r0 * out_row;
    if (c >= 2) ok = ok && cudaStreamWaitEvent(hp->h2d, hp->kern_done[s], 0) == cudaSuccess;
    ok = ok && cudaMemcpy2DAsync(in_buf[s], (size_t)in_row, xs, (size_t)(p->ld * ein), (size_t)in_row, (size_t)nr,
                                 cudaMemcpyHostToDevice, hp->h2d) == cudaSuccess;
    ok = ok && cudaEventRecord(hp->in_ready[s], hp->h2d) == cudaSuccess;
    ok = ok && cudaStreamWaitEvent(st, hp->in_ready[s], 0) == cudaSuccess;
    if (c >= 2) ok = ok && cudaStreamWaitEvent(st, hp->out_done[s], 0) == cudaSuccess;
    if (ok) {
      MxJob j{};
      j.x = in_buf[s];
      j.ld = p->K;
      j.in_bf16 = p->in_dtype == FP4Q_BF16;
      j.out_bf16 = p->out_dtype == FP4Q_BF16;
      j.G = 1;
      j.M = nr;
      j.K = p->K;
      j.y = out_buf[s];
      ok = launch_mxfp4(j, st) == cudaSuccess;
    }
    ok = ok && cudaEventRecord(hp->kern_done[s], st) == cudaSuccess;
    ok = ok && cudaStreamWaitEvent(hp->d2h, hp->kern_done[s], 0) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(ys, out_buf[s], (size_t)(nr * out_row), cudaMemcpyDeviceToHost, hp->d2h) == cudaSuccess;
    ok = ok && cudaEventRecord(hp->out_done[s], hp->d2h) == cudaSuccess;
  }
  // the call is complete on `stream` once both slots' last copies are
  for (int s = 0; ok && s < 2 && s < nchunks; ++s) ok = cudaStreamWaitEvent(st, hp->out_done[s], 0) == cudaSuccess;
  return ok ? FP4Q_OK : FP4Q_ERR_CUDA;
}
