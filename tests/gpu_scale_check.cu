// Exhaustive check of enc_ue5m3 against the general scale encoder enc_scale
// with the UE5M3 format, for every finite binary32 v >= 0 (test
// infrastructure: built and run by tests/test_gpu_device_numerics.py).
//
// Prints "checked N mismatches M" and, for the first mismatches, the input
// bits with both codes; exits 0 when the run completed (whatever M is).
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>

#include "fp4q_device.cuh"

__global__ void check(uint32_t hi, unsigned long long* count, uint32_t* first) {
  const fp4q::ScaleFmt f = fp4q::scale_fmt(1);
  for (uint32_t b = blockIdx.x * blockDim.x + threadIdx.x; b <= hi; b += gridDim.x * blockDim.x) {
    const float v = fp4q::bitsf(b);
    const uint32_t a = fp4q::enc_ue5m3(v), r = fp4q::enc_scale(v, f);
    if (a != r) {
      const unsigned long long k = atomicAdd(count, 1ull);
      if (k < 8) {
        first[3 * k] = b;
        first[3 * k + 1] = a;
        first[3 * k + 2] = r;
      }
    }
  }
}

int main() {
  const uint32_t hi = 0x7F7FFFFFu;  // largest finite binary32
  unsigned long long* count = nullptr;
  uint32_t* first = nullptr;
  if (cudaMalloc(&count, sizeof(*count)) != cudaSuccess || cudaMalloc(&first, 24 * sizeof(uint32_t)) != cudaSuccess) {
    std::printf("cuda alloc failed\n");
    return 2;
  }
  cudaMemset(count, 0, sizeof(*count));
  cudaMemset(first, 0, 24 * sizeof(uint32_t));
  check<<<152 * 8, 256>>>(hi, count, first);
  if (cudaDeviceSynchronize() != cudaSuccess) {
    std::printf("kernel failed\n");
    return 2;
  }
  unsigned long long c = 0;
  uint32_t fr[24];
  cudaMemcpy(&c, count, sizeof(c), cudaMemcpyDeviceToHost);
  cudaMemcpy(fr, first, sizeof(fr), cudaMemcpyDeviceToHost);
  std::printf("checked %llu mismatches %llu\n", (unsigned long long)hi + 1ull, c);
  for (unsigned long long k = 0; k < c && k < 8; ++k)
    std::printf("v=%08x enc_ue5m3=%02x enc_scale=%02x\n", fr[3 * k], fr[3 * k + 1], fr[3 * k + 2]);
  return 0;
}
