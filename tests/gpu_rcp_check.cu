// Exhaustive check of rcp_markstein against the IEEE reciprocal rcp.rn.f32
// for every binary32 s with 2^-125 <= s <= 2^125, both signs (test
// infrastructure: built and run by tests/test_gpu_device_numerics.py).
//
// Prints "checked N mismatches M" and, for the first mismatches, the input
// bits with both results; exits 0 when the run completed (whatever M is).
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>

#include "fp4q_device.cuh"

__global__ void check(uint32_t lo, uint32_t hi, unsigned long long* count, uint32_t* first) {
  const uint32_t n = hi - lo + 1u;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
#pragma unroll
    for (int sgn = 0; sgn < 2; ++sgn) {
      const float s = fp4q::bitsf((lo + i) | (sgn ? 0x80000000u : 0u));
      const uint32_t a = fp4q::fbits(fp4q::rcp_markstein(s)), b = fp4q::fbits(fp4q::ieee_rcp(s));
      if (a != b) {
        const unsigned long long k = atomicAdd(count, 1ull);
        if (k < 8) {
          first[3 * k] = fp4q::fbits(s);
          first[3 * k + 1] = a;
          first[3 * k + 2] = b;
        }
      }
    }
  }
}

int main() {
  const uint32_t lo = 0x01000000u, hi = 0x7E000000u;  // 2^-125 .. 2^125
  unsigned long long* count = nullptr;
  uint32_t* first = nullptr;
  if (cudaMalloc(&count, sizeof(*count)) != cudaSuccess || cudaMalloc(&first, 24 * sizeof(uint32_t)) != cudaSuccess) {
    std::printf("cuda alloc failed\n");
    return 2;
  }
  cudaMemset(count, 0, sizeof(*count));
  cudaMemset(first, 0, 24 * sizeof(uint32_t));
  check<<<152 * 8, 256>>>(lo, hi, count, first);
  if (cudaDeviceSynchronize() != cudaSuccess) {
    std::printf("kernel failed\n");
    return 2;
  }
  unsigned long long c = 0;
  uint32_t f[24];
  cudaMemcpy(&c, count, sizeof(c), cudaMemcpyDeviceToHost);
  cudaMemcpy(f, first, sizeof(f), cudaMemcpyDeviceToHost);
  std::printf("checked %llu mismatches %llu\n", 2ull * (hi - lo + 1u), c);
  for (unsigned long long k = 0; k < c && k < 8; ++k)
    std::printf("s=%08x markstein=%08x rcp.rn=%08x\n", f[3 * k], f[3 * k + 1], f[3 * k + 2]);
  return 0;
}
