// Exhaustive check of the two hardware conversions every fast kernel takes
// its codes from, against the oracle's encoders (test infrastructure: built
// and run by tests/test_gpu_device_numerics.py, linked with the oracle's
// shared library):
//
//   - e2m1x2_rne (cvt.rn.satfinite.e2m1x2.f32): the E2M1 code of every
//     finite binary32 t >= 0 against orc_e2m1_rne (nearest of the eight grid
//     points, ties to the even code, saturation at 6), and on the device
//     code(-t) == code(t) | 8 (the sign bit kept, -0 included);
//   - enc_e4m3_hw (cvt.rn.satfinite.e4m3x2.f32): the E4M3 scale code of
//     every finite binary32 v >= 0 against orc_scale_encode in the E4M3
//     format (nearest, ties to the even code, saturation at 448).
//
// Prints "checked N mismatches M" (N = both encoders over all 0x7F800000
// patterns) and the first mismatches; exits 0 when the run completed.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <thread>
#include <vector>

#include <cuda_runtime.h>

#include "fp4q_device.cuh"

extern "C" uint8_t orc_e2m1_rne(double t);
extern "C" uint8_t orc_scale_encode(int fmt, float v);

constexpr uint32_t kN = 0x7F800000u;  // every finite binary32 >= 0 (bit patterns 0 .. 0x7F7FFFFF)

__global__ void encode_all(uint8_t* e2, uint8_t* e4, unsigned long long* asym) {
  for (uint32_t b = blockIdx.x * blockDim.x + threadIdx.x; b < kN; b += gridDim.x * blockDim.x) {
    const float t = fp4q::bitsf(b);
    const uint32_t c = fp4q::e2m1x2_rne(t, 0.0f) & 0xFu;
    const uint32_t cn = fp4q::e2m1x2_rne(fp4q::bitsf(b | 0x80000000u), 0.0f) & 0xFu;
    if (cn != (c | 8u)) atomicAdd(asym, 1ull);
    e2[b] = (uint8_t)c;
    e4[b] = (uint8_t)fp4q::enc_e4m3_hw(t);
  }
}

int main() {
  uint8_t *d2 = nullptr, *d4 = nullptr;
  unsigned long long* dasym = nullptr;
  if (cudaMalloc(&d2, kN) != cudaSuccess || cudaMalloc(&d4, kN) != cudaSuccess ||
      cudaMalloc(&dasym, sizeof(*dasym)) != cudaSuccess) {
    std::printf("cuda alloc failed\n");
    return 2;
  }
  cudaMemset(dasym, 0, sizeof(*dasym));
  encode_all<<<152 * 8, 256>>>(d2, d4, dasym);
  if (cudaDeviceSynchronize() != cudaSuccess) {
    std::printf("kernel failed\n");
    return 2;
  }
  std::vector<uint8_t> e2(kN), e4(kN);
  unsigned long long asym = 0;
  if (cudaMemcpy(e2.data(), d2, kN, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(e4.data(), d4, kN, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(&asym, dasym, sizeof(asym), cudaMemcpyDeviceToHost) != cudaSuccess) {
    std::printf("copy failed\n");
    return 2;
  }
  // the oracle over the same patterns, in slices across the host's cores
  const unsigned nt = std::thread::hardware_concurrency() ? std::thread::hardware_concurrency() : 4;
  std::vector<unsigned long long> bad2(nt, 0), bad4(nt, 0);
  std::vector<uint32_t> first2(nt, 0xFFFFFFFFu), first4(nt, 0xFFFFFFFFu);
  std::vector<std::thread> pool;
  for (unsigned k = 0; k < nt; ++k) {
    pool.emplace_back([&, k] {
      const uint32_t lo = (uint32_t)((uint64_t)kN * k / nt), hi = (uint32_t)((uint64_t)kN * (k + 1) / nt);
      for (uint32_t b = lo; b < hi; ++b) {
        float v;
        std::memcpy(&v, &b, 4);
        if (e2[b] != orc_e2m1_rne((double)v)) {
          if (bad2[k]++ == 0) first2[k] = b;
        }
        if (e4[b] != orc_scale_encode(0, v)) {
          if (bad4[k]++ == 0) first4[k] = b;
        }
      }
    });
  }
  for (auto& th : pool) th.join();
  unsigned long long m2 = 0, m4 = 0;
  for (unsigned k = 0; k < nt; ++k) {
    m2 += bad2[k];
    m4 += bad4[k];
  }
  std::printf("checked %llu mismatches %llu\n", 2ull * kN, m2 + m4 + asym);
  std::printf("e2m1 mismatches %llu, e2m1 sign asymmetries %llu, e4m3 mismatches %llu\n", m2, asym, m4);
  for (unsigned k = 0; k < nt; ++k) {
    if (first2[k] != 0xFFFFFFFFu) {
      float v;
      std::memcpy(&v, &first2[k], 4);
      std::printf("e2m1 t=%08x device=%x oracle=%x\n", first2[k], e2[first2[k]], orc_e2m1_rne((double)v));
    }
    if (first4[k] != 0xFFFFFFFFu) {
      float v;
      std::memcpy(&v, &first4[k], 4);
      std::printf("e4m3 v=%08x device=%02x oracle=%02x\n", first4[k], e4[first4[k]], orc_scale_encode(0, v));
    }
  }
  return 0;
}
