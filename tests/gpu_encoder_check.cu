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
//     format (nearest, ties to the even code, saturation at 448);
//   - e2m1_sr (the branch-free stochastic rounding): the E2M1 code of every
//     binary32 t in [0, 8] with the random word w = hash(t) against
//     orc_e2m1_sr, and code(-t, w) == code(t, w) | 8 on the device;
//   - philox4x32_10 (the random words of stochastic rounding): 2^26
//     counters and keys that vary in every word, all four output words,
//     against orc_philox4x32_10.
//
// Prints "checked N mismatches M" (N = 2 x 0x7F800000 + 0x41000001 codes +
// 2^26 Philox blocks) and the first mismatches; exits 0 when the run
// completed.
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
extern "C" uint8_t orc_e2m1_sr(double t, uint32_t w);
extern "C" void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]);

constexpr uint32_t kN = 0x7F800000u;  // every finite binary32 >= 0 (bit patterns 0 .. 0x7F7FFFFF)
constexpr uint32_t kS = 0x41000001u;  // binary32 0 .. 8

constexpr uint32_t kP = 1u << 26;     // Philox blocks

// the random word of pattern b (a multiplicative hash)
__host__ __device__ inline uint32_t word_of(uint32_t b) { return (b * 2654435761u) ^ 0x5BD1E995u; }
// Philox counter and key of block i: every word varies
__host__ __device__ inline void philox_in(uint32_t i, uint32_t (&c)[4], uint32_t (&k)[2]) {
  c[0] = i * 0x9E3779B9u;
  c[1] = ~i;
  c[2] = i * 0x85EBCA6Bu + 7u;
  c[3] = i & 3u;
  k[0] = word_of(i);
  k[1] = i ^ 0xA5A5A5A5u;
}

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

__global__ void round_sr_all(uint8_t* sr, unsigned long long* asym) {
  for (uint32_t b = blockIdx.x * blockDim.x + threadIdx.x; b < kS; b += gridDim.x * blockDim.x) {
    const uint32_t w = word_of(b);
    const uint32_t c = fp4q::e2m1_sr(fp4q::bitsf(b), w);
    if (fp4q::e2m1_sr(fp4q::bitsf(b | 0x80000000u), w) != (c | 8u)) atomicAdd(asym, 1ull);
    sr[b] = (uint8_t)c;
  }
}

__global__ void philox_all(uint4* out) {
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < kP; i += gridDim.x * blockDim.x) {
    uint32_t c[4], k[2];
    philox_in(i, c, k);
    out[i] = fp4q::philox4x32_10(make_uint4(c[0], c[1], c[2], c[3]), k[0], k[1]);
  }
}

int main() {
  uint8_t *d2 = nullptr, *d4 = nullptr, *ds = nullptr;
  uint4* dp = nullptr;
  unsigned long long* dasym = nullptr;
  if (cudaMalloc(&d2, kN) != cudaSuccess || cudaMalloc(&d4, kN) != cudaSuccess || cudaMalloc(&ds, kS) != cudaSuccess ||
      cudaMalloc(&dp, (size_t)kP * sizeof(uint4)) != cudaSuccess ||
      cudaMalloc(&dasym, sizeof(*dasym)) != cudaSuccess) {
    std::printf("cuda alloc failed\n");
    return 2;
  }
  cudaMemset(dasym, 0, sizeof(*dasym));
  encode_all<<<152 * 8, 256>>>(d2, d4, dasym);
  round_sr_all<<<152 * 8, 256>>>(ds, dasym);
  philox_all<<<152 * 8, 256>>>(dp);
  if (cudaDeviceSynchronize() != cudaSuccess) {
    std::printf("kernel failed\n");
    return 2;
  }
  std::vector<uint8_t> e2(kN), e4(kN), esr(kS);
  std::vector<uint4> ph(kP);
  unsigned long long asym = 0;
  if (cudaMemcpy(e2.data(), d2, kN, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(e4.data(), d4, kN, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(esr.data(), ds, kS, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(ph.data(), dp, (size_t)kP * sizeof(uint4), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(&asym, dasym, sizeof(asym), cudaMemcpyDeviceToHost) != cudaSuccess) {
    std::printf("copy failed\n");
    return 2;
  }
  // the oracle over the same patterns, in slices across the host's cores
  const unsigned nt = std::thread::hardware_concurrency() ? std::thread::hardware_concurrency() : 4;
  std::vector<unsigned long long> bad2(nt, 0), bad4(nt, 0), bads(nt, 0), badp(nt, 0);
  std::vector<uint32_t> first2(nt, 0xFFFFFFFFu), first4(nt, 0xFFFFFFFFu), firsts(nt, 0xFFFFFFFFu);
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
        if (b < kS && esr[b] != orc_e2m1_sr((double)v, word_of(b))) {
          if (bads[k]++ == 0) firsts[k] = b;
        }
        if (b < kP) {
          uint32_t c[4], key[2], o[4];
          philox_in(b, c, key);
          orc_philox4x32_10(c, key, o);
          const uint4 d = ph[b];
          if (d.x != o[0] || d.y != o[1] || d.z != o[2] || d.w != o[3]) {
            if (badp[k]++ == 0) std::printf("philox i=%u device=%08x oracle=%08x\n", b, d.x, o[0]);
          }
        }
      }
    });
  }
  for (auto& th : pool) th.join();
  unsigned long long m2 = 0, m4 = 0, ms = 0, mp = 0;
  for (unsigned k = 0; k < nt; ++k) {
    m2 += bad2[k];
    m4 += bad4[k];
    ms += bads[k];
    mp += badp[k];
  }
  std::printf("checked %llu mismatches %llu\n", 2ull * kN + kS + kP, m2 + m4 + ms + mp + asym);
  std::printf("e2m1 mismatches %llu, sign asymmetries %llu, e4m3 mismatches %llu, sr mismatches %llu, "
              "philox mismatches %llu\n", m2, asym, m4, ms, mp);
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
    if (firsts[k] != 0xFFFFFFFFu) {
      float v;
      std::memcpy(&v, &firsts[k], 4);
      std::printf("sr t=%08x w=%08x device=%x oracle=%x\n", firsts[k], word_of(firsts[k]), esr[firsts[k]],
                  orc_e2m1_sr((double)v, word_of(firsts[k])));
    }
  }
  return 0;
}
