// k_row.cu -- rowwise quantize / QDQ of a contiguous tensor as a flat stream
// of 1 x 16 blocks.
//
// With the rows packed back to back (leading dimension K) and every outer
// block inside one row (ob divides K), the rowwise method never needs the
// row index: element n = (g M + i) K + j is the flat index, its codes sit at
// byte n / 2, its inner scale at n / 16, a 1 x ob outer scale at n / ob, and
// the stochastic-rounding counter and the residual are indexed by n too
// ("NVFP4 / AMD-FP4 outer-block (two-level) scaling for FP4 training",
// "Technical design"; fp4-train README, "Method" and "API" for the residual).
// So the kernel streams blocks: lane l of a warp
// owns block 32 w + l of its step, loads its 32 bytes (bf16) or 64 bytes
// (binary32) with 256-bit loads, and a 1 x ob outer block is ob / 16
// adjacent lanes, reduced with xor-shuffles.  No shared-memory tile, no
// barrier in the loop; the only shared memory is the inner-scale table.
// The bf16 round-to-nearest quantize takes a second form, row_bulk_kernel,
// whose input arrives by 1-D bulk copies into shared memory (below).
#include "fp4q_block.cuh"
#include "fp4q_device.cuh"
#include "fp4q_internal.h"
#include "fp4q_pair.cuh"
#include "fp4q_tma.cuh"

namespace fp4q {
namespace {

constexpr int RT = 256;  // threads per CTA
constexpr int RU = 2;    // blocks per thread in flight

// Where the rowwise kernel takes S from.
enum RowOuter : int {
  RO_NONE = 0,     // mode none
  RO_UNIFORM = 1,  // one S for the tensor (tensorwise, or its stored value)
  RO_WARP = 2,     // 1 x ob outer blocks computed across ob / 16 lanes
  RO_BUFFER = 3,   // 1 x ob outer scales read from the row buffer
};

__device__ __forceinline__ void ld256(const void* p, uint32_t (&a)[8]) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7])
               : "l"(p));
}
__device__ __forceinline__ void ld256_rw(const void* p, uint32_t (&a)[8]) {
  asm volatile("ld.global.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7])
               : "l"(p)
               : "memory");
}

template <bool IN_BF16>
struct Raw {
  uint32_t w[IN_BF16 ? 8 : 16];
};

template <bool IN_BF16>
__device__ __forceinline__ void load_raw(const void* x, int64_t b, Raw<IN_BF16>& r) {
  if (IN_BF16) {
    ld256(static_cast<const uint16_t*>(x) + 16 * b, *reinterpret_cast<uint32_t(*)[8]>(r.w));
  } else {
    const float* p = static_cast<const float*>(x) + 16 * b;
    ld256(p, *reinterpret_cast<uint32_t(*)[8]>(r.w));
    ld256(p + 8, *reinterpret_cast<uint32_t(*)[8]>(r.w + 8));
  }
}

// |max| of a block straight from its raw words when nothing is added:
// packed bf16 pairs; a non-finite result is sent to the sanitizing path.
template <bool IN_BF16>
__device__ __forceinline__ float raw_amax(const Raw<IN_BF16>& r) {
  if (IN_BF16) {
    uint32_t m = bf16x2_amax(bf16x2_amax(bf16x2_amax(r.w[0], r.w[1]), bf16x2_amax(r.w[2], r.w[3])),
                             bf16x2_amax(bf16x2_amax(r.w[4], r.w[5]), bf16x2_amax(r.w[6], r.w[7])));
    m &= 0x7FFF7FFFu;
    const uint32_t hi = m >> 16, lo = m & 0xFFFFu;
    return bitsf((hi > lo ? hi : lo) << 16);
  } else {
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = f32_amax(bitsf(r.w[2 * i]), bitsf(r.w[2 * i + 1]));
#pragma unroll
    for (int i = 0; i < 4; ++i) m[i] = f32_amax(m[2 * i], m[2 * i + 1]);
    return bitsf(fbits(f32_amax(f32_amax(m[0], m[1]), f32_amax(m[2], m[3]))) & 0x7FFFFFFFu);
  }
}

template <bool IN_BF16>
__device__ __forceinline__ void unpack(const Raw<IN_BF16>& r, float (&u)[16]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (IN_BF16) {
      u[2 * i] = bf16lo(r.w[i]);
      u[2 * i + 1] = bf16hi(r.w[i]);
    } else {
      u[2 * i] = bitsf(r.w[2 * i]);
      u[2 * i + 1] = bitsf(r.w[2 * i + 1]);
    }
  }
}

struct TabView {
  const float4* tab;
};

template <bool IN_BF16, bool SR, bool UE5M3, int RO>
__global__ void __launch_bounds__(RT) row_kernel(const QuantJob j) {
  pdl_wait_then_release();
  __shared__ float4 tab[256];
  build_scale_table<UE5M3>(tab, threadIdx.x, RT);
  const TabView tv{tab};
  const int lane = threadIdx.x & 31;
  const int64_t nblk = j.G * j.M * j.K / 16;
  const int64_t warp0 = (int64_t)blockIdx.x * (RT / 32) + (threadIdx.x >> 5);
  const int64_t nwarp = (int64_t)gridDim.x * (RT / 32);
  const int per = RO == RO_WARP || RO == RO_BUFFER ? j.ob / 16 : 1;  // inner blocks per outer block
  const bool per_pow2 = (per & (per - 1)) == 0;
  const int lper = 31 - __clz(per);
  const bool deq = j.qdq_orient == 1 || j.residual != nullptr;
  const uint32_t maxfin = IN_BF16 ? 0x7F7F0000u : 0x7F7FFFFFu;
  float S_u = 1.0f, r_u = 1.0f;
  if (RO == RO_UNIFORM) {
    if (j.s_src == S_TENSORWISE_WS) {
      S_u = ieee_div(bitsf(*j.tw_amax), UE5M3 ? 688128.0f : 2688.0f);
      if (blockIdx.x == 0 && threadIdx.x == 0 && j.tile_outer) j.tile_outer[0] = S_u;
    } else {
      S_u = j.tile_outer[0];
    }
    r_u = ieee_rcp(S_u);
  }
  __syncthreads();

  // warp-uniform loop: every lane runs every step (shuffles use full masks)
  for (int64_t base = warp0 * 32; base < nblk; base += nwarp * 32 * RU) {
    Raw<IN_BF16> raw[RU];
    int64_t b[RU];
    bool valid[RU];
#pragma unroll
    for (int q = 0; q < RU; ++q) {
      b[q] = base + (int64_t)q * nwarp * 32 + lane;
      valid[q] = b[q] < nblk;
      if (valid[q]) load_raw<IN_BF16>(j.x, b[q], raw[q]);
      else
#pragma unroll
        for (int i = 0; i < (IN_BF16 ? 8 : 16); ++i) raw[q].w[i] = 0u;
    }
#pragma unroll
    for (int q = 0; q < RU; ++q) {
      float u[16];
      unpack<IN_BF16>(raw[q], u);
      float am;
      if (j.residual) {
        if (valid[q]) {
          uint32_t rr[8];
          const float* rp = j.residual + 16 * b[q];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            ld256_rw(rp + 8 * h, rr);
#pragma unroll
            for (int i = 0; i < 8; ++i) u[8 * h + i] = ieee_add(u[8 * h + i], bitsf(rr[i]));
          }
        }
        am = amax16(u);
      } else {
        am = raw_amax<IN_BF16>(raw[q]);
      }
      if (fbits(am) >= 0x7F800000u) {  // inf / NaN present: sanitize the block
#pragma unroll
        for (int i = 0; i < 16; ++i) u[i] = sanitize(u[i], maxfin);
        am = amax16(u);
      }
      Norm n;
      n.none = RO == RO_NONE;
      n.S = 1.0f;
      n.r = 1.0f;
      if (RO == RO_UNIFORM) {
        n.S = S_u;
        n.r = r_u;
      } else if (RO == RO_WARP) {
        uint32_t g = fbits(am);
        for (int o = 1; o < per; o <<= 1) g = umax(g, __shfl_xor_sync(0xFFFFFFFFu, g, o));
        outer_sr<UE5M3>(bitsf(g), n.S, n.r);
        if (j.row_outer && j.do_row && valid[q] && (lane & (per - 1)) == 0) j.row_outer[b[q] >> lper] = n.S;
      } else if (RO == RO_BUFFER) {
        if (valid[q]) n.S = j.row_outer[per_pow2 ? (b[q] >> lper) : b[q] / per];
        n.r = ieee_rcp(n.S);
      }
      uint32_t sc, w0, w1;
      float dq[16];
      // round-to-nearest quantize without dequantized values: the fast form
      // when every lane's block is in its range (one warp-uniform branch)
      float a = am;
      const bool fast = !SR && !deq && __all_sync(0xFFFFFFFFu, RO == RO_NONE || fast_block(am, n.S, n.r, a));
      if (fast) {
        sc = block_fast<false, UE5M3, RO != RO_NONE, false>(tab, u, a, n.S, n.r, j.srk, 0u, 0u, 0ull, w0, w1);
      } else {
        n.pos = n.none || positive(n.S);
        n.fast = !n.none && positive_normal(n.S) && positive_normal(n.r);
        float4 T;
        sc = block_scale<UE5M3>(tv, am, n, T);
        float x[16];
        normalize16<SR>(u, x, n);
        if (deq) encode16<SR, true>(x, T, n, j.srk, j.step, 0u, sr_row_n(j, 16 * b[q]), w0, w1, dq);
        else encode16<SR, false>(x, T, n, j.srk, j.step, 0u, sr_row_n(j, 16 * b[q]), w0, w1, dq);
      }
      if (!valid[q]) continue;
      if (j.row_codes) {
        *reinterpret_cast<uint2*>(j.row_codes + 8 * b[q]) = make_uint2(w0, w1);
        j.row_scales[b[q]] = (uint8_t)sc;
      }
      if (j.residual) {
        uint32_t rr[8];
        float* rp = j.residual + 16 * b[q];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int i = 0; i < 8; ++i) rr[i] = fbits(ieee_sub(u[8 * h + i], dq[8 * h + i]));
          st256(rp + 8 * h, rr);
        }
      }
      if (j.qdq_orient == 1) {
        if (j.out_bf16) {
          uint32_t yy[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) yy[i] = pack_bf16x2(dq[2 * i], dq[2 * i + 1]);
          st256(static_cast<uint16_t*>(j.y) + 16 * b[q], yy);
        } else {
          uint32_t yy[8];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int i = 0; i < 8; ++i) yy[i] = fbits(dq[8 * h + i]);
            st256(static_cast<float*>(j.y) + 16 * b[q] + 8 * h, yy);
          }
        }
      }
    }
  }
}

// ---- bf16 round-to-nearest quantize fed by 1-D bulk copies ----
// The same per-block steps with the input moved by the copy engine: a CTA
// walks chunks of QB blocks (8 KB of bf16; chunk c = blockIdx.x + i
// gridDim.x), QS chunks in flight in shared memory, each completed on an
// mbarrier (bounded waits), so the loads hold no registers while they are
// in flight.  Thread t takes block t of the chunk, so the lanes of a 1 x ob
// outer block stay adjacent (a chunk starts on a multiple of QB blocks).
constexpr int QB = 256, QS = 4;

__device__ unsigned int g_row_timeout = 0;

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// With 1 x ob outer blocks or one tensorwise scale (PAIR) the kernel takes
// the pair-table path of fp4q_pair.cuh when the outer amax (a bf16 value) is
// in its range: the table image arrives by one more bulk copy, and per value
// pair the codes cost two packed multiplies; the general per-block steps
// then take their inner-scale entries computed on demand.
// OB64: the outer block is 1 x 64 (four lanes), a compile-time constant.
template <bool UE5M3, int RO, bool OB64 = false>
__global__ void __launch_bounds__(RT) row_bulk_kernel(const QuantJob j) {
  constexpr bool PAIR = RO == RO_WARP || RO == RO_UNIFORM;
  __shared__ __align__(128) unsigned char buf[QS][QB * 32];
  __shared__ __align__(16) unsigned char img[PAIR ? kImgOuter : 16];  // the pair-table image
  __shared__ float4 tab_s[PAIR ? 1 : 256];                            // inner-scale table (other forms)
  __shared__ __align__(8) uint64_t bars[QS + 1];
  const int t = threadIdx.x, lane = t & 31;
  const int64_t nblk = j.G * j.M * j.K / 16, nch = (nblk + QB - 1) / QB;
  const unsigned char* xb = static_cast<const unsigned char*>(j.x);
  auto issue = [&](int64_t c, int s) {
    const int64_t nb = nblk - c * QB < QB ? nblk - c * QB : QB;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_expect_tx(&bars[s], (uint32_t)(nb * 32));
    bulk_load(buf[s], xb + c * QB * 32, (uint32_t)(nb * 32), &bars[s]);
  };
  if (t == 0) {
#pragma unroll
    for (int s = 0; s <= QS; ++s) mbar_init(&bars[s]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (PAIR) {  // constant data: the copy may start before the previous grid has finished
      mbar_expect_tx(&bars[QS], kImgOuter);
      bulk_load(img, kCtlTab[UE5M3 ? 1 : 0], kImgOuter, &bars[QS]);
    }
  }
  pdl_wait_then_release();
  __syncthreads();
  if (t == 0) {
#pragma unroll
    for (int s = 0; s < QS - 1; ++s) {
      const int64_t c = blockIdx.x + (int64_t)s * gridDim.x;
      if (c < nch) issue(c, s);
    }
  }
  if (!PAIR) build_scale_table<UE5M3>(tab_s, t, RT);
  // the inner-scale entries: the shared table, or computed on demand
  auto entries = [&]() {
    if constexpr (PAIR) return EntryCalc<UE5M3>{};
    else return static_cast<const float4*>(tab_s);
  };
  const auto tab = entries();
  struct {
    decltype(entries()) tab;
  } tv{tab};
  const unsigned char* ptb = img;
  const uint32_t* ctab = reinterpret_cast<const uint32_t*>(PAIR ? img + 10240 : img);
  const int per = OB64 ? 4 : RO == RO_WARP || RO == RO_BUFFER ? j.ob / 16 : 1;
  const bool per_pow2 = (per & (per - 1)) == 0;
  const int lper = OB64 ? 2 : 31 - __clz(per);
  float S_u = 1.0f, r_u = 1.0f;
  uint32_t A_u = 0;  // the tensorwise amax, when it is computed here (bf16 input: a bf16 value)
  if (RO == RO_UNIFORM) {
    if (j.s_src == S_TENSORWISE_WS) {
      A_u = *j.tw_amax;
      S_u = ieee_div(bitsf(A_u), UE5M3 ? 688128.0f : 2688.0f);
      if (blockIdx.x == 0 && t == 0 && j.tile_outer) j.tile_outer[0] = S_u;
    } else {
      S_u = j.tile_outer[0];
    }
    r_u = ieee_rcp(S_u);
  }
  __syncthreads();
  if (PAIR && !mbar_wait(&bars[QS], 0u, 1u << 22)) atomicExch(&g_row_timeout, 1u);
  float zh_u = 0.0f, zl_u = 0.0f;
  const bool u_z = RO == RO_UNIFORM && j.s_src == S_TENSORWISE_WS && (A_u & 0xFFFFu) == 0u && table_ok<UE5M3>(A_u);
  if (u_z) outer_rcp(ptb, A_u, zh_u, zl_u);
  int slot = 0;
  uint32_t phase = 0;
  for (int64_t c = blockIdx.x; c < nch; c += gridDim.x) {
    if (t == 0) {
      const int64_t cn = c + (int64_t)(QS - 1) * gridDim.x;
      if (cn < nch) issue(cn, slot == 0 ? QS - 1 : slot - 1);
    }
    if (!mbar_wait(&bars[slot], phase, 1u << 22)) atomicExch(&g_row_timeout, 1u);
    const int64_t b = c * QB + t;
    const bool valid = b < nblk;
    Raw<true> raw;
    if (valid) {
      const uint4 lo = *reinterpret_cast<const uint4*>(buf[slot] + 32 * t);
      const uint4 hi = *reinterpret_cast<const uint4*>(buf[slot] + 32 * t + 16);
      raw.w[0] = lo.x; raw.w[1] = lo.y; raw.w[2] = lo.z; raw.w[3] = lo.w;
      raw.w[4] = hi.x; raw.w[5] = hi.y; raw.w[6] = hi.z; raw.w[7] = hi.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) raw.w[i] = 0u;
    }
    float u[16];
    unpack<true>(raw, u);
    float am = raw_amax<true>(raw);
    if (fbits(am) >= 0x7F800000u) {  // inf / NaN present: sanitize the block
#pragma unroll
      for (int i = 0; i < 16; ++i) u[i] = sanitize(u[i], 0x7F7F0000u);
      am = amax16(u);
    }
    Norm n;
    n.none = RO == RO_NONE;
    n.S = 1.0f;
    n.r = 1.0f;
    bool zfast = u_z;  // the pair-table path
    float zh = zh_u, zl = zl_u;
    uint32_t A = A_u;  // the outer amax bits (pair path)
    if (RO == RO_UNIFORM) {
      n.S = S_u;
      n.r = r_u;
    } else if (RO == RO_WARP) {
      uint32_t g = fbits(am);
      for (int o = 1; o < per; o <<= 1) g = umax(g, __shfl_xor_sync(0xFFFFFFFFu, g, o));
      // the outer amax of bf16 inputs is a bf16 value: the pair table when
      // the warp's scales are in its range
      zfast = __all_sync(0xFFFFFFFFu, table_ok<UE5M3>(g));
      if (zfast) {
        n.S = div_bmr(bitsf(g), bitsf(UE5M3 ? kDenHiU5 : kDenHiE4), bitsf(UE5M3 ? kDenLoU5 : kDenLoE4));  // exact
        outer_rcp(ptb, g, zh, zl);
        A = g;
      } else {
        outer_sr<UE5M3>(bitsf(g), n.S, n.r);
      }
      if (j.row_outer && j.do_row && valid && (lane & (per - 1)) == 0) j.row_outer[b >> lper] = n.S;
    } else if (RO == RO_BUFFER) {
      if (valid) n.S = j.row_outer[per_pow2 ? (b >> lper) : b / per];
      n.r = ieee_rcp(n.S);
    }
    uint32_t sc, w0, w1;
    if (PAIR && zfast) {
      // a = RN(am / S), v = RN(a / 6) by the known-divisor method; the codes
      // by the pair's multipliers, two values per instruction
      sc = encode_scale<UE5M3>(div_bmr(div_bmr(am, zh, zl), bitsf(kSixHi), bitsf(kSixLo)));
      float c1, c2;
      pair_mults(ptb, ctab, sc, A, c1, c2);
      const uint64_t C1 = pk2(c1, c1), C2 = pk2(c2, c2);
      float tq[16];
#pragma unroll
      for (int i = 0; i < 16; i += 2) upk2(mul2(mul2(pk2(u[i], u[i + 1]), C1), C2), tq[i], tq[i + 1]);
      w0 = e2m1x8_rne(tq);
      w1 = e2m1x8_rne(tq + 8);
    } else {
      float a = am;
      const bool fast = __all_sync(0xFFFFFFFFu, RO == RO_NONE || fast_block(am, n.S, n.r, a));
      if (fast) {
        sc = block_fast<false, UE5M3, RO != RO_NONE, false>(tab, u, a, n.S, n.r, j.srk, 0u, 0u, 0ull, w0, w1);
      } else {
        n.pos = n.none || positive(n.S);
        n.fast = !n.none && positive_normal(n.S) && positive_normal(n.r);
        float4 T;
        sc = block_scale<UE5M3>(tv, am, n, T);
        float x[16], dq[16];
        normalize16<false>(u, x, n);
        encode16<false, false>(x, T, n, j.srk, 0u, 0u, 0ull, w0, w1, dq);
      }
    }
    if (valid) {
      *reinterpret_cast<uint2*>(j.row_codes + 8 * b) = make_uint2(w0, w1);
      j.row_scales[b] = (uint8_t)sc;
    }
    __syncthreads();  // the slot is free for the copy issued next iteration
    if (++slot == QS) {
      slot = 0;
      phase ^= 1u;
    }
  }
}

template <bool UE5M3, int RO, bool OB64 = false>
cudaError_t launch_row_bulk_t(const QuantJob& j, cudaStream_t st) {
  auto kern = row_bulk_kernel<UE5M3, RO, OB64>;
  static int per_sm_cache[128] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 128) dev = 0;
  int& per_sm = per_sm_cache[dev];
  if (per_sm == 0) {
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, RT, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
  }
  const int64_t nch = (j.G * j.M * j.K / 16 + QB - 1) / QB;
  const int64_t cap = (int64_t)num_sms() * per_sm;
  return launch_pdl(kern, dim3((unsigned)(nch < cap ? nch : cap)), dim3(RT), 0, st, j);
}

template <bool UE5M3>
cudaError_t launch_row_bulk_o(const QuantJob& j, cudaStream_t st) {
  if (j.s_src == S_ONE) return launch_row_bulk_t<UE5M3, RO_NONE>(j, st);
  if (j.s_src == S_TENSORWISE_WS || j.mode == 1) return launch_row_bulk_t<UE5M3, RO_UNIFORM>(j, st);
  if (j.s_src == S_IN_TILE)
    return j.ob == 64 ? launch_row_bulk_t<UE5M3, RO_WARP, true>(j, st) : launch_row_bulk_t<UE5M3, RO_WARP>(j, st);
  return launch_row_bulk_t<UE5M3, RO_BUFFER>(j, st);
}

template <bool IN_BF16, bool SR, bool UE5M3, int RO>
cudaError_t launch_row_t(const QuantJob& j, cudaStream_t st) {
  auto kern = row_kernel<IN_BF16, SR, UE5M3, RO>;
  static int per_sm_cache[128] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 128) dev = 0;
  int& per_sm = per_sm_cache[dev];
  if (per_sm == 0) {
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, RT, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
  }
  const int64_t nblk = j.G * j.M * j.K / 16;
  const int64_t need = (nblk + RT * RU - 1) / (RT * RU);
  const int64_t cap = (int64_t)num_sms() * per_sm;
  return launch_pdl(kern, dim3((unsigned)(need < cap ? need : cap)), dim3(RT), 0, st, j);
}

template <bool IN_BF16, bool SR, bool UE5M3>
cudaError_t launch_row_o(const QuantJob& j, cudaStream_t st) {
  if (j.s_src == S_ONE) return launch_row_t<IN_BF16, SR, UE5M3, RO_NONE>(j, st);
  if (j.s_src == S_TENSORWISE_WS || j.mode == 1) return launch_row_t<IN_BF16, SR, UE5M3, RO_UNIFORM>(j, st);
  if (j.s_src == S_IN_TILE) return launch_row_t<IN_BF16, SR, UE5M3, RO_WARP>(j, st);
  return launch_row_t<IN_BF16, SR, UE5M3, RO_BUFFER>(j, st);
}

template <bool IN_BF16>
cudaError_t launch_row_d(const QuantJob& j, cudaStream_t st) {
  if (j.sr) return j.ue5m3 ? launch_row_o<IN_BF16, true, true>(j, st) : launch_row_o<IN_BF16, true, false>(j, st);
  return j.ue5m3 ? launch_row_o<IN_BF16, false, true>(j, st) : launch_row_o<IN_BF16, false, false>(j, st);
}

bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

}  // namespace

bool row_supports(const QuantJob& j) {
  if (j.do_col || j.inner_2d || j.outer_2d || j.qdq_orient == 2) return false;
  if (j.ld != j.K && j.G * j.M > 1) return false;  // rows must be packed back to back
  if (!aligned32(j.x) || (j.residual && !aligned32(j.residual)) || (j.qdq_orient == 1 && !aligned32(j.y)))
    return false;
  if (j.s_src == S_IN_TILE && !(j.ob == 16 || j.ob == 32 || j.ob == 64)) return false;
  if (j.rsl.mma) return false;  // the tensor-core scale layout is written by the tile kernels
  return true;
}

cudaError_t launch_row(const QuantJob& j, cudaStream_t st) {
  // bf16 round-to-nearest quantize (codes out, no residual): the bulk-copy form
  if (j.in_bf16 && !j.sr && !j.residual && j.qdq_orient == 0 && j.row_codes && j.G * j.M * j.K > 0)
    return j.ue5m3 ? launch_row_bulk_o<true>(j, st) : launch_row_bulk_o<false>(j, st);
  return j.in_bf16 ? launch_row_d<true>(j, st) : launch_row_d<false>(j, st);
}

cudaError_t row_timeout_flag(uint32_t* v, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(v, g_row_timeout, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_row_timeout, &z, sizeof z);
  }
  return e;
}

}  // namespace fp4q
