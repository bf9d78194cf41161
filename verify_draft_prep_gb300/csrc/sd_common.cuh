// sd_common.cuh -- device helpers shared by the sm_103a kernels of libsd_gb300.
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sd.h"

namespace sdk {

namespace cg = cooperative_groups;

// ---------------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
// SC'11). Each round multiplies words 0 and 2 by the two round constants (32x32 -> 64), xors
// the high halves with the other two words and the round key, and moves the low halves across;
// the key advances by the two Weyl constants after every round. The key is uniform across a
// launch, so the ten round keys stay in uniform registers.
// ---------------------------------------------------------------------------------------------
struct PhiloxKey {
  uint32_t k0, k1;
};

__host__ __device__ __forceinline__ PhiloxKey philox_key(uint64_t seed) {
  return PhiloxKey{(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, PhiloxKey key) {
  uint32_t k0 = key.k0, k1 = key.k1;
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t lo0 = 0xD2511F53u * c.x;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// The ten round keys precomputed on the host (k0 + i*W0, k1 + i*W1), kept in the kernel's
// parameter space so that every round reads its key as a constant operand.
struct PhiloxRoundKeys {
  uint32_t k0[10], k1[10];
};

inline PhiloxRoundKeys philox_round_keys(uint64_t seed) {
  PhiloxRoundKeys rk;
  uint32_t k0 = (uint32_t)(seed & 0xffffffffu), k1 = (uint32_t)(seed >> 32);
  for (int i = 0; i < 10; ++i) {
    rk.k0[i] = k0;
    rk.k1[i] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return rk;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxRoundKeys& rk) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t lo0 = 0xD2511F53u * c.x;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ rk.k0[i], lo1, hi0 ^ c.w ^ rk.k1[i], lo0);
  }
  return c;
}

__device__ __forceinline__ uint32_t word_of(uint4 v, uint32_t i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Accept uniform of draft d_{j+1} of request r: word 0 of block (0, j, r, 0), top 24 bits.
__device__ __forceinline__ double accept_uniform(PhiloxKey key, uint32_t r, uint32_t j) {
  const uint4 w = philox4x32_10(make_uint4(0u, j, r, 0u), key);
  return (double)(w.x >> 8) * (1.0 / 16777216.0);
}

// Race block of vocab entries 4g..4g+3 on row j of request r: block (g, j, r, tag); tag 1 is
// the verify races' stream, tag 2 the drafter-side sampling's.
constexpr uint32_t kTagVerify = 1u, kTagDraft = 2u;
__device__ __forceinline__ uint4 race_block(PhiloxKey key, uint32_t g, uint32_t r, uint32_t j,
                                            uint32_t tag = kTagVerify) {
  return philox4x32_10(make_uint4(g, j, r, tag), key);
}
__device__ __forceinline__ uint4 race_block(const PhiloxRoundKeys& rk, uint32_t g, uint32_t r,
                                            uint32_t j, uint32_t tag = kTagVerify) {
  return philox4x32_10(make_uint4(g, j, r, tag), rk);
}
__device__ __forceinline__ double accept_uniform(const PhiloxRoundKeys& rk, uint32_t r,
                                                 uint32_t j) {
  const uint4 w = philox4x32_10(make_uint4(0u, j, r, 0u), rk);
  return (double)(w.x >> 8) * (1.0 / 16777216.0);
}

// Exact race variate: E = fp32 rounding of the double -log(v), v = (w + 0.5) * 2^-32 (exact).
__device__ __forceinline__ float race_E_exact(uint32_t w) {
  const double v = ((double)w + 0.5) * (1.0 / 4294967296.0);
  return __double2float_rn(-log(v));
}

// Fast filter value for the race: R ~= 2^64 / (-log2 v), proportional to 1/E, from one hardware
// lg2 and one hardware reciprocal on an fp32 v. Within 2^-11 of v = 1 (w >= kNearOne, one word
// in 2048) the hardware lg2 loses relative accuracy, so there -log2(v) is formed from m = 1 - v
// by its series instead. The scale 2^64 keeps r * R in the normal range for every positive fp32
// residual r <= 2^30. The worst relative error of R against 2^64 / (E * log2(e)) over all 2^32
// words is measured exhaustively by sd_race_E_approx_error; the race filter's band is 8x wider.
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kNearOne = 0xFFE00000u;  // w >= this: 1 - v < 2^-11

// The operands of these two are always normal numbers here (v >= 2^-33; -log2(v) * 2^-64 in
// [2^-98, 2^-58]), so the flush-to-zero forms give the same results without subnormal handling.
__device__ __forceinline__ float fast_lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^x by the hardware approximation with flush-to-zero: results below 2^-126 become 0. The
// softmax terms that flush are more than 2^126 times smaller than the row's largest term.
__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float race_R_main(uint32_t w) {
  const float v = fmaf(__uint2float_rn(w), 0x1p-32f, 0x1p-33f);
  return fast_rcp(fast_lg2(v) * -0x1p-64f);
}

__device__ __forceinline__ float race_R_near_one(uint32_t w) {
  const float m = fmaf(__uint2float_rn(~w), 0x1p-32f, 0x1p-33f);  // 1 - v, m < 2^-11
  // -ln(1 - m) = m (1 + m/2 + m^2/3 + ...); the dropped terms are below 2^-25 relative.
  return fast_rcp((m * fmaf(m, fmaf(m, 0.33333334f, 0.5f), 1.0f)) * (kLog2e * 0x1p-64f));
}

__device__ __forceinline__ float race_R(uint32_t w) {
  return w < kNearOne ? race_R_main(w) : race_R_near_one(w);
}

// ---------------------------------------------------------------------------------------------
// Packed argmax keys: (orderable 32-bit key << 32) | (0xffffffff - x). The unsigned maximum
// picks the largest key and, among equal keys, the lowest x, whatever order CTAs finish in.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t pack_key(uint32_t key_bits, uint32_t x) {
  return ((uint64_t)key_bits << 32) | (uint64_t)(0xffffffffu - x);
}
__device__ __forceinline__ uint32_t packed_index(uint64_t p) {
  return 0xffffffffu - (uint32_t)(p & 0xffffffffu);
}
__device__ __forceinline__ uint32_t packed_key_bits(uint64_t p) { return (uint32_t)(p >> 32); }

// Total order on fp32 values as unsigned integers (-0 is folded into +0 first).
__device__ __forceinline__ uint32_t orderable(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------------------------
// Block reductions (NT threads, NT a multiple of 32). `scratch` holds NT/32 entries.
// ---------------------------------------------------------------------------------------------
template <int NT>
__device__ __forceinline__ uint64_t block_max_u64(uint64_t v, uint64_t* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t other = __shfl_xor_sync(0xffffffffu, v, o);
    v = other > v ? other : v;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < NT / 32 ? scratch[lane] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint64_t other = __shfl_xor_sync(0xffffffffu, v, o);
      v = other > v ? other : v;
    }
    if (lane == 0) scratch[0] = v;
  }
  __syncthreads();
  return scratch[0];
}

// ---------------------------------------------------------------------------------------------
// Cluster helpers (thread-block clusters; distributed shared memory).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void cluster_barrier() { cg::this_cluster().sync(); }

template <typename T>
__device__ __forceinline__ T load_from_rank(T* local_ptr, unsigned rank) {
  T* remote = cg::this_cluster().map_shared_rank(local_ptr, rank);
  return *remote;  // ordered by the preceding cluster barrier
}

// ---------------------------------------------------------------------------------------------
// Streaming loads. Rows are read once; keep them out of L1.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) {
  return __uint_as_float(b16 << 16);
}

// Error bits are rare; one atomic per affected request.
__device__ __forceinline__ void raise_err(int32_t* err, int32_t bits) {
  if (err && bits) atomicOr(err, bits);
}

}  // namespace sdk
