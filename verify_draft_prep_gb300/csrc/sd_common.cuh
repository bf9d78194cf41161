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

// Each round's two products as full 64-bit results (one wide multiply each, high and low halves
// together): fewer issue slots than separate high and low multiplies, the same words.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxRoundKeys& rk) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c.x;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ rk.k0[i], (uint32_t)p1,
                   (uint32_t)(p0 >> 32) ^ c.w ^ rk.k1[i], (uint32_t)p0);
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
__device__ __forceinline__ float race_E_exact_double(uint32_t w) {
  const double v = ((double)w + 0.5) * (1.0 / 4294967296.0);
  return __double2float_rn(-log(v));
}

// ---------------------------------------------------------------------------------------------
// The same E from pairs of fp32 (hi + lo, about 48 significant bits), because GB300 runs FP64 at a
// small fraction of its FP32 rate (one double log costs a warp about 2000 cycles). -ln v is formed
// from the series 2 atanh(z) = 2 (z + z^3/3 + z^5/5 + ...):
//   v >= 1/sqrt(2): u = 1 - v (exact from the integer 2^32 - 1 - w), -ln v = 2 atanh(u / (2 - u));
//   v <  1/sqrt(2): v = 2^(k-32) m with m in [1/sqrt(2), sqrt(2)), -ln v = (32 - k) ln 2 - ln m,
//                   ln m = 2 atanh((m - 1) / (m + 1)).
// |z| <= 0.1716 in both, so the series to z^17 leaves a relative truncation below 2^-49; the
// pair arithmetic (error-free sums and FMA products) keeps the whole evaluation within about
// 2^-44. The pair's hi is its fp32 rounding; where the value lies within 2^-36 (relative) of an
// fp32 rounding boundary the double path decides instead, so the result is always the double
// path's (checked against it on the GPU over all 2^32 words).
// ---------------------------------------------------------------------------------------------
struct FF {
  float hi, lo;
};
__device__ __forceinline__ FF ff_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return FF{s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ FF ff_fast_two_sum(float a, float b) {  // |a| >= |b| or a == 0
  const float s = __fadd_rn(a, b);
  return FF{s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ FF ff_add(FF a, FF b) {
  const FF s = ff_two_sum(a.hi, b.hi);
  return ff_fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}
__device__ __forceinline__ FF ff_mul(FF a, FF b) {
  const float p = __fmul_rn(a.hi, b.hi);
  float e = fmaf(a.hi, b.hi, -p);  // the exact error of p
  e = fmaf(a.hi, b.lo, e);
  e = fmaf(a.lo, b.hi, e);
  return ff_fast_two_sum(p, e);
}
__device__ __forceinline__ FF ff_div(FF a, FF b) {
  const float q1 = __fdiv_rn(a.hi, b.hi);
  const FF p = ff_mul(FF{q1, 0.0f}, b);
  const FF r = ff_add(a, FF{-p.hi, -p.lo});
  return ff_fast_two_sum(q1, __fdiv_rn(r.hi, b.hi));
}

// 2 atanh(z) = 2z (1 + t/3 + t^2/5 + ... + t^8/17), t = z^2 <= 0.0295: the five leading
// coefficients in pairs, the tail in fp32.
__device__ __forceinline__ FF ff_two_atanh(FF z) {
  const FF t = ff_mul(z, z);
  const float tf = t.hi;
  float q = fmaf(tf, 0x1.e1e1e2p-5f /*1/17*/, 0x1.111112p-4f /*1/15*/);
  q = fmaf(tf, q, 0x1.3b13b2p-4f /*1/13*/);
  q = fmaf(tf, q, 0x1.745d18p-4f /*1/11*/);
  FF a = ff_add(FF{0x1.c71c72p-4f, -0x1.c71c72p-31f} /*1/9*/, ff_mul(t, FF{q, 0.0f}));
  a = ff_add(FF{0x1.24924ap-3f, -0x1.b6db6ep-28f} /*1/7*/, ff_mul(t, a));
  a = ff_add(FF{0x1.99999ap-3f, -0x1.99999ap-29f} /*1/5*/, ff_mul(t, a));
  a = ff_add(FF{0x1.555556p-2f, -0x1.555556p-27f} /*1/3*/, ff_mul(t, a));
  const FF P = ff_add(FF{1.0f, 0.0f}, ff_mul(t, a));
  return ff_mul(FF{2.0f * z.hi, 2.0f * z.lo}, P);
}

// The fp32 rounding of the pair's value; near = true where it may lie within 2^-36 (relative) of
// a rounding boundary, and the caller takes the double path.
__device__ __forceinline__ float race_E_pair(uint32_t w, bool& near) {
  FF y;
  if (w >= 0xB504F334u) {  // v >= 1/sqrt(2)
    const uint32_t n = 0xFFFFFFFFu - w;  // u = (n + 0.5) 2^-32 = 1 - v, n < 2^31
    const FF u = ff_two_sum(__uint2float_rn(n & ~0xFFu) * 0x1p-32f,
                            (__uint2float_rn(n & 0xFFu) + 0.5f) * 0x1p-32f);
    const FF d = ff_add(FF{2.0f, 0.0f}, FF{-u.hi, -u.lo});
    y = ff_two_atanh(ff_div(u, d));
  } else {
    FF x = ff_two_sum(__uint2float_rn(w & ~0xFFu), __uint2float_rn(w & 0xFFu) + 0.5f);
    int k = (int)((__float_as_uint(x.hi) >> 23) & 0xFFu) - 127;  // x.hi in [2^k, 2^(k+1))
    float sc = __uint_as_float((uint32_t)(127 - k) << 23);        // 2^-k, exact
    FF m{x.hi * sc, x.lo * sc};
    if (m.hi > 1.41421356f) {
      ++k;
      m.hi *= 0.5f;
      m.lo *= 0.5f;
    }
    const FF lnm = ff_two_atanh(ff_div(ff_add(m, FF{-1.0f, 0.0f}), ff_add(m, FF{1.0f, 0.0f})));
    const float K = (float)(32 - k);                          // 1..33
    const float l2lo = __fmul_rn(K, 0x1.7f7d1cp-20f);         // K ln2, second part
    FF kl = ff_fast_two_sum(__fmul_rn(K, 0x1.62e4p-1f),        // exact (17 x 6 bits)
                            l2lo);
    kl = ff_add(kl, FF{fmaf(K, 0x1.7f7d1cp-20f, -l2lo), __fmul_rn(K, 0x1.ef357ap-45f)});
    y = ff_add(kl, FF{-lnm.hi, -lnm.lo});
  }
  // y.hi is the pair's fp32 rounding; accept it unless the value may lie near a boundary
  const uint32_t hb = __float_as_uint(y.hi);
  const float ulp = __uint_as_float(hb & 0x7F800000u) * 0x1p-23f;
  const bool pow2 = (hb & 0x007FFFFFu) == 0u;
  const float half = (y.lo < 0.0f && pow2) ? 0.25f * ulp : 0.5f * ulp;
  near = !(fabsf(y.lo) + y.hi * 0x1p-36f < half);
  return y.hi;
}

// Exact race variate: the pair's rounding, or the double path near a rounding boundary (about
// one word in 2900); bit for bit the double path's value for every w.
__device__ __forceinline__ float race_E_exact(uint32_t w) {
  bool near;
  const float e = race_E_pair(w, near);
  return near ? race_E_exact_double(w) : e;
}

// Fast filter value for the race: R ~= 2^64 / (-log2 v), proportional to 1/E, from one hardware
// lg2 and one hardware reciprocal on an fp32 v. Within 2^-11 of v = 1 (w >= kNearOne, one word
// in 2048) the hardware lg2 loses relative accuracy, so there -log2(v) is formed from m = 1 - v
// by its series instead. The scale 2^64 keeps r * R in the normal range for every positive fp32
// residual r <= 2^30. The worst relative error of R against 2^64 / (E * log2(e)) over all 2^32
// words is measured exhaustively by sd_race_E_approx_error; the race filter's band (2^-7) is 47x
// wider.
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

// The GPU's nanosecond clock (%globaltimer), for waits bounded by time.
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Error bits are rare; one atomic per affected request.

__device__ __forceinline__ void raise_err(int32_t* err, int32_t bits) {
  if (err && bits) atomicOr(err, bits);
}

}  // namespace sdk
