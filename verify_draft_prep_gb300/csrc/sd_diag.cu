// sd_diag.cu -- diagnostic kernels: the device Philox stream, the exact race variate, and the
// exhaustive error bound of the race filter's fast -log approximation.

#include <math.h>

#include "sd_common.cuh"

namespace sdk {

__global__ void philox_kernel(int n, const uint32_t* ctr, PhiloxKey key, uint32_t* out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    const uint4 c = make_uint4(ctr[4 * i], ctr[4 * i + 1], ctr[4 * i + 2], ctr[4 * i + 3]);
    const uint4 o = philox4x32_10(c, key);
    out[4 * i] = o.x;
    out[4 * i + 1] = o.y;
    out[4 * i + 2] = o.z;
    out[4 * i + 3] = o.w;
  }
}

__global__ void race_E_kernel(int n, const uint32_t* w, float* E) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) E[i] = race_E_exact(w[i]);
}

// max over w of |R(w) * E(w) * log2(e) / 2^64 - 1|, evaluated in double.
__global__ void approx_error_kernel(uint32_t w_begin, unsigned long long count, float* max_rel) {
  const double scale = 1.4426950408889634 / 18446744073709551616.0;
  double worst = 0.0;
  for (unsigned long long k = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
       k < count; k += (unsigned long long)gridDim.x * blockDim.x) {
    const uint32_t w = (uint32_t)(w_begin + k);
    const double rel = fabs((double)race_R(w) * (double)race_E_exact(w) * scale - 1.0);
    worst = rel > worst ? rel : worst;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) worst = fmax(worst, __shfl_xor_sync(0xffffffffu, worst, o));
  if ((threadIdx.x & 31) == 0) {
    const float f = (float)worst * 1.0000001f;  // round up
    atomicMax(reinterpret_cast<int*>(max_rel), __float_as_int(f));
  }
}

// Counts, over every w in [w_begin, w_begin + count), the words where the exact race variate
// differs from the double path (counts[0]) and the words that took the double path (counts[1]).
__global__ void E_check_kernel(uint32_t w_begin, unsigned long long count,
                               unsigned long long* counts) {
  unsigned long long mis = 0, near_n = 0;
  for (unsigned long long k = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
       k < count; k += (unsigned long long)gridDim.x * blockDim.x) {
    const uint32_t w = (uint32_t)(w_begin + k);
    bool near;
    const float e = race_E_pair(w, near);
    near_n += near;
    const float got = near ? race_E_exact_double(w) : e;
    // the reference value: the double path for every word
    mis += __float_as_uint(got) != __float_as_uint(race_E_exact_double(w));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mis += __shfl_xor_sync(0xffffffffu, mis, o);
    near_n += __shfl_xor_sync(0xffffffffu, near_n, o);
  }
  if ((threadIdx.x & 31) == 0) {
    if (mis) atomicAdd(counts, mis);
    if (near_n) atomicAdd(counts + 1, near_n);
  }
}

}  // namespace sdk

extern "C" int sd_philox_launch(int n, const uint32_t* ctr, uint64_t seed, uint32_t* out,
                                cudaStream_t stream) {
  if (n == 0) return SD_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((n + 255) / 256), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, sdk::philox_kernel, n, ctr, sdk::philox_key(seed), out) ==
                 cudaSuccess
             ? SD_OK
             : SD_E_LAUNCH;
}

extern "C" int sd_race_E_launch(int n, const uint32_t* w, float* E, cudaStream_t stream) {
  if (n == 0) return SD_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((n + 255) / 256), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, sdk::race_E_kernel, n, w, E) == cudaSuccess ? SD_OK
                                                                             : SD_E_LAUNCH;
}

extern "C" int sd_approx_error_launch(uint32_t w_begin, uint64_t count, float* max_rel,
                                      cudaStream_t stream) {
  if (count == 0) return SD_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(152 * 8, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, sdk::approx_error_kernel, w_begin,
                            (unsigned long long)count, max_rel) == cudaSuccess
             ? SD_OK
             : SD_E_LAUNCH;
}

extern "C" int sd_E_check_launch(uint32_t w_begin, uint64_t count, unsigned long long* counts,
                                 cudaStream_t stream) {
  if (count == 0) return SD_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(152 * 8, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, sdk::E_check_kernel, w_begin, (unsigned long long)count,
                            counts) == cudaSuccess
             ? SD_OK
             : SD_E_LAUNCH;
}
