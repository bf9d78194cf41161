// sd_gather.cu -- drafter hidden states (sm_103a).
//
// P-EAGLE blog (vLLM), section "Hidden State 管理": target hidden states go to their drafter
// slots and the learned h_shared fills the MASK slots. The page scatters and then applies
// torch.where; here each output row gathers its source row directly (the map is injective on
// the accepted rows, so both forms write the same bytes), which needs one pass and no mask.
//
// A row is H bf16 values moved bit for bit. ROWS output rows per CTA, NT/ROWS threads per row,
// 128-bit loads and stores when every row start is 16-byte aligned. The number of rows to write
// (*total_out) is read on the device, so the launch covers the fixed capacity and stays
// capturable in a CUDA graph.

#include "sd_common.cuh"

namespace sdk {

constexpr int GNT = 256;
constexpr int GROWS = 4;  // output rows per CTA
constexpr int GTPR = GNT / GROWS;

struct GatherParams {
  int capacity, H;
  const int32_t* total_out;
  const int32_t* hidden_map;
  const uint16_t* target;
  long ld_in;
  int n_in_rows;
  const uint16_t* h_shared;
  uint16_t* out;
  long ld_out;
  int32_t* err;
  int vec;  // 16-byte aligned rows, H % 8 == 0
};

__global__ void __launch_bounds__(GNT) gather_kernel(const GatherParams P) {
  int total = __ldg(P.total_out);
  int32_t e = 0;
  if (total < 0 || total > P.capacity) {
    if (blockIdx.x == 0 && threadIdx.x == 0) e |= SD_ERR_TOTAL_RANGE;
    total = total < 0 ? 0 : P.capacity;
  }
  const int sub = threadIdx.x / GTPR;
  const int t = threadIdx.x % GTPR;
  const long row = (long)blockIdx.x * GROWS + sub;
  if (row < total) {
    const int m = __ldg(P.hidden_map + row);
    const uint16_t* src = P.h_shared;
    if (m >= 0) {
      if (m < P.n_in_rows) src = P.target + (size_t)m * P.ld_in;
      else if (t == 0) e |= SD_ERR_MAP_RANGE;
    }
    uint16_t* dst = P.out + (size_t)row * P.ld_out;
    if (P.vec) {
      const int nv = P.H >> 3;
      const uint4* s4 = reinterpret_cast<const uint4*>(src);
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      int v = t;
      for (; v + 3 * GTPR < nv; v += 4 * GTPR) {
        const uint4 a0 = __ldg(s4 + v);
        const uint4 a1 = __ldg(s4 + v + GTPR);
        const uint4 a2 = __ldg(s4 + v + 2 * GTPR);
        const uint4 a3 = __ldg(s4 + v + 3 * GTPR);
        d4[v] = a0;
        d4[v + GTPR] = a1;
        d4[v + 2 * GTPR] = a2;
        d4[v + 3 * GTPR] = a3;
      }
      for (; v < nv; v += GTPR) d4[v] = __ldg(s4 + v);
    } else {
      for (int x = t; x < P.H; x += GTPR) dst[x] = __ldg(src + x);
    }
  }
  raise_err(P.err, e);
}

}  // namespace sdk

extern "C" int sd_gather_launch(int capacity, int H, const int32_t* total_out,
                                const int32_t* hidden_map, const void* target_hidden, long ld_in,
                                int n_in_rows, const void* h_shared, void* out_hidden,
                                long ld_out, int32_t* err, cudaStream_t stream) {
  sdk::GatherParams P;
  P.capacity = capacity;
  P.H = H;
  P.total_out = total_out;
  P.hidden_map = hidden_map;
  P.target = (const uint16_t*)target_hidden;
  P.ld_in = ld_in;
  P.n_in_rows = n_in_rows;
  P.h_shared = (const uint16_t*)h_shared;
  P.out = (uint16_t*)out_hidden;
  P.ld_out = ld_out;
  P.err = err;
  P.vec = (H % 8 == 0) && ((uintptr_t)target_hidden % 16 == 0) &&
          ((uintptr_t)h_shared % 16 == 0) && ((uintptr_t)out_hidden % 16 == 0) &&
          (ld_in % 8 == 0) && (ld_out % 8 == 0);
  const int grid = capacity > 0 ? (capacity + sdk::GROWS - 1) / sdk::GROWS : 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(sdk::GNT, 1, 1);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, sdk::gather_kernel, P) == cudaSuccess ? SD_OK : SD_E_LAUNCH;
}
