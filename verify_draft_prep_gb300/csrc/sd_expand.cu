// sd_expand.cu -- P-EAGLE drafter-batch rebuild in one pass (sm_103a).
//
// P-EAGLE blog (vLLM), sections "并行草稿生成的挑战" and "Triton Kernel": the drafter batch has
// a different shape from the verify batch ([token, MASK, MASK, ...]), so ids, positions, the KV
// slot mapping and the per-request start indices are rebuilt, and the same pass emits the
// rejected-token mask, the masked-token mask, the new-token indices and the hidden-state map.
// Section "核心方法" fixes the pairing (drafter slot j takes the token and hidden state of verify
// position j); "Hidden State 管理" fixes PADDING_SLOT_ID = -1.
//
// One launch, no inter-CTA communication: each CTA owns NT consecutive requests and recomputes
// the prefix of L_r = a_r + K over the requests before it (B int32 reads from L2), scans its own
// requests in shared memory, then writes its requests' slots with consecutive threads on
// consecutive slots (coalesced) and its share of the padding tail.

#include "sd_common.cuh"

namespace sdk {

constexpr int XNT = 256;

struct ExpandParams {
  int B, K;
  const int32_t* out_tokens;
  const int32_t* num_accepted;
  const int32_t* pos0;
  const int32_t* block_table;
  int max_blocks, block_size;
  int32_t mask_id;
  int capacity;
  int32_t* input_ids;
  int32_t* positions;
  int32_t* slot_mapping;
  int32_t* hidden_map;
  uint8_t* is_masked;
  uint8_t* is_rejected;
  int32_t* start_loc;
  int32_t* new_token_idx;
  int32_t* total_out;
  int32_t* err;
};

__device__ __forceinline__ int clamp_accepted(int a, int K, int32_t& e) {
  if (a < 0 || a > K) {
    e |= SD_ERR_NUM_ACCEPTED;
    a = a < 0 ? 0 : K;
  }
  return a;
}

__device__ __forceinline__ long long block_sum_ll(long long v, long long* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  long long t = 0;
#pragma unroll
  for (int w = 0; w < XNT / 32; ++w) t += scratch[w];
  return t;
}

__global__ void __launch_bounds__(XNT) expand_kernel(const ExpandParams P) {
  __shared__ long long red[2][XNT / 32];
  __shared__ int excl[XNT + 1];   // local exclusive scan of L over this CTA's requests
  __shared__ int acc[XNT];
  __shared__ int warp_tot[XNT / 32];
  __shared__ int s_err;
  const int K = P.K;
  const int tid = threadIdx.x;
  const int r0 = blockIdx.x * XNT;
  if (tid == 0) s_err = 0;

  // 1. prefix (requests before this CTA) and total over all requests
  long long pre = 0, tot = 0;
  for (int r = tid; r < P.B; r += XNT) {
    int32_t dummy = 0;
    const long long L = clamp_accepted(__ldg(P.num_accepted + r), K, dummy) + K;
    tot += L;
    if (r < r0) pre += L;
  }
  pre = block_sum_ll(pre, red[0]);
  tot = block_sum_ll(tot, red[1]);

  // 2. this CTA's requests: scan of L, per-request outputs
  int32_t e = 0;
  const int r = r0 + tid;
  int a = 0, L = 0;
  if (r < P.B) {
    a = clamp_accepted(__ldg(P.num_accepted + r), K, e);
    L = a + K;
  }
  // block exclusive scan of L (warp scan, then warp totals)
  int incl = L;
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int woff = 0;
  for (int w = 0; w < warp; ++w) woff += warp_tot[w];
  const int ex = woff + incl - L;
  excl[tid] = ex;
  acc[tid] = a;
  if (tid == XNT - 1) excl[XNT] = ex + L;
  __syncthreads();
  const int local_total = excl[XNT];
  if (r < P.B) {
    const long long start = pre + ex;
    P.start_loc[r] = (int32_t)start;
    for (int k = 0; k < K; ++k) P.new_token_idx[(size_t)r * K + k] = (int32_t)(start + a + k);
    for (int j = 0; j <= K; ++j) P.is_rejected[(size_t)r * (K + 1) + j] = (j >= 1 && j > a) ? 1 : 0;
  }

  // 3. this CTA's slots, consecutive threads on consecutive slots
  const int nreq = min(XNT, P.B - r0);
  for (int i = tid; i < local_total; i += XNT) {
    int lo = 0, hi = nreq - 1;  // last request q with excl[q] <= i
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (excl[mid] <= i) lo = mid;
      else hi = mid - 1;
    }
    const int q = lo;
    const int rq = r0 + q;
    const int j = i - excl[q];
    const int aq = acc[q];
    const long long g = pre + i;
    if (g >= P.capacity) {
      e |= SD_ERR_TOTAL_RANGE;
      continue;
    }
    P.input_ids[g] = (j <= aq) ? __ldg(P.out_tokens + (size_t)rq * (K + 1) + j) : P.mask_id;
    const long long pos = (long long)__ldg(P.pos0 + rq) + 1 + j;
    P.positions[g] = (int32_t)pos;
    int32_t slot = -1;
    const long long blk = pos >= 0 ? pos / P.block_size : -1;
    if (blk < 0 || blk >= P.max_blocks) {
      e |= SD_ERR_BLOCK_TABLE;
    } else {
      const long long phys = __ldg(P.block_table + (size_t)rq * P.max_blocks + blk);
      const long long s = phys * P.block_size + pos % P.block_size;
      if (phys < 0 || s > 2147483647LL) e |= SD_ERR_BLOCK_TABLE;
      else slot = (int32_t)s;
    }
    P.slot_mapping[g] = slot;
    P.hidden_map[g] = (j <= aq) ? (int32_t)((long long)rq * (K + 1) + j) : -1;
    P.is_masked[g] = (j > aq) ? 1 : 0;
  }

  // 4. padding tail [total, capacity), split evenly over the CTAs
  if (tot < P.capacity) {
    const long long n = P.capacity - tot;
    const long long per = (n + gridDim.x - 1) / gridDim.x;
    const long long b0 = tot + per * blockIdx.x;
    const long long b1 = min((long long)P.capacity, b0 + per);
    for (long long i = b0 + tid; i < b1; i += XNT) {
      P.input_ids[i] = -1;
      P.positions[i] = 0;
      P.slot_mapping[i] = -1;
      P.hidden_map[i] = -1;
      P.is_masked[i] = 0;
    }
  }
  if (blockIdx.x == 0 && tid == 0) {
    P.start_loc[P.B] = (int32_t)tot;
    *P.total_out = (int32_t)tot;
  }
  if (e) atomicOr(&s_err, e);
  __syncthreads();
  if (tid == 0) raise_err(P.err, s_err);
}

}  // namespace sdk

extern "C" int sd_expand_launch(int B, int K, const int32_t* out_tokens,
                                const int32_t* num_accepted, const int32_t* pos0,
                                const int32_t* block_table, int max_blocks, int block_size,
                                int32_t mask_token_id, int capacity, int32_t* input_ids,
                                int32_t* positions, int32_t* slot_mapping, int32_t* hidden_map,
                                uint8_t* is_masked, uint8_t* is_rejected, int32_t* start_loc,
                                int32_t* new_token_idx, int32_t* total_out, int32_t* err,
                                cudaStream_t stream) {
  sdk::ExpandParams P{B,         K,          out_tokens, num_accepted, pos0,          block_table,
                      max_blocks, block_size, mask_token_id, capacity,  input_ids,     positions,
                      slot_mapping, hidden_map, is_masked, is_rejected, start_loc, new_token_idx,
                      total_out, err};
  const int grid = B > 0 ? (B + sdk::XNT - 1) / sdk::XNT : 1;
  sdk::expand_kernel<<<grid, sdk::XNT, 0, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? SD_OK : SD_E_LAUNCH;
}
