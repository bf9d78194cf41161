// sd_prep.cu -- P-EAGLE drafter-batch rebuild, optionally fused with the hidden-state gather
// (sm_103a).
//
// P-EAGLE blog (vLLM), sections "并行草稿生成的挑战" and "Triton Kernel": the drafter batch
// ([token, MASK, MASK, ...] per request) has a different shape from the verify batch, so ids,
// positions, the KV slot mapping and the per-request start indices are rebuilt in one pass that
// also emits the rejected-token mask, the masked-token mask, the new-token indices and the
// hidden-state map. Section "核心方法" fixes the pairing (drafter slot j takes the token and
// hidden state of verify position j); "Hidden State 管理" fixes PADDING_SLOT_ID = -1 and the
// h_shared fill of MASK slots, done here in the same launch (gather form).
//
// Layout of the work: CTA c owns requests [c*RPC, (c+1)*RPC). No CTA waits for another: each
// recomputes the prefix of L_r = a_r + K over the requests before it (B int32 reads, served by
// L2), scans its own requests in shared memory, writes its requests' slots with consecutive
// threads on consecutive slots, copies its rows of hidden states (128-bit accesses), and writes
// its share of the padding tail. Dependent global round trips after the wait on sd_verify: the
// accepted counts, then the final tokens and block-table entries together.
//
// Programmatic dependent launch: when launched right after sd_verify on the same stream, the
// kernel is scheduled while sd_verify finishes; it loads the inputs sd_verify does not write
// (positions) and then waits (griddepcontrol.wait) until sd_verify's results are visible. It lets
// its own dependent be scheduled only at its end.

#include "sd_rebuild.cuh"

namespace sdk {

constexpr int PNT = 256;
constexpr int RPC_MAX = 1024;

struct PrepParams {
  int B, K;
  const int32_t* out_tokens;
  const int32_t* num_accepted;
  const int32_t* cu;  // nullable: per-request draft counts as a prefix [B+1] (K is then K_max)
  const int32_t* pos0;
  const int32_t* block_table;
  int max_blocks, block_size;
  int32_t mask_id;
  int capacity;
  int rpc;
  int32_t* input_ids;
  int32_t* positions;
  int32_t* slot_mapping;
  int32_t* hidden_map;
  uint8_t* is_masked;
  uint8_t* is_rejected;
  int32_t* start_loc;
  int32_t* new_token_idx;
  int32_t* total_out;
  // hidden-state gather (used when GATHER)
  int H;
  const uint16_t* hidden;
  long ld_in;
  int n_in_rows;
  const uint16_t* h_shared;
  uint16_t* out_hidden;
  long ld_out;
  int vec;
  int32_t* err;
};

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ int clamp_acc(int a, int K, int32_t& e) {
  if (a < 0 || a > K) {
    e |= SD_ERR_NUM_ACCEPTED;
    a = a < 0 ? 0 : K;
  }
  return a;
}

// Request r's draft count K_r (cu[r+1] - cu[r], clamped to [0, K] with SD_ERR_DRAFT_COUNT; K
// without cu) and the index c0 with its first target hidden row at c0 + r.
__device__ __forceinline__ int draft_count(const int32_t* cu, int r, int K, int& c0,
                                           int32_t& e) {
  if (!cu) {
    c0 = r * K;
    return K;
  }
  c0 = __ldg(cu + r);
  int k = __ldg(cu + r + 1) - c0;
  if (k < 0 || k > K || c0 < 0) {
    e |= SD_ERR_DRAFT_COUNT;
    k = (k < 0 || c0 < 0) ? 0 : K;
    c0 = c0 < 0 ? 0 : c0;
  }
  return k;
}

template <bool GATHER>
__global__ void __launch_bounds__(PNT) prep_kernel(const PrepParams P) {
  __shared__ int s_off[RPC_MAX + 1];  // local exclusive offsets of the CTA's requests
  __shared__ int s_a[RPC_MAX];
  __shared__ int s_pos[RPC_MAX];
  __shared__ int s_k[RPC_MAX];   // draft counts
  __shared__ int s_c0[RPC_MAX];  // first target hidden row - r
  __shared__ long long s_red[2][PNT / 32];
  __shared__ int s_wtot[PNT / 32];
  __shared__ int s_err;
  const int K = P.K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r0 = blockIdx.x * P.rpc;
  const int nreq = max(0, min(P.rpc, P.B - r0));
  int32_t e = 0;
  if (tid == 0) s_err = 0;

  // inputs not written by sd_verify
  for (int q = tid; q < nreq; q += PNT) s_pos[q] = __ldg(P.pos0 + r0 + q);
  grid_dependency_wait();

  // this CTA's first PNT accepted counts, loaded together with the prefix's (one round trip)
  const int a_first = tid < nreq ? P.num_accepted[r0 + tid] : 0;
  // prefix over the requests before this CTA and the total over all requests
  long long pre = 0, tot = 0;
  for (int r = tid; r < P.B; r += PNT) {
    int32_t ignored = 0;
    int c0;
    const int kr = draft_count(P.cu, r, K, c0, ignored);
    const long long L = clamp_acc(P.num_accepted[r], kr, ignored) + kr;
    tot += L;
    pre += (r < r0) ? L : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    pre += __shfl_xor_sync(0xffffffffu, pre, o);
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
  }
  if (lane == 0) {
    s_red[0][warp] = pre;
    s_red[1][warp] = tot;
  }
  __syncthreads();
  pre = 0;
  tot = 0;
#pragma unroll
  for (int w = 0; w < PNT / 32; ++w) {
    pre += s_red[0][w];
    tot += s_red[1][w];
  }

  // exclusive scan of L over this CTA's requests, PNT at a time
  int running = 0;
  for (int c = 0; c < nreq; c += PNT) {
    const int q = c + tid;
    int a = 0, L = 0, kr = 0, c0 = 0;
    if (q < nreq) {
      kr = draft_count(P.cu, r0 + q, K, c0, e);
      a = clamp_acc(c == 0 ? a_first : P.num_accepted[r0 + q], kr, e);
      L = a + kr;
    }
    int incl = L;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    __syncthreads();  // s_wtot reuse
    if (lane == 31) s_wtot[warp] = incl;
    __syncthreads();
    int woff = 0, ctot = 0;
#pragma unroll
    for (int w = 0; w < PNT / 32; ++w) {
      woff += (w < warp) ? s_wtot[w] : 0;
      ctot += s_wtot[w];
    }
    if (q < nreq) {
      s_off[q] = running + woff + incl - L;
      s_a[q] = a;
      s_k[q] = kr;
      s_c0[q] = c0;
    }
    running += ctot;
  }
  if (tid == 0) s_off[nreq] = running;
  __syncthreads();
  const int local_total = running;

  // per-request outputs
  for (int q = tid; q < nreq; q += PNT) P.start_loc[r0 + q] = (int32_t)(pre + s_off[q]);
  for (int i = tid; i < nreq * K; i += PNT) {
    const int q = i / K, k = i - q * K;
    P.new_token_idx[(size_t)r0 * K + i] =
        k < s_k[q] ? (int32_t)(pre + s_off[q] + s_a[q] + k) : -1;
  }
  for (int i = tid; i < nreq * (K + 1); i += PNT) {
    const int q = i / (K + 1), j = i - q * (K + 1);
    P.is_rejected[(size_t)r0 * (K + 1) + i] = (j >= 1 && j > s_a[q] && j <= s_k[q]) ? 1 : 0;
  }

  // this CTA's drafter slots
  for (int i = tid; i < local_total; i += PNT) {
    int lo = 0, hi = nreq - 1;  // last q with s_off[q] <= i
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_off[mid] <= i) lo = mid;
      else hi = mid - 1;
    }
    const int q = lo, rq = r0 + q, j = i - s_off[q], a = s_a[q];
    const long long g = pre + i;
    if (g >= P.capacity) {
      e |= SD_ERR_TOTAL_RANGE;
      continue;
    }
    const int32_t tok = (j <= a) ? P.out_tokens[(size_t)rq * (K + 1) + j] : P.mask_id;
    write_drafter_slot(g, j, a, tok, P.mask_id, s_pos[q],
                       P.block_table + (size_t)rq * P.max_blocks, P.max_blocks, P.block_size,
                       (long long)s_c0[q] + rq, P.input_ids, P.positions, P.slot_mapping,
                       P.hidden_map, P.is_masked, e);
  }

  // padding tail [total, capacity), split evenly over the CTAs
  if (tot < P.capacity) {
    const long long n = P.capacity - tot;
    const long long per = (n + gridDim.x - 1) / gridDim.x;
    const long long b0 = tot + per * blockIdx.x;
    const long long b1 = min((long long)P.capacity, b0 + per);
    for (long long i = b0 + tid; i < b1; i += PNT)
      write_padding_slot(i, P.input_ids, P.positions, P.slot_mapping, P.hidden_map, P.is_masked);
  }
  if (blockIdx.x == 0 && tid == 0) {
    P.start_loc[P.B] = (int32_t)tot;
    *P.total_out = (int32_t)tot;
  }

  if (GATHER) {
    // one warp per drafter row: target hidden row r*(K+1)+j (cu[r]+r+j with per-request counts)
    // for j <= a_r, h_shared otherwise
    const long long nrows = min((long long)local_total, (long long)P.capacity - pre);
    for (long long i = warp; i < nrows; i += PNT / 32) {
      int lo = 0, hi = nreq - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_off[mid] <= (int)i) lo = mid;
        else hi = mid - 1;
      }
      const int q = lo, j = (int)i - s_off[q];
      const long long m = (j <= s_a[q]) ? (long long)s_c0[q] + (r0 + q) + j : -1;
      gather_row_warp(m, P.hidden, P.ld_in, P.n_in_rows, P.h_shared,
                      P.out_hidden + (pre + i) * P.ld_out, P.H, P.vec != 0, lane, e);
    }
  }

  if (e) atomicOr(&s_err, e);
  __syncthreads();
  if (tid == 0) raise_err(P.err, s_err);
  // Only now may a programmatically dependent launch (the next kernel on the stream, e.g. the
  // next step's verify) be scheduled: with its CTAs already waiting at griddepcontrol.wait beside
  // this grid, a step on 1024 requests of 201088-entry logit rows took 8-11 us longer.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ padded drafter batch
// The fixed-width form of the same rebuild (P-EAGLE blog, "Hidden State 管理": rejected tokens
// are sent to PADDING_SLOT_ID = -1; target hidden states are scattered to their drafter rows):
// request r owns drafter rows [r*2K, (r+1)*2K); its first a_r + K rows are the packed layout's,
// the remaining K - a_r rows are rejected leftovers (token MASK, KV slot -1, hidden map -1 and
// h_shared, rejected 1). No prefix is needed, so every row is independent: one warp per row, lane
// 0 writing the row's metadata while the warp copies its hidden state.
struct PaddedParams {
  int B, K;
  const int32_t* out_tokens;
  const int32_t* num_accepted;
  const int32_t* pos0;
  const int32_t* block_table;
  int max_blocks, block_size;
  int32_t mask_id;
  int32_t* input_ids;
  int32_t* positions;
  int32_t* slot_mapping;
  int32_t* hidden_map;
  uint8_t* is_masked;
  uint8_t* rejected;
  int32_t* scatter_map;
  int32_t* new_token_idx;
  int H;
  const uint16_t* hidden;
  long ld_in;
  int n_in_rows;
  const uint16_t* h_shared;
  uint16_t* out_hidden;  // nullptr: metadata only
  long ld_out;
  int vec;
  int32_t* err;
};

__global__ void __launch_bounds__(PNT) prep_padded_kernel(const PaddedParams P) {
  __shared__ int s_err;
  const int K = P.K, W = 2 * K;
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * (PNT / 32) + (threadIdx.x >> 5);
  const long long n = (long long)P.B * W;
  if (threadIdx.x == 0) s_err = 0;
  const bool active = row < n;
  const int r = active ? (int)(row / W) : 0, j = active ? (int)(row - (long long)r * W) : 0;
  const int p0 = active ? __ldg(P.pos0 + r) : 0;  // not written by sd_verify
  grid_dependency_wait();
  __syncthreads();
  int32_t e = 0;
  if (active) {
    const int a = clamp_acc(P.num_accepted[r], K, e);
    const bool live = j < a + K;
    long long m = (j <= a) ? (long long)r * (K + 1) + j : -1;
    if (lane == 0) {
      const long long pos = (long long)p0 + 1 + j;
      int32_t slot = -1;
      if (live) {
        const long long blk = pos >= 0 ? pos / P.block_size : -1;
        if (blk < 0 || blk >= P.max_blocks) {
          e |= SD_ERR_BLOCK_TABLE;
        } else {
          const long long phys = __ldg(P.block_table + (size_t)r * P.max_blocks + blk);
          const long long sl = phys * P.block_size + pos % P.block_size;
          if (phys < 0 || sl > 2147483647LL) e |= SD_ERR_BLOCK_TABLE;
          else slot = (int32_t)sl;
        }
      }
      P.input_ids[row] = (j <= a) ? P.out_tokens[(size_t)r * (K + 1) + j] : P.mask_id;
      P.positions[row] = (int32_t)pos;
      P.slot_mapping[row] = slot;
      P.hidden_map[row] = (int32_t)m;
      P.is_masked[row] = (live && j > a) ? 1 : 0;
      P.rejected[row] = live ? 0 : 1;
      if (j <= K)
        P.scatter_map[(size_t)r * (K + 1) + j] = (j <= a) ? (int32_t)((long long)r * W + j) : -1;
      if (j < K) P.new_token_idx[(size_t)r * K + j] = (int32_t)((long long)r * W + a + j);
    }
    if (P.out_hidden) {
      if (m >= P.n_in_rows) {
        if (lane == 0) e |= SD_ERR_MAP_RANGE;
        m = -1;
      }
      const uint16_t* src = m >= 0 ? P.hidden + m * P.ld_in : P.h_shared;
      uint16_t* dst = P.out_hidden + row * P.ld_out;
      if (P.vec) {
        const int nv = P.H >> 3;
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
        uint4* d4 = reinterpret_cast<uint4*>(dst);
        copy_row_warp(s4, d4, nv, lane);
      } else {
        for (int x = lane; x < P.H; x += 32) dst[x] = __ldg(src + x);
      }
    }
  }
  if (e) atomicOr(&s_err, e);
  __syncthreads();
  if (threadIdx.x == 0) raise_err(P.err, s_err);
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // late, as in prep_kernel
}

}  // namespace sdk

extern "C" int sd_prep_launch(int B, int K, const int32_t* out_tokens, const int32_t* num_accepted,
                              const int32_t* cu_drafts, const int32_t* pos0, const int32_t* block_table, int max_blocks,
                              int block_size, int32_t mask_token_id, int capacity,
                              int32_t* input_ids, int32_t* positions, int32_t* slot_mapping,
                              int32_t* hidden_map, uint8_t* is_masked, uint8_t* is_rejected,
                              int32_t* start_loc, int32_t* new_token_idx, int32_t* total_out,
                              int H, const void* target_hidden, long ld_in, int n_in_rows,
                              const void* h_shared, void* out_hidden, long ld_out, int32_t* err,
                              cudaStream_t stream) {
  sdk::PrepParams P;
  P.B = B;
  P.K = K;
  P.out_tokens = out_tokens;
  P.num_accepted = num_accepted;
  P.cu = cu_drafts;
  P.pos0 = pos0;
  P.block_table = block_table;
  P.max_blocks = max_blocks;
  P.block_size = block_size;
  P.mask_id = mask_token_id;
  P.capacity = capacity;
  int rpc = (B + 255) / 256;
  if (rpc < 1) rpc = 1;
  if (rpc > sdk::RPC_MAX) rpc = sdk::RPC_MAX;
  P.rpc = rpc;
  P.input_ids = input_ids;
  P.positions = positions;
  P.slot_mapping = slot_mapping;
  P.hidden_map = hidden_map;
  P.is_masked = is_masked;
  P.is_rejected = is_rejected;
  P.start_loc = start_loc;
  P.new_token_idx = new_token_idx;
  P.total_out = total_out;
  P.H = H;
  P.hidden = (const uint16_t*)target_hidden;
  P.ld_in = ld_in;
  P.n_in_rows = n_in_rows;
  P.h_shared = (const uint16_t*)h_shared;
  P.out_hidden = (uint16_t*)out_hidden;
  P.ld_out = ld_out;
  P.vec = out_hidden && (H % 8 == 0) && ((uintptr_t)target_hidden % 16 == 0) &&
          ((uintptr_t)h_shared % 16 == 0) && ((uintptr_t)out_hidden % 16 == 0) &&
          (ld_in % 8 == 0) && (ld_out % 8 == 0);
  P.err = err;
  const int grid = B > 0 ? (B + rpc - 1) / rpc : 1;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(sdk::PNT, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t rc;
  if (out_hidden) rc = cudaLaunchKernelEx(&cfg, sdk::prep_kernel<true>, P);
  else rc = cudaLaunchKernelEx(&cfg, sdk::prep_kernel<false>, P);
  return rc == cudaSuccess ? SD_OK : SD_E_LAUNCH;
}

extern "C" int sd_prep_padded_launch(int B, int K, const int32_t* out_tokens,
                                     const int32_t* num_accepted, const int32_t* pos0,
                                     const int32_t* block_table, int max_blocks, int block_size,
                                     int32_t mask_token_id, int32_t* input_ids,
                                     int32_t* positions, int32_t* slot_mapping,
                                     int32_t* hidden_map, uint8_t* is_masked, uint8_t* rejected,
                                     int32_t* scatter_map, int32_t* new_token_idx, int H,
                                     const void* target_hidden, long ld_in, int n_in_rows,
                                     const void* h_shared, void* out_hidden, long ld_out,
                                     int32_t* err, cudaStream_t stream) {
  if (B == 0) return SD_OK;
  sdk::PaddedParams P;
  P.B = B;
  P.K = K;
  P.out_tokens = out_tokens;
  P.num_accepted = num_accepted;
  P.pos0 = pos0;
  P.block_table = block_table;
  P.max_blocks = max_blocks;
  P.block_size = block_size;
  P.mask_id = mask_token_id;
  P.input_ids = input_ids;
  P.positions = positions;
  P.slot_mapping = slot_mapping;
  P.hidden_map = hidden_map;
  P.is_masked = is_masked;
  P.rejected = rejected;
  P.scatter_map = scatter_map;
  P.new_token_idx = new_token_idx;
  P.H = H;
  P.hidden = (const uint16_t*)target_hidden;
  P.ld_in = ld_in;
  P.n_in_rows = n_in_rows;
  P.h_shared = (const uint16_t*)h_shared;
  P.out_hidden = (uint16_t*)out_hidden;
  P.ld_out = ld_out;
  P.vec = out_hidden && (H % 8 == 0) && ((uintptr_t)target_hidden % 16 == 0) &&
          ((uintptr_t)h_shared % 16 == 0) && ((uintptr_t)out_hidden % 16 == 0) &&
          (ld_in % 8 == 0) && (ld_out % 8 == 0);
  P.err = err;
  const long long rows = (long long)B * 2 * K;
  const long long grid = (rows + sdk::PNT / 32 - 1) / (sdk::PNT / 32);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(sdk::PNT, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sdk::prep_padded_kernel, P) == cudaSuccess ? SD_OK
                                                                             : SD_E_LAUNCH;
}
