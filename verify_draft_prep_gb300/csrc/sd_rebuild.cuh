// sd_rebuild.cuh -- per-slot and per-row pieces of the P-EAGLE drafter-batch rebuild, shared by
// the rebuild kernel (sd_prep.cu) and the verify kernel's fused rebuild (sd_verify.cu), so that
// both write exactly the same bytes.
//
// P-EAGLE blog (vLLM), sections "并行草稿生成的挑战" and "Triton Kernel": drafter slot j of
// request r (position pos0_r + 1 + j) takes the accepted draft d_{j+1} for j < a_r, the final
// token for j = a_r, and MASK after it; its KV slot comes from the block table (PADDING_SLOT_ID
// -1 where the table does not cover it); slots j <= a_r map the target hidden row of verify
// position j, the MASK slots h_shared ("Hidden State 管理").
#pragma once

#include "sd_common.cuh"

namespace sdk {

// Writes drafter slot j (global index g, g < capacity) of a request whose first target hidden
// row is hrow0; `tok` is the slot's token for j <= a (ignored after a). input_ids may be NULL
// (the token is written elsewhere).
__device__ __forceinline__ void write_drafter_slot(long long g, int j, int a, int32_t tok,
                                                   int32_t mask_id, int pos0,
                                                   const int32_t* bt_row, int max_blocks,
                                                   int block_size, long long hrow0,
                                                   int32_t* input_ids, int32_t* positions,
                                                   int32_t* slot_mapping, int32_t* hidden_map,
                                                   uint8_t* is_masked, int32_t& e) {
  const long long pos = (long long)pos0 + 1 + j;
  const long long blk = pos >= 0 ? pos / block_size : -1;
  const bool blk_ok = blk >= 0 && blk < max_blocks;
  const long long phys = blk_ok ? (long long)__ldg(bt_row + blk) : -1;
  int32_t slot = -1;
  const long long sl = phys * block_size + pos % block_size;
  if (!blk_ok || phys < 0 || sl > 2147483647LL) e |= SD_ERR_BLOCK_TABLE;
  else slot = (int32_t)sl;
  if (input_ids) input_ids[g] = (j <= a) ? tok : mask_id;
  positions[g] = (int32_t)pos;
  slot_mapping[g] = slot;
  hidden_map[g] = (j <= a) ? (int32_t)(hrow0 + j) : -1;
  is_masked[g] = (j > a) ? 1 : 0;
}

// One slot of the padding tail [total, capacity).
__device__ __forceinline__ void write_padding_slot(long long i, int32_t* input_ids,
                                                   int32_t* positions, int32_t* slot_mapping,
                                                   int32_t* hidden_map, uint8_t* is_masked) {
  input_ids[i] = -1;
  positions[i] = 0;
  slot_mapping[i] = -1;
  hidden_map[i] = -1;
  is_masked[i] = 0;
}

// One warp copies a row of nv 16-byte words: each lane issues all of its loads (up to
// kCopyBatch) before its stores, so a row of a few KB costs one memory round trip. The stores
// are streaming (evict-first): the rows are written once and read by a later kernel, so they
// leave L2 while this kernel runs instead of being written back during the next one's reads.
constexpr int kCopyBatch = 12;
__device__ __forceinline__ void copy_row_warp(const uint4* __restrict__ src,
                                              uint4* __restrict__ dst, int nv, int lane) {
  for (int v0 = lane; v0 < nv; v0 += 32 * kCopyBatch) {
    uint4 x[kCopyBatch];
#pragma unroll
    for (int k = 0; k < kCopyBatch; ++k)
      if (v0 + 32 * k < nv) x[k] = __ldg(src + v0 + 32 * k);
#pragma unroll
    for (int k = 0; k < kCopyBatch; ++k)
      if (v0 + 32 * k < nv) __stcs(dst + v0 + 32 * k, x[k]);
  }
}

// One warp writes drafter row `dst` from target hidden row m (m >= 0, m < n_in_rows) or from
// h_shared (m < 0, or m out of range with SD_ERR_MAP_RANGE). vec: 16-byte aligned rows and H a
// multiple of 8.
__device__ __forceinline__ void gather_row_warp(long long m, const uint16_t* hidden, long ld_in,
                                                int n_in_rows, const uint16_t* h_shared,
                                                uint16_t* dst, int H, bool vec, int lane,
                                                int32_t& e) {
  const uint16_t* src = h_shared;
  if (m >= 0) {
    if (m < n_in_rows) src = hidden + m * ld_in;
    else if (lane == 0) e |= SD_ERR_MAP_RANGE;
  }
  if (vec) {
    copy_row_warp(reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), H >> 3,
                  lane);
  } else {
    for (int x = lane; x < H; x += 32) dst[x] = __ldg(src + x);
  }
}

}  // namespace sdk
