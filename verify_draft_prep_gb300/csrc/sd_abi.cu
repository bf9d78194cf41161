// sd_abi.cu -- the exported C entry points of libsd_gb300: host-side argument checks, then one
// asynchronous launch on the caller's stream. See include/sd.h for the contract of each call.

#include <cuda_runtime.h>
#include <stdint.h>

#include "sd.h"

extern "C" {
int sd_verify_launch(int, int, int, int, const void*, long, const void*, long, const int32_t*,
                     const int32_t*, const float*, uint64_t, uint32_t, int32_t*, int32_t*, float*,
                     float*, void*, int32_t*, cudaStream_t);
size_t sd_verify_workspace_launch(int);
int sd_verify_noalloc_launch(int, int, int, int, const void*, long, const void*, long,
                             const int32_t*, const float*, uint64_t, uint32_t, int32_t*, int32_t*,
                             float*, float*, int32_t*, cudaStream_t);
int sd_verify_kernel_count(int, int, int, int);
int sd_sample_launch(int, int, int, int, const void*, long, const float*, uint64_t, uint32_t,
                     int32_t*, int32_t*, cudaStream_t);
int sd_prep_launch(int, int, const int32_t*, const int32_t*, const int32_t*, const int32_t*,
                   const int32_t*, int, int, int32_t, int, int32_t*, int32_t*, int32_t*, int32_t*,
                   uint8_t*, uint8_t*, int32_t*, int32_t*, int32_t*, int, const void*, long, int,
                   const void*, void*, long, int32_t*, cudaStream_t);
int sd_prep_padded_launch(int, int, const int32_t*, const int32_t*, const int32_t*,
                          const int32_t*, int, int, int32_t, int32_t*, int32_t*, int32_t*,
                          int32_t*, uint8_t*, uint8_t*, int32_t*, int32_t*, int, const void*, long,
                          int, const void*, void*, long, int32_t*, cudaStream_t);
int sd_gather_launch(int, int, const int32_t*, const int32_t*, const void*, long, int,
                     const void*, void*, long, int32_t*, cudaStream_t);
int sd_philox_launch(int, const uint32_t*, uint64_t, uint32_t*, cudaStream_t);
int sd_race_E_launch(int, const uint32_t*, float*, cudaStream_t);
int sd_approx_error_launch(uint32_t, uint64_t, float*, cudaStream_t);
int sd_E_check_launch(uint32_t, uint64_t, unsigned long long*, cudaStream_t);
int sd_verify_prepare_launch(int, int, int, int, const void*, long, const void*, long,
                             const int32_t*, const int32_t*, const float*, uint64_t, uint32_t,
                             int32_t*, int32_t*,
                             float*, float*, const int32_t*, const int32_t*, int, int, int32_t,
                             int, int32_t*, int32_t*, int32_t*, int32_t*, uint8_t*, uint8_t*,
                             int32_t*, int32_t*, int32_t*, int, const void*, long, int,
                             const void*, void*, long, void*, int32_t*, cudaStream_t);
int sd_verify_prepare_withheld_launch(int, uint32_t, int, int, int, int, const void*, long,
                                      const void*, long, const int32_t*, const int32_t*,
                                      const float*, uint64_t, uint32_t, int32_t*, int32_t*,
                                      float*, float*, const int32_t*, const int32_t*, int, int,
                                      int32_t, int, int32_t*, int32_t*, int32_t*, int32_t*,
                                      uint8_t*, uint8_t*, int32_t*, int32_t*, int32_t*, int,
                                      const void*, long, int, const void*, void*, long, void*,
                                      int32_t*, cudaStream_t);
int sd_verify_prepare_kernel_count(int, int, int, int, int);
int sd_verify_prepare_padded_launch(int, int, int, int, const void*, long, const void*, long,
                                    const int32_t*, const float*, uint64_t, uint32_t, int32_t*,
                                    int32_t*, float*, float*, const int32_t*, const int32_t*, int,
                                    int, int32_t, int32_t*, int32_t*, int32_t*, int32_t*,
                                    uint8_t*, uint8_t*, int32_t*, int32_t*, int, const void*, long,
                                    int, const void*, void*, long, void*, int32_t*, cudaStream_t);
}

namespace {

constexpr int kMaxDevices = 64;
int g_device_ok[kMaxDevices];  // 0 unknown, 1 sm_103, -1 other

// The kernels are built for sm_103a only.
int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return SD_E_DEVICE;
  if (dev < kMaxDevices && g_device_ok[dev] != 0) return g_device_ok[dev] > 0 ? SD_OK : SD_E_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return SD_E_DEVICE;
  const int ok = (major == 10 && minor == 3) ? 1 : -1;
  if (dev < kMaxDevices) g_device_ok[dev] = ok;
  return ok > 0 ? SD_OK : SD_E_DEVICE;
}

}  // namespace

extern "C" {

int sd_version(void) { return 100; }

const char* sd_status_string(int status) {
  switch (status) {
    case SD_OK: return "ok";
    case SD_E_NULL: return "a required pointer is NULL";
    case SD_E_SHAPE: return "a size or stride is out of range";
    case SD_E_DTYPE: return "unknown dtype";
    case SD_E_ALIGN: return "a pointer or stride breaks the required alignment";
    case SD_E_LAUNCH: return "CUDA launch failed";
    case SD_E_DEVICE: return "the current device is not an sm_103 GPU";
    case SD_E_NOALLOC_LIMIT:
      return "B exceeds the fixed scratch of sd_verify_noalloc (SD_VERIFY_NOALLOC_MAX_B requests)";
    default: return "unknown status";
  }
}

size_t sd_verify_workspace_bytes(int B, int K, int V, int dtype) {
  (void)K;
  (void)V;
  (void)dtype;
  return B > 0 ? sd_verify_workspace_launch(B) : 0;
}

int sd_verify_kernels(int B, int V, int dtype, int has_temperature) {
  if (dtype != SD_F32_PROBS && dtype != SD_BF16_LOGITS) return SD_E_DTYPE;
  if (B < 0 || V < 1) return SD_E_SHAPE;
  if (B == 0) return 0;
  const int dev = check_device();
  if (dev != SD_OK) return dev;
  return sd_verify_kernel_count(B, V, dtype, has_temperature);
}

int sd_verify(int B, int K, int V, int dtype, const void* target, long ld_t, const void* draft,
              long ld_d, const int32_t* drafts, const float* temperature, uint64_t seed,
              uint32_t request_base, int32_t* out_tokens, int32_t* num_accepted,
              float* p_at_draft, float* q_at_draft, void* workspace, size_t workspace_bytes,
              int32_t* err, void* stream) {
  if (dtype != SD_F32_PROBS && dtype != SD_BF16_LOGITS) return SD_E_DTYPE;
  if (B < 0 || K < 1 || K > SD_K_MAX || V < 1 || ld_t < V || ld_d < V) return SD_E_SHAPE;
  if ((long long)B * (K + 1) > 2147483647LL) return SD_E_SHAPE;
  if ((unsigned long long)request_base + (unsigned long long)B > 4294967296ULL) return SD_E_SHAPE;
  if (B == 0) return SD_OK;
  if (!target || !draft || !drafts || !out_tokens || !num_accepted || !workspace) return SD_E_NULL;
  if (workspace_bytes < sd_verify_workspace_bytes(B, K, V, dtype)) return SD_E_SHAPE;
  const int esize = dtype == SD_F32_PROBS ? 4 : 2;
  if ((uintptr_t)target % esize || (uintptr_t)draft % esize) return SD_E_ALIGN;
  if ((uintptr_t)workspace % 16) return SD_E_ALIGN;
  const int dev = check_device();
  if (dev != SD_OK) return dev;
  return sd_verify_launch(B, K, V, dtype, target, ld_t, draft, ld_d, drafts, nullptr,
                          temperature, seed, request_base, out_tokens, num_accepted, p_at_draft,
                          q_at_draft, workspace, err, (cudaStream_t)stream);
}

int sd_verify_ragged(int B, int K_max, int V, int dtype, const void* target, long ld_t,
                     const void* draft, long ld_d, const int32_t* drafts,
                     const int32_t* cu_drafts, const float* temperature, uint64_t seed,
                     uint32_t request_base, int32_t* out_tokens, int32_t* num_accepted,
                     float* p_at_draft, float* q_at_draft, void* workspace,
                     size_t workspace_bytes, int32_t* err, void* stream) {
  if (dtype != SD_F32_PROBS && dtype != SD_BF16_LOGITS) return SD_E_DTYPE;
  if (B < 0 || K_max < 1 || K_max > SD_K_MAX || V < 1 || ld_t < V || ld_d < V)
    return SD_E_SHAPE;
  if ((long long)B * (K_max + 1) > 2147483647LL) return SD_E_SHAPE;
  if ((unsigned long long)request_base + (unsigned long long)B > 4294967296ULL) return SD_E_SHAPE;
  if (B == 0) return SD_OK;
  if (!target || !draft || !drafts || !cu_drafts || !out_tokens || !num_accepted || !workspace)
    return SD_E_NULL;
  if (workspace_bytes < sd_verify_workspace_bytes(B, K_max, V, dtype)) return SD_E_SHAPE;
  const int esize = dtype == SD_F32_PROBS ? 4 : 2;
  if ((uintptr_t)target % esize || (uintptr_t)draft % esize) return SD_E_ALIGN;
  if ((uintptr_t)workspace % 16) return SD_E_ALIGN;
  const int dev = check_device();
  if (dev != SD_OK) return dev;
  return sd_verify_launch(B, K_max, V, dtype, target, ld_t, draft, ld_d, drafts, cu_drafts,
                          temperature, seed, request_base, out_tokens, num_accepted, p_at_draft,
                          q_at_draft, workspace, err, (cudaStream_t)stream);
}

int sd_draft_sample(int B, int K, int V, int dtype, const void* rows, long ld,
                    const float* temperature, uint64_t seed, uint32_t request_base,
                    int32_t* drafts, int32_t* err, void* stream) {
  if (dtype != SD_F32_PROBS && dtype != SD_BF16_LOGITS) return SD_E_DTYPE;
  if (B < 0 || K < 1 || K > SD_K_MAX || V < 1 || ld < V) return SD_E_SHAPE;
  // B*K rows of up to 8 CTAs each
  if ((long long)B * K * 8 > 2147483647LL) return SD_E_SHAPE;
  if ((unsigned long long)request_base + (unsigned long long)B > 4294967296ULL) return SD_E_SHAPE;
  if (B == 0) return SD_OK;
  if (!rows || !drafts) return SD_E_NULL;
  const int esize = dtype == SD_F32_PROBS ? 4 : 2;
  if ((uintptr_t)rows % esize) return SD_E_ALIGN;
  const int dev = check_device();
  if (dev != SD_OK) return dev;
  return sd_sample_launch(B, K, V, dtype, rows, ld, temperature, seed, request_base, drafts, err,
                          (cudaStream_t)stream);
}

int sd_verify_noalloc(int B, int K, int V, int dtype, const void* target, long ld_t,
                      const void* draft, long ld_d, const int32_t* drafts,
                      const float* temperature, uint64_t seed, uint32_t request_base,
                      int32_t* out_tokens, int32_t* num_accepted, float* p_at_draft,
                      float* q_at_draft, int32_t* err, void* stream) {
  if (dtype != SD_F32_PROBS && dtype != SD_BF16_LOGITS) return SD_E_DTYPE;
  if (B < 0 || K < 1 || K > SD_K_MAX || V < 1 || ld_t < V || ld_d < V) return SD_E_SHAPE;
  if (B > SD_VERIFY_NOALLOC_MAX_B) return SD_E_NOALLOC_LIMIT;
  if ((unsigned long long)request_base + (unsigned long long)B > 4294967296ULL) return SD_E_SHAPE;
  if (B == 0) return SD_OK;
  if (!target || !draft || !drafts || !out_tokens || !num_accepted) return SD_E_NULL;
  const int esize = dtype == SD_F32_PROBS ? 4 : 2;
  if ((uintptr_t)target % esize || (uintptr_t)draft % esize) return SD_E_ALIGN;
  const int dev = check_device();
  if (dev != SD_OK) return dev;
  return sd_verify_noalloc_launch(B, K, V, dtype, target, ld_t, draft, ld_d, drafts, temperature,
                                  seed, request_base, out_tokens, num_accepted, p_at_draft,
                                  q_at_draft, err, (cudaStream_t)stream);
}

namespace {

int check_expand_args(int B, int K, const int32_t* out_tokens, const int32_t* num_accepted,
                      const int32_t* pos0, const int32_t* block_table, int max_blocks,
                      int block_size, int capacity, int32_t* input_ids, int32_t* positions,
                      int32_t* slot_mapping, int32_t* hidden_map, uint8_t* is_masked,
                      uint8_t* is_rejected, int32_t* start_loc, int32_t* new_token_idx,
                      int32_t* total_out) {
  if (B < 0 || K < 1 || K > SD_K_MAX || max_blocks < 0 || block_size < 1 || capacity < 0)
    return SD_E_SHAPE;
  if ((long long)B * 2 * K > 2147483647LL) return SD_E_SHAPE;
  if (!start_loc || !total_out) return SD_E_NULL;
  if (B > 0 && (!out_tokens || !num_accepted || !pos0 || !is_rejected || !new_token_idx ||
                (max_blocks > 0 && !block_table)))
    return SD_E_NULL;
  if (capacity > 0 && (!input_ids || !positions || !slot_mapping || !hidden_map || !is_masked))
    return SD_E_NULL;
  return SD_OK;
}

}  // namespace

int sd_pdraft_expand(int B, int K, const int32_t* out_tokens, const int32_t* num_accepted,
                     const int32_t* pos0, const int32_t* block_table, int max_blocks,
                     int block_size, int32_t mask_token_id, int capacity, int32_t* input_ids,
                     int32_t* positions, int32_t* slot_mapping, int32_t* hidden_map,
                     uint8_t* is_masked, uint8_t* is_rejected, int32_t* start_loc,
                     int32_t* new_token_idx, int32_t* total_out, int32_t* err, void* stream) {
  int rc = check_expand_args(B, K, out_tokens, num_accepted, pos0, block_table, max_blocks,
                             block_size, capacity, input_ids, positions, slot_mapping, hidden_map,
                             is_masked, is_rejected, start_loc, new_token_idx, total_out);
  if (rc != SD_OK) return rc;
  rc = check_device();
  if (rc != SD_OK) return rc;
  return sd_prep_launch(B, K, out_tokens, num_accepted, nullptr, pos0, block_table, max_blocks,
                        block_size, mask_token_id, capacity, input_ids, positions, slot_mapping,
                        hidden_map, is_masked, is_rejected, start_loc, new_token_idx, total_out,
                        0, nullptr, 0, 0, nullptr, nullptr, 0, err, (cudaStream_t)stream);
}

namespace {
int prepare(int B, int K, const int32_t* out_tokens, const int32_t* num_accepted,
            const int32_t* cu_drafts, const int32_t* pos0, const int32_t* block_table,
            int max_blocks, int block_size, int32_t mask_token_id, int capacity,
            int32_t* input_ids, int32_t* positions, int32_t* slot_mapping, int32_t* hidden_map,
            uint8_t* is_masked, uint8_t* is_rejected, int32_t* start_loc, int32_t* new_token_idx,
            int32_t* total_out, int H, const void* target_hidden, long ld_in, int n_in_rows,
            const void* h_shared, void* out_hidden, long ld_out, int32_t* err, void* stream) {
  int rc = check_expand_args(B, K, out_tokens, num_accepted, pos0, block_table, max_blocks,
                             block_size, capacity, input_ids, positions, slot_mapping, hidden_map,
                             is_masked, is_rejected, start_loc, new_token_idx, total_out);
  if (rc != SD_OK) return rc;
  if (H < 1 || ld_in < H || ld_out < H || n_in_rows < 0) return SD_E_SHAPE;
  if (!h_shared || (capacity > 0 && !out_hidden) || (n_in_rows > 0 && !target_hidden))
    return SD_E_NULL;
  if ((uintptr_t)target_hidden % 2 || (uintptr_t)h_shared % 2 || (uintptr_t)out_hidden % 2)
    return SD_E_ALIGN;
  rc = check_device();
  if (rc != SD_OK) return rc;
  if (capacity == 0) out_hidden = nullptr;
  return sd_prep_launch(B, K, out_tokens, num_accepted, cu_drafts, pos0, block_table,
                        max_blocks, block_size, mask_token_id, capacity, input_ids, positions,
                        slot_mapping, hidden_map, is_masked, is_rejected, start_loc,
                        new_token_idx, total_out, H, target_hidden, ld_in, n_in_rows, h_shared,
                        out_hidden, ld_out, err, (cudaStream_t)stream);
}
}  // namespace

int sd_pdraft_prepare(int B, int K, const int32_t* out_tokens, const int32_t* num_accepted,
                      const int32_t* pos0, const int32_t* block_table, int max_blocks,
                      int block_size, int32_t mask_token_id, int capacity, int32_t* input_ids,
                      int32_t* positions, int32_t* slot_mapping, int32_t* hidden_map,
                      uint8_t* is_masked, uint8_t* is_rejected, int32_t* start_loc,
                      int32_t* new_token_idx, int32_t* total_out, int H,
                      const void* target_hidden, long ld_in, int n_in_rows, const void* h_shared,
                      void* out_hidden, long ld_out, int32_t* err, void* stream) {
  return prepare(B, K, out_tokens, num_accepted, nullptr, pos0, block_table, max_blocks,
                 block_size, mask_token_id, capacity, input_ids, positions, slot_mapping,
                 hidden_map, is_masked, is_rejected, start_loc, new_token_idx, total_out, H,
                 target_hidden, ld_in, n_in_rows, h_shared, out_hidden, ld_out, err, stream);
}

int sd_pdraft_prepare_ragged(int B, int K_max, const int32_t* out_tokens,
                             const int32_t* num_accepted, const int32_t* cu_drafts,
                             const int32_t* pos0, const int32_t* block_table, int max_blocks,
                             int block_size, int32_t mask_token_id, int capacity,
                             int32_t* input_ids, int32_t* positions, int32_t* slot_mapping,
                             int32_t* hidden_map, uint8_t* is_masked, uint8_t* is_rejected,
                             int32_t* start_loc, int32_t* new_token_idx, int32_t* total_out,
                             int H, const void* target_hidden, long ld_in, int n_in_rows,
                             const void* h_shared, void* out_hidden, long ld_out, int32_t* err,
                             void* stream) {
  if (B > 0 && !cu_drafts) return SD_E_NULL;
  return prepare(B, K_max, out_tokens, num_accepted, cu_drafts, pos0, block_table, max_blocks,
                 block_size, mask_token_id, capacity, input_ids, positions, slot_mapping,
                 hidden_map, is_masked, is_rejected, start_loc, new_token_idx, total_out, H,
                 target_hidden, ld_in, n_in_rows, h_shared, out_hidden, ld_out, err, stream);
}

int sd_pdraft_prepare_padded(int B, int K, const int32_t* out_tokens,
                             const int32_t* num_accepted, const int32_t* pos0,
                             const int32_t* block_table, int max_blocks, int block_size,
                             int32_t mask_token_id, int32_t* input_ids, int32_t* positions,
                             int32_t* slot_mapping, int32_t* hidden_map, uint8_t* is_masked,
                             uint8_t* rejected, int32_t* scatter_map, int32_t* new_token_idx,
                             int H, const void* target_hidden, long ld_in, int n_in_rows,
                             const void* h_shared, void* out_hidden, long ld_out, int32_t* err,
                             void* stream) {
  if (B < 0 || K < 1 || K > SD_K_MAX || max_blocks < 0 || block_size < 1) return SD_E_SHAPE;
  if ((long long)B * 2 * K > 2147483647LL) return SD_E_SHAPE;
  if (B == 0) return SD_OK;
  if (!out_tokens || !num_accepted || !pos0 || (max_blocks > 0 && !block_table) || !input_ids ||
      !positions || !slot_mapping || !hidden_map || !is_masked || !rejected || !scatter_map ||
      !new_token_idx)
    return SD_E_NULL;
  if (out_hidden) {
    if (H < 1 || ld_in < H || ld_out < H || n_in_rows < 0) return SD_E_SHAPE;
    if (!h_shared || (n_in_rows > 0 && !target_hidden)) return SD_E_NULL;
    if ((uintptr_t)target_hidden % 2 || (uintptr_t)h_shared % 2 || (uintptr_t)out_hidden % 2)
      return SD_E_ALIGN;
  }
  const int rc = check_device();
  if (rc != SD_OK) return rc;
  return sd_prep_padded_launch(B, K, out_tokens, num_accepted, pos0, block_table, max_blocks,
                               block_size, mask_token_id, input_ids, positions, slot_mapping,
                               hidden_map, is_masked, rejected, scatter_map, new_token_idx, H,
                               target_hidden, ld_in, n_in_rows, h_shared, out_hidden, ld_out, err,
                               (cudaStream_t)stream);
}

int sd_hidden_gather(int capacity, int H, const int32_t* total_out, const int32_t* hidden_map,
                     const void* target_hidden, long ld_in, int n_in_rows, const void* h_shared,
                     void* out_hidden, long ld_out, int32_t* err, void* stream) {
  if (capacity < 0 || H < 1 || ld_in < H || ld_out < H || n_in_rows < 0) return SD_E_SHAPE;
  if (!total_out || !h_shared) return SD_E_NULL;
  if (capacity > 0 && (!hidden_map || !out_hidden)) return SD_E_NULL;
  if (n_in_rows > 0 && !target_hidden) return SD_E_NULL;
  if ((uintptr_t)target_hidden % 2 || (uintptr_t)h_shared % 2 || (uintptr_t)out_hidden % 2)
    return SD_E_ALIGN;
  const int dev = check_device();
  if (dev != SD_OK) return dev;
  return sd_gather_launch(capacity, H, total_out, hidden_map, target_hidden, ld_in, n_in_rows,
                          h_shared, out_hidden, ld_out, err, (cudaStream_t)stream);
}

int sd_philox_words(int n, const uint32_t* ctr, uint64_t seed, uint32_t* out, void* stream) {
  if (n < 0) return SD_E_SHAPE;
  if (n > 0 && (!ctr || !out)) return SD_E_NULL;
  const int dev = check_device();
  if (dev != SD_OK) return dev;
  return sd_philox_launch(n, ctr, seed, out, (cudaStream_t)stream);
}

int sd_race_E(int n, const uint32_t* w, float* E, void* stream) {
  if (n < 0) return SD_E_SHAPE;
  if (n > 0 && (!w || !E)) return SD_E_NULL;
  const int dev = check_device();
  if (dev != SD_OK) return dev;
  return sd_race_E_launch(n, w, E, (cudaStream_t)stream);
}

int sd_race_E_approx_error(uint32_t w_begin, uint64_t count, float* max_rel, void* stream) {
  if (count > (1ull << 32)) return SD_E_SHAPE;
  if (!max_rel) return SD_E_NULL;
  const int dev = check_device();
  if (dev != SD_OK) return dev;
  return sd_approx_error_launch(w_begin, count, max_rel, (cudaStream_t)stream);
}

int sd_race_E_check(uint32_t w_begin, uint64_t count, uint64_t* counts, void* stream) {
  if (count > (1ull << 32)) return SD_E_SHAPE;
  if (!counts) return SD_E_NULL;
  const int dev = check_device();
  if (dev != SD_OK) return dev;
  return sd_E_check_launch(w_begin, count, reinterpret_cast<unsigned long long*>(counts),
                           (cudaStream_t)stream);
}

size_t sd_verify_prepare_workspace_bytes(int B) {
  return B > 0 ? sd_verify_workspace_launch(B) : 0;
}

int sd_verify_prepare_kernels(int B, int K, int V, int dtype, int has_temperature) {
  if (dtype != SD_F32_PROBS && dtype != SD_BF16_LOGITS) return SD_E_DTYPE;
  if (B < 0 || K < 1 || K > SD_K_MAX || V < 1) return SD_E_SHAPE;
  if (B == 0) return 0;
  const int dev = check_device();
  if (dev != SD_OK) return dev;
  return sd_verify_prepare_kernel_count(B, K, V, dtype, has_temperature);
}

}  // extern "C"

namespace {
// sd_verify_prepare and sd_verify_prepare_ragged (cu_drafts NULL: K drafts per request).
int verify_prepare(int B, int K, int V, int dtype, const void* target, long ld_t,
                   const void* draft, long ld_d, const int32_t* drafts, const int32_t* cu_drafts,
                   const float* temperature, uint64_t seed, uint32_t request_base,
                   int32_t* out_tokens, int32_t* num_accepted, float* p_at_draft,
                   float* q_at_draft, const int32_t* pos0, const int32_t* block_table,
                   int max_blocks, int block_size, int32_t mask_token_id, int capacity,
                   int32_t* input_ids, int32_t* positions, int32_t* slot_mapping,
                   int32_t* hidden_map, uint8_t* is_masked, uint8_t* is_rejected,
                   int32_t* start_loc, int32_t* new_token_idx, int32_t* total_out, int H,
                   const void* target_hidden, long ld_in, int n_in_rows, const void* h_shared,
                   void* out_hidden, long ld_out, void* workspace, size_t workspace_bytes,
                   int32_t* err, void* stream, int withhold = -1, uint32_t wait_us = 0) {
  // sd_verify's checks
  if (dtype != SD_F32_PROBS && dtype != SD_BF16_LOGITS) return SD_E_DTYPE;
  if (B < 0 || K < 1 || K > SD_K_MAX || V < 1 || ld_t < V || ld_d < V) return SD_E_SHAPE;
  if ((long long)B * (K + 1) > 2147483647LL) return SD_E_SHAPE;
  if ((unsigned long long)request_base + (unsigned long long)B > 4294967296ULL) return SD_E_SHAPE;
  // sd_pdraft_prepare's checks (on this call's own out_tokens / num_accepted)
  int rc = check_expand_args(B, K, out_tokens, num_accepted, pos0, block_table, max_blocks,
                             block_size, capacity, input_ids, positions, slot_mapping, hidden_map,
                             is_masked, is_rejected, start_loc, new_token_idx, total_out);
  if (rc != SD_OK) return rc;
  if (H < 1 || ld_in < H || ld_out < H || n_in_rows < 0) return SD_E_SHAPE;
  if (!h_shared || (capacity > 0 && !out_hidden) || (n_in_rows > 0 && !target_hidden))
    return SD_E_NULL;
  if ((uintptr_t)target_hidden % 2 || (uintptr_t)h_shared % 2 || (uintptr_t)out_hidden % 2)
    return SD_E_ALIGN;
  if (B == 0) {
    // no request: the rebuild still reports an empty batch
    rc = check_device();
    if (rc != SD_OK) return rc;
    return sd_prep_launch(0, K, out_tokens, num_accepted, cu_drafts, pos0, block_table, max_blocks,
                          block_size, mask_token_id, capacity, input_ids, positions,
                          slot_mapping, hidden_map, is_masked, is_rejected, start_loc,
                          new_token_idx, total_out, H, target_hidden, ld_in, n_in_rows, h_shared,
                          capacity == 0 ? nullptr : out_hidden, ld_out, err,
                          (cudaStream_t)stream);
  }
  if (!target || !draft || !drafts || !workspace) return SD_E_NULL;
  if (workspace_bytes < sd_verify_prepare_workspace_bytes(B)) return SD_E_SHAPE;
  const int esize = dtype == SD_F32_PROBS ? 4 : 2;
  if ((uintptr_t)target % esize || (uintptr_t)draft % esize) return SD_E_ALIGN;
  if ((uintptr_t)workspace % 16) return SD_E_ALIGN;
  rc = check_device();
  if (rc != SD_OK) return rc;
  if (withhold >= 0)
    return sd_verify_prepare_withheld_launch(
        withhold, wait_us, B, K, V, dtype, target, ld_t, draft, ld_d, drafts, cu_drafts,
        temperature, seed, request_base, out_tokens, num_accepted, p_at_draft, q_at_draft, pos0,
        block_table, max_blocks, block_size, mask_token_id, capacity, input_ids, positions,
        slot_mapping, hidden_map, is_masked, is_rejected, start_loc, new_token_idx, total_out, H,
        target_hidden, ld_in, n_in_rows, h_shared, capacity == 0 ? nullptr : out_hidden, ld_out,
        workspace, err, (cudaStream_t)stream);
  return sd_verify_prepare_launch(B, K, V, dtype, target, ld_t, draft, ld_d, drafts, cu_drafts,
                                  temperature, seed, request_base, out_tokens, num_accepted,
                                  p_at_draft, q_at_draft, pos0, block_table, max_blocks, block_size,
                                  mask_token_id, capacity, input_ids, positions, slot_mapping,
                                  hidden_map, is_masked, is_rejected, start_loc, new_token_idx,
                                  total_out, H, target_hidden, ld_in, n_in_rows, h_shared,
                                  capacity == 0 ? nullptr : out_hidden, ld_out, workspace, err,
                                  (cudaStream_t)stream);
}

}  // namespace

extern "C" {
int sd_verify_prepare(int B, int K, int V, int dtype, const void* target, long ld_t,
                      const void* draft, long ld_d, const int32_t* drafts,
                      const float* temperature, uint64_t seed, uint32_t request_base,
                      int32_t* out_tokens, int32_t* num_accepted, float* p_at_draft,
                      float* q_at_draft, const int32_t* pos0, const int32_t* block_table,
                      int max_blocks, int block_size, int32_t mask_token_id, int capacity,
                      int32_t* input_ids, int32_t* positions, int32_t* slot_mapping,
                      int32_t* hidden_map, uint8_t* is_masked, uint8_t* is_rejected,
                      int32_t* start_loc, int32_t* new_token_idx, int32_t* total_out, int H,
                      const void* target_hidden, long ld_in, int n_in_rows,
                      const void* h_shared, void* out_hidden, long ld_out, void* workspace,
                      size_t workspace_bytes, int32_t* err, void* stream) {
  return verify_prepare(B, K, V, dtype, target, ld_t, draft, ld_d, drafts, nullptr, temperature,
                        seed, request_base, out_tokens, num_accepted, p_at_draft, q_at_draft,
                        pos0, block_table, max_blocks, block_size, mask_token_id, capacity,
                        input_ids, positions, slot_mapping, hidden_map, is_masked, is_rejected,
                        start_loc, new_token_idx, total_out, H, target_hidden, ld_in, n_in_rows,
                        h_shared, out_hidden, ld_out, workspace, workspace_bytes, err, stream);
}

int sd_diag_verify_prepare_withheld(int withhold_request, uint32_t wait_us, int B, int K, int V,
                                    int dtype, const void* target, long ld_t, const void* draft,
                                    long ld_d, const int32_t* drafts, const float* temperature,
                                    uint64_t seed, uint32_t request_base, int32_t* out_tokens,
                                    int32_t* num_accepted, float* p_at_draft, float* q_at_draft,
                                    const int32_t* pos0, const int32_t* block_table,
                                    int max_blocks, int block_size, int32_t mask_token_id,
                                    int capacity, int32_t* input_ids, int32_t* positions,
                                    int32_t* slot_mapping, int32_t* hidden_map,
                                    uint8_t* is_masked, uint8_t* is_rejected,
                                    int32_t* start_loc, int32_t* new_token_idx,
                                    int32_t* total_out, int H, const void* target_hidden,
                                    long ld_in, int n_in_rows, const void* h_shared,
                                    void* out_hidden, long ld_out, void* workspace,
                                    size_t workspace_bytes, int32_t* err, void* stream) {
  if (withhold_request < 0 || withhold_request >= B || wait_us < 1 || wait_us > 1000000)
    return SD_E_SHAPE;
  return verify_prepare(B, K, V, dtype, target, ld_t, draft, ld_d, drafts, nullptr, temperature,
                        seed, request_base, out_tokens, num_accepted, p_at_draft, q_at_draft,
                        pos0, block_table, max_blocks, block_size, mask_token_id, capacity,
                        input_ids, positions, slot_mapping, hidden_map, is_masked, is_rejected,
                        start_loc, new_token_idx, total_out, H, target_hidden, ld_in, n_in_rows,
                        h_shared, out_hidden, ld_out, workspace, workspace_bytes, err, stream,
                        withhold_request, wait_us);
}

int sd_verify_prepare_ragged(int B, int K_max, int V, int dtype, const void* target, long ld_t,
                             const void* draft, long ld_d, const int32_t* drafts,
                             const int32_t* cu_drafts, const float* temperature, uint64_t seed,
                             uint32_t request_base, int32_t* out_tokens, int32_t* num_accepted,
                             float* p_at_draft, float* q_at_draft, const int32_t* pos0,
                             const int32_t* block_table, int max_blocks, int block_size,
                             int32_t mask_token_id, int capacity, int32_t* input_ids,
                             int32_t* positions, int32_t* slot_mapping, int32_t* hidden_map,
                             uint8_t* is_masked, uint8_t* is_rejected, int32_t* start_loc,
                             int32_t* new_token_idx, int32_t* total_out, int H,
                             const void* target_hidden, long ld_in, int n_in_rows,
                             const void* h_shared, void* out_hidden, long ld_out,
                             void* workspace, size_t workspace_bytes, int32_t* err,
                             void* stream) {
  if (B > 0 && !cu_drafts) return SD_E_NULL;
  return verify_prepare(B, K_max, V, dtype, target, ld_t, draft, ld_d, drafts, cu_drafts,
                        temperature, seed, request_base, out_tokens, num_accepted, p_at_draft,
                        q_at_draft, pos0, block_table, max_blocks, block_size, mask_token_id,
                        capacity, input_ids, positions, slot_mapping, hidden_map, is_masked,
                        is_rejected, start_loc, new_token_idx, total_out, H, target_hidden,
                        ld_in, n_in_rows, h_shared, out_hidden, ld_out, workspace,
                        workspace_bytes, err, stream);
}

int sd_verify_prepare_padded(int B, int K, int V, int dtype, const void* target, long ld_t,
                             const void* draft, long ld_d, const int32_t* drafts,
                             const float* temperature, uint64_t seed, uint32_t request_base,
                             int32_t* out_tokens, int32_t* num_accepted, float* p_at_draft,
                             float* q_at_draft, const int32_t* pos0, const int32_t* block_table,
                             int max_blocks, int block_size, int32_t mask_token_id,
                             int32_t* input_ids, int32_t* positions, int32_t* slot_mapping,
                             int32_t* hidden_map, uint8_t* is_masked, uint8_t* rejected,
                             int32_t* scatter_map, int32_t* new_token_idx, int H,
                             const void* target_hidden, long ld_in, int n_in_rows,
                             const void* h_shared, void* out_hidden, long ld_out,
                             void* workspace, size_t workspace_bytes, int32_t* err, void* stream) {
  // sd_verify's checks
  if (dtype != SD_F32_PROBS && dtype != SD_BF16_LOGITS) return SD_E_DTYPE;
  if (B < 0 || K < 1 || K > SD_K_MAX || V < 1 || ld_t < V || ld_d < V) return SD_E_SHAPE;
  if ((long long)B * (K + 1) > 2147483647LL) return SD_E_SHAPE;
  if ((unsigned long long)request_base + (unsigned long long)B > 4294967296ULL) return SD_E_SHAPE;
  // sd_pdraft_prepare_padded's checks
  if (max_blocks < 0 || block_size < 1) return SD_E_SHAPE;
  if ((long long)B * 2 * K > 2147483647LL) return SD_E_SHAPE;
  if (B == 0) return SD_OK;
  if (!out_tokens || !num_accepted || !pos0 || (max_blocks > 0 && !block_table) || !input_ids ||
      !positions || !slot_mapping || !hidden_map || !is_masked || !rejected || !scatter_map ||
      !new_token_idx)
    return SD_E_NULL;
  if (out_hidden) {
    if (H < 1 || ld_in < H || ld_out < H || n_in_rows < 0) return SD_E_SHAPE;
    if (!h_shared || (n_in_rows > 0 && !target_hidden)) return SD_E_NULL;
    if ((uintptr_t)target_hidden % 2 || (uintptr_t)h_shared % 2 || (uintptr_t)out_hidden % 2)
      return SD_E_ALIGN;
  }
  if (!target || !draft || !drafts || !workspace) return SD_E_NULL;
  if (workspace_bytes < sd_verify_workspace_bytes(B, K, V, dtype)) return SD_E_SHAPE;
  const int esize = dtype == SD_F32_PROBS ? 4 : 2;
  if ((uintptr_t)target % esize || (uintptr_t)draft % esize) return SD_E_ALIGN;
  if ((uintptr_t)workspace % 16) return SD_E_ALIGN;
  const int rc = check_device();
  if (rc != SD_OK) return rc;
  return sd_verify_prepare_padded_launch(
      B, K, V, dtype, target, ld_t, draft, ld_d, drafts, temperature, seed, request_base,
      out_tokens, num_accepted, p_at_draft, q_at_draft, pos0, block_table, max_blocks, block_size,
      mask_token_id, input_ids, positions, slot_mapping, hidden_map, is_masked, rejected,
      scatter_map, new_token_idx, H, target_hidden, ld_in, n_in_rows, h_shared, out_hidden,
      ld_out, workspace, err, (cudaStream_t)stream);
}

}  // extern "C"
