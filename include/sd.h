/*
 * sd.h -- C ABI of the GB300 (sm_103a) speculative-decoding verify and P-EAGLE draft-batch
 * rebuild library (libsd_gb300.so).
 *
 * Three calls make one decoding step's hot path, in this order on one stream:
 *   sd_verify         lossless verification of K drafts per request (rejection sampling with a
 *                     residual resample, or greedy argmax at temperature 0);
 *   sd_pdraft_expand  rebuild of the drafter batch for the next parallel-drafting pass;
 *   sd_hidden_gather  drafter hidden states from the target's hidden states or h_shared.
 *
 * Conventions for every call:
 *   - Every pointer is a DEVICE pointer owned by the caller, or, for the read-only row inputs
 *     (target, draft, hidden states), host memory the GPU can address (page-locked or
 *     registered): the kernels then read over the host link only the parts the step needs.
 *     Outputs, the workspace and *err are device memory. The library allocates nothing and keeps
 *     no state between calls.
 *   - Calls only enqueue work on `stream` (a cudaStream_t; 0 = the legacy default stream) and
 *     never synchronise, so a step can be captured in a CUDA graph.
 *   - The return value is SD_OK or a negative SD_E_* code for errors the host can see (null
 *     pointer, bad size, misaligned pointer, launch failure). Nothing is enqueued on error.
 *   - Data errors found on the device (a draft token outside [0, V), a position the block table
 *     does not cover, ...) are OR-ed as SD_ERR_* bits into *err (a device int32 the caller
 *     zeroes; may be NULL). The kernel then takes the documented fallback. No kernel traps or
 *     asserts. One kernel waits on a value written by another CTA of the same launch: the
 *     single launch of sd_verify_prepare (see there), whose wait is bounded by time (20 ms on
 *     the GPU clock) and ends with SD_ERR_WAIT, never with a hang.
 *
 * Notation: B requests, K drafts per request (1 <= K <= SD_K_MAX), V vocabulary entries,
 * H hidden size. Target rows p_0..p_K of request r are rows r*(K+1)+j of `target`; draft rows
 * q_0..q_{K-1} are rows r*K+j of `draft`; draft d_{j+1} (drafts[r*K+j]) is checked against row j.
 */
#ifndef SD_GB300_H
#define SD_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SD_API __attribute__((visibility("default")))
#else
#define SD_API
#endif

#define SD_K_MAX 16

/* host-visible status codes */
#define SD_OK 0
#define SD_E_NULL (-1)     /* a required pointer is NULL */
#define SD_E_SHAPE (-2)    /* a size or stride is out of range */
#define SD_E_DTYPE (-3)    /* unknown dtype */
#define SD_E_ALIGN (-4)    /* a pointer or stride breaks the stated alignment */
#define SD_E_LAUNCH (-5)   /* the CUDA launch failed (cudaGetLastError is left set) */
#define SD_E_DEVICE (-6)   /* no usable sm_103 device is current */
#define SD_E_NOALLOC_LIMIT (-7) /* B > SD_VERIFY_NOALLOC_MAX_B for sd_verify_noalloc */

/* device-side data error bits, OR-ed into *err */
#define SD_ERR_TOKEN_RANGE 1    /* a draft token outside [0, V): treated as rejected */
#define SD_ERR_BLOCK_TABLE 2    /* drafter position not covered by the block table: slot -1 */
#define SD_ERR_NUM_ACCEPTED 4   /* num_accepted outside [0, K]: clamped */
#define SD_ERR_MAP_RANGE 8      /* hidden_map row >= n_in_rows: h_shared written instead */
#define SD_ERR_ZERO_ROW 16      /* a race row without a positive key even on p: token 0 */
#define SD_ERR_TOTAL_RANGE 32   /* total_out outside [0, capacity]: clamped */
#define SD_ERR_WAIT 64          /* sd_verify_prepare: a request's first drafter slot was not
                                   published within the bounded wait (20 ms); its final token is
                                   not written to input_ids */
#define SD_ERR_DRAFT_COUNT 128  /* cu_drafts gives a request a draft count outside [0, K_max]:
                                   clamped (sd_verify_ragged) */

/* input kinds for sd_verify */
#define SD_F32_PROBS 0    /* fp32 probabilities, already at the sampling temperature */
#define SD_BF16_LOGITS 1  /* bf16 logits; softmax(l / T_r) is taken inside the kernel */

/*
 * sd_verify -- batched lossless verification of K drafts per request.
 *
 * Speculative-decoding explainer (ainews.alishangtian.com), sections "核心思想" (verify K+1
 * positions, discard after the first rejection, K+1 tokens when all are accepted),
 * "修正拒绝采样" (accept with probability min(1, p(x)/q(x)); on rejection resample from the
 * normalised residual max(0, p - q)) and "边界与代价" (temperature 0 must equal greedy decoding).
 *
 * Per request r, with T_r = temperature[r] (NULL: every T_r = 1):
 *   T_r > 0: draft d_{j+1} is accepted iff u_j * Q < P, with P = p_j(d_{j+1}),
 *            Q = q_j(d_{j+1}), compared exactly in double, and u_j = (w >> 8) * 2^-24 where w
 *            is word 0 of Philox4x32-10 block (0, j, r, 0) under key (seed lo, seed hi).
 *            a_r = index of the first rejection, or K. The final token b_r is
 *              a_r < K:  argmax_x r(x) / E_x, r = max(0, p_{a_r} - q_{a_r}),
 *              a_r == K: argmax_x max(0, p_K(x)) / E_x   (the bonus token),
 *            with E_x = fp32(-log(v)) from the double log, v = (w + 0.5) * 2^-32 and w word
 *            (x & 3) of block (x >> 2, j, r, 1), j the race row. Keys are fp32 quotients for
 *            SD_F32_PROBS; ties go to the lowest x. If no key of the residual race is
 *            positive, the race is re-run on p of the same row with the same E_x; if that has
 *            none either, b_r = 0 and SD_ERR_ZERO_ROW is raised.
 *   T_r == 0: accept iff d_{j+1} == argmax_x p_j(x) (lowest x on ties); b_r = argmax p_{a_r}.
 * For SD_BF16_LOGITS, p_j = softmax(l^t_j / T_r) and q_j = softmax(l^d_j / T_r) are formed in
 * fp32 inside the kernel (results match a double-precision evaluation within the documented
 * tolerance, not bit for bit); T_r == 0 works on the raw logits (bit-exact).
 * Rows after the first rejection are never read.
 *
 * Arguments:
 *   B >= 0, 1 <= K <= SD_K_MAX, V >= 1; dtype SD_F32_PROBS or SD_BF16_LOGITS.
 *   target [B*(K+1) rows, stride ld_t elements], draft [B*K rows, stride ld_d elements]
 *     (fp32 or bf16 per dtype; ld >= V). Rows whose start is 16-byte aligned are read with
 *     128-bit loads, other layouts with scalar loads.
 *   drafts [B, K] int32; temperature [B] fp32 or NULL (every request samples at T = 1; for
 *     large probability rows the library then balances the race over the whole GPU);
 *   seed: Philox key; request_base: the request index that local request 0 has in the Philox
 *     counters (r in the blocks above is request_base + local index), so that a batch split
 *     over several GPUs by request draws exactly what one GPU would draw for the whole batch;
 *     request_base + B <= 2^32.
 * Outputs:
 *   out_tokens [B, K+1] int32: d_1..d_{a_r}, b_r, then -1.
 *   num_accepted [B] int32: a_r.
 *   p_at_draft, q_at_draft [B, K] fp32, each may be NULL: P and Q of every examined draft
 *     j <= min(a_r, K-1) (probabilities; raw target/draft values for T_r == 0; 0 for an
 *     out-of-range token), -1 for drafts never examined.
 *   workspace, workspace_bytes: device scratch of at least sd_verify_workspace_bytes(B, K, V,
 *     dtype) bytes, zeroed before first use and left zeroed by every call (see below).
 *   err: see above.
 */
SD_API int sd_verify(int B, int K, int V, int dtype, const void* target, long ld_t,
                     const void* draft, long ld_d, const int32_t* drafts,
                     const float* temperature, uint64_t seed, uint32_t request_base,
                     int32_t* out_tokens, int32_t* num_accepted, float* p_at_draft,
                     float* q_at_draft, void* workspace, size_t workspace_bytes, int32_t* err,
                     void* stream);

/*
 * sd_verify_ragged -- sd_verify with a number of drafts of its own for every request.
 *
 * Request r has K_r = cu_drafts[r+1] - cu_drafts[r] drafts (0 <= K_r <= K_max; cu_drafts is the
 * exclusive prefix [B+1] of the counts, on the device). Its rows are packed: target rows
 * p_0..p_{K_r} at rows cu_drafts[r] + r .. cu_drafts[r] + r + K_r of target, draft rows
 * q_0..q_{K_r - 1} and draft tokens at cu_drafts[r] .. of draft and drafts. Each request is
 * verified exactly as sd_verify verifies it with K = K_r (the same Philox counters: request
 * request_base + r, row j); K_r = 0 samples the bonus token from p_0 alone. Outputs keep the
 * stride of K_max: out_tokens [B, K_max+1] (-1 after b_r), p_at_draft / q_at_draft [B, K_max]
 * (-1 where no draft was examined). cu_drafts must be consistent with the arrays: rows are
 * addressed from its entries. A count outside [0, K_max] (a decreasing entry, a step beyond K_max)
 * is clamped and raises SD_ERR_DRAFT_COUNT; the rows it then addresses must still lie inside the
 * arrays. Other arguments, workspace and errors as for sd_verify (with K = K_max).
 */
SD_API int sd_verify_ragged(int B, int K_max, int V, int dtype, const void* target, long ld_t,
                            const void* draft, long ld_d, const int32_t* drafts,
                            const int32_t* cu_drafts, const float* temperature, uint64_t seed,
                            uint32_t request_base, int32_t* out_tokens, int32_t* num_accepted,
                            float* p_at_draft, float* q_at_draft, void* workspace,
                            size_t workspace_bytes, int32_t* err, void* stream);

/*
 * Size in bytes of the workspace sd_verify needs for B requests: 16 bytes per request, where the
 * CTAs that share a request's race row merge their results. The caller allocates it (16-byte
 * aligned) and zeroes it once; every sd_verify call leaves it zeroed again. Calls that may run
 * concurrently need separate workspaces.
 */
SD_API size_t sd_verify_workspace_bytes(int B, int K, int V, int dtype);

/*
 * Number of kernels one sd_verify (or sd_verify_noalloc) call with these sizes launches on the
 * current device: 0 for B == 0, else 1 (the cluster kernel, or for an all-sampled batch on large
 * probability rows the race kernel that balances the batch over every SM). A planning query for
 * callers that count launches (a CUDA-graph budget, a profiler filter); it launches nothing.
 * Returns a negative status for an unknown dtype or B < 0, V < 1.
 */
SD_API int sd_verify_kernels(int B, int V, int dtype, int has_temperature);

/*
 * sd_verify_noalloc -- sd_verify for callers that cannot allocate device memory. This call has
 * no counterpart in the method's sources; it exists for callers such as a plugin or engine
 * that is handed only its input and output buffers and may not call cudaMalloc (allocation
 * would stall or break the host runtime's memory pool, or happen inside a stream capture that
 * forbids it). Same arguments, semantics and results as sd_verify, minus the workspace: the
 * merge slots live in a fixed device array of SD_VERIFY_NOALLOC_MAX_B entries (16 bytes each)
 * that every GPU loading the library holds until the process exits.
 *   - B > SD_VERIFY_NOALLOC_MAX_B returns SD_E_NOALLOC_LIMIT and enqueues nothing.
 *   - The first call on a device looks the array's address up (cudaGetSymbolAddress) with that
 *     device current; make that first call before any stream capture.
 *   - Each call enqueues a clear of the slots it uses (one cudaMemsetAsync of B*16 bytes) and
 *     then the verify kernel: two stream operations, of which sd_verify_kernels counts only the
 *     kernel. It calls no allocator.
 *   - All calls on a device share the one array: calls that may overlap on the GPU (other
 *     streams, other host threads) race on it and must be serialised by the caller.
 */
#define SD_VERIFY_NOALLOC_MAX_B 4096
SD_API int sd_verify_noalloc(int B, int K, int V, int dtype, const void* target, long ld_t,
                             const void* draft, long ld_d, const int32_t* drafts,
                             const float* temperature, uint64_t seed, uint32_t request_base,
                             int32_t* out_tokens, int32_t* num_accepted, float* p_at_draft,
                             float* q_at_draft, int32_t* err, void* stream);

/*
 * sd_draft_sample -- the drafter's K new drafts per request, sampled from its output rows.
 *
 * P-EAGLE blog (vLLM), section "Triton Kernel": new_token_idx marks the drafter slots whose
 * logits become the next drafts; the drafter runs its head on those slots, giving one row per
 * (request, draft). Each row is sampled the way the verify step samples a bonus token
 * (speculative-decoding explainer, "修正拒绝采样": an exact sample of the row's distribution):
 * d_{k+1} of request r = argmax_x q(x) / E_x over row (r*K + k), E_x = fp32(-log((w + 0.5) 2^-32))
 * with w word (x & 3) of Philox4x32-10 block (x >> 2, k, request_base + r, 2) -- tag 2, a stream
 * separate from the verify races' tag 1 -- ties to the lowest x; temperature[r] == 0 takes the
 * argmax of the row (lowest x on ties).
 * Arguments:
 *   rows: [B*K, V] with row stride ld elements: SD_F32_PROBS probabilities (already at the
 *     sampling temperature; only temperature == 0 matters), or SD_BF16_LOGITS logits, sampled
 *     from softmax(l / temperature[r]) computed in the kernel.
 *   temperature: [B] fp32 or NULL (= 1); seed, request_base: as for sd_verify.
 *   drafts: [B, K] int32 output (may serve as the next step's sd_verify drafts).
 *   err: SD_ERR_ZERO_ROW when a sampled row has no positive entry (draft 0).
 * Returns SD_OK, or SD_E_SHAPE (K outside [1, SD_K_MAX], V < 1, ld < V, B*K rows beyond 2^31
 * CTAs, request_base + B > 2^32), SD_E_DTYPE, SD_E_NULL, SD_E_ALIGN (rows not aligned to its
 * element), SD_E_DEVICE, SD_E_LAUNCH.
 */
SD_API int sd_draft_sample(int B, int K, int V, int dtype, const void* rows, long ld,
                           const float* temperature, uint64_t seed, uint32_t request_base,
                           int32_t* drafts, int32_t* err, void* stream);

/*
 * sd_pdraft_expand -- rebuild of the drafter batch for P-EAGLE parallel drafting.
 *
 * P-EAGLE blog (vLLM), sections "核心方法" (drafter position i takes the token and hidden state
 * of position i-1; MASK positions take emb(mask) and h_shared), "并行草稿生成的挑战" (expand ids,
 * hidden states and positions with MASK slots, bump positions per request, recompute the slot
 * mapping and per-request start indices), "Triton Kernel" (one pass also emits the rejected-token
 * mask, the masked-token mask, the new-token indices and the hidden-state mapping) and
 * "Hidden State 管理" (PADDING_SLOT_ID = -1).
 *
 * Request r with a_r = num_accepted[r] gets L_r = a_r + K consecutive drafter slots starting at
 * start_loc[r] = sum_{r' < r} L_{r'}. Slot j of request r (i = start_loc[r] + j):
 *   input_ids[i]    = out_tokens[r][j] for j <= a_r (d_1..d_{a_r}, b_r), else mask_token_id
 *   positions[i]    = pos0[r] + 1 + j          (pos0[r] = position of verify slot 0)
 *   slot_mapping[i] = block_table[r][pos / block_size] * block_size + pos % block_size, or -1
 *                     with SD_ERR_BLOCK_TABLE when the table does not cover pos
 *   hidden_map[i]   = r*(K+1) + j for j <= a_r (target hidden row), else -1 (h_shared)
 *   is_masked[i]    = (j > a_r)
 * Slots total_out <= i < capacity are padding: id -1, position 0, slot -1, map -1, mask 0.
 * is_rejected [B, K+1]: 1 for verify slots 1 <= j <= K with j > a_r, else 0.
 * new_token_idx [B, K]: start_loc[r] + a_r + k, the slots whose drafter logits become the next
 *   drafts. start_loc has B+1 entries; start_loc[B] = *total_out = sum_r L_r.
 * Arguments: B >= 0, 1 <= K <= SD_K_MAX; out_tokens [B, K+1] and num_accepted [B] as written by
 *   sd_verify; pos0 [B]; block_table [B, max_blocks] int32 (entries < 0 unused);
 *   block_size >= 1; capacity >= 0 (B*2*K holds every outcome; a smaller capacity truncates
 *   with SD_ERR_TOTAL_RANGE). Outputs have `capacity` entries (is_masked uint8).
 */
SD_API int sd_pdraft_expand(int B, int K, const int32_t* out_tokens, const int32_t* num_accepted,
                     const int32_t* pos0, const int32_t* block_table, int max_blocks,
                     int block_size, int32_t mask_token_id, int capacity, int32_t* input_ids,
                     int32_t* positions, int32_t* slot_mapping, int32_t* hidden_map,
                     uint8_t* is_masked, uint8_t* is_rejected, int32_t* start_loc,
                     int32_t* new_token_idx, int32_t* total_out, int32_t* err, void* stream);

/*
 * sd_pdraft_prepare -- sd_pdraft_expand and the hidden-state gather of sd_hidden_gather in one
 * launch: every output of sd_pdraft_expand, plus out_hidden[i, :] for i < total_out (clamped to
 * capacity) = target_hidden[hidden_map[i], :], or h_shared[:] where hidden_map[i] == -1, as
 * sd_hidden_gather defines it (same sources: P-EAGLE blog, "Hidden State 管理"). Rows from
 * total_out on are not written. Arguments are those of the two calls; target_hidden has n_in_rows
 * rows of stride ld_in, out_hidden `capacity` rows of stride ld_out (both >= H), bf16.
 * When enqueued right after sd_verify it is launched as a programmatic dependent of it: it is
 * scheduled while sd_verify drains and waits on the device for sd_verify's results.
 */
SD_API int sd_pdraft_prepare(int B, int K, const int32_t* out_tokens, const int32_t* num_accepted,
                             const int32_t* pos0, const int32_t* block_table, int max_blocks,
                             int block_size, int32_t mask_token_id, int capacity,
                             int32_t* input_ids, int32_t* positions, int32_t* slot_mapping,
                             int32_t* hidden_map, uint8_t* is_masked, uint8_t* is_rejected,
                             int32_t* start_loc, int32_t* new_token_idx, int32_t* total_out,
                             int H, const void* target_hidden, long ld_in, int n_in_rows,
                             const void* h_shared, void* out_hidden, long ld_out, int32_t* err,
                             void* stream);

/*
 * sd_verify_prepare -- one step of the hot path in one call: sd_verify followed by
 * sd_pdraft_prepare on its outputs.
 *
 * The two operations are those of sd_verify (speculative-decoding explainer, sections "核心思想"
 * and "修正拒绝采样") and sd_pdraft_prepare (P-EAGLE blog, sections "Triton Kernel" and "Hidden
 * State 管理"), with sd_verify's out_tokens and num_accepted feeding the rebuild. When every
 * request samples (temperature NULL) on probability rows, the batch is small enough for one
 * wave of CTAs (B <= 192, and 2B no more than 5 CTAs per SM) and sd_verify would split each row
 * over a request's CTAs (rather than its large-batch race kernel), both run in a single launch:
 * B extra CTAs rebuild the drafter batch while the others race. The single launch is taken
 * only when every one of its CTAs fits on the device at once (the occupancy API's count of
 * resident CTAs per SM times the SMs).
 * A rebuild CTA recomputes the accept decisions of its request and of those before it (they
 * depend on the inputs only), takes its first drafter slot as their prefix, and writes its
 * request's rows and hidden states; only the final token at slot a_r waits for the race, and the
 * CTA that completes request r's race row writes it at the slot the rebuild CTA published in the
 * workspace. If that CTA finds nothing published, it polls for at most 20 ms of the GPU clock
 * (in practice it never waits: the slot appears microseconds after the launch starts, the race
 * rows complete tens of microseconds later; a rebuild CTA kept off the GPU, for instance by
 * other work on another stream filling the SMs, is the only way to run the wait out). When the
 * wait runs out, SD_ERR_WAIT is raised and that request's final token is not written to
 * input_ids (every other output is); the two CTAs still leave the workspace zeroed. Other
 * batches run the two kernels back to back. Either way every output is bit for bit what
 * sd_verify then sd_pdraft_prepare write.
 *
 * Arguments: sd_verify's (without cu_drafts) then sd_pdraft_prepare's from pos0 on (out_tokens
 * and num_accepted are this call's own outputs), with one workspace of at least
 * sd_verify_prepare_workspace_bytes(B) bytes (as much as sd_verify's), 16-byte aligned, zeroed
 * before first use and left zeroed by every call. Errors: those of both calls; SD_ERR_WAIT if a
 * request's published slot never appeared (its final token is then not written to input_ids).
 */
SD_API int sd_verify_prepare(
    int B, int K, int V, int dtype, const void* target, long ld_t, const void* draft, long ld_d,
    const int32_t* drafts, const float* temperature, uint64_t seed, uint32_t request_base,
    int32_t* out_tokens, int32_t* num_accepted, float* p_at_draft, float* q_at_draft,
    const int32_t* pos0, const int32_t* block_table, int max_blocks, int block_size,
    int32_t mask_token_id, int capacity, int32_t* input_ids, int32_t* positions,
    int32_t* slot_mapping, int32_t* hidden_map, uint8_t* is_masked, uint8_t* is_rejected,
    int32_t* start_loc, int32_t* new_token_idx, int32_t* total_out, int H,
    const void* target_hidden, long ld_in, int n_in_rows, const void* h_shared, void* out_hidden,
    long ld_out, void* workspace, size_t workspace_bytes, int32_t* err, void* stream);

/*
 * sd_verify_prepare_ragged -- sd_verify_ragged then sd_pdraft_prepare_ragged on its outputs, in
 * one call: a draft count per request (cu_drafts [B+1], rows packed as sd_verify_ragged reads
 * them, K_max the output stride), with the same single launch for all-sampled one-wave batches
 * (the rebuild CTAs recompute every request's decisions over its own K_r drafts). Every output is
 * bit for bit what the two ragged calls write; arguments and errors as for them and
 * sd_verify_prepare.
 */
SD_API int sd_verify_prepare_ragged(
    int B, int K_max, int V, int dtype, const void* target, long ld_t, const void* draft,
    long ld_d, const int32_t* drafts, const int32_t* cu_drafts, const float* temperature,
    uint64_t seed, uint32_t request_base, int32_t* out_tokens, int32_t* num_accepted,
    float* p_at_draft, float* q_at_draft, const int32_t* pos0, const int32_t* block_table,
    int max_blocks, int block_size, int32_t mask_token_id, int capacity, int32_t* input_ids,
    int32_t* positions, int32_t* slot_mapping, int32_t* hidden_map, uint8_t* is_masked,
    uint8_t* is_rejected, int32_t* start_loc, int32_t* new_token_idx, int32_t* total_out, int H,
    const void* target_hidden, long ld_in, int n_in_rows, const void* h_shared, void* out_hidden,
    long ld_out, void* workspace, size_t workspace_bytes, int32_t* err, void* stream);

/* Workspace of sd_verify_prepare (and _ragged): sd_verify's merge slots, one per request. */
SD_API size_t sd_verify_prepare_workspace_bytes(int B);

/* Kernels one sd_verify_prepare call with these sizes launches (0, 1 fused, or 2); a planning
 * query like sd_verify_kernels. */
SD_API int sd_verify_prepare_kernels(int B, int K, int V, int dtype, int has_temperature);

/*
 * sd_pdraft_prepare_ragged -- sd_pdraft_prepare with a draft count per request, the rebuild
 * that follows sd_verify_ragged (adaptive per-request k): request r with K_r = cu_drafts[r+1] -
 * cu_drafts[r] drafts (0 <= K_r <= K_max) gets L_r = a_r + K_r drafter slots (its accepted
 * drafts, its final token, K_r - 1 MASK slots); its target hidden rows are cu_drafts[r] + r ..
 * (the packing sd_verify_ragged reads). is_rejected [B, K_max+1] is 1 for 1 <= j <= K_r with
 * j > a_r; new_token_idx [B, K_max] is start_loc[r] + a_r + k for k < K_r and -1 after;
 * num_accepted outside [0, K_r] is clamped (SD_ERR_NUM_ACCEPTED), a count outside [0, K_max]
 * too (SD_ERR_DRAFT_COUNT). capacity B*2*K_max holds every outcome. Other arguments and outputs
 * as for sd_pdraft_prepare (with K = K_max).
 */
SD_API int sd_pdraft_prepare_ragged(int B, int K_max, const int32_t* out_tokens,
                                    const int32_t* num_accepted, const int32_t* cu_drafts,
                                    const int32_t* pos0, const int32_t* block_table,
                                    int max_blocks, int block_size, int32_t mask_token_id,
                                    int capacity, int32_t* input_ids, int32_t* positions,
                                    int32_t* slot_mapping, int32_t* hidden_map,
                                    uint8_t* is_masked, uint8_t* is_rejected, int32_t* start_loc,
                                    int32_t* new_token_idx, int32_t* total_out, int H,
                                    const void* target_hidden, long ld_in, int n_in_rows,
                                    const void* h_shared, void* out_hidden, long ld_out,
                                    int32_t* err, void* stream);

/*
 * sd_pdraft_prepare_padded -- the drafter batch in fixed-width rows, with its hidden states.
 *
 * P-EAGLE blog (vLLM), sections "并行草稿生成的挑战" and "Triton Kernel" (the rebuilt ids,
 * positions, slot mapping, masks and new-token indices) and "Hidden State 管理" (rejected tokens
 * map to PADDING_SLOT_ID = -1 so that they write no KV cache; the target hidden states are
 * scattered to their drafter rows; MASK rows take h_shared). In this form every request keeps a
 * row of W = 2K drafter slots whatever it accepted, so start indices are r*W, the batch size is
 * fixed at B*W and no prefix over the batch is needed. Slot j of request r (i = r*W + j):
 *   j < a_r + K: as sd_pdraft_expand defines slot j of request r (input_ids, positions =
 *     pos0 + 1 + j, slot_mapping, hidden_map, is_masked), rejected[i] = 0;
 *   j >= a_r + K (K - a_r rejected leftovers): input_ids = mask_token_id, positions =
 *     pos0 + 1 + j, slot_mapping = -1, hidden_map = -1, is_masked = 0, rejected[i] = 1.
 *   scatter_map [B*(K+1)]: target row r*(K+1)+j -> drafter row r*W + j for j <= a_r, else -1
 *     (the same copies as hidden_map, indexed by source).
 *   new_token_idx [B, K]: r*W + a_r + k.
 *   out_hidden (nullable: metadata only) [B*W, H] bf16 with row stride ld_out: row i =
 *     target_hidden[hidden_map[i]] or h_shared (also for map rows >= n_in_rows, with
 *     SD_ERR_MAP_RANGE). Every row is written.
 * Arguments as for sd_pdraft_prepare; outputs input_ids .. rejected have B*W entries.
 * Errors: SD_ERR_NUM_ACCEPTED (clamped), SD_ERR_BLOCK_TABLE (live slot not covered: -1).
 */
SD_API int sd_pdraft_prepare_padded(int B, int K, const int32_t* out_tokens,
                                    const int32_t* num_accepted, const int32_t* pos0,
                                    const int32_t* block_table, int max_blocks, int block_size,
                                    int32_t mask_token_id, int32_t* input_ids, int32_t* positions,
                                    int32_t* slot_mapping, int32_t* hidden_map,
                                    uint8_t* is_masked, uint8_t* rejected, int32_t* scatter_map,
                                    int32_t* new_token_idx, int H, const void* target_hidden,
                                    long ld_in, int n_in_rows, const void* h_shared,
                                    void* out_hidden, long ld_out, int32_t* err, void* stream);

/*
 * sd_verify_prepare_padded -- sd_verify then sd_pdraft_prepare_padded in one call.
 *
 * The step of sd_verify_prepare with the drafter batch in the fixed-width layout of
 * sd_pdraft_prepare_padded (P-EAGLE blog, "Hidden State 管理": rejected tokens on
 * PADDING_SLOT_ID, target hidden states scattered to their drafter rows). When every request
 * samples on probability rows (temperature NULL) and the batch fits one wave (the conditions of
 * sd_verify_prepare's single launch), this is one launch: CTA r (r < B) recomputes request r's
 * accept decisions from the inputs -- in this layout no request's rows depend on another's counts
 * -- and writes all 2K rows of request r but the token at row r*2K + a_r, which the CTA that
 * completes the request's race writes; nothing waits. Other batches run the verify kernel and
 * then the padded rebuild kernel. Either way every output is bit for bit what sd_verify then
 * sd_pdraft_prepare_padded write; sd_verify_prepare_kernels gives the number of launches.
 *
 * Arguments: sd_verify's (workspace of at least sd_verify_workspace_bytes(B, K, V, dtype),
 * 16-byte aligned, zeroed before first use and left zeroed by every call) then
 * sd_pdraft_prepare_padded's from pos0 on (out_tokens and num_accepted are this call's own
 * outputs). Errors: those of both calls.
 */
SD_API int sd_verify_prepare_padded(
    int B, int K, int V, int dtype, const void* target, long ld_t, const void* draft, long ld_d,
    const int32_t* drafts, const float* temperature, uint64_t seed, uint32_t request_base,
    int32_t* out_tokens, int32_t* num_accepted, float* p_at_draft, float* q_at_draft,
    const int32_t* pos0, const int32_t* block_table, int max_blocks, int block_size,
    int32_t mask_token_id, int32_t* input_ids, int32_t* positions, int32_t* slot_mapping,
    int32_t* hidden_map, uint8_t* is_masked, uint8_t* rejected, int32_t* scatter_map,
    int32_t* new_token_idx, int H, const void* target_hidden, long ld_in, int n_in_rows,
    const void* h_shared, void* out_hidden, long ld_out, void* workspace, size_t workspace_bytes,
    int32_t* err, void* stream);

/*
 * sd_hidden_gather -- drafter hidden states.
 *
 * P-EAGLE blog (vLLM), section "Hidden State 管理": target hidden states are copied to their
 * drafter slots and the learned h_shared fills the MASK slots. Written here in gather form:
 *   out_hidden[i, :] = hidden_map[i] >= 0 ? target_hidden[hidden_map[i], :] : h_shared[:]
 * for i < *total_out (read on the device, clamped to capacity with SD_ERR_TOTAL_RANGE). Rows
 * from *total_out on are not written. A map entry >= n_in_rows writes h_shared and raises
 * SD_ERR_MAP_RANGE. Rows are H bf16 values moved bit for bit; target_hidden has n_in_rows rows
 * of stride ld_in elements, out_hidden `capacity` rows of stride ld_out (both >= H).
 */
SD_API int sd_hidden_gather(int capacity, int H, const int32_t* total_out, const int32_t* hidden_map,
                     const void* target_hidden, long ld_in, int n_in_rows, const void* h_shared,
                     void* out_hidden, long ld_out, int32_t* err, void* stream);

/* ---- diagnostics (test support; same conventions) ---- */

/* Philox4x32-10 of n counters ctr[n][4] under key (seed lo, seed hi) -> out[n][4]. */
SD_API int sd_philox_words(int n, const uint32_t* ctr, uint64_t seed, uint32_t* out, void* stream);

/* The race variates E = fp32(-log((w + 0.5) * 2^-32)) of n words w[n] -> E[n] (the exact path
 * the kernels use). */
SD_API int sd_race_E(int n, const uint32_t* w, float* E, void* stream);

/* Worst relative error, over every w in [w_begin, w_begin + count), of the fast approximation
 * the race filter uses for -log(v) against the exact E above. Writes max_rel[0] (fp32,
 * caller-zeroed) with atomicMax on the float bits. */
SD_API int sd_race_E_approx_error(uint32_t w_begin, uint64_t count, float* max_rel, void* stream);

/* Bit-exactness check of the exact race variate: the kernels evaluate E from pairs of fp32 and
 * take the double path only near an fp32 rounding boundary. Over every w in
 * [w_begin, w_begin + count) adds to counts[0] (uint64, caller-zeroed) the words whose E differs
 * from the double path's fp32(-log((w + 0.5) * 2^-32)), and to counts[1] the words that took
 * the double path. */
SD_API int sd_race_E_check(uint32_t w_begin, uint64_t count, uint64_t* counts, void* stream);

/* sd_verify_prepare with its single launch's wait made to run out (test support for the
 * bounded wait; same arguments from B on): in the single launch, request withhold_request's
 * rebuild CTA publishes its first drafter slot only after the CTA completing that request's race
 * row has polled for wait_us microseconds (1..10^6) of the GPU clock and given up, so that the
 * call raises SD_ERR_WAIT and leaves that request's final token unwritten in input_ids while
 * every other output matches sd_verify_prepare's. Batches that take two kernels run as
 * sd_verify_prepare does (they have no wait). Returns SD_E_SHAPE for a request outside [0, B) or
 * wait_us outside the range. */
SD_API int sd_diag_verify_prepare_withheld(
    int withhold_request, uint32_t wait_us, int B, int K, int V, int dtype, const void* target,
    long ld_t, const void* draft, long ld_d, const int32_t* drafts, const float* temperature,
    uint64_t seed, uint32_t request_base, int32_t* out_tokens, int32_t* num_accepted,
    float* p_at_draft, float* q_at_draft, const int32_t* pos0, const int32_t* block_table,
    int max_blocks, int block_size, int32_t mask_token_id, int capacity, int32_t* input_ids,
    int32_t* positions, int32_t* slot_mapping, int32_t* hidden_map, uint8_t* is_masked,
    uint8_t* is_rejected, int32_t* start_loc, int32_t* new_token_idx, int32_t* total_out, int H,
    const void* target_hidden, long ld_in, int n_in_rows, const void* h_shared, void* out_hidden,
    long ld_out, void* workspace, size_t workspace_bytes, int32_t* err, void* stream);

/* Text for a status code (static storage). */
SD_API const char* sd_status_string(int status);

/* Library version (major * 100 + minor). */
SD_API int sd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SD_GB300_H */
