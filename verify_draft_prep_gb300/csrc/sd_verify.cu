// sd_verify.cu -- batched lossless verification of K drafts per request (sm_103a).
//
// Speculative-decoding explainer (ainews.alishangtian.com), sections "核心思想" and
// "修正拒绝采样": accept a draft with probability min(1, p/q), resample the first rejected
// position from the normalised residual max(0, p - q), emit a bonus token from p_K when every
// draft is accepted; section "边界与代价": temperature 0 must reproduce greedy decoding.
//
// Design (one GB300, HBM-bound):
//  * Greedy and logit requests: one thread-block cluster of CL CTAs per request. Each CTA owns
//    1/CL of every vocab row; the CTAs combine row-wide results (argmax keys, softmax
//    statistics) through distributed shared memory, so a request's rows are visited in order and
//    nothing is read past the first rejection (greedy rows two at a time, at the cost of one
//    speculative row). No spin-waits.
//  * Sampled requests on probability rows: the accept scan is K scalar gathers (one lane per
//    draft); only the one residual (or bonus) row pair is streamed, with 128-bit loads, split
//    over the request's CTAs (no cluster needed when no request is greedy), which merge their
//    exact best through a 16-byte slot per request (atomicMax of the packed key, a unit count).
//    Batches that fill the GPU twice or more go to race_kernel, which splits all race rows
//    evenly over a whole number of CTAs per SM and runs each CTA's few accept scans first.
//  * The residual resample is an exponential race argmax_x r(x)/E_x. E_x needs a double log,
//    which GB300 executes slowly, so each thread filters with an fp32 approximation (one
//    hardware lg2) and keeps only elements whose approximate key lies within a relative band
//    of its running best; the CTA then evaluates the exact key r / fp32(-log(v)) for the few
//    candidates. The band is 23x twice the exhaustively measured worst error of the
//    approximation, so the winner (including the lowest-index rule on exact ties) is always
//    among the candidates. A per-unit upper bound against the CTA's running best skips units
//    that cannot hold a candidate.
//  * Logit rows (bf16): per row the cluster forms the sums of 2^(l c - ref c) (c = log2(e)/T_r,
//    ref the draft token's logit: no running maximum) for the target and draft rows together,
//    exchanges them while the next row's first quarter streams, decides the draft, and on
//    rejection races on the same row pair (the target unit re-read for the skip bound, the
//    draft unit only for the units that pass it).
//  * sd_verify_prepare and sd_verify_prepare_padded fold the drafter-batch rebuild into the
//    launch of an all-sampled one-wave batch: B extra CTAs recompute the accept decisions and
//    write the drafter rows while the others race; only the final token comes from the race.
//  * Per-request draft counts (a prefix of the counts) address each request's packed rows; the
//    drafter-side sampler (sample_kernel) races each drafter row on its own Philox stream, in the
//    log domain for logit rows (one pass: the softmax normaliser cancels).

#include <float.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <type_traits>

#include "sd_common.cuh"
#include "sd_rebuild.cuh"

namespace sdk {

constexpr int NT = 256;        // threads per CTA
constexpr int UNROLL = 3;      // 16-byte units in flight per thread and row (logit statistics)
constexpr int kArgmaxUnroll = 6;  // the same for greedy argmax rows (loads only: more in flight)
constexpr int CL_MAX = 8;      // CTAs per request (portable cluster size)
// Resident CTAs per SM of the verify kernel (48 registers). On fp32 rows it keeps 2 race units in
// flight per thread (measured better than 4 CTAs with 4 units for the one-wave and mixed
// batches); on logit rows 3 statistics units per row and 1 race unit (measured better than 4
// CTAs with 4 and 2: more clusters resident).
constexpr int kMinBlocksF32 = 5;
constexpr int kMinBlocks = 5;
constexpr int min_blocks(int dt) { return dt == SD_F32_PROBS ? kMinBlocksF32 : kMinBlocks; }
constexpr int kRaceMinBlocks = 4;  // the same for race_kernel (its loop keeps 3 units in flight)
constexpr float kBand = 1.0f / 128.0f;  // race candidate band (relative)
constexpr int kCandCap = 32;            // candidate units evaluated thread-parallel per CTA
constexpr int kMaxSeg = NT / 32;        // requests one race-kernel CTA may touch (a warp each)
// A unit whose bound r_max * R(w_max) * kSkip stays below the CTA's running best is skipped (see
// race_take): (1 + kBand) for the filter's band, 2^-9 for the approximations inside the bound.
constexpr float kSkip = (1.0f + kBand) * (1.0f + 0x1p-9f);

// Per-request merge slot in the caller's workspace: the packed (key, ~x) maximum over the
// request's CTAs and the number of CTAs that have merged. The last CTA resets both to zero.
struct RaceSlot {
  unsigned long long best;
  unsigned int count;
  // Fused launch only: 0 until the rebuild CTA publishes request r's first drafter slot + 1, or
  // kGaveUp once the CTA that completed r's race row stopped waiting for it. Whichever of the
  // two CTAs comes second puts it back to 0, so every launch leaves it at 0.
  unsigned int off1;
};
constexpr unsigned kGaveUp = 0xFFFFFFFFu;
// The completing race CTA waits for the published slot at most this long (and at least
// kMinPolls polls, so that a context switch in mid-wait does not end it early); in the fused
// launch every CTA is resident from the start and the slot appears microseconds after it, so
// running out means the rebuild CTA was kept off the GPU (SD_ERR_WAIT).
constexpr uint64_t kWaitNs = 20000000ull;  // 20 ms
constexpr uint32_t kMinPolls = 1024;

// The drafter-batch rebuild fused into the verify launch (sd_verify_prepare): the same outputs
// as the rebuild kernel, written by one extra CTA per request while the others race.
struct RebuildArgs {
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
  int H;
  const uint16_t* hidden;
  long ld_in;
  int n_in_rows;
  const uint16_t* h_shared;
  uint16_t* out_hidden;  // nullptr: metadata only
  long ld_out;
  int hvec;              // 16-byte aligned hidden rows, H a multiple of 8
  // the padded layout (sd_verify_prepare_padded): fixed 2K-slot rows, per-slot rejected mask
  // and the scatter form of the hidden map; capacity, start_loc and total_out are unused
  int padded;
  uint8_t* rejected;
  int32_t* scatter_map;
};

struct VerifyParams {
  int B, K, V;
  const void* target;
  long ld_t;
  const void* draft;
  long ld_d;
  const int32_t* drafts;
  const float* temperature;
  const int32_t* cu;  // nullable: per-request draft counts as a prefix [B+1] (K is then K_max)
  PhiloxRoundKeys rk;
  uint32_t rbase;  // request index of row 0 in the Philox counters (global index of a shard)
  int32_t* out_tokens;
  int32_t* num_accepted;
  float* p_at;
  float* q_at;
  struct RaceSlot* slots;  // one per request (sampled probability requests)
  int32_t* err;
  int cl;   // cluster size: CTAs that share a greedy or logit request's rows
  int nc;   // CTAs per request in the cluster role (a multiple of cl)
  int cluster_blocks;  // blocks [0, cluster_blocks) take the cluster role: B * nc
  int race_blocks;     // blocks after them take the race role (0: sampled requests stay per
                       // request in the cluster role)
  int vec;  // 1: every row starts on a 16-byte boundary
  int fuse;  // 1: CTAs [0, B) rebuild the drafter batch, CTAs [B, grid) race (spread over the
             // requests as evenly as they go); 2: the same with the padded layout
  RebuildArgs rb;
  uint64_t wait_ns;  // bound of the completing race CTA's wait for the published slot
  int withhold;      // diagnostic (-1: none): this request's rebuild CTA publishes its slot only
                     // once the race CTA has given up waiting, so that the wait runs out
};

// Request r's rows: K_r drafts (cu[r+1] - cu[r] when per-request counts are given, clamped to
// [0, K] with SD_ERR_DRAFT_COUNT; else K), target rows t0 .. t0 + K_r (t0 = cu[r] + r, or
// r*(K+1)), draft rows and draft tokens from d0 (cu[r], or r*K). Outputs keep the stride of K.
struct ReqRows {
  int k;
  size_t t0, d0;
  int32_t e;
};
__device__ __forceinline__ ReqRows req_rows(const VerifyParams& P, int r) {
  if (!P.cu) return ReqRows{P.K, (size_t)r * (P.K + 1), (size_t)r * P.K, 0};
  const int c0 = __ldg(P.cu + r), c1 = __ldg(P.cu + r + 1);
  int k = c1 - c0;
  int32_t e = 0;
  if (k < 0 || k > P.K || c0 < 0) {
    e = SD_ERR_DRAFT_COUNT;
    k = c0 < 0 ? 0 : (k < 0 ? 0 : P.K);
  }
  const size_t base = c0 < 0 ? 0 : (size_t)c0;
  return ReqRows{k, base + (size_t)r, base, e};
}

// ---------------------------------------------------------------------------------- row sources
// A "unit" is 16 bytes of a row: 4 fp32 or 8 bf16 elements. Units past V (the ragged tail) and
// rows that are not 16-byte aligned use scalar loads; elements past V take a neutral fill.

__device__ __forceinline__ float4 ld_f4(const float* p) {
  const uint4 v = ld_stream_u4(p);
  return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                     __uint_as_float(v.w));
}

__device__ __forceinline__ void f32_unit(const float* row, uint32_t u, uint32_t V, bool vec,
                                         float fill, float (&v)[4]) {
  const uint32_t x0 = u * 4u;
  if (vec && x0 + 4u <= V) {
    const float4 t = ld_f4(row + x0);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (x0 + i < V) ? __ldg(row + x0 + i) : fill;
  }
}

// 8 bf16 values as raw 16-bit words; entries past V read as bf16 -inf (0xff80).
__device__ __forceinline__ uint4 bf16_raw(const uint16_t* row, uint32_t u, uint32_t V, bool vec) {
  const uint32_t x0 = u * 8u;
  if (vec && x0 + 8u <= V) return ld_stream_u4(row + x0);
  uint32_t h[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = (x0 + i < V) ? (uint32_t)__ldg(row + x0 + i) : 0xff80u;
  return make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                    h[6] | (h[7] << 16));
}

__device__ __forceinline__ float bf16_at(const uint4& w, int i) {
  const uint32_t v = (i < 2) ? w.x : (i < 4) ? w.y : (i < 6) ? w.z : w.w;
  return (i & 1) ? __uint_as_float(v & 0xffff0000u) : __uint_as_float(v << 16);
}

// Residual (or bonus) values r(x) over fp32 probability rows.
template <bool HAS_Q>
struct F32Residual {
  static constexpr int EPU = 4;
  static constexpr int UNR = 2;  // units in flight per thread
  static constexpr bool kLean = false;
  const float* p;
  const float* q;
  uint32_t V;
  bool vec;
  struct Raw {
    float p[4], q[4];
  };
  __device__ __forceinline__ void fetch(uint32_t u, Raw& raw) const {
    f32_unit(p, u, V, vec, 0.0f, raw.p);
    if (HAS_Q) f32_unit(q, u, V, vec, 0.0f, raw.q);
  }
  // units entirely inside the row, read with unchecked 128-bit loads when vec is set
  __device__ __forceinline__ uint32_t full_units() const { return V / 4u; }
  __device__ __forceinline__ void fetch_fast(uint32_t u, Raw& raw) const {
    const float4 a = ld_f4(p + 4u * u);
    raw.p[0] = a.x; raw.p[1] = a.y; raw.p[2] = a.z; raw.p[3] = a.w;
    if (HAS_Q) {
      const float4 b = ld_f4(q + 4u * u);
      raw.q[0] = b.x; raw.q[1] = b.y; raw.q[2] = b.z; raw.q[3] = b.w;
    }
  }
  // the rest of a unit fetched by fetch_fast (here nothing: both rows are in)
  __device__ __forceinline__ void complete(uint32_t, Raw&) const {}
  __device__ __forceinline__ void residual(const Raw& raw, float (&r)[4]) const {
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = HAS_Q ? __fsub_rn(raw.p[i], raw.q[i]) : raw.p[i];
  }
  // an upper bound of the unit's residuals (here their maximum)
  __device__ __forceinline__ float residual_bound(const Raw& raw) const {
    float r[4];
    residual(raw, r);
    return fmaxf(fmaxf(r[0], r[1]), fmaxf(r[2], r[3]));
  }
  __device__ __forceinline__ float at(uint32_t x) const {
    return HAS_Q ? __fsub_rn(__ldg(p + x), __ldg(q + x)) : __ldg(p + x);
  }
};

// The same residual source with q chosen at run time (nullptr: the bonus race on p), so that one
// copy of the race loop serves both cases.
struct F32ResidualAny {
  static constexpr int EPU = 4;
  static constexpr int UNR = 3;
  static constexpr bool kLean = false;
  const float* p;
  const float* q;  // nullptr: r = p
  uint32_t V;
  bool vec;
  struct Raw {
    float p[4], q[4];
  };
  __device__ __forceinline__ void fetch(uint32_t u, Raw& raw) const {
    f32_unit(p, u, V, vec, 0.0f, raw.p);
    if (q) f32_unit(q, u, V, vec, 0.0f, raw.q);
    else raw.q[0] = raw.q[1] = raw.q[2] = raw.q[3] = 0.0f;
  }
  __device__ __forceinline__ uint32_t full_units() const { return V / 4u; }
  __device__ __forceinline__ void fetch_fast(uint32_t u, Raw& raw) const {
    const float4 a = ld_f4(p + 4u * u);
    raw.p[0] = a.x; raw.p[1] = a.y; raw.p[2] = a.z; raw.p[3] = a.w;
    if (q) {
      const float4 b = ld_f4(q + 4u * u);
      raw.q[0] = b.x; raw.q[1] = b.y; raw.q[2] = b.z; raw.q[3] = b.w;
    } else {
      raw.q[0] = raw.q[1] = raw.q[2] = raw.q[3] = 0.0f;
    }
  }
  __device__ __forceinline__ void complete(uint32_t, Raw&) const {}
  // p - 0 == p exactly, so the bonus race sees r = p as the definition asks
  __device__ __forceinline__ void residual(const Raw& raw, float (&r)[4]) const {
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = __fsub_rn(raw.p[i], raw.q[i]);
  }
  __device__ __forceinline__ float residual_bound(const Raw& raw) const {
    float r[4];
    residual(raw, r);
    return fmaxf(fmaxf(r[0], r[1]), fmaxf(r[2], r[3]));
  }
  __device__ __forceinline__ float at(uint32_t x) const {
    return q ? __fsub_rn(__ldg(p + x), __ldg(q + x)) : __ldg(p + x);
  }
};

// p(x) = exp2(l c - ref c) / S with c = log2(e) / T and S the row's sum of the same terms for a
// fixed reference logit ref (nrc = -(ref c)); written with explicit roundings so that the
// streamed statistics, the streamed race and the scalar re-evaluation of a candidate give the
// same bits for the same element.
__device__ __forceinline__ float logit_term(float l, float c, float nrc) {
  return fast_ex2(fmaf(l, c, nrc));
}
__device__ __forceinline__ float logit_prob(float l, float c, float nrc, float invS) {
  return __fmul_rn(logit_term(l, c, nrc), invS);
}

template <bool HAS_Q>
struct Bf16Residual {
  static constexpr int EPU = 8;
  static constexpr int UNR = 1;  // target units in flight per thread
  static constexpr bool kLean = true;
  const uint16_t* t;
  const uint16_t* d;
  float nrct, invSt, nrcd, invSd, c;
  uint32_t V;
  bool vec;
  struct Raw {
    uint4 t, d;
  };
  __device__ __forceinline__ void fetch(uint32_t u, Raw& raw) const {
    raw.t = bf16_raw(t, u, V, vec);
    if (HAS_Q) raw.d = bf16_raw(d, u, V, vec);
  }
  __device__ __forceinline__ uint32_t full_units() const { return V / 8u; }
  // The streamed pass reads the target unit alone: the skip bound needs only p (r <= p, as
  // q >= 0), and the draft unit is read (complete) for the units that pass it.
  __device__ __forceinline__ void fetch_fast(uint32_t u, Raw& raw) const {
    raw.t = ld_stream_u4(t + 8u * u);
  }
  __device__ __forceinline__ void complete(uint32_t u, Raw& raw) const {
    if (HAS_Q) raw.d = ld_stream_u4(d + 8u * u);
  }
  __device__ __forceinline__ void residual(const Raw& raw, float (&r)[8]) const {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float pv = logit_prob(bf16_at(raw.t, i), c, nrct, invSt);
      r[i] = HAS_Q ? __fsub_rn(pv, logit_prob(bf16_at(raw.d, i), c, nrcd, invSd)) : pv;
    }
  }
  // An upper bound of the unit's residuals without their exponentials: r(x) <= p(x) (q >= 0),
  // and p at the unit's largest target logit bounds every p(x) of the unit up to the hardware
  // exponential's non-monotonicity (far below the 2^-9 allowed for in kSkip).
  __device__ __forceinline__ float residual_bound(const Raw& raw) const {
    uint32_t m01, m23, m;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(m01) : "r"(raw.t.x), "r"(raw.t.y));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(m23) : "r"(raw.t.z), "r"(raw.t.w));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(m01), "r"(m23));
    const float lmax = fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    return logit_prob(lmax, c, nrct, invSt);
  }
  __device__ __forceinline__ float at(uint32_t x) const {
    const float pv = logit_prob(bf16_bits_to_float(__ldg(t + x)), c, nrct, invSt);
    return HAS_Q ? __fsub_rn(pv, logit_prob(bf16_bits_to_float(__ldg(d + x)), c, nrcd, invSd))
                 : pv;
  }
};

// -------------------------------------------------------------------------------- shared state
struct Smem {
  uint64_t red[NT / 32];
  float2 redf[2][NT / 32];  // block sums of a row pair (double-buffered by call parity)
  uint64_t slot[2];   // per-CTA cluster exchange (double-buffered)
  uint64_t slot2[2];  // second value of a paired exchange (greedy rows two at a time)
  uint64_t red2[NT / 32];
  uint64_t bcast2;
  float2 xslot[2];    // this CTA's row sums for the cluster (row parity)
  float2 xslot_fb;    // the same for a row's max-referenced recomputation
  uint64_t bcast;
  float lt[SD_K_MAX + 1], ld[SD_K_MAX];  // logit rows: the draft token's logits (references)
  float P[SD_K_MAX], Q[SD_K_MAX];
  int a;
  int e;
  int ncand;
  uint32_t cand[kCandCap];
  int last;
  uint32_t tau;  // race_take's running best of the current race_chunk call (fp32 bits)
  uint64_t race_best;  // race_chunk's exact maximum over the CTA
};

// Cluster-wide maximum of a CTA-uniform value. Every CTA of the cluster calls it the same
// number of times (control flow is uniform across the cluster by construction).
__device__ uint64_t cluster_max_u64(uint64_t v, Smem& sm, int& phase, int cl) {
  if (cl == 1) return v;
  if (threadIdx.x == 0) sm.slot[phase] = v;
  cluster_barrier();
  if (threadIdx.x < 32) {
    uint64_t m = (threadIdx.x < (unsigned)cl) ? load_from_rank(&sm.slot[phase], threadIdx.x) : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint64_t other = __shfl_xor_sync(0xffffffffu, m, o);
      m = other > m ? other : m;
    }
    if (threadIdx.x == 0) sm.bcast = m;
  }
  __syncthreads();
  const uint64_t m = sm.bcast;
  phase ^= 1;
  return m;
}

// The same for two values at once: one cluster barrier for both.
__device__ void cluster_max2_u64(uint64_t& v0, uint64_t& v1, Smem& sm, int& phase, int cl) {
  if (cl == 1) return;
  if (threadIdx.x == 0) {
    sm.slot[phase] = v0;
    sm.slot2[phase] = v1;
  }
  cluster_barrier();
  if (threadIdx.x < 32) {
    const bool in = threadIdx.x < (unsigned)cl;
    uint64_t m0 = in ? load_from_rank(&sm.slot[phase], threadIdx.x) : 0ull;
    uint64_t m1 = in ? load_from_rank(&sm.slot2[phase], threadIdx.x) : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint64_t x0 = __shfl_xor_sync(0xffffffffu, m0, o);
      const uint64_t x1 = __shfl_xor_sync(0xffffffffu, m1, o);
      m0 = x0 > m0 ? x0 : m0;
      m1 = x1 > m1 ? x1 : m1;
    }
    if (threadIdx.x == 0) {
      sm.bcast = m0;
      sm.bcast2 = m1;
    }
  }
  __syncthreads();
  v0 = sm.bcast;
  v1 = sm.bcast2;
  phase ^= 1;
}

// ------------------------------------------------------------------------------------ the race
// Filter: the approximate key of element x is alpha_x = r(x) * R(w_x), proportional to r/E within
// the measured relative error. Each thread keeps, branch-free, the largest unit maximum a1 (with
// its unit) and the largest maximum among its other units a2. With A the CTA's largest a1, only
// units whose maximum m satisfies m * (1 + kBand) >= A can hold the exact winner: the thread's
// best unit if a1 qualifies, and any other of its units only if a2 does (then it rescans). Every
// element of a candidate unit gets its exact key, so exact ties are settled by index.

__device__ __forceinline__ uint64_t exact_key(float r, uint32_t w, uint32_t x) {
  const float key = __fdiv_rn(fmaxf(r, 0.0f), race_E_exact(w));
  return pack_key(__float_as_uint(key), x);
}

template <int EPU>
__device__ __forceinline__ uint32_t unit_wmax(const uint4 (&w)[EPU / 4]) {
  uint32_t wmax = 0;
#pragma unroll
  for (int h = 0; h < EPU / 4; ++h) wmax = max(wmax, max(max(w[h].x, w[h].y), max(w[h].z, w[h].w)));
  return wmax;
}

// Largest approximate key of one unit (0 when no residual is positive); wmax = unit_wmax(w).
template <int EPU>
__device__ __forceinline__ float unit_max_alpha(const float (&r)[EPU], const uint4 (&w)[EPU / 4],
                                                uint32_t wmax) {
  float R[EPU];
#pragma unroll
  for (int h = 0; h < EPU / 4; ++h) {
    R[4 * h + 0] = race_R_main(w[h].x);
    R[4 * h + 1] = race_R_main(w[h].y);
    R[4 * h + 2] = race_R_main(w[h].z);
    R[4 * h + 3] = race_R_main(w[h].w);
  }
  if (wmax >= kNearOne) {  // one word in 8192: redo those few near v = 1
#pragma unroll
    for (int e = 0; e < EPU; ++e) {
      const uint32_t we = word_of(w[e >> 2], e & 3);
      if (we >= kNearOne) R[e] = race_R_near_one(we);
    }
  }
  float m = 0.0f;
#pragma unroll
  for (int e = 0; e < EPU; ++e) m = fmaxf(m, r[e] * R[e]);
  return m;
}

template <class Src>
__device__ __forceinline__ void unit_words(const PhiloxRoundKeys& rk, uint32_t u, uint32_t rid,
                                           uint32_t j, uint32_t tag, uint4 (&w)[Src::EPU / 4]) {
#pragma unroll
  for (int h = 0; h < Src::EPU / 4; ++h)
    w[h] = race_block(rk, u * (Src::EPU / 4) + h, rid, j, tag);
}

// Exact keys of the positive elements of unit u, folded into `best` (one thread, rare path).
template <class Src>
__device__ __noinline__ void exact_unit(const Src& src, uint32_t u, const PhiloxRoundKeys& rk,
                                        uint32_t rid, uint32_t j, uint32_t tag, uint64_t& best) {
  constexpr int EPU = Src::EPU;
  typename Src::Raw raw;
  src.fetch(u, raw);
  float r[EPU];
  src.residual(raw, r);
  uint4 w[EPU / 4];
  unit_words<Src>(rk, u, rid, j, tag, w);
#pragma unroll
  for (int e = 0; e < EPU; ++e) {
    if (r[e] > 0.0f) {
      const uint64_t k = exact_key(r[e], word_of(w[e >> 2], e & 3), u * EPU + e);
      best = k > best ? k : best;
    }
  }
}

// One unit of the streaming pass. *tau is the largest unit maximum any thread of the CTA has
// posted for this row so far (0 at the start of each race_chunk call); it and a1 are maxima of
// computed units, so neither exceeds A. A unit whose bound r_max * R(w_max) * kSkip (R rises with
// the word, so R(w_max) bounds R(w_x) of the unit up to the approximation error) stays below
// max(a1, *tau) has m * (1 + kBand) < A: it cannot be a candidate, and skipping it changes
// neither A nor a thread's candidate units; its keys are not computed.
// The largest Philox word of unit u: all the skip bound needs (the words themselves are
// recomputed for the few units that pass it, so that they need no registers in the loop).
template <int EPU>
__device__ __forceinline__ uint32_t unit_wmax_of(const PhiloxRoundKeys& rk, uint32_t u,
                                                 uint32_t rid, uint32_t j, uint32_t tag) {
  uint32_t m = 0;
#pragma unroll
  for (int h = 0; h < EPU / 4; ++h) {
    const uint4 w = race_block(rk, u * (EPU / 4) + h, rid, j, tag);
    m = max(m, max(max(w.x, w.y), max(w.z, w.w)));
  }
  return m;
}

template <class Src>
__device__ __forceinline__ void race_take(const Src& src, typename Src::Raw& raw,
                                          const PhiloxRoundKeys& rk, uint32_t rid, uint32_t j,
                                          uint32_t tag, uint32_t u, float& a1, float& a2,
                                          uint32_t& best_u, uint32_t* tau, bool fetched = false) {
  // Logit rows (two Philox blocks per unit) keep only the largest word through the bound and
  // recompute the words for the units that pass it, which keeps the loop's registers down;
  // probability rows (one block per unit) keep the words.
  uint4 w[Src::EPU / 4];
  uint32_t wmax;
  if (Src::kLean) {
    wmax = unit_wmax_of<Src::EPU>(rk, u, rid, j, tag);
  } else {
    unit_words<Src>(rk, u, rid, j, tag, w);
    wmax = unit_wmax<Src::EPU>(w);
  }
  const float thr = fmaxf(a1, __uint_as_float(*(volatile uint32_t*)tau));
  if (src.residual_bound(raw) * race_R(wmax) * kSkip < thr) return;
  if (!fetched) src.complete(u, raw);
  if (Src::kLean) unit_words<Src>(rk, u, rid, j, tag, w);
  float r[Src::EPU];
  src.residual(raw, r);
  const float m = unit_max_alpha<Src::EPU>(r, w, wmax);
  a2 = fmaxf(a2, fminf(m, a1));
  best_u = m > a1 ? u : best_u;
  if (m > thr) atomicMax(tau, __float_as_uint(m));  // keys are >= 0: ordered as integers
  a1 = fmaxf(a1, m);
}

// Exact race winner over units [u0, u1) of one row: the CTA's packed (key, ~x) maximum, or 0 when
// no element of the chunk has a positive residual.
template <class Src>
__device__ __forceinline__ uint64_t race_chunk(const Src& src, uint32_t u0, uint32_t u1,
                                               const PhiloxRoundKeys& rk,
                               uint32_t rid, uint32_t j, Smem& sm, uint32_t tag = kTagVerify) {
  constexpr int EPU = Src::EPU, UNR = Src::UNR;
  float a1 = 0.0f, a2 = 0.0f;
  uint32_t best_u = 0xffffffffu;
  // units [u0, uf) lie inside 16-byte aligned rows: unchecked 128-bit loads, software-pipelined
  // so that UNR units are always in flight (each buffer is refilled right after it is consumed)
  const uint32_t uf = src.vec ? max(u0, min(u1, src.full_units())) : u0;
  uint32_t ub = u0 + threadIdx.x;
  if (ub + (UNR - 1) * NT < uf) {
    typename Src::Raw raw[UNR];
#pragma unroll
    for (int k = 0; k < UNR; ++k) src.fetch_fast(ub + k * NT, raw[k]);
    for (; ub + (2 * UNR - 1) * NT < uf; ub += UNR * NT) {
#pragma unroll
      for (int k = 0; k < UNR; ++k) {
        const uint32_t u = ub + k * NT;
        race_take(src, raw[k], rk, rid, j, tag, u, a1, a2, best_u, &sm.tau);
        src.fetch_fast(u + UNR * NT, raw[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < UNR; ++k) {  // drain the last UNR units in flight
      const uint32_t u = ub + k * NT;
      race_take(src, raw[k], rk, rid, j, tag, u, a1, a2, best_u, &sm.tau);
    }
    ub += UNR * NT;
  }
  for (; ub < u1; ub += NT) {  // the rest, bounds-checked (fetch reads every row of the unit)
    typename Src::Raw raw;
    src.fetch(ub, raw);
    race_take(src, raw, rk, rid, j, tag, ub, a1, a2, best_u, &sm.tau, true);
  }
  if (threadIdx.x == 0) {
    sm.ncand = 0;
    sm.race_best = 0ull;
  }
  // A, the CTA's largest unit maximum, is in tau once every thread has left the streaming pass:
  // a unit maximum not posted there was at most the value tau held when the thread read it
  __syncthreads();
  const float A = __uint_as_float(*(volatile uint32_t*)&sm.tau);
  uint64_t best = 0ull;
  if (A > 0.0f) {
    // A CTA maximum below about 2^-100 in key units: fp32 keys are near the subnormal range
    // and no longer carry relative precision, so every positive element is evaluated exactly.
    const bool tiny = A < 0x1p-37f;
    bool rescan = tiny || a2 * (1.0f + kBand) >= A;
    if (!rescan && a1 * (1.0f + kBand) >= A) {
      const int slot = atomicAdd(&sm.ncand, 1);
      if (slot < kCandCap) sm.cand[slot] = best_u;
      else rescan = true;
    }
    if (rescan) {  // this thread's other units may hold candidates too (rare)
      for (uint32_t u = u0 + threadIdx.x; u < u1; u += NT) {
        bool take = tiny;
        if (!take) {
          typename Src::Raw raw;
          src.fetch(u, raw);
          float r[EPU];
          src.residual(raw, r);
          uint4 w[EPU / 4];
          unit_words<Src>(rk, u, rid, j, tag, w);
          take = unit_max_alpha<EPU>(r, w, unit_wmax<EPU>(w)) * (1.0f + kBand) >= A;
        }
        if (take) exact_unit(src, u, rk, rid, j, tag, best);
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) sm.tau = 0u;  // every thread has read A
    // the listed candidate units, one element per thread (kCandCap * EPU <= NT: one round, so
    // the candidates' scattered loads are in flight together)
    const int nc = min(sm.ncand, kCandCap);
    for (int l = (int)threadIdx.x; l < nc * EPU; l += NT) {
      const uint32_t u = sm.cand[l / EPU];
      const uint32_t x = u * EPU + (uint32_t)(l % EPU);
      const float r = x < src.V ? src.at(x) : 0.0f;  // the last unit may pass the row end
      if (r > 0.0f) {
        const uint4 w4 = race_block(rk, x >> 2, rid, j, tag);
        const uint64_t k = exact_key(r, word_of(w4, x & 3u), x);
        best = k > best ? k : best;
      }
    }
  } else {
    __syncthreads();
    if (threadIdx.x == 0) sm.tau = 0u;  // every thread has read A
  }
  // the CTA's best exact key: warp maxima into one shared 64-bit maximum
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t other = __shfl_xor_sync(0xffffffffu, best, o);
    best = other > best ? other : best;
  }
  if ((threadIdx.x & 31) == 0 && best)
    atomicMax((unsigned long long*)&sm.race_best, (unsigned long long)best);
  __syncthreads();
  const uint64_t m = sm.race_best;
  __syncthreads();  // every thread has read it before the next call resets it
  return m;
}

// ------------------------------------------------------------- log-domain race on logit rows
// For a race on softmax(l c ln2) itself (the drafter-side sampler), the winner
// argmax_x q(x)/E_x equals argmax_x (l_x c - log2 E_x): the softmax's maximum and normaliser are
// common factors, so one pass over the row suffices. The filter key is
// beta_x = l_x c - lg2(L_x), with L_x ~= -log2 v_x = E_x log2(e) from the hardware lg2 (the series
// near v = 1, as for R); it differs from the exact log key by the constant log2(log2 e) and an
// error below 2.5e-4 (L's measured relative error 1.669e-4 times log2 e, plus fp32 rounding of
// l c), far inside kLogBand, the band log2(1 + 2^-7) of the linear filter. Exact keys, for
// candidate units only: l_x c - log2(E_x) in double with E_x exactly as the verify race's,
// rounded to fp32 and packed as an orderable float (a tie within one fp32 step of the key goes
// to the lowest x).
constexpr float kLogBand = 0.01122f;   // log2(1 + 2^-7)
constexpr float kLogSlack = 0.002f;    // approximation allowance inside the per-unit bound

__device__ __forceinline__ float race_L(uint32_t w) {  // ~ -log2 v, v = (w + 0.5) 2^-32
  if (w < kNearOne) return -fast_lg2(fmaf(__uint2float_rn(w), 0x1p-32f, 0x1p-33f));
  const float m = fmaf(__uint2float_rn(~w), 0x1p-32f, 0x1p-33f);  // 1 - v
  return (m * fmaf(m, fmaf(m, 0.33333334f, 0.5f), 1.0f)) * kLog2e;
}

__device__ __forceinline__ uint64_t log_exact_key(float l, float c, uint32_t w, uint32_t x) {
  const double key = (double)l * (double)c - log2((double)race_E_exact(w));
  return pack_key(orderable((float)key), x);
}

__device__ __noinline__ void log_exact_unit(const uint16_t* row, uint32_t V, bool vec, float c,
                                            uint32_t u, const PhiloxRoundKeys& rk, uint32_t rid,
                                            uint32_t j, uint32_t tag, uint64_t& best) {
  const uint4 raw = bf16_raw(row, u, V, vec);
  uint4 w[2];
  w[0] = race_block(rk, 2u * u, rid, j, tag);
  w[1] = race_block(rk, 2u * u + 1u, rid, j, tag);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float l = bf16_at(raw, e);
    if (u * 8u + e < V && l > -INFINITY) {
      const uint64_t k = log_exact_key(l, c, word_of(w[e >> 2], e & 3), u * 8u + e);
      best = k > best ? k : best;
    }
  }
}

// Largest filter key of one unit (-inf when every logit is -inf).
__device__ __forceinline__ float log_unit_max(const uint4& raw, const uint4 (&w)[2], float c) {
  float m = -INFINITY;
#pragma unroll
  for (int e = 0; e < 8; ++e)
    m = fmaxf(m, fmaf(bf16_at(raw, e), c, -fast_lg2(race_L(word_of(w[e >> 2], e & 3)))));
  return m;
}

// One unit of the log-domain pass; *tau holds the CTA's running best (orderable bits, 0 = none).
__device__ __forceinline__ void log_take(const uint4& raw, const uint4 (&w)[2], float c,
                                         uint32_t u, float& a1, float& a2, uint32_t& best_u,
                                         uint32_t* tau) {
  uint32_t m01, m23, mm;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(m01) : "r"(raw.x), "r"(raw.y));
  asm("max.bf16x2 %0, %1, %2;" : "=r"(m23) : "r"(raw.z), "r"(raw.w));
  asm("max.bf16x2 %0, %1, %2;" : "=r"(mm) : "r"(m01), "r"(m23));
  const float lmax = fmaxf(__uint_as_float(mm << 16), __uint_as_float(mm & 0xffff0000u));
  const uint32_t wmax = unit_wmax<8>(w);
  const uint32_t tb = *(volatile uint32_t*)tau;
  const float shared_best = tb ? __uint_as_float(tb & 0x80000000u ? tb & 0x7fffffffu : ~tb)
                               : -INFINITY;
  const float thr = fmaxf(a1, shared_best);
  // bound of every beta_x of the unit: the largest logit and the largest word (L falls with w)
  if (fmaf(lmax, c, -fast_lg2(race_L(wmax))) + kLogSlack < thr - kLogBand) return;
  const float m = log_unit_max(raw, w, c);
  a2 = fmaxf(a2, fminf(m, a1));
  best_u = m > a1 ? u : best_u;
  if (m > thr) atomicMax(tau, orderable(m));
  a1 = fmaxf(a1, m);
}

// The exact log-domain race winner over units [u0, u1) of one logit row: the CTA's packed
// (orderable key, ~x) maximum, or 0 when every logit of the share is -inf.
__device__ uint64_t race_chunk_log(const uint16_t* row, uint32_t V, bool vec, float c,
                                   uint32_t u0, uint32_t u1, const PhiloxRoundKeys& rk,
                                   uint32_t rid, uint32_t j, uint32_t tag, Smem& sm) {
  float a1 = -INFINITY, a2 = -INFINITY;
  uint32_t best_u = 0xffffffffu;
  const uint32_t uf = vec ? max(u0, min(u1, V / 8u)) : u0;
  uint32_t ub = u0 + threadIdx.x;
  constexpr int UNR = 1;  // one unit in flight: the sampler fits 5 CTAs per SM unspilled
  if (ub + (UNR - 1) * NT < uf) {
    uint4 raw[UNR];
#pragma unroll
    for (int k = 0; k < UNR; ++k) raw[k] = ld_stream_u4(row + 8u * (ub + k * NT));
    for (; ub + (2 * UNR - 1) * NT < uf; ub += UNR * NT) {
#pragma unroll
      for (int k = 0; k < UNR; ++k) {
        const uint32_t u = ub + k * NT;
        uint4 w[2];
        w[0] = race_block(rk, 2u * u, rid, j, tag);
        w[1] = race_block(rk, 2u * u + 1u, rid, j, tag);
        log_take(raw[k], w, c, u, a1, a2, best_u, &sm.tau);
        raw[k] = ld_stream_u4(row + 8u * (u + UNR * NT));
      }
    }
#pragma unroll
    for (int k = 0; k < UNR; ++k) {
      const uint32_t u = ub + k * NT;
      uint4 w[2];
      w[0] = race_block(rk, 2u * u, rid, j, tag);
      w[1] = race_block(rk, 2u * u + 1u, rid, j, tag);
      log_take(raw[k], w, c, u, a1, a2, best_u, &sm.tau);
    }
    ub += UNR * NT;
  }
  for (; ub < u1; ub += NT) {  // the rest, bounds-checked (-inf past the row end)
    const uint4 raw = bf16_raw(row, ub, V, vec);
    uint4 w[2];
    w[0] = race_block(rk, 2u * ub, rid, j, tag);
    w[1] = race_block(rk, 2u * ub + 1u, rid, j, tag);
    log_take(raw, w, c, ub, a1, a2, best_u, &sm.tau);
  }
  if (threadIdx.x == 0) sm.ncand = 0;
  const uint32_t Ab = (uint32_t)block_max_u64<NT>(a1 > -INFINITY ? orderable(a1) : 0u, sm.red);
  if (threadIdx.x == 0) sm.tau = 0u;  // every thread has left the streaming pass
  uint64_t best = 0ull;
  if (Ab != 0u) {
    const float A = __uint_as_float(Ab & 0x80000000u ? Ab & 0x7fffffffu : ~Ab);
    bool rescan = a2 >= A - kLogBand;
    if (!rescan && a1 >= A - kLogBand) {
      const int slot = atomicAdd(&sm.ncand, 1);
      if (slot < kCandCap) sm.cand[slot] = best_u;
      else rescan = true;
    }
    if (rescan) {  // this thread's other units may hold candidates too (rare)
      for (uint32_t u = u0 + threadIdx.x; u < u1; u += NT) {
        const uint4 raw = bf16_raw(row, u, V, vec);
        uint4 w[2];
        w[0] = race_block(rk, 2u * u, rid, j, tag);
        w[1] = race_block(rk, 2u * u + 1u, rid, j, tag);
        if (log_unit_max(raw, w, c) >= A - kLogBand)
          log_exact_unit(row, V, vec, c, u, rk, rid, j, tag, best);
      }
    }
    __syncthreads();
    const int nc = min(sm.ncand, kCandCap);
    for (int l = (int)threadIdx.x; l < nc * 8; l += NT) {  // one element per thread
      const uint32_t x = sm.cand[l / 8] * 8u + (uint32_t)(l % 8);
      if (x < V) {
        const float lv = bf16_bits_to_float(__ldg(row + x));
        if (lv > -INFINITY) {
          const uint4 w4 = race_block(rk, x >> 2, rid, j, tag);
          const uint64_t k = log_exact_key(lv, c, word_of(w4, x & 3u), x);
          best = k > best ? k : best;
        }
      }
    }
  }
  return block_max_u64<NT>(best, sm.red);
}

// --------------------------------------------------------------------------------- greedy rows
__device__ __forceinline__ void argmax_take(float v, uint32_t x, float& best, uint32_t& bx) {
  if (v > best) {
    best = v;
    bx = x;
  }
}

template <int DT>
__device__ uint64_t argmax_chunk(const void* row, uint32_t V, bool vec, uint32_t u0, uint32_t u1,
                                 Smem& sm) {
  constexpr int EPU = DT == SD_F32_PROBS ? 4 : 8;
  float best = -INFINITY;
  uint32_t bx = 0xffffffffu;
  const uint32_t uf = vec ? max(u0, min(u1, V / EPU)) : u0;
  uint32_t ub = u0 + threadIdx.x;
  auto take = [&](const uint4& v, uint32_t u) {
    const uint32_t x0 = u * EPU;
    if (DT == SD_F32_PROBS) {
      argmax_take(__uint_as_float(v.x), x0 + 0, best, bx);
      argmax_take(__uint_as_float(v.y), x0 + 1, best, bx);
      argmax_take(__uint_as_float(v.z), x0 + 2, best, bx);
      argmax_take(__uint_as_float(v.w), x0 + 3, best, bx);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) argmax_take(bf16_at(v, i), x0 + i, best, bx);
    }
  };
  auto load = [&](uint32_t u) { return ld_stream_u4((const char*)row + (size_t)u * 16u); };
  if (ub + (kArgmaxUnroll - 1) * NT < uf) {  // unchecked 128-bit loads, kArgmaxUnroll units always in flight
    uint4 v[kArgmaxUnroll];
#pragma unroll
    for (int k = 0; k < kArgmaxUnroll; ++k) v[k] = load(ub + k * NT);
    for (; ub + (2 * kArgmaxUnroll - 1) * NT < uf; ub += kArgmaxUnroll * NT) {
#pragma unroll
      for (int k = 0; k < kArgmaxUnroll; ++k) {
        take(v[k], ub + k * NT);
        v[k] = load(ub + (k + kArgmaxUnroll) * NT);
      }
    }
#pragma unroll
    for (int k = 0; k < kArgmaxUnroll; ++k) take(v[k], ub + k * NT);
    ub += kArgmaxUnroll * NT;
  }
  for (; ub < u1; ub += NT) {  // the rest, bounds-checked
    if (DT == SD_F32_PROBS) {
      float v[4];
      f32_unit((const float*)row, ub, V, vec, -INFINITY, v);
#pragma unroll
      for (int i = 0; i < 4; ++i) argmax_take(v[i], ub * 4 + i, best, bx);
    } else {
      const uint4 v = bf16_raw((const uint16_t*)row, ub, V, vec);
#pragma unroll
      for (int i = 0; i < 8; ++i) argmax_take(bf16_at(v, i), ub * 8 + i, best, bx);
    }
  }
  const uint64_t pk = (bx == 0xffffffffu) ? 0ull : pack_key(orderable(best), bx);
  return block_max_u64<NT>(pk, sm.red);
}

// Argmax of two rows at once over units [u0, u1) (greedy rows j and j+1): both rows' loads in
// flight together, the two block maxima in one reduction.
template <int DT>
__device__ void argmax_chunk2(const void* row0, const void* row1, uint32_t V, bool vec,
                              uint32_t u0, uint32_t u1, Smem& sm, uint64_t& pk0, uint64_t& pk1) {
  constexpr int EPU = DT == SD_F32_PROBS ? 4 : 8;
  constexpr int U = kArgmaxUnroll / 2;  // units in flight per row
  float best0 = -INFINITY, best1 = -INFINITY;
  uint32_t bx0 = 0xffffffffu, bx1 = 0xffffffffu;
  const uint32_t uf = vec ? max(u0, min(u1, V / EPU)) : u0;
  uint32_t ub = u0 + threadIdx.x;
  auto take = [&](const uint4& v, uint32_t u, float& best, uint32_t& bx) {
    const uint32_t x0 = u * EPU;
    if (DT == SD_F32_PROBS) {
      argmax_take(__uint_as_float(v.x), x0 + 0, best, bx);
      argmax_take(__uint_as_float(v.y), x0 + 1, best, bx);
      argmax_take(__uint_as_float(v.z), x0 + 2, best, bx);
      argmax_take(__uint_as_float(v.w), x0 + 3, best, bx);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) argmax_take(bf16_at(v, i), x0 + i, best, bx);
    }
  };
  auto load = [&](const void* row, uint32_t u) {
    return ld_stream_u4((const char*)row + (size_t)u * 16u);
  };
  if (ub + (U - 1) * NT < uf) {  // unchecked 128-bit loads, U units of each row in flight
    uint4 v0[U], v1[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      v0[k] = load(row0, ub + k * NT);
      v1[k] = load(row1, ub + k * NT);
    }
    for (; ub + (2 * U - 1) * NT < uf; ub += U * NT) {
#pragma unroll
      for (int k = 0; k < U; ++k) {
        take(v0[k], ub + k * NT, best0, bx0);
        take(v1[k], ub + k * NT, best1, bx1);
        v0[k] = load(row0, ub + (k + U) * NT);
        v1[k] = load(row1, ub + (k + U) * NT);
      }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      take(v0[k], ub + k * NT, best0, bx0);
      take(v1[k], ub + k * NT, best1, bx1);
    }
    ub += U * NT;
  }
  for (; ub < u1; ub += NT) {  // the rest, bounds-checked
    if (DT == SD_F32_PROBS) {
      float a[4], b[4];
      f32_unit((const float*)row0, ub, V, vec, -INFINITY, a);
      f32_unit((const float*)row1, ub, V, vec, -INFINITY, b);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        argmax_take(a[i], ub * 4 + i, best0, bx0);
        argmax_take(b[i], ub * 4 + i, best1, bx1);
      }
    } else {
      const uint4 a = bf16_raw((const uint16_t*)row0, ub, V, vec);
      const uint4 b = bf16_raw((const uint16_t*)row1, ub, V, vec);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        argmax_take(bf16_at(a, i), ub * 8 + i, best0, bx0);
        argmax_take(bf16_at(b, i), ub * 8 + i, best1, bx1);
      }
    }
  }
  uint64_t p0 = (bx0 == 0xffffffffu) ? 0ull : pack_key(orderable(best0), bx0);
  uint64_t p1 = (bx1 == 0xffffffffu) ? 0ull : pack_key(orderable(best1), bx1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t x0 = __shfl_xor_sync(0xffffffffu, p0, o);
    const uint64_t x1 = __shfl_xor_sync(0xffffffffu, p1, o);
    p0 = x0 > p0 ? x0 : p0;
    p1 = x1 > p1 ? x1 : p1;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) {
    sm.red[warp] = p0;
    sm.red2[warp] = p1;
  }
  __syncthreads();
  p0 = 0ull;
  p1 = 0ull;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    p0 = sm.red[w] > p0 ? sm.red[w] : p0;
    p1 = sm.red2[w] > p1 ? sm.red2[w] : p1;
  }
  pk0 = p0;
  pk1 = p1;
}

// ------------------------------------------------------------ softmax statistics (bf16 rows)
// Per row the cluster forms S = sum_x 2^(l_x c - ref c) for a fixed reference logit ref: the
// draft token's own logit (element 0 of the row for the bonus row or an out-of-range draft).
// p(x) = 2^(l_x c - ref c) / S is the softmax whatever the reference, so no running maximum is
// kept and the partial sums combine by plain addition, in a fixed order (the results do not
// depend on timing). Every term is at most S, so S < kRefSumLimit certifies that no term
// overflowed; otherwise (extreme logits or temperatures) the row is summed again with the
// row's maximum as the reference. Terms flush to 0 below 2^-126, far below the reference term.
constexpr float kRefSumLimit = 0x1p100f;
constexpr int kLookAhead = 4;  // the next row's first 1/kLookAhead is streamed during the exchange

// Compensated running sums, kept as two lanes (even and odd elements of each 32-bit word pair)
// so that the scaling, the sums and the compensation run as packed fp32x2 instructions: half the
// issue slots of the scalar forms, each lane rounded exactly as the scalar operation would be.
struct RefAcc {
  float2 s = make_float2(0.0f, 0.0f), comp = make_float2(0.0f, 0.0f);
  __device__ __forceinline__ float total() const { return (s.x - comp.x) + (s.y - comp.y); }
};

__device__ __forceinline__ void absorb_ref(RefAcc& a, const uint4& raw, float c, float nrc) {
  const float2 c2 = make_float2(c, c), n2 = make_float2(nrc, nrc), m1 = make_float2(-1.0f, -1.0f);
  const uint32_t v[4] = {raw.x, raw.y, raw.z, raw.w};
  float2 e[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // elements 2i (low half) and 2i+1 (high half): l c + nrc, as logit_term rounds it
    const float2 l = make_float2(__uint_as_float(v[i] << 16), __uint_as_float(v[i] & 0xffff0000u));
    const float2 y = __ffma2_rn(l, c2, n2);
    e[i] = make_float2(fast_ex2(y.x), fast_ex2(y.y));
  }
  const float2 part = __fadd2_rn(__fadd2_rn(e[0], e[1]), __fadd2_rn(e[2], e[3]));
  const float2 y = __ffma2_rn(a.comp, m1, part);               // part - comp
  const float2 t = __fadd2_rn(a.s, y);
  a.comp = __ffma2_rn(y, m1, __ffma2_rn(a.s, m1, t));          // (t - s) - y
  a.s = t;
}

// Units [u0, u1) of target row trow (and, with HAS_Q, draft row drow) into the accumulators.
template <bool HAS_Q>
__device__ __forceinline__ void ref_sums(const uint16_t* trow, const uint16_t* drow, uint32_t V,
                                         bool vec, uint32_t u0, uint32_t u1, float c, float nrct,
                                         float nrcd, RefAcc& at, RefAcc& ad) {
  const uint32_t uf = vec ? max(u0, min(u1, V / 8u)) : u0;
  uint32_t ub = u0 + threadIdx.x;
  if (ub + (UNROLL - 1) * NT < uf) {  // unchecked 128-bit loads, UNROLL units always in flight
    uint4 vt[UNROLL], vd[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      vt[k] = ld_stream_u4(trow + 8u * (ub + k * NT));
      if (HAS_Q) vd[k] = ld_stream_u4(drow + 8u * (ub + k * NT));
    }
    for (; ub + (2 * UNROLL - 1) * NT < uf; ub += UNROLL * NT) {
#pragma unroll
      for (int k = 0; k < UNROLL; ++k) {
        absorb_ref(at, vt[k], c, nrct);
        if (HAS_Q) absorb_ref(ad, vd[k], c, nrcd);
        vt[k] = ld_stream_u4(trow + 8u * (ub + (k + UNROLL) * NT));
        if (HAS_Q) vd[k] = ld_stream_u4(drow + 8u * (ub + (k + UNROLL) * NT));
      }
    }
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      absorb_ref(at, vt[k], c, nrct);
      if (HAS_Q) absorb_ref(ad, vd[k], c, nrcd);
    }
    ub += UNROLL * NT;
  }
  for (; ub < u1; ub += NT) {  // the rest, bounds-checked (-inf past the row end: term 0)
    absorb_ref(at, bf16_raw(trow, ub, V, vec), c, nrct);
    if (HAS_Q) absorb_ref(ad, bf16_raw(drow, ub, V, vec), c, nrcd);
  }
}

// Sums of two values over the CTA, in a fixed order (every thread gets them). `par` alternates
// between calls, so one barrier per call suffices.
__device__ __forceinline__ float2 block_sum2(float a, float b, Smem& sm, int& par) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) sm.redf[par][warp] = make_float2(a, b);
  __syncthreads();
  float2 t = sm.redf[par][0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) {
    t.x += sm.redf[par][w].x;
    t.y += sm.redf[par][w].y;
  }
  par ^= 1;
  return t;
}

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Post this CTA's row sums for the cluster and arrive (the wait comes later, in
// cluster_collect, so that the exchange overlaps the next row's first units).
__device__ __forceinline__ void cluster_post(float2 v, float2* slot, int cl) {
  if (cl == 1) return;
  if (threadIdx.x == 0) *slot = v;
  cluster_arrive_release();
}

// Wait, then the cluster's sums (mine for cl == 1): in every warp lanes 0..cl-1 read rank
// lane's slot and reduce in a fixed order, so every CTA gets the same bits.
__device__ __forceinline__ float2 cluster_collect(float2 mine, float2* slot, int cl) {
  if (cl == 1) return mine;
  cluster_wait_acquire();
  const int lane = threadIdx.x & 31;
  float2 v = make_float2(0.0f, 0.0f);
  if (lane < cl) v = load_from_rank(slot, (unsigned)lane);
  for (int o = cl >> 1; o > 0; o >>= 1) {
    v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
    v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
  }
  v.x = __shfl_sync(0xffffffffu, v.x, 0);
  v.y = __shfl_sync(0xffffffffu, v.y, 0);
  return v;
}

// Largest logit of two rows over the cluster (drow may be NULL: -inf), for the max-referenced
// recomputation of a row's sums.
__device__ void row_max2(const uint16_t* trow, const uint16_t* drow, uint32_t V, bool vec,
                         uint32_t u0, uint32_t u1, Smem& sm, int& phase, int cl, float& mt,
                         float& md) {
  float a = -INFINITY, b = -INFINITY;
  for (uint32_t u = u0 + threadIdx.x; u < u1; u += NT) {
    const uint4 t = bf16_raw(trow, u, V, vec);
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, bf16_at(t, i));
    if (drow) {
      const uint4 d = bf16_raw(drow, u, V, vec);
#pragma unroll
      for (int i = 0; i < 8; ++i) b = fmaxf(b, bf16_at(d, i));
    }
  }
  // maxima as orderable bits, over the CTA, then over the cluster
  uint64_t pa = orderable(a), pb = orderable(b);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t xa = __shfl_xor_sync(0xffffffffu, pa, o);
    const uint64_t xb = __shfl_xor_sync(0xffffffffu, pb, o);
    pa = xa > pa ? xa : pa;
    pb = xb > pb ? xb : pb;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) {
    sm.red[warp] = pa;
    sm.red2[warp] = pb;
  }
  __syncthreads();
  pa = 0ull;
  pb = 0ull;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    pa = sm.red[w] > pa ? sm.red[w] : pa;
    pb = sm.red2[w] > pb ? sm.red2[w] : pb;
  }
  cluster_max2_u64(pa, pb, sm, phase, cl);
  auto unorder = [](uint32_t u) {
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
  };
  mt = unorder((uint32_t)pa);
  md = unorder((uint32_t)pb);
}

// The race on a logit row pair (HAS_Q) or on p alone, over the cluster: out of line, so that its
// registers do not add to the statistics loop's.
template <bool HAS_Q>
__device__ __forceinline__ uint64_t logit_race(const uint16_t* t, const uint16_t* d, float nrct,
                                            float invSt, float nrcd, float invSd, float c,
                                            uint32_t V, bool vec, uint32_t u0, uint32_t u1,
                                            const PhiloxRoundKeys& rk, uint32_t rid, uint32_t j,
                                            Smem& sm, int& phase, int cl) {
  const Bf16Residual<HAS_Q> src{t, d, nrct, invSt, nrcd, invSd, c, V, vec};
  return cluster_max_u64(race_chunk(src, u0, u1, rk, rid, j, sm), sm, phase, cl);
}

// A row's sums again against the row maxima (the rare case where the draft token's logit is too
// far below the row's largest for the terms to stay finite). Returns S and the new nrc's.
__device__ __noinline__ float2 logit_row_refit(const uint16_t* trow, const uint16_t* drow,
                                               uint32_t V, bool vec, uint32_t u0, uint32_t u1,
                                               float c, Smem& sm, int& phase, int& par, int cl,
                                               float& nrct, float& nrcd) {
  float mt, md;
  row_max2(trow, drow, V, vec, u0, u1, sm, phase, cl, mt, md);
  nrct = -__fmul_rn(mt, c);
  nrcd = drow ? -__fmul_rn(md, c) : 0.0f;
  RefAcc ft, fd;
  if (drow) ref_sums<true>(trow, drow, V, vec, u0, u1, c, nrct, nrcd, ft, fd);
  else ref_sums<false>(trow, nullptr, V, vec, u0, u1, c, nrct, 0.0f, ft, fd);
  const float2 fm = block_sum2(ft.total(), fd.total(), sm, par);
  cluster_post(fm, &sm.xslot_fb, cl);
  return cluster_collect(fm, &sm.xslot_fb, cl);
}

// -------------------------------------------------------- sampled probability requests (shared)
// Accept scan of request r by one warp (lane j checks draft d_{j+1}); P/Q of the examined drafts
// go to Ps/Qs (others stay as they are). Returns a_r; *bad_out receives SD_ERR_TOKEN_RANGE when
// the first rejection came from an out-of-range draft.
// Whether draft j of request r (rows rr, probability rows) is accepted: d_{j+1} in [0, V) and
// u_j * Q < P, compared exactly in double (u*Q is exact there). P, Q: the values at the draft
// (0 for an out-of-range token, which sets bad and counts as rejected).
__device__ __forceinline__ bool draft_accepted(const VerifyParams& P, const ReqRows& rr, int r,
                                               int j, float& Pv, float& Qv, bool& bad) {
  const uint32_t V = (uint32_t)P.V;
  Pv = 0.0f;
  Qv = 0.0f;
  bad = false;
  const int d = __ldg(P.drafts + rr.d0 + j);
  if (d < 0 || (uint32_t)d >= V) {
    bad = true;
    return false;
  }
  Pv = __ldg((const float*)P.target + (rr.t0 + j) * P.ld_t + d);
  Qv = __ldg((const float*)P.draft + (rr.d0 + j) * P.ld_d + d);
  const double u = accept_uniform(P.rk, P.rbase + (uint32_t)r, (uint32_t)j);
  return u * (double)Qv < (double)Pv;
}

__device__ int accept_scan_warp(const VerifyParams& P, int r, float* Ps, float* Qs, int* bad_out) {
  const ReqRows rr = req_rows(P, r);
  const int K = rr.k;
  const int j = threadIdx.x & 31;
  bool acc = false, bad = false;
  float Pv = 0.0f, Qv = 0.0f;
  if (j < K) acc = draft_accepted(P, rr, r, j, Pv, Qv, bad);
  const unsigned rej = __ballot_sync(0xffffffffu, j < K && !acc);
  const int av = rej ? __ffs(rej) - 1 : K;
  if (j < K && j <= av) {
    Ps[j] = Pv;
    Qs[j] = Qv;
  }
  const unsigned badm = __ballot_sync(0xffffffffu, bad && j == av);
  *bad_out = (badm ? SD_ERR_TOKEN_RANGE : 0) | rr.e;
  return av;
}

// Outputs of one request: d_1..d_a, b, -1 padding, a, P/Q at the drafts (the whole CTA writes).
__device__ void write_request(const VerifyParams& P, int r, int a, uint32_t b, int32_t e,
                              const float* Ps, const float* Qs) {
  const int K = P.K;
  const size_t d0 = req_rows(P, r).d0;
  const int t = threadIdx.x;
  if (t <= K) {
    int32_t tok = -1;
    if (t < a) tok = __ldg(P.drafts + d0 + t);
    else if (t == a) tok = (int32_t)b;
    P.out_tokens[(size_t)r * (K + 1) + t] = tok;
  }
  if (t < K) {
    if (P.p_at) P.p_at[(size_t)r * K + t] = Ps[t];
    if (P.q_at) P.q_at[(size_t)r * K + t] = Qs[t];
  }
  if (t == 0) {
    P.num_accepted[r] = a;
    raise_err(P.err, e);
  }
}

// Merge a CTA's packed race maximum over `units` units of request r's race row into its slot.
// Returns (in every thread) whether this CTA completed the row, and then the row's maximum.
__device__ bool merge_slot(RaceSlot* slot, uint64_t pk, uint32_t units, uint32_t row_units,
                           Smem& sm, uint64_t& row_max) {
  if (threadIdx.x == 0) {
    if (pk) atomicMax(&slot->best, (unsigned long long)pk);
    __threadfence();
    const unsigned prev = atomicAdd(&slot->count, units);
    const bool last = prev + units == row_units;
    sm.last = last;
    if (last) {
      __threadfence();
      sm.bcast = atomicOr(&slot->best, 0ull);  // every other part of the row is merged by now
    }
  }
  __syncthreads();
  const bool last = sm.last != 0;
  row_max = sm.bcast;
  __syncthreads();
  return last;
}

// The CTA that completed request r's race row: fallback and outputs, then the slot is zeroed.
// Request r's final token from its completed race row (maximum pk): the fallback race on p when
// no residual key is positive, SD_ERR_ZERO_ROW into e when even p has none; the merge slot is
// cleared for the next call.
__device__ uint32_t final_token(const VerifyParams& P, int r, int a, uint64_t pk, int32_t& e,
                                Smem& sm) {
  const ReqRows rr = req_rows(P, r);
  const int K = rr.k;
  const uint32_t V = (uint32_t)P.V;
  const uint32_t NU = (V + 3u) / 4u;
  const bool vec = P.vec != 0;
  const int jr = a < K ? a : K;
  const float* prow = (const float*)P.target + (rr.t0 + jr) * P.ld_t;
  if (packed_key_bits(pk) == 0u && a < K) {
    // no positive residual key anywhere in the row: race on p of the same row, whole row
    F32Residual<false> src{prow, nullptr, V, vec};
    pk = race_chunk(src, 0u, NU, P.rk, P.rbase + (uint32_t)r, (uint32_t)jr, sm);
  }
  uint32_t b = 0;
  if (packed_key_bits(pk) == 0u) e |= SD_ERR_ZERO_ROW;
  else b = packed_index(pk);
  if (threadIdx.x == 0) {
    P.slots[r].best = 0ull;
    P.slots[r].count = 0u;
  }
  return b;
}

__device__ __noinline__ uint32_t finish_sampled(const VerifyParams& P, int r, int a, int32_t e,
                                                uint64_t pk, const float* Ps, const float* Qs,
                                                Smem& sm) {
  const uint32_t b = final_token(P, r, a, pk, e, sm);
  write_request(P, r, a, b, e, Ps, Qs);
  return b;
}

// ------------------------------------------------------------------------- fused rebuild
// Sum over the CTA (every thread gets it).
__device__ long long block_sum_ll(long long v, Smem& sm) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();  // sm.red may still be read by a previous reduction
  if ((threadIdx.x & 31) == 0) sm.red[threadIdx.x >> 5] = (uint64_t)v;
  __syncthreads();
  long long t = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) t += (long long)sm.red[w];
  return t;
}

// Largest batch the fused rebuild takes: every rebuild CTA redoes the accept scans of the
// requests before its own (kMaxFuseB * SD_K_MAX draft decisions at most, two loads each).
constexpr int kMaxFuseB = 192;

// The rebuild role of request r (sd_verify_prepare, CTA r of the launch). It needs the accepted
// counts of requests 0..r, which depend only on the inputs: it recomputes them (the same
// decisions as the accept scan, all drafts at once), takes its request's first drafter slot as
// their prefix, and writes r's drafter rows and hidden states -- all while the other CTAs race.
// Only the final token at slot a_r waits for the race: the CTA that completes r's race row writes
// it, at the slot this CTA publishes in r's merge slot. The rebuild CTA of the last request also
// writes total_out, start_loc[B] and the padding tail.
__device__ __noinline__ void rebuild_role(const VerifyParams& P, int r, Smem& sm) {
  __shared__ int acc_s[kMaxFuseB];  // a_q, then (after the scan) a_q + K_q
  const RebuildArgs& R = P.rb;
  const int KM = P.K, n = r + 1;  // K_max with per-request counts
  for (int q = threadIdx.x; q < n; q += NT) acc_s[q] = req_rows(P, q).k;
  __syncthreads();
  for (int p = threadIdx.x; p < n * KM; p += NT) {
    const int q = p / KM, j = p - q * KM;
    const ReqRows rq = req_rows(P, q);
    if (j >= rq.k) continue;
    float Pv, Qv;
    bool bad;
    if (!draft_accepted(P, rq, q, j, Pv, Qv, bad)) atomicMin(&acc_s[q], j);
  }
  __syncthreads();
  const ReqRows rr = req_rows(P, r);
  const int K = rr.k, a = acc_s[r], L = a + K;
  long long part = 0;
  for (int q = threadIdx.x; q < r; q += NT) part += acc_s[q] + req_rows(P, q).k;
  const long long off = block_sum_ll(part, sm);
  int32_t e = 0;
  const int pos0 = __ldg(R.pos0 + r);
  const int32_t* bt_row = R.block_table + (size_t)r * R.max_blocks;
  for (int j = threadIdx.x; j < L; j += NT) {
    const long long g = off + j;
    if (g >= R.capacity) {
      e |= SD_ERR_TOTAL_RANGE;
      continue;
    }
    // slot a_r's token is the race's result: its CTA writes it (the tail of the race role)
    const int32_t tok = j < a ? __ldg(P.drafts + rr.d0 + j) : R.mask_id;
    write_drafter_slot(g, j, a, tok, R.mask_id, pos0, bt_row, R.max_blocks, R.block_size,
                       (long long)rr.t0, j == a ? nullptr : R.input_ids, R.positions,
                       R.slot_mapping, R.hidden_map, R.is_masked, e);
  }
  const int t = threadIdx.x;
  if (t <= KM) R.is_rejected[(size_t)r * (KM + 1) + t] = (t >= 1 && t > a && t <= K) ? 1 : 0;
  if (t < KM) R.new_token_idx[(size_t)r * KM + t] = t < K ? (int32_t)(off + a + t) : -1;
  if (t == 0) {
    R.start_loc[r] = (int32_t)off;
    unsigned* slot = &P.slots[r].off1;
    if (r == P.withhold) {
      // diagnostic: hold the publication back until the race CTA has given up (bounded)
      const uint64_t t0 = globaltimer_ns();
      while (*(volatile unsigned*)slot != kGaveUp &&
             globaltimer_ns() - t0 < 4 * P.wait_ns + 50000000ull) {
      }
    }
    // publish, unless the completing race CTA already gave up: then put the slot back to 0
    if (atomicCAS(slot, 0u, (unsigned)(off + 1)) == kGaveUp) atomicExch(slot, 0u);
  }
  if (R.out_hidden) {
    const long long nrows = min((long long)L, (long long)R.capacity - off);
    for (long long j = t >> 5; j < nrows; j += NT / 32)
      gather_row_warp(j <= a ? (long long)rr.t0 + j : -1, R.hidden, R.ld_in, R.n_in_rows,
                      R.h_shared, R.out_hidden + (off + j) * R.ld_out, R.H, R.hvec != 0, t & 31,
                      e);
  }
  if (r == P.B - 1) {
    const long long tot = off + L;
    if (t == 0) {
      R.start_loc[P.B] = (int32_t)tot;
      *R.total_out = (int32_t)tot;
    }
    for (long long i = tot + t; i < R.capacity; i += NT)
      write_padding_slot(i, R.input_ids, R.positions, R.slot_mapping, R.hidden_map, R.is_masked);
  }
  if (e) raise_err(P.err, e);
}

// The padded rebuild role of request r (sd_verify_prepare_padded, CTA r of the launch): request r
// owns drafter rows [r*2K, (r+1)*2K) whatever the other requests accept, so the CTA needs only
// its own request's accept decisions (recomputed from the inputs, all K at once) and writes every
// row of the request -- the same bytes as the padded rebuild kernel -- except the token at row
// r*2K + a_r, which the CTA that completes the request's race writes.
__device__ __noinline__ void padded_rebuild_role(const VerifyParams& P, int r, Smem& sm) {
  const RebuildArgs& R = P.rb;
  const int K = P.K, W = 2 * K;
  const ReqRows rr = req_rows(P, r);
  if (threadIdx.x == 0) sm.a = K;
  __syncthreads();
  if (threadIdx.x < (unsigned)K) {
    float Pv, Qv;
    bool bad;
    if (!draft_accepted(P, rr, r, (int)threadIdx.x, Pv, Qv, bad)) atomicMin(&sm.a, (int)threadIdx.x);
  }
  __syncthreads();
  const int a = sm.a;
  int32_t e = 0;
  const int p0 = __ldg(R.pos0 + r);
  const long long row0 = (long long)r * W;
  for (int j = threadIdx.x; j < W; j += NT) {
    const long long row = row0 + j;
    const bool live = j < a + K;
    const long long pos = (long long)p0 + 1 + j;
    int32_t slot = -1;
    if (live) {
      const long long blk = pos >= 0 ? pos / R.block_size : -1;
      if (blk < 0 || blk >= R.max_blocks) {
        e |= SD_ERR_BLOCK_TABLE;
      } else {
        const long long phys = __ldg(R.block_table + (size_t)r * R.max_blocks + blk);
        const long long sl = phys * R.block_size + pos % R.block_size;
        if (phys < 0 || sl > 2147483647LL) e |= SD_ERR_BLOCK_TABLE;
        else slot = (int32_t)sl;
      }
    }
    // row a_r's token is the race's result: its CTA writes it
    if (j < a) R.input_ids[row] = __ldg(P.drafts + rr.d0 + j);
    else if (j > a) R.input_ids[row] = R.mask_id;
    R.positions[row] = (int32_t)pos;
    R.slot_mapping[row] = slot;
    R.hidden_map[row] = (j <= a) ? (int32_t)(rr.t0 + j) : -1;
    R.is_masked[row] = (live && j > a) ? 1 : 0;
    R.rejected[row] = live ? 0 : 1;
    if (j <= K) R.scatter_map[rr.t0 + j] = (j <= a) ? (int32_t)row : -1;
    if (j < K) R.new_token_idx[(size_t)r * K + j] = (int32_t)(row0 + a + j);
  }
  if (R.out_hidden) {
    for (int j = threadIdx.x >> 5; j < W; j += NT / 32)
      gather_row_warp(j <= a ? (long long)rr.t0 + j : -1, R.hidden, R.ld_in, R.n_in_rows,
                      R.h_shared, R.out_hidden + (row0 + j) * R.ld_out, R.H, R.hvec != 0,
                      threadIdx.x & 31, e);
  }
  if (e) raise_err(P.err, e);
}

// The CTA that completed request r's race row in the fused launch: the verify outputs (as
// write_request) and the final token at slot a_r of the drafter batch, at the first slot the
// rebuild CTA published (long before any race row completes; the wait is bounded by time all
// the same, and if it runs out the token is not written and SD_ERR_WAIT is raised).
// tok_pre (thread t < K: draft t) and off_pre (thread 0: the published slot + 1, or 0 if not yet
// seen) were read before the merge, so that their round trips overlap the merge's. No acquire is
// needed: the CTA reads nothing else the rebuild CTA wrote, and writes a slot it leaves alone.
__device__ __noinline__ void fused_finish(const VerifyParams& P, int r, int a, int32_t e,
                                          uint64_t pk, const float* Ps, const float* Qs,
                                          int32_t tok_pre, unsigned off_pre, Smem& sm) {
  const uint32_t b = final_token(P, r, a, pk, e, sm);
  const int K = P.K, t = threadIdx.x;
  if (t <= K) P.out_tokens[(size_t)r * (K + 1) + t] = t < a ? tok_pre : (t == a ? (int32_t)b : -1);
  if (t < K) {
    if (P.p_at) P.p_at[(size_t)r * K + t] = Ps[t];
    if (P.q_at) P.q_at[(size_t)r * K + t] = Qs[t];
  }
  if (t == 0 && P.fuse == 2) {
    // the padded layout: request r's row a_r is r*2K + a_r, no published slot to wait for
    P.num_accepted[r] = a;
    P.rb.input_ids[(size_t)r * 2 * K + a] = (int32_t)b;
    raise_err(P.err, e);
  } else if (t == 0) {
    P.num_accepted[r] = a;
    unsigned* slot = &P.slots[r].off1;
    unsigned v = off_pre;
    if (v == 0u) {
      const uint64_t t0 = globaltimer_ns();
      for (uint32_t it = 0;; ++it) {
        v = *(volatile unsigned*)slot;
        if (v != 0u) break;
        if (it >= kMinPolls && globaltimer_ns() - t0 > P.wait_ns) {
          // give up, unless the slot was published in the meantime; the rebuild CTA then sees
          // kGaveUp and puts the slot back to 0
          v = atomicCAS(slot, 0u, kGaveUp);
          break;
        }
      }
    }
    if (v == 0u) {
      e |= SD_ERR_WAIT;
    } else {
      // slot a_r exists when the request has drafter slots at all (K_r > 0: L_r = a_r + K_r)
      const long long g = (long long)v - 1 + a;
      if (req_rows(P, r).k > 0 && g < P.rb.capacity) P.rb.input_ids[g] = (int32_t)b;
      atomicExch(slot, 0u);
    }
    raise_err(P.err, e);
  }
}

// The race kernel: an all-sampled batch in one launch. The requests' race rows are laid end to
// end (unit u of request r at position r*NU + u) and that line is split evenly over race_blocks
// CTAs (a whole number per SM). Every unit costs the same Philox and filter arithmetic, and that,
// more than the one or two rows a unit reads, sets a CTA's time (measured: balancing by bytes
// instead was slower), so every SM gets the same number of units. The split does not depend on
// which row a request races on, so each CTA first runs the accept scan of the few requests its
// share touches (one warp each; CTAs sharing a request compute the same result), then races over
// its segments; the CTA that completes a request's row writes all of that request's outputs.
struct AcceptState {
  float P[kMaxSeg][SD_K_MAX], Q[kMaxSeg][SD_K_MAX];
  int a[kMaxSeg], e[kMaxSeg];
};

__device__ __forceinline__ void race_role(const VerifyParams& P, uint32_t c, Smem& sm,
                                          AcceptState& as) {
  const uint32_t V = (uint32_t)P.V;
  const uint32_t NU = (V + 3u) / 4u;
  const bool vec = P.vec != 0;
  const unsigned long long W = (unsigned long long)P.B * NU;
  const unsigned long long w0 = W * c / (unsigned)P.race_blocks;
  const unsigned long long w1 = W * (c + 1) / (unsigned)P.race_blocks;
  if (w1 <= w0) return;  // CTA-uniform
  const int r0 = (int)(w0 / NU), r1 = (int)((w1 - 1) / NU);  // at most kMaxSeg requests
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp <= r1 - r0) {  // warp-uniform
    if (lane < SD_K_MAX) {
      as.P[warp][lane] = -1.0f;
      as.Q[warp][lane] = -1.0f;
    }
    __syncwarp();
    int bad;
    const int a = accept_scan_warp(P, r0 + warp, as.P[warp], as.Q[warp], &bad);
    if (lane == 0) {
      as.a[warp] = a;
      as.e[warp] = bad;
    }
  }
  if (threadIdx.x == 0) sm.tau = 0u;
  __syncthreads();
  for (int r = r0; r <= r1; ++r) {
    const unsigned long long base = (unsigned long long)r * NU;
    const uint32_t lo = (uint32_t)(max(w0, base) - base);
    const uint32_t hi = (uint32_t)(min(w1, base + NU) - base);
    const int i = r - r0;
    const int a = as.a[i];
    const ReqRows rr = req_rows(P, r);
    const int K = rr.k;
    const int jr = a < K ? a : K;
    const float* prow = (const float*)P.target + (rr.t0 + jr) * P.ld_t;
    const float* qrow = a < K ? (const float*)P.draft + (rr.d0 + jr) * P.ld_d : nullptr;
    const F32ResidualAny src{prow, qrow, V, vec};
    const uint64_t pk = race_chunk(src, lo, hi, P.rk, P.rbase + (uint32_t)r, (uint32_t)jr, sm);
    uint64_t row_max;
    if (merge_slot(P.slots + r, pk, hi - lo, NU, sm, row_max))
      finish_sampled(P, r, a, as.e[i], row_max, as.P[i], as.Q[i], sm);
  }
}

// ---------------------------------------------------------------------------------- the kernel
template <int DT>
__global__ void __launch_bounds__(NT, min_blocks(DT))
    verify_kernel(const __grid_constant__ VerifyParams P) {
  __shared__ Smem sm;
  constexpr int EPU = (DT == SD_F32_PROBS) ? 4 : 8;
  using Elt = typename std::conditional<DT == SD_F32_PROBS, float, uint16_t>::type;
  // When launched as a programmatic dependent, wait until the preceding grid's writes (possibly
  // this launch's inputs) are visible; otherwise this returns at once.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int nc = P.nc;
  uint32_t rank;  // this CTA's index within its request
  int r;
  if constexpr (DT == SD_F32_PROBS) {
    if (P.fuse) {
      // sd_verify_prepare's single launch: CTAs [0, B) rebuild the drafter batch, CTAs
      // [B, grid) race, dealt out to the requests as evenly as they go (request r takes race
      // CTAs [floor(r G / B), floor((r+1) G / B)) of the G = grid - B)
      if (blockIdx.x < (unsigned)P.B) {
        if (P.fuse == 2) padded_rebuild_role(P, (int)blockIdx.x, sm);
        else rebuild_role(P, (int)blockIdx.x, sm);
        return;
      }
      const uint64_t G = gridDim.x - (uint64_t)P.B, Bq = (uint64_t)P.B;
      const uint64_t c = blockIdx.x - (uint64_t)P.B;
      r = (int)(((c + 1) * Bq - 1) / G);
      const uint64_t s0 = (uint64_t)r * G / Bq;
      nc = (int)((uint64_t)(r + 1) * G / Bq - s0);
      rank = (uint32_t)(c - s0);
    }
  }
  if (!(DT == SD_F32_PROBS && P.fuse)) {
    rank = blockIdx.x % (unsigned)nc;
    r = (int)(blockIdx.x / (unsigned)nc);
  }
  const ReqRows rr = req_rows(P, r);
  const int K = rr.k;    // this request's drafts
  const int KM = P.K;    // the output stride
  const uint32_t V = (uint32_t)P.V;
  const bool vec = P.vec != 0;
  const uint32_t NU = (V + EPU - 1) / EPU;
  const Elt* tbase = (const Elt*)P.target + rr.t0 * P.ld_t;
  const Elt* dbase = (const Elt*)P.draft + rr.d0 * P.ld_d;
  auto trow = [&](int j) { return tbase + (size_t)j * P.ld_t; };
  auto drow = [&](int j) { return dbase + (size_t)j * P.ld_d; };
  const int32_t* dr = P.drafts + rr.d0;
  const float T = P.temperature ? P.temperature[r] : 1.0f;
  const bool greedy = (T == 0.0f);
  const bool sampled_probs = DT == SD_F32_PROBS && !greedy;
  // Sampled probability requests split their race row over the request's CTAs (in a cluster
  // launch, a mixed batch, over half of them: each then streams twice the units between its
  // fixed costs, the accept scan and the merge, and the others leave at once; 1% faster on 256
  // requests of 151936-entry rows, half of them greedy, with the same outputs); greedy and logit
  // requests use the first cluster only (whole clusters beyond it leave at once).
  // sampled probability requests belong to race_kernel when it is launched
  if (sampled_probs && P.race_blocks > 0) return;
  const int cl = sampled_probs ? (P.cl > 1 ? nc / 2 : nc) : P.cl;
  if (rank >= (uint32_t)cl) return;
  const uint32_t crank = rank;
  const uint32_t u0 = (uint32_t)(((uint64_t)NU * crank) / (unsigned)cl);
  const uint32_t u1 = (uint32_t)(((uint64_t)NU * (crank + 1)) / (unsigned)cl);
  int phase = 0;
  int a = K;
  uint32_t b = 0;
  int32_t e = rr.e;
  bool writer = crank == 0;  // the CTA that writes the request's outputs
  const int lane = threadIdx.x & 31;

  if (threadIdx.x < SD_K_MAX) {
    sm.P[threadIdx.x] = -1.0f;
    sm.Q[threadIdx.x] = -1.0f;
  }
  if constexpr (DT == SD_BF16_LOGITS) {
    // logit rows: each row's reference logits (the draft token's, element 0 when it is out of
    // range or for the bonus row), read once before any row is streamed
    if (!greedy && threadIdx.x <= (unsigned)K) {
      const int j = threadIdx.x;
      int x = 0;
      if (j < K) {
        const int d = __ldg(dr + j);
        x = (d >= 0 && (uint32_t)d < V) ? d : 0;
        sm.ld[j] = bf16_bits_to_float(__ldg((const uint16_t*)drow(j) + x));
      }
      sm.lt[j] = bf16_bits_to_float(__ldg((const uint16_t*)trow(j) + x));
    }
  }
  if (threadIdx.x == 0) sm.tau = 0u;
  __syncthreads();

  if (greedy) {
    // ---- temperature 0: accept while the draft is the row's argmax (lowest index on ties).
    // Rows go two at a time (j, j+1): one pass and one cluster exchange per pair, at the cost
    // of reading row j+1 for nothing when draft j is rejected.
    bool done = false;
    for (int j0 = 0; j0 <= K && !done; j0 += 2) {
      uint64_t pks[2];
      if (j0 + 1 <= K) {
        argmax_chunk2<DT>(trow(j0), trow(j0 + 1), V, vec, u0, u1, sm, pks[0], pks[1]);
        cluster_max2_u64(pks[0], pks[1], sm, phase, cl);
      } else {
        pks[0] = cluster_max_u64(argmax_chunk<DT>(trow(j0), V, vec, u0, u1, sm), sm, phase, cl);
        pks[1] = 0ull;
      }
      for (int t = 0; t < 2 && !done; ++t) {
        const int j = j0 + t;
        const uint64_t pk = pks[t];
        const uint32_t am = pk ? packed_index(pk) : 0u;  // no value above -inf: entry 0
        if (j == K) {
          b = am;
          done = true;
          break;
        }
        const int d = __ldg(dr + j);
        const bool valid = d >= 0 && (uint32_t)d < V;
        if (threadIdx.x == 0) {
          if (valid) {
            if (DT == SD_F32_PROBS) {
              sm.P[j] = __ldg((const float*)trow(j) + d);
              sm.Q[j] = __ldg((const float*)drow(j) + d);
            } else {
              sm.P[j] = bf16_bits_to_float(__ldg((const uint16_t*)trow(j) + d));
              sm.Q[j] = bf16_bits_to_float(__ldg((const uint16_t*)drow(j) + d));
            }
          } else {
            sm.P[j] = 0.0f;
            sm.Q[j] = 0.0f;
          }
        }
        if (!valid) e |= SD_ERR_TOKEN_RANGE;
        if (!valid || (uint32_t)d != am) {
          a = j;
          b = am;
          done = true;
        }
      }
    }
  } else if (DT == SD_F32_PROBS) {
    // ---- sampled, probability rows (small vocabularies): scalar accept scan, then the CTA's
    // share of the one race row, merged through the request's slot
    if (threadIdx.x < 32) {
      int bad;
      const int av = accept_scan_warp(P, r, sm.P, sm.Q, &bad);
      if (lane == 0) {
        sm.a = av;
        sm.e = bad;
      }
    }
    __syncthreads();
    a = sm.a;
    e = sm.e;
    const int jr = a < K ? a : K;
    uint64_t pk;
    if (a < K) {
      F32Residual<true> src{(const float*)trow(jr), (const float*)drow(jr), V, vec};
      pk = race_chunk(src, u0, u1, P.rk, P.rbase + (uint32_t)r, (uint32_t)jr, sm);
    } else {
      F32Residual<false> src{(const float*)trow(jr), nullptr, V, vec};
      pk = race_chunk(src, u0, u1, P.rk, P.rbase + (uint32_t)r, (uint32_t)jr, sm);
    }
    uint64_t row_max;
    // fused launch: the final token's inputs, read now so that they arrive during the merge
    int32_t tok_pre = 0;
    unsigned off_pre = 0u;
    if (P.fuse) {
      if (threadIdx.x < (unsigned)K) tok_pre = __ldg(dr + threadIdx.x);
      if (threadIdx.x == 0) off_pre = *(volatile unsigned*)&P.slots[r].off1;
    }
    if (merge_slot(P.slots + r, pk, u1 - u0, NU, sm, row_max)) {
      if (P.fuse) fused_finish(P, r, a, e, row_max, sm.P, sm.Q, tok_pre, off_pre, sm);
      else finish_sampled(P, r, a, e, row_max, sm.P, sm.Q, sm);
    }
    writer = false;  // finish_sampled wrote the outputs (in the CTA that completed the row)
  } else {
    // ---- sampled, bf16 logit rows: per row the sums S_t, S_d against the draft token's
    // logits, decide, race on the rejected row (or on p_K when every draft is accepted). The
    // cluster exchange of row j's sums overlaps the first units of row j+1.
    const float c = 1.4426950408889634f / T;
    const uint16_t* t16 = (const uint16_t*)tbase;
    const uint16_t* d16 = (const uint16_t*)dbase;
    auto tr = [&](int j) { return t16 + (size_t)j * P.ld_t; };
    auto dq = [&](int j) { return d16 + (size_t)j * P.ld_d; };
    // a row's references: the draft token's logits (element 0 when it is out of range; element
    // 0 of row K for the bonus row)
    auto nrc_of = [&](float ref) { return -__fmul_rn(ref, c); };
    auto ref_t = [&](int j) { return sm.lt[j]; };
    auto ref_d = [&](int j) { return sm.ld[j]; };
    const uint32_t us = u0 + (u1 - u0) / kLookAhead;
    int par = 0;
    // one row's units [lo, hi): target and draft rows j < K, the target row alone for j == K
    auto stream = [&](int j, uint32_t lo, uint32_t hi, RefAcc& at, RefAcc& ad) {
      if (j < K)
        ref_sums<true>(tr(j), dq(j), V, vec, lo, hi, c, nrc_of(ref_t(j)), nrc_of(ref_d(j)), at, ad);
      else
        ref_sums<false>(tr(j), nullptr, V, vec, lo, hi, c, nrc_of(ref_t(j)), 0.0f, at, ad);
    };
    RefAcc at, ad;
    stream(0, u0, u1, at, ad);
    float2 mine = block_sum2(at.total(), ad.total(), sm, par);
    cluster_post(mine, &sm.xslot[0], cl);
    for (int j = 0;; ++j) {
      // look-ahead: the first units of row j+1 while the cluster's sums of row j arrive
      RefAcc nt, nd;
      if (j + 1 <= K) stream(j + 1, u0, us, nt, nd);
      float2 S = cluster_collect(mine, &sm.xslot[j & 1], cl);
      float nrct = nrc_of(ref_t(j)), nrcd = j < K ? nrc_of(ref_d(j)) : 0.0f;
      if (!(S.x < kRefSumLimit) || (j < K && !(S.y < kRefSumLimit))) {
        // a term may have overflowed: sum the row again against its maximum (cluster-uniform)
        S = logit_row_refit(tr(j), j < K ? dq(j) : nullptr, V, vec, u0, u1, c, sm, phase, par,
                            cl, nrct, nrcd);
      }
      bool accept = false;
      if (j < K) {
        const int d = __ldg(dr + j);
        const bool valid = d >= 0 && (uint32_t)d < V;
        float Pv = 0.0f, Qv = 0.0f;
        if (valid) {
          Pv = __fdiv_rn(logit_term(ref_t(j), c, nrct), S.x);
          Qv = __fdiv_rn(logit_term(ref_d(j), c, nrcd), S.y);
          // the exact double test in one lane per warp (GB300's FP64 rate is low), shared
          int acc = 0;
          if ((threadIdx.x & 31) == 0) {
            const double u = accept_uniform(P.rk, P.rbase + (uint32_t)r, (uint32_t)j);
            acc = u * (double)Qv < (double)Pv;
          }
          accept = __shfl_sync(0xffffffffu, acc, 0) != 0;
        } else {
          e |= SD_ERR_TOKEN_RANGE;
        }
        if (threadIdx.x == 0) {
          sm.P[j] = Pv;
          sm.Q[j] = Qv;
        }
      }
      if (!accept) {
        // the race on row j: the residual of the rejected pair, or p_K for the bonus token
        a = j;
        const float invSt = 1.0f / S.x;
        uint64_t pk;
        const uint32_t rid = P.rbase + (uint32_t)r;
        if (j < K)
          pk = logit_race<true>(tr(j), dq(j), nrct, invSt, nrcd, 1.0f / S.y, c, V, vec, u0, u1,
                                P.rk, rid, (uint32_t)j, sm, phase, cl);
        else
          pk = 0ull;
        if (packed_key_bits(pk) == 0u)  // the bonus race, or no positive residual: p itself
          pk = logit_race<false>(tr(j), nullptr, nrct, invSt, 0.0f, 0.0f, c, V, vec, u0, u1, P.rk,
                                 rid, (uint32_t)j, sm, phase, cl);
        if (packed_key_bits(pk) == 0u) {
          e |= SD_ERR_ZERO_ROW;
          b = 0;
        } else {
          b = packed_index(pk);
        }
        break;
      }
      // accepted: the rest of row j+1, then its sums go to the cluster
      stream(j + 1, us, u1, nt, nd);
      mine = block_sum2(nt.total(), nd.total(), sm, par);
      cluster_post(mine, &sm.xslot[(j + 1) & 1], cl);
    }
  }

  // Let a programmatically dependent launch (the draft-batch rebuild) get scheduled; it waits
  // for this grid's completion before it reads any result.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __syncthreads();
  if (writer) {
    const int t = threadIdx.x;
    if (t <= KM) {
      int32_t tok = -1;
      if (t < a) tok = __ldg(dr + t);
      else if (t == a) tok = (int32_t)b;
      P.out_tokens[(size_t)r * (KM + 1) + t] = tok;
    }
    if (t < KM) {
      if (P.p_at) P.p_at[(size_t)r * KM + t] = sm.P[t];
      if (P.q_at) P.q_at[(size_t)r * KM + t] = sm.Q[t];
    }
    if (t == 0) {
      P.num_accepted[r] = a;
      raise_err(P.err, e);
    }
  }
  // greedy and logit requests exchanged data through distributed shared memory: peers may still
  // read this CTA's shared memory until all have passed this barrier
  if (cl > 1 && !sampled_probs) cluster_barrier();
}

// Sampled probability requests with large vocabularies: the race role over a whole number of
// CTAs per SM (see race_role).
__global__ void __launch_bounds__(NT, kRaceMinBlocks)
    race_kernel(const __grid_constant__ VerifyParams P) {
  __shared__ Smem sm;
  __shared__ AcceptState as;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  race_role(P, blockIdx.x, sm, as);
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------- drafter-side sampling
// Row (r*K + k) of `rows` is the drafter's output for draft k of request r: probabilities, or
// logits turned into probabilities by the request's temperature. The new draft is the
// exponential race argmax_x q(x)/E_x on the tag-2 Philox stream (block (x >> 2, k, r, 2)), or the
// argmax at temperature 0 -- the verify kernel's bonus race and greedy scan on a row of their
// own. One cluster of cl CTAs per row, each CTA a contiguous share of the row; logit rows take
// the softmax statistics first (exchanged over the cluster), then the race.
struct SampleParams {
  int B, K, V;
  const void* rows;
  long ld;
  const float* temperature;
  PhiloxRoundKeys rk;
  uint32_t rbase;
  int32_t* drafts;
  int32_t* err;
  int cl;
  int vec;
};

template <int DT>
// 5 CTAs per SM (48 registers): fp32 rows 1.4 to 6% faster than at 4 despite a few spills,
// logit rows (one unit in flight, no spills) 6.5% faster
__global__ void __launch_bounds__(NT, kMinBlocksF32)
    sample_kernel(const __grid_constant__ SampleParams P) {
  __shared__ Smem sm;
  constexpr int EPU = (DT == SD_F32_PROBS) ? 4 : 8;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int cl = P.cl;
  const uint32_t crank = blockIdx.x % (unsigned)cl;
  const int row = (int)(blockIdx.x / (unsigned)cl);
  const int r = row / P.K, k = row - r * P.K;
  const uint32_t V = (uint32_t)P.V;
  const bool vec = P.vec != 0;
  const uint32_t NU = (V + EPU - 1) / EPU;
  const uint32_t u0 = (uint32_t)(((uint64_t)NU * crank) / (unsigned)cl);
  const uint32_t u1 = (uint32_t)(((uint64_t)NU * (crank + 1)) / (unsigned)cl);
  const float T = P.temperature ? P.temperature[r] : 1.0f;
  const uint32_t rid = P.rbase + (uint32_t)r;
  int phase = 0;
  int32_t e = 0;
  if (threadIdx.x == 0) sm.tau = 0u;
  __syncthreads();
  uint64_t pk;
  if (T == 0.0f) {
    const void* rp = DT == SD_F32_PROBS
                         ? (const void*)((const float*)P.rows + (size_t)row * P.ld)
                         : (const void*)((const uint16_t*)P.rows + (size_t)row * P.ld);
    pk = cluster_max_u64(argmax_chunk<DT>(rp, V, vec, u0, u1, sm), sm, phase, cl);
  } else if (DT == SD_F32_PROBS) {
    F32Residual<false> src{(const float*)P.rows + (size_t)row * P.ld, nullptr, V, vec};
    pk = cluster_max_u64(race_chunk(src, u0, u1, P.rk, rid, (uint32_t)k, sm, kTagDraft), sm,
                         phase, cl);
  } else {
    // one pass: the log-domain race needs no softmax statistics
    const uint16_t* rp = (const uint16_t*)P.rows + (size_t)row * P.ld;
    const float c = 1.4426950408889634f / T;
    pk = cluster_max_u64(race_chunk_log(rp, V, vec, c, u0, u1, P.rk, rid, (uint32_t)k, kTagDraft,
                                        sm),
                         sm, phase, cl);
  }
  uint32_t b = 0;
  if (T == 0.0f) {
    b = pk ? packed_index(pk) : 0u;
  } else if (packed_key_bits(pk) == 0u) {
    e |= SD_ERR_ZERO_ROW;
  } else {
    b = packed_index(pk);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (crank == 0 && threadIdx.x == 0) {
    P.drafts[row] = (int32_t)b;
    raise_err(P.err, e);
  }
  if (cl > 1) cluster_barrier();  // peers may read this CTA's shared memory until here
}

}  // namespace sdk

// ------------------------------------------------------------------------------------ launcher
namespace {

}  // namespace

extern "C" size_t sd_verify_workspace_launch(int B) { return (size_t)B * sizeof(sdk::RaceSlot); }

namespace {

int sm_count() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cached[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 152;
  int n = cached[dev].load();
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 152;
    cached[dev].store(n);
  }
  return n;
}

// CTAs of the fp32 verify kernel that the device holds at once (occupancy query × SMs): the fused
// launch needs every one of its CTAs resident together.
int resident_f32() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cached[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  int n = cached[dev].load();
  if (n == 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, sdk::verify_kernel<SD_F32_PROBS>, sdk::NT, 0) != cudaSuccess)
      per_sm = 0;
    n = per_sm > 0 ? per_sm * sm_count() : -1;
    cached[dev].store(n);
  }
  return n > 0 ? n : 0;
}

int choose_cluster(int V, int epu) {
  const long units = ((long)V + epu - 1) / epu;
  int cl = sdk::CL_MAX;
  while (cl > 1 && units / cl < (long)sdk::NT * 2) cl >>= 1;
  return cl;
}

}  // namespace

// CTAs of the race kernel for an all-sampled batch (temperature NULL) on probability rows of at
// least 8192 entries whose cluster grid would span two waves or more (a whole number of CTAs per
// SM), or 0 for the cluster kernel.
static int race_grid(int B, int V, int dtype, bool has_temperature, int nc) {
  if (dtype != SD_F32_PROBS || (V + 3) / 4 < 2048 || has_temperature) return 0;
  const int sms = sm_count();
  if ((long)B * nc < 2L * sdk::kMinBlocksF32 * sms) return 0;  // measured faster per request
  long g = (long)sdk::kRaceMinBlocks * sms;
  // a CTA's share spans at most B/g + 2 requests: g >= B/6 keeps that within kMaxSeg
  if (g < (B + 5) / 6) g = (B + 5) / 6;
  return (int)g;
}

extern "C" int sd_verify_kernel_count(int B, int V, int dtype, int has_temperature) {
  (void)V;
  (void)dtype;
  (void)has_temperature;
  return B == 0 ? 0 : 1;  // the cluster kernel or the race kernel
}

// Launch shape of a verify call: cluster size cl, CTAs per request nc, race-kernel CTAs (0: the
// cluster kernel takes the batch), and whether a rebuild can join the launch (fusable).
struct VerifyShape {
  int cl, nc, race_blocks;
  bool fusable;
};
static VerifyShape verify_shape(int B, int V, int dtype, bool has_temperature) {
  VerifyShape v;
  const int epu = dtype == SD_F32_PROBS ? 4 : 8;
  v.cl = choose_cluster(V, epu);
  // Logit rows: the request's CTAs exchange every row's sums, so fewer CTAs per request spend
  // less of their time in exchanges and reductions; clusters of 4 once those still fill a wave
  // (V = 201088: 4-17% faster from B = 192 to 1024, while at B = 96 clusters of 8 are 12% faster).
  if (dtype == SD_BF16_LOGITS && v.cl > 4 && (long)B * 4 >= (long)sdk::kMinBlocks * sm_count())
    v.cl = 4;
  v.nc = v.cl;  // CTAs per request in the cluster role
  v.race_blocks = race_grid(B, V, dtype, has_temperature, v.nc);
  if (v.race_blocks == 0 && dtype == SD_F32_PROBS && !has_temperature) {
    // every request samples: its CTAs exchange nothing through shared memory, so no cluster is
    // needed, and each row splits over as many CTAs as fill one wave of kMinBlocksF32 per SM
    const int nu = (V + 3) / 4;
    int nc = sdk::kMinBlocksF32 * sm_count() / std::max(B, 1);
    nc = std::min(nc, std::max(1, nu / (2 * sdk::NT)));
    v.cl = 1;
    v.nc = std::max(nc, 1);
  }
  // The fused launch: one wave of kMinBlocksF32 CTAs per SM, B of them rebuilding the drafter
  // batch and at least as many racing (the race CTAs wait for the rebuild CTAs' published slots
  // only at their very end, and every CTA of the wave is resident from the start).
  v.fusable = v.race_blocks == 0 && v.cl == 1 && dtype == SD_F32_PROBS && !has_temperature &&
              B <= sdk::kMaxFuseB && 2L * B <= (long)resident_f32();
  return v;
}

// The verify launch; with rb, the drafter-batch rebuild joins it when the batch takes the
// one-wave all-sampled path (*fused = true), else the caller launches the rebuild kernel.
static int verify_launch_impl(int B, int K, int V, int dtype, const void* target, long ld_t,
                              const void* draft, long ld_d, const int32_t* drafts,
                              const int32_t* cu_drafts, const float* temperature, uint64_t seed,
                              uint32_t request_base, int32_t* out_tokens, int32_t* num_accepted,
                              float* p_at_draft, float* q_at_draft, void* workspace,
                              int32_t* err, cudaStream_t stream, const sdk::RebuildArgs* rb,
                              bool* fused, uint64_t wait_ns = sdk::kWaitNs, int withhold = -1) {
  const int esize = dtype == SD_F32_PROBS ? 4 : 2;
  sdk::VerifyParams P;
  memset(&P, 0, sizeof(P));
  P.B = B;
  P.K = K;
  P.V = V;
  P.target = target;
  P.ld_t = ld_t;
  P.draft = draft;
  P.ld_d = ld_d;
  P.drafts = drafts;
  P.temperature = temperature;
  P.cu = cu_drafts;
  P.rk = sdk::philox_round_keys(seed);
  P.rbase = request_base;
  P.out_tokens = out_tokens;
  P.num_accepted = num_accepted;
  P.p_at = p_at_draft;
  P.q_at = q_at_draft;
  P.slots = (sdk::RaceSlot*)workspace;
  P.err = err;
  const VerifyShape shape = verify_shape(B, V, dtype, temperature != nullptr);
  P.cl = shape.cl;
  P.nc = shape.nc;
  P.race_blocks = shape.race_blocks;
  P.cluster_blocks = B * P.nc;  // (unused when the race kernel takes the batch)
  P.vec = ((uintptr_t)target % 16 == 0) && ((uintptr_t)draft % 16 == 0) &&
          ((ld_t * esize) % 16 == 0) && ((ld_d * esize) % 16 == 0);
  P.fuse = (rb != nullptr && shape.fusable) ? (rb->padded ? 2 : 1) : 0;
  P.wait_ns = wait_ns;
  P.withhold = withhold;
  if (P.fuse) {
    // B rebuild CTAs, then up to one wave's worth of race CTAs, no more per request than a row
    // splits into (every race CTA gets at least 2 NT units)
    P.rb = *rb;
    const long per = std::max(1, ((V + 3) / 4) / (2 * sdk::NT));
    const long race = std::min((long)resident_f32() - B, (long)B * per);
    P.cluster_blocks = (int)(B + race);
  }
  if (fused) *fused = P.fuse != 0;
  if (B == 0) return SD_OK;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)P.cluster_blocks, 1, 1);
  cfg.blockDim = dim3(sdk::NT, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)P.cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // scheduled while the preceding kernel drains; the kernel waits on the device (see above)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t rc = cudaSuccess;
  if (P.race_blocks == 0) {
    // one kernel: clusters per request (greedy and logit rows in order; sampled probability
    // rows split over the request's CTAs)
    if (dtype == SD_F32_PROBS) rc = cudaLaunchKernelEx(&cfg, sdk::verify_kernel<SD_F32_PROBS>, P);
    else rc = cudaLaunchKernelEx(&cfg, sdk::verify_kernel<SD_BF16_LOGITS>, P);
    return rc == cudaSuccess ? SD_OK : SD_E_LAUNCH;
  }
  {
    // every request sampled on probability rows: accept scans and the race, balanced over every
    // SM (a programmatic dependent of what precedes it)
    cudaLaunchConfig_t rcfg = {};
    rcfg.gridDim = dim3((unsigned)P.race_blocks, 1, 1);
    rcfg.blockDim = dim3(sdk::NT, 1, 1);
    rcfg.stream = stream;
    cudaLaunchAttribute rattr[1];
    rattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    rattr[0].val.programmaticStreamSerializationAllowed = 1;
    rcfg.attrs = rattr;
    rcfg.numAttrs = 1;
    rc = cudaLaunchKernelEx(&rcfg, sdk::race_kernel, P);
  }
  return rc == cudaSuccess ? SD_OK : SD_E_LAUNCH;
}

extern "C" int sd_verify_launch(int B, int K, int V, int dtype, const void* target, long ld_t,
                                const void* draft, long ld_d, const int32_t* drafts,
                                const int32_t* cu_drafts, const float* temperature,
                                uint64_t seed, uint32_t request_base, int32_t* out_tokens,
                                int32_t* num_accepted, float* p_at_draft, float* q_at_draft,
                                void* workspace, int32_t* err, cudaStream_t stream) {
  return verify_launch_impl(B, K, V, dtype, target, ld_t, draft, ld_d, drafts, cu_drafts,
                            temperature, seed, request_base, out_tokens, num_accepted,
                            p_at_draft, q_at_draft, workspace, err, stream, nullptr, nullptr);
}

extern "C" int sd_prep_launch(int B, int K, const int32_t* out_tokens, const int32_t* num_accepted,
                              const int32_t* cu_drafts, const int32_t* pos0,
                              const int32_t* block_table, int max_blocks, int block_size,
                              int32_t mask_token_id, int capacity, int32_t* input_ids,
                              int32_t* positions, int32_t* slot_mapping, int32_t* hidden_map,
                              uint8_t* is_masked, uint8_t* is_rejected, int32_t* start_loc,
                              int32_t* new_token_idx, int32_t* total_out, int H,
                              const void* target_hidden, long ld_in, int n_in_rows,
                              const void* h_shared, void* out_hidden, long ld_out, int32_t* err,
                              cudaStream_t stream);

// Verify and rebuild in one call: one launch when the batch takes the one-wave all-sampled path,
// else the verify kernel and then the rebuild kernel (the same outputs either way). The
// workspace holds the B merge slots (each also carries its request's first drafter slot from the
// rebuild CTA to the CTA that writes the final token).
static int verify_prepare_impl(
    int B, int K, int V, int dtype, const void* target, long ld_t, const void* draft, long ld_d,
    const int32_t* drafts, const int32_t* cu_drafts, const float* temperature, uint64_t seed,
    uint32_t request_base,
    int32_t* out_tokens, int32_t* num_accepted, float* p_at_draft, float* q_at_draft,
    const int32_t* pos0, const int32_t* block_table, int max_blocks, int block_size,
    int32_t mask_token_id, int capacity, int32_t* input_ids, int32_t* positions,
    int32_t* slot_mapping, int32_t* hidden_map, uint8_t* is_masked, uint8_t* is_rejected,
    int32_t* start_loc, int32_t* new_token_idx, int32_t* total_out, int H,
    const void* target_hidden, long ld_in, int n_in_rows, const void* h_shared, void* out_hidden,
    long ld_out, void* workspace, int32_t* err, cudaStream_t stream, uint64_t wait_ns,
    int withhold) {
  sdk::RebuildArgs rb = {};
  rb.pos0 = pos0;
  rb.block_table = block_table;
  rb.max_blocks = max_blocks;
  rb.block_size = block_size;
  rb.mask_id = mask_token_id;
  rb.capacity = capacity;
  rb.input_ids = input_ids;
  rb.positions = positions;
  rb.slot_mapping = slot_mapping;
  rb.hidden_map = hidden_map;
  rb.is_masked = is_masked;
  rb.is_rejected = is_rejected;
  rb.start_loc = start_loc;
  rb.new_token_idx = new_token_idx;
  rb.total_out = total_out;
  rb.H = H;
  rb.hidden = (const uint16_t*)target_hidden;
  rb.ld_in = ld_in;
  rb.n_in_rows = n_in_rows;
  rb.h_shared = (const uint16_t*)h_shared;
  rb.out_hidden = (uint16_t*)out_hidden;
  rb.ld_out = ld_out;
  rb.hvec = out_hidden && (H % 8 == 0) && ((uintptr_t)target_hidden % 16 == 0) &&
            ((uintptr_t)h_shared % 16 == 0) && ((uintptr_t)out_hidden % 16 == 0) &&
            (ld_in % 8 == 0) && (ld_out % 8 == 0);
  bool fused = false;
  int rc = verify_launch_impl(B, K, V, dtype, target, ld_t, draft, ld_d, drafts, cu_drafts,
                              temperature, seed, request_base, out_tokens, num_accepted,
                              p_at_draft, q_at_draft, workspace, err, stream, &rb, &fused,
                              wait_ns, withhold);
  if (rc != SD_OK || fused) return rc;
  return sd_prep_launch(B, K, out_tokens, num_accepted, cu_drafts, pos0, block_table, max_blocks,
                        block_size, mask_token_id, capacity, input_ids, positions, slot_mapping,
                        hidden_map, is_masked, is_rejected, start_loc, new_token_idx, total_out,
                        H, target_hidden, ld_in, n_in_rows, h_shared, out_hidden, ld_out, err,
                        stream);
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
                                     int32_t* err, cudaStream_t stream);

// Verify and the padded drafter-batch rebuild in one call: one launch when the batch takes the
// one-wave all-sampled path (each rebuild CTA recomputes its own request's decisions; the race
// writes the final token at its fixed row), else the verify kernel and then the padded rebuild
// kernel (the same outputs either way).
extern "C" int sd_verify_prepare_padded_launch(
    int B, int K, int V, int dtype, const void* target, long ld_t, const void* draft, long ld_d,
    const int32_t* drafts, const float* temperature, uint64_t seed, uint32_t request_base,
    int32_t* out_tokens, int32_t* num_accepted, float* p_at_draft, float* q_at_draft,
    const int32_t* pos0, const int32_t* block_table, int max_blocks, int block_size,
    int32_t mask_token_id, int32_t* input_ids, int32_t* positions, int32_t* slot_mapping,
    int32_t* hidden_map, uint8_t* is_masked, uint8_t* rejected, int32_t* scatter_map,
    int32_t* new_token_idx, int H, const void* target_hidden, long ld_in, int n_in_rows,
    const void* h_shared, void* out_hidden, long ld_out, void* workspace, int32_t* err,
    cudaStream_t stream) {
  sdk::RebuildArgs rb = {};
  rb.padded = 1;
  rb.pos0 = pos0;
  rb.block_table = block_table;
  rb.max_blocks = max_blocks;
  rb.block_size = block_size;
  rb.mask_id = mask_token_id;
  rb.input_ids = input_ids;
  rb.positions = positions;
  rb.slot_mapping = slot_mapping;
  rb.hidden_map = hidden_map;
  rb.is_masked = is_masked;
  rb.rejected = rejected;
  rb.scatter_map = scatter_map;
  rb.new_token_idx = new_token_idx;
  rb.H = H;
  rb.hidden = (const uint16_t*)target_hidden;
  rb.ld_in = ld_in;
  rb.n_in_rows = n_in_rows;
  rb.h_shared = (const uint16_t*)h_shared;
  rb.out_hidden = (uint16_t*)out_hidden;
  rb.ld_out = ld_out;
  rb.hvec = out_hidden && (H % 8 == 0) && ((uintptr_t)target_hidden % 16 == 0) &&
            ((uintptr_t)h_shared % 16 == 0) && ((uintptr_t)out_hidden % 16 == 0) &&
            (ld_in % 8 == 0) && (ld_out % 8 == 0);
  bool fused = false;
  int rc = verify_launch_impl(B, K, V, dtype, target, ld_t, draft, ld_d, drafts, nullptr,
                              temperature, seed, request_base, out_tokens, num_accepted,
                              p_at_draft, q_at_draft, workspace, err, stream, &rb, &fused);
  if (rc != SD_OK || fused) return rc;
  return sd_prep_padded_launch(B, K, out_tokens, num_accepted, pos0, block_table, max_blocks,
                               block_size, mask_token_id, input_ids, positions, slot_mapping,
                               hidden_map, is_masked, rejected, scatter_map, new_token_idx, H,
                               target_hidden, ld_in, n_in_rows, h_shared, out_hidden, ld_out, err,
                               stream);
}

#define SD_VERIFY_PREPARE_PARAMS                                                                \
  int B, int K, int V, int dtype, const void *target, long ld_t, const void *draft, long ld_d, \
      const int32_t *drafts, const int32_t *cu_drafts, const float *temperature,               \
      uint64_t seed, uint32_t request_base, int32_t *out_tokens, int32_t *num_accepted,        \
      float *p_at_draft, float *q_at_draft, const int32_t *pos0, const int32_t *block_table,   \
      int max_blocks, int block_size, int32_t mask_token_id, int capacity, int32_t *input_ids, \
      int32_t *positions, int32_t *slot_mapping, int32_t *hidden_map, uint8_t *is_masked,      \
      uint8_t *is_rejected, int32_t *start_loc, int32_t *new_token_idx, int32_t *total_out,    \
      int H, const void *target_hidden, long ld_in, int n_in_rows, const void *h_shared,       \
      void *out_hidden, long ld_out, void *workspace, int32_t *err, cudaStream_t stream
#define SD_VERIFY_PREPARE_ARGS                                                                 \
  B, K, V, dtype, target, ld_t, draft, ld_d, drafts, cu_drafts, temperature, seed,             \
      request_base, out_tokens, num_accepted, p_at_draft, q_at_draft, pos0, block_table,       \
      max_blocks, block_size, mask_token_id, capacity, input_ids, positions, slot_mapping,     \
      hidden_map, is_masked, is_rejected, start_loc, new_token_idx, total_out, H,              \
      target_hidden, ld_in, n_in_rows, h_shared, out_hidden, ld_out, workspace, err, stream

extern "C" int sd_verify_prepare_launch(SD_VERIFY_PREPARE_PARAMS) {
  return verify_prepare_impl(SD_VERIFY_PREPARE_ARGS, sdk::kWaitNs, -1);
}

// Diagnostic form: in the fused launch, request `withhold`'s rebuild CTA publishes its first
// drafter slot only after the completing race CTA has waited wait_us microseconds and given up
// (SD_ERR_WAIT), so that a test can run the wait out without a fault.
extern "C" int sd_verify_prepare_withheld_launch(int withhold, uint32_t wait_us,
                                                 SD_VERIFY_PREPARE_PARAMS) {
  return verify_prepare_impl(SD_VERIFY_PREPARE_ARGS, (uint64_t)wait_us * 1000ull, withhold);
}

// Kernels one sd_verify_prepare call launches.
extern "C" int sd_verify_prepare_kernel_count(int B, int K, int V, int dtype,
                                              int has_temperature) {
  (void)K;
  if (B == 0) return 0;
  return verify_shape(B, V, dtype, has_temperature != 0).fusable ? 1 : 2;
}

// ------------------------------------------------------------------ no-allocation entry point
// Scratch for sd_verify_noalloc: the same per-request merge slots sd_verify keeps in the caller's
// workspace, here in a fixed array that every GPU loading the library holds until exit
// (SD_VERIFY_NOALLOC_MAX_B * 16 bytes). Host code may not pass the array's name to a kernel (on
// the host it is only a stand-in for the device symbol); its device address is looked up once
// per device, with that device current.
static __device__ __align__(256) sdk::RaceSlot g_noalloc_slots[SD_VERIFY_NOALLOC_MAX_B];

namespace {
constexpr int kNoallocMaxDevices = 64;
std::atomic<void*> g_noalloc_addr[kNoallocMaxDevices];
}  // namespace

extern "C" int sd_verify_noalloc_launch(int B, int K, int V, int dtype, const void* target,
                                        long ld_t, const void* draft, long ld_d,
                                        const int32_t* drafts, const float* temperature,
                                        uint64_t seed, uint32_t request_base,
                                        int32_t* out_tokens, int32_t* num_accepted,
                                        float* p_at_draft, float* q_at_draft, int32_t* err,
                                        cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoallocMaxDevices)
    return SD_E_DEVICE;
  void* slots = g_noalloc_addr[dev].load();
  if (!slots) {
    if (cudaGetSymbolAddress(&slots, g_noalloc_slots) != cudaSuccess || !slots)
      return SD_E_LAUNCH;
    g_noalloc_addr[dev].store(slots);
  }
  // The slots must start at zero; every call leaves them zeroed, but clear them anyway so that
  // no earlier call's state can leak into this one.
  if (cudaMemsetAsync(slots, 0, (size_t)B * sizeof(sdk::RaceSlot), stream) != cudaSuccess)
    return SD_E_LAUNCH;
  return sd_verify_launch(B, K, V, dtype, target, ld_t, draft, ld_d, drafts, nullptr,
                          temperature, seed, request_base, out_tokens, num_accepted, p_at_draft,
                          q_at_draft, slots, err, stream);
}

// Drafter-side sampling: one cluster per row.
extern "C" int sd_sample_launch(int B, int K, int V, int dtype, const void* rows, long ld,
                                const float* temperature, uint64_t seed, uint32_t request_base,
                                int32_t* drafts, int32_t* err, cudaStream_t stream) {
  if (B == 0) return SD_OK;
  const int esize = dtype == SD_F32_PROBS ? 4 : 2;
  const int epu = dtype == SD_F32_PROBS ? 4 : 8;
  sdk::SampleParams P;
  P.B = B;
  P.K = K;
  P.V = V;
  P.rows = rows;
  P.ld = ld;
  P.temperature = temperature;
  P.rk = sdk::philox_round_keys(seed);
  P.rbase = request_base;
  P.drafts = drafts;
  P.err = err;
  // CTAs per row: as few as still give the launch about 1.5 waves of kMinBlocksF32 CTAs per SM
  // (a row's CTAs meet at a cluster barrier and share the candidate pass; more rows per wave
  // amortise both), no more than the row splits into
  P.cl = choose_cluster(V, epu);
  const long rows_n = (long)B * K, want = 3L * sdk::kMinBlocksF32 * sm_count() / 2;
  while (P.cl > 1 && rows_n * (P.cl / 2) >= want) P.cl >>= 1;
  P.vec = ((uintptr_t)rows % 16 == 0) && ((ld * esize) % 16 == 0);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * K * P.cl), 1, 1);
  cfg.blockDim = dim3(sdk::NT, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)P.cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t rc;
  if (dtype == SD_F32_PROBS) rc = cudaLaunchKernelEx(&cfg, sdk::sample_kernel<SD_F32_PROBS>, P);
  else rc = cudaLaunchKernelEx(&cfg, sdk::sample_kernel<SD_BF16_LOGITS>, P);
  return rc == cudaSuccess ? SD_OK : SD_E_LAUNCH;
}
