// sd_oracle.cpp -- plain, slow CPU oracle for the speculative-decoding verify step and the
// P-EAGLE draft-batch rebuild.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product path may call this code: only the tests,
// the smoke check and the CPU-baseline leg of the benchmark load it. It shares no source,
// header, table or constant with the CUDA library; the two meet only at the seeded synthetic
// inputs.
//
// Sources (page title, then section):
//  [SD]  "Speculative decoding explainer" (ainews.alishangtian.com), sections
//        "修正拒绝采样" (modified rejection sampling: accept with min(1, p/q), resample from
//        the normalised residual max(0, p - q)), "核心思想" (the K-draft verify loop, discard
//        after the first rejection, K+1 tokens when every draft is accepted) and "边界与代价"
//        (greedy decoding must reproduce the target's argmax token for token).
//  [PE]  "P-EAGLE: parallel speculative decoding in vLLM" (vLLM blog), sections "核心方法"
//        (input shift by one: drafter slot i takes the token and hidden state of position
//        i-1; MASK slots take emb(mask) and h_shared), "并行草稿生成的挑战" (rebuild of ids,
//        positions, slot mapping and per-request start indices), "Triton Kernel" (the
//        metadata one pass emits) and "Hidden State 管理" (hidden-state copy, h_shared
//        fill, PADDING_SLOT_ID = -1).
//  [PX]  Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11):
//        the Philox4x32-10 bijection.
//
// Readings where the pages are silent (each is listed in the design notes):
//  R1 counter layout of the Philox stream: accept uniform = word 0 of block (0, j, r, 0);
//     race variate for vocab entry x on row j = word (x & 3) of block (x >> 2, j, r, 1);
//     key = (seed & 0xffffffff, seed >> 32).
//  R2 u = (w >> 8) * 2^-24; v = (w + 0.5) * 2^-32; E = fp32 rounding of the double -log(v).
//  R3 the residual sample is argmax_x r(x)/E_x (exponential race), keys compared as fp32 for
//     probability inputs (double for logits inputs), ties to the lowest x.
//  R4 if the residual race has no positive key (r == 0 everywhere) the race is re-run on
//     p of the same row with the same E's; if that has none either the token is 0 and
//     SD_ORACLE_ERR_ZERO_ROW is raised.
//  R5 drafter slot j of request r takes target hidden row r*(K+1)+j for j <= a_r, MASK slots
//     take h_shared (map -1); positions are pos0 + 1 + j.
//  R6 is_rejected is over the verify batch [B, K+1]: 1 for draft slots j > a_r, 0 for slot 0.
//  R13 drafter-side sampling (the drafter's K outputs per request become the next step's drafts):
//     draft k of request r is the exponential race argmax_x q(x)/E_x over the drafter's row k,
//     with E from word (x & 3) of block (x >> 2, k, r, 2) (tag 2, a stream of its own), the
//     R2/R3 rules otherwise; temperature 0 takes argmax q, lowest index on ties.
//  R14 padded drafter batch ([PE] "Hidden State 管理": rejected tokens get PADDING_SLOT_ID; the
//     target hidden states are scattered to their drafter rows): request r owns the fixed row of
//     W = 2K slots [r*W, (r+1)*W). Slots j < a_r + K are those of the packed layout (R5);
//     slots j >= a_r + K are rejected leftovers: token mask_token_id, position pos0 + 1 + j,
//     KV slot -1, hidden map -1 (h_shared), is_masked 0, rejected 1. new_token_idx =
//     r*W + a_r + k; the scatter map sends target row r*(K+1)+j to drafter row r*W + j for
//     j <= a_r and is -1 for the rejected target rows.
//  R17 per-request draft counts in the rebuild (cu = exclusive prefix of K_r, as in the verify):
//     L_r = a_r + K_r slots (K_r - 1 MASK slots), target hidden row of slot j = cu[r] + r + j,
//     is_rejected[r][j] = 1 for 1 <= j <= K_r with j > a_r (0 past K_r), new_token_idx[r][k] =
//     start_r + a_r + k for k < K_r and -1 after; a_r outside [0, K_r] is clamped.
//
// Build: g++ -std=c++17 -O2 -ffp-contract=off -fno-fast-math (no FMA contraction, so every
// fp32 operation below is one IEEE-754 round-to-nearest operation on both x86-64 and aarch64).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// Error bits (the oracle's own copy of the documented values).
constexpr int32_t ERR_TOKEN_RANGE = 1;    // draft token outside [0, V)
constexpr int32_t ERR_BLOCK_TABLE = 2;    // position not covered by the block table
constexpr int32_t ERR_NUM_ACCEPTED = 4;   // num_accepted outside [0, K]
constexpr int32_t ERR_MAP_RANGE = 8;      // hidden map row outside the target hidden rows
constexpr int32_t ERR_ZERO_ROW = 16;      // race row without a positive key even on p
constexpr int32_t ERR_TOTAL_RANGE = 32;   // total_out outside [0, capacity]
constexpr int32_t ERR_DRAFT_COUNT = 128;  // a per-request draft count outside [0, K]

// ---------------------------------------------------------------- [PX] Philox4x32-10
// One round: two 32x32->64 products, the high halves xor-ed with the other two words and the
// round key, the low halves moved across. The Weyl key schedule adds the two constants
// after every round.
void philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    const uint64_t prod0 = (uint64_t)M0 * (uint64_t)x0;
    const uint64_t prod1 = (uint64_t)M1 * (uint64_t)x2;
    const uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    const uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    const uint32_t n0 = hi1 ^ x1 ^ k0;
    const uint32_t n1 = lo1;
    const uint32_t n2 = hi0 ^ x3 ^ k1;
    const uint32_t n3 = lo0;
    x0 = n0; x1 = n1; x2 = n2; x3 = n3;
    k0 += W0;
    k1 += W1;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

uint32_t philox_word(uint64_t seed, uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                     int word) {
  const uint32_t ctr[4] = {c0, c1, c2, c3};
  const uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
  uint32_t out[4];
  philox4x32_10(ctr, key, out);
  return out[word];
}

// R1/R2: the accept uniform of draft d_{j+1} of request r.
double accept_uniform(uint64_t seed, uint32_t r, uint32_t j) {
  const uint32_t w = philox_word(seed, 0u, j, r, 0u, 0);
  return (double)(w >> 8) * (1.0 / 16777216.0);
}

// R1/R2: the exponential variate E_x of vocab entry x on row j of request r (tag 1: the verify
// races; tag 2: drafter-side sampling, R13).
float race_E(uint64_t seed, uint32_t r, uint32_t j, uint32_t x, uint32_t tag = 1u) {
  const uint32_t w = philox_word(seed, x >> 2, j, r, tag, (int)(x & 3u));
  const double v = ((double)w + 0.5) * (1.0 / 4294967296.0);
  return (float)(-std::log(v));
}

// ---------------------------------------------------------------- fp32-input race [SD] + R3/R4
// Returns the winning x; `margin` receives (k1 - k2) / k1 over the two largest keys.
// `use_q` false races on max(p, 0) (bonus race, or the R4 fallback).
int race_f32(const float* p, const float* q, bool use_q, int V, uint64_t seed, uint32_t r,
             uint32_t j, double* margin) {
  int best_x = 0;
  float best_k = -1.0f, second_k = -1.0f;
  for (int x = 0; x < V; ++x) {
    const float diff = use_q ? (p[x] - q[x]) : p[x];
    const float res = std::fmax(diff, 0.0f);           // NaN -> 0, negatives -> 0
    const float E = race_E(seed, r, j, (uint32_t)x);
    const float key = res / E;                          // one IEEE fp32 division
    if (key > best_k) {
      second_k = best_k;
      best_k = key;
      best_x = x;
    } else if (key > second_k) {
      second_k = key;
    }
  }
  if (margin) {
    *margin = (best_k > 0.0f) ? ((double)best_k - (double)std::max(second_k, 0.0f)) / best_k
                              : 0.0;
  }
  return (best_k > 0.0f) ? best_x : -1;  // -1: no positive key
}

// Greedy: argmax with the lowest index on ties (plain strict-greater scan).
template <typename Get>
int argmax_row(Get get, int V, double* margin) {
  int best_x = 0;
  double best = get(0), second = -INFINITY;
  for (int x = 1; x < V; ++x) {
    const double v = get(x);
    if (v > best) {
      second = best;
      best = v;
      best_x = x;
    } else if (v > second) {
      second = v;
    }
  }
  if (margin) *margin = best - second;
  return best_x;
}

float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

template <typename F>
void parallel_for(int n, int nthreads, F fn) {
  if (nthreads <= 0) nthreads = (int)std::thread::hardware_concurrency();
  if (nthreads <= 1 || n <= 1) {
    for (int i = 0; i < n; ++i) fn(i);
    return;
  }
  nthreads = std::min(nthreads, n);
  std::vector<std::thread> pool;
  pool.reserve(nthreads);
  for (int t = 0; t < nthreads; ++t) {
    pool.emplace_back([=] {
      for (int i = t; i < n; i += nthreads) fn(i);
    });
  }
  for (auto& th : pool) th.join();
}

struct VerifyOut {
  int32_t* out_tokens;
  int32_t* num_accepted;
  float* p_at;
  float* q_at;
  double* acc_margin;   // [B, K] optional
  double* race_margin;  // [B] optional
};

}  // namespace

extern "C" {

int oracle_version() { return 1; }

void oracle_philox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
  philox4x32_10(ctr, key, out);
}

double oracle_accept_uniform(uint64_t seed, uint32_t r, uint32_t j) {
  return accept_uniform(seed, r, j);
}

float oracle_race_E(uint64_t seed, uint32_t r, uint32_t j, uint32_t x) {
  return race_E(seed, r, j, x);
}

float oracle_race_E_tag(uint64_t seed, uint32_t r, uint32_t j, uint32_t x, uint32_t tag) {
  return race_E(seed, r, j, x, tag);
}

// Exponential race on one row of fp32 values (exposed for the pin tests).
int oracle_race_row_f32(const float* p, const float* q, int use_q, int V, uint64_t seed,
                        uint32_t r, uint32_t j, double* margin) {
  return race_f32(p, q, use_q != 0, V, seed, r, j, margin);
}

// Verify on fp32 probability rows [SD].
//  target: row (i*(K+1)+j) at target + row*ld_t, j = 0..K;  draft: row (i*K+j), j = 0..K-1.
//  req_ids (nullable): the global request index of local request i, used in the Philox
//  counters, so that a sample of a batch reproduces the batch's own draws.
//  temperature (nullable = all 1): 0 selects greedy verification, anything else sampling.
//  p_at/q_at (nullable) [B, K]: p_j(d_{j+1}), q_j(d_{j+1}) for every examined draft
//  j <= min(a, K-1) (0 for an out-of-range token), -1 for the rest.
int oracle_verify_probs(int B, int K, int V, const float* target, long ld_t, const float* draft,
                        long ld_d, const int32_t* drafts, const float* temperature, uint64_t seed,
                        const int32_t* req_ids, int32_t* out_tokens, int32_t* num_accepted,
                        float* p_at, float* q_at, double* acc_margin, double* race_margin,
                        int32_t* err, int nthreads) {
  if (B < 0 || K < 0 || V < 1) return -1;  // K == 0: the bonus token from p_0 alone
  std::vector<int32_t> errs((size_t)std::max(B, 1), 0);
  parallel_for(B, nthreads, [&](int i) {
    const uint32_t rid = req_ids ? (uint32_t)req_ids[i] : (uint32_t)i;
    const bool greedy = temperature && temperature[i] == 0.0f;
    const float* trow0 = target + (long)i * (K + 1) * ld_t;
    const float* drow0 = draft + (long)i * K * ld_d;
    int a = K;
    int32_t e = 0;
    for (int j = 0; j < K; ++j) {
      if (p_at) p_at[(long)i * K + j] = -1.0f;
      if (q_at) q_at[(long)i * K + j] = -1.0f;
      if (acc_margin) acc_margin[(long)i * K + j] = -1.0;
    }
    for (int j = 0; j < K; ++j) {
      const int d = drafts[(long)i * K + j];
      const float* trow = trow0 + (long)j * ld_t;
      const float* drow = drow0 + (long)j * ld_d;
      if (d < 0 || d >= V) {
        e |= ERR_TOKEN_RANGE;
        if (p_at) p_at[(long)i * K + j] = 0.0f;
        if (q_at) q_at[(long)i * K + j] = 0.0f;
        a = j;
        break;
      }
      const float P = trow[d], Q = drow[d];
      if (p_at) p_at[(long)i * K + j] = P;
      if (q_at) q_at[(long)i * K + j] = Q;
      bool accept;
      if (greedy) {
        double m;
        const int am = argmax_row([&](int x) { return (double)trow[x]; }, V, &m);
        accept = (am == d);
        if (acc_margin) acc_margin[(long)i * K + j] = m;
      } else {
        const double u = accept_uniform(seed, rid, (uint32_t)j);
        const double uq = u * (double)Q;  // exact: 24-bit u times 24-bit Q
        accept = uq < (double)P;
        if (acc_margin) {
          const double mx = std::max((double)P, uq);
          acc_margin[(long)i * K + j] = mx > 0 ? std::fabs((double)P - uq) / mx : 0.0;
        }
      }
      if (!accept) {
        a = j;
        break;
      }
    }
    int b;
    double rm = 0.0;
    if (greedy) {
      const float* trow = trow0 + (long)a * ld_t;
      b = argmax_row([&](int x) { return (double)trow[x]; }, V, &rm);
    } else if (a < K) {
      const float* trow = trow0 + (long)a * ld_t;
      const float* drow = drow0 + (long)a * ld_d;
      b = race_f32(trow, drow, true, V, seed, rid, (uint32_t)a, &rm);
      if (b < 0) b = race_f32(trow, nullptr, false, V, seed, rid, (uint32_t)a, &rm);  // R4
    } else {
      const float* trow = trow0 + (long)K * ld_t;
      b = race_f32(trow, nullptr, false, V, seed, rid, (uint32_t)K, &rm);
    }
    if (b < 0) {
      e |= ERR_ZERO_ROW;
      b = 0;
    }
    for (int t = 0; t <= K; ++t) {
      int32_t tok = -1;
      if (t < a) tok = drafts[(long)i * K + t];
      else if (t == a) tok = b;
      out_tokens[(long)i * (K + 1) + t] = tok;
    }
    num_accepted[i] = a;
    if (race_margin) race_margin[i] = rm;
    errs[i] = e;
  });
  if (err) {
    int32_t e = 0;
    for (int i = 0; i < B; ++i) e |= errs[i];
    *err |= e;
  }
  return 0;
}

// Verify on bf16 logit rows with per-request temperature softmax, all in double.
//  p_j = softmax(l^t_j / T), q_j = softmax(l^d_j / T) (the same T for both, reading); T == 0
//  verifies greedily on the raw logits. Race keys are r/E in double with
//  r = max(0, p - q) in double. Rows after the first rejection are never read.
//  Greedy requests report the raw logits at the draft in p_at/q_at.
int oracle_verify_logits(int B, int K, int V, const uint16_t* target, long ld_t,
                         const uint16_t* draft, long ld_d, const int32_t* drafts,
                         const float* temperature, uint64_t seed, const int32_t* req_ids,
                         int32_t* out_tokens, int32_t* num_accepted, float* p_at, float* q_at,
                         double* acc_margin, double* race_margin, int32_t* err, int nthreads) {
  if (B < 0 || K < 0 || V < 1) return -1;  // K == 0: the bonus token from p_0 alone
  std::vector<int32_t> errs((size_t)std::max(B, 1), 0);
  parallel_for(B, nthreads, [&](int i) {
    const uint32_t rid = req_ids ? (uint32_t)req_ids[i] : (uint32_t)i;
    const double T = temperature ? (double)temperature[i] : 1.0;
    const bool greedy = (T == 0.0);
    const uint16_t* trow0 = target + (long)i * (K + 1) * ld_t;
    const uint16_t* drow0 = draft + (long)i * K * ld_d;
    // softmax of one row: p(x) = exp((l(x) - m) / T) / S
    auto softmax_row = [&](const uint16_t* row, std::vector<double>& out) {
      out.resize(V);
      double m = -INFINITY;
      for (int x = 0; x < V; ++x) m = std::max(m, (double)bf16_to_float(row[x]));
      double S = 0.0;
      for (int x = 0; x < V; ++x) {
        out[x] = std::exp(((double)bf16_to_float(row[x]) - m) / T);
        S += out[x];
      }
      for (int x = 0; x < V; ++x) out[x] /= S;
    };
    auto race_d = [&](const std::vector<double>& p, const std::vector<double>* q, uint32_t j,
                      double* margin) {
      int best_x = -1;
      double best_k = 0.0, second_k = 0.0;
      for (int x = 0; x < V; ++x) {
        const double res = q ? std::max(p[x] - (*q)[x], 0.0) : std::max(p[x], 0.0);
        const double key = res / (double)race_E(seed, rid, j, (uint32_t)x);
        if (key > best_k) {
          second_k = best_k;
          best_k = key;
          best_x = x;
        } else if (key > second_k) {
          second_k = key;
        }
      }
      *margin = best_k > 0.0 ? (best_k - second_k) / best_k : 0.0;
      return best_x;
    };
    int a = K;
    int32_t e = 0;
    for (int j = 0; j < K; ++j) {
      if (p_at) p_at[(long)i * K + j] = -1.0f;
      if (q_at) q_at[(long)i * K + j] = -1.0f;
      if (acc_margin) acc_margin[(long)i * K + j] = -1.0;
    }
    std::vector<double> p, q;
    for (int j = 0; j < K; ++j) {
      const int d = drafts[(long)i * K + j];
      const uint16_t* trow = trow0 + (long)j * ld_t;
      const uint16_t* drow = drow0 + (long)j * ld_d;
      if (d < 0 || d >= V) {
        e |= ERR_TOKEN_RANGE;
        if (p_at) p_at[(long)i * K + j] = 0.0f;
        if (q_at) q_at[(long)i * K + j] = 0.0f;
        a = j;
        break;
      }
      bool accept;
      if (greedy) {
        double m;
        const int am = argmax_row([&](int x) { return (double)bf16_to_float(trow[x]); }, V, &m);
        accept = (am == d);
        if (p_at) p_at[(long)i * K + j] = bf16_to_float(trow[d]);
        if (q_at) q_at[(long)i * K + j] = bf16_to_float(drow[d]);
        if (acc_margin) acc_margin[(long)i * K + j] = m;
      } else {
        softmax_row(trow, p);
        softmax_row(drow, q);
        const double P = p[d], Q = q[d];
        if (p_at) p_at[(long)i * K + j] = (float)P;
        if (q_at) q_at[(long)i * K + j] = (float)Q;
        const double uq = accept_uniform(seed, rid, (uint32_t)j) * Q;
        accept = uq < P;
        if (acc_margin) {
          const double mx = std::max(P, uq);
          acc_margin[(long)i * K + j] = mx > 0 ? std::fabs(P - uq) / mx : 0.0;
        }
      }
      if (!accept) {
        a = j;
        break;
      }
    }
    int b;
    double rm = 0.0;
    if (greedy) {
      const uint16_t* trow = trow0 + (long)a * ld_t;
      b = argmax_row([&](int x) { return (double)bf16_to_float(trow[x]); }, V, &rm);
    } else if (a < K) {
      // p and q of row a are still the ones computed for the rejected draft, unless the
      // rejection came from an out-of-range token, in which case compute them now.
      if (e & ERR_TOKEN_RANGE) {
        softmax_row(trow0 + (long)a * ld_t, p);
        softmax_row(drow0 + (long)a * ld_d, q);
      }
      b = race_d(p, &q, (uint32_t)a, &rm);
      if (b < 0) b = race_d(p, nullptr, (uint32_t)a, &rm);  // R4
    } else {
      softmax_row(trow0 + (long)K * ld_t, p);
      b = race_d(p, nullptr, (uint32_t)K, &rm);
    }
    if (b < 0) {
      e |= ERR_ZERO_ROW;
      b = 0;
    }
    for (int t = 0; t <= K; ++t) {
      int32_t tok = -1;
      if (t < a) tok = drafts[(long)i * K + t];
      else if (t == a) tok = b;
      out_tokens[(long)i * (K + 1) + t] = tok;
    }
    num_accepted[i] = a;
    if (race_margin) race_margin[i] = rm;
    errs[i] = e;
  });
  if (err) {
    int32_t e = 0;
    for (int i = 0; i < B; ++i) e |= errs[i];
    *err |= e;
  }
  return 0;
}

// P-EAGLE draft-batch rebuild [PE] "并行草稿生成的挑战", "Triton Kernel", "Hidden State 管理".
// Request r gets L_r = a_r + K drafter slots: its accepted drafts d_1..d_a, the final verify
// token b_r, then K-1 MASK slots; start_loc is the exclusive prefix sum of L. Slots from
// total_out to capacity are padding (id -1, position 0, slot -1, map -1, not masked).
int oracle_pdraft_expand(int B, int K, const int32_t* out_tokens, const int32_t* num_accepted,
                         const int32_t* pos0, const int32_t* block_table, int max_blocks,
                         int block_size, int32_t mask_token_id, int capacity, int32_t* input_ids,
                         int32_t* positions, int32_t* slot_mapping, int32_t* hidden_map,
                         uint8_t* is_masked, uint8_t* is_rejected, int32_t* start_loc,
                         int32_t* new_token_idx, int32_t* total_out, int32_t* err,
                         const int32_t* cu) {
  if (B < 0 || K < 1 || block_size < 1 || max_blocks < 0) return -1;
  int32_t e = 0;
  long total = 0;
  for (int r = 0; r < B; ++r) {
    int Kr = K;          // this request's draft count (R17)
    long t0 = (long)r * (K + 1);  // its first target hidden row
    if (cu) {
      Kr = cu[r + 1] - cu[r];
      if (Kr < 0 || Kr > K) {
        e |= ERR_DRAFT_COUNT;
        Kr = Kr < 0 ? 0 : K;
      }
      t0 = (long)cu[r] + r;
    }
    int a = num_accepted[r];
    if (a < 0 || a > Kr) {
      e |= ERR_NUM_ACCEPTED;
      a = std::min(std::max(a, 0), Kr);
    }
    const int L = a + Kr;
    start_loc[r] = (int32_t)total;
    for (int j = 0; j < L; ++j) {
      const long i = total + j;
      if (i >= capacity) {
        e |= ERR_TOTAL_RANGE;
        break;
      }
      input_ids[i] = (j <= a) ? out_tokens[(long)r * (K + 1) + j] : mask_token_id;
      const long pos = (long)pos0[r] + 1 + j;
      positions[i] = (int32_t)pos;
      int32_t slot = -1;
      const long blk = pos >= 0 ? pos / block_size : -1;
      if (blk < 0 || blk >= max_blocks) {
        e |= ERR_BLOCK_TABLE;
      } else {
        const long phys = block_table[(long)r * max_blocks + blk];
        const long s = phys * block_size + pos % block_size;
        if (phys < 0 || s > 2147483647L) e |= ERR_BLOCK_TABLE;
        else slot = (int32_t)s;
      }
      slot_mapping[i] = slot;
      hidden_map[i] = (j <= a) ? (int32_t)(t0 + j) : -1;
      is_masked[i] = (j > a) ? 1 : 0;
    }
    for (int j = 0; j <= K; ++j)
      is_rejected[(long)r * (K + 1) + j] = (j >= 1 && j > a && j <= Kr) ? 1 : 0;
    for (int k = 0; k < K; ++k)
      new_token_idx[(long)r * K + k] = k < Kr ? (int32_t)(total + a + k) : -1;
    total += L;
  }
  start_loc[B] = (int32_t)total;
  *total_out = (int32_t)total;
  for (long i = total; i < capacity; ++i) {
    input_ids[i] = -1;
    positions[i] = 0;
    slot_mapping[i] = -1;
    hidden_map[i] = -1;
    is_masked[i] = 0;
  }
  if (err) *err |= e;
  return 0;
}

// Padded drafter batch (R14) with its hidden states: every one of the B*2K rows is written.
int oracle_pdraft_prepare_padded(int B, int K, const int32_t* out_tokens,
                                 const int32_t* num_accepted, const int32_t* pos0,
                                 const int32_t* block_table, int max_blocks, int block_size,
                                 int32_t mask_token_id, int32_t* input_ids, int32_t* positions,
                                 int32_t* slot_mapping, int32_t* hidden_map, uint8_t* is_masked,
                                 uint8_t* rejected, int32_t* scatter_map, int32_t* new_token_idx,
                                 int H, const uint16_t* target_hidden, long ld_in, int n_in_rows,
                                 const uint16_t* h_shared, uint16_t* out_hidden, long ld_out,
                                 int32_t* err) {
  if (B < 0 || K < 1 || block_size < 1 || max_blocks < 0 || H < 1) return -1;
  const int W = 2 * K;
  int32_t e = 0;
  for (int r = 0; r < B; ++r) {
    int a = num_accepted[r];
    if (a < 0 || a > K) {
      e |= ERR_NUM_ACCEPTED;
      a = std::min(std::max(a, 0), K);
    }
    for (int j = 0; j < W; ++j) {
      const long i = (long)r * W + j;
      const bool live = j < a + K;
      const long pos = (long)pos0[r] + 1 + j;
      input_ids[i] = (j <= a) ? out_tokens[(long)r * (K + 1) + j] : mask_token_id;
      positions[i] = (int32_t)pos;
      int32_t slot = -1;
      if (live) {
        const long blk = pos >= 0 ? pos / block_size : -1;
        if (blk < 0 || blk >= max_blocks) {
          e |= ERR_BLOCK_TABLE;
        } else {
          const long phys = block_table[(long)r * max_blocks + blk];
          const long sl = phys * block_size + pos % block_size;
          if (phys < 0 || sl > 2147483647L) e |= ERR_BLOCK_TABLE;
          else slot = (int32_t)sl;
        }
      }
      slot_mapping[i] = slot;
      long m = (j <= a) ? (long)r * (K + 1) + j : -1;
      hidden_map[i] = (int32_t)m;
      is_masked[i] = (live && j > a) ? 1 : 0;
      rejected[i] = live ? 0 : 1;
      if (m >= n_in_rows) {
        e |= ERR_MAP_RANGE;
        m = -1;
      }
      const uint16_t* src = m >= 0 ? target_hidden + m * ld_in : h_shared;
      std::memcpy(out_hidden + i * ld_out, src, (size_t)H * sizeof(uint16_t));
    }
    for (int j = 0; j <= K; ++j)
      scatter_map[(long)r * (K + 1) + j] = (j <= a) ? (int32_t)((long)r * W + j) : -1;
    for (int k = 0; k < K; ++k) new_token_idx[(long)r * K + k] = (int32_t)((long)r * W + a + k);
  }
  if (err) *err |= e;
  return 0;
}

// Hidden-state gather [PE] "Hidden State 管理": row i < total_out takes the target hidden
// row hidden_map[i], or h_shared where the map is -1. Rows from total_out on are not written.
// Rows are bf16, moved as raw 16-bit words.
int oracle_hidden_gather(int capacity, int H, const int32_t* total_out, const int32_t* hidden_map,
                         const uint16_t* target_hidden, long ld_in, int n_in_rows,
                         const uint16_t* h_shared, uint16_t* out_hidden, long ld_out,
                         int32_t* err) {
  if (capacity < 0 || H < 1) return -1;
  int32_t e = 0;
  long n = *total_out;
  if (n < 0 || n > capacity) {
    e |= ERR_TOTAL_RANGE;
    n = std::min<long>(std::max<long>(n, 0), capacity);
  }
  for (long i = 0; i < n; ++i) {
    const long m = hidden_map[i];
    const uint16_t* src = h_shared;
    if (m >= 0) {
      if (m < n_in_rows) src = target_hidden + m * ld_in;
      else e |= ERR_MAP_RANGE;
    }
    std::memcpy(out_hidden + i * ld_out, src, (size_t)H * sizeof(uint16_t));
  }
  if (err) *err |= e;
  return 0;
}

// Drafter-side sampling (R13) on fp32 probability rows: row (i*K + k) at q + row*ld is the
// drafter's distribution for draft k of request i. Keys q(x)/E_x are fp32 divisions (R3), the
// largest wins, lowest x on ties; T == 0 takes the argmax. A row without a positive key gives
// token 0 and ERR_ZERO_ROW. margin (nullable) [B*K] receives (k1 - k2) / k1.
int oracle_draft_sample_probs(int B, int K, int V, const float* q, long ld,
                              const float* temperature, uint64_t seed, const int32_t* req_ids,
                              int32_t* drafts, double* margin, int32_t* err, int nthreads) {
  if (B < 0 || K < 1 || V < 1) return -1;
  std::vector<int32_t> errs((size_t)std::max(B, 1), 0);
  parallel_for(B, nthreads, [&](int i) {
    const uint32_t rid = req_ids ? (uint32_t)req_ids[i] : (uint32_t)i;
    const bool greedy = temperature && temperature[i] == 0.0f;
    for (int k = 0; k < K; ++k) {
      const float* row = q + ((long)i * K + k) * ld;
      double m = 0.0;
      int x;
      if (greedy) {
        x = argmax_row([&](int t) { return (double)row[t]; }, V, &m);
      } else {
        int best_x = -1;
        float best_k = 0.0f, second_k = 0.0f;
        for (int t = 0; t < V; ++t) {
          const float key = std::fmax(row[t], 0.0f) / race_E(seed, rid, (uint32_t)k, t, 2u);
          if (key > best_k) {
            second_k = best_k;
            best_k = key;
            best_x = t;
          } else if (key > second_k) {
            second_k = key;
          }
        }
        m = best_k > 0.0f ? ((double)best_k - (double)second_k) / best_k : 0.0;
        x = best_x;
        if (x < 0) {
          errs[i] |= ERR_ZERO_ROW;
          x = 0;
        }
      }
      drafts[(long)i * K + k] = x;
      if (margin) margin[(long)i * K + k] = m;
    }
  });
  if (err) {
    int32_t e = 0;
    for (int i = 0; i < B; ++i) e |= errs[i];
    *err |= e;
  }
  return 0;
}

// Drafter-side sampling (R13) on bf16 logit rows: q = softmax(l / T) in double, keys q/E in
// double; T == 0 takes the argmax of the raw logits.
int oracle_draft_sample_logits(int B, int K, int V, const uint16_t* logits, long ld,
                               const float* temperature, uint64_t seed, const int32_t* req_ids,
                               int32_t* drafts, double* margin, int32_t* err, int nthreads) {
  if (B < 0 || K < 1 || V < 1) return -1;
  std::vector<int32_t> errs((size_t)std::max(B, 1), 0);
  parallel_for(B, nthreads, [&](int i) {
    const uint32_t rid = req_ids ? (uint32_t)req_ids[i] : (uint32_t)i;
    const double T = temperature ? (double)temperature[i] : 1.0;
    std::vector<double> qv((size_t)V);
    for (int k = 0; k < K; ++k) {
      const uint16_t* row = logits + ((long)i * K + k) * ld;
      double m = 0.0;
      int x;
      if (T == 0.0) {
        x = argmax_row([&](int t) { return (double)bf16_to_float(row[t]); }, V, &m);
      } else {
        double mx = -INFINITY;
        for (int t = 0; t < V; ++t) mx = std::max(mx, (double)bf16_to_float(row[t]));
        double S = 0.0;
        for (int t = 0; t < V; ++t) {
          qv[t] = std::exp(((double)bf16_to_float(row[t]) - mx) / T);
          S += qv[t];
        }
        int best_x = -1;
        double best_k = 0.0, second_k = 0.0;
        for (int t = 0; t < V; ++t) {
          const double key = (qv[t] / S) / (double)race_E(seed, rid, (uint32_t)k, t, 2u);
          if (key > best_k) {
            second_k = best_k;
            best_k = key;
            best_x = t;
          } else if (key > second_k) {
            second_k = key;
          }
        }
        m = best_k > 0.0 ? (best_k - second_k) / best_k : 0.0;
        x = best_x;
        if (x < 0) {
          errs[i] |= ERR_ZERO_ROW;
          x = 0;
        }
      }
      drafts[(long)i * K + k] = x;
      if (margin) margin[(long)i * K + k] = m;
    }
  });
  if (err) {
    int32_t e = 0;
    for (int i = 0; i < B; ++i) e |= errs[i];
    *err |= e;
  }
  return 0;
}

}  // extern "C"
