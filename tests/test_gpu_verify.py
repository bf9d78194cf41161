"""GPU parity of sd_verify on probability rows against the oracle: every integer output bit-exact,
p/q at the drafts bit-exact, error bits equal. Cases span several CTA chunks, ragged vocabulary
tails, unaligned rows (scalar loads), greedy and sampled requests, out-of-range drafts, rows
without residual mass, zero rows and exact key ties; then the lossless and expected-tokens
workloads of 10^6 requests, compared request by request."""

import numpy as np
import pytest
import torch

import oracle
import verify_draft_prep_gb300 as sd
from devrun import assert_verify_equal, oracle_verify_rows, random_probs_case, run_verify, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,K,V,greedy,seed", [
    (1, 4, 1024, 0.0, 0),
    (7, 3, 1001, 0.3, 1),          # ragged tail (V % 4 == 1)
    (16, 5, 4099, 0.5, 2),         # V % 4 == 3
    (33, 8, 20000, 0.25, 3),       # several CTAs per row
    (9, 16, 70001, 0.4, 4),        # K = SD_K_MAX, cluster of 8, ragged
    (64, 1, 8, 0.2, 5),            # tiny vocabulary
    (5, 2, 1, 0.4, 6),             # V = 1
])
def test_random_cases_bit_exact(B, K, V, greedy, seed):
    rng = np.random.default_rng(100 + seed)
    p, q, d, T = random_probs_case(rng, B, K, V, sigma=0.7, greedy_frac=greedy)
    got = run_verify(to_dev(p), to_dev(q), to_dev(d), to_dev(T), seed=seed * 7919)
    want = oracle_verify_rows(torch.from_numpy(p), torch.from_numpy(q), torch.from_numpy(d),
                              torch.from_numpy(T), seed=seed * 7919)
    assert_verify_equal(got, want)


def test_unaligned_rows_use_scalar_path():
    rng = np.random.default_rng(11)
    B, K, V, ld = 12, 3, 5003, 5005  # row stride not a multiple of 4 elements
    p, q, d, T = random_probs_case(rng, B, K, V, greedy_frac=0.3)
    pt = torch.zeros(B * (K + 1), ld)
    qt = torch.zeros(B * K, ld)
    pt[:, :V] = torch.from_numpy(p)
    qt[:, :V] = torch.from_numpy(q)
    got = run_verify(pt.cuda()[:, :V], qt.cuda()[:, :V], to_dev(d), to_dev(T), seed=5)
    want = oracle_verify_rows(torch.from_numpy(p), torch.from_numpy(q), torch.from_numpy(d),
                              torch.from_numpy(T), seed=5)
    assert_verify_equal(got, want)
    # an offset base pointer (4-byte aligned only)
    big = torch.zeros(B * (K + 1) * V + 1).cuda()
    big[1:] = torch.from_numpy(p).reshape(-1).cuda()
    got2 = run_verify(big[1:].view(B * (K + 1), V), to_dev(q), to_dev(d), to_dev(T), seed=5)
    assert_verify_equal(got2, want)


def test_edge_cases_bit_exact():
    rng = np.random.default_rng(12)
    B, K, V = 10, 4, 3000
    p, q, d, T = random_probs_case(rng, B, K, V, zero_frac=0.3, greedy_frac=0.2)
    d[0, 0] = V          # out of range at the first draft
    d[1, 2] = -3         # out of range later (examined only if drafts 0, 1 pass)
    p3 = p.reshape(B, K + 1, V)
    q3 = q.reshape(B, K, V)
    q3[2] = p3[2, :K] * 2          # p <= q: no residual mass on any row
    p3[3] = 0                      # a zero request: zero-row fallback
    q3[3] = 0
    T[2] = T[3] = 1.0
    got = run_verify(to_dev(p), to_dev(q), to_dev(d), to_dev(T), seed=77)
    want = oracle_verify_rows(torch.from_numpy(p), torch.from_numpy(q), torch.from_numpy(d),
                              torch.from_numpy(T), seed=77)
    assert want["err"] & oracle.ERR_TOKEN_RANGE and want["err"] & oracle.ERR_ZERO_ROW
    assert_verify_equal(got, want)


def test_exact_key_ties():
    # two entries with equal fp32 E and equal residual on a rejected row: lowest index wins
    V = 60000
    seed, j = 4, 0
    E = np.array([oracle.race_E(seed, 0, j, x) for x in range(V)], np.float32)
    order = np.argsort(E, kind="stable")
    same = np.nonzero(E[order[1:]] == E[order[:-1]])[0]
    lo, hi = sorted((int(order[same[0]]), int(order[same[0] + 1])))
    p = np.zeros((2, V), np.float32)
    q = np.zeros((1, V), np.float32)
    p[0, [lo, hi]] = 0.5
    p[1] = 1.0 / V
    q[0, 7] = 1.0
    d = np.array([[7]], np.int32)   # P = 0 at 7: always rejected, residual = p
    got = run_verify(to_dev(p), to_dev(q), to_dev(d), seed=seed)
    assert got["num_accepted"][0] == 0 and got["out_tokens"][0, 0] == lo
    want = oracle_verify_rows(torch.from_numpy(p), torch.from_numpy(q), torch.from_numpy(d),
                              seed=seed)
    assert_verify_equal(got, want)


def test_lossless_workload_million_requests():
    V, K, N = 8, 2, 1_000_000
    P = np.array([[0.30, 0.05, 0.15, 0.02, 0.20, 0.08, 0.12, 0.08],
                  [0.05, 0.05, 0.40, 0.10, 0.10, 0.05, 0.05, 0.20],
                  [0.125, 0.25, 0.05, 0.075, 0.1, 0.2, 0.1, 0.1]], np.float32)
    Q = np.array([[0.10, 0.25, 0.15, 0.10, 0.05, 0.15, 0.10, 0.10],
                  [0.20, 0.10, 0.20, 0.10, 0.10, 0.10, 0.10, 0.10]], np.float32)
    rng = np.random.default_rng(13)
    drafts = np.stack([rng.choice(V, size=N, p=Q[j].astype(np.float64) / Q[j].astype(np.float64).sum())
                       for j in range(K)], 1).astype(np.int32)
    target = np.ascontiguousarray(np.broadcast_to(P, (N, K + 1, V))).reshape(N * (K + 1), V)
    draft = np.ascontiguousarray(np.broadcast_to(Q, (N, K, V))).reshape(N * K, V)
    got = run_verify(to_dev(target), to_dev(draft), to_dev(drafts), seed=13)
    want = oracle.verify_probs(target.reshape(N, K + 1, V), draft.reshape(N, K, V), drafts,
                               seed=13)
    assert_verify_equal(got, want)
    # and the first token follows p_0 (chi-square, alpha 1e-3)
    from scipy import stats
    c = np.bincount(got["out_tokens"][:, 0], minlength=V)
    e = N * P[0].astype(np.float64) / P[0].sum()
    assert ((c - e) ** 2 / e).sum() < stats.chi2.ppf(1 - 1e-3, V - 1)


@pytest.mark.parametrize("beta,gamma", [(0.5, 4), (0.8, 4), (0.9, 6)])
def test_expected_tokens_workload(beta, gamma):
    V, N = 8, 1_000_000
    q = np.array([0.25] * 4 + [0.0] * 4, np.float32)
    p = np.array([beta * 0.25] * 4 + [(1 - beta) * 0.25] * 4, np.float32)
    rng = np.random.default_rng(gamma)
    drafts = rng.integers(0, 4, size=(N, gamma), dtype=np.int32)
    target = np.broadcast_to(p, (N * (gamma + 1), V))
    draft = np.broadcast_to(q, (N * gamma, V))
    got = run_verify(to_dev(target), to_dev(draft), to_dev(drafts), seed=gamma)
    want = oracle.verify_probs_strided(N, gamma, V, p, 0, q, 0, drafts, seed=gamma)
    assert_verify_equal(got, want)
    mean = (got["num_accepted"] + 1).mean()
    cf = (1 - beta ** (gamma + 1)) / (1 - beta)
    assert abs(mean - cf) < 4 * (got["num_accepted"] + 1).std() / np.sqrt(N)


def test_err_pointer_optional_and_stream_order():
    rng = np.random.default_rng(14)
    p, q, d, T = random_probs_case(rng, 4, 2, 500)
    B, K = d.shape
    s = torch.cuda.Stream()
    outs = torch.zeros(B, K + 1, dtype=torch.int32, device="cuda")
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    pt, qt, dt = to_dev(p), to_dev(q), to_dev(d)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        sd.sd_verify(pt, qt, dt, outs, acc, seed=3)
    s.synchronize()
    want = oracle_verify_rows(torch.from_numpy(p), torch.from_numpy(q), torch.from_numpy(d),
                              seed=3)
    assert np.array_equal(outs.cpu().numpy(), want["out_tokens"])
    assert np.array_equal(acc.cpu().numpy(), want["num_accepted"])


@pytest.mark.parametrize("B,K,V,seed", [
    (1, 4, 8192, 20),       # one request spread over every CTA of the grid
    (3, 5, 20001, 21),      # ragged tail
    (64, 5, 50000, 22),
    (700, 2, 9000, 23),     # more requests than CTAs: several segments per CTA
    (40, 16, 131071, 24),
])
def test_all_sampled_path_bit_exact(B, K, V, seed):
    # temperature NULL: every request samples; the library takes its accept + race kernels
    rng = np.random.default_rng(300 + seed)
    p, q, d, _ = random_probs_case(rng, B, K, V, sigma=0.8)
    got = run_verify(to_dev(p), to_dev(q), to_dev(d), None, seed=seed)
    want = oracle_verify_rows(torch.from_numpy(p), torch.from_numpy(q), torch.from_numpy(d),
                              None, seed=seed)
    assert_verify_equal(got, want)


def test_all_sampled_path_edge_cases():
    rng = np.random.default_rng(25)
    B, K, V = 12, 4, 10007
    p, q, d, _ = random_probs_case(rng, B, K, V, zero_frac=0.3)
    d[0, 0] = V
    d[1, 1] = -5
    p3 = p.reshape(B, K + 1, V)
    q3 = q.reshape(B, K, V)
    q3[2] = p3[2, :K] * 2          # no residual mass: whole-row fallback on p
    p3[3] = 0                      # zero request
    q3[3] = 0
    got = run_verify(to_dev(p), to_dev(q), to_dev(d), None, seed=99)
    want = oracle_verify_rows(torch.from_numpy(p), torch.from_numpy(q), torch.from_numpy(d),
                              None, seed=99)
    assert want["err"] & oracle.ERR_TOKEN_RANGE and want["err"] & oracle.ERR_ZERO_ROW
    assert_verify_equal(got, want)
    # unaligned rows (scalar loads) on the same path
    pt = torch.zeros(B * (K + 1) * V + 1).cuda()
    pt[1:] = torch.from_numpy(p).reshape(-1).cuda()
    got2 = run_verify(pt[1:].view(B * (K + 1), V), to_dev(q), to_dev(d), None, seed=99)
    assert_verify_equal(got2, want)


@pytest.mark.parametrize("temperature", ["mixed", None])
def test_request_base_shards_reproduce_the_whole_batch(temperature):
    # a batch verified as two shards, each with request_base = its first request's index,
    # gives bit for bit what one call over the whole batch gives (both kernel paths)
    rng = np.random.default_rng(31)
    B, K, V = 10, 4, 30011
    p, q, d, T = random_probs_case(rng, B, K, V, greedy_frac=0.3 if temperature else 0.0)
    T = to_dev(T) if temperature else None
    pt, qt, dt = to_dev(p), to_dev(q), to_dev(d)
    whole = run_verify(pt, qt, dt, T, seed=7)
    s = 3
    lo = run_verify(pt[:s * (K + 1)], qt[:s * K], dt[:s], None if T is None else T[:s], seed=7)
    hi = run_verify(pt[s * (K + 1):], qt[s * K:], dt[s:], None if T is None else T[s:], seed=7,
                    request_base=s)
    for k in ("out_tokens", "num_accepted", "p_at_draft", "q_at_draft"):
        assert np.array_equal(np.concatenate([lo[k], hi[k]]).view(np.int32),
                              whole[k].view(np.int32)), k
    want = oracle_verify_rows(torch.from_numpy(p), torch.from_numpy(q), torch.from_numpy(d),
                              None if T is None else T.cpu(), seed=7, req_ids=np.arange(s, B))
    assert_verify_equal(hi, want, check_err=False)
    # a shard without request_base draws other numbers: the shifted counters matter
    if temperature is None:
        shifted = run_verify(pt[s * (K + 1):], qt[s * K:], dt[s:], None, seed=7)
        assert not np.array_equal(shifted["out_tokens"], hi["out_tokens"])


def test_pinned_host_inputs_match_device_inputs():
    # the kernels may read their row inputs straight from pinned host memory (over the host link)
    rng = np.random.default_rng(61)
    B, K, V = 6, 3, 20011
    p, q, d, T = random_probs_case(rng, B, K, V, greedy_frac=0.3)
    dev = run_verify(to_dev(p), to_dev(q), to_dev(d), to_dev(T), seed=5)
    hp = torch.from_numpy(p).pin_memory()
    hq = torch.from_numpy(q).pin_memory()
    out = dict(out_tokens=torch.empty(B, K + 1, dtype=torch.int32, device="cuda"),
               num_accepted=torch.empty(B, dtype=torch.int32, device="cuda"))
    sd.sd_verify(hp, hq, to_dev(d), out["out_tokens"], out["num_accepted"],
                 temperature=to_dev(T), seed=5,
                 workspace_buf=torch.zeros(16 * B, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert np.array_equal(out["out_tokens"].cpu().numpy(), dev["out_tokens"])
    assert np.array_equal(out["num_accepted"].cpu().numpy(), dev["num_accepted"])
