"""Pins for greedy verification and the exponential race.

Greedy (speculative-decoding explainer, section "边界与代价": at temperature 0 the output
matches greedy decoding token for token) reduces to numpy.argmax, which returns the first
maximal index -- the tie rule. The race argmax r(x)/E_x reduces to known answers on special
rows: a one-hot residual picks its only token whatever E is; a residual that is constant on a
set S picks the member of S with the smallest E; and over many requests the race token follows
r / sum(r) (the exponential-race identity), checked by chi-square.
"""

import numpy as np
from scipy import stats

import oracle


def test_greedy_matches_numpy_argmax_with_ties():
    rng = np.random.default_rng(7)
    B, K, V = 400, 4, 50
    p = rng.dirichlet(np.ones(V), size=(B, K + 1)).astype(np.float32)
    # plant exact ties at the maximum on a third of the rows
    for b in range(0, B, 3):
        for j in range(K + 1):
            m = p[b, j].max()
            idx = rng.choice(V, size=2, replace=False)
            p[b, j, idx] = m
    q = rng.dirichlet(np.ones(V), size=(B, K)).astype(np.float32)
    am = p.argmax(axis=-1)  # first maximal index
    drafts = am[:, :K].copy().astype(np.int32)
    # make request b wrong at row b % (K+1) (no wrong draft when b % (K+1) == K)
    for b in range(B):
        j = b % (K + 1)
        if j < K:
            drafts[b, j] = (am[b, j] + 1 + rng.integers(0, V - 1)) % V
    res = oracle.verify_probs(p, q, drafts, temperature=np.zeros(B, np.float32))
    for b in range(B):
        a = 0
        while a < K and drafts[b, a] == am[b, a]:
            a += 1
        assert res["num_accepted"][b] == a
        assert list(res["out_tokens"][b, :a]) == list(drafts[b, :a])
        assert res["out_tokens"][b, a] == am[b, a]
        assert np.all(res["out_tokens"][b, a + 1:] == -1)


def test_one_hot_residual():
    V = 300
    for x in (0, 1, 137, 299):
        p = np.zeros(V, np.float32)
        q = np.zeros(V, np.float32)
        p[x] = 0.5
        p[(x + 1) % V] = 0.5
        q[(x + 1) % V] = 0.5  # residual max(0, p - q) is one-hot at x
        for seed in range(5):
            tok, _ = oracle.race_row(p, q, seed, 3, 2)
            assert tok == x


def test_constant_residual_on_a_set_picks_smallest_E():
    rng = np.random.default_rng(8)
    V = 97
    for trial in range(50):
        S = np.sort(rng.choice(V, size=int(rng.integers(1, 20)), replace=False))
        p = np.zeros(V, np.float32)
        p[S] = 1.0 / 64
        seed, r, j = int(rng.integers(0, 2**32)), int(trial), 1
        tok, _ = oracle.race_row(p, None, seed, r, j)
        E = np.array([oracle.race_E(seed, r, j, int(x)) for x in S], np.float32)
        assert tok == int(S[np.argmin(E)])  # argmin: lowest index among equal E


def test_all_zero_residual_falls_back_to_p():
    # p <= q everywhere (the rows do not carry the same total), so a rejection leaves no
    # residual mass: the resample races on p of the same row with the same E's.
    V, N = 16, 400
    rng = np.random.default_rng(15)
    q = rng.dirichlet(np.ones(V)).astype(np.float32)
    p = (q * np.float32(0.5)).astype(np.float32)
    assert oracle.race_row(p, q, 9, 0, 0)[0] == -1
    target = np.ascontiguousarray(np.broadcast_to(np.stack([p, q]), (N, 2, V)))
    draft = np.ascontiguousarray(np.broadcast_to(q, (N, 1, V)))
    drafts = rng.integers(0, V, (N, 1)).astype(np.int32)
    res = oracle.verify_probs(target, draft, drafts, seed=9)
    rejected = np.nonzero(res["num_accepted"] == 0)[0]
    assert 100 < rejected.size < 300  # accept probability p/q = 1/2
    for r in rejected:
        assert res["out_tokens"][r, 0] == oracle.race_row(p, None, 9, int(r), 0)[0]
    assert res["err"] == 0
    # a fully-zero target row raises the zero-row flag and emits token 0
    z = np.zeros((1, 2, V), np.float32)
    res = oracle.verify_probs(z, z[:, :1], np.array([[5]], np.int32), seed=1)
    assert res["num_accepted"][0] == 0 and res["out_tokens"][0, 0] == 0
    assert res["err"] & oracle.ERR_ZERO_ROW


def test_race_follows_residual_over_requests():
    V = 10
    rng = np.random.default_rng(9)
    r = rng.random(V).astype(np.float32)
    r[[2, 7]] = 0
    n = 200_000
    toks = np.array([oracle.race_row(r, None, 5, i, 0)[0] for i in range(n)])
    counts = np.bincount(toks, minlength=V)
    prob = r.astype(np.float64) / r.sum()
    keep = prob > 0
    assert counts[~keep].sum() == 0
    stat = ((counts[keep] - n * prob[keep]) ** 2 / (n * prob[keep])).sum()
    assert stat < stats.chi2.ppf(1 - 1e-3, keep.sum() - 1), stat


def test_exact_key_tie_goes_to_lowest_index():
    # Find two vocab entries whose fp32 E values are equal, give them the same residual and
    # nothing else: their keys tie exactly and the lower index must win (argmax tie rule).
    seed, r, j = 4, 0, 0
    E = np.array([oracle.race_E(seed, r, j, x) for x in range(60000)], np.float32)
    order = np.argsort(E, kind="stable")
    same = np.nonzero(E[order[1:]] == E[order[:-1]])[0]
    assert same.size > 0
    pairs = [(int(min(order[k], order[k + 1])), int(max(order[k], order[k + 1]))) for k in same[:5]]
    for lo, hi in pairs:
        p = np.zeros(60000, np.float32)
        p[[lo, hi]] = 0.5
        tok, margin = oracle.race_row(p, None, seed, r, j)
        assert tok == lo and margin == 0.0
