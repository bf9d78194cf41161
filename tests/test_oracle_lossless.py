"""Lossless pins (speculative-decoding explainer, section "修正拒绝采样"): whatever the drafter,
the verified output follows the target distribution p.

V = 8, one fixed pair (p, q) with a non-trivial overlap, 10^6 requests, one seed. Chi-square
at alpha = 1e-3 against the exact law. A dropped residual term, a flipped accept inequality, a
wrong row index or a race on q instead of p each fail one of these.
"""

import numpy as np
from scipy import stats

import oracle

N = 1_000_000
ALPHA = 1e-3

P0 = np.array([0.30, 0.05, 0.15, 0.02, 0.20, 0.08, 0.12, 0.08], np.float32)
Q0 = np.array([0.10, 0.25, 0.15, 0.10, 0.05, 0.15, 0.10, 0.10], np.float32)
P1 = np.array([0.05, 0.05, 0.40, 0.10, 0.10, 0.05, 0.05, 0.20], np.float32)
Q1 = np.array([0.20, 0.10, 0.20, 0.10, 0.10, 0.10, 0.10, 0.10], np.float32)
P2 = np.array([0.125, 0.25, 0.05, 0.075, 0.1, 0.2, 0.1, 0.1], np.float32)


def _chi2(counts, expected_prob, n):
    counts = np.asarray(counts, np.float64)
    exp = np.asarray(expected_prob, np.float64) * n
    keep = exp >= 5
    c = np.append(counts[keep], counts[~keep].sum())
    e = np.append(exp[keep], exp[~keep].sum())
    if e[-1] == 0:
        c, e = c[:-1], e[:-1]
    stat = ((c - e) ** 2 / e).sum()
    return stat, len(c) - 1


def _run(rows_p, rows_q, seed, rng):
    K = len(rows_q)
    V = rows_p[0].size
    target = np.ascontiguousarray(np.broadcast_to(np.stack(rows_p), (N, K + 1, V)))
    draft = np.ascontiguousarray(np.broadcast_to(np.stack(rows_q), (N, K, V)))
    drafts = np.stack([rng.choice(V, size=N, p=q.astype(np.float64) / q.astype(np.float64).sum())
                       for q in rows_q], axis=1).astype(np.int32)
    return oracle.verify_probs(target, draft, drafts, seed=seed)


def test_first_token_follows_p():
    rng = np.random.default_rng(1)
    res = _run([P0, P1], [Q0], seed=11, rng=rng)
    t1 = res["out_tokens"][:, 0]
    stat, df = _chi2(np.bincount(t1, minlength=8), P0 / P0.sum(), N)
    assert stat < stats.chi2.ppf(1 - ALPHA, df), (stat, df)
    # acceptance rate = sum min(p, q)
    beta = np.minimum(P0, Q0).astype(np.float64).sum()
    acc = (res["num_accepted"] == 1).mean()
    assert abs(acc - beta) < 4 * np.sqrt(beta * (1 - beta) / N)


def test_bonus_follows_p_K():
    rng = np.random.default_rng(2)
    res = _run([P0, P1], [Q0], seed=12, rng=rng)
    sel = res["num_accepted"] == 1
    bonus = res["out_tokens"][sel, 1]
    stat, df = _chi2(np.bincount(bonus, minlength=8), P1 / P1.sum(), sel.sum())
    assert stat < stats.chi2.ppf(1 - ALPHA, df), (stat, df)
    # requests that rejected emit exactly one token
    assert np.all(res["out_tokens"][~sel, 1] == -1)


def test_joint_first_two_tokens_K2():
    rng = np.random.default_rng(3)
    res = _run([P0, P1, P2], [Q0, Q1], seed=13, rng=rng)
    toks = res["out_tokens"]
    a = res["num_accepted"]
    V = 8
    # cells: (t1, none) when a == 0; (t1, t2) when a >= 1
    cell = np.where(a == 0, toks[:, 0], V + toks[:, 0] * V + toks[:, 1])
    counts = np.bincount(cell, minlength=V + V * V)
    p0 = P0.astype(np.float64) / P0.sum()
    q0 = Q0.astype(np.float64)
    beta0 = np.minimum(P0, Q0).astype(np.float64).sum()
    res0 = np.maximum(P0 - Q0, 0).astype(np.float64)
    res0 /= res0.sum()
    p1 = P1.astype(np.float64) / P1.sum()
    prob = np.zeros(V + V * V)
    prob[:V] = (1 - beta0) * res0
    prob[V:] = np.outer(np.minimum(p0, q0), p1).ravel()
    assert abs(prob.sum() - 1) < 1e-6
    stat, df = _chi2(counts, prob / prob.sum(), N)
    assert stat < stats.chi2.ppf(1 - ALPHA, df), (stat, df)
