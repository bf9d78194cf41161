"""Brute-force pins on tiny inputs (speculative-decoding explainer, sections "核心思想" and
"修正拒绝采样").

1. The exact joint law of (a, emitted tokens) for V <= 4, K = 2 is enumerated from the
   definitions -- accept probability = the share of the 2^24-point u grid with u*Q < P,
   residual resample with probability r/sum(r), bonus from p_K -- and compared with a 10^6-
   request histogram of the oracle (chi-square).
2. An independent pure-Python statement of the same step (tests/pyref.py) must match the oracle
   token for token on 1000 random tiny cases, greedy and sampled, with zeros, ties and
   out-of-range drafts.
"""

import itertools
import math

import numpy as np
from scipy import stats

import oracle
import pyref

N = 1_000_000


def _accept_prob(P, Q):
    # u = k / 2^24, k = 0 .. 2^24-1; accept iff k * Q / 2^24 < P (exact in double)
    P, Q = float(P), float(Q)
    if Q == 0.0:
        return 1.0 if P > 0 else 0.0
    t = P * 2**24 / Q
    return min(2**24, math.ceil(t)) / 2**24


def _exact_law(p, q, V):
    """Joint law for K = 2: outcome tuple -> probability."""
    K = 2
    law = {}

    def residual(j):
        r = np.maximum(p[j] - q[j], np.float32(0)).astype(np.float64)
        return r / r.sum()

    def walk(j, prefix, prob):
        if j == K:
            pk = p[K].astype(np.float64)
            for z in range(V):
                law[tuple(prefix + [z])] = law.get(tuple(prefix + [z]), 0) + prob * pk[z] / pk.sum()
            return
        rej_mass = 0.0
        for x in range(V):
            px = q[j][x] / q[j].astype(np.float64).sum() * _accept_prob(p[j][x], q[j][x])
            rej_mass += q[j][x] / q[j].astype(np.float64).sum() * (1 - _accept_prob(p[j][x], q[j][x]))
            if px > 0:
                walk(j + 1, prefix + [x], prob * px)
        if rej_mass > 0:
            res = residual(j)
            for y in range(V):
                if res[y] > 0:
                    key = tuple(prefix + [y, None])
                    law[key] = law.get(key, 0) + prob * rej_mass * res[y]

    walk(0, [], 1.0)
    return law


def test_exact_joint_law_K2():
    rng = np.random.default_rng(5)
    for case in range(3):
        V = 3 + case % 2
        K = 2
        p = rng.dirichlet(np.ones(V), size=K + 1).astype(np.float32)
        q = rng.dirichlet(np.ones(V), size=K).astype(np.float32)
        law = _exact_law(p, q, V)
        assert abs(sum(law.values()) - 1) < 1e-5
        target = np.ascontiguousarray(np.broadcast_to(p, (N, K + 1, V)))
        draft = np.ascontiguousarray(np.broadcast_to(q, (N, K, V)))
        qn = q.astype(np.float64) / q.astype(np.float64).sum(axis=1, keepdims=True)
        drafts = np.stack([rng.choice(V, size=N, p=qn[j]) for j in range(K)], 1).astype(np.int32)
        res = oracle.verify_probs(target, draft, drafts, seed=100 + case)
        a = res["num_accepted"]
        toks = res["out_tokens"]
        keys = list(law.keys())
        index = {k: i for i, k in enumerate(keys)}
        counts = np.zeros(len(keys))
        # encode each request's outcome
        for av in range(K + 1):
            sel = np.nonzero(a == av)[0]
            sub = toks[sel, : av + 1]
            uniq, cnt = np.unique(sub, axis=0, return_counts=True)
            for row, c in zip(uniq, cnt):
                key = tuple(int(v) for v in row) + ((None,) if av < K else ())
                assert key in index, key  # the oracle never emits an impossible outcome
                counts[index[key]] += c
        exp = np.array([law[k] for k in keys]) * N
        keep = exp >= 5
        c = np.append(counts[keep], counts[~keep].sum())
        e = np.append(exp[keep], exp[~keep].sum())
        stat = ((c - e) ** 2 / np.maximum(e, 1e-12)).sum()
        assert stat < stats.chi2.ppf(1 - 1e-3, len(c) - 1), (case, stat, len(c))


def _random_case(rng):
    V = int(rng.integers(1, 7))
    K = int(rng.integers(1, 4))
    kind = rng.integers(0, 4)
    p = rng.dirichlet(np.ones(V), size=K + 1).astype(np.float32)
    q = rng.dirichlet(np.ones(V), size=K).astype(np.float32)
    if kind == 1:  # zeros in both, ties
        p[rng.random(p.shape) < 0.3] = 0
        q[rng.random(q.shape) < 0.3] = 0
        p = np.round(p * 4) / 4
    if kind == 2:  # q == p on some rows: no residual mass
        q[0] = p[0]
    drafts = rng.integers(0, V, size=K).astype(np.int32)
    if kind == 3 and rng.random() < 0.5:
        drafts[rng.integers(0, K)] = V + 3 if rng.random() < 0.5 else -1
    greedy = bool(rng.random() < 0.3)
    if greedy and rng.random() < 0.7:
        drafts = np.array([int(np.argmax(p[j])) for j in range(K)], np.int32)
    return V, K, p, q, drafts, greedy


def test_independent_python_statement_matches():
    rng = np.random.default_rng(6)
    for case in range(1000):
        V, K, p, q, drafts, greedy = _random_case(rng)
        seed = int(rng.integers(0, 2**63))
        rid = int(rng.integers(0, 2**31))
        res = oracle.verify_probs(p[None], q[None], drafts[None],
                                  temperature=np.array([0.0 if greedy else 1.0], np.float32),
                                  seed=seed, req_ids=np.array([rid], np.int32))
        a, toks = pyref.verify_one(p, q, drafts, greedy, seed, rid)
        assert int(res["num_accepted"][0]) == a, case
        assert [int(t) for t in res["out_tokens"][0]] == toks, case
