"""Pins for the oracle's logits variant: per-request temperature softmax, then the same verify.

softmax(l / T) is checked against scipy.special.softmax, greedy (T == 0) against numpy.argmax on
the bf16 logits (exact ties included), and the lossless property against p = softmax(l / T) by
chi-square; the temperature reading (divide the logits by T) is what the chi-square pins.
"""

import numpy as np
import torch
from scipy import special, stats

import oracle


def _bf16(x):
    t = torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16)
    vals = t.float().numpy()
    return bits, vals


def test_probabilities_at_drafts_match_scipy_softmax():
    rng = np.random.default_rng(10)
    B, K, V = 6, 3, 500
    lt_bits, lt = _bf16(2 * rng.standard_normal((B, K + 1, V)))
    ld_bits, ld = _bf16(lt[:, :K] + 0.5 * rng.standard_normal((B, K, V)))
    T = rng.uniform(0.5, 1.2, B).astype(np.float32)
    drafts = rng.integers(0, V, (B, K)).astype(np.int32)
    res = oracle.verify_logits(lt_bits, ld_bits, drafts, temperature=T, seed=3)
    for b in range(B):
        a = res["num_accepted"][b]
        for j in range(K):
            if j <= min(a, K - 1):
                p = special.softmax(lt[b, j].astype(np.float64) / float(T[b]))
                q = special.softmax(ld[b, j].astype(np.float64) / float(T[b]))
                assert abs(res["p_at_draft"][b, j] - p[drafts[b, j]]) < 1e-7
                assert abs(res["q_at_draft"][b, j] - q[drafts[b, j]]) < 1e-7
            else:
                assert res["p_at_draft"][b, j] == -1.0


def test_greedy_on_logits_matches_numpy_argmax():
    rng = np.random.default_rng(11)
    B, K, V = 200, 4, 300
    lt_bits, lt = _bf16(np.round(4 * rng.standard_normal((B, K + 1, V))) / 4)  # many exact ties
    ld_bits, _ = _bf16(rng.standard_normal((B, K, V)))
    am = lt.argmax(axis=-1)
    drafts = am[:, :K].astype(np.int32).copy()
    for b in range(B):
        j = b % (K + 1)
        if j < K:
            drafts[b, j] = (am[b, j] + 1) % V
    res = oracle.verify_logits(lt_bits, ld_bits, drafts, temperature=np.zeros(B, np.float32))
    for b in range(B):
        a = 0
        while a < K and drafts[b, a] == am[b, a]:
            a += 1
        assert res["num_accepted"][b] == a
        assert res["out_tokens"][b, a] == am[b, a]


def test_lossless_with_temperature():
    rng = np.random.default_rng(12)
    V, K, N = 8, 1, 300_000
    T = 0.7
    lt_bits, lt = _bf16(rng.standard_normal((K + 1, V)))
    ld_bits, ld = _bf16(lt[:K] + 0.8 * rng.standard_normal((K, V)))
    q = special.softmax(ld[0].astype(np.float64) / T)
    drafts = rng.choice(V, size=(N, 1), p=q).astype(np.int32)
    res = oracle.verify_logits(np.broadcast_to(lt_bits, (N, K + 1, V)),
                               np.broadcast_to(ld_bits, (N, K, V)), drafts,
                               temperature=np.full(N, T, np.float32), seed=21, margins=False)
    p = special.softmax(lt[0].astype(np.float64) / T)
    counts = np.bincount(res["out_tokens"][:, 0], minlength=V)
    stat = ((counts - N * p) ** 2 / (N * p)).sum()
    assert stat < stats.chi2.ppf(1 - 1e-3, V - 1), stat
    # T = 1 would be a different law: the test would notice a dropped temperature
    p1 = special.softmax(lt[0].astype(np.float64))
    stat1 = ((counts - N * p1) ** 2 / (N * p1)).sum()
    assert stat1 > stats.chi2.ppf(1 - 1e-3, V - 1)
